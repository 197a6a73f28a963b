"""tq_gemm_fp8 (prefill with FP8 E4M3 operands) against the oracle.

Two comparisons:
* with the oracle's own FP8 statement (oracle.linear_fp8): without the block transform the two sides
  round the same numbers to E4M3 (bf16 activations and fp16 scales times powers of two are exact in
  fp32 and fp64), so the operands agree bit for bit and the only differences are the tensor cores'
  accumulation and the bf16 output: |y - y8| <= ACC * Aq + half a bf16 ulp, Aq the sum of the
  quantised products' magnitudes.  With the transform (fp32 on the GPU, fp64 in the oracle) an operand
  lying within rounding of an E4M3 midpoint may round the other way: each such flip moves a product
  by at most 2^-3 of max|x~| * max|w|, and two are allowed per output;
* with the exact result (oracle.ternary_linear): within the E4M3 bound the oracle pins derive
  (tq_testlib.fp8_bound), plus the accumulation and output terms above.
"""
import numpy as np
import pytest
import torch

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import LinearCase, bf16_half_ulp, fp8_bound, sample_rows

pytestmark = pytest.mark.gpu

B3, B2 = tq.TQ_PACK_B3, tq.TQ_PACK_2BIT
# Tensor-core accumulation of the E4M3 products, relative to their absolute sum: fp32 accumulation
# order plus the MMA's internal alignment of addends (FP8 MMAs align within a K = 32 step).
ACC = 2.0 ** -12


def run(case):
    y = tq.tq_gemm_fp8(case.desc, case.codes, case.scales, case.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    return y.float().cpu().numpy()


def refs(case, rows=None, x=None):
    """y8 (oracle.linear_fp8), exact y and A, Aq, the flip allowance and the E4M3 bound."""
    rows = np.arange(case.N) if rows is None else np.asarray(rows)
    t, s = case.host_rows(rows)
    codes = O.pack(t, case.packing)
    x = case.x_host.float().numpy() if x is None else x
    y8, A, bad = O.linear_fp8(codes, s, x, case.K, case.group, case.packing, case.fwht_block)
    y, _, _ = O.ternary_linear(codes, s, x, case.K, case.group, case.packing, case.fwht_block)
    assert bad == 0
    xt = O.block_fwht(np.asarray(x, dtype=np.float64), case.fwht_block)
    W = O.dequant(t, s, case.group)
    ea = O.pow2_exponent(np.abs(xt).max(axis=1))
    eb = O.pow2_exponent(np.abs(s.astype(np.float64)).max(axis=1))
    aq = O.e4m3(xt * np.ldexp(1.0, -ea)[:, None])
    wq = O.e4m3(W * np.ldexp(1.0, -eb)[:, None])
    Aq = (np.abs(aq) @ np.abs(wq).T) * np.ldexp(1.0, ea[:, None] + eb[None, :])
    flip = 2 * 2.0 ** -3 * np.outer(np.abs(xt).max(axis=1), np.abs(W).max(axis=1)) * 1.07
    return dict(y8=y8, y=y, A=A, Aq=Aq, flip=flip, bound=fp8_bound(xt, W, ea, eb))


def check(yg, r, transform, what=""):
    out = bf16_half_ulp(np.maximum(np.abs(yg), np.abs(r["y8"])))
    tight = ACC * r["Aq"] + out + 1e-30
    if transform:
        tight = tight + r["flip"]
    err = np.abs(yg - r["y8"])
    assert np.isfinite(yg).all()
    worst = np.unravel_index(np.argmax(err / tight), err.shape)
    assert err[worst] <= tight[worst], (f"{what} vs linear_fp8 at {worst}: {yg[worst]!r} vs {r['y8'][worst]!r}, "
                                         f"err {err[worst]:.3e} > {tight[worst]:.3e}")
    loose = r["bound"] + ACC * r["Aq"] + bf16_half_ulp(np.maximum(np.abs(yg), np.abs(r["y"]))) + 1e-30
    err2 = np.abs(yg - r["y"])
    worst = np.unravel_index(np.argmax(err2 / loose), err2.shape)
    assert err2[worst] <= loose[worst], f"{what} vs exact at {worst}: err {err2[worst]:.3e} > {loose[worst]:.3e}"
    return float((err / tight).max())


@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("group", [128, 64])
@pytest.mark.parametrize("M,N,K", [(1, 64, 128), (77, 200, 384), (256, 128, 1024), (300, 257, 640), (130, 96, 2560)])
def test_small_ragged_no_transform(packing, group, M, N, K):
    """Operands identical on both sides: accumulation and bf16 rounding only."""
    case = LinearCase(31, M + N + K, N, K, group, packing, M, fwht_block=0)
    check(run(case), refs(case), False)


@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("M,N,K", [(64, 256, 512), (129, 300, 1280), (200, 512, 3072)])
def test_small_ragged_transform(packing, M, N, K):
    case = LinearCase(32, M + N + K, N, K, 128, packing, M)
    check(run(case), refs(case), True)


def test_row_magnitudes_and_zero_rows():
    """Token rows of magnitude 1e5, 1, 1e-6 and 0 in one call (each row has its own factor), and a
    weight row whose scales are all zero: zero rows give exact zeros."""
    case = LinearCase(33, 5, 192, 1024, 128, B2, 8, fwht_block=0)
    mags = torch.tensor([1e5, 1.0, 1e-6, 0.0, 3e2, 1e-2, 1.0, 7.0])[:, None]
    case.x_host = (case.x_host.float() * mags).to(torch.bfloat16)
    case.x = case.x_host.cuda()
    case.scales[17].zero_()
    yg = run(case)
    t, _ = case.host_rows(np.arange(case.N))
    check(yg, refs_with_scales(case, case.scales.cpu().numpy(), t), False)
    assert (yg[3] == 0).all() and (yg[:, 17] == 0).all()


def refs_with_scales(case, s, t):
    """refs() for scales modified on the device (taken back from it)."""
    class C:
        pass
    c = C()
    c.__dict__.update(case.__dict__)
    c.host_rows = lambda rows: (t[rows], s[rows])
    return refs(c)


def test_inf_records_range_error():
    case = LinearCase(34, 6, 128, 512, 128, B2, 4)
    x = case.x_host.clone()
    x[2, 7] = float("inf")
    tq.tq_gemm_fp8(case.desc, case.codes, case.scales, x.cuda())
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 8   # TQ_ERR_RANGE
    assert tq.tq_device_status() == 0


def test_prefill_full_size_every_output():
    """(M, K, N) = (2048, 5120, 17408), 2-bit, group 128, with the transform: all 35.6 M outputs."""
    M, K, N = inputs.PREFILL["shapes"][0]
    case = LinearCase(inputs.seed_of(4), K, N, K, 128, B2, M)
    yg = run(case)
    worst = 0.0
    for r0 in range(0, N, 2048):
        rows = np.arange(r0, min(N, r0 + 2048))
        worst = max(worst, check(yg[:, rows], refs(case, rows), True, what=f"rows {r0}.."))
    print(f"worst error / bound: {worst:.3f}")


@pytest.mark.parametrize("packing", [B2, B3])
def test_prefill_second_shape_sampled(packing):
    """(M, K, N) = (4096, 17408, 5120): sampled weight rows, every token."""
    M, K, N = inputs.PREFILL["shapes"][1]
    case = LinearCase(inputs.seed_of(4), K + packing, N, K, 128, packing, M)
    yg = run(case)
    rows = sample_rows(N, 40, seed=3)
    check(yg[:, rows], refs(case, rows), True)


def test_matches_fp16_path_closely():
    """The FP8 result stays within the E4M3 bound of the FP16 path's result on the same call."""
    case = LinearCase(35, 7, 512, 2048, 128, B3, 256)
    y8 = run(case)
    y16 = tq.tq_gemm(case.desc, case.codes, case.scales, case.x).float().cpu().numpy()
    r = refs(case)
    assert (np.abs(y8 - y16) <= r["bound"] + ACC * r["Aq"] + 2e-3 * r["A"] + 1e-30).all()


@pytest.mark.parametrize("packing", [B2, B3])
def test_negative_scales(packing):
    """Negative FP16 scales (the E4M3 sign bit flips for t = -1 whatever the scale's sign)."""
    case = LinearCase(36, 8, 200, 1024, 64, packing, 64, fwht_block=0)
    case.scales[:, 1::2] = -case.scales[:, 1::2]
    yg = run(case)
    t, _ = case.host_rows(np.arange(case.N))
    check(yg, refs_with_scales(case, case.scales.cpu().numpy(), t), False)

