"""tq_quantize (offline: rotate, absmean FP16 group scale, ternarize, pack) against the oracle:
bit-exact codes and scales on the same bf16 W, and the quantized matrix working in tq_gemv."""
import numpy as np
import pytest
import torch

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import check_tolerance

pytestmark = pytest.mark.gpu

B3, B2 = tq.TQ_PACK_B3, tq.TQ_PACK_2BIT


def weights(seed, tid, N, K, scale=2.0 ** -6):
    """bf16 W ~ N(0, 1) * 2^-6 with 0.1 % of the entries x20 (the outliers the rotation spreads);
    the power-of-two factor keeps the values bf16-exact."""
    w = inputs.activations(seed, tid, N, K, outlier_frac=0.001)
    return (w.float() * scale).to(torch.bfloat16)


def check_exact(w, group, packing, fwht_block, rows=None):
    N, K = w.shape
    d = tq.desc(N, K, group, packing, fwht_block)
    codes, scales = tq.tq_quantize(d, w.cuda())
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    codes = codes.cpu().numpy().view(np.uint32)
    scales = scales.cpu().numpy()
    rows = np.arange(N) if rows is None else np.asarray(rows)
    wh = w.float().numpy()
    for r0 in range(0, len(rows), 1024):
        rr = rows[r0:r0 + 1024]
        c_ref, s_ref, _ = O.quantize(wh[rr], group, packing, fwht_block)
        assert np.array_equal(codes[rr], c_ref), "codes differ"
        assert np.array_equal(scales[rr].view(np.uint16), s_ref.view(np.uint16)), "scales differ"
    return codes, scales


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("fwht_block", [128, 0])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (33, 1280), (130, 2560)])
def test_bit_exact_small(packing, group, fwht_block, N, K):
    check_exact(weights(31, N + K, N, K), group, packing, fwht_block)


@pytest.mark.parametrize("packing", [B3, B2])
def test_bit_exact_full_size(packing):
    """The 27B-class down projection (5120 x 17408) and gate/up shape (17408 x 5120), every row."""
    for tid, (N, K) in enumerate([(5120, 17408), (17408, 5120)]):
        check_exact(weights(32, tid, N, K), 128, packing, 128)


def test_special_values():
    """All-zero groups (scale 0, t = 0), ties and exact halves, and a scale beyond the FP16 range."""
    w = torch.zeros((3, 256), dtype=torch.bfloat16)
    w[1, :64] = 3 / 16
    w[1, 64:128] = 1 / 16       # without the transform: mean 1/8, so 1/16 is exactly halfway -> 0
    w[2] = -2.0 ** -20
    check_exact(w, 128, B2, 0)
    check_exact(w, 64, B3, 128)
    big = torch.full((1, 128), 3.0e38, dtype=torch.bfloat16)
    d = tq.desc(1, 128, 128, B2, 0)
    tq.tq_quantize(d, big.cuda())
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 8          # TQ_ERR_RANGE


@pytest.mark.parametrize("packing", [B3, B2])
def test_quantized_matrix_in_gemv(packing):
    """The quantized matrix through tq_gemv with the same activations matches the oracle's contraction
    of the oracle's own quantization (which the codes equal bit for bit)."""
    N, K, group, batch = 512, 2048, 128, 4
    w = weights(33, 0, N, K)
    d = tq.desc(N, K, group, packing, 128)
    codes, scales = tq.tq_quantize(d, w.cuda())
    x = inputs.activations(33, 1, batch, K)
    y = tq.tq_gemv(d, codes, scales, x.cuda())
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    c_ref, s_ref, _ = O.quantize(w.float().numpy(), group, packing, 128)
    y_ref, A, bad = O.ternary_linear(c_ref, s_ref, x.float().numpy(), K, group, packing, 128)
    assert bad == 0
    check_tolerance(y.cpu().numpy(), y_ref, A)
    # the ternary layer approximates the dense one, and the rotation helps: with outliers in W, the
    # same quantizer without the transform is clearly worse (the pages' reason for rotating first)
    dense = x.float().numpy().astype(np.float64) @ w.float().numpy().astype(np.float64).T
    rel = np.linalg.norm(y.cpu().numpy() - dense) / np.linalg.norm(dense)
    d0 = tq.desc(N, K, group, packing, 0)
    c0, s0 = tq.tq_quantize(d0, w.cuda())
    y0 = tq.tq_gemv(d0, c0, s0, x.cuda())
    rel0 = np.linalg.norm(y0.cpu().numpy() - dense) / np.linalg.norm(dense)
    assert rel < 0.55 and rel < 0.8 * rel0
