"""tq_gemm (prefill) against the oracle: bf16 output within the tolerance plus half a bf16 ulp."""
import numpy as np
import pytest
import torch

import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import LinearCase, bf16_half_ulp, check_tolerance, sample_rows

pytestmark = pytest.mark.gpu

B3, B2 = tq.TQ_PACK_B3, tq.TQ_PACK_2BIT


def run(case):
    y = tq.tq_gemm(case.desc, case.codes, case.scales, case.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    return y.float().cpu().numpy()


def check_bf16(y, y_ref, A):
    check_tolerance(y, y_ref, A, extra=bf16_half_ulp(np.maximum(np.abs(y_ref), np.abs(y))))


@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("group", [128, 64])
@pytest.mark.parametrize("M,N,K", [(1, 64, 128), (77, 200, 384), (256, 128, 1024), (300, 257, 640), (130, 96, 2560)])
def test_small_ragged(packing, group, M, N, K):
    case = LinearCase(21, M + N + K, N, K, group, packing, M)
    y_ref, A = case.oracle()
    check_bf16(run(case), y_ref, A)


@pytest.mark.parametrize("shape", inputs.PREFILL["shapes"], ids=lambda s: "x".join(map(str, s)))
def test_prefill_full_size_sampled(shape):
    """(M, K, N) = (2048, 5120, 17408) and (4096, 17408, 5120), 2-bit, group 128: sampled outputs."""
    M, K, N = shape
    case = LinearCase(inputs.seed_of(4), K, N, K, 128, B2, M)
    y = run(case)
    rows = sample_rows(N, 24, seed=1)
    toks = sample_rows(M, 12, seed=2)
    t, s = case.host_rows(rows)
    import oracle as O
    x = case.x_host.float().numpy()[toks]
    y_ref, A, _ = O.ternary_linear(O.pack(t, B2), s, x, K, 128, B2, 128)
    check_bf16(y[np.ix_(toks, rows)], y_ref, A)


def test_prefill_full_size_every_output():
    """(M, K, N) = (2048, 5120, 17408), 2-bit, group 128: all 35.6 M outputs against the oracle."""
    import oracle as O
    M, K, N = inputs.PREFILL["shapes"][0]
    case = LinearCase(inputs.seed_of(4), K, N, K, 128, B2, M)
    y = run(case)
    x = case.x_host.float().numpy()
    for r0 in range(0, N, 2048):
        rows = np.arange(r0, min(N, r0 + 2048))
        t, s = case.host_rows(rows)
        y_ref, A, _ = O.ternary_linear(O.pack(t, B2), s, x, K, 128, B2, 128)
        check_bf16(y[:, rows], y_ref, A)


@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("mag", [1e3, 1e-4])
def test_activation_magnitudes(packing, mag):
    """Large and small activations (x~ held as FP16 without block scaling): within the tolerance."""
    case = LinearCase(22, 3, 200, 1280, 128, packing, 130)
    case.x_host = (case.x_host.float() * mag).to(torch.bfloat16)
    case.x = case.x_host.cuda()
    y_ref, A = case.oracle()
    check_bf16(run(case), y_ref, A)


def test_out_of_fp16_range_is_reported():
    """|x~| beyond the FP16 range (activations ~1e5) records TQ_ERR_RANGE in the device status."""
    case = LinearCase(23, 4, 128, 512, 128, B2, 64)
    case.x = (case.x_host.float() * 1e5).to(torch.bfloat16).cuda()
    tq.tq_gemm(case.desc, case.codes, case.scales, case.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 8          # TQ_ERR_RANGE
    assert tq.tq_device_status() == 0
    # an in-range call afterwards is correct
    case2 = LinearCase(23, 5, 128, 512, 128, B2, 64)
    y_ref, A = case2.oracle()
    check_bf16(run(case2), y_ref, A)


@pytest.mark.parametrize("packing", [B2, B3])
def test_negative_scales(packing):
    """FP16 scales of either sign (the decode flips the sign bit for t = -1): every other group negated."""
    import oracle as O
    case = LinearCase(24, 5, 136, 1280, 64, packing, 96)
    case.scales[:, ::2] = -case.scales[:, ::2]
    y = run(case)
    t, _ = case.host_rows(np.arange(case.N))
    y_ref, A, _ = O.ternary_linear(O.pack(t, packing), case.scales.cpu().numpy(), case.x_host.float().numpy(),
                                   case.K, case.group, packing, 128)
    check_bf16(y, y_ref, A)

