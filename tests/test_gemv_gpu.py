"""tq_gemv (decode) against the oracle: element by element on small and ragged shapes, and on
sampled rows of every linear of the 27B-class decode layer at its full size."""
import numpy as np
import pytest
import torch

import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import LinearCase, check_tolerance, sample_rows

pytestmark = pytest.mark.gpu

B3, B2 = tq.TQ_PACK_B3, tq.TQ_PACK_2BIT


def run(case: LinearCase):
    y = tq.tq_gemv(case.desc, case.codes, case.scales, case.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    return y.cpu().numpy()


def test_single_linear_1024():
    """K = N = 1024, batch 1, base-3, group 128, 0.5 % x20 outliers, seed 0: every output."""
    c = inputs.SINGLE_LINEAR
    case = LinearCase(inputs.seed_of(1), 0, c["N"], c["K"], c["group"], c["packing"], c["B"],
                      outlier_frac=c["outlier_frac"])
    y_ref, A = case.oracle()
    check_tolerance(run(case), y_ref, A)


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("N,K,batch", [(1, 128, 1), (33, 384, 3), (200, 1024, 16), (129, 640, 5), (7, 2560, 8),
                                        (300, 1280, 2)])
def test_small_ragged(packing, group, N, K, batch):
    case = LinearCase(11, N * 7 + batch, N, K, group, packing, batch)
    y_ref, A = case.oracle()
    check_tolerance(run(case), y_ref, A)


@pytest.mark.parametrize("packing", [B3, B2])
def test_no_transform(packing):
    case = LinearCase(12, 3, 96, 512, 128, packing, 4, fwht_block=0)
    y_ref, A = case.oracle()
    check_tolerance(run(case), y_ref, A)


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("batch", [1, 4, 16])
@pytest.mark.parametrize("lin", inputs.dense_layer_linears(), ids=lambda l: l.name)
def test_dense_layer_full_size_sampled(lin, batch, packing):
    """Full-size weights, the launch configuration the benchmark times; 48 sampled rows checked."""
    tid = 100 + inputs.dense_layer_linears().index(lin)
    case = LinearCase(inputs.seed_of(2), tid, lin.N, lin.K, 128, packing, batch)
    y = run(case)
    rows = sample_rows(lin.N, 48, seed=tid)
    y_ref, A = case.oracle(rows)
    check_tolerance(y[:, rows], y_ref, A)


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("batch", [1, 8])
@pytest.mark.parametrize("lin", inputs.stacked_layer_linears()[::2], ids=lambda l: l.name)
def test_stacked_projections_full_size_sampled(lin, batch, packing):
    """The stacked qkv (7168 x 5120) and gate_up (34816 x 5120) projections the stream benchmark calls."""
    tid = 200 + inputs.stacked_layer_linears().index(lin)
    case = LinearCase(inputs.seed_of(5), tid, lin.N, lin.K, 128, packing, batch)
    y = run(case)
    rows = sample_rows(lin.N, 48, seed=tid)
    y_ref, A = case.oracle(rows)
    check_tolerance(y[:, rows], y_ref, A)


def test_zero_trits_and_determinism():
    d = tq.desc(64, 1024, 128, B3)
    codes = tq.tq_pack(d, torch.zeros((64, 1024), dtype=torch.int8, device="cuda"))
    scales = inputs.scales(1, 1, 64, 8, device="cuda")
    x = inputs.activations(1, 1, 4, 1024).cuda()
    y = tq.tq_gemv(d, codes, scales, x)
    # all-zero trits: sum |s t x~| = 0, so the bound is the absolute 1e-5 (the tensor-core path sums
    # (t + 1) x~ and subtracts sum x~, which cancels to ~1e-6 rather than to an exact 0)
    assert torch.max(torch.abs(y)).item() <= 1e-5
    case = LinearCase(13, 1, 512, 2048, 128, B2, 16)
    y1 = tq.tq_gemv(case.desc, case.codes, case.scales, case.x)
    y2 = tq.tq_gemv(case.desc, case.codes, case.scales, case.x)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("mag", [1e4, 1e-6, 0.0])
def test_activation_magnitudes(packing, mag):
    """Per-block exponent handling: very large, very small and all-zero activations."""
    case = LinearCase(14, 2, 160, 1280, 128, packing, 3)
    case.x_host = (case.x_host.float() * mag).to(torch.bfloat16)
    case.x = case.x_host.cuda()
    y_ref, A = case.oracle()
    y = run(case)
    check_tolerance(y, y_ref, A)
    if mag == 0.0:
        assert np.count_nonzero(y) == 0


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("N,K,batch", [(200, 17408, 1), (1, 17408, 16), (1000, 640, 2), (257, 3200, 7)])
def test_split_tiles(packing, N, K, batch):
    """Few rows, long K: tiles are split across many CTAs and summed by the last arriver."""
    case = LinearCase(15, N + batch, N, K, 128, packing, batch)
    y_ref, A = case.oracle()
    check_tolerance(run(case), y_ref, A)
    y2 = tq.tq_gemv(case.desc, case.codes, case.scales, case.x).cpu().numpy()
    assert np.array_equal(y2, run(case))   # deterministic across calls


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("N,K,batch", [(300, 1280, 2), (5120, 17408, 1), (17408, 5120, 4), (129, 640, 16)])
def test_static_weights_flag(packing, N, K, batch):
    """TQ_STATIC_WEIGHTS only moves the first weight loads before the dependent-launch wait: the result
    is bit-identical to the default path, also when the preceding kernel on the stream is a GEMV."""
    case = LinearCase(16, N + batch, N, K, 128, packing, batch)
    d_static = tq.desc(N, K, 128, packing, flags=tq.TQ_STATIC_WEIGHTS)
    y_default = tq.tq_gemv(case.desc, case.codes, case.scales, case.x)
    y_static = [tq.tq_gemv(d_static, case.codes, case.scales, case.x) for _ in range(3)]
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    for y in y_static:
        assert torch.equal(y, y_default)
    rows = sample_rows(N, 64, seed=N)
    y_ref, A = case.oracle(rows)
    check_tolerance(y_default.cpu().numpy()[:, rows], y_ref, A)


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("batch", [2, 16])
@pytest.mark.parametrize("N,K", [(300, 1280), (7168, 5120)])
def test_mixed_magnitude_batch(packing, batch, N, K):
    """Rows of one call 1e7 apart in size (even rows x 1e4, odd rows x 1e-3): each row is held to its
    own bound 1e-3 * sum |s t x~| + 1e-5, so a small row next to a large one must keep its precision."""
    case = LinearCase(17, batch + N, N, K, 128, packing, batch)
    mult = torch.tensor([1e4 if b % 2 == 0 else 1e-3 for b in range(batch)]).reshape(batch, 1)
    case.x_host = (case.x_host.float() * mult).to(torch.bfloat16)
    case.x = case.x_host.cuda()
    rows = np.arange(N) if N <= 1024 else sample_rows(N, 512, seed=N)
    y_ref, A = case.oracle(rows)
    y = run(case)
    check_tolerance(y[:, rows], y_ref, A)


def _graph_of(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("packing", [B3, B2])
@pytest.mark.parametrize("batch", [1, 8])
def test_stacked_projections_graph_replayed_every_output(packing, batch):
    """The launch configuration of the per-call decode stream: the stacked qkv (7168 x 5120) and
    gate_up (34816 x 5120) projections with TQ_STATIC_WEIGHTS, called back to back (qkv, gate_up,
    qkv again) inside a CUDA graph; after a replay every output of every call is compared with the
    oracle."""
    lins = inputs.stacked_layer_linears()
    cases = []
    for lin in (lins[0], lins[2]):
        tid = 300 + lins.index(lin)
        c = LinearCase(inputs.seed_of(5), tid, lin.N, lin.K, 128, packing, batch)
        c.desc = tq.desc(lin.N, lin.K, 128, packing, flags=tq.TQ_STATIC_WEIGHTS)
        cases.append(c)
    ws = torch.empty(max(tq.tq_gemv_workspace_bytes(c.desc, batch) for c in cases), dtype=torch.uint8, device="cuda")
    ys = [torch.empty((batch, c.N), dtype=torch.float32, device="cuda") for c in cases]
    y_again = torch.empty_like(ys[0])

    def step():
        tq.tq_gemv(cases[0].desc, cases[0].codes, cases[0].scales, cases[0].x, y=ys[0], workspace=ws)
        tq.tq_gemv(cases[1].desc, cases[1].codes, cases[1].scales, cases[1].x, y=ys[1], workspace=ws)
        tq.tq_gemv(cases[0].desc, cases[0].codes, cases[0].scales, cases[0].x, y=y_again, workspace=ws)

    g = _graph_of(step)
    for y in ys + [y_again]:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    for c, y in zip(cases, ys):
        yh = y.cpu().numpy()
        for r0 in range(0, c.N, 4096):
            rows = np.arange(r0, min(c.N, r0 + 4096))
            y_ref, A = c.oracle(rows)
            check_tolerance(yh[:, rows], y_ref, A, what=f"N={c.N} rows {r0}..")
    assert torch.equal(y_again, ys[0])


def test_same_shape_every_packing_in_one_process():
    """A 2-bit call, then base-3 and 3-bit calls of the same shape and batch in the same process: each
    packing takes its own kernel (the work-split caches are per packing) and matches the oracle."""
    import oracle as O
    N, K, B = 2048, 5120, 1
    for packing in (tq.TQ_PACK_2BIT, tq.TQ_PACK_B3):
        case = LinearCase(61, packing, N, K, 128, packing, B)
        y = tq.tq_gemv(case.desc, case.codes, case.scales, case.x)
        torch.cuda.synchronize()
        assert tq.tq_device_status() == 0
        y_ref, A = case.oracle()
        check_tolerance(y.cpu().numpy(), y_ref, A, what=f"packing {packing}")
    q = inputs.codes3(61, 3, N, K)
    d3 = tq.desc(N, K, 128, tq.TQ_PACK_3BIT)
    s3 = inputs.scales(61, 4, N, K // 128)
    x3 = inputs.activations(61, 5, B, K)
    y3 = tq.tq_gemv(d3, tq.tq_pack(d3, q.cuda()), s3.cuda(), x3.cuda())
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    y_ref, A, _ = O.ternary_linear(O.pack(q.numpy(), O.PACK_3BIT), s3.numpy(), x3.float().numpy(), K, 128,
                                   O.PACK_3BIT)
    check_tolerance(y3.cpu().numpy(), y_ref, A, what="3-bit")
    assert tq.tq_gemv_kernel_count(d3, B) == 2

