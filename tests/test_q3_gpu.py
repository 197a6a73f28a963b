"""3-bit codes of the non-expert linears: tq_pack / tq_unpack bit-exact against the oracle, and
tq_gemv on them within the stated bound, on small ragged shapes and at full size."""
import numpy as np
import pytest
import torch

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import check_tolerance, sample_rows

pytestmark = pytest.mark.gpu

Q3 = tq.TQ_PACK_3BIT


@pytest.mark.parametrize("N,K", [(1, 1), (3, 63), (5, 64), (7, 200), (33, 640), (64, 5120)])
def test_pack_unpack_bit_exact(N, K):
    q = inputs.codes3(71, N + K, N, K)
    d = tq.desc(N, K, 128, Q3)
    codes = tq.tq_pack(d, q.cuda())
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), O.pack(q.numpy(), O.PACK_3BIT))
    back, bad = tq.tq_unpack(d, codes)
    assert bad.item() == 0 and np.array_equal(back.cpu().numpy(), q.numpy())
    # an invalid word (bit 15 set: the gap between the two halves) is counted
    c2 = codes.clone()
    c2[0, 0] |= 1 << 15
    _, bad2 = tq.tq_unpack(d, c2)
    torch.cuda.synchronize()
    assert bad2.item() == 1
    assert tq.tq_device_status() == 4   # TQ_ERR_INVALID_CODE
    assert tq.tq_device_status() == 0


class Q3Case:
    def __init__(self, seed, tid, N, K, group, batch, fwht_block=128, flags=0):
        self.seed, self.tid, self.N, self.K, self.group = seed, tid, N, K, group
        self.desc = tq.desc(N, K, group, Q3, fwht_block, flags)
        self.fwht_block = fwht_block
        self.codes = tq.tq_pack(self.desc, inputs.codes3(seed, 2 * tid, N, K, device="cuda"))
        self.scales = inputs.scales(seed, 2 * tid + 1, N, K // group, device="cuda").contiguous()
        self.x_host = inputs.activations(seed, tid, batch, K)
        self.x = self.x_host.cuda()

    def oracle(self, rows):
        q = inputs.codes3(self.seed, 2 * self.tid, self.N, self.K, rows=rows).numpy()
        s = inputs.scales(self.seed, 2 * self.tid + 1, self.N, self.K // self.group, rows=rows).numpy()
        y, A, bad = O.ternary_linear(O.pack(q, O.PACK_3BIT), s, self.x_host.float().numpy(), self.K, self.group,
                                     O.PACK_3BIT, self.fwht_block)
        assert bad == 0
        return y, A


@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("N,K,batch", [(1, 128, 1), (37, 384, 3), (200, 1280, 8), (129, 640, 5), (5, 2560, 2),
                                     (300, 896, 16), (64, 128, 11), (190, 3200, 6)])
def test_gemv_small(group, N, K, batch):
    c = Q3Case(72, N + batch, N, K, group, batch)
    y = tq.tq_gemv(c.desc, c.codes, c.scales, c.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    y_ref, A = c.oracle(np.arange(N))
    check_tolerance(y.cpu().numpy(), y_ref, A)


@pytest.mark.parametrize("N,K,batch", [(64, 17408, 2), (128, 9984, 1)])
def test_gemv_k_split(N, K, batch):
    """Few rows, long K: the K-range is split over the CTAs of a cluster (and ragged last units)."""
    c = Q3Case(75, N + K, N, K, 64, batch)
    y = tq.tq_gemv(c.desc, c.codes, c.scales, c.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    y_ref, A = c.oracle(np.arange(N))
    check_tolerance(y.cpu().numpy(), y_ref, A)


def test_noalloc_static_weights_and_graph():
    """tq_gemv_noalloc and TQ_STATIC_WEIGHTS on 3-bit codes: same bits as tq_gemv, and a captured
    graph replays to the same bits."""
    c = Q3Case(76, 3, 1536, 2048, 128, 4, flags=tq.TQ_STATIC_WEIGHTS)
    y = tq.tq_gemv(c.desc, c.codes, c.scales, c.x)
    y_na = tq.tq_gemv_noalloc(c.desc, c.codes, c.scales, c.x)
    torch.cuda.synchronize()
    assert torch.equal(y, y_na)
    y_ref, A = c.oracle(np.arange(1536))
    check_tolerance(y.cpu().numpy(), y_ref, A)
    out = torch.empty_like(y)
    ws = torch.empty(tq.tq_gemv_workspace_bytes(c.desc, 4), dtype=torch.uint8, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tq.tq_gemv(c.desc, c.codes, c.scales, c.x, y=out, workspace=ws)   # warm-up outside capture
        with torch.cuda.graph(g, stream=s):
            tq.tq_gemv(c.desc, c.codes, c.scales, c.x, y=out, workspace=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, y)


def test_gemv_no_transform():
    c = Q3Case(73, 1, 96, 512, 128, 4, fwht_block=0)
    y = tq.tq_gemv(c.desc, c.codes, c.scales, c.x)
    y_ref, A = c.oracle(np.arange(96))
    check_tolerance(y.cpu().numpy(), y_ref, A)


@pytest.mark.parametrize("N,K,batch", [(5120, 5120, 1), (7168, 5120, 4), (4096, 17408, 1), (2048, 4096, 16)])
def test_gemv_full_size_every_output(N, K, batch):
    """Attention-sized and FFN-sized 3-bit linears: every output."""
    c = Q3Case(74, N + K, N, K, 128, batch)
    y = tq.tq_gemv(c.desc, c.codes, c.scales, c.x)
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    yh = y.cpu().numpy()
    for r0 in range(0, N, 2048):
        rows = np.arange(r0, min(N, r0 + 2048))
        y_ref, A = c.oracle(rows)
        check_tolerance(yh[:, rows], y_ref, A, what=f"rows {r0}..")


def test_unsupported_elsewhere():
    d = tq.desc(128, 256, 128, Q3)
    assert tq.tq_gemv_kernel_count(d, 1) == 2
    assert tq.tq_gemv_kernel_count(d, 17) == -1
    assert tq.tq_gemm_workspace_bytes(d, 64) == 0


def test_gemv_wide_output_sampled():
    """The wide-output 3-bit shape the bench times (131072 x 2048, lm_head-like): rows sampled across
    the whole output (the first and last 2048 and two chunks between), batch 1 and 3."""
    for batch in (1, 3):
        c = Q3Case(77, batch, 131072, 2048, 128, batch)
        y = tq.tq_gemv(c.desc, c.codes, c.scales, c.x)
        torch.cuda.synchronize()
        assert tq.tq_device_status() == 0
        yh = y.cpu().numpy()
        for r0 in (0, 40960, 90112, 131072 - 2048):
            rows = np.arange(r0, r0 + 2048)
            y_ref, A = c.oracle(rows)
            check_tolerance(yh[:, rows], y_ref, A, what=f"rows {r0}..")

