"""tq_seq (a decode step: a chain of dependent 2-bit or base-3 GEMVs in one launch) against the oracle.

Each call of the chain is checked on its own input: call 0 on the bf16 x, a TQ_SEQ_X_PREV call on
the GPU's own output of the call before it, a TQ_SEQ_X_SWIGLU_PREV call on silu(gate) * up formed
in fp64 from the GPU's own gate/up output.  The bound is the per-output 1e-3 * sum|s t x~| + 1e-5;
for a SwiGLU input it adds the effect of the kernel forming silu(g) * u in fp32 (a relative input
error below 1e-6, carried through the block transform: |FWHT(dx)_k| <= ||dx_block||_1 / sqrt(128)).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import check_tolerance

pytestmark = pytest.mark.gpu

B2, B3 = tq.TQ_PACK_2BIT, tq.TQ_PACK_B3
BF16, PREV, SWIGLU, RMS = tq.TQ_SEQ_X_BF16, tq.TQ_SEQ_X_PREV, tq.TQ_SEQ_X_SWIGLU_PREV, tq.TQ_SEQ_X_RMS_PREV


class Chain:
    """Seeded weights for a list of (N, K, x_src) calls, the plan, and the per-call oracle check."""

    def __init__(self, seed, shapes, batch, group=128, x_tid=999, packing=B2):
        self.seed, self.shapes, self.batch, self.group, self.packing = seed, shapes, batch, group, packing
        self.descs, self.codes, self.scales, self.ys = [], [], [], []
        for j, (N, K, _) in enumerate(shapes):
            d = tq.desc(N, K, group, packing)
            self.descs.append(d)
            self.codes.append(tq.tq_pack(d, inputs.trits(seed, 2 * j, N, K, device="cuda")))
            self.scales.append(inputs.scales(seed, 2 * j + 1, N, K // group, device="cuda").contiguous())
            self.ys.append(torch.full((batch, N), float("nan"), dtype=torch.float32, device="cuda"))
        self.x_host = inputs.activations(seed, x_tid, batch, shapes[0][1])
        self.x = self.x_host.cuda()
        calls = [(self.descs[j], self.codes[j], self.scales[j], src, self.x if j == 0 else None, self.ys[j])
                 for j, (_, _, src) in enumerate(shapes)]
        self.plan = tq.SeqPlan(calls, batch)

    def run(self):
        self.plan.run()
        torch.cuda.synchronize()
        assert tq.tq_device_status() == 0
        return [y.cpu().numpy() for y in self.ys]

    def call_input(self, j, ys):
        N, K, src = self.shapes[j]
        if src == BF16:
            return self.x_host.float().numpy().astype(np.float64), None
        prev = ys[j - 1].astype(np.float64)
        if src == PREV:
            return prev[:, :K], None
        if src == RMS:
            x = prev[:, :K]
            return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 1e-6), "rms"
        g, u = prev[:, :K], prev[:, K:2 * K]
        return g / (1.0 + np.exp(-g)) * u, "swiglu"

    def check_call(self, j, ys, rows=None, chunk=2048):
        N, K, _ = self.shapes[j]
        x, kind = self.call_input(j, ys)
        rows = np.arange(N) if rows is None else np.asarray(rows)
        worst = 0.0
        for r0 in range(0, len(rows), chunk):
            rr = rows[r0:r0 + chunk]
            t = inputs.trits(self.seed, 2 * j, N, K, rows=rr).numpy()
            s = inputs.scales(self.seed, 2 * j + 1, N, K // self.group, rows=rr).numpy()
            y_ref, A, bad = O.ternary_linear(O.pack(t, self.packing), s, x, K, self.group, self.packing, 128)
            assert bad == 0
            extra = None
            if kind == "rms":
                # the kernel's 1 / rms in fp32 (a sum of K squares): relative error below 2e-6
                extra = 2e-6 * A
            elif kind == "swiglu":
                # relative input error <= 1e-6, through the block transform and |s t|
                W = np.abs(O.dequant(t, s, self.group))                       # [rows, K]
                wsum = W.reshape(len(rr), K // 128, 128).sum(axis=2)          # [rows, blocks]
                xsum = np.abs(x).reshape(x.shape[0], K // 128, 128).sum(axis=2)  # [batch, blocks]
                extra = 1e-6 / math.sqrt(128) * (xsum @ wsum.T)
            worst = max(worst, check_tolerance(ys[j][:, rr], y_ref, A, extra=extra, what=f"call {j} rows {r0}.."))
        return worst


SMALL_G128 = [(2048, 1024, BF16), (1024, 1024, PREV), (4096, 1024, RMS), (1024, 2048, SWIGLU), (1000, 1024, RMS)]
SMALL_G64 = [(512, 512, BF16), (2048, 512, RMS), (512, 1024, SWIGLU), (96, 512, PREV)]


# Base-3 items are 640 trits x 64 rows: K = 1024 and 512 end in a partial item (3 of 5 groups of 128,
# 8 of 10 groups of 64), N = 1000 and 96 in a partial row unit (rows past N read as zero codes).
@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("batch", [1, 2, 3, 4])
def test_chain_small_group128(packing, batch):
    c = Chain(41 + batch, SMALL_G128, batch, packing=packing)
    ys = c.run()
    for j in range(len(SMALL_G128)):
        c.check_call(j, ys)


@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("batch", [1, 2, 8])
def test_chain_small_group64(packing, batch):
    c = Chain(51 + batch, SMALL_G64, batch, group=64, packing=packing)
    ys = c.run()
    for j in range(len(SMALL_G64)):
        c.check_call(j, ys)


@pytest.mark.parametrize("packing", [B2, B3])
def test_chain_full_size_layer_every_output(packing):
    """One 27B-class decoder layer as the decode step calls it (qkv 7168 x 5120 on x; o on the
    attention stand-in = the q part of qkv; gate_up 34816 x 5120 on the RMS-normalised o output;
    down 5120 x 17408 on SwiGLU), then the next layer's qkv on the RMS-normalised layer output;
    batch 1, the configuration of the decode benchmark.
    Every output of every call is compared with the oracle."""
    shapes = [(7168, 5120, BF16), (5120, 5120, PREV), (34816, 5120, RMS), (5120, 17408, SWIGLU), (7168, 5120, RMS)]
    c = Chain(inputs.seed_of(5) + 7, shapes, 1, packing=packing)
    ys = c.run()
    for j in range(len(shapes)):
        c.check_call(j, ys)


def test_base3_full_size_batch8_sampled():
    """The same layer in base-3 at batch 8 (the largest batch tile): 512 sampled rows of each call."""
    shapes = [(7168, 5120, BF16), (5120, 5120, PREV), (34816, 5120, RMS), (5120, 17408, SWIGLU)]
    c = Chain(inputs.seed_of(5) + 9, shapes, 8, packing=B3)
    ys = c.run()
    rng = np.random.default_rng(5)
    for j, (N, _, _) in enumerate(shapes):
        c.check_call(j, ys, rows=np.sort(rng.choice(N, 512, replace=False)))


@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("batch", [1, 2])
def test_many_runs_and_reupload(packing, batch):
    """Forty back-to-back runs of one plan (each run a new launch: the base-3 kernel's handoff words
    carry a launch-unique epoch from the count of completed launches), then a fresh upload (which
    resets that count and clears the words) and ten more: every run's outputs are bit-identical to the
    first run's, and the first run matches the oracle."""
    c = Chain(71 + batch, SMALL_G128, batch, packing=packing)
    first = c.run()
    for j in range(len(SMALL_G128)):
        c.check_call(j, first)
    for _ in range(39):
        c.plan.run()
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    for a, y in zip(first, c.ys):
        assert np.array_equal(a, y.cpu().numpy())
    tq.tq_seq_upload(c.plan.handle, c.plan.workspace)
    for _ in range(10):
        c.plan.run()
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    for a, y in zip(first, c.ys):
        assert np.array_equal(a, y.cpu().numpy())


@pytest.mark.parametrize("packing", [B2, B3])
def test_determinism_and_graph_replay(packing):
    """Results do not depend on timing: two runs and a CUDA-graph replay are bit-identical."""
    c = Chain(61, SMALL_G128, 2, packing=packing)
    first = c.run()
    second = c.run()
    for a, b in zip(first, second):
        assert np.array_equal(a, b)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.plan.run(stream=s)
    for y in c.ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert tq.tq_device_status() == 0
    for a, y in zip(first, c.ys):
        assert np.array_equal(a, y.cpu().numpy())


def test_rejected_on_the_host():
    d = tq.desc(1024, 1024, 128, B2)
    codes = torch.zeros((1024, 64), dtype=torch.int32, device="cuda")
    scales = torch.ones((1024, 8), dtype=torch.float16, device="cuda")
    x = torch.zeros((1, 1024), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((8, 1024), dtype=torch.float32, device="cuda")

    def status(calls, batch=1):
        with pytest.raises(tq.TQError) as e:
            tq.tq_seq_create(calls, batch)
        return e.value.status

    assert status([(d, codes, scales, PREV, None, y)]) == 1                   # call 0 needs an x
    assert status([(d, codes, scales, BF16, x, y)], batch=9) == 1             # batch above 8
    assert status([(d, codes, scales, BF16, x, y), (d, codes, scales, SWIGLU, None, y)]) == 1  # N_prev != 2K
    d640 = tq.desc(1024, 640, 128, B2)
    assert status([(d640, codes, scales, BF16, x, y)]) == 2                   # scale rows of 10 bytes
    d3 = tq.desc(1024, 1024, 128, tq.TQ_PACK_B3)
    assert status([(d, codes, scales, BF16, x, y), (d3, codes, scales, PREV, None, y)]) == 2  # mixed packings
    dq = tq.desc(1024, 1024, 128, tq.TQ_PACK_3BIT)
    assert status([(dq, codes, scales, BF16, x, y)]) == 2                     # 3-bit codes
    ok = tq.tq_seq_create([(d, codes, scales, BF16, x, y)], 1)
    assert tq.tq_seq_kernel_count(ok) == 1
    tq.tq_seq_destroy(ok)


@pytest.mark.parametrize("packing", [B2, B3])
@pytest.mark.parametrize("batch", [2, 8])
def test_chain_mixed_magnitude_rows(packing, batch):
    """Batch rows 1e7 apart in size in one decode step (even rows x 1e4, odd rows x 1e-3): every call
    holds each row to its own bound (per-row block exponents; RMS normalisation per row)."""
    c = Chain(81 + batch, SMALL_G128[:4], batch, packing=packing)
    mult = torch.tensor([1e4 if b % 2 == 0 else 1e-3 for b in range(batch)]).reshape(batch, 1)
    c.x_host = (c.x_host.float() * mult).to(torch.bfloat16)
    c.x.copy_(c.x_host.cuda())
    ys = c.run()
    for j in range(4):
        c.check_call(j, ys)
