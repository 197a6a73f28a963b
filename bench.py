"""Benchmark of the ternary-weight linear layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference] [--no-extras]

Default workload: one decode token through the linears of a 27B-class dense model - per layer the
stacked q/k/v projection (7168 x 5120), o (5120 x 5120), the stacked gate/up projection (34816 x 5120)
and down (5120 x 17408) - over 64 layers with distinct weights, 2-bit packing, group-128 FP16 scales,
fused block-128 FWHT, batch 1.  The step is the dependent chain a decode step is: qkv reads the
RMS-normalised layer input, o reads the q part of qkv's output (attention is not part of this
library; it stands in as the identity), gate_up reads o's output RMS-normalised, down reads
silu(gate) * up, and the next layer reads down's output.  All 256 calls run as one tq_seq launch
(the decode-step entry point); 5.62 GB of codes + FP16 scales per token, far larger than L2, stream
from HBM every step.  The metric is packed-weight HBM GB/s (codes + scales, pitch included) with
model-equivalent decode tok/s beside it.

Other rows of the hot path are measured in the same run under "extras": the same stream as 256
separate tq_gemv launches (per-call path, both packings, batch 1 and 8), the decode step at batch 8,
the seven linears of one layer called one by one at batch 1 / 4 / 16 in both packings (tok/s =
batch / (64 x the sum of the seven times)), the single 1024 x 1024 base-3 linear (latency and
L2-cold GB/s), the 256-expert top-8 MoE expert layer (1 / 8 / 64 tokens) and the two prefill GEMM
shapes.  ``--impl reference`` times the CPU oracle (fp64 numpy) on a bounded sample of the same
workload, on the host cores.

Multi-GPU: independent replicas, one process per GPU (torchrun); each rank streams its own copy
of the weights; value = bytes of all ranks / max time over ranks ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import ternary_weight_quantized_unpack_b300 as tq  # noqa: E402
from ternary_weight_quantized_unpack_b300 import inputs  # noqa: E402

GB = 1e9
LAYERS = 64
PACKINGS = {"2bit": tq.TQ_PACK_2BIT, "base3": tq.TQ_PACK_B3}
PACKING_NAMES = {tq.TQ_PACK_2BIT: "2bit", tq.TQ_PACK_B3: "base3", tq.TQ_PACK_3BIT: "3bit"}
METRIC = "packed-weight HBM GB/s (% of B300 peak) and model-equivalent decode tok/s"


# ----------------------------------------------------------------------------------------------
# environment: ranks, peaks, clocks
# ----------------------------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


class ClockSampler:
    """Samples SM clock, max clock and throttle reasons while the timed region runs: NVML when it
    loads, else ``nvidia-smi -lms 20`` in a subprocess."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}
    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                  "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self.mode, self.err = None, None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:  # NVML library missing: fall back to nvidia-smi
            self.err = repr(e)
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for name, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(0.002)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run_nvml, daemon=True)
            self.t.start()
        elif self.mode == "nvidia-smi":
            import subprocess
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.SMI_FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)   # let the first sample land before the timed region starts
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self.t.join()
        elif self.mode == "nvidia-smi":
            time.sleep(0.05)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for n, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(n)
        return False

    def summary(self):
        if self.mode is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "error": self.err}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples), "source": self.mode}


# ----------------------------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------------------------

class Stream:
    """64 layers of the 27B-class shapes, distinct weights per layer.  stacked=True calls the layer the
    way an inference engine does (qkv, o, gate_up, down: 4 calls); stacked=False calls each of the 7
    linears separately.  The weights read per token are the same either way."""

    def __init__(self, packing, batch, layers=LAYERS, seed=inputs.seed_of(5), device="cuda", stacked=True):
        self.packing, self.batch, self.layers, self.stacked = packing, batch, layers, stacked
        self.linears = inputs.stacked_layer_linears() if stacked else inputs.dense_layer_linears()
        gen = torch.Generator(device=device)
        gen.manual_seed(seed + 10 * packing + batch)
        self.calls = []  # (desc, codes, scales, x, y, ws, bytes)
        self.x_bufs = {}
        ws_bytes = max(tq.tq_gemv_workspace_bytes(tq.desc(l.N, l.K, 128, packing), batch) for l in self.linears)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        for i, lin in enumerate(self.linears):   # one activation buffer per linear shape (fed each layer)
            x = inputs.activations(seed, 500 + i, batch, lin.K)
            self.x_bufs[lin.name] = (x.to(device), x.pin_memory() if torch.cuda.is_available() else x)
        self.y_bufs = {l.name: torch.empty((batch, l.N), dtype=torch.float32, device=device) for l in self.linears}
        for layer in range(layers):
            for lin in self.linears:
                # the weights do not change during the stream: let each GEMV start streaming them
                # while the previous call is still finishing
                d = tq.desc(lin.N, lin.K, 128, packing, flags=tq.TQ_STATIC_WEIGHTS)
                t = torch.randint(-1, 2, (lin.N, lin.K), dtype=torch.int8, device=device, generator=gen)
                codes = tq.tq_pack(d, t)
                del t
                s = torch.exp(torch.randn((lin.N, lin.K // 128), generator=gen, device=device) * 0.5 - 4).half()
                self.calls.append((d, codes, s, lin.name, tq.tq_packed_bytes(d) + tq.tq_scale_bytes(d)))
        torch.cuda.synchronize()
        self.bytes_per_step = sum(c[4] for c in self.calls)

    def step(self, events=None):
        for i, (d, codes, s, name, _) in enumerate(self.calls):
            if events is not None:
                events[i][0].record()
            tq.tq_gemv(d, codes, s, self.x_bufs[name][0], y=self.y_bufs[name], workspace=self.ws)
            if events is not None:
                events[i][1].record()

    def step_e2e(self, y_host):
        """One token in, one result out: H2D of the first call's input from pinned memory, every call,
        D2H of the last call's output."""
        name0 = self.calls[0][3]
        xd, xh = self.x_bufs[name0]
        xd.copy_(xh, non_blocking=True)
        self.step()
        y_host.copy_(self.y_bufs[self.calls[-1][3]], non_blocking=True)

    def h2d_bytes(self):
        return self.x_bufs[self.calls[0][3]][0].numel() * 2

    def d2h_bytes(self):
        return self.y_bufs[self.calls[-1][3]].numel() * 4


class SeqStep:
    """The decode step of a Stream's weights (stacked, 2-bit or base-3) as one tq_seq launch: the dependent
    chain qkv(RMS-normalised input) -> o(q part) -> gate_up(RMS-normalised) -> down(SwiGLU) per layer."""

    SRC = {"qkv": tq.TQ_SEQ_X_RMS_PREV, "o": tq.TQ_SEQ_X_PREV, "gate_up": tq.TQ_SEQ_X_RMS_PREV,
           "down": tq.TQ_SEQ_X_SWIGLU_PREV}

    def __init__(self, stream: "Stream", device="cuda"):
        assert stream.stacked and stream.packing in (tq.TQ_PACK_2BIT, tq.TQ_PACK_B3)
        self.batch = stream.batch
        lins = {l.name: l for l in stream.linears}
        self.x_dev, self.x_host = stream.x_bufs["qkv"]
        self.ys = {n: torch.empty((self.batch, l.N), dtype=torch.float32, device=device) for n, l in lins.items()}
        calls = []
        for i, (d, codes, s, name, _) in enumerate(stream.calls):
            d0 = tq.desc(d.N, d.K, d.group, d.packing, d.fwht_block)
            src = tq.TQ_SEQ_X_BF16 if i == 0 else self.SRC[name]
            calls.append((d0, codes, s, src, self.x_dev if i == 0 else None, self.ys[name]))
        self.out = self.ys[stream.calls[-1][3]]
        self.plan = tq.SeqPlan(calls, self.batch)
        self.bytes_per_step = stream.bytes_per_step

    def step(self):
        self.plan.run()

    def step_e2e(self, y_host):
        """One token in, one result out: H2D of the input from pinned memory, the step, D2H of the
        last call's output."""
        self.x_dev.copy_(self.x_host, non_blocking=True)
        self.plan.run()
        y_host.copy_(self.out, non_blocking=True)

    def h2d_bytes(self):
        return self.x_dev.numel() * 2

    def d2h_bytes(self):
        return self.out.numel() * 4


def capture(fn, warm=1):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, reps, world, clocks_index=None):
    """Replay ``g`` reps times inside a barrier/synchronize-bracketed region timed with CUDA events."""
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(clocks_index) if clocks_index is not None else None
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    return ms, (sampler.summary() if sampler is not None else None)


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def traffic_from_profiles(kernel_key: str):
    """DRAM bytes recorded by an ncu capture (profiles/ncu_traffic.txt: key, bytes, hash, source files),
    if the kernel sources it was taken on (the files listed, under the package's csrc/) are unchanged."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel_key:
            if parts[2] == source_hash(parts[3].split(",")):
                return float(parts[1])
    return None


def source_hash(files=None):
    """First 16 hex digits of the SHA-256 of the kernel sources (all of csrc/, or the files named)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ternary_weight_quantized_unpack_b300", "csrc")
    for f in sorted(files if files else os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------------------------
# extras: MoE and prefill
# ----------------------------------------------------------------------------------------------

def bench_moe(T, steps, warmup, seed=inputs.seed_of(3)):
    m = inputs.MOE
    E, H, F, G, k = m["E"], m["H"], m["F"], m["group"], m["topk"]
    gu, dn = tq.desc(2 * F, H, G, m["packing"]), tq.desc(H, F, G, m["packing"])
    dev = "cuda"
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    # stacked [E][rows][P]: pack all experts' rows at once (rows of different experts are independent)
    gu_all = tq.desc(E * 2 * F, H, G, m["packing"])
    dn_all = tq.desc(E * H, F, G, m["packing"])
    gu_codes = tq.tq_pack(gu_all, torch.randint(-1, 2, (E * 2 * F, H), dtype=torch.int8, device=dev, generator=gen))
    d_codes = tq.tq_pack(dn_all, torch.randint(-1, 2, (E * H, F), dtype=torch.int8, device=dev, generator=gen))
    gu_s = torch.exp(torch.randn((E * 2 * F, H // G), generator=gen, device=dev) * 0.5 - 4).half()
    d_s = torch.exp(torch.randn((E * H, F // G), generator=gen, device=dev) * 0.5 - 4).half()
    logits = inputs.router_logits(seed, T, T, E).to(dev)
    x = inputs.activations(seed, T, T, H).to(dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_moe_workspace_bytes(T, E, k, H, F), dtype=torch.uint8, device=dev)

    def call():
        tq.tq_moe_gemv(gu, dn, E, k, gu_codes, gu_s, d_codes, d_s, logits, x, topk_idx=idx, topk_gate=gate, y=y,
                       workspace=ws)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    n_active = len(set(idx.cpu().numpy().reshape(-1).tolist()))
    per_expert = (tq.tq_packed_bytes(gu) + tq.tq_scale_bytes(gu) + tq.tq_packed_bytes(dn) + tq.tq_scale_bytes(dn))
    g = capture(call)
    # the MoE weights (193 MB) exceed L2; between replays flush L2 by rewriting a 256 MB buffer
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    for _ in range(steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    byts = n_active * per_expert + logits.numel() * 4
    return {"tokens": T, "active_experts": n_active, "ms": ms, "GB_s": byts / (ms * 1e-3) / GB,
            "tok_s_40_layers": T / (40 * ms * 1e-3), "bytes": byts}


def bench_quantize(reps, seed=inputs.seed_of(2)):
    """The offline quantizer on the 27B-class gate/up shape (17408 x 5120 dense bf16 W): rotate, scale,
    ternarize and pack, timed per call; GB/s of W read."""
    N, K = 17408, 5120
    w = (inputs.activations(seed, 900, N, K, outlier_frac=0.001).float() * 2.0 ** -6).to(torch.bfloat16).cuda()
    out = {}
    for name, pk in (("2bit", tq.TQ_PACK_2BIT), ("base3", tq.TQ_PACK_B3)):
        d = tq.desc(N, K, 128, pk)
        codes, scales = tq.tq_quantize(d, w)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            tq.tq_quantize(d, w, codes, scales)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        out[name] = {"N": N, "K": K, "ms": ms, "GB_s_of_W": N * K * 2 / (ms * 1e-3) / GB}
    return out


def bench_moe_prefill(T, steps, warmup, seed=inputs.seed_of(3)):
    """The expert layer at prefill sizes (tq_moe_gemm: grouped tcgen05 GEMM), T tokens; TFLOP/s of the
    expert GEMMs (2 * T * topk * (2F * H + H * F))."""
    m = inputs.MOE
    E, H, F, G, k = m["E"], m["H"], m["F"], m["group"], m["topk"]
    gu, dn = tq.desc(2 * F, H, G, m["packing"]), tq.desc(H, F, G, m["packing"])
    dev = "cuda"
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + T)
    gu_all, dn_all = tq.desc(E * 2 * F, H, G, m["packing"]), tq.desc(E * H, F, G, m["packing"])
    gu_codes = tq.tq_pack(gu_all, torch.randint(-1, 2, (E * 2 * F, H), dtype=torch.int8, device=dev, generator=gen))
    d_codes = tq.tq_pack(dn_all, torch.randint(-1, 2, (E * H, F), dtype=torch.int8, device=dev, generator=gen))
    gu_s = torch.exp(torch.randn((E * 2 * F, H // G), generator=gen, device=dev) * 0.5 - 4).half()
    d_s = torch.exp(torch.randn((E * H, F // G), generator=gen, device=dev) * 0.5 - 4).half()
    logits = inputs.router_logits(seed, T, T, E).to(dev)
    x = inputs.activations(seed, T, T, H).to(dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_moe_gemm_workspace_bytes(T, E, k, H, F), dtype=torch.uint8, device=dev)

    def call():
        tq.tq_moe_gemm(gu, dn, E, k, gu_codes, gu_s, d_codes, d_s, logits, x, topk_idx=idx, topk_gate=gate, y=y,
                       workspace=ws)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    flops = 2.0 * T * k * (2 * F * H + H * F)
    return {"tokens": T, "ms": ms, "TFLOP_s": flops / (ms * 1e-3) / 1e12, "tok_s_40_layers": T / (40 * ms * 1e-3),
            "launches_per_call": 9}


def bench_prefill(shape, steps, warmup, seed=inputs.seed_of(4), fp8=False):
    """One prefill call (FP16 operands, or FP8 E4M3 with tq_gemm_fp8), device time per call."""
    M, K, N = shape
    d = tq.desc(N, K, 128, tq.TQ_PACK_2BIT)
    dev = "cuda"
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + K)
    codes = tq.tq_pack(d, torch.randint(-1, 2, (N, K), dtype=torch.int8, device=dev, generator=gen))
    s = torch.exp(torch.randn((N, K // 128), generator=gen, device=dev) * 0.5 - 4).half()
    x = inputs.activations(seed, K, M, K).to(dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    gemm = tq.tq_gemm_fp8 if fp8 else tq.tq_gemm
    ws_bytes = (tq.tq_gemm_fp8_workspace_bytes if fp8 else tq.tq_gemm_workspace_bytes)(d, M)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        gemm(d, codes, s, x, y=y, workspace=ws)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        gemm(d, codes, s, x, y=y, workspace=ws)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    flops = 2.0 * M * N * K
    return {"M": M, "K": K, "N": N, "operands": "fp8_e4m3" if fp8 else "fp16", "ms": ms,
            "TFLOP_s": flops / (ms * 1e-3) / 1e12}


def l2_cold_times(fn, reps, flush):
    """Per-call device time of fn() after an L2 flush (a 256 MB write; the flush keeps the device busy
    while the host enqueues the call, so no host launch latency enters the events)."""
    times = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def bench_single_linear(reps, seed=inputs.seed_of(1)):
    """The single 1024 x 1024 base-3 linear (batch 1, 0.5 % x20 outliers): latency with L2 flushed
    before every call, and back-to-back graph replays (L2-warm)."""
    c = inputs.SINGLE_LINEAR
    N, K, G, pk = c["N"], c["K"], c["group"], c["packing"]
    d = tq.desc(N, K, G, pk, c["fwht_block"])
    codes = tq.tq_pack(d, inputs.trits(seed, 0, N, K, device="cuda"))
    s = inputs.scales(seed, 1, N, K // G, device="cuda").contiguous()
    x = inputs.activations(seed, 0, c["B"], K, outlier_frac=c["outlier_frac"]).cuda()
    y = torch.empty((c["B"], N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, tq.tq_gemv_workspace_bytes(d, c["B"])), dtype=torch.uint8, device="cuda")
    call = lambda: tq.tq_gemv(d, codes, s, x, y=y, workspace=ws)  # noqa: E731
    for _ in range(3):
        call()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    cold = l2_cold_times(call, reps, flush)
    g = capture(lambda: [call() for _ in range(20)], warm=0)
    g.replay()
    torch.cuda.synchronize()
    warm_ms, _ = time_graph(g, max(3, reps // 4), 1)
    warm = warm_ms / (20 * max(3, reps // 4))
    byts = tq.tq_packed_bytes(d) + tq.tq_scale_bytes(d)
    return {"N": N, "K": K, "packing": "base3", "batch": c["B"], "bytes": byts,
            "latency_us_l2_cold": cold * 1e3, "GB_s_l2_cold": byts / (cold * 1e-3) / GB,
            "latency_us_l2_warm_back_to_back": warm * 1e3,
            "kernels_per_call": tq.tq_gemv_kernel_count(d, c["B"])}


# 3-bit linears timed alone: a 27B-class gate/up-sized matrix and a wide-output one (the shape class of
# an lm_head over a 2048-wide hidden state; no page gives the model's vocabulary size)
GEMV3_SHAPES = ((17408, 5120), (131072, 2048))


def bench_gemv_linear(N, K, packing, batch, reps, seed=inputs.seed_of(2)):
    """One linear called alone with L2 flushed before each call: device time and GB/s of codes + scales."""
    d = tq.desc(N, K, 128, packing)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + N + packing)
    lo, hi = (-4, 4) if packing == tq.TQ_PACK_3BIT else (-1, 2)
    codes = tq.tq_pack(d, torch.randint(lo, hi, (N, K), dtype=torch.int8, device="cuda", generator=gen))
    s = torch.exp(torch.randn((N, K // 128), generator=gen, device="cuda") * 0.5 - 4).half()
    x = inputs.activations(seed, N, batch, K).cuda()
    y = torch.empty((batch, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, tq.tq_gemv_workspace_bytes(d, batch)), dtype=torch.uint8, device="cuda")
    call = lambda: tq.tq_gemv(d, codes, s, x, y=y, workspace=ws)  # noqa: E731
    for _ in range(3):
        call()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ms = l2_cold_times(call, max(3, reps), flush)
    byts = tq.tq_packed_bytes(d) + tq.tq_scale_bytes(d)
    return {"N": N, "K": K, "packing": PACKING_NAMES[packing], "batch": batch, "us_l2_cold": ms * 1e3,
            "GB_s": byts / (ms * 1e-3) / GB, "kernels_per_call": tq.tq_gemv_kernel_count(d, batch)}


def bench_layer_linears(packing, batches, reps, seed=inputs.seed_of(2)):
    """The seven linears of one 27B-class layer, each called alone with L2 flushed before it; per
    batch: per-linear device times and tok/s = batch / (64 x sum of the seven times)."""
    lins = inputs.dense_layer_linears()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + packing)
    ws_bytes = max(tq.tq_gemv_workspace_bytes(tq.desc(l.N, l.K, 128, packing), b) for l in lins for b in batches)
    ws = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    w = []
    for lin in lins:
        d = tq.desc(lin.N, lin.K, 128, packing)
        lo, hi = (-4, 4) if packing == tq.TQ_PACK_3BIT else (-1, 2)
        codes = tq.tq_pack(d, torch.randint(lo, hi, (lin.N, lin.K), dtype=torch.int8, device="cuda", generator=gen))
        s = torch.exp(torch.randn((lin.N, lin.K // 128), generator=gen, device="cuda") * 0.5 - 4).half()
        w.append((lin, d, codes, s))
    out = []
    for b in batches:
        per = {}
        for i, (lin, d, codes, s) in enumerate(w):
            x = inputs.activations(seed, 700 + i, b, lin.K).cuda()
            y = torch.empty((b, lin.N), dtype=torch.float32, device="cuda")
            call = lambda: tq.tq_gemv(d, codes, s, x, y=y, workspace=ws)  # noqa: E731
            call()
            per[lin.name] = l2_cold_times(call, reps, flush) * 1e3
        tot_us = sum(per.values())
        byts = sum(tq.tq_packed_bytes(d) + tq.tq_scale_bytes(d) for _, d, _, _ in w)
        out.append({"packing": PACKING_NAMES[packing], "batch": b,
                    "us_per_linear_l2_cold": per, "us_sum_7": tot_us,
                    "GB_s": byts / (tot_us * 1e-6) / GB,
                    "tok_s_64_layers": b / (LAYERS * tot_us * 1e-6)})
    return out


def bench_seq(st: "Stream", steps, world=1, clocks_index=None, warmup=3):
    """The decode step of ``st`` as one tq_seq launch, graph-replayed; returns (engine, graph, ms for
    all steps, clocks)."""
    eng = SeqStep(st)
    for _ in range(warmup):
        eng.step()
    torch.cuda.synchronize()
    g = capture(eng.step, warm=0)
    g.replay()
    torch.cuda.synchronize()
    ms, clocks = time_graph(g, steps, world, clocks_index=clocks_index)
    return eng, g, ms, clocks


def bench_per_call(st: "Stream", steps, world=1, clocks_index=None, warmup=3):
    """The step as one tq_gemv launch per call (graph-replayed); returns (graph, ms for all steps, clocks)."""
    for _ in range(warmup):
        st.step()
    torch.cuda.synchronize()
    g = capture(st.step, warm=0)
    g.replay()
    torch.cuda.synchronize()
    ms, clocks = time_graph(g, steps, world, clocks_index=clocks_index)
    return g, ms, clocks


# ----------------------------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ----------------------------------------------------------------------------------------------

def oracle_sample_seconds(packing, batch, rows_per_linear, seed=inputs.seed_of(5)):
    """Time the oracle (unpack + FWHT + contraction, fp64) on rows_per_linear rows of each of the 7
    linears; returns (seconds, packed bytes covered)."""
    import oracle as O
    total_s, total_b = 0.0, 0
    for i, lin in enumerate(inputs.dense_layer_linears()):
        rows = np.arange(min(rows_per_linear, lin.N))
        t = inputs.trits(seed, 900 + i, lin.N, lin.K, rows=rows).numpy()
        s = inputs.scales(seed, 950 + i, lin.N, lin.K // 128, rows=rows).numpy()
        codes = O.pack(t, packing)
        x = inputs.activations(seed, 500 + i, batch, lin.K).float().numpy()
        t0 = time.perf_counter()
        O.ternary_linear(codes, s, x, lin.K, 128, packing, 128)
        total_s += time.perf_counter() - t0
        total_b += codes.nbytes + s.nbytes
    return total_s, total_b


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(packing, batch, target_s=12.0):
    s, b = oracle_sample_seconds(packing, batch, 32)
    rows = int(min(17408, max(32, 32 * target_s / max(s, 1e-3))))
    s, b = oracle_sample_seconds(packing, batch, rows)
    return {"value": b / s / GB, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle on the first {rows} rows of each of the 7 linears (batch {batch}); "
                      f"{b / 1e6:.1f} MB of packed weights in {s:.1f} s, scaled by bytes"}


# ----------------------------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------------------------

def config_of(packing, batch, layers=None, stacked=True, seq=False):
    layers = LAYERS if layers is None else layers
    return {"workload": f"27B-class dense decode: {layers} layers x {{q,k,v,o,gate,up,down}} ternary GEMV "
                        "(hidden 5120, FFN 17408, 40/8 heads x 128), distinct weights per layer",
            "calls_per_layer": "4: qkv (q,k,v stacked, 7168 x 5120), o, gate_up (34816 x 5120), down" if stacked
            else "7: one per linear",
            "engine": "tq_seq: the dependent chain (RMS norm -> qkv -> o -> RMS norm -> gate_up -> SwiGLU -> down) "
                      "in one launch" if seq else "tq_gemv per call, graph-replayed",
            "packing": "base3_20_per_u32" if packing == tq.TQ_PACK_B3 else "2bit", "batch": batch,
            "group": 128, "fwht_block": 128, "layers": layers,
            "l2": "inputs larger than L2 (4.56 GB base-3 / 5.62 GB 2-bit of weights per step)"}


def oracle_linear_bytes(lin, packing, group=128):
    """Codes + scales of one linear, from the oracle's own size rules (no library call)."""
    import oracle as O
    return O.packed_bytes(lin.N, lin.K, packing) + O.scale_bytes(lin.N, lin.K, group)


def run_reference(args, rank, world):
    """The oracle arm: each step runs the fp64 oracle on a fixed row sample (the first 64 rows of each
    of the seven linears of a layer) on the host cores; value = packed bytes of the sample / time."""
    if rank != 0:
        return
    packing, batch = PACKINGS[args.packing], 1
    for _ in range(args.warmup):
        oracle_sample_seconds(packing, batch, 16)
    t0 = time.perf_counter()
    total_b = 0
    for _ in range(args.steps):
        _, b = oracle_sample_seconds(packing, batch, 64)
        total_b += b
    secs = time.perf_counter() - t0
    v = total_b / secs / GB
    full_bytes = sum(oracle_linear_bytes(l, packing) for l in inputs.dense_layer_linears()) * LAYERS
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(packing, batch),
            "step": "one step = the oracle on the first 64 rows of each of the 7 linears of a layer "
                    f"({total_b / args.steps / 1e6:.2f} MB of packed weights)",
            "projected_ms_per_token": full_bytes / (v * GB) * 1e3,
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": "each step: fp64 numpy oracle on the first 64 rows of each of the 7 "
                                       "linears of one layer; value = packed bytes of the sample / time"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def e2e_time(fn, steps, world):
    """Wall time of ``steps`` calls of fn(), each followed by a synchronize (the step's result is read
    on the host), max over ranks."""
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        fn()
        torch.cuda.synchronize()
    return max_over_ranks(time.perf_counter() - t0, world)


def run_tq(args, rank, world, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (libtq has no CPU path)")
    peaks = measured_peaks()
    packing, batch = PACKINGS[args.packing], args.batch
    st = Stream(packing, batch, layers=args.layers)
    seq = args.engine == "seq" and packing in (tq.TQ_PACK_2BIT, tq.TQ_PACK_B3) and batch <= 8
    if seq:
        eng, g, ms_total, clocks = bench_seq(st, args.steps, world, clocks_index=local, warmup=args.warmup)
        launches_per_step = tq.tq_seq_kernel_count(eng.plan.handle)
        kname = "gemv_seq_b3_kernel" if packing == tq.TQ_PACK_B3 else "gemv_seq_kernel"
        kernel = (f"{kname}: the whole step (256 dependent calls) is this one persistent launch; "
                  "duration = CUDA-event time of the graph-replayed steps / steps")
    else:
        eng = st
        g, ms_total, clocks = bench_per_call(st, args.steps, world, clocks_index=local, warmup=args.warmup)
        launches_per_step = sum(tq.tq_gemv_kernel_count(c[0], batch) for c in st.calls)
        kernel = ("tq_gemv launches (decode GEMV kernel, plus the activation prep kernel above batch 4 or for "
                  "base-3); duration = graph-replayed step time")
    ms_max = max_over_ranks(ms_total, world)
    ms_step = ms_max / args.steps
    bytes_all = st.bytes_per_step * args.steps * world
    value = bytes_all / (ms_max * 1e-3) / GB
    achieved = st.bytes_per_step / (ms_step * 1e-3) / GB
    # end to end through the public API: one token's input in from pinned host memory, one result out
    y_host = torch.empty_like(eng.out if seq else st.y_bufs[st.calls[-1][3]], device="cpu").pin_memory()
    for _ in range(2):
        eng.step_e2e(y_host)
    e2e_s = e2e_time(lambda: eng.step_e2e(y_host), args.steps, world)
    e2e_value = st.bytes_per_step * args.steps * world / e2e_s / GB
    tkey = f"gemv_seq_{'b3' if packing == tq.TQ_PACK_B3 else '2b'}_b{batch}_per_layer" if seq else \
        f"dense_decode_{'b3' if packing == tq.TQ_PACK_B3 else '2b'}_b{batch}_stacked_per_layer"
    per_layer = traffic_from_profiles(tkey)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32-accumulate (fp16 x~ operand, ternary weights)", "data": "synthetic",
        "config": config_of(packing, batch, args.layers, seq=seq),
        "tok_s": world * batch / (ms_step * 1e-3),
        "pct_of_hbm_peak": 100.0 * value / world / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": None if per_layer is None else per_layer * args.layers,
                     "traffic_unit": "DRAM bytes per step: ncu dram__bytes_read.sum + dram__bytes_write.sum of a "
                                     "short stream, per layer, x layers",
                     "kernel": kernel, "kernel_ms": ms_step,
                     "algorithmic_bytes_per_step": st.bytes_per_step, "calls_per_step": len(st.calls),
                     "algorithmic_bytes_per_layer": st.bytes_per_step // max(1, args.layers),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": eng.h2d_bytes(),
                "d2h_bytes_per_step": eng.d2h_bytes(),
                "path": "per step: H2D of the token's bf16 input (pinned), the step, D2H of the last output, "
                        "host synchronize"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
        "source_hash": source_hash(),
    }
    del eng, g
    if rank == 0 and world == 1 and args.cpu:
        line["cpu_baseline"] = cpu_baseline(packing, batch)
    if args.extras and world == 1:
        ex = {"decode_step": [], "per_call_stream": [], "single_linear": None, "layer_linears": [],
              "moe": [], "prefill": [], "quantize": None, "moe_prefill": []}
        reps = max(5, args.steps // 4)
        if seq:   # the same weights called one launch per call
            g2, ms2, _ = bench_per_call(st, reps)
            ms2 /= reps
            ex["per_call_stream"].append({"packing": PACKING_NAMES[packing], "batch": batch, "calls_per_layer": 4,
                                          "ms": ms2,
                                          "GB_s": st.bytes_per_step / (ms2 * 1e-3) / GB,
                                          "tok_s": batch / (ms2 * 1e-3)})
            del g2
        del st
        torch.cuda.empty_cache()
        for pk, b in ((tq.TQ_PACK_2BIT, 8), (tq.TQ_PACK_B3, 1), (tq.TQ_PACK_B3, 8)):
            s2 = Stream(pk, b)
            e2, g2, ms2, _ = bench_seq(s2, reps)
            ms2 /= reps
            ex["decode_step"].append({"packing": PACKING_NAMES[pk], "batch": b, "engine": "tq_seq (one launch per step)",
                                      "ms": ms2, "GB_s": s2.bytes_per_step / (ms2 * 1e-3) / GB,
                                      "pct_of_hbm_peak": 100.0 * s2.bytes_per_step / (ms2 * 1e-3) / GB / peaks["hbm_gbs"],
                                      "tok_s": b / (ms2 * 1e-3)})
            del e2, g2
            g2, ms2, _ = bench_per_call(s2, reps)
            ms2 /= reps
            ex["per_call_stream"].append({"packing": "base3" if pk == tq.TQ_PACK_B3 else "2bit", "batch": b,
                                          "calls_per_layer": 4, "ms": ms2,
                                          "GB_s": s2.bytes_per_step / (ms2 * 1e-3) / GB, "tok_s": b / (ms2 * 1e-3)})
            del s2, g2
            torch.cuda.empty_cache()
        ex["single_linear"] = bench_single_linear(max(20, args.steps // 2))
        for pk in (tq.TQ_PACK_2BIT, tq.TQ_PACK_B3):
            ex["layer_linears"] += bench_layer_linears(pk, inputs.DENSE_DECODE["batches"], max(10, args.steps // 5))
        # 3-bit codes (the precision the non-expert linears keep)
        ex["layer_linears"] += bench_layer_linears(tq.TQ_PACK_3BIT, inputs.DENSE_DECODE["batches"],
                                                   max(10, args.steps // 5))
        ex["gemv3"] = [bench_gemv_linear(N, K, tq.TQ_PACK_3BIT, 1, 20) for N, K in GEMV3_SHAPES]
        torch.cuda.empty_cache()
        for T in inputs.MOE["tokens"]:
            r = bench_moe(T, max(10, args.steps // 2), 3)
            r["latency_us"] = r["ms"] * 1e3
            r["launches_per_call"] = 3
            ex["moe"].append(r)
        ex["quantize"] = bench_quantize(5)
        ex["moe_prefill"] = [bench_moe_prefill(T, 10, 3) for T in (256, 1024, 4096)]
        for r in ex["moe_prefill"]:
            r["pct_of_bf16_peak"] = 100.0 * r["TFLOP_s"] / peaks["bf16_tflops"]
        for shape in inputs.PREFILL["shapes"]:
            ex["prefill"].append(bench_prefill(shape, 20, 3))
            ex["prefill"].append(bench_prefill(shape, 20, 3, fp8=True))
        for p in ex["prefill"]:
            if p["operands"] == "fp16":
                p["pct_of_bf16_peak"] = 100.0 * p["TFLOP_s"] / peaks["bf16_tflops"]
            else:  # FP8 peak: the measured bf16 burst x the nominal FP8 / BF16 ratio (4.5 / 2.25)
                p["pct_of_fp8_peak"] = 100.0 * p["TFLOP_s"] / (2.0 * peaks["bf16_tflops"])
        line["extras"] = ex
    if rank == 0:
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tq", "reference"], default="tq")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--packing", choices=sorted(PACKINGS), default="2bit",
                    help="packing of the decode stream (the other one is measured under extras)")
    ap.add_argument("--layers", type=int, default=LAYERS, help="layers of the weight stream (profiling runs use 1)")
    ap.add_argument("--engine", choices=["seq", "per_call"], default="seq",
                    help="seq: the whole step as one tq_seq launch (2-bit, batch <= 8); per_call: one tq_gemv per call")
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu", action="store_false")
    ap.add_argument("--workload", choices=["stream", "prefill", "prefill_fp8", "moe", "moe_prefill", "gemv3"],
                    default="stream",
                    help="stream: the headline decode line; prefill / prefill_fp8 / moe / moe_prefill / gemv3: one "
                         "line per shape of those workloads")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload in ("prefill", "prefill_fp8"):
        if rank == 0:
            peaks = measured_peaks()
            fp8 = args.workload == "prefill_fp8"
            for shape in inputs.PREFILL["shapes"]:
                r = bench_prefill(shape, args.steps, args.warmup, fp8=fp8)
                r["pct_of_peak"] = 100.0 * r["TFLOP_s"] / (peaks["bf16_tflops"] * (2.0 if fp8 else 1.0))
                print(json.dumps({"workload": args.workload, **r}))
    elif args.workload == "gemv3":
        if rank == 0:
            for N, K in GEMV3_SHAPES:
                for b in (1, 16):
                    print(json.dumps({"workload": "gemv3", **bench_gemv_linear(N, K, tq.TQ_PACK_3BIT, b, args.steps)}))
    elif args.workload == "moe":
        if rank == 0:
            for T in inputs.MOE["tokens"]:
                print(json.dumps({"workload": "moe", **bench_moe(T, args.steps, args.warmup)}))
    elif args.workload == "moe_prefill":
        if rank == 0:
            for T in (256, 1024, 4096):
                print(json.dumps({"workload": "moe_prefill", **bench_moe_prefill(T, args.steps, args.warmup)}))
    else:
        run_tq(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
