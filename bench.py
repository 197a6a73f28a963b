"""Benchmark of the ternary-weight linear layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference] [--no-extras]

Default workload: decode of the 27B-class dense model's linears - the seven ternary linears of one
decoder layer (q/k/v/o 5120x5120 / 1024x5120, gate/up 17408x5120, down 5120x17408), 2-bit packing
(--packing base3: 20 trits per uint32), group-128 FP16 scales, fused block-128 FWHT, batch 1 - run
over 64 layers with distinct weights.  q/k/v and gate/up are stacked as an inference engine calls
them (4 GEMV calls per layer, 256 per step, replayed from a CUDA graph); the weights (5.62 GB 2-bit,
4.56 GB base-3, codes + FP16 scales) are far larger than L2, so every step streams them from HBM.
The metric is packed-weight HBM GB/s (codes + FP16 scales, pitch included) with model-equivalent
decode tok/s beside it.

Other rows of the hot path are measured in the same run under "extras": the other packing, batch 8
and one call per linear of the same stream, the 256-expert top-8 MoE expert layer (1 / 8 / 64
tokens), and the two prefill GEMM shapes.  ``--impl reference`` times the CPU oracle (fp64 numpy) on a bounded sample of the same
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

def linear_bytes(lin, packing, group=128):
    d = tq.desc(lin.N, lin.K, group, packing)
    return tq.tq_packed_bytes(d) + tq.tq_scale_bytes(d)


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
        """Per step: H2D of each linear's activations from pinned memory, the GEMV, D2H of the output."""
        for i, (d, codes, s, name, _) in enumerate(self.calls):
            xd, xh = self.x_bufs[name]
            xd.copy_(xh, non_blocking=True)
            tq.tq_gemv(d, codes, s, xd, y=self.y_bufs[name], workspace=self.ws)
        last = self.calls[-1][3]
        y_host.copy_(self.y_bufs[last], non_blocking=True)

    def h2d_bytes(self):
        return sum(self.x_bufs[c[3]][0].numel() * 2 for c in self.calls)

    def d2h_bytes(self):
        return self.y_bufs[self.calls[-1][3]].numel() * 4


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


def per_call_durations(stream: Stream):
    """Capture one step with external timing events around every call; replay once; per-call ms."""
    n = len(stream.calls)
    events = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
              for _ in range(n)]
    g = capture(lambda: stream.step(events))
    g.replay()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in events]


def traffic_from_profiles(kernel_key: str):
    """DRAM bytes recorded by an ncu capture (profiles/ncu_traffic.txt: key, bytes, source hash), if
    the kernel sources it was taken on are unchanged."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    src_hash = hashlib.sha256()
    csrc = os.path.join(ROOT, "ternary_weight_quantized_unpack_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            src_hash.update(fh.read())
    cur = src_hash.hexdigest()[:16]
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key and parts[2] == cur:
            return float(parts[1])
    return None


def traffic_per_step(packing, batch, layers):
    """ncu DRAM bytes of one layer (profiles/ncu_traffic.txt) x layers, or None."""
    per_layer = traffic_from_profiles(
        f"dense_decode_{'b3' if packing == tq.TQ_PACK_B3 else '2b'}_b{batch}_stacked_per_layer")
    return None if per_layer is None else per_layer * layers


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ternary_weight_quantized_unpack_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
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


def bench_prefill(shape, steps, warmup, seed=inputs.seed_of(4)):
    M, K, N = shape
    d = tq.desc(N, K, 128, tq.TQ_PACK_2BIT)
    dev = "cuda"
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + K)
    codes = tq.tq_pack(d, torch.randint(-1, 2, (N, K), dtype=torch.int8, device=dev, generator=gen))
    s = torch.exp(torch.randn((N, K // 128), generator=gen, device=dev) * 0.5 - 4).half()
    x = inputs.activations(seed, K, M, K).to(dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tq.tq_gemm_workspace_bytes(d, M), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        tq.tq_gemm(d, codes, s, x, y=y, workspace=ws)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        tq.tq_gemm(d, codes, s, x, y=y, workspace=ws)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    flops = 2.0 * M * N * K
    return {"M": M, "K": K, "N": N, "ms": ms, "TFLOP_s": flops / (ms * 1e-3) / 1e12}


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

def config_of(packing, batch, layers=None, stacked=True):
    layers = LAYERS if layers is None else layers
    return {"workload": f"27B-class dense decode: {layers} layers x {{q,k,v,o,gate,up,down}} ternary GEMV "
                        "(hidden 5120, FFN 17408, 40/8 heads x 128), distinct weights per layer",
            "calls_per_layer": "4: qkv (q,k,v stacked, 7168 x 5120), o, gate_up (34816 x 5120), down" if stacked
            else "7: one per linear",
            "packing": "base3_20_per_u32" if packing == tq.TQ_PACK_B3 else "2bit", "batch": batch,
            "group": 128, "fwht_block": 128, "layers": layers,
            "l2": "inputs larger than L2 (4.56 GB base-3 / 5.62 GB 2-bit of weights per step)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    packing, batch = PACKINGS[args.packing], 1
    per_step = []
    for _ in range(args.warmup):
        oracle_sample_seconds(packing, batch, 16)
    for _ in range(args.steps):
        s, b = oracle_sample_seconds(packing, batch, 64)
        per_step.append(b / s / GB)
    full_bytes = sum(linear_bytes(l, packing) for l in inputs.dense_layer_linears()) * LAYERS
    v = statistics.median(per_step)
    ms = full_bytes / (v * GB) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_of(packing, batch),
            "tok_s": batch / (ms * 1e-3),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": "each step: fp64 numpy oracle on the first 64 rows of each of the 7 linears, "
                                       "scaled by packed bytes to the 64-layer stream"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_tq(args, rank, world, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (libtq has no CPU path)")
    peaks = measured_peaks()
    packing, batch = PACKINGS[args.packing], args.batch
    st = Stream(packing, batch, layers=args.layers)
    # warm-up: W eager steps, then capture one step into a graph
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    g = capture(st.step, warm=0)
    g.replay()
    torch.cuda.synchronize()
    ms_total, clocks = time_graph(g, args.steps, world, clocks_index=local)
    ms_max = max_over_ranks(ms_total, world)
    ms_step = ms_max / args.steps
    bytes_all = st.bytes_per_step * args.steps * world
    value = bytes_all / (ms_max * 1e-3) / GB
    # dominant kernel: the GEMV call, timed per call inside a captured step (external events)
    durs = per_call_durations(st)
    achieved = sum(c[4] for c in st.calls) / (sum(durs) * 1e-3) / GB
    # end to end through the public API with host buffers
    y_host = torch.empty_like(st.y_bufs[st.calls[-1][3]], device="cpu").pin_memory()
    ge = capture(lambda: st.step_e2e(y_host), warm=1)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ge.replay()
        torch.cuda.synchronize()   # the step's result is read on the host
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = st.bytes_per_step * args.steps * world / e2e_s / GB
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32-accumulate (fp16 x~ operand, ternary weights)", "data": "synthetic",
        "config": config_of(packing, batch, args.layers),
        "tok_s": world * batch / (ms_step * 1e-3),
        "pct_of_hbm_peak": 100.0 * value / world / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": traffic_per_step(packing, batch, args.layers),
                     "traffic_unit": "DRAM bytes per step: ncu bytes of one layer's launches x layers",
                     "kernel": "tq_gemv calls (decode GEMV kernel, plus the activation prep kernel above batch 4 "
                               "or for base-3), per-call CUDA events",
                     "algorithmic_bytes_per_step": st.bytes_per_step, "calls_per_step": len(st.calls),
                     "algorithmic_bytes_per_layer": st.bytes_per_step // max(1, args.layers),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": st.h2d_bytes(),
                "d2h_bytes_per_step": st.d2h_bytes()},
        "gpu_launches": args.steps * sum(tq.tq_gemv_kernel_count(c[0], batch) for c in st.calls),
        "clocks": clocks,
        "source_hash": source_hash(),
    }
    del st, g, ge
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and args.cpu:
        line["cpu_baseline"] = cpu_baseline(packing, batch)
    if args.extras and world == 1:
        ex = {"stream": [], "moe": [], "prefill": []}
        other = tq.TQ_PACK_B3 if packing == tq.TQ_PACK_2BIT else tq.TQ_PACK_2BIT
        for pk, b, stk in ((packing, 8, True), (other, 1, True), (other, 8, True), (packing, 1, False),
                           (other, 1, False)):
            s2 = Stream(pk, b, stacked=stk)
            s2.step()
            g2 = capture(s2.step, warm=0)
            g2.replay()
            ms2, _ = time_graph(g2, max(3, args.steps // 2), 1)
            ms2 /= max(3, args.steps // 2)
            ex["stream"].append({"packing": "base3" if pk == tq.TQ_PACK_B3 else "2bit", "batch": b,
                                 "calls_per_layer": 4 if stk else 7, "ms": ms2,
                                 "GB_s": s2.bytes_per_step / (ms2 * 1e-3) / GB, "tok_s": b / (ms2 * 1e-3)})
            del s2, g2
            torch.cuda.empty_cache()
        for T in inputs.MOE["tokens"]:
            ex["moe"].append(bench_moe(T, max(5, args.steps // 2), 3))
        for shape in inputs.PREFILL["shapes"]:
            ex["prefill"].append(bench_prefill(shape, 3, 1))
        for p in ex["prefill"]:
            p["pct_of_bf16_peak"] = 100.0 * p["TFLOP_s"] / peaks["bf16_tflops"]
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
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu", action="store_false")
    ap.add_argument("--workload", choices=["stream", "prefill", "moe"], default="stream",
                    help="stream: the headline decode line; prefill / moe: one line per shape of those workloads")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload == "prefill":
        if rank == 0:
            peaks = measured_peaks()
            for shape in inputs.PREFILL["shapes"]:
                r = bench_prefill(shape, args.steps, args.warmup)
                r["pct_of_bf16_peak"] = 100.0 * r["TFLOP_s"] / peaks["bf16_tflops"]
                print(json.dumps({"workload": "prefill", **r}))
    elif args.workload == "moe":
        if rank == 0:
            for T in inputs.MOE["tokens"]:
                print(json.dumps({"workload": "moe", **bench_moe(T, args.steps, args.warmup)}))
    else:
        run_tq(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
