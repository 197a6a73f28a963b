"""Seeded synthetic inputs for the ternary-weight linear layer.

This module only draws numbers.  It holds none of the layer's arithmetic (no
packing, no transform, no contraction), so both the CPU oracle and the CUDA
path can take their inputs from it without sharing any of the method.

Distributions (the workload shapes come from the models the pages describe:
27B dense with group-128 FP16 scales, and the 256-expert top-8 MoE with
group-64 ternary experts):

* trits t in {-1, 0, +1}, i.i.d. uniform.  Element (n, k) of tensor ``tid``
  is ``(h mod 3) - 1`` where ``h`` is a counter-based 32-bit hash of
  ``(seed, tid, n*K + k)``.  Being counter-based, the same element can be
  produced on the host (for the rows an oracle samples) or on the device (for
  the multi-GB weight streams) and the two agree bit for bit: the hash uses
  only integer multiply / xor / shift on int64 tensors whose values stay below
  2**63, so CPU and CUDA torch produce identical bits.
* FP16 group scales ~ lognormal(mu=-4, sigma=0.5), taken as one of 4096
  equiprobable quantiles (a fixed table built on the host), indexed by the top
  12 bits of the same kind of hash.  The table makes host and device agree
  exactly without relying on transcendental functions being bit-identical.
* activations x ~ N(0, 1) rounded to bf16 (numpy PCG64); for the single-layer
  case 0.5 % of the entries are multiplied by 20 before rounding.
* router logits ~ N(0, 1) fp32 (numpy PCG64).
"""
from __future__ import annotations

import dataclasses
import math
from statistics import NormalDist

import numpy as np
import torch

_M32 = 0xFFFFFFFF
_MUL = 0x45D9F3B  # < 2**27, so x * _MUL < 2**59 for x < 2**32: no int64 overflow


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """32-bit integer avalanche (xor-shift-multiply, two rounds) on int64 values in [0, 2**32)."""
    x = ((x >> 16) ^ x) * _MUL & _M32
    x = ((x >> 16) ^ x) * _MUL & _M32
    return (x >> 16) ^ x


def _key(seed: int, tid: int) -> int:
    k = torch.tensor([(seed * 0x9E3779B1 + tid * 0x85EBCA77 + 0x27D4EB2F) & _M32], dtype=torch.int64)
    return int(_mix32(_mix32(k))[0])


def hash_u32(seed: int, tid: int, idx: torch.Tensor) -> torch.Tensor:
    """Counter-based hash of element indices ``idx`` (int64, < 2**32) -> int64 in [0, 2**32)."""
    k = _key(seed, tid)
    return _mix32(_mix32(idx ^ k) ^ ((k * 0x2545F491) & _M32))


def trits(seed: int, tid: int, N: int, K: int, rows=None, device="cpu", chunk_rows: int = 2048) -> torch.Tensor:
    """int8 trits [len(rows) or N, K] in {-1,0,1}; element (n,k) depends only on (seed, tid, n*K+k)."""
    assert N * K < 2**32
    row_list = torch.arange(N, dtype=torch.int64) if rows is None else torch.as_tensor(rows, dtype=torch.int64)
    out = torch.empty((row_list.numel(), K), dtype=torch.int8, device=device)
    kk = torch.arange(K, dtype=torch.int64, device=device)
    for r0 in range(0, row_list.numel(), chunk_rows):
        r = row_list[r0:r0 + chunk_rows].to(device)
        idx = r[:, None] * K + kk[None, :]
        out[r0:r0 + r.numel()] = (hash_u32(seed, tid, idx) % 3 - 1).to(torch.int8)
    return out


def codes3(seed: int, tid: int, N: int, K: int, rows=None, device="cpu", chunk_rows: int = 2048) -> torch.Tensor:
    """int8 3-bit codes [len(rows) or N, K], uniform on {-4..3}; element (n,k) depends only on
    (seed, tid, n*K+k)."""
    assert N * K < 2**32
    row_list = torch.arange(N, dtype=torch.int64) if rows is None else torch.as_tensor(rows, dtype=torch.int64)
    out = torch.empty((row_list.numel(), K), dtype=torch.int8, device=device)
    kk = torch.arange(K, dtype=torch.int64, device=device)
    for r0 in range(0, row_list.numel(), chunk_rows):
        r = row_list[r0:r0 + chunk_rows].to(device)
        idx = r[:, None] * K + kk[None, :]
        out[r0:r0 + r.numel()] = ((hash_u32(seed, tid, idx) >> 8) % 8 - 4).to(torch.int8)
    return out


_SCALE_TABLE_CACHE: dict = {}


def scale_table(mu: float = -4.0, sigma: float = 0.5, n: int = 4096) -> np.ndarray:
    """fp16 table of the n equiprobable quantiles of lognormal(mu, sigma)."""
    key = (mu, sigma, n)
    if key not in _SCALE_TABLE_CACHE:
        nd = NormalDist()
        q = [math.exp(mu + sigma * nd.inv_cdf((i + 0.5) / n)) for i in range(n)]
        _SCALE_TABLE_CACHE[key] = np.asarray(q, dtype=np.float64).astype(np.float16)
    return _SCALE_TABLE_CACHE[key]


def scales(seed: int, tid: int, N: int, n_groups: int, rows=None, device="cpu") -> torch.Tensor:
    """fp16 group scales [len(rows) or N, n_groups], lognormal(-4, 0.5) quantiles."""
    table = torch.from_numpy(scale_table().view(np.int16).astype(np.int64)).to(device)
    row_list = torch.arange(N, dtype=torch.int64) if rows is None else torch.as_tensor(rows, dtype=torch.int64)
    idx = row_list.to(device)[:, None] * n_groups + torch.arange(n_groups, dtype=torch.int64, device=device)[None, :]
    h = hash_u32(seed, tid + 0x5CA1E, idx)
    bits = table[h >> 20].to(torch.int16)
    return bits.view(torch.float16)


def activations(seed: int, tid: int, B: int, K: int, outlier_frac: float = 0.0, outlier_mult: float = 20.0) -> torch.Tensor:
    """bf16 [B, K] ~ N(0,1); a fraction ``outlier_frac`` of entries (exact count) multiplied by ``outlier_mult``."""
    rng = np.random.Generator(np.random.PCG64([seed, tid, 0xAC7]))
    x = rng.standard_normal((B, K), dtype=np.float32)
    n_out = int(round(outlier_frac * B * K))
    if n_out:
        pos = rng.choice(B * K, size=n_out, replace=False)
        x.reshape(-1)[pos] *= np.float32(outlier_mult)
    return torch.from_numpy(x).to(torch.bfloat16)


def router_logits(seed: int, tid: int, T: int, E: int) -> torch.Tensor:
    """fp32 router logits [T, E] ~ N(0,1)."""
    rng = np.random.Generator(np.random.PCG64([seed, tid, 0x70E]))
    return torch.from_numpy(rng.standard_normal((T, E), dtype=np.float32))


# ----------------------------------------------------------------------------------------------
# Workload shapes
# ----------------------------------------------------------------------------------------------

PACK_B3 = 1   # base-3, 20 trits per uint32
PACK_2BIT = 2  # 2 bits per trit, 16 trits per uint32


@dataclasses.dataclass(frozen=True)
class Linear:
    name: str
    N: int   # output features (rows of W)
    K: int   # input features (reduction dim)


def dense_layer_linears(hidden: int = 5120, ffn: int = 17408, n_q: int = 40, n_kv: int = 8, head_dim: int = 128):
    """The seven ternary linears of one 27B-class decoder layer (q/k/v/o attention + gate/up/down FFN)."""
    return [
        Linear("q", n_q * head_dim, hidden),
        Linear("k", n_kv * head_dim, hidden),
        Linear("v", n_kv * head_dim, hidden),
        Linear("o", hidden, n_q * head_dim),
        Linear("gate", ffn, hidden),
        Linear("up", ffn, hidden),
        Linear("down", hidden, ffn),
    ]


def stacked_layer_linears(hidden: int = 5120, ffn: int = 17408, n_q: int = 40, n_kv: int = 8, head_dim: int = 128):
    """The same seven linears grouped as an inference engine calls them: q, k and v read the same input
    and are stacked into one projection (rows q, then k, then v), gate and up likewise (rows gate, then
    up).  Every weight is still read once per token; four calls per layer instead of seven."""
    return [
        Linear("qkv", (n_q + 2 * n_kv) * head_dim, hidden),
        Linear("o", hidden, n_q * head_dim),
        Linear("gate_up", 2 * ffn, hidden),
        Linear("down", hidden, ffn),
    ]


def seed_of(config: int) -> int:
    """Seed of workload ``config`` (1..5): the single-layer case uses seed 0, workload c uses 1000*c."""
    return 0 if config == 1 else 1000 * config


SINGLE_LINEAR = dict(N=1024, K=1024, B=1, group=128, packing=PACK_B3, fwht_block=128, outlier_frac=0.005)
MOE = dict(E=256, topk=8, H=2048, F=512, group=64, packing=PACK_B3, fwht_block=128, tokens=(1, 8, 64))
PREFILL = dict(shapes=((2048, 5120, 17408), (4096, 17408, 5120)), group=128, packing=PACK_2BIT, fwht_block=128)
DENSE_DECODE = dict(batches=(1, 4, 16), group=128, packings=(PACK_B3, PACK_2BIT), fwht_block=128)
STREAM = dict(layers=64, batches=(1, 8), group=128, fwht_block=128)
