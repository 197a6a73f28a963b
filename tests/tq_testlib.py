"""Shared helpers for the parity tests: build inputs on both sides, check the tolerance."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import ternary_weight_quantized_unpack_b300 as tq
from ternary_weight_quantized_unpack_b300 import inputs

REL_TOL = 1e-3   # |y - y_ref| <= REL_TOL * sum_k |s t x~| + ABS_TOL  (per output)
ABS_TOL = 1e-5


def check_tolerance(y, y_ref, A, extra=None, what="y"):
    """Elementwise |y - y_ref| <= 1e-3 * A + 1e-5 (+ extra).  Returns the worst error / bound ratio."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    bound = REL_TOL * np.asarray(A, dtype=np.float64) + ABS_TOL
    if extra is not None:
        bound = bound + extra
    err = np.abs(y - y_ref)
    assert np.all(np.isfinite(y)), f"{what}: non-finite values"
    ratio = err / bound
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert ratio[worst] <= 1.0, (f"{what}: worst at {worst}: got {y[worst]!r}, ref {y_ref[worst]!r}, "
                                 f"err {err[worst]:.3e} > bound {bound[worst]:.3e}")
    return float(ratio[worst])


def bf16_half_ulp(v):
    """Half a bf16 ulp at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return 0.5 * 2.0 ** (np.floor(np.log2(a)) - 7)


class LinearCase:
    """One ternary linear: seeded trits/scales/x, packed on the GPU by tq_pack, and the host copies
    the oracle reads (drawn from the same counter-based generator)."""

    def __init__(self, seed, tid, N, K, group, packing, batch, fwht_block=128, outlier_frac=0.0, device="cuda"):
        self.seed, self.tid, self.N, self.K, self.group, self.packing = seed, tid, N, K, group, packing
        self.batch, self.fwht_block = batch, fwht_block
        self.desc = tq.desc(N, K, group, packing, fwht_block)
        ng = O.n_groups(K, group)
        trits_dev = inputs.trits(seed, 2 * tid, N, K, device=device)
        self.codes = tq.tq_pack(self.desc, trits_dev)
        del trits_dev
        self.scales = inputs.scales(seed, 2 * tid + 1, N, ng, device=device).contiguous()
        self.x_host = inputs.activations(seed, tid, batch, K, outlier_frac=outlier_frac)
        self.x = self.x_host.to(device)

    def host_rows(self, rows):
        t = inputs.trits(self.seed, 2 * self.tid, self.N, self.K, rows=rows).numpy()
        s = inputs.scales(self.seed, 2 * self.tid + 1, self.N, O.n_groups(self.K, self.group), rows=rows).numpy()
        return t, s

    def oracle(self, rows=None):
        """(y_ref [batch, rows], A [batch, rows]) from the oracle, for all rows or a subset."""
        rows = np.arange(self.N) if rows is None else np.asarray(rows)
        t, s = self.host_rows(rows)
        codes = O.pack(t, self.packing)
        x = self.x_host.float().numpy()
        y, A, bad = O.ternary_linear(codes, s, x, self.K, self.group, self.packing, self.fwht_block)
        assert bad == 0
        return y, A


def sample_rows(N, n, seed=0):
    """A spread of rows: first, last, and n random ones (sorted, unique)."""
    r = np.random.Generator(np.random.PCG64(seed)).choice(N, size=min(n, N), replace=False)
    return np.unique(np.concatenate([[0, N - 1], r]))


def silu(z):
    return z / (1 + np.exp(-z))


def silu_prime(z):
    s = 1 / (1 + np.exp(-z))
    return s * (1 + z * (1 - s))


def moe_bounds(out, down_dense, fwht_block):
    """Tolerances of the expert layer derived from the per-linear bound 1e-3 * A + 1e-5.

    out: the oracle's moe_layer result for the checked tokens; down_dense: expert -> dense W_d
    (fp64 s * t).  Returns (hb, A_e2e, extra):
      hb     per-output bound on h = silu(g) * u, propagated from the bounds on g and u through
             silu (first order plus the second-order term, silu'' <= 1/2) and the product;
      A_e2e  sum_j gate_j * A_down, the plain down-stage scale;
      extra  the h bound carried through FWHT (a sum of |.| over each block / sqrt(block)) and |W_d|,
             weighted by the gates, plus a relative 1e-6 for the gates' own error.
    """
    Eg = 1e-3 * out["A_g"] + 1e-5
    Eu = 1e-3 * out["A_u"] + 1e-5
    g, u = out["g"], out["u"]
    hb = np.abs(silu(g)) * Eu + (np.abs(silu_prime(g)) * Eg + 0.25 * Eg ** 2) * (np.abs(u) + Eu) \
        + 1e-6 * np.abs(out["h"]) + 1e-7
    T, k, F = hb.shape
    H = out["y"].shape[1]
    blk = fwht_block or 1
    dht = np.repeat(hb.reshape(T, k, -1, blk).sum(axis=3), blk, axis=2) / math.sqrt(blk)
    extra = np.zeros((T, H))
    for ti in range(T):
        for j in range(k):
            Wd_abs = np.abs(down_dense[int(out["idx"][ti, j])])
            extra[ti] += out["gate"][ti, j] * (Wd_abs @ dht[ti, j]) + 1e-6 * np.abs(out["y_parts"][ti, j])
    A_e2e = np.einsum("tj,tjh->th", out["gate"], out["A_d"])
    return hb, A_e2e, extra


def fp8_bound(xt, W, ea, eb):
    """|y_fp8 - y| for the E4M3 operands: relative 2^-4 per operand (normals, half a 3-bit ulp) and,
    below 2^-6 after scaling, an absolute 2^-10 (half the subnormal spacing) times the row factor."""
    ax, aw = np.abs(xt), np.abs(W)
    A = ax @ aw.T
    fa = np.ldexp(1.0, ea)[:, None]
    fb = np.ldexp(1.0, eb)[None, :]
    K = xt.shape[1]
    return ((2.0 ** -3 + 2.0 ** -8) * A + 2.0 ** -10 * 1.07 * (fb * ax.sum(axis=1)[:, None] + fa * aw.sum(axis=1)[None, :])
            + K * 2.0 ** -20 * fa * fb)
