"""Pins for the CPU oracle: each check compares the oracle with something other than itself.

Every ``pin_*`` function takes an oracle-like namespace and raises AssertionError if it disagrees
with an independent statement of the same fact: Python's own base-3 / base-4 integer parsing, the
closed form of Sylvester Hadamard entries, orthogonality, brute-force pure-Python contractions on
tiny inputs, closed forms of special cases, and brute-force routing.  The tests run every pin on
the real oracle (must pass) and on oracles with one planted mistake each (must fail), so a
plausible slip in the oracle - wrong digit order, wrong sign in the Hadamard recursion, a missing
normalisation, a transposed operand, a wrong tie-break - cannot pass unnoticed.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O_real
from ternary_weight_quantized_unpack_b300 import inputs
from tq_testlib import fp8_bound

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "format_constants.txt")


def golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, value = line.split()[:2]
            vals[name] = float(value) if "." in value else int(value)
    return vals


def rng(seed=0):
    return np.random.Generator(np.random.PCG64(seed))


def popcount(v):
    return bin(v).count("1")


def fwht_closed_form(xrow, block):
    """x~_r = sum_c (-1)^popcount(r & c) x_c / sqrt(block), per block, pure Python."""
    out = []
    for b0 in range(0, len(xrow), block):
        xs = xrow[b0:b0 + block]
        for r in range(block):
            out.append(sum(((-1) ** popcount(r & c)) * xs[c] for c in range(block)) / math.sqrt(block))
    return out


# ----------------------------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------------------------

def pin_pack_b3(O):
    r = rng(1)
    for K in (1, 19, 20, 21, 67, 160):
        t = r.integers(-1, 2, size=(3, K)).astype(np.int8)
        codes = O.pack(t, O.PACK_B3)
        P = codes.shape[1]
        assert P == -(-(-(-K // 20)) // 4) * 4
        for n in range(3):
            digits = [int(v) + 1 for v in t[n]] + [1] * (P * 20 - K)
            for j in range(P):
                d = digits[20 * j: 20 * j + 20]
                # Python parses the most significant digit first; digit i has weight 3**i
                assert int(codes[n, j]) == int("".join(str(v) for v in reversed(d)), 3)


def pin_pack_2b(O):
    r = rng(2)
    for K in (1, 15, 16, 17, 100, 128):
        t = r.integers(-1, 2, size=(3, K)).astype(np.int8)
        codes = O.pack(t, O.PACK_2BIT)
        P = codes.shape[1]
        assert P == -(-(-(-K // 16)) // 4) * 4
        for n in range(3):
            digits = [int(v) + 1 for v in t[n]] + [1] * (P * 16 - K)
            for j in range(P):
                d = digits[16 * j: 16 * j + 16]
                assert int(codes[n, j]) == int("".join(str(v) for v in reversed(d)), 4)


def pin_unpack(O):
    r = rng(3)
    for packing in (O.PACK_B3, O.PACK_2BIT):
        for K in (1, 37, 128, 301):
            t = r.integers(-1, 2, size=(4, K)).astype(np.int8)
            back, bad = O.unpack(O.pack(t, packing), K, packing)
            assert bad == 0 and back.dtype == np.int8 and np.array_equal(back, t)
    # all 3^5 patterns in the low five digits, the rest random; and the extremes
    low = np.array(np.meshgrid(*[[-1, 0, 1]] * 5, indexing="ij")).reshape(5, -1).T
    hi = r.integers(-1, 2, size=(low.shape[0], 15))
    t = np.concatenate([low, hi], axis=1).astype(np.int8)
    codes = O.pack(t, O.PACK_B3)
    back, bad = O.unpack(codes, 20, O.PACK_B3)
    assert bad == 0 and np.array_equal(back, t)
    assert len(set(int(c) for c in codes[:, 0])) == 243
    # hand-decoded words: 5 = 12 in base 3 -> digits (2, 1, 0, ...) -> t = (+1, 0, -1, -1, ...)
    one, bad = O.unpack(np.array([[5, 0, 0, 0]], dtype=np.uint32), 3, O.PACK_B3)
    assert bad == 0 and one.tolist() == [[1, 0, -1]]
    # 2-bit: 0b10_01_00 = 36 -> fields (0, 1, 2) -> t = (-1, 0, +1)
    one, bad = O.unpack(np.array([[36, 0, 0, 0]], dtype=np.uint32), 3, O.PACK_2BIT)
    assert bad == 0 and one.tolist() == [[-1, 0, 1]]
    # invalid words are counted
    bad_b3 = np.array([[3 ** 20, 2 ** 32 - 1, 3 ** 20 - 1, 0]], dtype=np.uint32)
    assert O.unpack(bad_b3, 80, O.PACK_B3)[1] == 2
    bad_2b = np.array([[0x55555555, 0x55555557, 0xC0000000, 0]], dtype=np.uint32)
    assert O.unpack(bad_2b, 64, O.PACK_2BIT)[1] == 2


def pin_format_constants(O):
    g = golden()
    assert g["trits_per_b3_word"] == O.B3_TRITS == 20
    assert 3 ** 20 - 1 == g["b3_max_word"] == O.B3_MAX < g["two_pow_32"] < 3 ** 21
    plus = O.pack(np.ones((1, 20), np.int8), O.PACK_B3)[0, 0]
    zero = O.pack(np.zeros((1, 20), np.int8), O.PACK_B3)[0, 0]
    minus = O.pack(-np.ones((1, 20), np.int8), O.PACK_B3)[0, 0]
    assert (int(plus), int(zero), int(minus)) == (g["b3_max_word"], g["b3_all_zero_word"], g["b3_all_minus_word"])
    assert int(O.pack(np.zeros((1, 16), np.int8), O.PACK_2BIT)[0, 0]) == g["b2_all_zero_word"]
    # bits per weight of the codes alone (K a multiple of 80 so the 16-byte pitch adds nothing)
    N, K = 64, 5120
    assert O.packed_bytes(N, K, O.PACK_B3) * 8 / (N * K) == g["b3_bits_per_weight"]
    assert O.packed_bytes(N, K, O.PACK_2BIT) * 8 / (N * K) == 2.0
    assert O.scale_bytes(N, K, g["group_size_dense"]) * 8 / (N * K) == 16 / 128
    assert round(math.log2(3), 2) == g["trit_entropy_bits"]
    # the pages' own size arithmetic: 27B weights at 1.76 bpw is the 5.93 GB file, 1/9 of FP16
    assert abs(27e9 * g["avg_bits_with_scales"] / 8 / 1e9 - g["file_27b_gb"]) < 0.02
    assert abs(g["fp16_27b_gb"] / g["file_27b_gb"] - 9) < 0.1
    # the 7.21 GB tier is consistent with 2-bit codes + FP16 group-128 scales (2.125 bpw) within 1 %
    bpw_2b = (O.packed_bytes(N, K, O.PACK_2BIT) + O.scale_bytes(N, K, 128)) * 8 / (N * K)
    assert bpw_2b == 2.125 and abs(27e9 * bpw_2b / 8 / 1e9 / g["gguf_tier2_gb"] - 1) < 0.01


def pin_hadamard(O):
    assert O.hadamard(2).tolist() == [[1, 1], [1, -1]]
    assert O.hadamard(4).tolist() == [[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]]
    for n in (1, 2, 4, 8, 16, 32, 64, 128):
        H = O.hadamard(n)
        for i in range(n):
            for j in range(n):
                assert H[i, j] == (-1) ** popcount(i & j)
        assert np.array_equal(H @ H.T, n * np.eye(n))


def pin_fwht(O):
    n = 128
    eye = np.eye(n)
    out = O.block_fwht(eye, n)
    for i in range(n):  # transform of e_i is column i of H / sqrt(n), from the closed form
        for r in range(n):
            assert abs(out[i, r] - ((-1) ** popcount(r & i)) / math.sqrt(n)) < 1e-15
    x = rng(4).standard_normal((3, 4 * n))
    y = O.block_fwht(x, n)
    assert np.allclose(O.block_fwht(y, n), x, atol=1e-13)       # orthonormal & symmetric: involution
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    small = rng(5).standard_normal((1, 2 * n))
    assert np.allclose(O.block_fwht(small, n)[0], fwht_closed_form(list(small[0]), n), atol=1e-12)
    assert np.array_equal(O.block_fwht(x, 0), x)


def pin_rotation_identity(O):
    """y = W x = (W H^T / sqrt n)(H x / sqrt n) for a dense W: the pre-rotation is lossless."""
    r = rng(6)
    n = 128
    W = r.standard_normal((5, 2 * n))
    x = r.standard_normal((2, 2 * n))
    Hb = np.kron(np.eye(2), O.hadamard(n)) / math.sqrt(n)
    lhs = x @ W.T
    rhs = O.block_fwht(x, n) @ (W @ Hb.T).T
    assert np.allclose(lhs, rhs, atol=1e-12)


def pin_contraction_bruteforce(O):
    """ternary_linear against pure-Python loops on tiny ragged inputs, both packings."""
    r = rng(7)
    for packing, group in ((O.PACK_B3, 128), (O.PACK_2BIT, 64), (O.PACK_B3, 64)):
        N, K, B = 3, 256, 2
        t = r.integers(-1, 2, size=(N, K)).astype(np.int8)
        s = np.exp(r.normal(-4, 0.5, size=(N, K // group))).astype(np.float16)
        x = r.standard_normal((B, K)).astype(np.float32)
        y, A, bad = O.ternary_linear(O.pack(t, packing), s, x, K, group, packing, 128)
        assert bad == 0
        for b in range(B):
            xt = fwht_closed_form([float(v) for v in x[b]], 128)
            for nn in range(N):
                acc = 0.0
                aab = 0.0
                for k in range(K):
                    term = float(s[nn, k // group]) * int(t[nn, k]) * xt[k]
                    acc += term
                    aab += abs(term)
                assert abs(y[b, nn] - acc) <= 1e-12 * max(1.0, aab)
                assert abs(A[b, nn] - aab) <= 1e-12 * max(1.0, aab)


def pin_pack_3bit(O):
    """3-bit codes against Python's own base-8 parsing of each 16-bit half of a word (five digits
    q + 4, least significant first, bit 15 left zero; blocks of 64 codes in 7 words, word 6 holding
    codes 60, 61 in its low half and 62, 63 in its high half, every other digit q = 0), a hand-worked
    block, the row pitch, the invalid-word count and the contraction by brute force."""
    r = rng(31)

    def half(digits):
        return int("".join(str(d) for d in reversed(digits)), 8)

    for K in (1, 10, 63, 64, 65, 200, 640):
        q = r.integers(-4, 4, size=(3, K)).astype(np.int8)
        codes = O.pack(q, O.PACK_3BIT)
        nb = -(-K // 64)
        assert codes.shape == (3, -(-nb * 7 // 4) * 4)
        for n in range(3):
            for b in range(nb):
                def dig(c):
                    k = 64 * b + c
                    return int(q[n, k]) + 4 if k < K else 4
                for i in range(6):
                    lo = [dig(10 * i + j) for j in range(5)]
                    hi = [dig(10 * i + 5 + j) for j in range(5)]
                    assert int(codes[n, 7 * b + i]) == half(lo) + (half(hi) << 16)
                lo6 = [dig(60), dig(61), 4, 4, 4]
                hi6 = [dig(62), dig(63), 4, 4, 4]
                assert int(codes[n, 7 * b + 6]) == half(lo6) + (half(hi6) << 16)
        back, bad = O.unpack(codes, K, O.PACK_3BIT)
        assert bad == 0 and np.array_equal(back, q)
    q = np.array([[k % 8 - 4 for k in range(64)]], dtype=np.int8)   # digit of code k is k % 8
    c = O.pack(q, O.PACK_3BIT)
    assert int(c[0, 0]) == 0o43210 | (0o10765 << 16)
    assert int(c[0, 1]) == 0o65432 | (0o32107 << 16)
    assert int(c[0, 6]) == 0o44454 | (0o44476 << 16)
    back, bad = O.unpack(c, 64, O.PACK_3BIT)
    assert bad == 0 and np.array_equal(back, q)
    for bit in (15, 31):
        bad_codes = c.copy()
        bad_codes[0, 2] |= np.uint32(1 << bit)
        assert O.unpack(bad_codes, 64, O.PACK_3BIT)[1] == 1
    ok_codes = c.copy()
    ok_codes[0, 6] ^= np.uint32(7 << 6)    # a padding slot of word 6: not validated, not read
    back, bad = O.unpack(ok_codes, 64, O.PACK_3BIT)
    assert bad == 0 and np.array_equal(back, q)
    # the contraction on 3-bit codes: y = sum_k s q x~, brute force
    N, K, B, group = 2, 256, 2, 64
    q = r.integers(-4, 4, size=(N, K)).astype(np.int8)
    sc = np.exp(r.normal(-4, 0.5, size=(N, K // group))).astype(np.float16)
    x = r.standard_normal((B, K)).astype(np.float32)
    y, A, bad = O.ternary_linear(O.pack(q, O.PACK_3BIT), sc, x, K, group, O.PACK_3BIT, 128)
    assert bad == 0
    for b in range(B):
        xt = fwht_closed_form([float(v) for v in x[b]], 128)
        for nn in range(N):
            terms = [float(sc[nn, k // group]) * int(q[nn, k]) * xt[k] for k in range(K)]
            assert abs(y[b, nn] - sum(terms)) <= 1e-12 * max(1.0, sum(abs(v) for v in terms))


def pin_special_cases(O):
    r = rng(8)
    N, K, B = 4, 384, 3
    x = r.standard_normal((B, K)).astype(np.float32)
    s = np.exp(r.normal(-4, 0.5, size=(N, K // 128))).astype(np.float16)
    # all t = 0 -> exactly 0
    y, A, _ = O.ternary_linear(O.pack(np.zeros((N, K), np.int8), O.PACK_B3), s, x, K, 128, O.PACK_B3)
    assert np.all(y == 0) and np.all(A == 0)
    # all t = +1 with s = 1: sum over a block of H x / sqrt(n) is sqrt(n) * x[first of block]
    ones = np.ones((N, K // 128), np.float16)
    y, _, _ = O.ternary_linear(O.pack(np.ones((N, K), np.int8), O.PACK_2BIT), ones, x, K, 128, O.PACK_2BIT)
    expect = math.sqrt(128) * x[:, ::128].astype(np.float64).sum(axis=1)
    assert np.allclose(y, expect[:, None], atol=1e-12)
    # one non-zero trit at k with scale s -> +-s * x~_k, x~_k from the popcount closed form
    k = 200
    t = np.zeros((N, K), np.int8)
    t[1, k] = -1
    y, _, _ = O.ternary_linear(O.pack(t, O.PACK_B3), s, x, K, 128, O.PACK_B3)
    blk, rr = divmod(k, 128)
    for b in range(B):
        xk = sum(((-1) ** popcount(rr & c)) * float(x[b, 128 * blk + c]) for c in range(128)) / math.sqrt(128)
        assert abs(y[b, 1] - (-float(s[1, blk]) * xk)) < 1e-12
        assert y[b, 0] == 0 and y[b, 2] == 0


def route_bruteforce(logits, k):
    idx, gates = [], []
    for row in logits:
        vals = [float(v) for v in row]
        chosen = []
        for _ in range(k):
            best = None
            for e, v in enumerate(vals):
                if e in chosen:
                    continue
                if best is None or v > vals[best]:  # strict '>' keeps the lower index on ties
                    best = e
            chosen.append(best)
        m = max(vals[e] for e in chosen)
        ex = [math.exp(vals[e] - m) for e in chosen]
        idx.append(chosen)
        gates.append([v / sum(ex) for v in ex])
    return idx, gates


def pin_moe_route(O):
    r = rng(9)
    logits = r.standard_normal((5, 256)).astype(np.float32)
    logits[3, [7, 100, 200]] = 4.0      # three-way tie at the top
    logits[4, :] = 0.25                 # everything tied
    idx, gate = O.moe_route(logits, 8)
    bi, bg = route_bruteforce(logits, 8)
    assert idx.tolist() == bi
    assert np.allclose(gate, np.array(bg), atol=1e-15)
    assert np.allclose(gate.sum(axis=1), 1.0, atol=1e-15)
    assert idx[3, :3].tolist() == [7, 100, 200] and idx[4].tolist() == list(range(8))


def _moe_case(O, r, E=6, H=256, F=128, group=64, T=3):
    P_H = O.row_pitch_words(H, O.PACK_B3)
    P_F = O.row_pitch_words(F, O.PACK_B3)
    gu_t = r.integers(-1, 2, size=(E, 2 * F, H)).astype(np.int8)
    d_t = r.integers(-1, 2, size=(E, H, F)).astype(np.int8)
    gu_c = np.stack([O.pack(gu_t[e], O.PACK_B3) for e in range(E)])
    d_c = np.stack([O.pack(d_t[e], O.PACK_B3) for e in range(E)])
    assert gu_c.shape == (E, 2 * F, P_H) and d_c.shape == (E, H, P_F)
    gu_s = np.exp(r.normal(-2, 0.5, size=(E, 2 * F, H // group))).astype(np.float16)
    d_s = np.exp(r.normal(-2, 0.5, size=(E, H, F // group))).astype(np.float16)
    x = r.standard_normal((T, H)).astype(np.float32)
    return gu_c, gu_s, d_c, d_s, x


def _ffn(O, gc, gs, dc, ds, x, H, F, group):
    gu, _, _ = O.ternary_linear(gc, gs, x, H, group, O.PACK_B3)
    h = gu[:, :F] / (1 + np.exp(-gu[:, :F])) * gu[:, F:]
    y, _, _ = O.ternary_linear(dc, ds, h, F, group, O.PACK_B3)
    return y


def pin_moe_layer(O):
    r = rng(10)
    E, H, F, group, T = 6, 256, 128, 64, 3
    gu_c, gu_s, d_c, d_s, x = _moe_case(O, r, E, H, F, group, T)
    # one expert forced (+50): the layer reduces to that expert's SwiGLU FFN
    logits = r.standard_normal((T, E)).astype(np.float32)
    logits[:, 4] = 50.0
    out = O.moe_layer(logits, x, gu_c, gu_s, d_c, d_s, H, F, group, O.PACK_B3, topk=2)
    ref = _ffn(O, gu_c[4], gu_s[4], d_c[4], d_s[4], x, H, F, group)
    assert np.allclose(out["y"], ref, rtol=1e-9, atol=1e-12)
    assert (out["idx"][:, 0] == 4).all()
    # all experts identical: gates sum to one, so the layer equals the single FFN exactly
    same = [np.repeat(a[:1], E, axis=0) for a in (gu_c, gu_s, d_c, d_s)]
    logits = r.standard_normal((T, E)).astype(np.float32)
    out = O.moe_layer(logits, x, *same, H, F, group, O.PACK_B3, topk=3)
    ref = _ffn(O, same[0][0], same[1][0], same[2][0], same[3][0], x, H, F, group)
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-12)
    # generic case: y = sum_j gate_j * FFN_{e_j}(x), with experts evaluated one by one
    out = O.moe_layer(logits, x, gu_c, gu_s, d_c, d_s, H, F, group, O.PACK_B3, topk=3)
    for t in range(T):
        acc = 0
        for j in range(3):
            e = int(out["idx"][t, j])
            acc = acc + out["gate"][t, j] * _ffn(O, gu_c[e], gu_s[e], d_c[e], d_s[e], x[t:t + 1], H, F, group)[0]
        assert np.allclose(out["y"][t], acc, rtol=1e-12, atol=1e-12)


def pin_silu(O):
    """silu(z) = z * sigmoid(z), checked against facts of the logistic function that do not restate
    the formula: sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4 (so
    silu(+-ln 3) = +-(3/4) ln 3 and -(1/4) ln 3), silu(z) - silu(-z) = z (because
    sigmoid(z) + sigmoid(-z) = 1), silu(z) -> z for large z and -> 0 for very negative z, and the
    slope 1/2 at the origin."""
    ln3 = math.log(3.0)
    z = np.array([0.0, ln3, -ln3, 1.0, -2.5, 7.0])
    v = O.silu(z)
    assert v[0] == 0.0
    assert abs(v[1] - 0.75 * ln3) <= 1e-15 and abs(v[2] + 0.25 * ln3) <= 1e-15
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=0, atol=1e-14)
    assert abs(O.silu(np.array([40.0]))[0] - 40.0) <= 40.0 * 1e-15
    assert 0 > O.silu(np.array([-40.0]))[0] > -1e-15
    h = 1e-8
    assert abs(O.silu(np.array([h]))[0] / h - 0.5) < 1e-7


def pin_moe_down_from_h(O):
    """The down-projection + combine stage restated from a given h (the form the GPU test uses to
    check that stage on the GPU's own h) equals the full layer when given the layer's own h."""
    r = rng(12)
    E, H, F, group, T, k = 6, 256, 128, 64, 4, 3
    gu_c, gu_s, d_c, d_s, x = _moe_case(O, r, E, H, F, group, T)
    logits = r.standard_normal((T, E)).astype(np.float32)
    out = O.moe_layer(logits, x, gu_c, gu_s, d_c, d_s, H, F, group, O.PACK_B3, topk=k)
    downs = {e: (d_c[e], d_s[e]) for e in range(E)}
    y, A = O.moe_down_from_h(out["h"], out["idx"], out["gate"], downs, F, group, O.PACK_B3)
    assert np.allclose(y, out["y"], rtol=1e-12, atol=1e-12)
    assert np.allclose(A, np.einsum("tj,tjh->th", out["gate"], out["A_d"]), rtol=1e-12, atol=1e-12)
    # and a single routed slot reduces to one plain ternary linear on FWHT(h)
    y1, _ = O.moe_down_from_h(out["h"][:1, :1], out["idx"][:1, :1], np.ones((1, 1)), downs, F, group, O.PACK_B3)
    ref, _, _ = O.ternary_linear(d_c[int(out["idx"][0, 0])], d_s[int(out["idx"][0, 0])], out["h"][0, :1], F, group,
                                 O.PACK_B3)
    assert np.allclose(y1, ref, rtol=1e-12, atol=1e-12)


def bf16_round(a):
    """Round float values to bf16 (nearest even) and back, with torch as the converter."""
    import torch
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def scipy_rotation(W, block=128):
    """w' = W_blk @ H^T / sqrt(block), with scipy's Hadamard matrix (a separate construction)."""
    from scipy.linalg import hadamard as scipy_hadamard
    H = scipy_hadamard(block).astype(np.float64)
    N, K = W.shape
    return (np.asarray(W, np.float64).reshape(N, K // block, block) @ H.T / math.sqrt(block)).reshape(N, K)


def pin_quantize_closed_form(O):
    """One non-zero a at column j of a 128-block rotates to a * (-1)^popcount(r & j) / sqrt(128) at
    every r: all |w'| equal, so the scale is fp16(|a| / sqrt(128)) for each group of the block and
    t_r = sign(a) (-1)^popcount(r & j).  Every block of a row gets its own a and j (one block is all
    zero: scale 0, t 0), so group bookkeeping, the sign pattern and the normalisation all show.
    Without the transform a group of 64 values 3/16 and 64 values 1/16 has mean 1/8 = its scale, and
    the 1/16 entries sit exactly halfway between 0 and 1/8: they go to 0."""
    r = rng(21)
    N, nb = 3, 4
    K = 128 * nb
    W = np.zeros((N, K))
    pos = {}
    for n in range(N):
        for b in range(nb):
            if (n, b) == (1, 2):
                continue
            a = float(bf16_round([r.choice([-1, 1]) * 2.0 ** r.integers(-8, 3) * (1 + r.integers(0, 128) / 128)])[0])
            j = int(r.integers(0, 128))
            W[n, 128 * b + j] = a
            pos[(n, b)] = (a, j)
    for group in (128, 64):
        codes, scales, trits = O.quantize(W, group, O.PACK_2BIT)
        for n in range(N):
            for b in range(nb):
                gs = slice(b * 128 // group, (b + 1) * 128 // group)
                if (n, b) not in pos:
                    assert np.all(scales[n, gs] == 0) and np.all(trits[n, 128 * b:128 * (b + 1)] == 0)
                    continue
                a, j = pos[(n, b)]
                want_s = np.float16(abs(a) / math.sqrt(128.0))
                assert np.all(np.abs(scales[n, gs].astype(np.float64) - float(want_s)) <= float(want_s) * 2 ** -10)
                want_t = [int(np.sign(a)) * (-1) ** popcount(rr & j) for rr in range(128)]
                assert trits[n, 128 * b:128 * (b + 1)].tolist() == want_t
        t_back, bad = O.unpack(codes, K, O.PACK_2BIT)
        assert bad == 0 and np.array_equal(t_back, trits)
    W0 = np.array([[3 / 16] * 64 + [1 / 16] * 64 + [-3 / 16] * 64 + [-1 / 16] * 64])
    _, s0, t0 = O.quantize(W0, 128, O.PACK_B3, fwht_block=0)
    assert s0.tolist() == [[0.125, 0.125]]
    assert t0.tolist() == [[1] * 64 + [0] * 64 + [-1] * 64 + [0] * 64]


def pin_quantize_nearest_level(O):
    """On Gaussian bf16 weights with outliers: the scale is fp16 of the group's mean |w'| (w' from
    scipy's Hadamard matrix), every t is the level of S * {-1, 0, +1} nearest to w', negating W
    negates t, and scaling W by 4 keeps t and scales S by 4."""
    r = rng(22)
    N, K = 6, 512
    W = r.standard_normal((N, K)) * 0.02
    W[r.random((N, K)) < 0.01] *= 20
    W = bf16_round(W)
    wr = scipy_rotation(W)
    for group in (128, 64):
        _, S, t = O.quantize(W, group, O.PACK_B3)
        mean = np.abs(wr).reshape(N, K // group, group).mean(axis=2)
        assert np.all(np.abs(S.astype(np.float64) - mean) <= mean * 2 ** -10)
        Sf = np.repeat(S.astype(np.float64), group, axis=1)
        dist = np.stack([np.abs(wr - Sf * lv) for lv in (-1, 0, 1)])
        best = dist.min(axis=0)
        chosen = np.abs(wr - Sf * t)
        assert np.all(chosen <= best + 1e-12 * Sf)
        assert np.mean(t != 0) > 0.4
        _, Sn, tn = O.quantize(-W, group, O.PACK_B3)
        assert np.array_equal(tn, -t) and np.array_equal(Sn, S)
        _, S4, t4 = O.quantize(4 * W, group, O.PACK_B3)
        assert np.array_equal(t4, t) and np.array_equal(S4.astype(np.float64), 4 * S.astype(np.float64))


def pin_quantize_round_trip(O):
    """The rotation loses nothing: weights that are already ternary times a group scale in the
    rotated basis, rotated back (scipy's Hadamard) and rounded to bf16, quantize back to the same
    trits; each scale comes back as S times the group's fraction of non-zero trits (the mean |w'|)."""
    r = rng(23)
    N, K = 5, 768
    for group in (128, 64):
        for packing in (O.PACK_B3, O.PACK_2BIT):
            T = r.integers(-1, 2, size=(N, K)).astype(np.int8)
            S = np.exp(r.standard_normal((N, K // group)) * 0.5 - 4).astype(np.float16).astype(np.float64)
            wr = np.repeat(S, group, axis=1) * T
            from scipy.linalg import hadamard as scipy_hadamard
            H = scipy_hadamard(128).astype(np.float64)
            W = bf16_round((wr.reshape(N, K // 128, 128) @ H / math.sqrt(128)).reshape(N, K))
            codes, S_q, t_q = O.quantize(W, group, packing)
            assert np.array_equal(t_q, T)
            t_back, bad = O.unpack(codes, K, packing)
            assert bad == 0 and np.array_equal(t_back, T)
            frac = (T != 0).reshape(N, K // group, group).mean(axis=2)
            assert np.allclose(S_q.astype(np.float64), S * frac, rtol=4e-3, atol=0)


def e4m3_grid():
    """Every finite FP8 E4M3 value from its bit fields (exponent e, mantissa m), by Python
    arithmetic, with the mantissa field of each."""
    grid = {}
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue  # the NaN pattern
            v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            grid[v] = m
            grid[-v] = m
    return grid


def pin_e4m3(O):
    """Rounding to FP8 E4M3: the grid enumerated from its bit fields is fixed, midpoints go to the
    even mantissa, points just off a midpoint to the nearer neighbour, magnitudes past 448 to 448, and
    torch's own E4M3 conversion agrees on random values in range."""
    grid = e4m3_grid()
    vals = np.array(sorted(grid))
    assert vals.max() == 448.0 and vals[vals > 0].min() == 2.0 ** -9 and len(vals) == 253
    assert np.array_equal(O.e4m3(vals), vals)
    pos = [v for v in sorted(grid) if v >= 0]
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = (lo + hi) / 2
        even = lo if grid[lo] % 2 == 0 else hi
        assert O.e4m3(mid) == even and O.e4m3(-mid) == -even, (lo, hi)
        assert O.e4m3(mid - (hi - lo) / 8) == lo and O.e4m3(mid + (hi - lo) / 8) == hi
    assert O.e4m3(1000.0) == 448.0 and O.e4m3(-470.0) == -448.0 and O.e4m3(2.0 ** -11) == 0.0
    r = rng(41)
    v = r.standard_normal(4000) * 10.0 ** r.uniform(-4, 2.5, 4000)
    v = v[np.abs(v) < 440]
    lib = torch.tensor(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3(v), lib)


def pin_pow2_exponent(O):
    """e = floor(log2 m) - 7: m * 2^-e in [128, 256), by Python's frexp; 0 for m = 0."""
    assert list(O.pow2_exponent([0.0, 1.0, 128.0, 255.9, 256.0, 2.0 ** -20])) == [0, -7, 0, 0, 1, -27]
    r = rng(42)
    m = np.exp(r.uniform(-30, 30, 500))
    e = O.pow2_exponent(m)
    scaled = m * np.exp2(-e.astype(np.float64))
    assert ((scaled >= 128) & (scaled < 256)).all()


def pin_linear_fp8(O):
    """The FP8 contraction: (a) operands already on the E4M3 grid under their row factors give the
    exact ternary result; (b) brute force with Python loops (frexp exponents, the pinned rounding) on a
    small case; (c) the distance to the exact result stays inside the derived bound."""
    r = rng(43)
    grid = np.array(sorted(v for v in e4m3_grid() if 16 <= abs(v) < 256))
    # (a) rows of x with a maximum in [128, 256), weights with group scales on the grid in [128, 256)
    N, K, B, group = 5, 256, 3, 64
    x = r.choice(grid, size=(B, K))
    x[:, 0] = 240.0
    t = r.integers(-1, 2, size=(N, K)).astype(np.int8)
    sc = r.choice(grid[(grid >= 128)], size=(N, K // group)).astype(np.float16)
    codes = O.pack(t, O.PACK_2BIT)
    y8, A8, bad = O.linear_fp8(codes, sc, x, K, group, O.PACK_2BIT, 0)
    y, A, _ = O.ternary_linear(codes, sc, x, K, group, O.PACK_2BIT, 0)
    assert bad == 0 and np.array_equal(y8, y) and np.array_equal(A8, A)
    # (b) brute force
    N, K, B, group = 3, 256, 2, 128
    t = r.integers(-1, 2, size=(N, K)).astype(np.int8)
    sc = np.exp(r.normal(-4, 0.5, size=(N, K // group))).astype(np.float16)
    x = (r.standard_normal((B, K)) * np.array([[1e-3], [50.0]])).astype(np.float32)
    codes = O.pack(t, O.PACK_B3)
    y8, _, _ = O.linear_fp8(codes, sc, x, K, group, O.PACK_B3, 128)
    for b in range(B):
        xt = fwht_closed_form([float(v) for v in x[b]], 128)
        ea = math.frexp(max(abs(v) for v in xt))[1] - 1 - 7
        for n in range(N):
            eb = math.frexp(max(abs(float(v)) for v in sc[n]))[1] - 1 - 7
            acc = 0.0
            for k in range(K):
                w = float(sc[n, k // group]) * int(t[n, k])
                acc += float(O.e4m3(xt[k] * 2.0 ** -ea)) * float(O.e4m3(w * 2.0 ** -eb))
            ref = acc * 2.0 ** (ea + eb)
            assert abs(y8[b, n] - ref) <= 1e-12 * max(1.0, abs(ref)), (b, n, y8[b, n], ref)
    # (c) the bound, on a case with a wide range of magnitudes
    N, K, B, group = 16, 512, 4, 64
    t = r.integers(-1, 2, size=(N, K)).astype(np.int8)
    sc = np.exp(r.normal(-4, 1.5, size=(N, K // group))).astype(np.float16)
    x = (r.standard_normal((B, K)) * np.exp(r.normal(0, 3, size=(B, K)))).astype(np.float32)
    codes = O.pack(t, O.PACK_2BIT)
    y8, _, _ = O.linear_fp8(codes, sc, x, K, group, O.PACK_2BIT, 128)
    y, _, _ = O.ternary_linear(codes, sc, x, K, group, O.PACK_2BIT, 128)
    xt = O.block_fwht(x, 128)
    W = O.dequant(t, sc, group)
    ea = np.array([math.frexp(np.abs(row).max())[1] - 8 for row in xt])
    eb = np.array([math.frexp(float(np.abs(row.astype(np.float64)).max()))[1] - 8 for row in sc])
    assert (np.abs(y8 - y) <= fp8_bound(xt, W, ea, eb)).all()
    assert np.abs(y8 - y).max() > 0   # the quantisation is not a no-op here


PINS = [pin_pack_b3, pin_pack_2b, pin_unpack, pin_format_constants, pin_hadamard, pin_fwht,
        pin_rotation_identity, pin_contraction_bruteforce, pin_special_cases, pin_moe_route, pin_moe_layer,
        pin_silu, pin_moe_down_from_h, pin_quantize_closed_form, pin_quantize_nearest_level,
        pin_quantize_round_trip, pin_pack_3bit, pin_e4m3, pin_pow2_exponent, pin_linear_fp8]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(O_real)


# ----------------------------------------------------------------------------------------------
# planted mistakes: each mutant must fail at least one pin
# ----------------------------------------------------------------------------------------------

ORIG = {k: getattr(O_real, k) for k in ("pack", "unpack", "hadamard", "block_fwht", "moe_route", "dequant",
                                        "silu", "moe_down_from_h", "quantize")}


def _pack3_blocks_of_60(trits, packing):
    """3-bit codes packed densely (no block padding: 6 words of 10 per 60 codes)."""
    if packing != O_real.PACK_3BIT:
        return ORIG["pack"](trits, packing)
    q = np.asarray(trits)
    N, K = q.shape
    P = O_real.row_pitch_words(K, packing)
    d = np.full((N, P * 10), 4, dtype=np.int64)
    d[:, :K] = q.astype(np.int64) + 4
    shifts = np.array([O_real.q3_slot_bit(j) for j in range(10)])
    w = (d.reshape(N, P, 10) << shifts).sum(axis=2)
    return w.astype(np.uint32)


def _pack3_no_half_gap(trits, packing):
    """3-bit slots at bits 3j for all ten slots (the high half starting at bit 15)."""
    if packing != O_real.PACK_3BIT:
        return ORIG["pack"](trits, packing)
    w = ORIG["pack"](trits, packing).astype(np.int64)
    hi = (w >> 16) & 0x7FFF
    return ((w & 0x7FFF) | (hi << 15)).astype(np.uint32)


def _pack_msd_first(trits, packing):
    return ORIG["pack"](np.asarray(trits)[:, ::-1].copy(), packing)  # digit order reversed per row


def _hadamard_wrong_sign(n):
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [-H, H]])
    return H


def _fwht_unnormalised(x, block=128):
    return ORIG["block_fwht"](x, block) * (math.sqrt(block) if block else 1.0)


def _fwht_skipped(x, block=128):
    return np.asarray(x, dtype=np.float64).copy()


def _route_ties_high(logits, topk=8):
    logits = np.asarray(logits, np.float32)
    idx, gate = ORIG["moe_route"](logits[:, ::-1].copy(), topk)
    return (logits.shape[1] - 1 - idx).astype(np.int32), gate


def _route_softmax_all(logits, topk=8):
    idx, _ = ORIG["moe_route"](logits, topk)
    l = np.asarray(logits, np.float64)
    e = np.exp(l - l.max(axis=1, keepdims=True))
    full = e / e.sum(axis=1, keepdims=True)
    return idx, np.take_along_axis(full, idx.astype(np.int64), axis=1)


def _dequant_tiled(trits, scales, group):
    t = np.asarray(trits, np.float64)
    s = np.asarray(scales, np.float64)
    return np.tile(s, (1, group))[:, :t.shape[1]] * t   # wrong: interleaves groups instead of repeating


def _dequant_sign_flipped(trits, scales, group):
    return -ORIG["dequant"](trits, scales, group)


def _silu_mirrored(z):
    return z / (1.0 + np.exp(z))    # z * sigmoid(-z)


def _down_without_gates(h, idx, gate, experts_down, F, group, packing, fwht_block=128):
    return ORIG["moe_down_from_h"](h, idx, np.ones_like(gate), experts_down, F, group, packing, fwht_block)


def _unpack_off_by_one(codes, K, packing):
    t, bad = ORIG["unpack"](codes, K, packing)
    return np.roll(t, 1, axis=1), bad


def _quantize_with(stat="mean", thr=0.5, rotate=True, c=None, ties_up=False, interleaved=False, flip=False):
    """The quantizer with one step changed (a planted mistake)."""
    def q(W, group, packing, fwht_block=128):
        W = np.asarray(W, np.float64)
        N, K = W.shape
        if rotate and fwht_block:
            u = (W.reshape(N, K // 128, 128) @ O_real.hadamard(128).T).reshape(N, K)
            cc = O_real.INV_SQRT128 if c is None else c
        else:
            u, cc = W.copy(), 1.0
        g = np.abs(u).reshape(N, group, K // group).transpose(0, 2, 1) if interleaved else \
            np.abs(u).reshape(N, K // group, group)
        m = g.max(axis=2) if stat == "max" else g.sum(axis=2) / group
        S = (m * cc).astype(np.float16)
        lim = np.repeat(S.astype(np.float64) * thr, group, axis=1)
        hit = np.abs(u) * cc >= lim if ties_up else np.abs(u) * cc > lim
        t = np.where(hit, np.sign(u), 0.0).astype(np.int8)
        if flip:
            t = -t
        return O_real.pack(t, packing), S, t
    return q


def _e4m3_ties_away(v):
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    step = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / step + 0.5) * step, 448.0), v)


def _pow2_exponent_one_high(m):
    return ORIG_FP8["pow2_exponent"](m) + 1


def _linear_fp8_without_weight_factor(codes, scales, x, K, group, packing, fwht_block=128):
    y, A, bad = ORIG_FP8["linear_fp8"](codes, scales, x, K, group, packing, fwht_block)
    eb = ORIG_FP8["pow2_exponent"](np.abs(np.asarray(scales, dtype=np.float64)).max(axis=1))
    return y * np.ldexp(1.0, -eb)[None, :], A, bad


ORIG_FP8 = {k: getattr(O_real, k) for k in ("e4m3", "pow2_exponent", "linear_fp8")}


MUTANTS = {
    "3-bit blocks not padded to 64": dict(pack=_pack3_blocks_of_60),
    "3-bit high half starting at bit 15": dict(pack=_pack3_no_half_gap),
    "quantize scale from max": dict(quantize=_quantize_with(stat="max")),
    "quantize threshold 0.7 S": dict(quantize=_quantize_with(thr=0.7)),
    "quantize without rotation": dict(quantize=_quantize_with(rotate=False)),
    "quantize rotation unnormalised": dict(quantize=_quantize_with(c=1.0)),
    "quantize ties to +-1": dict(quantize=_quantize_with(ties_up=True)),
    "quantize groups interleaved": dict(quantize=_quantize_with(interleaved=True)),
    "quantize sign flipped": dict(quantize=_quantize_with(flip=True)),
    "pack digit order reversed": dict(pack=_pack_msd_first),
    "hadamard recursion sign": dict(hadamard=_hadamard_wrong_sign),
    "fwht missing 1/sqrt(n)": dict(block_fwht=_fwht_unnormalised),
    "transform skipped": dict(block_fwht=_fwht_skipped),
    "route ties to higher index": dict(moe_route=_route_ties_high),
    "gates softmax over all experts": dict(moe_route=_route_softmax_all),
    "scales repeated wrongly": dict(dequant=_dequant_tiled),
    "weight sign flipped": dict(dequant=_dequant_sign_flipped),
    "unpack shifted by one trit": dict(unpack=_unpack_off_by_one),
    "silu with sigmoid(-z)": dict(silu=_silu_mirrored),
    "down stage ignores the gates": dict(moe_down_from_h=_down_without_gates),
    "e4m3 ties away from zero": dict(e4m3=_e4m3_ties_away),
    "fp8 row exponent one too high": dict(pow2_exponent=_pow2_exponent_one_high),
    "fp8 result missing the weight factor": dict(linear_fp8=_linear_fp8_without_weight_factor),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    for k, v in MUTANTS[name].items():
        monkeypatch.setattr(O_real, k, v)
    failures = 0
    for pin in PINS:
        try:
            pin(O_real)
        except AssertionError:
            failures += 1
    assert failures >= 1, f"planted mistake '{name}' passed every pin"


def test_inputs_host_device_agree_on_cpu():
    """The counter-based generator gives the same trits for a row whether drawn alone or in bulk."""
    full = inputs.trits(11, 3, 40, 300)
    some = inputs.trits(11, 3, 40, 300, rows=[5, 17, 39])
    assert np.array_equal(full[[5, 17, 39]].numpy(), some.numpy())
    t = full.numpy()
    frac = [(t == v).mean() for v in (-1, 0, 1)]
    assert all(abs(f - 1 / 3) < 0.01 for f in frac)
    s = inputs.scales(11, 3, 40, 7).float().numpy()
    assert s.min() > 0 and abs(np.log(s).mean() + 4) < 0.1 and abs(np.log(s).std() - 0.5) < 0.05
    x = inputs.activations(0, 0, 1, 1024, outlier_frac=0.005).float().numpy()
    assert (np.abs(x) > 8).sum() >= 1
