"""CPU oracle for the ternary-weight linear layer.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
``--impl reference`` arm) may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and this package imports nothing from the product.  The only
thing both sides share is the seeded input generator, which holds none of the method.

What it is: a plain, slow, fp64 numpy statement of what the method computes, written from the
pages in the order they give it.  No blocking, fusion or reordering beyond the definitions;
library primitives used as single steps are ``numpy.matmul`` and ``numpy.argsort``.

Sources (cited by title and section):
  [TT]  the page on the 1.58-bit TurboQuant-MLX build of Qwen3.6-35B-A3B on a 16 GB Mac,
        section "为什么 1.58bit 没变成乱码" (why 1.58 bit does not become gibberish), points 1-3.
  [CC]  "27B 大模型塞进 5.9GB：三值量化，凭什么「不崩」？",
        section 一 (what "ternary" means) and section 二 ①-③ (rotation, group scales, kernels).
  [NX]  the Ternary-Bonsai2-27B vs GSQ-RCO comparison page, §1.1 (ternary = sign + add/sub).

Readings where the pages are silent (each is listed in the design notes):
  * base-3 word = little-endian base-3 integer of the digits (t + 1); 20 digits per uint32,
    trits row-contiguous across group boundaries; trits past K are t = 0 (digit 1); each row is
    padded to a multiple of 4 words (16 bytes) with all-digit-1 words.
  * 2-bit word: field (t + 1) of trit k at bits 2*(k mod 16) of word k // 16; field 3 is invalid;
    padding fields are 1 (t = 0); rows padded to a multiple of 4 words.
  * Hadamard: Sylvester (natural) order, orthonormal scaling 1/sqrt(n), block 128 along K.
  * MoE: top-8 by raw logit, ties to the lower expert index; gates = softmax over the 8 chosen
    logits; SwiGLU expert h = silu(gate) * up; the expert input x and the down-projection input h
    are both block-Hadamard transformed; combine = sum_j gate_j * y_j.
  * Offline quantizer: the pages give the order (rotate, then one FP16 scale per group, then three
    levels) but not the rounding rule; this build takes the absmean rule of BitNet b1.58 (scale =
    mean |w'| over the group, t = the level of {-1, 0, +1} nearest to w' / scale, a tie at 1/2 to 0).

Parity pins (tests/test_oracle_pins.py): every function below is checked against something other
than itself - Python's own base-3/base-4 integer parsing, the closed form of Sylvester entries,
orthogonality, brute-force pure-Python contractions on tiny inputs, closed forms of special cases,
and brute-force routing.  End-to-end numbers printed on the pages: none exist for this path, so
no function here is pinned to a page-printed worked example.
"""
from __future__ import annotations

import math

import numpy as np

PACK_B3 = 1
PACK_2BIT = 2
PACK_3BIT = 3
B3_TRITS = 20      # [TT] point 3: base-3 code packs 20 ternary indices into one 32-bit integer
B2_TRITS = 16
B3_MAX = 3 ** 20 - 1  # largest valid base-3 word
# [TT] point 1: the non-expert linears (attention, GDN projections, lm_head) stay at 3 bits.  The
# page fixes no bit layout; this build's reading: integer codes q in {-4..3} (digit d = q + 4) times
# the group's FP16 scale.  A 32-bit word has ten 3-bit slots, five per 16-bit half: slot j < 5 at
# bits 3j, slot j >= 5 at bits 16 + 3(j - 5); bits 15 and 31 are zero.  Each block of 64 codes takes
# 7 words: word i < 6 holds codes 10i..10i+9 of the block in slots 0..9; word 6 holds codes 60, 61 in
# slots 0, 1 and codes 62, 63 in slots 5, 6, its other slots the padding digit.  No word straddles a
# group of 64 or 128.
Q3_PER_WORD = 10
Q3_BLOCK = 64
Q3_WORDS_PER_BLOCK = 7
Q3_PAD_DIGIT = 4   # q = 0
# (word, slot) of each code of a block, in code order
Q3_CODE_SLOTS = [(c // 10, c % 10) for c in range(60)] + [(6, 0), (6, 1), (6, 5), (6, 6)]


def q3_slot_bit(j: int) -> int:
    """Lowest bit of slot j of a 3-bit word."""
    return 3 * j if j < 5 else 16 + 3 * (j - 5)


# ----------------------------------------------------------------------------------------------
# Format: sizes
# ----------------------------------------------------------------------------------------------

def words_per_row(K: int, packing: int) -> int:
    """Words that hold one row of K trits (or 3-bit codes), before pitch padding."""
    if packing == PACK_3BIT:
        return -(-K // Q3_BLOCK) * Q3_WORDS_PER_BLOCK
    per = B3_TRITS if packing == PACK_B3 else B2_TRITS
    return -(-K // per)


def row_pitch_words(K: int, packing: int) -> int:
    """Row pitch in uint32 words: rounded up to a multiple of 4 (16 bytes)."""
    return -(-words_per_row(K, packing) // 4) * 4


def n_groups(K: int, group: int) -> int:
    return -(-K // group)


def packed_bytes(N: int, K: int, packing: int) -> int:
    return N * row_pitch_words(K, packing) * 4


def scale_bytes(N: int, K: int, group: int) -> int:
    """[CC] §二 ②: one FP16 scale per group of weights."""
    return N * n_groups(K, group) * 2


# ----------------------------------------------------------------------------------------------
# Format: pack / unpack   ([TT] point 3; 2-bit layout is this build's reading)
# ----------------------------------------------------------------------------------------------

def pack(trits: np.ndarray, packing: int) -> np.ndarray:
    """int8 trits [N, K] in {-1,0,1} -> uint32 codes [N, P].

    base-3: word j of a row = sum_{i<20} (t[20j+i] + 1) * 3**i.
    2-bit : word j of a row = sum_{i<16} (t[16j+i] + 1) << 2i.
    3-bit : codes q in {-4..3}; code c of 64-code block b sits as digit q + 4 in slot
            Q3_CODE_SLOTS[c] = (i, j) of word 7b + i, at bit q3_slot_bit(j) (padding digits 4, q = 0).
    """
    if packing == PACK_3BIT:
        return _pack3(trits)
    trits = np.asarray(trits)
    assert trits.ndim == 2 and np.isin(trits, (-1, 0, 1)).all()
    N, K = trits.shape
    P = row_pitch_words(K, packing)
    per = B3_TRITS if packing == PACK_B3 else B2_TRITS
    digits = np.ones((N, P * per), dtype=np.int64)           # padding trits are t = 0 -> digit 1
    digits[:, :K] = trits.astype(np.int64) + 1
    digits = digits.reshape(N, P, per)
    if packing == PACK_B3:
        weights = 3 ** np.arange(per, dtype=np.int64)
    else:
        weights = np.int64(1) << (2 * np.arange(per, dtype=np.int64))
    words = (digits * weights).sum(axis=2)
    return words.astype(np.uint32)


def _pack3(q: np.ndarray) -> np.ndarray:
    q = np.asarray(q)
    assert q.ndim == 2 and ((q >= -4) & (q <= 3)).all()
    N, K = q.shape
    nb = -(-K // Q3_BLOCK)
    P = row_pitch_words(K, PACK_3BIT)
    digits = np.full((N, nb, Q3_BLOCK), Q3_PAD_DIGIT, dtype=np.int64)
    digits.reshape(N, nb * Q3_BLOCK)[:, :K] = q.astype(np.int64) + 4
    slots = np.full((N, nb, Q3_WORDS_PER_BLOCK, Q3_PER_WORD), Q3_PAD_DIGIT, dtype=np.int64)
    for c, (i, j) in enumerate(Q3_CODE_SLOTS):
        slots[:, :, i, j] = digits[:, :, c]
    shifts = np.array([q3_slot_bit(j) for j in range(Q3_PER_WORD)], dtype=np.int64)
    words = (slots << shifts).sum(axis=3).reshape(N, nb * Q3_WORDS_PER_BLOCK)
    pad_word = sum(Q3_PAD_DIGIT << q3_slot_bit(j) for j in range(Q3_PER_WORD))
    out = np.full((N, P), pad_word, dtype=np.int64)
    out[:, :nb * Q3_WORDS_PER_BLOCK] = words
    return out.astype(np.uint32)


def _unpack3(codes: np.ndarray, K: int):
    codes = np.asarray(codes, dtype=np.uint32).astype(np.int64)
    N, P = codes.shape
    nb = -(-K // Q3_BLOCK)
    invalid = (codes & ((1 << 15) | (1 << 31))) != 0
    w = codes[:, :nb * Q3_WORDS_PER_BLOCK].reshape(N, nb, Q3_WORDS_PER_BLOCK)
    digits = np.empty((N, nb, Q3_BLOCK), dtype=np.int64)
    for c, (i, j) in enumerate(Q3_CODE_SLOTS):
        digits[:, :, c] = (w[:, :, i] >> q3_slot_bit(j)) & 7
    return (digits.reshape(N, nb * Q3_BLOCK)[:, :K] - 4).astype(np.int8), int(invalid.sum())


def unpack(codes: np.ndarray, K: int, packing: int):
    """uint32 codes [N, P] -> (int8 trits [N, K], number of invalid words).

    base-3: digit i of word v is (v // 3**i) % 3, t = digit - 1; a word above 3**20 - 1 is invalid.
    2-bit : field i is (v >> 2i) & 3, t = field - 1; a word holding a field equal to 3 is invalid.
    3-bit : slot j of word v is (v >> q3_slot_bit(j)) & 7, q = digit - 4; a word with bit 15 or 31 set
            is invalid.
    Every word of the row pitch is validated; the values of padding digits are not.
    """
    if packing == PACK_3BIT:
        return _unpack3(codes, K)
    codes = np.asarray(codes, dtype=np.uint32).astype(np.int64)
    N, P = codes.shape
    if packing == PACK_B3:
        per = B3_TRITS
        invalid = codes > B3_MAX
        digits = np.empty((N, P, per), dtype=np.int64)
        v = codes.copy()
        for i in range(per):
            digits[:, :, i] = v % 3
            v //= 3
    else:
        per = B2_TRITS
        digits = np.empty((N, P, per), dtype=np.int64)
        for i in range(per):
            digits[:, :, i] = (codes >> (2 * i)) & 3
        invalid = (digits == 3).any(axis=2)
    t = digits.reshape(N, P * per)[:, :K] - 1
    return t.astype(np.int8), int(invalid.sum())


# ----------------------------------------------------------------------------------------------
# Hadamard rotation   ([CC] §二 ①: weights rotated offline; a matching O(n log n) transform on
# the activations at inference undoes it)
# ----------------------------------------------------------------------------------------------

def hadamard(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix: H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]] (fp64, unnormalised)."""
    assert n >= 1 and n & (n - 1) == 0
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def block_fwht(x: np.ndarray, block: int = 128) -> np.ndarray:
    """x~[b, blk*block + r] = sum_c H[r, c] * x[b, blk*block + c] / sqrt(block)  (block 0 = identity).

    Written as the explicit matrix product with the Sylvester matrix; fp64 throughout.
    """
    x = np.asarray(x, dtype=np.float64)
    if block == 0:
        return x.copy()
    B, K = x.shape
    assert K % block == 0
    H = hadamard(block)
    xb = x.reshape(B, K // block, block)
    y = np.matmul(xb, H.T) / math.sqrt(block)
    return y.reshape(B, K)


# ----------------------------------------------------------------------------------------------
# Contraction   ([CC] §二 ②: 128 weights share one FP16 scale; [NX] §1.1: the product becomes
# sign tests and add/subtract; [CC] §二 ③: compute on the packed format)
# ----------------------------------------------------------------------------------------------

def dequant(trits: np.ndarray, scales: np.ndarray, group: int) -> np.ndarray:
    """Dense fp64 W[n, k] = s[n, k // group] * t[n, k]."""
    t = np.asarray(trits, dtype=np.float64)
    s = np.asarray(scales, dtype=np.float64)
    N, K = t.shape
    s_full = np.repeat(s, group, axis=1)[:, :K]
    return s_full * t


def ternary_linear(codes, scales, x, K: int, group: int, packing: int, fwht_block: int = 128):
    """y[b, n] = sum_k s[n, g(k)] * t[n, k] * x~[b, k]  with x~ = block_fwht(x).

    Steps in the pages' order: unpack the packed codes, apply the matching transform to the
    activations, contract.  Returns (y, A, n_invalid) with A[b, n] = sum_k |s t x~| (the scale of
    the tolerance |y_gpu - y| <= 1e-3 A + 1e-5) all in fp64.
    """
    t, n_invalid = unpack(codes, K, packing)
    W = dequant(t, scales, group)
    xt = block_fwht(np.asarray(x, dtype=np.float64), fwht_block)
    y = np.matmul(xt, W.T)
    A = np.matmul(np.abs(xt), np.abs(W).T)
    return y, A, n_invalid


# ----------------------------------------------------------------------------------------------
# MoE expert layer   ([TT] point 1: 256 routed experts, 8 active per token, router gate at full
# precision; point 2: top-8 of 256)
# ----------------------------------------------------------------------------------------------

def moe_route(logits: np.ndarray, topk: int = 8):
    """Top-k experts per token by raw fp32 logit (ties: lower expert index first), and
    gate_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k chosen logits (fp64)."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, topk), dtype=np.int32)
    gate = np.empty((T, topk), dtype=np.float64)
    for t in range(T):
        order = np.argsort(-logits[t].astype(np.float64), kind="stable")  # stable: equal logits keep index order
        sel = order[:topk]
        idx[t] = sel
        l = logits[t, sel].astype(np.float64)
        e = np.exp(l - l.max())
        gate[t] = e / e.sum()
    return idx, gate


def silu(z):
    return z / (1.0 + np.exp(-z))


def moe_layer(logits, x, gu_codes, gu_scales, d_codes, d_scales, H: int, F: int, group: int,
              packing: int, topk: int = 8, fwht_block: int = 128, experts=None):
    """Routed SwiGLU expert layer.

    gu_codes [E, 2F, P_H] holds, per expert, the gate rows (0..F-1) then the up rows (F..2F-1),
    both with K = H; d_codes [E, H, P_F] is the down projection with K = F.  ``experts`` may be a
    dict e -> (gu_codes, gu_scales, d_codes, d_scales) overriding the stacked arrays (for sampling).

    Per token: route; x~ = FWHT(x); for each chosen expert e_j: g = W_g x~, u = W_u x~,
    h = silu(g) * u, h~ = FWHT(h), y_j = W_d h~;  y = sum_j gate_j y_j.
    Returns dict with idx, gate, h [T, k, F], y [T, H], and the tolerance scales.
    """
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    idx, gate = moe_route(logits, topk)
    xt = block_fwht(x, fwht_block)
    h = np.zeros((T, topk, F))
    g_all = np.zeros((T, topk, F))
    u_all = np.zeros((T, topk, F))
    A_g = np.zeros((T, topk, F))
    A_u = np.zeros((T, topk, F))
    y_parts = np.zeros((T, topk, H))
    A_d = np.zeros((T, topk, H))
    cache = {}
    for t in range(T):
        for j in range(topk):
            e = int(idx[t, j])
            if e not in cache:
                if experts is not None and e in experts:
                    gc, gs, dc, ds = experts[e]
                else:
                    gc, gs, dc, ds = gu_codes[e], gu_scales[e], d_codes[e], d_scales[e]
                tg, _ = unpack(gc, H, packing)
                td, _ = unpack(dc, F, packing)
                cache[e] = (dequant(tg, gs, group), dequant(td, ds, group))
            Wgu, Wd = cache[e]
            gu = Wgu @ xt[t]
            Agu = np.abs(Wgu) @ np.abs(xt[t])
            g_all[t, j], u_all[t, j] = gu[:F], gu[F:]
            A_g[t, j], A_u[t, j] = Agu[:F], Agu[F:]
            h[t, j] = silu(gu[:F]) * gu[F:]
    ht = block_fwht(h.reshape(T * topk, F), fwht_block).reshape(T, topk, F)
    for t in range(T):
        for j in range(topk):
            Wd = cache[int(idx[t, j])][1]
            y_parts[t, j] = Wd @ ht[t, j]
            A_d[t, j] = np.abs(Wd) @ np.abs(ht[t, j])
    y = np.einsum("tj,tjh->th", gate, y_parts)
    return dict(idx=idx, gate=gate, g=g_all, u=u_all, A_g=A_g, A_u=A_u, h=h, h_t=ht,
                y_parts=y_parts, A_d=A_d, y=y)


def moe_down_from_h(h, idx, gate, experts_down: dict, F: int, group: int, packing: int, fwht_block: int = 128):
    """Down projection + combine from a given h [T, k, F] (used to check the down stage on the GPU's
    own h).  experts_down maps e -> (d_codes [H, P_F], d_scales)."""
    h = np.asarray(h, dtype=np.float64)
    T, k, _ = h.shape
    ht = block_fwht(h.reshape(T * k, F), fwht_block).reshape(T, k, F)
    y = None
    A = None
    for t in range(T):
        for j in range(k):
            dc, ds = experts_down[int(idx[t, j])]
            td, _ = unpack(dc, F, packing)
            Wd = dequant(td, ds, group)
            part = Wd @ ht[t, j]
            Apart = np.abs(Wd) @ np.abs(ht[t, j])
            if y is None:
                y = np.zeros((T, part.shape[0]))
                A = np.zeros((T, part.shape[0]))
            y[t] += gate[t, j] * part
            A[t] += gate[t, j] * Apart
    return y, A


# ----------------------------------------------------------------------------------------------
# Offline quantizer   ([CC] §二 ①: rotate the weights by a Hadamard transform before compressing;
# §二 ②: each group of 128 weights shares one FP16 scale; 一: three levels -1, 0, +1, the scale
# restoring the magnitude)
# ----------------------------------------------------------------------------------------------

INV_SQRT128 = math.sqrt(2.0) / 16.0   # 2^-3.5, rounded once to fp64


def quantize(W, group: int, packing: int, fwht_block: int = 128):
    """Dense W [N, K] (bf16 values, given as any float array) -> (codes, fp16 scales, int8 trits).

    1. Rotate each row block by block (same transform as the activations'): u = W_blk @ H^T with the
       unnormalised Sylvester H, in fp64; the rotated weight is w' = u * c with c = 2^-3.5
       (fwht_block 0: u = W, c = 1).  For bf16 input u is exact in fp64 whenever the magnitudes in
       one block span less than 2^38, and so are the group sums below when they span less than 2^31.
    2. Per group of ``group`` consecutive k: m = sum |u| / group, scale S = fp16(m * c) (the product
       rounded to fp64 once, then to fp16 to nearest even).
    3. t = sign(u) where fp64(|u| * c) > S / 2, else 0: the nearest of S * {-1, 0, +1} to w'
       (absmean rule), a value exactly halfway between 0 and S going to 0.
    4. Pack t (base-3 or 2-bit, as ``pack``).
    """
    W = np.asarray(W, dtype=np.float64)
    N, K = W.shape
    assert K % 128 == 0 and group in (64, 128) and fwht_block in (0, 128)
    if fwht_block:
        H = hadamard(fwht_block)
        u = np.matmul(W.reshape(N, K // fwht_block, fwht_block), H.T).reshape(N, K)
        c = INV_SQRT128
    else:
        u = W.copy()
        c = 1.0
    m = np.abs(u).reshape(N, K // group, group).sum(axis=2) / group
    scales = (m * c).astype(np.float16)
    half = np.repeat(scales.astype(np.float64) / 2.0, group, axis=1)
    trits = np.where(np.abs(u) * c > half, np.sign(u), 0.0).astype(np.int8)
    return pack(trits, packing), scales, trits


# ----------------------------------------------------------------------------------------------
# FP8 prefill variant.  No passage states it: it is this build's variant of the batched contraction
# ([CC] §二 ③ computes on the packed format; the FP8 operand type is the reading).  Each activation
# row and each weight row is brought to FP8 E4M3 under its own power-of-two factor; the tolerance
# against the exact result is the variant's own, stated with the GPU test.
# ----------------------------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3(v):
    """Nearest FP8 E4M3 value (4 exponent bits with bias 7, 3 mantissa bits, subnormals m * 2^-9,
    largest finite 448, no infinities), ties to the even mantissa; magnitudes that round above 448
    give 448.  fp64 in, fp64 out."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))       # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    E = np.maximum(ex - 1, -6)                      # binade; below 2^-6 the subnormal spacing 2^-9
    step = np.ldexp(1.0, E - 3)                     # grid spacing: 3 mantissa bits
    q = np.minimum(np.round(a / step) * step, E4M3_MAX)   # np.round: half to even
    return np.copysign(q, v)


def pow2_exponent(m):
    """e = floor(log2 m) - 7 for m > 0, so that m * 2^-e lies in [128, 256); 0 for m = 0."""
    m = np.asarray(m, dtype=np.float64)
    _, ex = np.frexp(np.where(m > 0, m, 1.0))
    return np.where(m > 0, ex - 1 - 7, 0).astype(np.int64)


def linear_fp8(codes, scales, x, K: int, group: int, packing: int, fwht_block: int = 128):
    """The contraction with FP8 E4M3 operands:

        y[b, n] = 2^(ea_b + eb_n) * sum_k e4m3(x~[b, k] * 2^-ea_b) * e4m3(s[n, g(k)] t[n, k] * 2^-eb_n)

    with ea_b = pow2_exponent(max_k |x~[b, k]|) and eb_n = pow2_exponent(max_g |s[n, g]|) (over the
    row's scales).  Products of E4M3 values and their sums are exact in fp64 at these sizes, so y is
    the exact value of the quantised operands' contraction.  Returns (y, A, n_invalid) with A the
    exact operands' sum_k |s t x~| (as ``ternary_linear``)."""
    t, n_invalid = unpack(codes, K, packing)
    W = dequant(t, scales, group)
    xt = block_fwht(np.asarray(x, dtype=np.float64), fwht_block)
    ea = pow2_exponent(np.abs(xt).max(axis=1))
    eb = pow2_exponent(np.abs(np.asarray(scales, dtype=np.float64)).max(axis=1))
    aq = e4m3(xt * np.ldexp(1.0, -ea)[:, None])
    wq = e4m3(W * np.ldexp(1.0, -eb)[:, None])
    y = np.matmul(aq, wq.T) * np.ldexp(1.0, ea[:, None] + eb[None, :])
    A = np.matmul(np.abs(xt), np.abs(W).T)
    return y, A, n_invalid
