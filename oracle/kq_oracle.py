"""CPU oracle for the k-quant weight matmul Y = dequant(W) . X.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares no
code with the CUDA library (no kernels, headers, helpers or tables); the only
thing the two sides have in common is the seeded input generator, which holds
none of the method's arithmetic.

Everything here is written as the plain definition, in numpy, so that a reader
can check it against the pages by eye:

* block formats are decoded field by field from raw bytes,
* weights are dequantised to fp64,
* activations are quantised to Q8_1 in fp32 exactly as the pages' quantiser does
  (the integer codes are decided in fp32 on both sides),
* the product is a plain fp64 matmul (a library primitive) of the dequantised
  operands, and the error bound Sum_k |w_k x_k| is a second fp64 matmul.

Sources (page title, section):

[MMVQ]  "06 · 8e/8e② — decode MMVQ: dp4a integer dot products + the llama.cpp
        launch table": §2 Principle (value of a Q4_K weight, the min-term
        identity, the activation quantiser), §3.2 Key code (``q4_k_q8_mmvq``
        byte offsets and nibble halves; ``quantize_pad40_block``), §3.3
        Pitfalls (Q6_K: ql[128] + qh[64] + scales[16], then fp16 d at byte 208).
[MMQv2] "ZINC MMQ v2 — Fused Q4_K×Q8_1 Tensor-Core GEMM (beat llama.cpp)":
        What they do right (Q8_1 activations, 1 byte per element), MoE routing
        (fused gather), Correctness gate (CPU dequant + matmul reference).
[GAP]   "Prefill Gap Closure Plan — ZINC CUDA vs llama.cpp": T2 (gather by
        expert: histogram, prefix sum, scatter of token-slot ids; "scatter
        back" to the tokens).

Where the pages leave a step open, the reading taken is stated at the function.
The bit layouts the pages elide (the Q4_K 6-bit scale/min packing, the Q6_K
ql/qh bit arrangement and the whole Q5_K block) follow the GGUF k-quant
layout; their agreement with GGUF files is "parity unpinned" (no GGUF file is
available to check against); every other function here is pinned by
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
Q4_K_BYTES = 144
Q6_K_BYTES = 210
Q5_K_BYTES = 176
QK8_1 = 32
Q8_1_BYTES = 36


# ----------------------------------------------------------------------------
# fp16 fields
# ----------------------------------------------------------------------------
def fp16_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) -> exact fp64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f32_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 values -> binary16 bit patterns, round to nearest, ties to even."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


# ----------------------------------------------------------------------------
# Q4_K
# ----------------------------------------------------------------------------
def q4_k_scale_min(scales: np.ndarray):
    """Unpack the eight 6-bit (scale, min) pairs of a Q4_K super-block.

    ``scales``: uint8 [..., 12], the bytes at offset 4 of each block. The page
    names this unpacking (``get_scale_min_k4``) but elides its body ([MMVQ]
    §3.2); the reading taken is the GGUF k-quant packing:

      sub-block j < 4 : sc = S[j] & 63,            m = S[j+4] & 63
      sub-block j >= 4: sc = (S[j+4] & 15) | (S[j-4] >> 6) << 4
                        m  = (S[j+4] >> 4) | (S[j]   >> 6) << 4

    Returns int64 arrays (sc, m) of shape [..., 8].
    """
    S = scales.astype(np.int64)
    sc = np.empty(S.shape[:-1] + (8,), dtype=np.int64)
    m = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = S[..., j] & 63
        m[..., j] = S[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (S[..., j + 4] & 15) | ((S[..., j - 4] >> 6) << 4)
        m[..., j] = (S[..., j + 4] >> 4) | ((S[..., j] >> 6) << 4)
    return sc, m


def q4_k_fields(blocks: np.ndarray):
    """Decode Q4_K super-blocks ([MMVQ] §3.2 ``q4_k_q8_mmvq``).

    ``blocks``: uint8 [..., 144]. Byte 0: fp16 d; byte 2: fp16 dmin; bytes 4..15:
    packed 6-bit scales and mins; bytes 16..143: ``qs``. Sub-block j (32 weights)
    reads the 32 bytes ``qs[32*(j>>1) : 32*(j>>1)+32]``: the low nibble when j is
    even, the high nibble when j is odd.

    Returns (d [...], dmin [...], sc [..., 8], m [..., 8], nib [..., 8, 32]).
    """
    blocks = np.asarray(blocks, dtype=np.uint8)
    d = fp16_to_f64(blocks[..., 0:2].copy().view(np.uint16)[..., 0])
    dmin = fp16_to_f64(blocks[..., 2:4].copy().view(np.uint16)[..., 0])
    sc, m = q4_k_scale_min(blocks[..., 4:16])
    qs = blocks[..., 16:144].astype(np.int64)
    nib = np.empty(blocks.shape[:-1] + (8, 32), dtype=np.int64)
    for j in range(8):
        chunk = qs[..., 32 * (j >> 1): 32 * (j >> 1) + 32]
        nib[..., j, :] = (chunk & 15) if j % 2 == 0 else (chunk >> 4)
    return d, dmin, sc, m, nib


def q4_k_dequant(W: np.ndarray, K: int) -> np.ndarray:
    """Dequantise a row-major Q4_K matrix to fp64 [M, K].

    Each weight is d*sc*nib - dmin*m ([MMVQ] §2: "a Q4_K dequantized value =
    d·s·nib − dm·m"), with the fp16 fields widened exactly."""
    W = np.asarray(W, dtype=np.uint8)
    M = W.shape[0]
    nb = K // QK_K
    blocks = W.reshape(M, nb, Q4_K_BYTES)
    d, dmin, sc, m, nib = q4_k_fields(blocks)
    w = (d[..., None, None] * sc[..., None] * nib
         - (dmin[..., None] * m)[..., None])
    return w.reshape(M, K)


# ----------------------------------------------------------------------------
# Q6_K
# ----------------------------------------------------------------------------
def q6_k_fields(blocks: np.ndarray):
    """Decode Q6_K super-blocks.

    ``blocks``: uint8 [..., 210]: ``ql[128]`` at byte 0 (low 4 bits of each
    code), ``qh[64]`` at byte 128 (high 2 bits), int8 ``scales[16]`` at byte 192
    (one per 16 weights), fp16 ``d`` at byte 208 ([MMVQ] §3.3 Pitfalls).

    The pages give only the field sizes; the bit arrangement taken is the GGUF
    one. For half h in {0,1}, quarter g in {0..3} and r in {0..31}, weight
    e = 128h + 32g + r has
      low 4 bits : g=0 low nibble of ql[64h + r],  g=1 low nibble of ql[64h+32+r],
                   g=2 high nibble of ql[64h + r], g=3 high nibble of ql[64h+32+r]
      high 2 bits: bits 2g..2g+1 of qh[32h + r]
      scale      : scales[e // 16]

    Returns (d [...], sc [..., 16], q [..., 256]) with q in [0, 63].
    """
    blocks = np.asarray(blocks, dtype=np.uint8)
    ql = blocks[..., 0:128].astype(np.int64)
    qh = blocks[..., 128:192].astype(np.int64)
    sc = blocks[..., 192:208].view(np.int8).astype(np.int64)
    d = fp16_to_f64(blocks[..., 208:210].copy().view(np.uint16)[..., 0])
    q = np.empty(blocks.shape[:-1] + (256,), dtype=np.int64)
    for h in range(2):
        for g in range(4):
            src = ql[..., 64 * h + 32 * (g & 1): 64 * h + 32 * (g & 1) + 32]
            low = (src & 15) if g < 2 else (src >> 4)
            high = (qh[..., 32 * h: 32 * h + 32] >> (2 * g)) & 3
            q[..., 128 * h + 32 * g: 128 * h + 32 * g + 32] = low | (high << 4)
    return d, sc, q


def q6_k_dequant(W: np.ndarray, K: int) -> np.ndarray:
    """Dequantise a row-major Q6_K matrix to fp64 [M, K]: d*sc*(q-32)."""
    W = np.asarray(W, dtype=np.uint8)
    M = W.shape[0]
    nb = K // QK_K
    blocks = W.reshape(M, nb, Q6_K_BYTES)
    d, sc, q = q6_k_fields(blocks)
    scale = np.repeat(sc, 16, axis=-1)                       # [M, nb, 256]
    w = d[..., None] * scale * (q - 32)
    return w.reshape(M, K)


# ----------------------------------------------------------------------------
# Q5_K
# ----------------------------------------------------------------------------
def q5_k_fields(blocks: np.ndarray):
    """Decode Q5_K super-blocks.

    The pages name Q5_K only as a sibling of the Q4_K and Q6_K decode kernels,
    with its own unpacking and no layout ([MMVQ] §3.2 "one kernel per type";
    the Q4_K value d·s·nib − dm·m of §2 with a fifth bit). The reading taken is
    the GGUF Q5_K block, 176 bytes: fp16 d at byte 0, fp16 dmin at byte 2, the
    Q4_K 6-bit scale/min packing at bytes 4..15, ``qh[32]`` at byte 16,
    ``qs[128]`` at byte 48. Sub-block j (32 weights) takes its low four bits
    like Q4_K (low nibbles of ``qs[32*(j>>1) : +32]`` for even j, high nibbles
    for odd j) and weight r of the sub-block its fifth bit from bit j of
    ``qh[r]``. Agreement with GGUF files is parity unpinned (no file here).

    Returns (d [...], dmin [...], sc [..., 8], m [..., 8], q [..., 8, 32]), q in [0, 31].
    """
    blocks = np.asarray(blocks, dtype=np.uint8)
    d = fp16_to_f64(blocks[..., 0:2].copy().view(np.uint16)[..., 0])
    dmin = fp16_to_f64(blocks[..., 2:4].copy().view(np.uint16)[..., 0])
    sc, m = q4_k_scale_min(blocks[..., 4:16])
    qh = blocks[..., 16:48].astype(np.int64)
    qs = blocks[..., 48:176].astype(np.int64)
    q = np.empty(blocks.shape[:-1] + (8, 32), dtype=np.int64)
    for j in range(8):
        chunk = qs[..., 32 * (j >> 1): 32 * (j >> 1) + 32]
        low = (chunk & 15) if j % 2 == 0 else (chunk >> 4)
        q[..., j, :] = low | (((qh >> j) & 1) << 4)
    return d, dmin, sc, m, q


def q5_k_dequant(W: np.ndarray, K: int) -> np.ndarray:
    """Dequantise a row-major Q5_K matrix to fp64 [M, K]: d*sc*q - dmin*m."""
    W = np.asarray(W, dtype=np.uint8)
    M = W.shape[0]
    nb = K // QK_K
    d, dmin, sc, m, q = q5_k_fields(W.reshape(M, nb, Q5_K_BYTES))
    w = (d[..., None, None] * sc[..., None] * q
         - (dmin[..., None] * m)[..., None])
    return w.reshape(M, K)


def dequant(wtype: str, W: np.ndarray, K: int) -> np.ndarray:
    if wtype == "q5_k":
        return q5_k_dequant(W, K)
    if wtype == "q4_k":
        return q4_k_dequant(W, K)
    if wtype == "q6_k":
        return q6_k_dequant(W, K)
    raise ValueError(wtype)


# ----------------------------------------------------------------------------
# Q8_1 activation quantisation
# ----------------------------------------------------------------------------
def quantize_q8_1(X: np.ndarray):
    """Quantise fp32 activations to Q8_1 blocks of 32.

    Follows the quantiser of [MMVQ] §2 and §3.2 (``quantize_pad40_block``), in
    fp32, step by step:
      amax = max |x| over the block
      d    = amax / 127                 (fp32 division)
      di   = 1 / d if d != 0 else 0     (fp32 division; also 0 where 1 / d
                                         overflows fp32, see below)
      q    = clamp(rint(x * di), -128, 127)   (fp32 product, ties to even)
      d_h  = fp16(d)                    (stored scale, round to nearest even)
    plus the block sum of the Q8_1 format, s = d * Sum(q) ([MMQv2]: Q8_1
    carries the sum used by the min term). Reading taken for the open point of
    which d multiplies Sum(q): the stored d_h, so that s is the sum of the
    block's dequantised activations; d_h * Sum(q) is exact in fp32 (11-bit by
    at most 13-bit integers) and is rounded once to fp16. Reading taken where
    the pages' formula has no finite value: when amax is below about 3.7e-37,
    1 / d overflows fp32 and x * di would be infinite or NaN; d_h = fp16(d) is
    0 there, so the block's dequantised values are 0 whatever its codes, and
    the codes are taken as 0 (di = 0), as for amax = 0.

    ``X``: fp32 [N, K] token-major, K % 32 == 0.
    Returns (q int8 [N, K/32, 32], d_h uint16 [N, K/32], s_h uint16 [N, K/32]).
    """
    X = np.asarray(X, dtype=np.float32)
    N, K = X.shape
    if K % QK8_1:
        raise ValueError("K must be a multiple of 32")
    xb = X.reshape(N, K // QK8_1, QK8_1)
    amax = np.max(np.abs(xb), axis=-1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    di = np.zeros_like(d)
    with np.errstate(over="ignore", divide="ignore"):
        np.divide(np.float32(1.0), d, out=di, where=(d != 0))
    di[~np.isfinite(di)] = 0
    prod = (xb * di[..., None]).astype(np.float32)
    q = np.clip(np.rint(prod), -128, 127).astype(np.int8)
    d_h = f32_to_fp16_bits(d)
    sumq = q.astype(np.int32).sum(axis=-1)
    s32 = (fp16_to_f64(d_h).astype(np.float32) * sumq.astype(np.float32)).astype(np.float32)
    s_h = f32_to_fp16_bits(s32)
    return q, d_h, s_h


def pack_q8_1(q: np.ndarray, d_h: np.ndarray, s_h: np.ndarray) -> np.ndarray:
    """Lay Q8_1 blocks out as bytes: [fp16 d][fp16 s][int8 q[32]] = 36 bytes.

    The pages show a 40-byte variant with a pad and an int32 sum; the Q8_1 byte
    layout taken here keeps "1 byte per element" plus the two fp16 fields, with
    the int8 payload 4-byte aligned. Returns uint8 [N, K/32, 36]."""
    N, nb, _ = q.shape
    out = np.empty((N, nb, Q8_1_BYTES), dtype=np.uint8)
    out[..., 0:2] = np.asarray(d_h, dtype=np.uint16)[..., None].view(np.uint8).reshape(N, nb, 2)
    out[..., 2:4] = np.asarray(s_h, dtype=np.uint16)[..., None].view(np.uint8).reshape(N, nb, 2)
    out[..., 4:36] = q.view(np.uint8)
    return out


def q8_1_dequant(q: np.ndarray, d_h: np.ndarray) -> np.ndarray:
    """x_hat = d_h * q in fp64, shape [N, K]."""
    N, nb, _ = q.shape
    return (fp16_to_f64(d_h)[..., None] * q.astype(np.float64)).reshape(N, nb * QK8_1)


# ----------------------------------------------------------------------------
# Matmul
# ----------------------------------------------------------------------------
def matmul(wtype: str, W: np.ndarray, X: np.ndarray, M: int, K: int):
    """Reference Y = dequant(W) . x_hat for every token, in fp64.

    ``W``: raw row-major blocks [M, ...]; ``X``: fp32 [N, K] token-major.
    The activations are quantised to Q8_1 first (the fused step of every path),
    then Y[n, m] = Sum_k w[m, k] * x_hat[n, k] ([MMQv2] Correctness gate: CPU
    dequant + matmul). Also returns the per-element error scale
    B[n, m] = Sum_k |w[m, k] * x_hat[n, k]|.

    Returns (Y fp64 [N, M], B fp64 [N, M]) with M contiguous per token.
    """
    w = dequant(wtype, W, K)
    assert w.shape == (M, K)
    q, d_h, _ = quantize_q8_1(X)
    xh = q8_1_dequant(q, d_h)
    Y = xh @ w.T
    B = np.abs(xh) @ np.abs(w).T
    return Y, B


def matmul_rows(wtype: str, W: np.ndarray, X: np.ndarray, K: int, rows: np.ndarray):
    """The same as ``matmul`` restricted to the weight rows in ``rows`` (used
    to check sampled outputs of full-size problems)."""
    w = dequant(wtype, np.asarray(W)[rows], K)
    q, d_h, _ = quantize_q8_1(X)
    xh = q8_1_dequant(q, d_h)
    return xh @ w.T, np.abs(xh) @ np.abs(w).T


def q4_k_min_term_matvec(W: np.ndarray, x: np.ndarray, K: int) -> np.ndarray:
    """Q4_K matvec by the min-term identity of [MMVQ] §2:

      W.x = Sum over sub-blocks [ d*sc * Sum(nib * q) * d8 - dmin*m * d8 * Sum(q) ]

    with the integer dot products taken exactly in int64 and the combination
    in fp64. This is a second formulation of the same product, used to check
    the plain one. ``x``: fp32 [K]. Returns fp64 [M]."""
    W = np.asarray(W, dtype=np.uint8)
    M = W.shape[0]
    nb = K // QK_K
    d, dmin, sc, m, nib = q4_k_fields(W.reshape(M, nb, Q4_K_BYTES))
    q, d_h, _ = quantize_q8_1(np.asarray(x, dtype=np.float32).reshape(1, K))
    q = q.reshape(nb, 8, 32).astype(np.int64)
    d8 = fp16_to_f64(d_h).reshape(nb, 8)
    dot = np.einsum("mbjk,bjk->mbj", nib, q)              # exact int64
    sq = q.sum(axis=-1)                                    # [nb, 8]
    terms = (d[..., None] * sc * dot - dmin[..., None] * m * sq[None]) * d8[None]
    return terms.sum(axis=(1, 2))


# ----------------------------------------------------------------------------
# MoE
# ----------------------------------------------------------------------------
def moe_buckets(expert_ids: np.ndarray, n_experts: int):
    """Group the (token, slot) pairs by expert ([GAP] T2 step 1: histogram ->
    prefix-sum offsets -> scatter of token-slot ids into per-expert buckets).

    Within a bucket the pairs keep token order, then slot order.
    Returns (counts int64 [E], offsets int64 [E+1], entries int64 [T*top_k])
    where an entry is the flat slot index t*top_k + j."""
    ids = np.asarray(expert_ids).reshape(-1)
    if ids.size and (ids.min() < 0 or ids.max() >= n_experts):
        raise ValueError("expert id out of range")
    counts = np.bincount(ids, minlength=n_experts).astype(np.int64)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    entries = np.argsort(ids, kind="stable").astype(np.int64)
    return counts, offsets, entries


def moe(wtype: str, W_experts: np.ndarray, expert_ids: np.ndarray, X: np.ndarray,
        n_experts: int, M: int, K: int):
    """MoE expert matmul: for every token t and slot j,
    Y[t, j, :] = dequant(W_{ids[t, j]}) . x_hat_t ([MMQv2] MoE routing; [GAP]
    T2). No router-probability weighting and no sum over slots: the combine is
    the step after this one.

    ``W_experts``: [n_experts * M, ...] raw blocks, expert-major.
    Returns (Y fp64 [T, top_k, M], B fp64 [T, top_k, M])."""
    ids = np.asarray(expert_ids)
    T, top_k = ids.shape
    q, d_h, _ = quantize_q8_1(X)
    xh = q8_1_dequant(q, d_h)
    Y = np.zeros((T, top_k, M))
    B = np.zeros((T, top_k, M))
    Wr = np.asarray(W_experts).reshape(n_experts, M, -1)
    for e in range(n_experts):
        t_idx, j_idx = np.nonzero(ids == e)
        if t_idx.size == 0:
            continue
        w = dequant(wtype, Wr[e], K)
        Y[t_idx, j_idx] = xh[t_idx] @ w.T
        B[t_idx, j_idx] = np.abs(xh[t_idx]) @ np.abs(w).T
    return Y, B


# ----------------------------------------------------------------------------
# The steps next to the matmul: the producer of the activations before it and
# the MoE combine after it
# ----------------------------------------------------------------------------
def rms_norm(X: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of every token row, the producer whose output the activation
    quantiser takes when it is fused into it ([MMVQ] §3.2 Key code: the Q8_1
    quantisation body moved into the RMSNorm and SwiGLU producers). The pages
    name the producer without its formula; the reading taken is the usual one,
    x / sqrt(mean(x^2) + eps) * gamma, in fp64.

    ``X``: [N, K]; ``gamma``: [K]. Returns fp64 [N, K]."""
    X = np.asarray(X, dtype=np.float64)
    ms = np.mean(X * X, axis=1, keepdims=True)
    return X / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)[None, :]


def swiglu(G: np.ndarray, U: np.ndarray) -> np.ndarray:
    """SwiGLU, the other producer named in [MMVQ] §3.2 Key code; reading taken:
    silu(g) * u with silu(g) = g / (1 + exp(-g)), element-wise in fp64."""
    G = np.asarray(G, dtype=np.float64)
    return G / (1.0 + np.exp(-G)) * np.asarray(U, dtype=np.float64)


def matmul_from(wtype: str, W: np.ndarray, Xp: np.ndarray, M: int, K: int):
    """``matmul`` for activations made by a producer (``rms_norm``, ``swiglu``):
    they are rounded to fp32 (the precision the quantiser receives them in),
    then quantised to Q8_1 and multiplied as in ``matmul``."""
    return matmul(wtype, W, np.asarray(Xp, dtype=np.float32), M, K)


def moe_combine(Y: np.ndarray, probs: np.ndarray) -> np.ndarray:
    """The step after the expert matmul: the slots' rows go back to their token
    ([GAP] T2, "scatter back"), read as the usual MoE combine weighted by the
    router probabilities: out[t, :] = Sum_j probs[t, j] * Y[t, j, :], in fp64.
    The probabilities are inputs (no normalisation here).

    ``Y``: [T, top_k, M]; ``probs``: [T, top_k]. Returns fp64 [T, M]."""
    return np.einsum("tj,tjm->tm", np.asarray(probs, dtype=np.float64), np.asarray(Y, dtype=np.float64))


def tolerance(B: np.ndarray) -> np.ndarray:
    """Per-element acceptance bound |y_gpu - y_ref| <= 1e-3 * B + 1e-5."""
    return 1e-3 * B + 1e-5
