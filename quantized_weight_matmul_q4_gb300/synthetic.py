"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and places them at the byte offsets the
block formats define. It holds none of the method's arithmetic: no
dequantisation, no activation quantisation, no matmul. Both the CUDA path and
the CPU oracle receive exactly the arrays produced here.

Distributions follow the workloads of the k-quant matmul pages:

* Q4_K super-block (256 weights, 144 bytes): fp16 ``d`` and ``dmin`` drawn
  from |N(0, 0.01)|, 6-bit sub-block scales and mins uniform on [0, 63],
  nibbles uniform on [0, 15]. Because every one of those integer fields is
  uniform over all of its bits, the 12 packed scale bytes and the 128 nibble
  bytes are exactly uniform random bytes, so they are drawn as bytes and no
  packing code is needed. Layout per "06 · 8e/8e② — decode MMVQ" (§3.2, the
  ``q4_k_q8_mmvq`` listing): d at byte 0, dmin at byte 2, scales at byte 4,
  nibbles at byte 16.
* Q6_K super-block (256 weights, 210 bytes): ``ql[128]`` at byte 0, ``qh[64]``
  at byte 128 (6-bit codes uniform on [0, 63], hence uniform bytes), int8
  ``scales[16]`` uniform on [-64, 63] at byte 192 and fp16 ``d`` at byte 208
  (the generator bug described in "06 · 8e/8e②", §3.3 Pitfalls, put d at byte
  0; it sits at 208). ``d`` is drawn like the Q4_K ``d``.
* Q5_K super-block (256 weights, 176 bytes; the GGUF layout, which the pages
  do not give): fp16 ``d`` at byte 0 and ``dmin`` at byte 2 drawn like the Q4_K
  ones, then 12 bytes of packed 6-bit scales/mins, ``qh[32]`` and ``qs[128]``;
  every one of those fields is uniform over all its bits, so bytes 4..175 are
  uniform random bytes.
* TQ4_1S block (32 weights, 20 bytes; "TQ4_1S Weight Kernel Optimization",
  Block Layout): fp16 ``d0`` at byte 0 and ``d1`` at byte 2, each drawn as
  0.02 * exp(0.25 * N(0, 1)) (positive half-block scales of the size of a
  7B model's weights), then 16 bytes of 4-bit centroid indices, element j in
  byte j / 2 (low nibble for even j). The indices are floor(8 + 3 z) clipped to
  [0, 15] with z ~ N(0, 1): symmetric and bell-shaped like the occupancy of
  the Lloyd-Max cells of N(0, 1), without the centroid table.
* Activations X: fp32 N(0, 1), token-major (K contiguous per token).
* MoE routing: for every token, the top-k experts of softmax(N(0,1) logits),
  ordered by descending probability, ties to the lower expert index.
"""
from __future__ import annotations

import numpy as np

QK_K = 256            # weights per k-quant super-block
Q4_K_BYTES = 144      # bytes per Q4_K super-block
Q6_K_BYTES = 210      # bytes per Q6_K super-block
Q5_K_BYTES = 176      # bytes per Q5_K super-block
Q8_1_BYTES = 36       # bytes per 32-element Q8_1 activation block
QK_TQ = 32            # weights per TQ4_1S block
TQ4_1S_BYTES = 20     # bytes per TQ4_1S block
QK8_1 = 32            # activations per Q8_1 block


def rngs(seed: int, n: int = 3):
    """Independent PCG64 streams spawned from one seed, in the fixed order
    (weights, activations, routing logits)."""
    return [np.random.Generator(np.random.PCG64(s))
            for s in np.random.SeedSequence(seed).spawn(n)]


def _fp16_abs_normal(rng: np.random.Generator, shape, sigma: float = 0.01) -> np.ndarray:
    """|N(0, sigma)| drawn in fp64 and stored as fp16 bit patterns (uint16)."""
    v = np.abs(rng.standard_normal(shape)) * sigma
    return v.astype(np.float16).view(np.uint16)


def q4_k_weights(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """Random Q4_K matrix: uint8 array of shape [M, (K/256)*144], row-major."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK_K
    w = rng.integers(0, 256, size=(M, nb, Q4_K_BYTES), dtype=np.uint8)
    d = _fp16_abs_normal(rng, (M, nb))
    dmin = _fp16_abs_normal(rng, (M, nb))
    w[:, :, 0:2] = d[..., None].view(np.uint8).reshape(M, nb, 2)
    w[:, :, 2:4] = dmin[..., None].view(np.uint8).reshape(M, nb, 2)
    return w.reshape(M, nb * Q4_K_BYTES)


def q6_k_weights(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """Random Q6_K matrix: uint8 array of shape [M, (K/256)*210], row-major."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK_K
    w = rng.integers(0, 256, size=(M, nb, Q6_K_BYTES), dtype=np.uint8)
    sc = rng.integers(-64, 64, size=(M, nb, 16), dtype=np.int64).astype(np.int8)
    w[:, :, 192:208] = sc.view(np.uint8)
    d = _fp16_abs_normal(rng, (M, nb))
    w[:, :, 208:210] = d[..., None].view(np.uint8).reshape(M, nb, 2)
    return w.reshape(M, nb * Q6_K_BYTES)


def tq4_1s_weights(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """Random TQ4_1S matrix: uint8 array of shape [M, (K/32)*20], row-major."""
    if K % QK_TQ:
        raise ValueError("K must be a multiple of 32")
    nb = K // QK_TQ
    w = np.empty((M, nb, TQ4_1S_BYTES), dtype=np.uint8)
    d = (0.02 * np.exp(0.25 * rng.standard_normal((M, nb, 2)))).astype(np.float16)
    w[:, :, 0:4] = d.view(np.uint8).reshape(M, nb, 4)
    idx = np.clip(np.floor(8 + 3 * rng.standard_normal((M, nb, QK_TQ))), 0, 15).astype(np.uint8)
    w[:, :, 4:20] = idx[..., 0::2] | (idx[..., 1::2] << 4)
    return w.reshape(M, nb * TQ4_1S_BYTES)


def q5_k_weights(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """Random Q5_K matrix: uint8 array of shape [M, (K/256)*176], row-major."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK_K
    w = rng.integers(0, 256, size=(M, nb, Q5_K_BYTES), dtype=np.uint8)
    d = _fp16_abs_normal(rng, (M, nb))
    dmin = _fp16_abs_normal(rng, (M, nb))
    w[:, :, 0:2] = d[..., None].view(np.uint8).reshape(M, nb, 2)
    w[:, :, 2:4] = dmin[..., None].view(np.uint8).reshape(M, nb, 2)
    return w.reshape(M, nb * Q5_K_BYTES)


def weights(wtype: str, rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    if wtype == "q5_k":
        return q5_k_weights(rng, M, K)
    if wtype == "tq4_1s":
        return tq4_1s_weights(rng, M, K)
    if wtype == "q4_k":
        return q4_k_weights(rng, M, K)
    if wtype == "q6_k":
        return q6_k_weights(rng, M, K)
    raise ValueError(f"unknown weight type {wtype!r}")


def activations(rng: np.random.Generator, K: int, N: int) -> np.ndarray:
    """X ~ N(0, 1) as fp32, shape [N, K] (token-major: K contiguous per token)."""
    return rng.standard_normal((N, K), dtype=np.float32)


def expert_ids(rng: np.random.Generator, T: int, n_experts: int, top_k: int) -> np.ndarray:
    """Top-k experts of softmax(N(0,1) logits) per token, int32 [T, top_k].

    Slots are ordered by descending probability; equal probabilities go to the
    lower expert index (stable sort)."""
    logits = rng.standard_normal((T, n_experts))
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    p = z / z.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")
    return np.ascontiguousarray(order[:, :top_k].astype(np.int32))


# Seeded workloads with the shapes of the pages. Seeds: the 512x2048 matvec
# uses seed 0; the others use 1..6. The TQ4_1S shapes are the FFN matvecs of the
# 7B model the TQ4_1S page decodes (hidden 3584, intermediate 18944).
WORKLOADS = {
    "matvec_q4k_512x2048": dict(kind="matvec", wtype="q4_k", M=512, K=2048, N=1, seed=0),
    "decode_q4k_4096x11008": dict(kind="matvec", wtype="q4_k", M=4096, K=11008, N=1, seed=1),
    "decode_q4k_11008x4096": dict(kind="matvec", wtype="q4_k", M=11008, K=4096, N=1, seed=1),
    "decode_q5k_4096x11008": dict(kind="matvec", wtype="q5_k", M=4096, K=11008, N=1, seed=1),
    "decode_q5k_11008x4096": dict(kind="matvec", wtype="q5_k", M=11008, K=4096, N=1, seed=1),
    "decode_q6k_4096x11008": dict(kind="matvec", wtype="q6_k", M=4096, K=11008, N=1, seed=1),
    "decode_q6k_11008x4096": dict(kind="matvec", wtype="q6_k", M=11008, K=4096, N=1, seed=1),
    "decode_tq4_1s_18944x3584": dict(kind="matvec", wtype="tq4_1s", M=18944, K=3584, N=1, seed=6),
    "decode_tq4_1s_3584x18944": dict(kind="matvec", wtype="tq4_1s", M=3584, K=18944, N=1, seed=6),
    "smalln_q4k_4096x11008_n4": dict(kind="gemm", wtype="q4_k", M=4096, K=11008, N=4, seed=5),
    "prefill_q4k_4096x4096_n64": dict(kind="gemm", wtype="q4_k", M=4096, K=4096, N=64, seed=2),
    "prefill_q4k_4096x4096_n512": dict(kind="gemm", wtype="q4_k", M=4096, K=4096, N=512, seed=2),
    "prefill_q4k_14336x4096_n2048": dict(kind="gemm", wtype="q4_k", M=14336, K=4096, N=2048, seed=3),
    "prefill_q5k_14336x4096_n2048": dict(kind="gemm", wtype="q5_k", M=14336, K=4096, N=2048, seed=3),
    "prefill_q6k_4096x14336_n2048": dict(kind="gemm", wtype="q6_k", M=4096, K=14336, N=2048, seed=3),
    "moe_q4k_128x768x2048_t1024_top8": dict(kind="moe", wtype="q4_k", M=768, K=2048, T=1024,
                                           n_experts=128, top_k=8, seed=4),
    "moe_q6k_128x768x2048_t1024_top8": dict(kind="moe", wtype="q6_k", M=768, K=2048, T=1024,
                                           n_experts=128, top_k=8, seed=4),
}


def make_workload(name: str, copies: int = 1):
    """Build the named workload's inputs (numpy arrays).

    Returns a dict with ``W`` (a list of ``copies`` independent weight sets,
    each drawn from its own stream), ``X`` and, for MoE, ``ids``."""
    cfg = dict(WORKLOADS[name])
    r_w, r_x, r_ids = rngs(cfg["seed"])
    out = dict(cfg)
    if cfg["kind"] == "moe":
        E, M, K = cfg["n_experts"], cfg["M"], cfg["K"]
        wr = [np.random.Generator(np.random.PCG64(s)) for s in r_w.bit_generator.seed_seq.spawn(copies)]
        out["W"] = [weights(cfg["wtype"], r, E * M, K) for r in wr]
        out["X"] = activations(r_x, K, cfg["T"])
        out["ids"] = expert_ids(r_ids, cfg["T"], E, cfg["top_k"])
    else:
        wr = [np.random.Generator(np.random.PCG64(s)) for s in r_w.bit_generator.seed_seq.spawn(copies)]
        out["W"] = [weights(cfg["wtype"], r, cfg["M"], cfg["K"]) for r in wr]
        out["X"] = activations(r_x, cfg["K"], cfg["N"])
    return out
