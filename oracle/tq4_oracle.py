"""CPU oracle for the TQ4_1S weight matvec y = W . x.

TEST INFRASTRUCTURE ONLY, like ``kq_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` use it.
It shares no code, header, table or constant with the CUDA library; its
centroid table is typed here from the page, independently of the kernel's.

Source: [TQ] "TQ4_1S Weight Kernel Optimization" — Architecture Overview
(32-weight blocks, two half-block scales, WHT-rotated 4-bit Lloyd-Max codes,
dequant = centroid[index] * half-block scale followed by the inverse WHT, and
the fused form that pre-rotates the activation instead), Block Layout
(block_tq4_1s: fp16 d0 for elements 0..15, fp16 d1 for 16..31, 16 bytes of
indices, element j in byte j/2, low nibble for even j), Centroid Table.

Readings taken where the page leaves a step open (each one is pinned by
``tests/test_oracle_tq4.py``):

* The WHT is the 32-point Walsh-Hadamard transform of one block in natural
  (Sylvester) order, H[i, j] = (-1)^popcount(i & j) / sqrt(32): orthonormal,
  so it is a rotation, and symmetric, so it is its own inverse. The page names
  no random sign flips, so there are none.
* A TQ4_1S row holds the WHT-rotated weights: r_b = H w_b for each 32-block b,
  and the stored codes give r_b ~ centroid[idx] * d. The weights are therefore
  w_b = H^-1 r_b, and y = Sum_b w_b . x_b.

Everything is fp64, computed by the plain definition: decode the bytes,
dequantise the rotated block, undo the rotation, take the dot product. The
fused form of the page (rotate the activation once, then dot the rotated
weights against it) is a separate function, used only to check the identity.
"""
from __future__ import annotations

import numpy as np

QK_TQ = 32           # weights per TQ4_1S block
TQ4_1S_BYTES = 20    # bytes per block: two fp16 scales + 16 bytes of 4-bit indices

# [TQ] Centroid Table: the 16 Lloyd-Max values for N(0, 1), index order.
CENTROIDS = np.array([
    -2.733, -2.069, -1.618, -1.256, -0.942, -0.657, -0.388, -0.128,
    0.128, 0.388, 0.657, 0.942, 1.256, 1.618, 2.069, 2.733,
], dtype=np.float64)


def wht_matrix(n: int = QK_TQ) -> np.ndarray:
    """Orthonormal Walsh-Hadamard matrix in natural order, from its definition
    H[i, j] = (-1)^popcount(i & j) / sqrt(n) (n a power of two)."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    parity = np.vectorize(lambda v: bin(int(v)).count("1") & 1)(i & j)
    return np.where(parity == 1, -1.0, 1.0) / np.sqrt(n)


def tq4_1s_fields(blocks: np.ndarray):
    """Decode raw blocks [..., 20] (uint8) field by field ([TQ] Block Layout).

    Returns (d0, d1) as fp64 [...] and the centroid indices [..., 32] (int64),
    index j = (qs[j / 2] >> 4 * (j % 2)) & 0xF."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    d0 = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    d1 = blocks[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    qs = blocks[..., 4:20].astype(np.int64)
    idx = np.empty(blocks.shape[:-1] + (QK_TQ,), dtype=np.int64)
    idx[..., 0::2] = qs & 0xF
    idx[..., 1::2] = qs >> 4
    return d0, d1, idx


def tq4_1s_dequant_rotated(W: np.ndarray, K: int) -> np.ndarray:
    """Rotated-space weights R [M, K] (fp64): centroid[idx] times the scale of
    the element's half block, d0 for elements 0..15, d1 for 16..31."""
    W = np.asarray(W, dtype=np.uint8)
    M = W.shape[0]
    nb = K // QK_TQ
    d0, d1, idx = tq4_1s_fields(W.reshape(M, nb, TQ4_1S_BYTES))
    scale = np.concatenate([np.repeat(d0[..., None], 16, axis=-1), np.repeat(d1[..., None], 16, axis=-1)], axis=-1)
    return (CENTROIDS[idx] * scale).reshape(M, K)


def tq4_1s_dequant(W: np.ndarray, K: int) -> np.ndarray:
    """Weights in the original space [M, K] (fp64): each block's rotated
    values through the inverse WHT, w_b = H^-1 r_b (H orthogonal: H^-1 = H^T)."""
    R = tq4_1s_dequant_rotated(W, K)
    M = R.shape[0]
    H_inv = wht_matrix().T
    return np.einsum("ij,mbj->mbi", H_inv, R.reshape(M, K // QK_TQ, QK_TQ)).reshape(M, K)


def tq4_1s_matmul(W: np.ndarray, X: np.ndarray, M: int, K: int):
    """Reference Y[n, m] = Sum_k w[m, k] x[n, k] with w = tq4_1s_dequant(W).

    ``X``: fp32 [N, K], taken exactly. Also returns the error scale
    B[n, m] = Sum_b Sum_j Sum_k |r[m, b, j] H[j, k] x[n, b, k]|, the sum of the
    absolute values of every term of the rotated bilinear form; it bounds both
    Sum_k |w x| and Sum_j |r (H x)|, whichever form a kernel adds up.

    Returns (Y fp64 [N, M], B fp64 [N, M])."""
    w = tq4_1s_dequant(W, K)
    assert w.shape == (M, K)
    X = np.asarray(X, dtype=np.float32).astype(np.float64).reshape(-1, K)
    Y = X @ w.T
    R = np.abs(tq4_1s_dequant_rotated(W, K)).reshape(M, K // QK_TQ, QK_TQ)
    xl1 = np.abs(X).reshape(X.shape[0], K // QK_TQ, QK_TQ).sum(axis=-1) / np.sqrt(QK_TQ)  # |H| |x_b| per element
    B = np.einsum("mbj,nb->nm", R, xl1)
    return Y, B


def tq4_1s_matmul_rows(W: np.ndarray, X: np.ndarray, K: int, rows: np.ndarray):
    """``tq4_1s_matmul`` restricted to the weight rows in ``rows``."""
    Wr = np.asarray(W)[rows]
    return tq4_1s_matmul(Wr, X, Wr.shape[0], K)


def tq4_1s_rotated_matvec(W: np.ndarray, x: np.ndarray, K: int) -> np.ndarray:
    """The fused form of [TQ] Architecture Overview: rotate the activation once
    per block (x_r = H x_b, the forward WHT), then y = Sum_b r_b . x_r with the
    rotated weights as stored. A second formulation of the same product, used
    to check the plain one. ``x``: fp32 [K]. Returns fp64 [M]."""
    R = tq4_1s_dequant_rotated(W, K)
    M = R.shape[0]
    xb = np.asarray(x, dtype=np.float32).astype(np.float64).reshape(K // QK_TQ, QK_TQ)
    xr = xb @ wht_matrix().T
    return np.einsum("mbj,bj->m", R.reshape(M, K // QK_TQ, QK_TQ), xr)
