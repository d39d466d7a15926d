"""Pins for the TQ4_1S oracle: each test ties it to something other than itself
(the Lloyd-Max conditions of N(0, 1), a library Hadamard matrix, a block
written out by hand, closed forms, brute force through the fast transform).

Source: "TQ4_1S Weight Kernel Optimization" (Architecture Overview, Block
Layout, Centroid Table).
"""
import math
import os

import numpy as np
import pytest

from oracle import tq4_oracle as tq
from quantized_weight_matmul_q4_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tq4_1s_block.txt")


def _block(d0: float, d1: float, idx) -> np.ndarray:
    """A block built from its fields by hand (little-endian fp16, two indices per byte)."""
    idx = np.asarray(idx, dtype=np.uint8)
    b = np.zeros(20, dtype=np.uint8)
    b[0:2] = np.array([d0], dtype=np.float16).view(np.uint8)
    b[2:4] = np.array([d1], dtype=np.float16).view(np.uint8)
    for j in range(16):
        b[4 + j] = idx[2 * j] | (idx[2 * j + 1] << 4)
    return b


def test_centroid_table_meets_lloyd_max_conditions_for_standard_normal():
    # Lloyd-Max for N(0,1): cell edges at the midpoints, each centroid the mean
    # of N(0,1) over its cell, (pdf(a) - pdf(b)) / (cdf(b) - cdf(a)). The table is
    # printed to 3 decimals, so it may be off by half a unit of the last digit.
    stats = pytest.importorskip("scipy.stats")
    c = tq.CENTROIDS
    assert c.shape == (16,) and np.all(np.diff(c) > 0)
    assert np.array_equal(c[::-1], -c)
    edges = np.concatenate([[-np.inf], (c[1:] + c[:-1]) / 2, [np.inf]])
    n = stats.norm
    mean = (n.pdf(edges[:-1]) - n.pdf(edges[1:])) / (n.cdf(edges[1:]) - n.cdf(edges[:-1]))
    assert np.max(np.abs(mean - c)) <= 5e-4


def test_wht_matrix_is_the_library_sylvester_hadamard():
    linalg = pytest.importorskip("scipy.linalg")
    H = tq.wht_matrix()
    assert np.array_equal(H * math.sqrt(32), linalg.hadamard(32).astype(np.float64))
    assert np.allclose(H @ H, np.eye(32), atol=1e-15)  # orthonormal and its own inverse


def test_golden_block_decodes_to_the_printed_values():
    lines = [ln for ln in open(GOLDEN) if not ln.startswith("#")]
    raw = np.array([int(t, 16) for t in lines[0].split(":")[1].split()], dtype=np.uint8)
    vals = np.array([float(t) for ln in lines[2:] for t in ln.split()])
    assert raw.shape == (20,) and vals.shape == (32,)
    got = tq.tq4_1s_dequant_rotated(raw.reshape(1, 20), 32)[0]
    assert np.allclose(got, vals, rtol=0, atol=1e-15)


@pytest.mark.parametrize("v", [0, 5, 8, 15])
def test_constant_block_has_one_nonzero_weight(v):
    # All 32 rotated values equal to c = centroid[v] * d: the block is c times
    # the all-ones vector, which the orthonormal WHT maps to c * sqrt(32) at
    # element 0 and zeros elsewhere.
    d = 0.75
    w = tq.tq4_1s_dequant(_block(d, d, [v] * 32).reshape(1, 20), 32)[0]
    want = np.zeros(32)
    want[0] = tq.CENTROIDS[v] * d * math.sqrt(32)
    assert np.allclose(w, want, rtol=0, atol=1e-12)


def test_two_scale_block_closed_form():
    # Rotated values c*d0 on elements 0..15 and c*d1 on 16..31: the inverse WHT
    # gives 16 (d0 + d1) c / sqrt(32) at element 0, 16 (d0 - d1) c / sqrt(32) at
    # element 16 (row 16 of H flips the sign of the upper half) and zeros elsewhere.
    d0, d1, v = 0.5, 0.125, 13
    c = tq.CENTROIDS[v]
    w = tq.tq4_1s_dequant(_block(d0, d1, [v] * 32).reshape(1, 20), 32)[0]
    want = np.zeros(32)
    want[0] = 16 * (d0 + d1) * c / math.sqrt(32)
    want[16] = 16 * (d0 - d1) * c / math.sqrt(32)
    assert np.allclose(w, want, rtol=0, atol=1e-12)


def _fwht(v):
    """In-place fast Walsh-Hadamard transform (butterflies, natural order), unnormalised."""
    v = list(v)
    h = 1
    while h < len(v):
        for i in range(0, len(v), 2 * h):
            for j in range(i, i + h):
                a, b = v[j], v[j + h]
                v[j], v[j + h] = a + b, a - b
        h *= 2
    return v


def test_brute_force_tiny_matvec():
    # Bytes -> values by explicit bit operations, the inverse rotation through
    # the fast transform, then the dot product, all in Python scalars.
    M, K = 3, 96
    rng = np.random.default_rng(11)
    W = syn.tq4_1s_weights(rng, M, K)
    x = syn.activations(rng, K, 1)[0]
    y = []
    for m in range(M):
        acc = 0.0
        for b in range(K // 32):
            blk = W[m, 20 * b:20 * b + 20]
            d0 = float(np.frombuffer(bytes(blk[0:2]), dtype="<f2")[0])
            d1 = float(np.frombuffer(bytes(blk[2:4]), dtype="<f2")[0])
            r = []
            for j in range(32):
                code = (int(blk[4 + j // 2]) >> (4 * (j % 2))) & 0xF
                r.append(float(tq.CENTROIDS[code]) * (d0 if j < 16 else d1))
            w = [t / math.sqrt(32) for t in _fwht(r)]
            acc += sum(w[i] * float(x[32 * b + i]) for i in range(32))
        y.append(acc)
    Y, B = tq.tq4_1s_matmul(W, x.reshape(1, K), M, K)
    assert np.allclose(Y[0], y, rtol=1e-13, atol=1e-15)


def test_plain_and_prerotated_forms_agree():
    # The page's fused form (rotate the activation, keep the weights rotated)
    # computes the same product as dequantise + inverse WHT + dot.
    M, K = 40, 1024
    rng = np.random.default_rng(3)
    W = syn.tq4_1s_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    Y, B = tq.tq4_1s_matmul(W, x, M, K)
    yf = tq.tq4_1s_rotated_matvec(W, x[0], K)
    assert np.allclose(Y[0], yf, rtol=0, atol=1e-12 * np.max(B))


def test_error_scale_bounds_both_sums():
    M, K = 16, 256
    rng = np.random.default_rng(4)
    W = syn.tq4_1s_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    _, B = tq.tq4_1s_matmul(W, x, M, K)
    w = tq.tq4_1s_dequant(W, K)
    plain = np.abs(w) @ np.abs(x[0].astype(np.float64))
    R = tq.tq4_1s_dequant_rotated(W, K).reshape(M, K // 32, 32)
    xr = x[0].astype(np.float64).reshape(K // 32, 32) @ tq.wht_matrix().T
    rotated = np.abs(np.einsum("mbj,bj->mbj", R, xr)).sum(axis=(1, 2))
    assert np.all(B[0] >= plain * (1 - 1e-12)) and np.all(B[0] >= rotated * (1 - 1e-12))


def test_planted_nibble_swap_is_caught_by_the_golden_block():
    # Reading the high nibble for even elements (a plausible slip) changes the
    # golden block's values, so the golden test above would fail on it.
    raw = np.array([int(t, 16) for t in open(GOLDEN).read().split("bytes:")[1].split("\n")[0].split()],
                   dtype=np.uint8)
    swapped = raw.copy()
    swapped[4:] = (raw[4:] >> 4) | ((raw[4:] & 0xF) << 4)
    a = tq.tq4_1s_dequant_rotated(raw.reshape(1, 20), 32)
    b = tq.tq4_1s_dequant_rotated(swapped.reshape(1, 20), 32)
    assert not np.allclose(a, b)
