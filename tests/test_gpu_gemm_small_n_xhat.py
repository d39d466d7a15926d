"""The tensor-core GEMM's activation operand, bit for bit, and small-N
prefill shapes against the oracle.

With the one-hot weights of tests/_onehot.py (code row k dequantises to the
unit vector e_k), output row k of every token is exactly that token's x_hat[k]
= fp16(d_h * q_k): one nonzero product in the fp32 accumulator, and a split-K
sum adds exact zeros to it. So the x_hat the GEMM multiplies (made from X by
quantize_xhat_kernel) is compared bit for bit with the oracle's Q8_1 codes and
scales ("06 · 8e/8e② — decode MMVQ", §2 Principle; "ZINC MMQ v2", What they do
right: Q8_1 activations), rounded to the fp16 operand the tensor cores take.
The small-N shapes (64-token tiles, split K, ragged token counts and a ragged
last row tile) are checked against the oracle within the per-element bound.
"""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_gemm, synthetic as syn
from _kqutil import assert_within_bound, to_dev
from _onehot import onehot_weights

pytestmark = pytest.mark.gpu


def _xhat_expected(X):
    q, d_h, _ = ora.quantize_q8_1(X)
    dh = np.asarray(d_h, dtype=np.uint16).view(np.float16).astype(np.float32)
    prod = dh[:, :, None] * q.astype(np.float32)        # exact: an fp16 value times an integer of at most 7 bits
    return prod.astype(np.float16).astype(np.float32).reshape(X.shape[0], -1)


def _tokens(K, N, seed):
    rng = np.random.default_rng(seed)
    X = syn.activations(rng, K, N)
    if N >= 4:
        X[1] = 0.0                                                  # an all-zero token
        X[2] *= np.repeat(np.exp(1.5 * rng.standard_normal(K // 32)), 32).astype(np.float32)  # mixed block scales (x_hat stays finite in fp16)
        X[3] = np.tile(np.arange(32, dtype=np.float32) - 15.5, K // 32)                  # halves: ties to even
    return X


@pytest.mark.parametrize("wtype,K,N", [
    ("q4_k", 1024, 64), ("q4_k", 1024, 17), ("q4_k", 4096, 8), ("q4_k", 4096, 64),
    ("q5_k", 1024, 64), ("q5_k", 4096, 33),
    ("q6_k", 4096, 64), ("q6_k", 4096, 5),   # Q6_K rows of K = 1024 are not 16-byte multiples
])
def test_in_kernel_xhat_is_exact(wtype, K, N):
    import torch
    W = onehot_weights(wtype, K)
    X = _tokens(K, N, K + N)
    Y = kq_gemm(wtype, to_dev(W, torch), to_dev(X, torch), W.shape[0], K).cpu().numpy()
    want = _xhat_expected(X)
    got = Y[:, :K]
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
        raise AssertionError(f"{wtype} K={K} N={N}: {bad.size} x_hat values differ; first flat index {bad[0]}: "
                             f"gpu={got.reshape(-1)[bad[0]]!r} want={want.reshape(-1)[bad[0]]!r}")


@pytest.mark.parametrize("wtype,M,K,N", [
    ("q4_k", 4096, 4096, 64),    # 32 row tiles, K split 4 ways
    ("q4_k", 300, 2048, 40),     # 3 row tiles (the last ragged), K split 8 ways
    ("q5_k", 1024, 512, 64),     # 8 row tiles, K split over its two super-blocks
    ("q6_k", 2048, 2048, 33),    # 16 row tiles, K split 8 ways
    ("q4_k", 14336, 4096, 64),   # 112 row tiles, K not split
    ("q6_k", 640, 2048, 9),      # 5 row tiles, K split 8 ways
])
def test_small_n_prefill_parity(wtype, M, K, N):
    import torch
    rng = np.random.default_rng(M + K + N)
    W = syn.weights(wtype, rng, M, K)
    X = syn.activations(rng, K, N)
    Y = kq_gemm(wtype, to_dev(W, torch), to_dev(X, torch), M, K).cpu().numpy()
    Yr, B = ora.matmul(wtype, W, X, M, K)
    assert_within_bound(Y, Yr, B, f"{wtype} {M}x{K}x{N}")


def test_small_n_prefill_deterministic():
    import torch
    rng = np.random.default_rng(5)
    M, K, N = 4096, 4096, 64
    Wd = to_dev(syn.q4_k_weights(rng, M, K), torch)
    Xd = to_dev(syn.activations(rng, K, N), torch)
    Y0 = kq_gemm("q4_k", Wd, Xd, M, K).cpu().numpy()
    for _ in range(3):
        assert np.array_equal(kq_gemm("q4_k", Wd, Xd, M, K).cpu().numpy(), Y0)
