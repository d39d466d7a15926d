"""Small-N decode (2 to 16 tokens at once) against the oracle, element by
element, within |y - y_ref| <= 1e-3 * Sum_k |w_k x_k| + 1e-5. Through the
public GEMM entry point: Q4_K and Q5_K with 2 <= N <= 7 run on the decode matvec path
("06 · 8e/8e② — decode MMVQ", §2 Principle: dp4a integer dots, the min term
from the Q8_1 block sum), the staged weights multiplied with every token;
larger N (the N = 8 and 16 cases) on the tensor-core GEMM."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_gemm, synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _run(W, X, M, K, wtype="q4_k"):
    import torch
    Y = kq_gemm(wtype, to_dev(W, torch), to_dev(X, torch), M, K)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


@pytest.mark.parametrize("M,K,N", [
    (512, 2048, 2),
    (300, 1024, 3),      # rows per CTA not a multiple of 32
    (1000, 4096, 4),
    (777, 2816, 5),      # two passes, the last with one token
    (640, 2048, 6),
    (4096, 11008, 7),    # the largest N on the decode path; two passes of four and three
    (2048, 1024, 8),     # tensor-core GEMM
    (129, 256, 16),      # one super-block per row (tensor-core GEMM)
])
def test_small_n_full_parity(M, K, N):
    rng = np.random.default_rng(M + 7 * N)
    W = syn.q4_k_weights(rng, M, K)
    X = syn.activations(rng, K, N)
    Y = _run(W, X, M, K)
    Yr, B = ora.matmul("q4_k", W, X, M, K)
    assert_within_bound(Y, Yr, B, f"q4_k {M}x{K} N={N}")


@pytest.mark.parametrize("M,K,N", [(4096, 11008, 4), (11008, 4096, 5), (11008, 4096, 16)])
def test_small_n_decode_shapes_sampled_rows(M, K, N):
    rng = np.random.default_rng(N)
    W = syn.q4_k_weights(rng, M, K)
    X = syn.activations(rng, K, N)
    Y = _run(W, X, M, K)
    rows = np.sort(np.concatenate([rng.choice(M, 160, replace=False), [0, 31, 32, M - 1]]))
    Yr, B = ora.matmul_rows("q4_k", W, X, K, rows)
    assert_within_bound(Y[:, rows], Yr, B, f"q4_k {M}x{K} N={N}")
    assert np.all(np.isfinite(Y))


def test_small_n_deterministic_and_per_token():
    # identical calls give identical bits; a token's row does not depend on the
    # other tokens of the call beyond rounding (the number of tokens changes how
    # the block sums are grouped), so it stays within the bound either way
    M, K = 1024, 2048
    rng = np.random.default_rng(5)
    W = syn.q4_k_weights(rng, M, K)
    X = syn.activations(rng, K, 6)
    a = _run(W, X, M, K)
    b = _run(W, X, M, K)
    assert np.array_equal(a, b)
    sub = np.ascontiguousarray(X[[3, 0, 5]])
    c = _run(W, sub, M, K)
    Yr, B = ora.matmul("q4_k", W, sub, M, K)
    assert_within_bound(c, Yr, B, "three tokens")
    assert_within_bound(a[[3, 0, 5]], Yr, B, "the same tokens among six")


@pytest.mark.parametrize("M,K,N", [(512, 2048, 2), (300, 1024, 3), (777, 2816, 5), (4096, 11008, 4), (1000, 2048, 7)])
def test_small_n_q5k(M, K, N):
    # Q5_K takes the same matvec path (its fifth bits merged into each dp4a word).
    rng = np.random.default_rng(M + 11 * N)
    W = syn.q5_k_weights(rng, M, K)
    X = syn.activations(rng, K, N)
    Y = _run(W, X, M, K, "q5_k")
    rows = np.arange(M) if M <= 1000 else np.sort(np.concatenate([rng.choice(M, 160, replace=False), [0, M - 1]]))
    Yr, B = ora.matmul_rows("q5_k", W, X, K, rows)
    assert_within_bound(Y[:, rows], Yr, B, f"q5_k {M}x{K} N={N}")
