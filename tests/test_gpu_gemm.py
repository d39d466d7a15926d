"""Prefill GEMM on the tensor cores against the oracle, element by element,
within |y - y_ref| <= 1e-3 * Sum_k |w_k x_k| + 1e-5 ("ZINC MMQ v2", Kernel
architecture and Correctness gate; "Prefill Gap Closure Plan", T1)."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_gemm, synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _run(wtype, W, X, M, K):
    import torch
    Y = kq_gemm(wtype, to_dev(W, torch), to_dev(X, torch), M, K)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


@pytest.mark.parametrize("wtype,M,K,N", [
    ("q4_k", 128, 256, 16),        # one tile, one super-block
    ("q4_k", 200, 512, 5),         # ragged M and N, split K
    ("q4_k", 256, 1024, 64),
    ("q4_k", 384, 768, 100),       # N tile of 128 rows, ragged
    ("q4_k", 130, 2048, 300),      # two N tiles (256 + 44), ragged M
    ("q4_k", 1, 256, 1),
    ("q6_k", 136, 2048, 40),
    ("q6_k", 256, 4096, 257),
    # CTA pairs (even number of 128-row tiles, token tile of 128 or 256)
    ("q4_k", 512, 1024, 128),      # bn = 128: one 64-row x_hat box per CTA
    ("q4_k", 500, 512, 200),       # bn = 256, ragged M and ragged second half
    ("q6_k", 512, 2048, 96),       # bn = 128, second half partly past N
    ("q4_k", 256, 4096, 256),      # one pair tile, K split 16 ways
    ("q4_k", 20480, 256, 100),     # 80 pair tiles: some pairs take two, alternating accumulators
])
def test_small_shapes_full_parity(wtype, M, K, N):
    rng = np.random.default_rng(M + 3 * K + 7 * N)
    W = syn.weights(wtype, rng, M, K)
    X = syn.activations(rng, K, N)
    Y = _run(wtype, W, X, M, K)
    Yr, B = ora.matmul(wtype, W, X, M, K)
    assert_within_bound(Y, Yr, B, f"{wtype} {M}x{K}x{N}")


@pytest.mark.parametrize("name", ["prefill_q4k_4096x4096_n64", "prefill_q4k_4096x4096_n512"])
def test_prefill_workloads_full_parity(name):
    wl = syn.make_workload(name)
    M, K = wl["M"], wl["K"]
    Y = _run(wl["wtype"], wl["W"][0], wl["X"], M, K)
    Yr, B = ora.matmul(wl["wtype"], wl["W"][0], wl["X"], M, K)
    assert_within_bound(Y, Yr, B, name)


@pytest.mark.parametrize("name", ["prefill_q4k_14336x4096_n2048", "prefill_q6k_4096x14336_n2048",
                                  "prefill_q5k_14336x4096_n2048"])
def test_large_workloads_sampled_rows(name):
    wl = syn.make_workload(name)
    M, K = wl["M"], wl["K"]
    Y = _run(wl["wtype"], wl["W"][0], wl["X"], M, K)
    # every 128-row tile (and so every 256-row pair tile) is checked: its first
    # and last rows and one random row inside it, plus the matrix's last row
    rng = np.random.default_rng(11)
    starts = np.arange(0, M, 128)
    inner = starts + rng.integers(1, 127, size=starts.size)
    rows = np.unique(np.concatenate([starts, np.minimum(starts + 127, M - 1), np.minimum(inner, M - 1), [M - 1]]))
    Yr, B = ora.matmul_rows(wl["wtype"], wl["W"][0], wl["X"], K, rows)
    assert_within_bound(Y[:, rows], Yr, B, name)
    assert np.all(np.isfinite(Y))


def test_deterministic_and_matches_matvec_semantics():
    M, K, N = 512, 2048, 64
    rng = np.random.default_rng(2)
    W = syn.q4_k_weights(rng, M, K)
    X = syn.activations(rng, K, N)
    a = _run("q4_k", W, X, M, K)
    b = _run("q4_k", W, X, M, K)
    assert np.array_equal(a, b)
