"""The decode kernels' own Q8_1 quantisers, bit for bit against the oracle.

The decode matvec quantises x inside each CTA and the small-N decode in a
pre-pass; neither writes Q8_1 blocks to memory. Multiplied with the one-hot
matrices of tests/_onehot.py, every activation code and every block sum
appears alone in one output element as an exact fp32 value (d_h * q_k, and
-d_h * Sum q per block, or d_h * Sum q per half block for Q6_K), so the codes,
scales and sums these kernels use are compared with the oracle's Q8_1 step
("06 · 8e/8e② — decode MMVQ", §2 Principle and §3.2 quantize_pad40_block) with
np.array_equal: a code off by one, a scale rounded from the wrong value or a
wrong block sum fails.

Covered: kq_matvec in its staged lane-row form (row slices of at most 4096
rows), its ring form and the item kernel (the whole matrix, replicated where
needed so that a CTA's rows no longer fit), kq_matvec_prefetch, and the small-N
decode path of kq_gemm (2 to 7 tokens), on the activations of every workload
and on edge blocks.
"""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_gemm, kq_matvec, kq_matvec_prefetch, synthetic as syn
from _kqutil import to_dev
from _onehot import expected_outputs, onehot_weights

pytestmark = pytest.mark.gpu

SLICE_ROWS = 4096          # rows per call of the staged lane-row form at the decode sizes
SLICE_ROWS_TOKENS = 2048   # rows per call of the small-N decode (its staged rows sit beside several tokens' codes)
RING_MIN_ROWS = 16896      # enough rows that a CTA's range no longer fits staged (K >= 4096)


def _workload_tokens():
    """(name, X [n, K]) for every workload: its first tokens (up to 7)."""
    out = []
    for name, cfg in syn.WORKLOADS.items():
        _, r_x, _ = syn.rngs(cfg["seed"])
        n = cfg.get("N", cfg.get("T", 1))
        X = syn.activations(r_x, cfg["K"], min(n, 7))
        out.append((name, X))
    return out


def _edge_tokens(K):
    rng = np.random.default_rng(K)
    X = np.zeros((8, K), np.float32)
    X[0] = rng.standard_normal(K)
    X[1, :K // 2] = np.tile(np.concatenate([np.zeros(32), -np.zeros(32)]), K // 128)  # all-zero blocks
    X[1, K // 2:] = np.tile(127.0 * np.sign(rng.standard_normal(32)), K // 64)   # amax = 127 -> d = 1
    X[2] = np.tile(np.arange(32) - 15.5, K // 32)                                   # halves: ties to even
    X[3] = rng.standard_normal(K) * 1e-30                                            # d_h underflows to 0
    X[4] = rng.standard_normal(K) * 3e2
    X[5] = np.repeat(rng.standard_normal(K // 32), 32)                               # constant blocks
    X[6] = rng.standard_normal(K) * np.repeat(np.exp(2 * rng.standard_normal(K // 32)), 32)  # mixed scales
    X[7] = np.linspace(-1, 1, K) * np.tile(np.repeat(np.float32([1e-38, 3e-37, 5e-37, 1.0]), 32), K // 128)  # 1/d overflow
    return X


def _expected(wtype, X):
    q, d_h, _ = ora.quantize_q8_1(X)
    return np.stack([expected_outputs(wtype, q[t], d_h[t]) for t in range(X.shape[0])])


def _check(got, want, what):
    got = np.asarray(got)
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} outputs differ; first at flat index {i}: "
                             f"gpu={got.reshape(-1)[i]!r} want={want.reshape(-1)[i]!r}")


def _matvec_all_forms(wtype, W, Wd, x, want, what):
    """kq_matvec on row slices (staged form), on the whole matrix replicated
    up to RING_MIN_ROWS rows (ring or item form), and kq_matvec_prefetch."""
    import torch
    M, K = W.shape[0], x.shape[0]
    xd = to_dev(x, torch)
    got = np.empty(M, np.float32)
    for r0 in range(0, M, SLICE_ROWS):
        r1 = min(M, r0 + SLICE_ROWS)
        got[r0:r1] = kq_matvec(wtype, Wd[r0:r1], xd, r1 - r0, K).cpu().numpy()
    _check(got, want, f"{what} staged slices")
    reps = max(1, -(-RING_MIN_ROWS // M))
    Wr = Wd.repeat(reps, 1) if reps > 1 else Wd
    y = kq_matvec(wtype, Wr, xd, Wr.shape[0], K).cpu().numpy()
    _check(y, np.tile(want, reps), f"{what} whole ({Wr.shape[0]} rows)")
    y = kq_matvec_prefetch(wtype, Wd[:min(M, SLICE_ROWS)], xd, min(M, SLICE_ROWS), K, W_next=Wd).cpu().numpy()
    _check(y, want[:min(M, SLICE_ROWS)], f"{what} prefetch")


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k", "q6_k"])
def test_decode_quantiser_exact_on_workload_activations(wtype):
    import torch
    for name, X in _workload_tokens():
        K = X.shape[1]
        if wtype == "q6_k" and ((K // 256) * 210) % 16 and K > 15360:
            continue                                   # such Q6_K rows are refused (K <= 15360)
        W = onehot_weights(wtype, K)
        Wd = to_dev(W, torch)
        want = _expected(wtype, X[:1])[0]
        _matvec_all_forms(wtype, W, Wd, X[0], want, f"{wtype} {name}")
        del Wd
        torch.cuda.empty_cache()


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("K", [512, 4096, 11008])
def test_decode_quantiser_exact_on_edge_blocks(wtype, K):
    import torch
    X = _edge_tokens(K)
    W = onehot_weights(wtype, K)
    Wd = to_dev(W, torch)
    want = _expected(wtype, X)
    for t in range(X.shape[0]):
        _matvec_all_forms(wtype, W, Wd, X[t], want[t], f"{wtype} K={K} edge token {t}")


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k"])
@pytest.mark.parametrize("K", [2048, 4096, 11008])
def test_small_n_quantiser_exact(wtype, K):
    # kq_gemm sends 2..7 tokens of Q4_K / Q5_K to the decode path, whose
    # pre-pass makes every token's codes and block sums once.
    import torch
    rng = np.random.default_rng(K + 1)
    X = np.concatenate([_edge_tokens(K), syn.activations(rng, K, 7)])
    W = onehot_weights(wtype, K)
    Wd = to_dev(W, torch)
    want = _expected(wtype, X)
    M = W.shape[0]
    for N in range(2, 8):
        for t0 in (0, 8):
            Xd = to_dev(X[t0:t0 + N], torch)
            for r0 in range(0, M, SLICE_ROWS_TOKENS):
                r1 = min(M, r0 + SLICE_ROWS_TOKENS)
                Y = kq_gemm(wtype, Wd[r0:r1], Xd, r1 - r0, K).cpu().numpy()
                _check(Y, want[t0:t0 + N, r0:r1], f"{wtype} K={K} N={N} tokens {t0}.. rows {r0}..{r1}")
