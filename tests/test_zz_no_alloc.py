"""kq_gemm_noalloc (the GEMM with the library's fixed per-device scratch)
through the C ABI, on two calls in a row: each call's output against the
oracle's Y_ref within the per-element bound, and against kq_gemm's output on
the same inputs within the same bound.

The file name sorts last so that it runs after every other test as well as
alone in a fresh process; both orders must pass."""
import ctypes

import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import _native as nat
from quantized_weight_matmul_q4_gb300 import kq_gemm, kq_gemm_noalloc, kq_workspace_bytes, synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wtype,M,K,N", [
    ("q4_k", 200, 512, 5),         # split K: partial sums in the scratch
    ("q4_k", 384, 1024, 300),      # two N tiles, ragged
    ("q6_k", 256, 2048, 40),
])
def test_noalloc_matches_gemm_twice(wtype, M, K, N):
    import torch
    rng = np.random.default_rng(M + 5 * K + 11 * N)
    W = syn.weights(wtype, rng, M, K)
    X = syn.activations(rng, K, N)
    Wd, Xd = to_dev(W, torch), to_dev(X, torch)
    Ygemm = kq_gemm(wtype, Wd, Xd, M, K)
    torch.cuda.synchronize()
    Ygemm = Ygemm.cpu().numpy().astype(np.float64)
    Yref, B = ora.matmul(wtype, W, X, M, K)
    for call in range(2):
        Y = kq_gemm_noalloc(wtype, Wd, Xd, M, K)
        torch.cuda.synchronize()
        Y = Y.cpu().numpy()
        assert_within_bound(Y, Yref, B, f"call {call} {wtype} {M}x{K}x{N} vs oracle")
        assert_within_bound(Y, Ygemm, B, f"call {call} {wtype} {M}x{K}x{N} vs kq_gemm")


def test_noalloc_prefill_workload_twice():
    import torch
    wl = syn.make_workload("prefill_q4k_4096x4096_n512")
    M, K = wl["M"], wl["K"]
    Wd, Xd = to_dev(wl["W"][0], torch), to_dev(wl["X"], torch)
    Ygemm = kq_gemm(wl["wtype"], Wd, Xd, M, K)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 2047, M - 1])
    Yref, B = ora.matmul_rows(wl["wtype"], wl["W"][0], wl["X"], K, rows)
    ref = Ygemm.cpu().numpy().astype(np.float64)
    for call in range(2):
        Y = kq_gemm_noalloc(wl["wtype"], Wd, Xd, M, K).cpu().numpy()
        assert_within_bound(Y[:, rows], Yref, B, f"call {call} vs oracle")
        assert_within_bound(Y[:, rows], ref[:, rows], B, f"call {call} vs kq_gemm")
        assert np.all(np.isfinite(Y))


def test_noalloc_rejects_oversize_scratch():
    import torch
    M, K, N = 256, 14336, 2048
    assert kq_workspace_bytes(nat.KQ_OP_GEMM, "q4_k", M, K, N) > nat.KQ_GEMM_STATIC_WS_BYTES
    W = torch.zeros((M, (K // 256) * 144), dtype=torch.uint8, device="cuda")
    X = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    Y = torch.full((N, M), 7.0, dtype=torch.float32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = nat.lib().kq_gemm_noalloc(nat.KQ_Q4_K, ctypes.c_void_p(W.data_ptr()), ctypes.c_void_p(X.data_ptr()),
                                   ctypes.c_void_p(Y.data_ptr()), M, K, N, s)
    assert st == nat.KQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool(torch.all(Y == 7.0))   # nothing was queued
