"""Q5_K on the tensor-core paths (prefill GEMM, MoE grouped GEMM) against the
oracle, element by element within the bound. The weights are unpacked to fp16
like Q4_K's (the 5-bit code as fp16 1024 + q), so the same operand rounding
applies ("ZINC MMQ v2 — Fused Q4_K×Q8_1 Tensor-Core GEMM": the goal names the
Q5_K prefill GEMMs beside Q4_K and Q6_K)."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_gemm, kq_moe_grouped_gemm, synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N", [
    (256, 1024, 40),     # one 64-token tile, unpaired
    (384, 2048, 3),      # a few tokens: Q5_K stays on the tensor-core path
    (1024, 2048, 128),   # 128-token tiles: CTA pairs
    (640, 4096, 300),    # ragged token tail, 256-token pair tiles
])
def test_gemm_full_parity(M, K, N):
    import torch
    rng = np.random.default_rng(M + 7 * N)
    W = syn.q5_k_weights(rng, M, K)
    X = syn.activations(rng, K, N)
    Y = kq_gemm("q5_k", to_dev(W, torch), to_dev(X, torch), M, K)
    torch.cuda.synchronize()
    Yr, B = ora.matmul("q5_k", W, X, M, K)
    assert_within_bound(Y.cpu().numpy(), Yr, B, f"q5_k gemm {M}x{K}x{N}")


def test_gemm_large_sampled_rows():
    import torch
    M, K, N = 4096, 4096, 512
    rng = np.random.default_rng(5)
    W = syn.q5_k_weights(rng, M, K)
    X = syn.activations(rng, K, N)
    Y = kq_gemm("q5_k", to_dev(W, torch), to_dev(X, torch), M, K).cpu().numpy()
    rows = np.unique(np.concatenate([rng.choice(M, 96, replace=False), [0, 127, 128, 255, 256, M - 1]]))
    Yr, B = ora.matmul_rows("q5_k", W, X, K, rows)
    assert_within_bound(Y[:, rows], Yr, B, "q5_k gemm 4096x4096x512 rows")


@pytest.mark.parametrize("E,M,K,T,top_k", [(4, 128, 1024, 50, 2), (8, 256, 2048, 96, 3)])
def test_moe_full_parity(E, M, K, T, top_k):
    import torch
    rng = np.random.default_rng(E * M + T)
    W = syn.q5_k_weights(rng, E * M, K)
    X = syn.activations(rng, K, T)
    ids = syn.expert_ids(rng, T, E, top_k)
    Y = kq_moe_grouped_gemm("q5_k", to_dev(W, torch), E, to_dev(ids, torch), to_dev(X, torch), M, K)
    torch.cuda.synchronize()
    Yr, B = ora.moe("q5_k", W, ids, X, E, M, K)
    assert_within_bound(Y.cpu().numpy(), Yr, B, f"q5_k moe E{E} {M}x{K} T{T} top{top_k}")
