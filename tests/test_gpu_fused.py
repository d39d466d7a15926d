"""The steps next to the matmul on the GPU against the oracle: the decode
matvec with its RMSNorm or SwiGLU producer fused into the Q8_1 quantiser
("06 · 8e/8e② — decode MMVQ", §3.2 Key code), and the router-weighted MoE
combine after the grouped expert GEMM ("Prefill Gap Closure Plan", T2,
"scatter back"). Element by element within |y - y_ref| <= 1e-3 * B + 1e-5,
B = Sum_k |w_k x_k| for the oracle's Q8_1 codes of the produced activations
(computed in fp64 and rounded to fp32; the GPU computes the producers in fp32,
so a code may differ by one at a rounding boundary, well inside the bound)."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
import quantized_weight_matmul_q4_gb300 as kq
from quantized_weight_matmul_q4_gb300 import synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu

# (wtype, M, K): the staged lane-row decode kernel (the decode shapes, a small
# one), its ring form (15200 x 4096: a CTA's rows do not fit whole), the item
# kernel for Q4_K (x too long for the lane-row forms) and for Q6_K (aligned and
# unaligned rows).
SHAPES = [("q4_k", 4096, 11008), ("q4_k", 11008, 4096), ("q4_k", 300, 2048), ("q4_k", 15200, 4096),
          ("q4_k", 256, 102400), ("q6_k", 1000, 4096), ("q6_k", 512, 11008)]


def _check(wtype, W, xp, y, M, K, what):
    """y against the oracle on all rows (M <= 2048) or on sampled rows."""
    rng = np.random.default_rng(M)
    rows = np.arange(M) if M <= 2048 else np.sort(np.concatenate([rng.choice(M, 256, replace=False), [0, M - 1]]))
    Yr, B = ora.matmul_rows(wtype, W, np.asarray(xp, dtype=np.float32)[None, :], K, rows)
    assert_within_bound(y[rows], Yr[0], B[0], what)


@pytest.mark.parametrize("wtype,M,K", SHAPES)
def test_matvec_swiglu(wtype, M, K):
    import torch
    rng = np.random.default_rng(M + K)
    W = syn.weights(wtype, rng, M, K)
    g = (rng.standard_normal(K) * 3).astype(np.float32)
    u = rng.standard_normal(K).astype(np.float32)
    y = kq.kq_matvec_swiglu(wtype, to_dev(W, torch), to_dev(g, torch), to_dev(u, torch), M, K)
    torch.cuda.synchronize()
    _check(wtype, W, ora.swiglu(g, u), y.cpu().numpy(), M, K, f"swiglu {wtype} {M}x{K}")


@pytest.mark.parametrize("wtype,M,K", SHAPES)
@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_matvec_rmsnorm(wtype, M, K, eps):
    import torch
    rng = np.random.default_rng(M + 3 * K)
    W = syn.weights(wtype, rng, M, K)
    x = (rng.standard_normal(K) * 7 + 1).astype(np.float32)
    gamma = rng.uniform(0.2, 2.0, K).astype(np.float32)
    y = kq.kq_matvec_rmsnorm(wtype, to_dev(W, torch), to_dev(x, torch), to_dev(gamma, torch), eps, M, K)
    torch.cuda.synchronize()
    _check(wtype, W, ora.rms_norm(x[None, :], gamma, eps)[0], y.cpu().numpy(), M, K,
           f"rmsnorm {wtype} {M}x{K} eps={eps}")


def test_fused_matvec_deterministic():
    import torch
    rng = np.random.default_rng(9)
    M, K = 4096, 11008
    W = to_dev(syn.q4_k_weights(rng, M, K), torch)
    x = to_dev(rng.standard_normal(K).astype(np.float32), torch)
    g = to_dev(rng.uniform(0.5, 1.5, K).astype(np.float32), torch)
    a = kq.kq_matvec_rmsnorm("q4_k", W, x, g, 1e-5, M, K)
    b = kq.kq_matvec_rmsnorm("q4_k", W, x, g, 1e-5, M, K)
    c = kq.kq_matvec_swiglu("q4_k", W, x, g, M, K)
    d = kq.kq_matvec_swiglu("q4_k", W, x, g, M, K)
    assert torch.equal(a, b) and torch.equal(c, d)


@pytest.mark.parametrize("T,top_k,M", [(37, 3, 200), (64, 8, 768), (5, 1, 13), (1, 16, 4)])
def test_moe_combine(T, top_k, M):
    import torch
    rng = np.random.default_rng(T * top_k + M)
    Y = rng.standard_normal((T, top_k, M)).astype(np.float32)
    P = rng.uniform(size=(T, top_k)).astype(np.float32)
    out = kq.kq_moe_combine(to_dev(Y, torch), to_dev(P, torch)).cpu().numpy()
    ref = ora.moe_combine(Y, P)
    # one fp32 rounding per fused multiply-add, top_k of them in a row
    bound = 2.0 ** -23 * top_k * np.einsum("tj,tjm->tm", np.abs(P).astype(np.float64), np.abs(Y).astype(np.float64))
    assert np.all(np.abs(out - ref) <= bound + 1e-30)


def test_moe_then_combine_matches_the_oracle():
    import torch
    wl = syn.make_workload("moe_q4k_128x768x2048_t1024_top8")
    E, M, K, T, top_k = wl["n_experts"], wl["M"], wl["K"], wl["T"], wl["top_k"]
    rng = np.random.default_rng(12)
    P = rng.dirichlet(np.ones(top_k), size=T).astype(np.float32)
    Y = kq.kq_moe_grouped_gemm("q4_k", to_dev(wl["W"][0], torch), E, to_dev(wl["ids"], torch),
                               to_dev(wl["X"], torch), M, K)
    out = kq.kq_moe_combine(Y, to_dev(P, torch)).cpu().numpy()
    Yr, B = ora.moe("q4_k", wl["W"][0], wl["ids"], wl["X"], E, M, K)
    ref = ora.moe_combine(Yr, P)
    bound = np.einsum("tj,tjm->tm", P.astype(np.float64), ora.tolerance(B)) + 1e-6 * ora.moe_combine(np.abs(Yr), P)
    assert np.all(np.abs(out - ref) <= bound)
