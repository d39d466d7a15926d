"""Q5_K decode matvec on the GPU against the oracle, element by element,
within |y - y_ref| <= 1e-3 * Sum_k |w_k x_k| + 1e-5. Q5_K is the pages' sibling
of the Q4_K and Q6_K decode kernels ("06 · 8e/8e② — decode MMVQ", §3.2 Key
code: one kernel per type); its block is read with the GGUF layout."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_matvec, kq_matvec_rmsnorm, kq_matvec_swiglu, synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _run(W, x, M, K, wtype="q5_k"):
    import torch
    y = kq_matvec(wtype, to_dev(W, torch), to_dev(np.ascontiguousarray(x).reshape(-1), torch), M, K)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("M,K", [
    (1, 256), (17, 512), (37, 11008), (300, 4096), (1000, 2304), (33, 65536),  # lane-row kernel, staged
    (20000, 512), (19457, 256),                                                 # more rows than a CTA takes: item kernel
])
def test_shapes_full_parity(M, K):
    rng = np.random.default_rng(M * 13 + K)
    W = syn.q5_k_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    y = _run(W, x, M, K)
    Y, B = ora.matmul("q5_k", W, x, M, K)
    assert_within_bound(y, Y[0], B[0], f"q5_k {M}x{K}")


@pytest.mark.parametrize("name", ["decode_q5k_4096x11008", "decode_q5k_11008x4096"])
def test_decode_workloads_sampled_rows(name):
    # Slices larger than shared memory: the ring form of the lane-row kernel.
    wl = syn.make_workload(name)
    M, K = wl["M"], wl["K"]
    W, x = wl["W"][0], wl["X"]
    y = _run(W, x, M, K)
    R = -(-M // 152)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.choice(M, 160, replace=False), [0, R - 1, R, M - 2, M - 1]]))
    Yr, B = ora.matmul_rows("q5_k", W, x, K, rows)
    assert_within_bound(y[rows], Yr[0], B[0], name)
    assert np.all(np.isfinite(y))


def test_zero_high_bits_agree_with_q4k():
    # The same fields as a Q4_K matrix with every fifth bit zero: both kernels
    # compute the same product.
    M, K = 512, 4096
    q4 = syn.q4_k_weights(np.random.default_rng(9), M, K).reshape(M, K // 256, 144)
    q5 = np.zeros((M, K // 256, 176), np.uint8)
    q5[..., 0:16] = q4[..., 0:16]
    q5[..., 48:176] = q4[..., 16:144]
    x = syn.activations(np.random.default_rng(10), K, 1)
    y4 = _run(q4.reshape(M, -1), x, M, K, "q4_k")
    y5 = _run(q5.reshape(M, -1), x, M, K, "q5_k")
    _, B = ora.matmul("q4_k", q4.reshape(M, -1), x, M, K)
    assert_within_bound(y5, y4.astype(np.float64), B[0], "q5_k with qh = 0 vs q4_k")


@pytest.mark.parametrize("prod", ["swiglu", "rmsnorm"])
def test_fused_producers(prod):
    import torch
    M, K = 2048, 11008
    rng = np.random.default_rng(4)
    W = syn.q5_k_weights(rng, M, K)
    a = syn.activations(rng, K, 1)
    b = syn.activations(rng, K, 1)
    if prod == "swiglu":
        y = kq_matvec_swiglu("q5_k", to_dev(W, torch), to_dev(a[0], torch), to_dev(b[0], torch), M, K)
        xp = ora.swiglu(a, b)
    else:
        g = np.abs(b).astype(np.float32) + 0.5
        y = kq_matvec_rmsnorm("q5_k", to_dev(W, torch), to_dev(a[0], torch), to_dev(g[0], torch), 1e-6, M, K)
        xp = ora.rms_norm(a, g[0], 1e-6)
    torch.cuda.synchronize()
    Y, B = ora.matmul_from("q5_k", W, xp, M, K)
    assert_within_bound(y.cpu().numpy(), Y[0], B[0], f"q5_k {prod}")


def test_deterministic():
    wl = syn.make_workload("decode_q5k_11008x4096")
    a = _run(wl["W"][0], wl["X"], wl["M"], wl["K"])
    b = _run(wl["W"][0], wl["X"], wl["M"], wl["K"])
    assert np.array_equal(a, b)
