"""TQ4_1S decode matvec on the GPU against the TQ4_1S oracle (dequantise,
inverse WHT, dot product in fp64), element by element within
|y - y_ref| <= 1e-3 * Sum |r H x| + 1e-5 ("TQ4_1S Weight Kernel Optimization":
Architecture Overview, Block Layout, Centroid Table)."""
import numpy as np
import pytest

from oracle import tq4_oracle as tq
from quantized_weight_matmul_q4_gb300 import kq_matvec, synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _run(W, x, M, K):
    import torch
    y = kq_matvec("tq4_1s", to_dev(W, torch), to_dev(np.ascontiguousarray(x).reshape(-1), torch), M, K)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("M,K", [
    (1, 32), (5, 32), (17, 96), (45, 4000), (7, 40000),      # K % 128 != 0: the direct kernel, one or more K segments
    (64, 65536),                                              # rotated activations too large to stage: direct kernel
    (1, 128), (152, 128), (153, 256), (37, 11008),           # one row per CTA: 32 quad slices per row
    (512, 2048), (300, 4096), (1000, 4096), (3000, 3584),    # 2 .. 20 rows per CTA: 4 .. 16 slices
    (19456, 128), (160, 18944),                               # 128 rows per CTA; two chunk slots
])
def test_shapes_full_parity(M, K):
    rng = np.random.default_rng(M * 31 + K)
    W = syn.tq4_1s_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    y = _run(W, x, M, K)
    Y, B = tq.tq4_1s_matmul(W, x, M, K)
    assert_within_bound(y, Y[0], B[0], f"tq4_1s {M}x{K}")


@pytest.mark.parametrize("name", ["decode_tq4_1s_18944x3584", "decode_tq4_1s_3584x18944"])
def test_decode_workloads_sampled_rows(name):
    # The 7B FFN shapes: ring-staged chunks (more chunks than slots); rows at
    # CTA range boundaries and the last rows are among the sampled ones.
    wl = syn.make_workload(name)
    M, K = wl["M"], wl["K"]
    W, x = wl["W"][0], wl["X"]
    y = _run(W, x, M, K)
    R = -(-M // 152)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(M, 160, replace=False), [0, R - 1, R, 2 * R - 1, M - 2, M - 1]]))
    Y, B = tq.tq4_1s_matmul_rows(W, x, K, rows)
    assert_within_bound(y[rows], Y[0], B[0], name)
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("M,K", [(4096, 14336), (14336, 4096)])
def test_other_ring_shapes_sampled_rows(M, K):
    rng = np.random.default_rng(M + K)
    W = syn.tq4_1s_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    y = _run(W, x, M, K)
    R = -(-M // 152)
    rows = np.unique(np.concatenate([rng.choice(M, 128, replace=False), [0, R - 1, R, M - 1]]))
    Y, B = tq.tq4_1s_matmul_rows(W, x, K, rows)
    assert_within_bound(y[rows], Y[0], B[0], f"tq4_1s {M}x{K}")


def test_deterministic():
    wl = syn.make_workload("decode_tq4_1s_3584x18944")
    a = _run(wl["W"][0], wl["X"], wl["M"], wl["K"])
    b = _run(wl["W"][0], wl["X"], wl["M"], wl["K"])
    assert np.array_equal(a, b)


def test_zero_activation_gives_zero():
    M, K = 200, 3584
    W = syn.tq4_1s_weights(np.random.default_rng(2), M, K)
    y = _run(W, np.zeros((1, K), np.float32), M, K)
    assert np.all(y == 0)


def test_constant_blocks_pick_element_zero():
    # Every block all index v with d0 = d1 = d: each block's weights are
    # c[v] d sqrt(32) at element 0 and zero elsewhere, so y = c[v] d sqrt(32) Sum_b x[32 b].
    M, K, v, d = 64, 1024, 13, 0.25
    blk = np.zeros(20, np.uint8)
    blk[0:4] = np.array([d, d], dtype=np.float16).view(np.uint8)
    blk[4:] = v | (v << 4)
    W = np.tile(blk, (M, K // 32))
    x = syn.activations(np.random.default_rng(3), K, 1)
    y = _run(W, x, M, K)
    want = tq.CENTROIDS[v] * d * np.sqrt(32) * x[0, ::32].astype(np.float64).sum()
    assert np.allclose(y, want, rtol=1e-5, atol=1e-5)
