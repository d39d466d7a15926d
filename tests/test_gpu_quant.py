"""Q8_1 activation quantisation on the GPU against the oracle: bit-exact bytes
(codes, fp16 scale, fp16 block sum) on every workload's activations and on edge
cases ("06 · 8e/8e② — decode MMVQ", §2 and §3.2 quantize_pad40_block)."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_quantize_q8_1, synthetic as syn
from _kqutil import to_dev

pytestmark = pytest.mark.gpu


def _gpu_q8(X):
    import torch
    Xq = kq_quantize_q8_1(to_dev(X, torch))
    torch.cuda.synchronize()
    return Xq.cpu().numpy()


def _ref_q8(X):
    q, d_h, s_h = ora.quantize_q8_1(X)
    return ora.pack_q8_1(q, d_h, s_h)


@pytest.mark.parametrize("name", list(syn.WORKLOADS))
def test_workload_activations_bit_exact(name):
    cfg = syn.WORKLOADS[name]
    _, r_x, _ = syn.rngs(cfg["seed"])
    N = cfg["N"] if "N" in cfg else cfg["T"]
    X = syn.activations(r_x, cfg["K"], N)
    got, want = _gpu_q8(X), _ref_q8(X)
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_edge_blocks_bit_exact():
    rng = np.random.default_rng(3)
    K = 32 * 16
    X = np.zeros((7, K), np.float32)
    X[0] = rng.standard_normal(K)
    X[1, :32] = 0.0                                        # all-zero block
    X[1, 32:64] = -0.0
    X[1, 64:96] = 127.0 * np.sign(rng.standard_normal(32))  # amax = 127 exactly -> d = 1
    X[1, 96:128] = np.arange(32) - 15.5                   # halves -> ties to even
    X[2] = rng.standard_normal(K) * 1e-30                  # tiny scales (d_h underflows to 0)
    X[3] = rng.standard_normal(K) * 3e2                    # large scales
    X[4] = np.repeat(rng.standard_normal(K // 32), 32)     # constant blocks
    X[5, ::32] = 1.0                                       # a single non-zero per block
    X[5, 1::32] = -1.0 + 2 ** -20
    # max|x| around the point where 1/d overflows fp32 (~3.7e-37): subnormal,
    # just below (codes 0), just above (codes as usual)
    for b, sc in enumerate([1e-38, 3.0e-37, 5.0e-37, 1e-36] * (K // 128)):
        X[6, 32 * b:32 * b + 32] = np.linspace(-1, 1, 32) * np.float32(sc)
    got, want = _gpu_q8(X), _ref_q8(X)
    assert np.array_equal(got, want)


def test_ragged_token_counts():
    for N, K in [(1, 32), (3, 96), (7, 2080)]:
        X = np.random.default_rng(N).standard_normal((N, K)).astype(np.float32)
        assert np.array_equal(_gpu_q8(X), _ref_q8(X))
