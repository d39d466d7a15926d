"""CPU pins of the one-hot weight matrices used to expose the fused Q8_1 codes
(tests/_onehot.py): the oracle's own dequantisation of each matrix is the
matrix the construction describes, and the oracle's product with it is the
list of exact codes and block sums that the GPU tests expect."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from _onehot import expected_outputs, onehot_weights


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k", "q6_k"])
@pytest.mark.parametrize("K", [256, 768])
def test_onehot_dequantises_to_the_described_matrix(wtype, K):
    W = onehot_weights(wtype, K)
    w = ora.dequant(wtype, W, K)
    assert np.array_equal(w[:K], np.eye(K))
    sums = w[K:]
    if wtype == "q6_k":
        want = np.kron(np.eye(K // 16), np.ones(16))
    else:
        want = -np.kron(np.eye(K // 32), np.ones(32))
    assert np.array_equal(sums, want)


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k", "q6_k"])
def test_onehot_product_is_the_codes_and_sums(wtype):
    K = 512
    rng = np.random.default_rng(17)
    X = (rng.standard_normal((1, K)) * np.repeat(np.exp(rng.standard_normal(K // 32)), 32)).astype(np.float32)
    W = onehot_weights(wtype, K)
    Y, _ = ora.matmul(wtype, W, X, W.shape[0], K)
    q, d_h, s_h = ora.quantize_q8_1(X)
    want = expected_outputs(wtype, q[0], d_h[0])
    assert np.array_equal(Y[0], want.astype(np.float64))
    if wtype != "q6_k":
        # the sum rows carry the Q8_1 block sum: s_h = fp16(d_h * Sum q) = fp16(-y)
        assert np.array_equal(ora.f32_to_fp16_bits(-want[K:]), s_h[0])


def test_a_code_off_by_one_changes_an_output():
    # The construction can see a plausible quantiser mistake: one code moved by one.
    K = 256
    X = np.random.default_rng(4).standard_normal((1, K)).astype(np.float32)
    q, d_h, _ = ora.quantize_q8_1(X)
    good = expected_outputs("q4_k", q[0], d_h[0])
    q2 = q.copy()
    q2[0, 3, 5] += 1 if q2[0, 3, 5] < 127 else -1
    bad = expected_outputs("q4_k", q2[0], d_h[0])
    assert not np.array_equal(good, bad)
