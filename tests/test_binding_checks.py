"""The binding's argument checks (CPU): every public call refuses what the
library cannot take before anything reaches the C ABI, with the same errors
whether or not the fast path of the checks applies."""
import numpy as np
import pytest

import quantized_weight_matmul_q4_gb300 as kq
from quantized_weight_matmul_q4_gb300 import _dev, _wt


def test_cpu_tensor_is_refused():
    torch = pytest.importorskip("torch")
    W = torch.zeros(144, dtype=torch.uint8)
    x = torch.zeros(256, dtype=torch.float32)
    with pytest.raises(TypeError, match="CUDA tensor"):
        kq.kq_matvec("q4_k", W, x, 1, 256, y=torch.zeros(1))
    with pytest.raises(TypeError, match="CUDA tensor"):
        _dev(x, "x", torch.float32)


def test_non_tensor_is_refused():
    pytest.importorskip("torch")
    with pytest.raises(TypeError, match="CUDA tensor"):
        _dev(np.zeros(4, np.float32), "x")
    with pytest.raises(TypeError, match="CUDA tensor"):
        _dev(None, "x")


def test_weight_type_names():
    assert _wt("q4_k") == kq.KQ_Q4_K
    assert _wt("Q6_K") == kq.KQ_Q6_K      # any case
    assert _wt("q5_k") == kq.KQ_Q5_K
    assert _wt("tq4_1s") == kq.KQ_TQ4_1S
    assert _wt(kq.KQ_Q4_K) == kq.KQ_Q4_K
    with pytest.raises(KeyError):
        _wt("q3_k")
