"""Failure detection on the GPU without a fault: a pipeline wait that runs out.

kq_test_hold_copies makes the weight producers issue nothing, so every
consumer wait of the next launch runs out after its limit (2 s). The kernel
must then record KQ_DEVERR_WAIT_TIMEOUT, leave its loops, free its tensor
memory and return (no copy is in flight), and the context must stay usable: a
normal call right after it meets the accuracy bound against the oracle and
records no error. Each kernel form is held once: the staged and ring lane-row
decode kernels, the item decode kernel (Q6_K), the unpaired and the paired
tensor-core GEMM, and the MoE grouped GEMM.
"""
import numpy as np
import pytest

import quantized_weight_matmul_q4_gb300 as kq
from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _held_then_normal(call):
    """Runs call() once held and once normally; returns the normal result."""
    import torch
    assert kq.kq_get_device_error() == kq.KQ_DEVERR_NONE
    kq.kq_test_hold_copies(True)
    try:
        call()
    finally:
        kq.kq_test_hold_copies(False)
    assert kq.kq_get_device_error() == kq.KQ_DEVERR_WAIT_TIMEOUT
    assert kq.kq_get_device_error() == kq.KQ_DEVERR_NONE       # read once, then cleared
    out = call()
    torch.cuda.synchronize()
    assert kq.kq_get_device_error() == kq.KQ_DEVERR_NONE
    return out


@pytest.mark.parametrize("wtype,M,K", [
    ("q4_k", 4096, 11008),    # lane-row kernel, all rows staged
    ("q4_k", 4096, 14336),    # lane-row kernel, ring of chunk slots
    ("q6_k", 300, 4096),      # item kernel
])
def test_matvec_wait_timeout_then_recovers(wtype, M, K):
    import torch
    rng = np.random.default_rng(M + K)
    W = syn.weights(wtype, rng, M, K)
    x = syn.activations(rng, K, 1)
    Wd, xd = to_dev(W, torch), to_dev(x.reshape(-1), torch)
    y = _held_then_normal(lambda: kq.kq_matvec(wtype, Wd, xd, M, K))
    Y, B = ora.matmul(wtype, W, x, M, K)
    assert_within_bound(y.cpu().numpy(), Y[0], B[0], f"{wtype} {M}x{K} after a timeout")


@pytest.mark.parametrize("M,K,N", [
    (256, 1024, 64),     # unpaired tiles, K split across CTAs
    (512, 1024, 256),    # CTA pairs
])
def test_gemm_wait_timeout_then_recovers(M, K, N):
    import torch
    rng = np.random.default_rng(M + N)
    W = syn.q4_k_weights(rng, M, K)
    X = syn.activations(rng, K, N)
    Wd, Xd = to_dev(W, torch), to_dev(X, torch)
    Y = _held_then_normal(lambda: kq.kq_gemm("q4_k", Wd, Xd, M, K))
    Yr, B = ora.matmul("q4_k", W, X, M, K)
    assert_within_bound(Y.cpu().numpy(), Yr, B, f"gemm {M}x{K}x{N} after a timeout")


def test_moe_wait_timeout_then_recovers():
    import torch
    E, M, K, T, top_k = 8, 256, 1024, 64, 2
    rng = np.random.default_rng(3)
    W = syn.q4_k_weights(rng, E * M, K)
    X = syn.activations(rng, K, T)
    ids = syn.expert_ids(rng, T, E, top_k)
    Wd, Xd, idd = to_dev(W, torch), to_dev(X, torch), to_dev(ids, torch)
    Y = _held_then_normal(lambda: kq.kq_moe_grouped_gemm("q4_k", Wd, E, idd, Xd, M, K))
    Yr, B = ora.moe("q4_k", W, ids, X, E, M, K)
    assert_within_bound(Y.cpu().numpy(), Yr, B, "moe after a timeout")
