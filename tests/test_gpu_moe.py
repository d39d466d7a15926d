"""MoE grouped expert GEMM on the GPU against the oracle ("ZINC MMQ v2", MoE
routing; "Prefill Gap Closure Plan", T2): every (token, slot) output equals the
dense product with the routed expert's weights, within the per-element bound."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
import quantized_weight_matmul_q4_gb300 as kq
from quantized_weight_matmul_q4_gb300 import synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _run(wtype, W, ids, X, E, M, K):
    import torch
    Y = kq.kq_moe_grouped_gemm(wtype, to_dev(W, torch), E, to_dev(ids.astype(np.int32), torch),
                               to_dev(X, torch), M, K)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


@pytest.mark.parametrize("name", ["moe_q4k_128x768x2048_t1024_top8", "moe_q6k_128x768x2048_t1024_top8"])
def test_workload_full_parity(name):
    wl = syn.make_workload(name)
    E, M, K, wtype = wl["n_experts"], wl["M"], wl["K"], wl["wtype"]
    Y = _run(wtype, wl["W"][0], wl["ids"], wl["X"], E, M, K)
    Yr, B = ora.moe(wtype, wl["W"][0], wl["ids"], wl["X"], E, M, K)
    assert_within_bound(Y, Yr, B, name)
    assert kq.kq_get_device_error() == kq.KQ_DEVERR_NONE


@pytest.mark.parametrize("wtype,E,M,K,T,top_k", [
    ("q4_k", 5, 200, 512, 37, 3),
    ("q4_k", 3, 128, 256, 300, 2),     # buckets larger than one 128-token tile
    ("q4_k", 16, 64, 1024, 9, 1),      # most experts get no token
    ("q6_k", 4, 136, 2048, 50, 2),
    ("q4_k", 6, 256, 512, 300, 2),     # buckets of more than one 128-token tile
    ("q6_k", 3, 512, 2048, 70, 3),
    ("q4_k", 1, 128, 256, 1, 1),       # one expert, one token
    ("q4_k", 1, 256, 512, 300, 1),     # every token to the only expert: a bucket of several tiles
    ("q4_k", 512, 128, 256, 20, 4),    # the most experts the call takes; nearly all get no token
])
def test_small_shapes_full_parity(wtype, E, M, K, T, top_k):
    rng = np.random.default_rng(E * 100 + T)
    W = syn.weights(wtype, rng, E * M, K)
    X = syn.activations(rng, K, T)
    ids = syn.expert_ids(rng, T, E, top_k)
    Y = _run(wtype, W, ids, X, E, M, K)
    Yr, B = ora.moe(wtype, W, ids, X, E, M, K)
    assert_within_bound(Y, Yr, B, f"moe {wtype} E={E} T={T}")


@pytest.mark.parametrize("M", [128, 256])
def test_all_tokens_to_one_expert(M):
    E, K, T = 4, 512, 260
    rng = np.random.default_rng(9)
    W = syn.q4_k_weights(rng, E * M, K)
    X = syn.activations(rng, K, T)
    ids = np.zeros((T, 1), np.int32) + 2
    Y = _run("q4_k", W, ids, X, E, M, K)
    Yr, B = ora.moe("q4_k", W, ids, X, E, M, K)
    assert_within_bound(Y, Yr, B, "one expert")


@pytest.mark.parametrize("M", [128, 256])
def test_out_of_range_expert_id_is_reported_and_zeroed(M):
    E, K, T, top_k = 4, 256, 10, 2
    rng = np.random.default_rng(4)
    W = syn.q4_k_weights(rng, E * M, K)
    X = syn.activations(rng, K, T)
    ids = syn.expert_ids(rng, T, E, top_k)
    ids[3, 1] = 7
    ids[5, 0] = -1
    kq.kq_get_device_error()                       # clear
    Y = _run("q4_k", W, ids, X, E, M, K)
    assert kq.kq_get_device_error() == kq.KQ_DEVERR_EXPERT_ID
    assert np.all(Y[3, 1] == 0) and np.all(Y[5, 0] == 0)
    ok = np.ones((T, top_k), bool)
    ok[3, 1] = ok[5, 0] = False
    good_ids = np.where(ok, ids, 0)
    Yr, B = ora.moe("q4_k", W, good_ids, X, E, M, K)
    assert_within_bound(Y[ok], Yr[ok], B[ok], "valid slots")


def test_deterministic():
    wl = syn.make_workload("moe_q4k_128x768x2048_t1024_top8")
    a = _run("q4_k", wl["W"][0], wl["ids"], wl["X"], 128, 768, 2048)
    b = _run("q4_k", wl["W"][0], wl["ids"], wl["X"], 128, 768, 2048)
    assert np.array_equal(a, b)
