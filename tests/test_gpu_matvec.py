"""Decode matvec (N = 1) on the GPU against the oracle, element by element,
within |y - y_ref| <= 1e-3 * Sum_k |w_k x_k| + 1e-5 ("06 · 8e/8e② — decode
MMVQ", §2 Principle and §3.2 Key code)."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import kq_matvec, synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu


def _run(wtype, W, x, M, K):
    import torch
    y = kq_matvec(wtype, to_dev(W, torch), to_dev(x.reshape(-1), torch), M, K)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("name", ["matvec_q4k_512x2048", "decode_q4k_4096x11008", "decode_q4k_11008x4096",
                                  "decode_q6k_4096x11008", "decode_q6k_11008x4096"])
def test_workload_full_parity(name):
    wl = syn.make_workload(name)
    M, K = wl["M"], wl["K"]
    y = _run(wl["wtype"], wl["W"][0], wl["X"], M, K)
    Y, B = ora.matmul(wl["wtype"], wl["W"][0], wl["X"], M, K)
    assert_within_bound(y, Y[0], B[0], name)


@pytest.mark.parametrize("wtype", ["q4_k", "q6_k"])
@pytest.mark.parametrize("M,K", [(1, 256), (17, 512), (37, 11008), (300, 4096), (1000, 2304), (33, 65536)])
def test_ragged_shapes(wtype, M, K):
    if wtype == "q6_k" and K == 65536:
        K = 14336                                    # Q6_K rows of 16-byte multiples
    rng = np.random.default_rng(M * 7 + K)
    W = syn.weights(wtype, rng, M, K)
    x = syn.activations(rng, K, 1)
    y = _run(wtype, W, x, M, K)
    Y, B = ora.matmul(wtype, W, x, M, K)
    assert_within_bound(y, Y[0], B[0], f"{wtype} {M}x{K}")


def test_q6k_ragged_tail_bytes():
    # 43 Q6_K blocks per row = 9030 bytes: rows are not 16-byte multiples, so
    # each CTA's copies start up to 14 bytes before its first row (one row per
    # CTA here: every even offset occurs) and the last copy ends in a <16-byte
    # tail copied by the producer thread.
    M, K = 45, 11008
    rng = np.random.default_rng(5)
    W = syn.q6_k_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    y = _run("q6_k", W, x, M, K)
    Y, B = ora.matmul("q6_k", W, x, M, K)
    assert_within_bound(y, Y[0], B[0], "q6_k tail")


def test_min_term_form_agrees_on_workload_rows():
    wl = syn.make_workload("decode_q4k_4096x11008")
    rows = np.arange(0, 4096, 97)
    y = _run("q4_k", wl["W"][0], wl["X"], 4096, 11008)
    y_min = ora.q4_k_min_term_matvec(wl["W"][0][rows], wl["X"][0], 11008)
    _, B = ora.matmul_rows("q4_k", wl["W"][0], wl["X"], 11008, rows)
    assert_within_bound(y[rows], y_min, B[0], "min-term rows")


def test_deterministic():
    wl = syn.make_workload("decode_q4k_11008x4096")
    a = _run("q4_k", wl["W"][0], wl["X"], 11008, 4096)
    b = _run("q4_k", wl["W"][0], wl["X"], 11008, 4096)
    assert np.array_equal(a, b)


def test_zero_activation_gives_zero():
    M, K = 64, 1024
    W = syn.q4_k_weights(np.random.default_rng(1), M, K)
    y = _run("q4_k", W, np.zeros((1, K), np.float32), M, K)
    assert np.all(y == 0)


@pytest.mark.parametrize("M,K", [(4096, 14336), (14336, 4096)])
def test_ring_staging_shapes_sampled_rows(M, K):
    # Row ranges too large to stage whole take the ring form of the lane-row
    # kernel (chunk slots refilled as they are consumed); rows at CTA range
    # boundaries and the ragged end are among the sampled ones.
    rng = np.random.default_rng(M + K)
    W = syn.q4_k_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    y = _run("q4_k", W, x, M, K)
    R = -(-M // 152)
    rows = np.unique(np.concatenate([rng.choice(M, 160, replace=False), [0, R - 1, R, M - 1],
                                     np.arange(R * 150, M)]))
    Yr, B = ora.matmul_rows("q4_k", W, x, K, rows)
    assert_within_bound(y[rows], Yr[0], B[0], f"ring {M}x{K}")
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("wtype,M,K", [
    ("q4_k", 256, 102400),    # item kernel, 3 ring slots for up to 8 chunks per CTA
    ("q6_k", 304, 102400),    # item kernel, 3 slots
    ("q6_k", 304, 102144),    # item kernel, 3 slots; rows of 399 blocks (83790 B), so CTA
                              # ranges start off 16-byte boundaries
    ("q4_k", 4560, 49152),    # lane-row ring form with 2 slots of 5-block chunks
])
def test_shallow_rings_sampled_rows(wtype, M, K):
    # Rings much shallower than the distance the consumers can run ahead: a
    # consumer must never take an older fill of its chunk's slot (same barrier
    # parity) for its chunk, and no copy may still be in flight when a CTA ends.
    rng = np.random.default_rng(M + K)
    W = syn.weights(wtype, rng, M, K)
    x = syn.activations(rng, K, 1)
    y = _run(wtype, W, x, M, K)
    rows = np.unique(np.concatenate([rng.choice(M, 128, replace=False), [0, 1, M - 2, M - 1]]))
    Yr, B = ora.matmul_rows(wtype, W, x, K, rows)
    assert_within_bound(y[rows], Yr[0], B[0], f"shallow ring {wtype} {M}x{K}")
    assert np.all(np.isfinite(y))


def test_prefetch_call_is_bit_identical():
    # kq_matvec_prefetch only adds an L2 prefetch of the next call's weights.
    import torch
    from quantized_weight_matmul_q4_gb300 import kq_matvec_prefetch
    for wtype, name in [("q4_k", "decode_q4k_4096x11008"), ("q5_k", "decode_q5k_11008x4096"),
                        ("q6_k", "decode_q6k_4096x11008"), ("tq4_1s", "decode_tq4_1s_3584x18944")]:
        wl = syn.make_workload(name, copies=2)
        M, K = wl["M"], wl["K"]
        W = to_dev(wl["W"][0], torch)
        W_next = to_dev(wl["W"][1], torch)
        x = to_dev(wl["X"].reshape(-1), torch)
        a = kq_matvec(wtype, W, x, M, K)
        b = kq_matvec_prefetch(wtype, W, x, M, K, W_next=W_next)
        c = kq_matvec_prefetch(wtype, W, x, M, K, W_next=None)
        torch.cuda.synchronize()
        assert torch.equal(a, b) and torch.equal(a, c), wtype


def test_largest_k_for_many_rows():
    # Many rows (more than a CTA of the staged kernel takes) put the activations
    # and two ring slots in one CTA's shared memory: K = 121600 is the largest K
    # that fits; the next multiple of 256 is refused before any launch.
    import torch
    import quantized_weight_matmul_q4_gb300 as kq
    M, K = 20000, 121600
    rng = np.random.default_rng(9)
    W = syn.q4_k_weights(rng, M, K)
    x = syn.activations(rng, K, 1)
    Wd = to_dev(W, torch)
    y = kq_matvec("q4_k", Wd, to_dev(x.reshape(-1), torch), M, K).cpu().numpy()
    rows = np.unique(np.concatenate([rng.choice(M, 48, replace=False), [0, M - 1]]))
    Yr, B = ora.matmul_rows("q4_k", W, x, K, rows)
    assert_within_bound(y[rows], Yr[0], B[0], "q4_k 20000x121600")
    K2 = K + 256
    W2 = torch.zeros((M, (K2 // 256) * 144), dtype=torch.uint8, device="cuda")
    with pytest.raises(kq.KQError):
        kq_matvec("q4_k", W2, torch.zeros(K2, device="cuda"), M, K2)
