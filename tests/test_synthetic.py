"""The seeded generators place fields where the formats put them and draw the
stated distributions ("06 · 8e/8e② — decode MMVQ", §3.3 Pitfalls: a Q6_K
generator that wrote d at byte 0 once passed for a kernel bug)."""
import numpy as np

from quantized_weight_matmul_q4_gb300 import synthetic as syn


def _f16(b2):
    return b2.copy().view(np.uint16).view(np.float16).astype(np.float64)


def test_q4k_generator_fields():
    W = syn.q4_k_weights(np.random.default_rng(0), 64, 1024)
    assert W.shape == (64, 4 * 144) and W.dtype == np.uint8
    blk = W.reshape(64, 4, 144)
    d = _f16(blk[..., 0:2]).ravel()
    dmin = _f16(blk[..., 2:4]).ravel()
    assert np.all(d >= 0) and np.all(dmin >= 0)
    assert 0.005 < d.mean() < 0.011 and 0.005 < dmin.mean() < 0.011   # E|N(0,.01)| = 0.008
    # packed scales and nibbles are uniform bytes: all 256 values occur
    assert len(np.unique(blk[..., 4:144])) == 256


def test_q6k_generator_fields_and_d_offset():
    W = syn.q6_k_weights(np.random.default_rng(1), 64, 512)
    assert W.shape == (64, 2 * 210)
    blk = W.reshape(64, 2, 210)
    sc = blk[..., 192:208].view(np.int8)
    assert sc.min() >= -64 and sc.max() <= 63 and sc.min() < -60 and sc.max() > 60
    d = _f16(blk[..., 208:210]).ravel()
    assert np.all(d >= 0) and 0.005 < d.mean() < 0.011
    # bytes 0..1 are ql codes (uniform), not the scale
    lead = _f16(blk[..., 0:2]).ravel()
    assert not (0.005 < np.abs(lead[np.isfinite(lead)]).mean() < 0.011)


def test_q5k_generator_fields():
    W = syn.q5_k_weights(np.random.default_rng(4), 64, 512)
    assert W.shape == (64, 2 * 176) and W.dtype == np.uint8
    blk = W.reshape(64, 2, 176)
    d = _f16(blk[..., 0:2]).ravel()
    dmin = _f16(blk[..., 2:4]).ravel()
    assert np.all(d >= 0) and np.all(dmin >= 0)
    assert 0.005 < d.mean() < 0.011 and 0.005 < dmin.mean() < 0.011
    assert len(np.unique(blk[..., 4:176])) == 256   # scales, qh, qs: uniform bytes


def test_tq4_1s_generator_fields():
    W = syn.tq4_1s_weights(np.random.default_rng(3), 32, 4096)
    assert W.shape == (32, 128 * 20) and W.dtype == np.uint8
    blk = W.reshape(32, 128, 20)
    d = _f16(blk[..., 0:4].reshape(32, 128, 2, 2)).ravel()
    assert np.all(d > 0) and 0.018 < np.median(d) < 0.022            # 0.02 * exp(0.25 N(0,1))
    lo, hi = blk[..., 4:20] & 0xF, blk[..., 4:20] >> 4
    idx = np.concatenate([lo.ravel(), hi.ravel()])
    counts = np.bincount(idx, minlength=16)
    assert np.all(counts > 0)                                        # every index occurs
    assert counts[7] + counts[8] > 5 * (counts[0] + counts[15])      # bell-shaped, symmetric
    assert abs(int(counts[:8].sum()) - int(counts[8:].sum())) < 0.02 * idx.size


def test_activations_and_ids():
    X = syn.activations(np.random.default_rng(2), 4096, 8)
    assert X.shape == (8, 4096) and X.dtype == np.float32
    assert abs(X.mean()) < 0.05 and abs(X.std() - 1) < 0.05
    ids = syn.expert_ids(np.random.default_rng(3), 1024, 128, 8)
    assert ids.shape == (1024, 8) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < 128
    assert all(len(set(r)) == 8 for r in ids.tolist())
    counts = np.bincount(ids.ravel(), minlength=128)
    assert counts.sum() == 8192 and counts.min() > 20 and counts.max() < 130


def test_workloads_are_reproducible():
    a = syn.make_workload("matvec_q4k_512x2048")
    b = syn.make_workload("matvec_q4k_512x2048", copies=2)
    assert np.array_equal(a["W"][0], b["W"][0]) and not np.array_equal(b["W"][0], b["W"][1])
    assert np.array_equal(a["X"], b["X"])
    assert a["W"][0].shape == (512, 8 * 144) and a["X"].shape == (1, 2048)
