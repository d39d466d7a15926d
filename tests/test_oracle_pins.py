"""Pins for the CPU oracle: each test ties an oracle function to something other
than itself (hand-built blocks with closed-form values, the IEEE-754 definition
checked by brute force, invariants of the quantiser, a second formulation of the
product, brute force on tiny shapes).

Sources: "06 · 8e/8e② — decode MMVQ: dp4a integer dot products + the llama.cpp
launch table" (§2 Principle, §3.2 Key code, §3.3 Pitfalls) and "ZINC MMQ v2 —
Fused Q4_K×Q8_1 Tensor-Core GEMM" (MoE routing, Correctness gate).
"""
import itertools
import math

import numpy as np
import pytest

from oracle import kq_oracle as ora
from quantized_weight_matmul_q4_gb300 import synthetic as syn


# ----------------------------------------------------------------------------
# fp16 fields against the IEEE-754 binary16 definition
# ----------------------------------------------------------------------------
def _binary16_value(bits: int) -> float:
    """Value of a binary16 pattern from the definition (sign, 5-bit biased
    exponent, 10-bit fraction; exponent 0 is subnormal)."""
    s = -1.0 if bits >> 15 else 1.0
    e = (bits >> 10) & 31
    f = bits & 1023
    if e == 31:
        return s * math.inf if f == 0 else math.nan
    if e == 0:
        return s * f * 2.0 ** -24
    return s * (1 + f / 1024) * 2.0 ** (e - 15)


def test_fp16_decode_every_pattern_matches_definition():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = ora.fp16_to_f64(bits)
    want = np.array([_binary16_value(int(b)) for b in range(65536)])
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(np.isinf(got), np.isinf(want))


def test_fp16_encode_is_nearest_even_by_brute_force():
    # All finite non-negative binary16 values, ascending.
    pos = np.array([_binary16_value(b) for b in range(0x7C00)])
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(0, 65504, 2000), rng.uniform(0, 1, 2000),
        rng.uniform(0, 2 ** -13, 2000),                     # subnormal range
        (pos[:-1] + pos[1:]) / 2,                           # every tie
    ]).astype(np.float32)
    got = ora.f32_to_fp16_bits(x)
    xf = x.astype(np.float64)
    idx = np.searchsorted(pos, xf)                          # pos[idx-1] < x <= pos[idx]
    idx = np.clip(idx, 1, len(pos) - 1)
    lo, hi = idx - 1, idx
    dlo, dhi = xf - pos[lo], pos[hi] - xf
    pick = np.where(dlo < dhi, lo, hi)
    tie = dlo == dhi
    pick = np.where(tie, np.where(lo % 2 == 0, lo, hi), pick)   # even fraction wins
    exact = pos[np.clip(np.searchsorted(pos, xf), 0, len(pos) - 1)] == xf
    pick = np.where(exact, np.searchsorted(pos, xf), pick)
    assert np.array_equal(got.astype(np.int64), pick)


def test_fp16_encode_literal_ties():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10: ties to the even 1.0 (0x3C00).
    # 1 + 3*2^-11 is halfway between 1 + 2^-10 and 1 + 2^-9: goes to 0x3C02.
    x = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 65504.0, 2.0 ** -24, 2.0 ** -25], np.float32)
    assert [int(b) for b in ora.f32_to_fp16_bits(x)] == [0x3C00, 0x3C02, 0x7BFF, 0x0001, 0x0000]


# ----------------------------------------------------------------------------
# Q4_K: a hand-built super-block with closed-form weights
# ----------------------------------------------------------------------------
# sub-block scales and mins chosen so that j >= 4 exercises the high-bit fields
Q4K_SC = [1, 2, 3, 4, 37, 46, 55, 63]
Q4K_M = [0, 5, 10, 63, 17, 34, 51, 60]
# the 12 packed bytes, worked out by hand from the GGUF packing:
#   S[0..3] = sc0..3 | (sc4..7 bits 4-5) << 6   -> 1|2<<6, 2|2<<6, 3|3<<6, 4|3<<6
#   S[4..7] = m0..3  | (m4..7  bits 4-5) << 6   -> 0|1<<6, 5|2<<6, 10|3<<6, 63|3<<6
#   S[8..11] = (sc4..7 & 15) | (m4..7 & 15) << 4 -> 5|1<<4, 14|2<<4, 7|3<<4, 15|12<<4
Q4K_SCALE_BYTES = [129, 130, 195, 196, 64, 133, 202, 255, 21, 46, 55, 207]


def _q4k_nib(j, i):
    """Closed-form nibble used by the hand-built block for sub-block j, element i."""
    return (i + 3 * j) % 16 if j % 2 == 0 else (15 - i - j) % 16


def _q4k_block(d_bits=0x3C00, dmin_bits=0x3800):
    blk = np.zeros(144, np.uint8)
    blk[0], blk[1] = d_bits & 255, d_bits >> 8          # d    = 1.0
    blk[2], blk[3] = dmin_bits & 255, dmin_bits >> 8    # dmin = 0.5
    blk[4:16] = Q4K_SCALE_BYTES
    for c in range(4):                                   # 32-byte chunk c: sub 2c low, 2c+1 high
        for i in range(32):
            blk[16 + 32 * c + i] = _q4k_nib(2 * c, i) | (_q4k_nib(2 * c + 1, i) << 4)
    return blk


def test_q4k_scale_min_unpack_hand_block():
    sc, m = ora.q4_k_scale_min(np.array(Q4K_SCALE_BYTES, np.uint8))
    assert sc.tolist() == Q4K_SC
    assert m.tolist() == Q4K_M


def test_q4k_dequant_hand_block_closed_form():
    blk = _q4k_block()
    w = ora.q4_k_dequant(blk.reshape(1, 144), 256)[0]
    want = [1.0 * Q4K_SC[j] * _q4k_nib(j, i) - 0.5 * Q4K_M[j] for j in range(8) for i in range(32)]
    assert w.tolist() == want


def test_q4k_d_and_dmin_not_swapped():
    # d = 2, dmin = 0: every weight is 2*sc*nib; d = 0, dmin = 2: every weight is -2*m.
    w = ora.q4_k_dequant(_q4k_block(0x4000, 0x0000).reshape(1, 144), 256)[0]
    assert w.tolist() == [2.0 * Q4K_SC[j] * _q4k_nib(j, i) for j in range(8) for i in range(32)]
    w = ora.q4_k_dequant(_q4k_block(0x0000, 0x4000).reshape(1, 144), 256)[0]
    assert w.tolist() == [-2.0 * Q4K_M[j] for j in range(8) for i in range(32)]


def test_q4k_multi_block_rows_keep_block_order():
    # two rows x two blocks; each block gets a distinct d so a wrong row or
    # block stride shows up.
    blocks = [_q4k_block(d_bits=b, dmin_bits=0) for b in (0x3C00, 0x4000, 0x4200, 0x4400)]  # 1,2,3,4
    W = np.concatenate(blocks).reshape(2, 2 * 144)
    w = ora.q4_k_dequant(W, 512)
    base = np.array([Q4K_SC[j] * _q4k_nib(j, i) for j in range(8) for i in range(32)], float)
    assert np.array_equal(w[0, :256], 1 * base) and np.array_equal(w[0, 256:], 2 * base)
    assert np.array_equal(w[1, :256], 3 * base) and np.array_equal(w[1, 256:], 4 * base)


# ----------------------------------------------------------------------------
# Q6_K: hand-built blocks
# ----------------------------------------------------------------------------
def _q6k_code(e):
    return (7 * e + 3) % 64


def _q6k_block(d_bits=0x4000):
    """Places the closed-form codes _q6k_code(e) bit by bit (GGUF arrangement)."""
    blk = np.zeros(210, np.uint8)
    for e in range(256):
        h, g, r = e // 128, (e % 128) // 32, e % 32
        q = _q6k_code(e)
        lo, hi = q & 15, q >> 4
        pos = 64 * h + 32 * (g & 1) + r
        blk[pos] |= lo if g < 2 else lo << 4
        blk[128 + 32 * h + r] |= hi << (2 * g)
    blk[192:208] = (np.arange(16) - 8).astype(np.int8).view(np.uint8)   # scales -8..7
    blk[208], blk[209] = d_bits & 255, d_bits >> 8                       # d = 2.0
    return blk


def test_q6k_dequant_hand_block_closed_form():
    w = ora.q6_k_dequant(_q6k_block().reshape(1, 210), 256)[0]
    want = [2.0 * (e // 16 - 8) * (_q6k_code(e) - 32) for e in range(256)]
    assert w.tolist() == want


def test_q6k_d_is_read_at_offset_208():
    # codes all 0 (so q - 32 = -32), scales all 1, d = 1.0 stored at byte 208,
    # bytes 0..1 (where a wrong reader would look) are zero.
    blk = np.zeros(210, np.uint8)
    blk[192:208] = 1
    blk[208], blk[209] = 0x00, 0x3C
    w = ora.q6_k_dequant(blk.reshape(1, 210), 256)[0]
    assert w.tolist() == [-32.0] * 256


# ----------------------------------------------------------------------------
# Q8_1 quantiser
# ----------------------------------------------------------------------------
def _rand_x(seed, N, K, scale=1.0):
    return (np.random.default_rng(seed).standard_normal((N, K)) * scale).astype(np.float32)


def test_q8_1_invariants_random():
    X = np.concatenate([_rand_x(1, 6, 1024), _rand_x(2, 2, 1024, 1e-3), _rand_x(3, 2, 1024, 300.0)])
    q, d_h, s_h = ora.quantize_q8_1(X)
    xb = X.reshape(X.shape[0], -1, 32).astype(np.float64)
    qi = q.astype(np.int64)
    amax = np.abs(xb).max(-1)
    d32 = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    assert np.abs(qi).max() <= 127
    # the largest |x| of each block maps to +-127
    arg = np.abs(xb).argmax(-1)
    assert np.all(np.abs(np.take_along_axis(qi, arg[..., None], -1)) == 127)
    # the sign is kept (or the code is 0)
    assert np.all((qi == 0) | (np.sign(qi) == np.sign(xb)))
    # reconstruction error at most half a step (plus fp32 rounding of 1/d and x/d)
    assert np.all(np.abs(xb - d32[..., None] * qi) <= d32[..., None] * (0.5 + 1e-6))
    # the stored scale is fp16(d); the block sum is fp16(d_h * Sum q) to half an ulp
    assert np.array_equal(d_h, d32.astype(np.float16).view(np.uint16))
    s_exact = ora.fp16_to_f64(d_h) * qi.sum(-1)
    s = ora.fp16_to_f64(s_h)
    ulp = np.spacing(np.abs(s_exact).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(s - s_exact) <= ulp / 2)


def test_q8_1_zero_block():
    X = np.zeros((1, 64), np.float32)
    X[0, 32:] = _rand_x(4, 1, 32)[0]
    q, d_h, s_h = ora.quantize_q8_1(X)
    assert np.all(q[0, 0] == 0) and d_h[0, 0] == 0 and s_h[0, 0] == 0
    assert d_h[0, 1] != 0


def test_q8_1_reciprocal_overflow_block_is_zero():
    # amax below ~3.7e-37: 1/d overflows fp32 and d_h = fp16(d) = 0, so the
    # block dequantises to 0 whatever the codes; the codes are taken as 0. Just
    # above the threshold 1/d is finite and the block quantises as usual.
    X = np.zeros((1, 128), np.float32)
    X[0, :32] = np.linspace(-1, 1, 32) * np.float32(1e-38)      # subnormal amax
    X[0, 32:64] = np.linspace(-1, 1, 32) * np.float32(3.0e-37)  # d ~ 2.4e-39: 1/d = inf
    X[0, 64:96] = np.linspace(-1, 1, 32) * np.float32(5.0e-37)  # d ~ 3.9e-39: 1/d finite
    X[0, 96:] = _rand_x(8, 1, 32)[0]
    d = (np.abs(X.reshape(4, 32)).max(-1) / np.float32(127)).astype(np.float32)
    with np.errstate(over="ignore"):
        assert np.isinf(np.float32(1) / d[1]) and np.isfinite(np.float32(1) / d[2])
    q, d_h, s_h = ora.quantize_q8_1(X)
    assert np.all(q[0, :2] == 0) and np.all(d_h[0, :3] == 0) and np.all(s_h[0, :3] == 0)
    assert q[0, 2].tolist() == ora.quantize_q8_1(X[:, 64:96] * np.float32(2.0 ** 100))[0][0, 0].tolist()
    assert np.abs(q[0, 2]).max() == 127


def test_q8_1_unit_scale_block_is_round_half_even():
    # amax = 127 gives d = 1 and di = 1, so q = rint(x): round half to even.
    x = [127, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.49, -3.51, 126.5, -126.5, 0.49999997,
         10.5, 11.5, -10.5, 0, 7, -7, 99.5, 100.5, 0.25, 64.5, 65.5, -64.5,
         1, 2, 3, 4, 5, 6, 8.5, 9.5]
    q, d_h, s_h = ora.quantize_q8_1(np.array([x], np.float32))
    want = [127, 0, 2, 2, 0, -2, -2, 3, -4, 126, -126, 0,
            10, 12, -10, 0, 7, -7, 100, 100, 0, 64, 66, -64,
            1, 2, 3, 4, 5, 6, 8, 10]
    assert q[0, 0].tolist() == want
    assert d_h[0, 0] == 0x3C00
    assert ora.fp16_to_f64(s_h[0, 0]) == float(sum(want))


def test_q8_1_power_of_two_scaling_keeps_codes():
    X = _rand_x(5, 3, 512)
    q0, d0, _ = ora.quantize_q8_1(X)
    for k in (-4, 3, 6):
        qk, dk, _ = ora.quantize_q8_1((X * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(q0, qk)
        assert np.array_equal(ora.fp16_to_f64(dk), ora.fp16_to_f64(d0) * 2.0 ** k)


def test_q8_1_pack_layout():
    X = _rand_x(6, 2, 64)
    q, d_h, s_h = ora.quantize_q8_1(X)
    b = ora.pack_q8_1(q, d_h, s_h)
    assert b.shape == (2, 2, 36)
    assert int(b[1, 1, 0]) | int(b[1, 1, 1]) << 8 == int(d_h[1, 1])
    assert int(b[1, 1, 2]) | int(b[1, 1, 3]) << 8 == int(s_h[1, 1])
    assert b[1, 1, 4:].view(np.int8).tolist() == q[1, 1].tolist()


# ----------------------------------------------------------------------------
# Matmul
# ----------------------------------------------------------------------------
def _q4k_random(seed, M, K):
    rng = np.random.default_rng(seed)
    W = rng.integers(0, 256, (M, K // 256, 144), dtype=np.uint8)
    W[..., 0:4] = np.abs(rng.standard_normal((M, K // 256, 2)) * 0.01).astype(np.float16).view(np.uint8).reshape(M, K // 256, 4)
    return W.reshape(M, -1)


def _q6k_random(seed, M, K):
    rng = np.random.default_rng(seed)
    W = rng.integers(0, 256, (M, K // 256, 210), dtype=np.uint8)
    W[..., 192:208] = rng.integers(-64, 64, (M, K // 256, 16)).astype(np.int8).view(np.uint8)
    W[..., 208:210] = np.abs(rng.standard_normal((M, K // 256, 1)) * 0.01).astype(np.float16).view(np.uint8)
    return W.reshape(M, -1)


def test_matmul_one_hot_picks_a_weight_column():
    # x = 127 * e_k quantises to q = 127 e_k with d = 1, so y[m] = 127 * w[m, k].
    W = np.concatenate([_q4k_block(), _q4k_block(0x4000, 0x3C00)]).reshape(1, 288)
    for k in (0, 37, 255, 256, 300, 511):
        x = np.zeros((1, 512), np.float32)
        x[0, k] = 127.0
        Y, B = ora.matmul("q4_k", W, x, 1, 512)
        j, i = (k % 256) // 32, k % 32
        if k < 256:
            want = 1.0 * Q4K_SC[j] * _q4k_nib(j, i) - 0.5 * Q4K_M[j]
        else:
            want = 2.0 * Q4K_SC[j] * _q4k_nib(j, i) - 1.0 * Q4K_M[j]
        assert Y[0, 0] == 127 * want
        assert B[0, 0] == abs(127 * want)


def test_matmul_q6k_one_hot():
    W = _q6k_block().reshape(1, 210)
    for k in (0, 15, 16, 100, 128, 255):
        x = np.zeros((1, 256), np.float32)
        x[0, k] = -127.0
        Y, _ = ora.matmul("q6_k", W, x, 1, 256)
        assert Y[0, 0] == -127 * 2.0 * (k // 16 - 8) * (_q6k_code(k) - 32)


@pytest.mark.parametrize("wtype", ["q4_k", "q6_k", "q5_k"])
def test_matmul_brute_force_tiny(wtype):
    M, N, K = 3, 4, 512
    W = syn.weights(wtype, np.random.default_rng(11), M, K)
    X = _rand_x(12, N, K)
    Y, B = ora.matmul(wtype, W, X, M, K)
    w = ora.dequant(wtype, W, K)
    q, d_h, _ = ora.quantize_q8_1(X)
    xh = ora.q8_1_dequant(q, d_h)
    for n, m in itertools.product(range(N), range(M)):
        acc = 0.0
        bnd = 0.0
        for k in range(K):
            acc += w[m, k] * xh[n, k]
            bnd += abs(w[m, k] * xh[n, k])
        assert abs(Y[n, m] - acc) <= 1e-12 * bnd
        assert abs(B[n, m] - bnd) <= 1e-12 * bnd


def test_min_term_identity_matches_direct_product():
    M, K = 16, 1024
    W = _q4k_random(21, M, K)
    x = _rand_x(22, 1, K)
    y_min = ora.q4_k_min_term_matvec(W, x[0], K)
    Y, B = ora.matmul("q4_k", W, x, M, K)
    assert np.all(np.abs(y_min - Y[0]) <= 1e-12 * B[0])


def test_matmul_rows_matches_full():
    M, N, K = 8, 3, 512
    W = _q4k_random(31, M, K)
    X = _rand_x(32, N, K)
    Y, B = ora.matmul("q4_k", W, X, M, K)
    rows = np.array([6, 1, 3])
    Yr, Br = ora.matmul_rows("q4_k", W, X, K, rows)
    assert np.array_equal(Yr, Y[:, rows]) and np.array_equal(Br, B[:, rows])


# ----------------------------------------------------------------------------
# MoE
# ----------------------------------------------------------------------------
def test_moe_buckets_are_a_stable_permutation():
    rng = np.random.default_rng(41)
    T, top_k, E = 37, 4, 9
    ids = np.stack([rng.permutation(E)[:top_k] for _ in range(T)]).astype(np.int32)
    counts, offsets, entries = ora.moe_buckets(ids, E)
    assert counts.sum() == T * top_k and offsets[-1] == T * top_k
    assert sorted(entries.tolist()) == list(range(T * top_k))
    flat = ids.reshape(-1)
    for e in range(E):
        seg = entries[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)          # token order, then slot order
    with pytest.raises(ValueError):
        ora.moe_buckets(np.array([[0, E]]), E)


def test_moe_equals_dense_per_slot():
    E, M, K, T, top_k = 5, 4, 256, 6, 2
    W = _q4k_random(51, E * M, K)
    X = _rand_x(52, T, K)
    rng = np.random.default_rng(53)
    ids = np.stack([rng.permutation(E)[:top_k] for _ in range(T)]).astype(np.int32)
    Y, B = ora.moe("q4_k", W, ids, X, E, M, K)
    for t in range(T):
        for j in range(top_k):
            e = ids[t, j]
            Yd, Bd = ora.matmul("q4_k", W[e * M:(e + 1) * M], X[t:t + 1], M, K)
            assert np.array_equal(Y[t, j], Yd[0]) and np.array_equal(B[t, j], Bd[0])


# ----------------------------------------------------------------------------
# Producers (RMSNorm, SwiGLU) and the MoE combine
# ----------------------------------------------------------------------------
def test_rms_norm_constant_row_and_unit_mean_square():
    K = 64
    gamma = np.linspace(0.5, 2.0, K)
    # a constant row c: mean square c^2, so the result is c / sqrt(c^2 + eps) * gamma
    y = ora.rms_norm(np.full((1, K), -3.0), gamma, 0.0)
    assert np.allclose(y[0], -gamma, rtol=0, atol=1e-15)
    y = ora.rms_norm(np.full((1, K), 2.0), gamma, 5.0)
    assert np.allclose(y[0], 2.0 / 3.0 * gamma, rtol=0, atol=1e-15)
    # with gamma = 1 and eps = 0 every row has mean square exactly 1 (up to rounding)
    rng = np.random.default_rng(71)
    X = rng.standard_normal((5, 257)) * rng.uniform(0.1, 10.0, size=(5, 1))
    y = ora.rms_norm(X, np.ones(257), 0.0)
    assert np.allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-13)


def test_rms_norm_is_scale_invariant_and_row_wise():
    rng = np.random.default_rng(72)
    X = rng.standard_normal((3, 96))
    g = rng.standard_normal(96)
    a = ora.rms_norm(X, g, 0.0)
    assert np.allclose(ora.rms_norm(7.5 * X, g, 0.0), a, rtol=1e-13)
    assert np.allclose(ora.rms_norm(X[1:2], g, 0.0), a[1:2], rtol=0, atol=0)


def test_swiglu_special_values_and_odd_part():
    g = np.array([0.0, 40.0, -40.0, 1.0])
    u = np.array([3.0, 2.0, 5.0, 1.0])
    y = ora.swiglu(g, u)
    assert y[0] == 0.0
    assert abs(y[1] - 80.0) < 1e-12 and abs(y[2]) < 1e-15
    assert abs(y[3] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    # silu(g) - silu(-g) = g for every g (sigma(g) + sigma(-g) = 1)
    rng = np.random.default_rng(73)
    g = rng.standard_normal(1000) * 5
    ones = np.ones_like(g)
    assert np.allclose(ora.swiglu(g, ones) - ora.swiglu(-g, ones), g, rtol=1e-12, atol=1e-12)


def test_moe_combine_one_hot_mean_and_linearity():
    rng = np.random.default_rng(74)
    T, top_k, M = 6, 4, 9
    Y = rng.standard_normal((T, top_k, M))
    pick = rng.integers(0, top_k, size=T)
    onehot = np.eye(top_k)[pick]
    assert np.array_equal(ora.moe_combine(Y, onehot), Y[np.arange(T), pick])
    assert np.allclose(ora.moe_combine(Y, np.full((T, top_k), 1.0 / top_k)), Y.mean(axis=1), rtol=1e-14)
    p1, p2 = rng.uniform(size=(T, top_k)), rng.uniform(size=(T, top_k))
    assert np.allclose(ora.moe_combine(Y, p1 + p2), ora.moe_combine(Y, p1) + ora.moe_combine(Y, p2), rtol=1e-13)


def test_moe_combine_equals_matmul_with_the_weighted_weights():
    # Sum_j p_j (W_{e_j} . x_hat) = (Sum_j p_j W_{e_j}) . x_hat
    E, M, K, T, top_k = 4, 3, 256, 5, 2
    W = _q4k_random(75, E * M, K)
    X = _rand_x(76, T, K)
    rng = np.random.default_rng(77)
    ids = np.stack([rng.permutation(E)[:top_k] for _ in range(T)]).astype(np.int32)
    probs = rng.uniform(size=(T, top_k))
    Y, _ = ora.moe("q4_k", W, ids, X, E, M, K)
    out = ora.moe_combine(Y, probs)
    w = ora.dequant("q4_k", W, K).reshape(E, M, K)
    q, d_h, _ = ora.quantize_q8_1(X)
    xh = ora.q8_1_dequant(q, d_h)
    for t in range(T):
        weff = sum(probs[t, j] * w[ids[t, j]] for j in range(top_k))
        assert np.allclose(out[t], weff @ xh[t], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# Q5_K (GGUF layout, a reading: the pages give none): the Q4_K value with a
# fifth bit, so it reduces to Q4_K exactly when every high bit is zero
# ----------------------------------------------------------------------------
def _q5k_from_q4k(q4: np.ndarray, qh: np.ndarray) -> np.ndarray:
    """Q5_K blocks holding the fields of Q4_K blocks q4 [..., 144] and the high-bit bytes qh [..., 32]."""
    out = np.zeros(q4.shape[:-1] + (176,), np.uint8)
    out[..., 0:16] = q4[..., 0:16]
    out[..., 16:48] = qh
    out[..., 48:176] = q4[..., 16:144]
    return out


def test_q5k_with_zero_high_bits_is_q4k():
    M, K = 5, 768
    q4 = syn.q4_k_weights(np.random.default_rng(31), M, K).reshape(M, K // 256, 144)
    q5 = _q5k_from_q4k(q4, np.zeros(q4.shape[:-1] + (32,), np.uint8)).reshape(M, -1)
    assert np.array_equal(ora.q5_k_dequant(q5, K), ora.q4_k_dequant(q4.reshape(M, -1), K))


def test_q5k_all_high_bits_add_16_d_sc():
    M, K = 4, 512
    q4 = syn.q4_k_weights(np.random.default_rng(32), M, K).reshape(M, K // 256, 144)
    q5 = _q5k_from_q4k(q4, np.full(q4.shape[:-1] + (32,), 0xFF, np.uint8)).reshape(M, -1)
    d, _, sc, _, _ = ora.q4_k_fields(q4)
    extra = (16 * d[..., None, None] * sc[..., None] * np.ones(32)).reshape(M, K)
    assert np.allclose(ora.q5_k_dequant(q5, K), ora.q4_k_dequant(q4.reshape(M, -1), K) + extra, rtol=0, atol=1e-12)


@pytest.mark.parametrize("j,r", [(0, 0), (1, 5), (4, 31), (7, 17)])
def test_q5k_one_high_bit_moves_one_weight(j, r):
    # bit j of qh[r] is the fifth bit of weight r of sub-block j, i.e. element 32 j + r
    q4 = _q4k_block()
    qh = np.zeros(32, np.uint8)
    base = ora.q5_k_dequant(_q5k_from_q4k(q4, qh).reshape(1, 176), 256)[0]
    qh[r] = 1 << j
    moved = ora.q5_k_dequant(_q5k_from_q4k(q4, qh).reshape(1, 176), 256)[0]
    diff = moved - base
    want = np.zeros(256)
    want[32 * j + r] = 16 * 1.0 * Q4K_SC[j]          # d = 1.0 in the hand block
    assert np.array_equal(diff, want)


def test_q5k_hand_block_closed_form():
    # the Q4_K hand block with fifth bits (i + j) % 3 == 0
    qh = np.zeros(32, np.uint8)
    for i in range(32):
        for j in range(8):
            if (i + j) % 3 == 0:
                qh[i] |= 1 << j
    w = ora.q5_k_dequant(_q5k_from_q4k(_q4k_block(), qh).reshape(1, 176), 256)[0]
    want = [1.0 * Q4K_SC[j] * (_q4k_nib(j, i) + (16 if (i + j) % 3 == 0 else 0)) - 0.5 * Q4K_M[j]
            for j in range(8) for i in range(32)]
    assert w.tolist() == want
