"""Weight matrices whose matvec exposes the activation's Q8_1 codes one by one.

The fused quantisers of the decode kernels never write their Q8_1 codes to
memory. These matrices make each code and each block sum appear alone in one
output element, as an exact fp32 value:

* code row k (one per activation element):  w = e_k, so y = d_h * q_k;
* sum row g (one per 32-block):              w = -1 on block g, so y = -d_h * Sum q;
* Q6_K half-sum row h (one per 16 values):   w = +1 on those 16, so y = d_h * Sum q.

Every product and partial sum involved is exact in fp32 (an fp16 scale times an
integer of at most 12 bits), and every other term a kernel adds is an exact
zero, so any correct kernel returns these values bit for bit. A code that is
off by one, a scale rounded from the wrong value or a wrong block sum changes
an output.

The matrices are built from the block layouts ("06 · 8e/8e② — decode MMVQ",
§3.2 Key code for Q4_K, §3.3 Pitfalls for Q6_K; the GGUF reading for the
scale/min packing and for Q5_K). ``tests/test_onehot_pins.py`` checks, on the
CPU, that the oracle's own dequantisation of them is the matrix described
above.
"""
import numpy as np

ONE_FP16 = (0x00, 0x3C)   # fp16 1.0, little-endian


def _kquant_rows(K: int, bb: int, qs_off: int) -> np.ndarray:
    """Q4_K (bb = 144, nibbles at 16) or Q5_K (bb = 176, nibbles at 48, qh = 0)."""
    nb = K // 256
    W = np.zeros((K + K // 32, nb * bb), dtype=np.uint8)
    # code rows: d = 1, dmin = 0, every sc_j = 1, every m_j = 0, one nibble = 1
    k = np.arange(K)
    b, e = k // 256, k % 256
    j, i = e // 32, e % 32
    base = b * bb
    W[k, base] = ONE_FP16[0]
    W[k, base + 1] = ONE_FP16[1]
    for t in range(4):
        W[k, base + 4 + t] = 1        # S[0..3]: sc_0..3 = 1
        W[k, base + 12 + t] = 1       # S[8..11]: low nibble = sc_4..7 = 1, high nibble = m_4..7 = 0
    W[k, base + qs_off + 32 * (j >> 1) + i] = np.where(j % 2 == 0, 0x01, 0x10)
    # sum rows: d = 0, dmin = 1, every sc = 0, m_j = 1 on sub-block j only, nibbles 0
    g = np.arange(K // 32)
    r = K + g
    b, j = g // 8, g % 8
    base = b * bb
    W[r, base + 2] = ONE_FP16[0]
    W[r, base + 3] = ONE_FP16[1]
    # m_j for j < 4 is S[j+4] & 63; for j >= 4 it is S[j+4] >> 4 (bits 4..5 from S[j] >> 6)
    W[r, base + 8 + j] = np.where(j < 4, 0x01, 0x10)
    return W


def _q6k_rows(K: int) -> np.ndarray:
    nb = K // 256
    bb = 210
    W = np.zeros((K + K // 16, nb * bb), dtype=np.uint8)
    for bk in range(nb):
        W[:, bk * bb + 128: bk * bb + 192] = 0xAA     # high 2 bits of every code = 2 (q = 32 + low 4 bits)
    # code rows: d = 1, every scale 1, q = 32 everywhere except q = 33 at element k
    k = np.arange(K)
    b, e = k // 256, k % 256
    h, rem = e // 128, e % 128
    g, r = rem // 32, rem % 32
    base = b * bb
    W[k[:, None], base[:, None] + 192 + np.arange(16)[None, :]] = 1
    W[k, base + 208] = ONE_FP16[0]
    W[k, base + 209] = ONE_FP16[1]
    ql = base + 64 * h + 32 * (g & 1) + r               # g = 0, 1: low nibble; g = 2, 3: high nibble
    W[k, ql] = np.where(g < 2, 0x01, 0x10)
    # half-sum rows: d = 1, scale 1 on one group of 16 only, q = 33 everywhere
    s = np.arange(K // 16)
    rr = K + s
    b, grp = s // 16, s % 16
    base = b * bb
    for bk in range(nb):
        W[rr[:, None], bk * bb + np.arange(128)[None, :]] = 0x11
    W[rr, base + 192 + grp] = 1
    W[rr, base + 208] = ONE_FP16[0]
    W[rr, base + 209] = ONE_FP16[1]
    return W


def onehot_weights(wtype: str, K: int) -> np.ndarray:
    """Rows [code rows (K) | sum rows (K/32; Q6_K: half-sum rows, K/16)]."""
    if wtype == "q4_k":
        return _kquant_rows(K, 144, 16)
    if wtype == "q5_k":
        return _kquant_rows(K, 176, 48)
    if wtype == "q6_k":
        return _q6k_rows(K)
    raise ValueError(wtype)


def expected_outputs(wtype: str, q: np.ndarray, d_h: np.ndarray) -> np.ndarray:
    """The exact fp32 outputs of ``onehot_weights`` applied to one token whose
    Q8_1 codes are q (int8 [K/32, 32]) and scales d_h (fp16 bits [K/32]):
    d_h * q_k per code row, then -d_h * Sum q per block (Q6_K: +d_h * Sum q per
    half block). Computed in fp64, where every value is exact, then cast."""
    dh = np.asarray(d_h, dtype=np.uint16).view(np.float16).astype(np.float64)
    qq = q.astype(np.int64)
    codes = (dh[:, None] * qq).reshape(-1)
    if wtype == "q6_k":
        halves = qq.reshape(-1, 2, 16).sum(axis=-1)               # [K/32, 2]
        sums = (dh[:, None] * halves).reshape(-1)
    else:
        sums = -dh * qq.sum(axis=-1)
    out = np.concatenate([codes, sums])
    assert np.array_equal(out.astype(np.float32).astype(np.float64), out)   # exact in fp32
    return out.astype(np.float32)
