"""The C-ABI library builds, loads and exports every function include/kq.h
declares; its host-side argument checks answer without touching a GPU."""
import ctypes

import pytest

from quantized_weight_matmul_q4_gb300 import _native as nat
from quantized_weight_matmul_q4_gb300.build import build


@pytest.fixture(scope="module")
def L():
    build()
    return nat.lib()


def test_header_declares_the_boundary():
    names = nat.header_symbols()
    assert {"kq_quantize_q8_1", "kq_matvec", "kq_matvec_swiglu", "kq_matvec_rmsnorm", "kq_gemm",
            "kq_moe_grouped_gemm", "kq_moe_combine", "kq_workspace_bytes", "kq_get_device_error",
            "kq_status_str"} <= set(names)


def test_every_declared_symbol_is_exported(L):
    for name in nat.header_symbols():
        assert hasattr(L, name), name
        assert name in nat.SIGNATURES, f"{name} has no ctypes signature"


def test_status_strings(L):
    for s in range(8):
        assert nat.status_str(s).startswith("KQ_")
    assert "unknown" in nat.status_str(99)


# Fake, never dereferenced device addresses: the checks below all fail before
# any CUDA call is made.
A = ctypes.c_void_p(1 << 20)           # 16-byte aligned
U = ctypes.c_void_p((1 << 20) + 4)     # misaligned
NUL = ctypes.c_void_p(0)


def test_quantize_argument_checks(L):
    assert L.kq_quantize_q8_1(NUL, A, 64, 1, NUL) == nat.KQ_ERR_NULL
    assert L.kq_quantize_q8_1(A, A, 48, 1, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_quantize_q8_1(A, A, 64, 0, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_quantize_q8_1(U, A, 64, 1, NUL) == nat.KQ_ERR_ALIGN


def test_matvec_argument_checks(L):
    assert L.kq_matvec(9, A, A, A, 16, 256, NUL) == nat.KQ_ERR_TYPE
    assert L.kq_matvec(nat.KQ_Q4_K, NUL, A, A, 16, 256, NUL) == nat.KQ_ERR_NULL
    assert L.kq_matvec(nat.KQ_Q4_K, A, A, A, 16, 300, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec(nat.KQ_Q6_K, A, A, A, 0, 256, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec(nat.KQ_Q4_K, A, U, A, 16, 256, NUL) == nat.KQ_ERR_ALIGN


def test_tq4_1s_argument_checks(L):
    # TQ4_1S: K a multiple of 32; the decode matvec is its only entry point.
    assert L.kq_matvec(nat.KQ_TQ4_1S, NUL, A, A, 16, 256, NUL) == nat.KQ_ERR_NULL
    assert L.kq_matvec(nat.KQ_TQ4_1S, A, A, A, 16, 48, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec(nat.KQ_TQ4_1S, A, A, A, 0, 64, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec(nat.KQ_TQ4_1S, U, A, A, 16, 64, NUL) == nat.KQ_ERR_ALIGN
    assert L.kq_matvec_swiglu(nat.KQ_TQ4_1S, A, A, A, A, 16, 256, NUL) == nat.KQ_ERR_TYPE
    assert L.kq_matvec_rmsnorm(nat.KQ_TQ4_1S, A, A, A, ctypes.c_float(1e-6), A, 16, 256, NUL) == nat.KQ_ERR_TYPE
    assert L.kq_gemm(nat.KQ_TQ4_1S, A, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_TYPE
    assert L.kq_gemm_noalloc(nat.KQ_TQ4_1S, A, A, A, 16, 256, 4, NUL) == nat.KQ_ERR_TYPE
    assert L.kq_moe_grouped_gemm(nat.KQ_TQ4_1S, A, 8, A, 2, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_TYPE


def test_prefetch_argument_checks(L):
    f = L.kq_matvec_prefetch
    assert f(nat.KQ_Q4_K, A, A, A, 16, 256, U, 1024, NUL) == nat.KQ_ERR_ALIGN    # misaligned W_next
    assert f(nat.KQ_Q4_K, NUL, A, A, 16, 256, A, 1024, NUL) == nat.KQ_ERR_NULL
    assert f(nat.KQ_Q4_K, A, A, A, 16, 300, A, 1024, NUL) == nat.KQ_ERR_SHAPE
    assert f(9, A, A, A, 16, 256, NUL, 0, NUL) == nat.KQ_ERR_TYPE


def test_q5k_argument_checks(L):
    # Q5_K is taken wherever Q4_K is (K a multiple of 256).
    assert L.kq_matvec(nat.KQ_Q5_K, NUL, A, A, 16, 256, NUL) == nat.KQ_ERR_NULL
    assert L.kq_matvec(nat.KQ_Q5_K, A, A, A, 16, 288, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec(nat.KQ_Q5_K, A, U, A, 16, 256, NUL) == nat.KQ_ERR_ALIGN
    assert L.kq_matvec_swiglu(nat.KQ_Q5_K, A, A, NUL, A, 16, 256, NUL) == nat.KQ_ERR_NULL
    assert L.kq_gemm(nat.KQ_Q5_K, A, A, A, 16, 256, 4, NUL, 1 << 30, NUL) == nat.KQ_ERR_NULL
    assert L.kq_gemm(nat.KQ_Q5_K, A, A, A, 16, 128, 4, A, 1 << 30, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_gemm_noalloc(nat.KQ_Q5_K, A, A, A, 16, 128, 4, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_moe_grouped_gemm(nat.KQ_Q5_K, A, 0, A, 1, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_SHAPE


def test_fused_matvec_argument_checks(L):
    f = ctypes.c_float
    assert L.kq_matvec_swiglu(nat.KQ_Q4_K, A, A, NUL, A, 16, 256, NUL) == nat.KQ_ERR_NULL
    assert L.kq_matvec_swiglu(nat.KQ_Q4_K, A, A, U, A, 16, 256, NUL) == nat.KQ_ERR_ALIGN
    assert L.kq_matvec_swiglu(nat.KQ_Q6_K, A, A, A, A, 16, 100, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec_rmsnorm(nat.KQ_Q4_K, A, A, NUL, f(1e-6), A, 16, 256, NUL) == nat.KQ_ERR_NULL
    assert L.kq_matvec_rmsnorm(nat.KQ_Q4_K, A, A, A, f(-1.0), A, 16, 256, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec_rmsnorm(nat.KQ_Q4_K, A, A, A, f(float("nan")), A, 16, 256, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_matvec_rmsnorm(nat.KQ_Q4_K, A, A, U, f(1e-6), A, 16, 256, NUL) == nat.KQ_ERR_ALIGN
    assert L.kq_matvec_rmsnorm(5, A, A, A, f(1e-6), A, 16, 256, NUL) == nat.KQ_ERR_TYPE


def test_moe_combine_argument_checks(L):
    assert L.kq_moe_combine(NUL, A, A, 16, 4, 2, NUL) == nat.KQ_ERR_NULL
    assert L.kq_moe_combine(A, A, A, 0, 4, 2, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_moe_combine(A, A, A, 16, 4, 0, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_moe_combine(A, A, A, 16, 4, 513, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_moe_combine(A, U, A, 16, 4, 2, NUL) == nat.KQ_ERR_ALIGN


def test_gemm_argument_checks(L):
    assert L.kq_gemm(0, A, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_TYPE
    assert L.kq_gemm(nat.KQ_Q4_K, A, A, A, 16, 256, 4, NUL, 1 << 30, NUL) == nat.KQ_ERR_NULL
    assert L.kq_gemm(nat.KQ_Q4_K, A, A, A, 16, 128, 4, A, 1 << 30, NUL) == nat.KQ_ERR_SHAPE
    # Q6_K rows must be a multiple of 16 bytes on the tensor-core path: K % 2048 == 0
    assert L.kq_gemm(nat.KQ_Q6_K, A, A, A, 16, 1024, 4, A, 1 << 30, NUL) == nat.KQ_ERR_SHAPE
    assert L.kq_gemm(nat.KQ_Q4_K, A, A, U, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_ALIGN


def test_gemm_noalloc_argument_checks(L):
    f = L.kq_gemm_noalloc
    assert f(0, A, A, A, 16, 256, 4, NUL) == nat.KQ_ERR_TYPE
    assert f(nat.KQ_Q4_K, A, NUL, A, 16, 256, 4, NUL) == nat.KQ_ERR_NULL
    assert f(nat.KQ_Q4_K, A, A, A, 16, 128, 4, NUL) == nat.KQ_ERR_SHAPE
    assert f(nat.KQ_Q6_K, A, A, A, 16, 1024, 4, NUL) == nat.KQ_ERR_SHAPE
    assert f(nat.KQ_Q4_K, A, A, U, 16, 256, 4, NUL) == nat.KQ_ERR_ALIGN


def test_moe_argument_checks(L):
    f = L.kq_moe_grouped_gemm
    assert f(nat.KQ_Q4_K, A, 8, A, 9, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_SHAPE   # top_k > E
    assert f(nat.KQ_Q4_K, A, 0, A, 1, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_SHAPE
    assert f(nat.KQ_Q4_K, A, 513, A, 1, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_SHAPE
    assert f(nat.KQ_Q4_K, A, 8, NUL, 2, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_NULL
    assert f(nat.KQ_Q4_K, A, 8, U, 2, A, A, 16, 256, 4, A, 1 << 30, NUL) == nat.KQ_ERR_ALIGN


def test_workspace_sizes(L):
    ws = L.kq_workspace_bytes
    assert ws(nat.KQ_OP_MATVEC, nat.KQ_Q4_K, 4096, 4096, 1, 0, 0) == 0
    g = ws(nat.KQ_OP_GEMM, nat.KQ_Q4_K, 4096, 4096, 512, 0, 0)
    assert g >= 512 * 4096 * 2                         # at least x_hat in fp16
    m = ws(nat.KQ_OP_MOE, nat.KQ_Q4_K, 768, 2048, 1024, 128, 8)
    assert m >= 8192 * 2048 * 2 + 2 * 8192 * 4         # gathered x_hat + bucket tables
    assert ws(nat.KQ_OP_MOE, nat.KQ_Q4_K, 768, 2048, 1024, 4, 8) == 0   # top_k > n_experts
    assert ws(nat.KQ_OP_GEMM, nat.KQ_Q4_K, 4096, 100, 512, 0, 0) == 0   # K % 256
    assert ws(99, nat.KQ_Q4_K, 4096, 4096, 512, 0, 0) == 0
