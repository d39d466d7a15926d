"""kq — k-quant (Q4_K / Q5_K / Q6_K) and TQ4_1S weight matmul for NVIDIA GB300.

Thin Python binding over the C ABI of libkq (include/kq.h): every function
here only checks and marshals its arguments (device pointers, sizes, the
current CUDA stream) and calls the library of the same name. All arithmetic
runs in the library's CUDA kernels; there is no CPU path. PyTorch provides
device memory and streams.
"""
from __future__ import annotations

import ctypes

from ._native import (KQ_DEVERR_EXPERT_ID, KQ_DEVERR_NONE, KQ_DEVERR_WAIT_TIMEOUT, KQ_GEMM_STATIC_WS_BYTES,
                      KQ_OP_GEMM, KQ_OP_MATVEC, KQ_OP_MOE, KQ_Q4_K, KQ_Q5_K, KQ_Q6_K, KQ_TQ4_1S, KQError, check, lib)

__all__ = [
    "KQ_Q4_K", "KQ_Q5_K", "KQ_Q6_K", "KQ_TQ4_1S", "KQ_OP_MATVEC", "KQ_OP_GEMM", "KQ_OP_MOE", "KQError",
    "KQ_DEVERR_NONE", "KQ_DEVERR_WAIT_TIMEOUT", "KQ_DEVERR_EXPERT_ID",
    "KQ_GEMM_STATIC_WS_BYTES", "kq_quantize_q8_1", "kq_matvec", "kq_matvec_prefetch", "kq_matvec_swiglu", "kq_matvec_rmsnorm",
    "kq_gemm", "kq_gemm_noalloc", "kq_moe_grouped_gemm", "kq_moe_combine", "kq_workspace_bytes",
    "kq_get_device_error", "kq_test_hold_copies", "block_bytes", "row_bytes",
]

_BLOCK_BYTES = {KQ_Q4_K: 144, KQ_Q5_K: 176, KQ_Q6_K: 210, KQ_TQ4_1S: 20}
_BLOCK_WEIGHTS = {KQ_Q4_K: 256, KQ_Q5_K: 256, KQ_Q6_K: 256, KQ_TQ4_1S: 32}


_WTYPES = {"q4_k": KQ_Q4_K, "q5_k": KQ_Q5_K, "q6_k": KQ_Q6_K, "tq4_1s": KQ_TQ4_1S}


def _wt(wtype) -> int:
    if isinstance(wtype, str):
        w = _WTYPES.get(wtype)
        return w if w is not None else _WTYPES[wtype.lower()]
    return int(wtype)


def block_bytes(wtype) -> int:
    return _BLOCK_BYTES[_wt(wtype)]


def row_bytes(wtype, K: int) -> int:
    return (K // _BLOCK_WEIGHTS[_wt(wtype)]) * block_bytes(wtype)


_TORCH = None
_TENSOR = None        # torch.Tensor
_RAW_STREAM = None    # the current stream's handle of a device, without a Stream object (or False)
_GET_DEVICE = None    # the current device index


def _torch():
    global _TORCH, _TENSOR, _RAW_STREAM, _GET_DEVICE
    if _TORCH is None:
        import torch
        _TENSOR = torch.Tensor
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None) or False
        _GET_DEVICE = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
        _TORCH = torch
    return _TORCH


def _dev(t, name: str, dtype=None):
    """Device pointer (an int) of a contiguous CUDA tensor of the given dtype."""
    # The checks of a decode loop's every call, with as few attribute reads as
    # possible; anything unusual takes the path below for its error.
    if type(t) is _TENSOR and t.is_cuda and (dtype is None or t.dtype is dtype) and t.is_contiguous():
        return t.data_ptr()
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (libkq has no CPU path)")
    if dtype is not None and t.dtype is not dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    """The cudaStream_t to queue on: `stream` (a torch stream or a raw handle),
    else the current stream of the current device."""
    torch = _torch()
    if stream is None:
        if _RAW_STREAM:
            return _RAW_STREAM(_GET_DEVICE())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def kq_quantize_q8_1(X, Xq=None, stream=None):
    """X: fp32 [N, K] -> Q8_1 bytes uint8 [N, K/32, 36]."""
    torch = _torch()
    N, K = X.shape
    if Xq is None:
        Xq = torch.empty((N, K // 32, 36), dtype=torch.uint8, device=X.device)
    check(lib().kq_quantize_q8_1(_dev(X, "X", torch.float32), _dev(Xq, "Xq", torch.uint8), K, N,
                                 _stream(stream)), "kq_quantize_q8_1")
    return Xq


def kq_matvec(wtype, W, x, M: int, K: int, y=None, stream=None):
    """y[M] = dequant(W) . x; W uint8 [M, row_bytes], x fp32 [K] (wtype q4_k, q5_k, q6_k or tq4_1s)."""
    torch = _torch()
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=x.device)
    check(lib().kq_matvec(_wt(wtype), _dev(W, "W", torch.uint8), _dev(x, "x", torch.float32),
                          _dev(y, "y", torch.float32), M, K, _stream(stream)), "kq_matvec")
    return y


def kq_matvec_prefetch(wtype, W, x, M: int, K: int, W_next=None, y=None, stream=None):
    """kq_matvec, and L2 is asked to prefetch W_next (the next call's weights,
    a uint8 CUDA tensor) while it runs; y is identical to kq_matvec's."""
    torch = _torch()
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=x.device)
    nxt = _dev(W_next, "W_next", torch.uint8) if W_next is not None else None
    nbytes = W_next.numel() if W_next is not None else 0
    check(lib().kq_matvec_prefetch(_wt(wtype), _dev(W, "W", torch.uint8), _dev(x, "x", torch.float32),
                                   _dev(y, "y", torch.float32), M, K, nxt, nbytes, _stream(stream)),
          "kq_matvec_prefetch")
    return y


def kq_matvec_swiglu(wtype, W, gate, up, M: int, K: int, y=None, stream=None):
    """y[M] = dequant(W) . Q8_1(silu(gate) * up); gate, up fp32 [K]."""
    torch = _torch()
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=gate.device)
    check(lib().kq_matvec_swiglu(_wt(wtype), _dev(W, "W", torch.uint8), _dev(gate, "gate", torch.float32),
                                 _dev(up, "up", torch.float32), _dev(y, "y", torch.float32), M, K,
                                 _stream(stream)), "kq_matvec_swiglu")
    return y


def kq_matvec_rmsnorm(wtype, W, x, gamma, eps: float, M: int, K: int, y=None, stream=None):
    """y[M] = dequant(W) . Q8_1(x / sqrt(mean(x^2) + eps) * gamma); x, gamma fp32 [K]."""
    torch = _torch()
    if y is None:
        y = torch.empty(M, dtype=torch.float32, device=x.device)
    check(lib().kq_matvec_rmsnorm(_wt(wtype), _dev(W, "W", torch.uint8), _dev(x, "x", torch.float32),
                                  _dev(gamma, "gamma", torch.float32), float(eps), _dev(y, "y", torch.float32),
                                  M, K, _stream(stream)), "kq_matvec_rmsnorm")
    return y


def kq_moe_combine(Y, probs, out=None, stream=None):
    """out[T, M] = Sum_j probs[:, j] * Y[:, j, :] for Y fp32 [T, top_k, M], probs fp32 [T, top_k]."""
    torch = _torch()
    T, top_k, M = Y.shape
    if out is None:
        out = torch.empty((T, M), dtype=torch.float32, device=Y.device)
    check(lib().kq_moe_combine(_dev(Y, "Y", torch.float32), _dev(probs, "probs", torch.float32),
                               _dev(out, "out", torch.float32), M, T, top_k, _stream(stream)), "kq_moe_combine")
    return out


def kq_workspace_bytes(op: int, wtype, M: int, K: int, N_or_T: int, n_experts: int = 0, top_k: int = 0) -> int:
    return int(lib().kq_workspace_bytes(int(op), _wt(wtype), M, K, N_or_T, n_experts, top_k))


def kq_gemm(wtype, W, X, M: int, K: int, Y=None, ws=None, stream=None):
    """Y[N, M] = (dequant(W) . X^T)^T for X fp32 [N, K]."""
    torch = _torch()
    N = X.shape[0]
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=X.device)
    if ws is None:
        ws = torch.empty(max(1, kq_workspace_bytes(KQ_OP_GEMM, wtype, M, K, N)), dtype=torch.uint8,
                         device=X.device)
    check(lib().kq_gemm(_wt(wtype), _dev(W, "W", torch.uint8), _dev(X, "X", torch.float32),
                        _dev(Y, "Y", torch.float32), M, K, N, _dev(ws, "ws", torch.uint8), ws.numel(),
                        _stream(stream)), "kq_gemm")
    return Y


def kq_gemm_noalloc(wtype, W, X, M: int, K: int, Y=None, stream=None):
    """kq_gemm with the library's fixed per-device scratch instead of a workspace.

    Raises KQError(KQ_ERR_WORKSPACE) when the shape needs more than
    KQ_GEMM_STATIC_WS_BYTES of scratch. Calls that may overlap race on the scratch.
    """
    torch = _torch()
    N = X.shape[0]
    if Y is None:
        Y = torch.empty((N, M), dtype=torch.float32, device=X.device)
    check(lib().kq_gemm_noalloc(_wt(wtype), _dev(W, "W", torch.uint8), _dev(X, "X", torch.float32),
                                _dev(Y, "Y", torch.float32), M, K, N, _stream(stream)), "kq_gemm_noalloc")
    return Y


def kq_moe_grouped_gemm(wtype, W_experts, n_experts: int, expert_ids, X, M: int, K: int, Y=None, ws=None,
                        stream=None):
    """Y[T, top_k, M]: per (token, slot) product with the routed expert's weights."""
    torch = _torch()
    T, top_k = expert_ids.shape
    if Y is None:
        Y = torch.empty((T, top_k, M), dtype=torch.float32, device=X.device)
    if ws is None:
        ws = torch.empty(max(1, kq_workspace_bytes(KQ_OP_MOE, wtype, M, K, T, n_experts, top_k)),
                         dtype=torch.uint8, device=X.device)
    check(lib().kq_moe_grouped_gemm(_wt(wtype), _dev(W_experts, "W_experts", torch.uint8), n_experts,
                                    _dev(expert_ids, "expert_ids", torch.int32), top_k,
                                    _dev(X, "X", torch.float32), _dev(Y, "Y", torch.float32), M, K, T,
                                    _dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)),
          "kq_moe_grouped_gemm")
    return Y


def kq_get_device_error(stream=None) -> int:
    """Waits for the stream; returns and clears the first recorded device error code."""
    code = ctypes.c_int32(0)
    st = lib().kq_get_device_error(ctypes.byref(code), _stream(stream))
    if st not in (0, 7):
        raise KQError(st, "kq_get_device_error")
    return int(code.value)


def kq_test_hold_copies(hold: bool) -> None:
    """Test hook: while set, the weight producers of the decode and tensor-core
    kernels issue nothing, so their waits run out (KQ_DEVERR_WAIT_TIMEOUT)."""
    check(lib().kq_test_hold_copies(1 if hold else 0), "kq_test_hold_copies")
