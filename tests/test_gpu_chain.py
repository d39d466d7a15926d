"""Decode calls chained on one stream, each reading the previous call's output
as its activations, with no synchronisation between them. Every decode kernel
starts streaming its weights before it waits for the previous kernel
(programmatic dependent launch); these tests check that no kernel reads its x
before the producer of x has finished. Each stage is compared with the oracle
applied to the GPU's own previous output, so a stage that read a stale or
half-written x fails on its own."""
import numpy as np
import pytest

from oracle import kq_oracle as ora
from oracle import tq4_oracle as tq
import quantized_weight_matmul_q4_gb300 as kq
from quantized_weight_matmul_q4_gb300 import synthetic as syn
from _kqutil import assert_within_bound, to_dev

pytestmark = pytest.mark.gpu

D = 4096  # every matrix is D x D, so each output feeds the next call

STAGES = [("q4_k", "plain"), ("q5_k", "prefetch"), ("tq4_1s", "plain"), ("q6_k", "plain"),
          ("q4_k", "rmsnorm"), ("q6_k", "prefetch"), ("q4_k", "prefetch")]


# Where each format keeps its fp16 scales (byte offsets in a block, block size),
# and a power of two that brings the stage's output to about the size of its
# input (random weights of the generator amplify by 260x to 590x at K = 4096, and
# an activation above 127 * 65504 is outside the Q8_1 format).
_SCALES = {"q4_k": ((0, 2), 144, -8), "q5_k": ((0, 2), 176, -9), "q6_k": ((208,), 210, -9), "tq4_1s": ((0, 2), 20, 0)}


def _scaled(W, wt):
    offs, bb, e = _SCALES[wt]
    blocks = W.reshape(W.shape[0], -1, bb).copy()
    for o in offs:
        f = blocks[..., o:o + 2].copy().view(np.float16)
        blocks[..., o:o + 2] = (f * np.float16(2.0 ** e)).view(np.uint8)
    return blocks.reshape(W.shape)


def _weights():
    rng = np.random.default_rng(77)
    return [_scaled(syn.weights(wt, rng, D, D), wt) for wt, _ in STAGES]


def _launch_chain(Wd, x0, ys, gamma):
    x = x0
    for i, (wt, how) in enumerate(STAGES):
        nxt = Wd[(i + 1) % len(Wd)]
        if how == "plain":
            kq.kq_matvec(wt, Wd[i], x, D, D, y=ys[i])
        elif how == "prefetch":
            kq.kq_matvec_prefetch(wt, Wd[i], x, D, D, W_next=nxt, y=ys[i])
        else:
            kq.kq_matvec_rmsnorm(wt, Wd[i], x, gamma, 1e-5, D, D, y=ys[i])
        x = ys[i]


def _check_stages(Ws, x0, outs, gamma):
    x = x0.astype(np.float32)
    for i, (wt, how) in enumerate(STAGES):
        xin = x.reshape(1, D)
        if wt == "tq4_1s":
            Y, B = tq.tq4_1s_matmul(Ws[i], xin, D, D)
        elif how == "rmsnorm":
            Y, B = ora.matmul_from(wt, Ws[i], ora.rms_norm(xin, gamma, 1e-5), D, D)
        else:
            Y, B = ora.matmul(wt, Ws[i], xin, D, D)
        assert_within_bound(outs[i], Y[0], B[0], f"stage {i} ({wt}, {how})")
        x = outs[i]  # the next stage's reference input is what the GPU produced


@pytest.mark.parametrize("graph", [False, True])
def test_chained_decode_calls(graph):
    import torch
    Ws = _weights()
    Wd = [to_dev(W, torch) for W in Ws]
    rng = np.random.default_rng(78)
    x0 = syn.activations(rng, D, 1)[0]
    gamma = (np.abs(syn.activations(rng, D, 1)[0]) + 0.5).astype(np.float32)
    x0d, gd = to_dev(x0, torch), to_dev(gamma, torch)
    ys = [torch.empty(D, dtype=torch.float32, device="cuda") for _ in STAGES]
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            _launch_chain(Wd, x0d, ys, gd)  # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for y in ys:
            y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            _launch_chain(Wd, x0d, ys, gd)
        g.replay()
    else:
        _launch_chain(Wd, x0d, ys, gd)
    torch.cuda.synchronize()
    assert kq.kq_get_device_error() == 0
    outs = [y.cpu().numpy() for y in ys]
    for o in outs:
        assert np.all(np.isfinite(o))
    _check_stages(Ws, x0, outs, gamma)


GEMM_D, GEMM_N = 2048, 96  # Q6_K on the tensor-core path needs K % 2048 == 0
GEMM_STAGES = ["q4_k", "q5_k", "q6_k"]


@pytest.mark.parametrize("graph", [False, True])
def test_chained_prefill_calls(graph):
    # Y_i = W_i . Y_{i-1} for 96 tokens: each call's activation quantiser and
    # epilogue wait for the previous kernel (programmatic dependent launch).
    import torch
    rng = np.random.default_rng(79)
    Ws = [_scaled(syn.weights(wt, rng, GEMM_D, GEMM_D), wt) for wt in GEMM_STAGES]
    Wd = [to_dev(W, torch) for W in Ws]
    X0 = syn.activations(rng, GEMM_D, GEMM_N)
    X0d = to_dev(X0, torch)
    ws = [torch.empty(kq.kq_workspace_bytes(kq.KQ_OP_GEMM, wt, GEMM_D, GEMM_D, GEMM_N), dtype=torch.uint8,
                      device="cuda") for wt in GEMM_STAGES]
    Ys = [torch.empty((GEMM_N, GEMM_D), dtype=torch.float32, device="cuda") for _ in GEMM_STAGES]

    def chain():
        x = X0d
        for i, wt in enumerate(GEMM_STAGES):
            kq.kq_gemm(wt, Wd[i], x, GEMM_D, GEMM_D, Y=Ys[i], ws=ws[i])
            x = Ys[i]

    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            chain()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for y in Ys:
            y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain()
        g.replay()
    else:
        chain()
    torch.cuda.synchronize()
    assert kq.kq_get_device_error() == 0
    x = X0
    for i, wt in enumerate(GEMM_STAGES):
        out = Ys[i].cpu().numpy()
        assert np.all(np.isfinite(out)), wt
        Yr, B = ora.matmul(wt, Ws[i], x, GEMM_D, GEMM_D)
        assert_within_bound(out, Yr, B, f"prefill stage {i} ({wt})")
        x = out
