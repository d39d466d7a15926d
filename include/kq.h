/*
 * kq.h — k-quant weight matmul on NVIDIA GB300 (sm_103a): C ABI of libkq.
 *
 *   Y[M, N] = dequant(W)[M, K] . X[K, N]
 *
 * W holds 4-bit Q4_K, 5-bit Q5_K or 6-bit Q6_K super-blocks; X is fp32 and is
 * quantised to
 * Q8_1 (int8 codes with an fp16 scale per 32 values) inside every call. The
 * decode matvec also takes TQ4_1S weights (WHT-rotated 4-bit Lloyd-Max codes),
 * which it multiplies with the fp32 activations directly.
 *
 * Sources (page title, section):
 *  [MMVQ]  "06 · 8e/8e② — decode MMVQ: dp4a integer dot products + the llama.cpp
 *          launch table": §2 Principle (Q4_K value d*sc*nib - dmin*m, the min-term
 *          identity, the q8 activation quantiser), §3.2 Key code (Q4_K byte
 *          offsets, quantize_pad40_block), §3.3 Pitfalls (Q6_K layout, d at 208).
 *  [MMQv2] "ZINC MMQ v2 — Fused Q4_K×Q8_1 Tensor-Core GEMM (beat llama.cpp)": What
 *          they do right (Q8_1 activations, fused dequant), Kernel architecture,
 *          Persistent kernel + atomic work queue, MoE routing (fused gather).
 *  [GAP]   "Prefill Gap Closure Plan — ZINC CUDA vs llama.cpp": T1 (fused dequant
 *          tensor-core GEMM), T2 (grouped MoE expert GEMM: histogram, prefix sum,
 *          scatter, per-expert GEMM).
 *  [TQ]    "TQ4_1S Weight Kernel Optimization": Architecture Overview (rotated
 *          4-bit weights, dequant = centroid[index] * half-block scale, inverse
 *          WHT, pre-rotated activation), Block Layout, Centroid Table.
 *
 * Conventions for every entry point
 *  - Pointers are device pointers owned by the caller (cudaMalloc / a framework
 *    allocator) unless stated otherwise. The library allocates no memory, keeps
 *    no pointer after the call returns, and does not synchronise the stream
 *    (except kq_get_device_error).
 *  - Layouts (row-major everywhere):
 *      W : M rows x (K/256) super-blocks; a Q4_K block is 144 bytes
 *          [fp16 d][fp16 dmin][12 B packed 6-bit scales/mins][128 B nibbles],
 *          a Q6_K block is 210 bytes [ql 128][qh 64][int8 scales 16][fp16 d].
 *          Q5_K (the GGUF layout; the pages give none): 176 bytes [fp16 d][fp16 dmin]
 *          [12 B scales/mins packed as Q4_K][qh 32][128 B nibbles], weight r of
 *          sub-block j taking its fifth bit from bit j of qh[r].
 *          TQ4_1S: M rows x (K/32) blocks of 20 bytes [fp16 d0][fp16 d1][qs 16],
 *          element j's centroid index in qs[j/2], low nibble for even j.
 *          For MoE the experts' matrices are concatenated, expert-major.
 *      X : fp32, token-major: token n occupies X[n*K .. n*K+K-1].
 *      Y : fp32, token-major: Y[n*M + m].
 *      Xq: N x (K/32) Q8_1 blocks of 36 bytes [fp16 d][fp16 s][int8 q[32]].
 *  - Alignment: W, X, Y, Xq and ws must be 16-byte aligned.
 *  - Sizes: K must be a multiple of 256 (32 for kq_quantize_q8_1 and for TQ4_1S);
 *    M, N, T >= 1; all sizes below 2^31.
 *  - Work is queued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *    A status other than KQ_OK means nothing was queued, except KQ_ERR_CUDA
 *    after a failed launch.
 *  - Results are deterministic: the same inputs give bit-identical outputs.
 *  - Per-device state: the library looks up, once per device, the device
 *    addresses of its error word (and of kq_gemm_noalloc's scratch) and sets
 *    its kernels' shared-memory limits. That state belongs to the device's
 *    primary context: do not call the library after cudaDeviceReset in the
 *    same process.
 *  - Accuracy: Q8_1 codes and block sums are bit-exact against the IEEE fp32
 *    definition. Y satisfies |Y - Y_ref| <= 1e-3 * Sum_k |w_k x_k| + 1e-5 per
 *    element, Y_ref being the exact product of the dequantised operands. The
 *    tensor-core paths (kq_gemm, kq_moe_grouped_gemm) round dequantised
 *    weights and activations to fp16, so they need |w|, |x| < 65504.
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KQ_API __attribute__((visibility("default")))
#else
#define KQ_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* kq_stream_t;

typedef enum kq_status {
  KQ_OK = 0,
  KQ_ERR_NULL = 1,      /* a required pointer is NULL */
  KQ_ERR_SHAPE = 2,     /* a size is out of range or not a multiple of its block */
  KQ_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned */
  KQ_ERR_TYPE = 4,      /* unknown weight type */
  KQ_ERR_WORKSPACE = 5, /* ws_bytes is smaller than kq_workspace_bytes() */
  KQ_ERR_CUDA = 6,      /* a CUDA runtime call failed (no device, launch failure) */
  KQ_ERR_DEVICE = 7     /* a kernel recorded an error; see kq_get_device_error */
} kq_status;

/* KQ_Q5_K is taken wherever Q4_K is; KQ_TQ4_1S by kq_matvec only (the other
 * entry points return KQ_ERR_TYPE for it). */
typedef enum kq_wtype { KQ_Q4_K = 1, KQ_Q6_K = 2, KQ_TQ4_1S = 3, KQ_Q5_K = 4 } kq_wtype;

typedef enum kq_op { KQ_OP_MATVEC = 1, KQ_OP_GEMM = 2, KQ_OP_MOE = 3 } kq_op;

/* Device error codes reported by kq_get_device_error. */
#define KQ_DEVERR_NONE 0
#define KQ_DEVERR_WAIT_TIMEOUT 1 /* a pipeline wait gave up (the kernel returned early) */
#define KQ_DEVERR_EXPERT_ID 2    /* an expert id was outside [0, n_experts) */

/*
 * kq_quantize_q8_1 — fp32 activations to Q8_1 blocks ([MMVQ] §2 and §3.2
 * quantize_pad40_block; the Q8_1 block sum of [MMQv2] "What they do right").
 * For every 32 consecutive values x of a token:
 *   d = max|x| / 127, q = clamp(rint(x * (d != 0 ? 1/d : 0)), -128, 127),
 *   stored d_h = fp16(d), s_h = fp16(d_h * Sum q), all in IEEE fp32 with
 *   round-half-even.
 * X: fp32 [N][K]; Xq: N*(K/32)*36 bytes, written. K % 32 == 0.
 */
KQ_API kq_status kq_quantize_q8_1(const float* X, void* Xq, int64_t K, int64_t N, kq_stream_t stream);

/*
 * kq_matvec — decode matvec y = dequant(W) . x for one token ([MMVQ] §2, §3.2:
 * integer dot products of the 4/6-bit codes with the Q8_1 codes of x, the
 * min term from the Q8_1 block sum, warp-shuffle row reductions). x is
 * quantised to Q8_1 inside the call. Needs no workspace.
 * wtype: KQ_Q4_K, KQ_Q6_K or KQ_Q5_K (the Q4_K value d*sc*q - dmin*m with a
 * 5-bit q; the pages ship it as a sibling decode kernel). W: M rows of K/256
 * blocks; x: fp32 [K];
 * y: fp32 [M], written.
 * Weight streaming starts before the kernel waits for the previous kernel on
 * the stream: W must not be written by a kernel that is still running when this
 * call starts, i.e. by a preceding kernel that allows programmatic dependent
 * launch. (A preceding ordinary kernel, copy or event is always complete.)
 * A Q6_K row whose byte length is not a multiple of 16 must have K <= 15360.
 * The k-quant decode kernels hold the whole Q8_1 activation in shared memory:
 * K <= 121600 is always taken; a larger K only when a CTA's rows fit the staged
 * kernel (few rows), else KQ_ERR_SHAPE with nothing queued. TQ4_1S has no such
 * limit (its fallback rotates x in segments).
 *
 * wtype KQ_TQ4_1S ([TQ]): W holds rotated weights r_b[j] = c[idx_j] * d_h(j)
 * per 32-block b (c the page's 16-entry centroid table, d0 for j < 16, d1
 * otherwise), and y[m] = Sum_b w_b . x_b with w_b = H^-1 r_b, H the orthonormal
 * 32-point Walsh-Hadamard transform in natural order (H[i][j] =
 * (-1)^popcount(i & j) / sqrt(32), its own inverse). The call rotates x once
 * (x_r = H x_b, fp32) and computes Sum_b r_b . x_r in fp32; no Q8_1 step.
 * K must be a multiple of 32 (multiples of 128 take the TMA-staged kernel).
 * Accuracy: |y - y_ref| <= 1e-3 * Sum_b Sum_j Sum_k |r_b[j] H[j][k] x_b[k]| + 1e-5,
 * y_ref the exact product. Weight streaming starts before the dependency wait,
 * as above.
 */
KQ_API kq_status kq_matvec(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t K,
                           kq_stream_t stream);

/*
 * kq_matvec_prefetch — kq_matvec, and while it runs each CTA also asks L2 to
 * fetch its share of W_next[0, W_next_bytes) (rounded down to a multiple of 16):
 * the weights of the call that follows on the stream, e.g. the next layer's
 * matrix in a decode step. That call's weight stream then starts from L2 while
 * this one computes (the staged lane-row forms and the item kernel of Q6_K
 * ask for it once their activations are in, so that it does not delay them;
 * the lane-row ring form once its ring is primed). y is bit-identical to
 * kq_matvec's; the prefetch is a hint (nothing waits for it). An addition of
 * this library (the pages launch one matrix per call without it). Every decode
 * kernel form takes it except the TQ4_1S fallback for K % 128 != 0.
 * W_next: NULL (no prefetch) or 16-byte aligned device memory readable for
 * W_next_bytes bytes (KQ_ERR_ALIGN otherwise). Other arguments as kq_matvec.
 */
KQ_API kq_status kq_matvec_prefetch(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t K,
                                    const void* W_next, size_t W_next_bytes, kq_stream_t stream);

/*
 * kq_matvec_swiglu, kq_matvec_rmsnorm — kq_matvec with the producer of its
 * activations fused into the Q8_1 quantiser ([MMVQ] §3.2 Key code: the
 * quantisation body moved into the RMSNorm and SwiGLU producers), so the
 * produced activations never go to memory:
 *   swiglu:  x[k] = silu(gate[k]) * up[k],  silu(g) = g / (1 + exp(-g));
 *   rmsnorm: x[k] = x_in[k] * r * gamma[k], r = 1 / sqrt(Sum_k x_in[k]^2 / K + eps)
 *            (eps >= 0; the sum of squares is taken in a fixed order).
 * gate, up, x_in, gamma: fp32 [K], 16-byte aligned. The producers compute in
 * fp32; the Q8_1 codes are then made from those fp32 values exactly as in
 * kq_matvec, and Y meets the accuracy bound against the exact product of the
 * dequantised weights with the Q8_1 codes of the produced activations.
 * Otherwise as kq_matvec (wtype, layouts, W streamed before the dependency wait);
 * KQ_TQ4_1S is not taken here (KQ_ERR_TYPE).
 */
KQ_API kq_status kq_matvec_swiglu(int wtype, const void* W, const float* gate, const float* up, float* y, int64_t M,
                                  int64_t K, kq_stream_t stream);
KQ_API kq_status kq_matvec_rmsnorm(int wtype, const void* W, const float* x, const float* gamma, float eps, float* y,
                                   int64_t M, int64_t K, kq_stream_t stream);

/*
 * kq_gemm — prefill GEMM Y = dequant(W) . X for N tokens ([MMQv2] Kernel
 * architecture; [GAP] T1). X is quantised to Q8_1 (as x_hat = fp16(d_h * q))
 * into the workspace once per call; weight super-blocks are staged by TMA and
 * unpacked to fp16 into tensor memory; tcgen05 MMAs accumulate in tensor memory.
 * A few tokens are a decode rather than a GEMM: Q4_K and Q5_K with 2 <= N <= 7 run on
 * the decode matvec path instead ([MMVQ] §2: dp4a on the Q8_1 codes, the min
 * term from the block sums; the tokens' codes are made once into the
 * workspace, the weights are read once for all tokens). Both paths meet the
 * accuracy bound above; a token's result may differ in the last bits with the
 * number of tokens in the call (the partial sums are grouped differently).
 * W: M x K weights; X: fp32 [N][K]; Y: fp32 [N][M], written.
 * ws: device workspace of at least kq_workspace_bytes(KQ_OP_GEMM, ...) bytes.
 * Q6_K needs K % 2048 == 0 (rows whose byte length is a multiple of 16).
 * As in kq_matvec, W is streamed before the GEMM waits for the previous kernel
 * on the stream: W must not be written by a still-running predecessor that
 * allows programmatic dependent launch.
 */
KQ_API kq_status kq_gemm(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K, int64_t N, void* ws,
                  size_t ws_bytes, kq_stream_t stream);

/*
 * kq_gemm_noalloc — kq_gemm without a workspace argument. This entry point is
 * an addition of this library; the source pages have no counterpart to it.
 * Same operation, arguments (minus ws/ws_bytes), layouts, accuracy and
 * determinism as kq_gemm; it runs the same kernels.
 *
 * Who needs it: callers that cannot hand the library device memory per call,
 * e.g. plain C hosts with no device allocator of their own, or runtimes that
 * plan all device memory ahead and forbid allocation on the per-token path
 * (cudaMalloc may synchronise the device, which such a loop cannot afford).
 * The library itself allocates nothing here: the scratch (fp16 x_hat and
 * split-K partials) is a fixed array of KQ_GEMM_STATIC_WS_BYTES per device,
 * part of the library's device image, which no caller has to clear. With
 * CUDA's default lazy module loading the array takes device memory only once
 * this entry point is first called on a device; with eager loading
 * (CUDA_MODULE_LOADING=EAGER) every context that loads the library reserves it.
 *
 * Limit: returns KQ_ERR_WORKSPACE, with nothing queued, when the call would
 * need more scratch than KQ_GEMM_STATIC_WS_BYTES, i.e. when
 * kq_workspace_bytes(KQ_OP_GEMM, wtype, M, K, N, 0, 0) > KQ_GEMM_STATIC_WS_BYTES
 * (for instance N = 2048 tokens with K = 14336). Use kq_gemm there.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the array's device address, which loads the array's module; make that first
 * call before any stream capture.
 *
 * Concurrency: all calls on one device share the one array. Two calls whose
 * kernels may overlap (on different streams, or from several host threads
 * without ordering) race on it and give wrong results; order them on one
 * stream (or with events).
 */
#define KQ_GEMM_STATIC_WS_BYTES ((size_t)32 << 20)

KQ_API kq_status kq_gemm_noalloc(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K,
                                 int64_t N, kq_stream_t stream);

/*
 * kq_moe_grouped_gemm — MoE expert matmul ([MMQv2] MoE routing; [GAP] T2).
 * For every token t and slot j < top_k: Y[t][j][:] = dequant(W_e) . x_t with
 * e = expert_ids[t*top_k + j]. The (token, slot) pairs are grouped by expert
 * (histogram, prefix sum, scatter), the activations are gathered per expert,
 * and each expert's weight tile is read once for all of its tokens.
 * W_experts: n_experts * M rows of K/256 blocks (expert-major);
 * expert_ids: int32 [T][top_k]; X: fp32 [T][K]; Y: fp32 [T][top_k][M], written.
 * No router weighting and no sum over slots. An out-of-range expert id records
 * KQ_DEVERR_EXPERT_ID and that slot's output row is written as zeros.
 * ws: at least kq_workspace_bytes(KQ_OP_MOE, ...) bytes.
 */
KQ_API kq_status kq_moe_grouped_gemm(int wtype, const void* W_experts, int32_t n_experts, const int32_t* expert_ids,
                              int32_t top_k, const float* X, float* Y, int64_t M, int64_t K, int64_t T, void* ws,
                              size_t ws_bytes, kq_stream_t stream);

/*
 * kq_moe_combine — the step after kq_moe_grouped_gemm: each token's slot rows
 * go back to the token, weighted by the router probabilities ([GAP] T2,
 * "scatter back"; read as the usual weighted MoE combine):
 *   out[t][m] = Sum_{j < top_k} probs[t][j] * Y[t][j][m],
 * summed in fp32 in slot order with one fused multiply-add per slot
 * (deterministic). Y: fp32 [T][top_k][M] (as kq_moe_grouped_gemm writes it);
 * probs: fp32 [T][top_k]; out: fp32 [T][M], written. 1 <= top_k <= 512.
 * Needs no workspace; out must not overlap Y or probs.
 */
KQ_API kq_status kq_moe_combine(const float* Y, const float* probs, float* out, int64_t M, int64_t T, int32_t top_k,
                                kq_stream_t stream);

/*
 * kq_workspace_bytes — device workspace needed by an operation (0 for
 * KQ_OP_MATVEC). N_or_T is N for KQ_OP_GEMM and T for KQ_OP_MOE; n_experts
 * and top_k are read for KQ_OP_MOE only. The size depends on the SM count of
 * the current device. Returns 0 for invalid arguments.
 */
KQ_API size_t kq_workspace_bytes(int op, int wtype, int64_t M, int64_t K, int64_t N_or_T, int32_t n_experts,
                          int32_t top_k);

/*
 * kq_get_device_error — waits for `stream`, then returns in *code the first
 * device error recorded on the current device since the previous call
 * (KQ_DEVERR_*), and clears it. Returns KQ_ERR_DEVICE when *code != 0.
 * There is one error word per device, shared by every stream and every call
 * on it (not one per workspace): with kernels in flight on other streams, a
 * code may come from one of those, and only `stream` is waited for.
 */
KQ_API kq_status kq_get_device_error(int32_t* code, kq_stream_t stream);

/*
 * kq_test_hold_copies — a test hook for the library's failure detection; the
 * source pages have no counterpart to it. While `hold` is non-zero, launches
 * made afterwards by kq_matvec, kq_matvec_prefetch and the fused matvecs (Q4_K,
 * Q5_K, Q6_K), by kq_gemm's tensor-core kernel and by kq_moe_grouped_gemm run
 * with their weight producer issuing no copy (and, on the tensor-core paths,
 * handing out no tile). Their consumers' pipeline waits then run out after
 * their limit (2 s), the kernel records KQ_DEVERR_WAIT_TIMEOUT, leaves its
 * loops, frees its tensor memory and returns: the path a wait that gives up
 * takes, with no copy in flight. Outputs of such calls are undefined. The
 * flag is per process and is read when a call queues its launch (a call
 * captured in a CUDA graph keeps the value it saw). Not for production use:
 * hold = 0 (the default) restores normal calls. Always returns KQ_OK.
 * Calls that take other kernels (TQ4_1S, the small-N decode of kq_gemm) are
 * not affected.
 */
KQ_API kq_status kq_test_hold_copies(int hold);

/* Name of a status code (static string). */
KQ_API const char* kq_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* KQ_H */
