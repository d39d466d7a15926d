// Internal declarations shared by the CUDA translation units of libkq.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kq.h"

namespace kq {

cudaError_t launch_quantize_q8_1(const float* X, void* Xq, int64_t K, int64_t N, cudaStream_t s);
cudaError_t launch_quantize_xhat(const float* X, __half* Xh, int64_t K, int64_t rows, int num_sms, cudaStream_t s);
// MoE activations: the x_hat row of token p (Q8_1 of X row p, as
// launch_quantize_xhat makes it) into bucket row slot_pos[s] of Xh for each
// slot s = p * top_k + j; entries[slot_pos[s]] = s. Negative positions are skipped.
cudaError_t launch_quantize_scatter(const float* X, __half* Xh, int64_t K, int64_t T, int top_k, const int* slot_pos,
                                   int* entries, cudaStream_t s);

// Producer of the decode matvec's activations (fused into its quantiser):
// x itself; silu(x) * aux (SwiGLU, x the gate, aux the up projection);
// x / sqrt(mean(x^2) + eps) * aux (RMSNorm, aux = gamma).
constexpr int PROD_X = 0;
constexpr int PROD_SWIGLU = 1;
constexpr int PROD_RMSNORM = 2;
// pf: the next call's weights, of which each CTA asks L2 to prefetch its share
// of pf_bytes (a multiple of 16) while it runs; null for none.
cudaError_t launch_matvec(int wtype, const void* W, const float* x, const float* aux, float eps, int prod, float* y,
                          int64_t M, int64_t K, const void* pf, uint64_t pf_bytes, int* err, int num_sms, cudaStream_t s,
                          int* status);

// TQ4_1S decode matvec y = W . x (K a multiple of 32; W 16-byte aligned); pf
// as for launch_matvec (the fallback for K % 128 != 0 ignores it).
cudaError_t launch_tq4_matvec(const void* W, const float* x, float* y, int64_t M, int64_t K, const void* pf,
                              uint64_t pf_bytes, int* err, int num_sms, cudaStream_t s, int* status);

// Several tokens (Q4_K or Q5_K, 2 <= N <= LR_TOKENS_MAX) on the decode matvec path:
// Y[N][M] = dequant(W) . X[N][K], the tokens' Q8_1 codes made once into
// `scratch` (device memory; at most ~1.25 N K + 256 N bytes are used);
// *handled = false when the shape or the scratch does not suit it (nothing
// queued).
constexpr int LR_TOKENS_MAX = 7;  // measured crossover with the tensor-core GEMM at the decode shapes
cudaError_t launch_matvec_tokens(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K, int64_t N,
                                 void* scratch, size_t scratch_bytes, int* err, int num_sms, cudaStream_t s,
                                 bool* handled);

// Dense prefill GEMM plan: tiles of 128 weight rows x up to bn = 256 tokens
// (256 rows for a CTA pair), with the K range optionally split across CTAs
// (fixed-order reduction after).
struct GemmPlan {
  int m_tiles;  // 128-row tiles
  int n_tiles, bn, splits;
  bool pair;    // run as CTA pairs (2-SM MMAs) when the device allows it
  int grid;     // CTAs of an unpaired launch
  int num_sms;
  size_t xhat_bytes, partial_bytes, total_bytes;
};
GemmPlan plan_gemm(int wtype, int64_t M, int64_t K, int64_t N, int num_sms);
cudaError_t launch_gemm(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K, int64_t N,
                        void* ws, const GemmPlan& plan, int* err, cudaStream_t s, int* status);

struct MoePlan {
  int m_tiles;
  size_t off_counts, off_offsets, off_tiles, off_queue, off_entries, off_src, off_xhat, total_bytes;
};
MoePlan plan_moe(int wtype, int64_t M, int64_t K, int64_t T, int n_experts, int top_k);
cudaError_t launch_moe(int wtype, const void* W, int n_experts, const int32_t* ids, int top_k, const float* X,
                       float* Y, int64_t M, int64_t K, int64_t T, void* ws, const MoePlan& plan, int* err,
                       int num_sms, cudaStream_t s, int* status);

// out[t][m] = Sum_j probs[t][j] * Y[t][j][m] (the MoE combine), fp32, slot order.
cudaError_t launch_moe_combine(const float* Y, const float* probs, float* out, int64_t M, int64_t T, int top_k,
                               int num_sms, cudaStream_t s);

// Current device, its SM count and the device address of its error word
// (looked up once per device).
cudaError_t device_context(int* dev, int* num_sms, int** err);

// The flag set by kq_test_hold_copies, read when a launch's parameters are made.
int test_hold_copies();

// Raises a kernel's dynamic shared-memory limit to the 227 KB maximum, once per
// device (later calls only read a flag, so launches stay cheap and capturable).
cudaError_t allow_max_smem(const void* kernel, int slot);
constexpr int kSmemSlots = 37;

// Launches `kernel` on `s` with programmatic stream serialization allowed (the
// kernel calls pdl_enter() before its first global memory access).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Builds a 2-D tiled tensor map through the driver entry point.
bool encode_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

}  // namespace kq
