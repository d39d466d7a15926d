// The MoE combine: each token's slot rows, weighted by the router
// probabilities, summed back into one row ("Prefill Gap Closure Plan", T2: the
// rows are scattered back to their tokens after the grouped expert GEMM):
//
//   out[t][m] = Sum_{j < top_k} probs[t][j] * Y[t][j][m]
//
// in fp32 with one fused multiply-add per slot in slot order, so the result
// does not depend on scheduling. Memory-bound: every Y element is read once.
#include <algorithm>

#include "kq_internal.h"
#include "kq_common.cuh"

namespace kq {

// Four consecutive outputs of one token per thread (M % 4 == 0: the rows of Y
// and out are then 16-byte aligned), grid-strided.
__global__ void __launch_bounds__(256) moe_combine4_kernel(const float* __restrict__ Y, const float* __restrict__ P,
                                                           float* __restrict__ out, int64_t M, int64_t T, int top_k) {
  pdl_enter();
  const int64_t m4 = M >> 2;
  const int64_t total = T * m4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t t = i / m4, c = i - t * m4;
    const float* y = Y + t * top_k * M + 4 * c;
    const float* p = P + t * top_k;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < top_k; ++j) {
      const float pj = __ldg(p + j);
      const float4 v = __ldg(reinterpret_cast<const float4*>(y + j * M));
      acc.x = fmaf(pj, v.x, acc.x);
      acc.y = fmaf(pj, v.y, acc.y);
      acc.z = fmaf(pj, v.z, acc.z);
      acc.w = fmaf(pj, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(out + t * M + 4 * c) = acc;
  }
}

// Any M: one output per thread.
__global__ void __launch_bounds__(256) moe_combine1_kernel(const float* __restrict__ Y, const float* __restrict__ P,
                                                           float* __restrict__ out, int64_t M, int64_t T, int top_k) {
  pdl_enter();
  const int64_t total = T * M;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t t = i / M, m = i - t * M;
    const float* y = Y + t * top_k * M + m;
    const float* p = P + t * top_k;
    float acc = 0.f;
    for (int j = 0; j < top_k; ++j) acc = fmaf(__ldg(p + j), __ldg(y + j * M), acc);
    out[i] = acc;
  }
}

cudaError_t launch_moe_combine(const float* Y, const float* probs, float* out, int64_t M, int64_t T, int top_k,
                               int num_sms, cudaStream_t s) {
  const bool vec4 = (M % 4) == 0;
  const int64_t work = vec4 ? T * (M / 4) : T * M;
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(num_sms) * 8));
  if (vec4)
    return launch_pdl(moe_combine4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, Y, probs, out, M, T,
                      top_k);
  return launch_pdl(moe_combine1_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, Y, probs, out, M, T,
                    top_k);
}

}  // namespace kq
