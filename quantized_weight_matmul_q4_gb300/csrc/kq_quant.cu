// Activation quantisation kernels: fp32 -> Q8_1 bytes, and fp32 -> x_hat fp16
// (the Q8_1 value d_h * q, rounded once to fp16) for the tensor-core paths.
#include "kq_internal.h"
#include "kq_quant.cuh"

namespace kq {

// X fp32 [nblk * 32] (token-major, K % 32 == 0) -> nblk Q8_1 blocks of 36 bytes
// laid out as [fp16 d][fp16 s][int8 q[32]].
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float* __restrict__ X, uint8_t* __restrict__ Xq,
                                                            int64_t nblk) {
  pdl_enter();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  const int64_t b = t >> 3;
  const int j = static_cast<int>(t & 7);
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (b < nblk) v = __ldg(reinterpret_cast<const float4*>(X) + t);
  const Q8Quad r = quantize_quad(v);
  if (b < nblk) {
    uint8_t* dst = Xq + b * Q8_1_BYTES;
    *reinterpret_cast<uint32_t*>(dst + 4 + 4 * j) = pack_q4(r.q);
    if (j == 0)
      *reinterpret_cast<uint32_t*>(dst) = static_cast<uint32_t>(__half_as_ushort(r.dh_h)) |
                                          (static_cast<uint32_t>(__half_as_ushort(r.s_h)) << 16);
  }
}

// x_hat = fp16(d_h * q) of four values: the product is exact in fp32 and is
// rounded once.
__device__ __forceinline__ uint2 xhat4(const Q8Quad& r) {
  const __half2 h01 = __halves2half2(__float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[0]))),
                                     __float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[1]))));
  const __half2 h23 = __halves2half2(__float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[2]))),
                                     __float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[3]))));
  return make_uint2(half2_bits(h01), half2_bits(h23));
}

constexpr int XH_UNROLL = 4;   // quads in flight per thread
constexpr int XH_CTAS_PER_SM = 8;

// Output row p of Xh (fp16 [rows][K]) is the Q8_1 value of input row p. Quads
// (4 values) are strided over a grid of a few CTAs per SM, XH_UNROLL loads in
// flight per thread. K / 4 is a multiple of 64 and the stride a multiple of 32,
// so a warp's 32 quads always lie in one row and take the same path.
__global__ void __launch_bounds__(256) quantize_xhat_kernel(const float* __restrict__ X, __half* __restrict__ Xh,
                                                            int K, int64_t rows) {
  pdl_enter();
  const int64_t total = rows * (K >> 2);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * 256;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; t0 < total; t0 += XH_UNROLL * stride) {
    float4 v[XH_UNROLL];
#pragma unroll
    for (int u = 0; u < XH_UNROLL; ++u) {
      const int64_t t = t0 + u * stride;
      if (t < total) v[u] = __ldg(reinterpret_cast<const float4*>(X) + t);
    }
#pragma unroll
    for (int u = 0; u < XH_UNROLL; ++u) {
      const int64_t t = t0 + u * stride;
      if (t < total) reinterpret_cast<uint2*>(Xh)[t] = xhat4(quantize_quad(v[u]));
    }
  }
}

// MoE gather: bucket row slot_pos[i] of Xh is the x_hat row of slot i's token
// (row i / top_k of Xtok, quantised once per token); slots with a negative
// position are skipped. One warp per slot, each lane moving 16-byte pieces of
// the row with GR_UNROLL loads in flight; lane 0 also records
// entries[slot_pos[i]] = i. K * 2 bytes is a multiple of 512, so every lane
// moves whole rounds of 32 x 16 bytes.
constexpr int GR_WARPS = 8;
constexpr int GR_UNROLL = 8;
__global__ void __launch_bounds__(GR_WARPS * 32) gather_rows_kernel(const __half* __restrict__ Xtok,
                                                                    __half* __restrict__ Xh, int K, int64_t n_slots,
                                                                    int top_k, const int* __restrict__ slot_pos,
                                                                    int* __restrict__ entries) {
  pdl_enter();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * GR_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n_slots) return;
  const int pos = __ldg(slot_pos + i);
  if (pos < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(Xtok + (i / top_k) * static_cast<int64_t>(K));
  uint4* dst = reinterpret_cast<uint4*>(Xh + static_cast<int64_t>(pos) * K);
  const int n16 = K / 8;  // 16-byte pieces per row
  for (int c0 = lane; c0 < n16; c0 += 32 * GR_UNROLL) {
    uint4 v[GR_UNROLL];
#pragma unroll
    for (int u = 0; u < GR_UNROLL; ++u)
      if (c0 + 32 * u < n16) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
    for (int u = 0; u < GR_UNROLL; ++u)
      if (c0 + 32 * u < n16) dst[c0 + 32 * u] = v[u];
  }
  if (lane == 0) entries[pos] = static_cast<int>(i);
}

static unsigned xhat_grid(int64_t quads, int num_sms) {
  const int64_t need = (quads + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * XH_CTAS_PER_SM;
  return static_cast<unsigned>(need < cap ? need : cap);
}

cudaError_t launch_quantize_xhat(const float* X, __half* Xh, int64_t K, int64_t rows, int num_sms, cudaStream_t s) {
  const int64_t quads = rows * (K / 4);
  if (quads == 0) return cudaSuccess;
  return launch_pdl(quantize_xhat_kernel, dim3(xhat_grid(quads, num_sms)), dim3(256), 0, s, X, Xh,
                    static_cast<int>(K), rows);
}

cudaError_t launch_gather_rows(const __half* Xtok, __half* Xh, int64_t K, int64_t n_slots, int top_k,
                               const int* slot_pos, int* entries, cudaStream_t s) {
  if (n_slots == 0) return cudaSuccess;
  return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>((n_slots + GR_WARPS - 1) / GR_WARPS)),
                    dim3(GR_WARPS * 32), 0, s, Xtok, Xh, static_cast<int>(K), n_slots, top_k, slot_pos, entries);
}

cudaError_t launch_quantize_q8_1(const float* X, void* Xq, int64_t K, int64_t N, cudaStream_t s) {
  const int64_t nblk = (K / QK8_1) * N;
  const int64_t threads = nblk * 8;
  const int64_t grid = (threads + 255) / 256;
  if (grid == 0) return cudaSuccess;
  return launch_pdl(quantize_q8_1_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, X,
                    static_cast<uint8_t*>(Xq), nblk);
}


}  // namespace kq
