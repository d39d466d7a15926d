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

// MoE activations: token p's x_hat row (the Q8_1 value of X row p, exactly as
// quantize_xhat_kernel makes it) is written to the bucket row slot_pos[s] of
// each of its slots s = p * top_k + j; slots with a negative position (an
// invalid expert id) are skipped, and entries[slot_pos[s]] = s records the slot
// of each bucket row. A warp takes one token's run of QS_ROUNDS rounds of 32
// quads (K / 4 is a multiple of 64, so a run is whole rounds and the eight lanes
// of a Q8_1 block stay together), quantises each round once and stores it to
// every bucket row of the token.
constexpr int QS_WARPS = 8;
constexpr int QS_ROUNDS = 4;
__global__ void __launch_bounds__(QS_WARPS * 32) quantize_scatter_kernel(const float* __restrict__ X,
                                                                        __half* __restrict__ Xh, int K, int64_t T,
                                                                        int top_k, const int* __restrict__ slot_pos,
                                                                        int* __restrict__ entries) {
  pdl_enter();
  const int rounds = K >> 7;  // rounds of 32 quads per row
  const int runs = (rounds + QS_ROUNDS - 1) / QS_ROUNDS;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * QS_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= T * runs) return;
  const int64_t p = w / runs;
  const int run = static_cast<int>(w - p * runs);
  const int r1 = min(rounds, (run + 1) * QS_ROUNDS);
  const float4* xrow = reinterpret_cast<const float4*>(X + p * K);
  uint2* hrow0 = reinterpret_cast<uint2*>(Xh);
  const int64_t quads = K >> 2;
  const int* sp = slot_pos + p * top_k;
  float4 v[QS_ROUNDS];
#pragma unroll
  for (int u = 0; u < QS_ROUNDS; ++u)
    if (run * QS_ROUNDS + u < r1) v[u] = __ldg(xrow + (run * QS_ROUNDS + u) * 32 + lane);
#pragma unroll
  for (int u = 0; u < QS_ROUNDS; ++u) {
    const int r = run * QS_ROUNDS + u;
    if (r >= r1) break;  // warp-uniform
    const uint2 h = xhat4(quantize_quad(v[u]));
    for (int j0 = 0; j0 < top_k; j0 += 32) {
      const int my = (j0 + lane < top_k) ? __ldg(sp + j0 + lane) : -1;
      const int nj = min(32, top_k - j0);
      for (int jj = 0; jj < nj; ++jj) {
        const int pos = __shfl_sync(0xffffffffu, my, jj);
        if (pos >= 0) hrow0[pos * quads + r * 32 + lane] = h;
      }
      if (run == 0 && u == 0 && my >= 0) entries[my] = static_cast<int>(p * top_k + j0 + lane);
    }
  }
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

cudaError_t launch_quantize_scatter(const float* X, __half* Xh, int64_t K, int64_t T, int top_k, const int* slot_pos,
                                   int* entries, cudaStream_t s) {
  const int64_t runs = ((K >> 7) + QS_ROUNDS - 1) / QS_ROUNDS;
  const int64_t warps = T * runs;
  if (warps == 0) return cudaSuccess;
  return launch_pdl(quantize_scatter_kernel, dim3(static_cast<unsigned>((warps + QS_WARPS - 1) / QS_WARPS)),
                    dim3(QS_WARPS * 32), 0, s, X, Xh, static_cast<int>(K), T, top_k, slot_pos, entries);
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
