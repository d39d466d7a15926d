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

// Output row p of Xh (fp16 [rows][K]) is the Q8_1 value of input row
// src_rows[p] (or row p when src_rows is null); a negative source row gives
// zeros. Each x_hat = fp16(d_h * q): the product is exact in fp32 and is
// rounded once.
__global__ void __launch_bounds__(256) quantize_xhat_kernel(const float* __restrict__ X, __half* __restrict__ Xh,
                                                            int K, int64_t rows, const int* __restrict__ src_rows) {
  pdl_enter();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;  // quad index in the output
  const int64_t kq4 = K >> 2;
  const int64_t row = t / kq4;
  const int64_t col = (t - row * kq4) << 2;
  bool valid = row < rows;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (valid) {
    const int64_t src = src_rows ? static_cast<int64_t>(__ldg(src_rows + row)) : row;
    if (src >= 0) v = __ldg(reinterpret_cast<const float4*>(X + src * K + col));
  }
  const Q8Quad r = quantize_quad(v);
  if (valid) {
    const __half2 h01 = __halves2half2(__float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[0]))),
                                       __float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[1]))));
    const __half2 h23 = __halves2half2(__float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[2]))),
                                       __float2half_rn(__fmul_rn(r.dh, static_cast<float>(r.q[3]))));
    uint2 o;
    o.x = half2_bits(h01);
    o.y = half2_bits(h23);
    *reinterpret_cast<uint2*>(Xh + row * K + col) = o;
  }
}

cudaError_t launch_quantize_q8_1(const float* X, void* Xq, int64_t K, int64_t N, cudaStream_t s) {
  const int64_t nblk = (K / QK8_1) * N;
  const int64_t threads = nblk * 8;
  const int64_t grid = (threads + 255) / 256;
  if (grid == 0) return cudaSuccess;
  return launch_pdl(quantize_q8_1_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, X,
                    static_cast<uint8_t*>(Xq), nblk);
}

cudaError_t launch_quantize_xhat(const float* X, __half* Xh, int64_t K, int64_t rows, const int* src_rows,
                                 cudaStream_t s) {
  const int64_t threads = rows * (K / 4);
  const int64_t grid = (threads + 255) / 256;
  if (grid == 0) return cudaSuccess;
  return launch_pdl(quantize_xhat_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, X, Xh,
                    static_cast<int>(K), rows, src_rows);
}

}  // namespace kq
