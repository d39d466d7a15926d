// fp32 -> Q8_1 activation quantisation, one 32-element block per 8 threads.
//
// The quantiser of "06 · 8e/8e② — decode MMVQ" (§2 Principle and §3.2
// ``quantize_pad40_block``), with the Q8_1 block sum of "ZINC MMQ v2" (What
// they do right: Q8_1 activations):
//   amax = max|x|, d = amax / 127, di = 1 / d (0 when d = 0, or when 1 / d
//   is not a finite fp32 value: max|x| below about 3.7e-37, where d_h = fp16(d)
//   is 0 and the block dequantises to 0 whatever its codes),
//   q = clamp(rint(x * di), -128, 127), stored scale d_h = fp16(d),
//   block sum s = fp16(d_h * Sum q).
// Every step is a single IEEE fp32 operation (correctly rounded division,
// product, round-half-even rint), so the integer codes are reproducible
// bit for bit on any IEEE machine. The file is compiled without fast-math.
#pragma once

#include "kq_common.cuh"

namespace kq {

// The reciprocal scale di of a block: 1 / d, or 0 when d is 0 or 1 / d
// overflows (the comparison is false for inf), so that every code is finite.
__device__ __forceinline__ float q8_inv_scale(float d) {
  const float di = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
  return (di <= 3.40282347e38f) ? di : 0.0f;
}

struct Q8Quad {
  int q[4];        // the four codes of this thread
  float dh;        // fp16-rounded scale d_h, as fp32
  __half dh_h;     // d_h
  __half s_h;      // fp16(d_h * Sum q) over the whole block
  int sumq;        // Sum q over the whole block
};

// Quantises the four values v of one thread; the 8 threads of an aligned
// group of 8 lanes hold one 32-element block (thread j holds elements 4j..4j+3).
// All 32 lanes of the warp must call this.
__device__ __forceinline__ Q8Quad quantize_quad(float4 v) {
  float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  const float d = __fdiv_rn(a, 127.0f);
  const float di = q8_inv_scale(d);
  Q8Quad r;
  const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float t = rintf(__fmul_rn(e[j], di));
    r.q[j] = static_cast<int>(fminf(fmaxf(t, -128.0f), 127.0f));
  }
  int s = r.q[0] + r.q[1] + r.q[2] + r.q[3];
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 4);
  r.sumq = s;
  r.dh_h = __float2half_rn(d);
  r.dh = __half2float(r.dh_h);
  r.s_h = __float2half_rn(__fmul_rn(r.dh, static_cast<float>(s)));  // exact product, one rounding
  return r;
}

__device__ __forceinline__ uint32_t pack_q4(const int (&q)[4]) {
  return (static_cast<uint32_t>(q[0]) & 0xFFu) | ((static_cast<uint32_t>(q[1]) & 0xFFu) << 8) |
         ((static_cast<uint32_t>(q[2]) & 0xFFu) << 16) | ((static_cast<uint32_t>(q[3]) & 0xFFu) << 24);
}

// Quantises 8 consecutive values v[0..7] held by one lane; the four lanes of an
// aligned lane quad hold one 32-element block (lane 4i + j: elements 8j..8j+7).
// Same arithmetic as quantize_quad. All four lanes of the quad must call it.
struct Q8Oct {
  uint32_t q[2];   // 8 packed int8 codes
  float dh;        // fp16-rounded block scale d_h, as fp32
  int sumq;        // Sum q over the whole 32-element block
};

__device__ __forceinline__ Q8Oct quantize_oct(const float (&v)[8]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  const float d = __fdiv_rn(a, 127.0f);
  const float di = q8_inv_scale(d);
  // q = rint(p) with p = fl(x * di): adding 1.5 * 2^23 to p (|p| < 2^22) rounds it
  // to the nearest integer, ties to even, into the low mantissa bits, whose low
  // byte is then q as a two's-complement int8; four such bytes are gathered by
  // byte permutes and summed by one dp4a. |p| never exceeds 127.0001 (amax * di
  // with di = 1 / fl(amax / 127), also for subnormal d; di = 0 where 1 / d
  // overflows), so the clamp to [-128, 127] of the definition never applies.
  Q8Oct r;
  int s = 0;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    uint32_t u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = __float_as_uint(__fadd_rn(__fmul_rn(v[4 * w + k], di), 12582912.0f));
    r.q[w] = __byte_perm(__byte_perm(u[0], u[1], 0x0040), __byte_perm(u[2], u[3], 0x0040), 0x5410);
    s = __dp4a(static_cast<int>(r.q[w]), 0x01010101, s);
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  r.sumq = s;
  r.dh = __half2float(__float2half_rn(d));
  return r;
}

}  // namespace kq
