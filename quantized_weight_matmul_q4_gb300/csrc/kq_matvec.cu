// Decode matvec y[M] = dequant(W)[M,K] . x[K] for Q4_K, Q5_K and Q6_K weights,
// with the fp32 -> Q8_1 quantisation of x (and optionally its RMSNorm or
// SwiGLU producer) fused in. Q5_K is the Q4_K value with a fifth bit per code
// (the page's "one kernel per type" sibling), read with the GGUF block layout.
//
// Method: "06 · 8e/8e② — decode MMVQ: dp4a integer dot products + the
// llama.cpp launch table", §2 Principle and §3.2 Key code: per 32-weight
// sub-block an exact integer dot of the 4-bit codes with the int8 activation
// codes (dp4a), the min term taken from the activation block sum
// (W.x = Sum_sub [d*sc*d8*Sum(nib*q) - dmin*m*d8*Sum(q)]), and a warp-shuffle
// reduction per row. The page's launch geometry (one 256-thread block per row,
// plain loads) was made for a 273 GB/s LPDDR part; here the rows of the
// row-major matrix are contiguous, so each CTA owns a balanced contiguous range
// of rows and streams it through a shared-memory ring of ~16 KB chunks with 1-D
// bulk copies (one elected producer thread, mbarrier completion): every byte of
// W is read from HBM once, and at the decode sizes a CTA's whole range is in
// flight within the first microsecond. The consumer threads quantise x into
// shared memory while the first chunks land; then each thread takes whole
// super-blocks (row, block) in arrival order, so a block's header is decoded
// once for its 256 weights, and writes one partial sum per block; each row's
// partials are added in a fixed order at the end (deterministic). That is the
// item kernel (matvec_kernel); the lane-row kernel further down stages whole row
// ranges by TMA and is the one the decode shapes take for Q4_K and Q5_K.
#include <algorithm>

#include "kq_internal.h"
#include "kq_quant.cuh"

namespace kq {

constexpr int MV_CWARPS = 16;                       // consumer warps
constexpr int MV_CTHREADS = MV_CWARPS * 32;
constexpr int MV_THREADS = MV_CTHREADS + 32;        // + one producer warp
constexpr int MV_SMEM_LIMIT = 227 * 1024;
constexpr int MV_PART_MAX = 4096;                   // block partials per row group
constexpr int MV_CHUNK_BLOCKS_Q4K = 112;            // 16128 B per chunk
constexpr int MV_CHUNK_BLOCKS_Q6K = 80;             // 16800 B per chunk
// Q6_K rows with K < 8192 take 25200-byte chunks, fewer and larger copies
// (measured: decode 11008 x 4096 went from 11.0 to 9.8 us per launch with them;
// 4096 x 11008 went from 11.6 to 11.8 us, so longer rows keep 80 blocks).
constexpr int MV_CHUNK_BLOCKS_Q6K_SHORT_K = 120;
constexpr int MV_Q6K_LONG_K = 8192;
constexpr int MV_CHUNK_BLOCKS_Q5K = 92;             // 16192 B per chunk
constexpr int MV_MAX_RING = 14;

struct MatvecParams {
  const uint8_t* W;
  const float* x;       // x, or the gate of SwiGLU
  const float* aux;     // SwiGLU: up; RMSNorm: gamma
  float eps;            // RMSNorm
  float* y;
  int M, K, nb;
  int bb;               // bytes per block (144 or 210)
  int rs;               // bytes per weight row
  int64_t w_bytes;      // M * rs: copies never read past this
  int chunk_blocks;     // blocks per ring chunk
  int chunk_bytes;      // chunk_blocks * bb (a multiple of 16)
  int slot_bytes;       // ring slot stride (multiple of 128)
  int n_ring;           // ring depth (chunks)
  int rows_per_group;   // rows whose block partials are reduced together
  int xq_bytes;         // int8 activation codes (block-swizzled 16-byte pieces)
  int xds_bytes;        // per-32 activation scales and sums
  const uint8_t* pf;    // the next call's weights, prefetched into L2 (or null)
  uint64_t pf_bytes;    // a multiple of 16
  int* err;
  int hold;             // kq_test_hold_copies: the producer issues nothing
};

// Activation codes live in 16-byte pieces; piece j (0..15) of K-block b is
// stored at piece j ^ (b & 7). Threads that read the same piece of eight
// consecutive blocks hit eight different bank groups.
__device__ __forceinline__ int xq_piece(int b, int j) { return (b << 8) + ((j ^ (b & 7)) << 4); }

// Q4_K: per (block b, 32-byte chunk c) one int4 {d8 of sub 2c, d8 of sub 2c+1,
// Sum q of sub 2c, Sum q of sub 2c+1}, stored at 4b + (c ^ ((b >> 1) & 3)).
__device__ __forceinline__ int xds_q4k(int b, int c) { return 4 * b + (c ^ ((b >> 1) & 3)); }
// Q6_K: per 32-block g8 (0..7) of block b one int4 {d8, Sum q of the first 16,
// Sum q of the last 16, 0}, stored at 8b + (g8 ^ (b & 7)).
__device__ __forceinline__ int xds_q6k(int b, int g8) { return 8 * b + (g8 ^ (b & 7)); }

__device__ __forceinline__ float i2f(int v) { return static_cast<float>(v); }

// The producer of the activations that the quantiser takes, fused into the
// matvec ("06 · 8e/8e② — decode MMVQ", §3.2 Key code: the Q8_1 quantisation
// moved into the RMSNorm and SwiGLU producers): PROD_X reads x; PROD_SWIGLU
// makes silu(g) * u from gate g = x and up u = aux; PROD_RMSNORM makes
// x * inv_rms * gamma with gamma = aux. All in fp32.
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Activations k .. k+3 (k a multiple of 4).
template <int PROD>
__device__ __forceinline__ float4 produce4(const float* __restrict__ x, const float* __restrict__ aux, int k,
                                           float inv_rms) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(x + k));
  if (PROD == PROD_X) return a;
  const float4 b = __ldg(reinterpret_cast<const float4*>(aux + k));
  if (PROD == PROD_SWIGLU)
    return make_float4(silu_f(a.x) * b.x, silu_f(a.y) * b.y, silu_f(a.z) * b.z, silu_f(a.w) * b.w);
  return make_float4(a.x * inv_rms * b.x, a.y * inv_rms * b.y, a.z * inv_rms * b.z, a.w * inv_rms * b.w);
}

// RMSNorm's 1 / sqrt(mean(x^2) + eps) over x[0 .. K), computed by the nthreads
// consumer threads of the CTA (named barrier 1) in a fixed order: each thread
// sums its quads, warps reduce by shuffles, then every thread adds the warp sums
// in warp order. red: nthreads / 32 floats of shared memory.
__device__ __forceinline__ float rms_inv(const float* __restrict__ x, int K, float eps, float* red, int nthreads) {
  float ss = 0.f;
  for (int q = threadIdx.x; q < (K >> 2); q += nthreads) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(x) + q);
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  ss = warp_sum_f(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  float tot = 0.f;
  for (int w = 0; w < (nthreads >> 5); ++w) tot += red[w];
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");  // red is free again
  return rsqrtf(tot / static_cast<float>(K) + eps);
}

// Sum over one Q4_K super-block (256 weights) of w * x_hat, by the min-term
// identity: d * Sum_sub d8*sc*dot(nib, q) - dmin * Sum_sub d8*m*Sum(q).
__device__ __forceinline__ float block_dot_q4k(const uint8_t* __restrict__ blk, int b, const uint8_t* __restrict__ xq,
                                               const int4* __restrict__ xds) {
  const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
  // 6-bit scales and mins, one per byte: sub-blocks 0..3 and 4..7
  const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
  const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
  const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
  float acc_lo = 0.f, acc_hi = 0.f, acc_m = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
    const int4 x0 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 0));
    const int4 x1 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 1));
    const int4 x2 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 2));
    const int4 x3 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 3));
    const int4 ds = xds[xds_q4k(b, c)];
    // sub-block 2c: low nibbles against elements 0..31 of the chunk
    int dA = __dp4a(static_cast<int>(qa.x & 0x0F0F0F0Fu), x0.x, 0);
    dA = __dp4a(static_cast<int>(qa.y & 0x0F0F0F0Fu), x0.y, dA);
    dA = __dp4a(static_cast<int>(qa.z & 0x0F0F0F0Fu), x0.z, dA);
    dA = __dp4a(static_cast<int>(qa.w & 0x0F0F0F0Fu), x0.w, dA);
    dA = __dp4a(static_cast<int>(qb.x & 0x0F0F0F0Fu), x1.x, dA);
    dA = __dp4a(static_cast<int>(qb.y & 0x0F0F0F0Fu), x1.y, dA);
    dA = __dp4a(static_cast<int>(qb.z & 0x0F0F0F0Fu), x1.z, dA);
    dA = __dp4a(static_cast<int>(qb.w & 0x0F0F0F0Fu), x1.w, dA);
    // sub-block 2c+1: high nibbles kept in place (16 x nibble), against 32..63
    int dB = dp4a_us(qa.x & 0xF0F0F0F0u, x2.x, 0);
    dB = dp4a_us(qa.y & 0xF0F0F0F0u, x2.y, dB);
    dB = dp4a_us(qa.z & 0xF0F0F0F0u, x2.z, dB);
    dB = dp4a_us(qa.w & 0xF0F0F0F0u, x2.w, dB);
    dB = dp4a_us(qb.x & 0xF0F0F0F0u, x3.x, dB);
    dB = dp4a_us(qb.y & 0xF0F0F0F0u, x3.y, dB);
    dB = dp4a_us(qb.z & 0xF0F0F0F0u, x3.z, dB);
    dB = dp4a_us(qb.w & 0xF0F0F0F0u, x3.w, dB);
    const uint32_t scw = (c < 2) ? sc_lo : sc_hi;
    const uint32_t mw = (c < 2) ? m_lo : m_hi;
    const int sh = (c & 1) * 16;
    const int scA = (scw >> sh) & 0xFF, scB = (scw >> (sh + 8)) & 0xFF;
    const int mA = (mw >> sh) & 0xFF, mB = (mw >> (sh + 8)) & 0xFF;
    const float d8A = __int_as_float(ds.x), d8B = __int_as_float(ds.y);
    acc_lo = fmaf(d8A, i2f(scA * dA), acc_lo);
    acc_hi = fmaf(d8B, i2f(scB * dB), acc_hi);
    acc_m = fmaf(d8A, i2f(mA * ds.z), acc_m);
    acc_m = fmaf(d8B, i2f(mB * ds.w), acc_m);
  }
  return d * fmaf(acc_hi, 0.0625f, acc_lo) - dmin * acc_m;
}

// Q5_K codes of four weights: the low (LO) or high nibbles of the four qs
// bytes in w, with the fifth bit, bit `BIT` of the matching qh bytes in h,
// moved to bit 4 of each byte (the Q5_K block: the Q4_K fields with qh[32] at
// byte 16 and the nibbles at byte 48; weight r of sub-block j has its fifth
// bit in bit j of qh[r]).
template <bool LO, int BIT>
__device__ __forceinline__ int q5_codes(uint32_t w, uint32_t h) {
  const uint32_t hb = (BIT <= 4 ? (h << (4 - BIT)) : (h >> (BIT - 4))) & 0x10101010u;
  return static_cast<int>(((LO ? w : (w >> 4)) & 0x0F0F0F0Fu) | hb);
}

// Integer dots of one 64-weight chunk of a Q5_K block: sub-block J (low
// nibbles, against x0 | x1) into dA and sub-block J + 1 (high nibbles, against
// x2 | x3) into dB. qa, qb: the chunk's 32 nibble bytes; ha, hb: qh[0..15] and
// qh[16..31].
template <int J>
__device__ __forceinline__ void q5_chunk_dots(const uint4& qa, const uint4& qb, const uint4& ha, const uint4& hb,
                                              const int4& x0, const int4& x1, const int4& x2, const int4& x3, int& dA,
                                              int& dB) {
  dA = __dp4a(q5_codes<true, J>(qa.x, ha.x), x0.x, 0);
  dA = __dp4a(q5_codes<true, J>(qa.y, ha.y), x0.y, dA);
  dA = __dp4a(q5_codes<true, J>(qa.z, ha.z), x0.z, dA);
  dA = __dp4a(q5_codes<true, J>(qa.w, ha.w), x0.w, dA);
  dA = __dp4a(q5_codes<true, J>(qb.x, hb.x), x1.x, dA);
  dA = __dp4a(q5_codes<true, J>(qb.y, hb.y), x1.y, dA);
  dA = __dp4a(q5_codes<true, J>(qb.z, hb.z), x1.z, dA);
  dA = __dp4a(q5_codes<true, J>(qb.w, hb.w), x1.w, dA);
  dB = __dp4a(q5_codes<false, J + 1>(qa.x, ha.x), x2.x, 0);
  dB = __dp4a(q5_codes<false, J + 1>(qa.y, ha.y), x2.y, dB);
  dB = __dp4a(q5_codes<false, J + 1>(qa.z, ha.z), x2.z, dB);
  dB = __dp4a(q5_codes<false, J + 1>(qa.w, ha.w), x2.w, dB);
  dB = __dp4a(q5_codes<false, J + 1>(qb.x, hb.x), x3.x, dB);
  dB = __dp4a(q5_codes<false, J + 1>(qb.y, hb.y), x3.y, dB);
  dB = __dp4a(q5_codes<false, J + 1>(qb.z, hb.z), x3.z, dB);
  dB = __dp4a(q5_codes<false, J + 1>(qb.w, hb.w), x3.w, dB);
}

// Sum over one Q5_K super-block of w * x_hat, w = d * sc * q - dmin * m with q
// the 5-bit code: the Q4_K form with the codes built by q5_codes.
__device__ __forceinline__ float block_dot_q5k(const uint8_t* __restrict__ blk, int b, const uint8_t* __restrict__ xq,
                                               const int4* __restrict__ xds) {
  const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
  const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
  const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
  const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
  const uint4 ha = *reinterpret_cast<const uint4*>(blk + 16);  // qh[0..15]
  const uint4 hb = *reinterpret_cast<const uint4*>(blk + 32);  // qh[16..31]
  float acc = 0.f, acc_m = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 48 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 64 + 32 * c);
    const int4 x0 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 0));
    const int4 x1 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 1));
    const int4 x2 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 2));
    const int4 x3 = *reinterpret_cast<const int4*>(xq + xq_piece(b, 4 * c + 3));
    const int4 ds = xds[xds_q4k(b, c)];
    int dA, dB;
    if (c == 0) q5_chunk_dots<0>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
    else if (c == 1) q5_chunk_dots<2>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
    else if (c == 2) q5_chunk_dots<4>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
    else q5_chunk_dots<6>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
    const uint32_t scw = (c < 2) ? sc_lo : sc_hi;
    const uint32_t mw = (c < 2) ? m_lo : m_hi;
    const int sh = (c & 1) * 16;
    const int scA = (scw >> sh) & 0xFF, scB = (scw >> (sh + 8)) & 0xFF;
    const int mA = (mw >> sh) & 0xFF, mB = (mw >> (sh + 8)) & 0xFF;
    const float d8A = __int_as_float(ds.x), d8B = __int_as_float(ds.y);
    acc = fmaf(d8A, i2f(scA * dA), acc);
    acc = fmaf(d8B, i2f(scB * dB), acc);
    acc_m = fmaf(d8A, i2f(mA * ds.z), acc_m);
    acc_m = fmaf(d8B, i2f(mB * ds.w), acc_m);
  }
  return d * acc - dmin * acc_m;
}

// Sum over one Q6_K super-block of w * x_hat, w = d * sc * (q - 32), taken as
// d * Sum_16 sc * d8 * (dot(q, x) - 32 * Sum x) per group of 16 weights.
// A 210-byte block is only 2-byte aligned in shared memory: its 53 words are
// read once as the 54 4-byte aligned words around it and each is rebuilt with
// one funnel shift (by 0 or 16 bits). Block word k: ql[4k..] for k < 32, qh
// for 32 <= k < 48, the int8 scales for 48..51, d in the low half of word 52.
// (The words read past the block's end stay inside its ring slot and only
// feed bits that are not used.)
__device__ __forceinline__ float block_dot_q6k(const uint8_t* __restrict__ blk, int b, const uint8_t* __restrict__ xq,
                                               const int4* __restrict__ xds) {
  const uint32_t* aw = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(blk) & ~uintptr_t(3));
  const uint32_t sh = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(blk) & 2) * 8;  // 0 or 16
  uint32_t u[54];
#pragma unroll
  for (int k = 0; k < 54; ++k) u[k] = aw[k];
  uint32_t w[53];
#pragma unroll
  for (int k = 0; k < 53; ++k) w[k] = __funnelshift_r(u[k], u[k + 1], sh);
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(w[52] & 0xFFFFu)));
  float acc = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int g8 = 4 * h + g;  // 32-weight group inside the block
      const int4 xa = *reinterpret_cast<const int4*>(xq + xq_piece(b, 2 * g8));
      const int4 xb = *reinterpret_cast<const int4*>(xq + xq_piece(b, 2 * g8 + 1));
      const int xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      int dot0 = 0, dot1 = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t l = w[16 * h + 8 * (g & 1) + i];   // ql[64h + 32(g & 1) + 4i ..]
        const uint32_t hq = w[32 + 8 * h + i];              // qh[32h + 4i ..]
        const uint32_t lo = (g < 2) ? l : (l >> 4);
        const uint32_t hi = (g < 2) ? (hq << (4 - 2 * g)) : (hq >> (2 * g - 4));
        const uint32_t q = (lo & 0x0F0F0F0Fu) | (hi & 0x30303030u);  // the 6-bit codes of four weights
        if (i < 4)
          dot0 = dp4a_us(q, xv[i], dot0);
        else
          dot1 = dp4a_us(q, xv[i], dot1);
      }
      const int4 ds = xds[xds_q6k(b, g8)];
      const int si = 8 * h + 2 * g;  // scale index of the first 16 weights
      const int sc0 = static_cast<int>(static_cast<int8_t>(w[48 + (si >> 2)] >> (8 * (si & 3))));
      const int sc1 = static_cast<int>(static_cast<int8_t>(w[48 + (si >> 2)] >> (8 * (si & 3) + 8)));
      const int t = sc0 * (dot0 - 32 * ds.y) + sc1 * (dot1 - 32 * ds.z);
      acc = fmaf(__int_as_float(ds.x), i2f(t), acc);
    }
  }
  return d * acc;
}

template <int WT, int PROD>
__global__ void __launch_bounds__(MV_THREADS, 1) matvec_kernel(const MatvecParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* xq = smem;
  int4* xds = reinterpret_cast<int4*>(smem + p.xq_bytes);
  float* part = reinterpret_cast<float*>(smem + p.xq_bytes + p.xds_bytes);
  uint8_t* ring = reinterpret_cast<uint8_t*>(part + MV_PART_MAX);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(p.n_ring) * p.slot_bytes);
  uint64_t* empty = full + p.n_ring;
  volatile int* abort = reinterpret_cast<volatile int*>(empty + p.n_ring);
  volatile int* issued = abort + 1;  // chunks the producer has issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.M / gridDim.x);
  const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.M / gridDim.x);
  const int n_items = (r1 - r0) * p.nb;                 // (row, block) pairs of this CTA
  const int n_chunks = (n_items + p.chunk_blocks - 1) / p.chunk_blocks;
  // Q6_K rows are 16-byte multiples only when K / 256 is a multiple of 8, so
  // a CTA's first row need not start on a 16-byte boundary: its copies then
  // start `lead` bytes early, at the aligned address below, and every item of
  // a slot sits `lead` bytes in.
  const int64_t start = static_cast<int64_t>(r0) * p.rs;
  const int lead = static_cast<int>(start & 15);

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_ring; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], p.chunk_blocks);
    }
    *abort = 0;
    *issued = 0;
    fence_mbar_init();
  }
  // Programmatic dependent launch: the weight stream does not depend on the
  // previous kernel (W is read-only; the caller's contract), so the producer
  // starts at once; the consumers wait for the previous grid before reading x.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();

  if (warp == MV_CWARPS) {
    // Producer: the CTA's contiguous byte range, chunk by chunk, through the ring.
    if (lane == 0 && !p.hold) {
      const uint8_t* base = p.W + (start - lead);         // 16-byte aligned
      const int64_t total = static_cast<int64_t>(n_items) * p.bb;
      for (int c = 0; c < n_chunks; ++c) {
        const int slot = c % p.n_ring;
        if (c >= p.n_ring && !mbar_wait(&empty[slot], ((c / p.n_ring) & 1) ^ 1, abort, p.err)) break;
        const int64_t off = static_cast<int64_t>(c) * p.chunk_bytes;  // a multiple of 16
        // The chunk's items end `bytes` past base + off. The copy rounds that up
        // to 16 bytes unless it would pass the end of W; then this thread copies
        // the ragged tail (< 16 B) itself.
        const uint32_t bytes =
            static_cast<uint32_t>(lead + min(static_cast<int64_t>(p.chunk_bytes), total - off));
        const int64_t room = p.w_bytes - (start - lead) - off;
        uint32_t main_bytes = (bytes + 15u) & ~15u;
        if (main_bytes > room) main_bytes = bytes & ~15u;
        uint8_t* dst = ring + static_cast<size_t>(slot) * p.slot_bytes;
        for (uint32_t i = main_bytes; i < bytes; ++i) dst[i] = base[off + i];
        mbar_expect_tx(&full[slot], main_bytes);
        if (main_bytes) bulk_g2s(dst, base + off, main_bytes, &full[slot]);
        *issued = c + 1;
      }
      // Every copy lands before the CTA may exit (also when the consumers gave up).
      const int done = *issued;
      for (int sl = 0; sl < min(done, p.n_ring); ++sl) {
        const int fills = (done - sl + p.n_ring - 1) / p.n_ring;
        if (!mbar_wait_bounded(&full[sl], (fills - 1) & 1)) report_error(p.err, ERR_WAIT_TIMEOUT);
      }
    }
    return;
  }

  // Consumers: quantise x to Q8_1 in shared memory while the first chunks land.
  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
  const float inv_rms = (PROD == PROD_RMSNORM) ? rms_inv(p.x, p.K, p.eps, part, MV_CTHREADS) : 0.f;
  const int nq = p.K >> 2;
  for (int base = 0; base < nq; base += 4 * MV_CTHREADS) {
    float4 xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qd = base + i * MV_CTHREADS + threadIdx.x;
      xv[i] = qd < nq ? produce4<PROD>(p.x, p.aux, 4 * qd, inv_rms) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qd = base + i * MV_CTHREADS + threadIdx.x;
      const Q8Quad r = quantize_quad(xv[i]);
      // Sum q over this thread's half (16 values) of the 32-block
      int s4 = r.q[0] + r.q[1] + r.q[2] + r.q[3];
      s4 += __shfl_xor_sync(0xffffffffu, s4, 1);
      s4 += __shfl_xor_sync(0xffffffffu, s4, 2);
      const int s_hi = __shfl_down_sync(0xffffffffu, s4, 4);
      if (qd < nq) {
        const int k = qd << 2;
        const int b = k >> 8, j = (k >> 4) & 15;
        *reinterpret_cast<uint32_t*>(xq + xq_piece(b, j) + (k & 15)) = pack_q4(r.q);
        if ((qd & 7) == 0) {
          const int g8 = (k >> 5) & 7;
          if (WT != KQ_Q6_K) {  // Q4_K and Q5_K share the sub-block layout
            int* e = reinterpret_cast<int*>(&xds[xds_q4k(b, g8 >> 1)]);
            e[g8 & 1] = __float_as_int(r.dh);
            e[2 + (g8 & 1)] = r.sumq;
          } else {
            xds[xds_q6k(b, g8)] = make_int4(__float_as_int(r.dh), s4, s_hi, 0);
          }
        }
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(MV_CTHREADS) : "memory");
  // The next call's weights are asked of L2 once x is in (eight warps, an eighth
  // each), as in the lane-row kernel: 12.3 -> 11.5 us per Q6_K decode launch.
  if (lane == 0 && warp < 8) prefetch_slice_l2(p.pf, p.pf_bytes, warp, 8);

  // Items (row, block) in arrival order; one partial per item, reduced per row.
  const int items_per_group = p.rows_per_group * p.nb;
  for (int g0 = 0; g0 < n_items; g0 += items_per_group) {
    const int g1 = min(n_items, g0 + items_per_group);
    bool ok = true;
    for (int it = g0 + threadIdx.x; it < g1; it += MV_CTHREADS) {
      const int c = it / p.chunk_blocks;
      const int slot = c % p.n_ring;
      // chunk c issued: the slot's completed fills are c / n_ring or one more,
      // so the parity wait below is unambiguous
      if (!wait_counter_above(issued, c, abort, p.err) || !mbar_wait(&full[slot], (c / p.n_ring) & 1, abort, p.err)) {
        ok = false;
        break;
      }
      const uint8_t* blk = ring + static_cast<size_t>(slot) * p.slot_bytes + lead +
                           static_cast<size_t>(it - c * p.chunk_blocks) * p.bb;
      const int b = it % p.nb;
      part[it - g0] = (WT == KQ_Q4_K)   ? block_dot_q4k(blk, b, xq, xds)
                      : (WT == KQ_Q5_K) ? block_dot_q5k(blk, b, xq, xds)
                                        : block_dot_q6k(blk, b, xq, xds);
      mbar_arrive(&empty[slot]);
    }
    (void)ok;
    asm volatile("bar.sync 1, %0;" ::"r"(MV_CTHREADS) : "memory");
    // Row sums: S lanes per row (the largest power of two up to 32 that keeps
    // every row of the group in one pass), each adding every S-th partial, then
    // a butterfly over the S lanes. The order is fixed: deterministic.
    const int rows = (g1 - g0) / p.nb;
    int S = 32;
    while (S > 1 && rows * S > MV_CTHREADS) S >>= 1;
    for (int t0 = 0; t0 < rows * S; t0 += MV_CTHREADS) {
      const int t = t0 + threadIdx.x, r = t / S, j = t % S;
      float acc = 0.f;
      if (r < rows) {
        const float* pr = part + r * p.nb;
        for (int i = j; i < p.nb; i += S) acc += pr[i];
      }
      for (int o = S >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (r < rows && j == 0) p.y[r0 + g0 / p.nb + r] = acc;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(MV_CTHREADS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// Q4_K decode matvec, "lane = row" form (the decode fast path, used when a
// CTA's rows fit in shared memory: decode matrices up to ~30 MB).
//
// CTA c owns the R rows [c*R, c*R + R) (R <= 128; the last CTA may have
// fewer) and stages all of them at once, so a whole call's weights are in
// flight within the first microsecond. The rows are cut into chunks of cb
// super-blocks (cb odd, up to 7: 1008 contiguous bytes per row); a chunk is one
// 2-D tensor copy of R rows x cb*144 bytes with its own mbarrier, and the
// producer thread issues every chunk as soon as the CTA starts, before the
// kernel waits for the previous kernel on the stream (the weights do not depend
// on it). The copies are contiguous row segments, which HBM streams at full
// rate, and chunks land in issue order.
//
// After the dependency wait the consumer warps quantise x to Q8_1 in shared
// memory (eight values per thread, four threads per 32-block). The work items
// (chunk, row group of 32 rows, block of the chunk) are dealt to the warps in
// chunk order, so the items of a chunk run on different warps as soon as it
// lands and only the last chunk's items remain once the stream ends. For an
// item, each lane takes one row: it decodes the block header (d, dmin, eight
// 6-bit scales and mins) once and accumulates the four 64-weight chunks with
// dp4a against the activation codes, which all lanes read at one address
// (broadcast). The row pitch cb*144 bytes is an odd number of 16-byte units, so
// 32 lanes reading one offset of 32 rows hit distinct bank groups. A warp
// adds its items into one register per row group, in item order; the warps'
// sums are added in warp order at the end (deterministic).
// ---------------------------------------------------------------------------
// Two builds: 24 consumer warps with all of a CTA's rows staged at once (one CTA
// per SM), or 14 consumer warps with a ring of chunk slots in at most half of
// an SM's shared memory (two CTAs per SM), for row ranges that do not fit
// whole.
constexpr int LR_NW_FULL = 24;
constexpr int LR_NW_RING = 14;
constexpr int LR_NW_TOK = 16;               // several-token kernel: its per-token sums need the
                                             // registers of a 17-warp CTA (96 a thread)
constexpr int LR_RING_SMEM = 113 * 1024;     // two CTAs per SM (228 KB, 1 KB reserved per CTA)
constexpr int LR_MAX_ROWS = 128;             // rows per CTA: at most four row groups
constexpr int LR_XT = 2;                     // 8-value activation tasks loaded per thread per round
constexpr int LR_NT = 4;                     // tokens per pass of the several-token kernel (else 2 when
                                             // four tokens' activations do not fit beside the weights)

struct MatvecLaneRowParams {
  const float* x;   // [n_tok][K]; one token: x, or the gate of SwiGLU
  const float* aux; // one token: SwiGLU up, or RMSNorm gamma
  float eps;        // RMSNorm
  float* y;         // [n_tok][M]
  int n_tok;        // tokens (1 for the decode matvec)
  int M, K, nb;
  int R;            // rows per CTA
  int n_groups;     // ceil(R / 32)
  int cb;           // super-blocks per chunk (odd)
  int tail_cb;      // super-blocks in the last chunk's slot (cb, or only the rest when the plan trims it)
  int n_chunks;     // ceil(nb / cb)
  int chunk_bytes;  // shared-memory stride of a chunk (R * cb * 144 rounded up to 128)
  int S;            // chunk slots (== n_chunks: everything staged at once; fewer: a ring)
  uint32_t inv_per_chunk, inv_cb;  // ceil(2^32 / d) for d = n_groups * cb and d = cb
  int xq_off, xs_off, part_off, bar_off;  // shared-memory layout (bytes)
  int xq_tok, xs_tok;                     // bytes of one token's codes and of its {d8, s} pairs
  const uint8_t* xq_g;                    // several tokens: codes [n_tok][xq_tok], quantised beforehand
  const uint8_t* xs_g;                    // several tokens: {d8, s} pairs [n_tok][xs_tok]
  const uint8_t* pf;                      // the next call's weights, prefetched into L2 (or null)
  uint64_t pf_bytes;                      // a multiple of 16
  int* err;
  int hold;                               // kq_test_hold_copies: the weight producer issues nothing
};


template <int NW, bool RING, int PROD, int WT = KQ_Q4_K>
__global__ void __launch_bounds__((NW + 1) * 32, RING ? 2 : 1)
    matvec_q4k_lanerow_kernel(const __grid_constant__ CUtensorMap tmW, const MatvecLaneRowParams p) {
  static_assert(WT == KQ_Q4_K || WT == KQ_Q5_K, "Q4_K or Q5_K super-blocks");
  constexpr int BB = (WT == KQ_Q5_K) ? Q5K_BYTES : Q4K_BYTES;  // bytes per super-block
  constexpr int LR_CT = NW * 32;
  extern __shared__ __align__(1024) uint8_t smem[];
  int8_t* xq = reinterpret_cast<int8_t*>(smem + p.xq_off);
  float2* xs = reinterpret_cast<float2*>(smem + p.xs_off);  // per 32-block: {d8, d8 * Sum q}
  float* part = reinterpret_cast<float*>(smem + p.part_off);  // [warp][row group][lane]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);  // one per slot
  uint64_t* empty = full + p.S;
  volatile int* abort = reinterpret_cast<volatile int*>(empty + p.S);
  volatile int* chunks_issued = abort + 1;  // ring form: chunks the producer has issued

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * p.R;
  const int rows = min(p.R, p.M - r0);

  const int per_chunk = p.n_groups * p.cb;  // work items per chunk
  if (threadIdx.x == 0) {
    for (int sl = 0; sl < p.S; ++sl) {
      mbar_init(&full[sl], 1);
      if (RING) mbar_init(&empty[sl], per_chunk);  // every item of a chunk, computed or skipped, arrives once
    }
    *abort = 0;
    *chunks_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {
    const uint32_t box = static_cast<uint32_t>(p.R * p.cb * BB);
    if (!RING) {
      // Staged form: chunk 0 at once, so that the first work items find their
      // weights; the other chunks only when the dependency wait returns, beside
      // the consumers' loads of x. Issued at the CTA's start, the whole range
      // (~167 KB per SM) held up those loads behind the wait (6.1 against 5.5 us
      // per decode launch); issued once x has landed, it came too late for the
      // dots (6.1 us).
      if (lane == 0 && !p.hold) {
        tma_prefetch_desc(&tmW);
        mbar_expect_tx(&full[0], box);
        tma_load_2d(smem, &tmW, &full[0], 0, r0);
      }
      __syncwarp();
      asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    if (lane == 0 && !p.hold) {
      if (!RING) {
        for (int c = 1; c < p.n_chunks; ++c) {
          mbar_expect_tx(&full[c], box);
          tma_load_2d(smem + static_cast<size_t>(c) * p.chunk_bytes, &tmW, &full[c], c * p.cb * (BB / 4), r0);
        }
        // Every copy lands before the CTA may exit (also when the consumers gave up).
        for (int c = 0; c < p.n_chunks; ++c)
          if (!mbar_wait_bounded(&full[c], 0)) report_error(p.err, ERR_WAIT_TIMEOUT);
      } else {
        tma_prefetch_desc(&tmW);
        int issued = 0;
        for (int c = 0; c < p.n_chunks; ++c) {
          const int sl = c % p.S;
          if (c == p.S) prefetch_share_l2(p.pf, p.pf_bytes);  // once the ring is primed
          if (c >= p.S && !mbar_wait(&empty[sl], ((c / p.S) - 1) & 1, abort, p.err)) break;
          mbar_expect_tx(&full[sl], box);
          tma_load_2d(smem + static_cast<size_t>(sl) * p.chunk_bytes, &tmW, &full[sl], c * p.cb * (BB / 4), r0);
          issued = c + 1;
          *chunks_issued = issued;
        }
        if (p.n_chunks <= p.S) prefetch_share_l2(p.pf, p.pf_bytes);
        // Every copy lands before the CTA may exit (also when the consumers gave up).
        for (int sl = 0; sl < min(issued, p.S); ++sl) {
          const int fills = (issued - sl + p.S - 1) / p.S;
          if (!mbar_wait_bounded(&full[sl], (fills - 1) & 1)) report_error(p.err, ERR_WAIT_TIMEOUT);
        }
      }
    }
    return;
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel

  // x -> Q8_1 in shared memory: task t quantises x[8t .. 8t+8); the four tasks
  // of a 32-block sit on four consecutive lanes. nt is a multiple of 32, so a
  // warp's tasks are all in range or all out of range.
  const float inv_rms = (PROD == PROD_RMSNORM) ? rms_inv(p.x, p.K, p.eps, part, LR_CT) : 0.f;
  const int nt = p.K >> 3;
  for (int t0 = 0; t0 < nt; t0 += LR_CT * LR_XT) {
    float v[LR_XT][8];
#pragma unroll
    for (int i = 0; i < LR_XT; ++i) {
      const int t = t0 + threadIdx.x + i * LR_CT;
      if (t < nt) {
        const float4 a = produce4<PROD>(p.x, p.aux, 8 * t, inv_rms);
        const float4 c = produce4<PROD>(p.x, p.aux, 8 * t + 4, inv_rms);
        v[i][0] = a.x; v[i][1] = a.y; v[i][2] = a.z; v[i][3] = a.w;
        v[i][4] = c.x; v[i][5] = c.y; v[i][6] = c.z; v[i][7] = c.w;
      }
    }
#pragma unroll
    for (int i = 0; i < LR_XT; ++i) {
      const int t = t0 + threadIdx.x + i * LR_CT;
      if (t < nt) {
        const Q8Oct r = quantize_oct(v[i]);
        *reinterpret_cast<uint2*>(xq + 8 * t) = make_uint2(r.q[0], r.q[1]);
        if ((lane & 3) == 0) xs[t >> 2] = make_float2(r.dh, __fmul_rn(r.dh, static_cast<float>(r.sumq)));  // exact
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(LR_CT) : "memory");
  // Staged form: the next call's weights are asked of L2 only now, once x is in:
  // issued at the CTA's start, that stream delayed the loads of x behind the
  // dependency wait (6.6 against 6.1 us per decode launch). Eight warps issue
  // an eighth each.
  if (!RING && lane == 0 && warp < 8) prefetch_slice_l2(p.pf, p.pf_bytes, warp, 8);

  const float4* xs4 = reinterpret_cast<const float4*>(xs);
  const int pitch = p.cb * BB;
  const int items = p.n_chunks * per_chunk;
  int ready = -1, sl = 0;  // last chunk this warp has seen land, and its slot
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // this warp's sums for row groups 0..3
  for (int i = warp; i < items; i += NW) {
    // i = (c * n_groups + g) * cb + j; quotients by multiply-high (exact in range)
    const int c = static_cast<int>(__umulhi(static_cast<uint32_t>(i), p.inv_per_chunk));
    const int rem = i - c * per_chunk;
    const int g = static_cast<int>(__umulhi(static_cast<uint32_t>(rem), p.inv_cb));
    const int j = rem - g * p.cb;
    const int b = c * p.cb + j;
    if (!RING) {
      if (b >= p.nb) continue;  // zero-filled tail of the last chunk
      if (c != ready) {
        if (!mbar_wait(&full[c], 0, abort, p.err)) break;
        ready = c;
      }
      sl = c;
    } else {
      if (c != ready) {
        sl = c % p.S;
        // chunk c issued first: the parity wait cannot take an older fill of the slot
        if (!wait_counter_above(chunks_issued, c, abort, p.err) || !mbar_wait(&full[sl], (c / p.S) & 1, abort, p.err))
          break;
        ready = c;
      }
      if (b >= p.nb) {  // zero-filled tail of the last chunk: release it all the same
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sl]);
        continue;
      }
    }
    const int row = 32 * g + lane;
    const int srow = min(row, p.R - 1);  // lanes past the last row repeat it; their result is dropped
    const uint8_t* blk = smem + static_cast<size_t>(sl) * p.chunk_bytes + srow * pitch + j * BB;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
    // 6-bit scales and mins, one per byte: sub-blocks 0..3 and 4..7
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    const int8_t* xb = xq + (b << 8);
    float lo = 0.f, mn = 0.f;
    uint4 ha, hb;  // Q5_K: qh[0..15], qh[16..31]
    if (WT == KQ_Q5_K) {
      ha = *reinterpret_cast<const uint4*>(blk + 16);
      hb = *reinterpret_cast<const uint4*>(blk + 32);
    }
    constexpr int QS = (WT == KQ_Q5_K) ? 48 : 16;  // byte offset of the nibbles
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // bytes 32q .. 32q+31 of the nibbles: low nibbles are sub-block 2q, high nibbles 2q+1
      const uint4 qa = *reinterpret_cast<const uint4*>(blk + QS + 32 * q);
      const uint4 qb = *reinterpret_cast<const uint4*>(blk + QS + 16 + 32 * q);
      const int4 x0 = *reinterpret_cast<const int4*>(xb + 64 * q);
      const int4 x1 = *reinterpret_cast<const int4*>(xb + 64 * q + 16);
      const int4 x2 = *reinterpret_cast<const int4*>(xb + 64 * q + 32);
      const int4 x3 = *reinterpret_cast<const int4*>(xb + 64 * q + 48);
      const float4 ds = xs4[(b << 2) + q];  // {d8, s} of sub-blocks 2q and 2q+1
      const uint32_t scw = (q < 2) ? sc_lo : sc_hi;
      const uint32_t mw = (q < 2) ? m_lo : m_hi;
      const int sh = (q & 1) * 16;
      const int scA = (scw >> sh) & 0xFF, scB = (scw >> (sh + 8)) & 0xFF;
      const int mA = (mw >> sh) & 0xFF, mB = (mw >> (sh + 8)) & 0xFF;
      if (WT == KQ_Q5_K) {
        int dA, dB;
        if (q == 0) q5_chunk_dots<0>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
        else if (q == 1) q5_chunk_dots<2>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
        else if (q == 2) q5_chunk_dots<4>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
        else q5_chunk_dots<6>(qa, qb, ha, hb, x0, x1, x2, x3, dA, dB);
        lo = fmaf(ds.x, i2f(scA * dA), lo);
        lo = fmaf(ds.z, i2f(scB * dB), lo);
        mn = fmaf(ds.y, i2f(mA), mn);
        mn = fmaf(ds.w, i2f(mB), mn);
        continue;
      }
      // high nibbles are taken in place (w & 0xF0F0F0F0 = 16 * nibble): the sums
      // h0, h1 are exact multiples of 16
      int a0 = __dp4a(static_cast<int>(qa.x & 0x0F0F0F0Fu), x0.x, 0);
      int a1 = __dp4a(static_cast<int>(qb.x & 0x0F0F0F0Fu), x1.x, 0);
      int h0 = dp4a_us(qa.x & 0xF0F0F0F0u, x2.x, 0);
      int h1 = dp4a_us(qb.x & 0xF0F0F0F0u, x3.x, 0);
      a0 = __dp4a(static_cast<int>(qa.y & 0x0F0F0F0Fu), x0.y, a0);
      a1 = __dp4a(static_cast<int>(qb.y & 0x0F0F0F0Fu), x1.y, a1);
      h0 = dp4a_us(qa.y & 0xF0F0F0F0u, x2.y, h0);
      h1 = dp4a_us(qb.y & 0xF0F0F0F0u, x3.y, h1);
      a0 = __dp4a(static_cast<int>(qa.z & 0x0F0F0F0Fu), x0.z, a0);
      a1 = __dp4a(static_cast<int>(qb.z & 0x0F0F0F0Fu), x1.z, a1);
      h0 = dp4a_us(qa.z & 0xF0F0F0F0u, x2.z, h0);
      h1 = dp4a_us(qb.z & 0xF0F0F0F0u, x3.z, h1);
      a0 = __dp4a(static_cast<int>(qa.w & 0x0F0F0F0Fu), x0.w, a0);
      a1 = __dp4a(static_cast<int>(qb.w & 0x0F0F0F0Fu), x1.w, a1);
      h0 = dp4a_us(qa.w & 0xF0F0F0F0u, x2.w, h0);
      h1 = dp4a_us(qb.w & 0xF0F0F0F0u, x3.w, h1);
      lo = fmaf(ds.x, i2f(scA * (a0 + a1)), lo);
      lo = fmaf(ds.z, i2f(scB * ((h0 + h1) >> 4)), lo);
      mn = fmaf(ds.y, i2f(mA), mn);
      mn = fmaf(ds.w, i2f(mB), mn);
    }
    const float v = fmaf(-dmin, mn, d * lo);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] += (g == k) ? v : 0.f;
    if (RING) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sl]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (k < p.n_groups) part[(warp * p.n_groups + k) * 32 + lane] = acc[k];
  asm volatile("bar.sync 1, %0;" ::"r"(LR_CT) : "memory");
  // y[row] = Sum over the warps, in warp order
  for (int r = threadIdx.x; r < rows; r += LR_CT) {
    const float* pr = part + (r >> 5) * 32 + (r & 31);
    float a = pr[0];
#pragma unroll 8
    for (int w = 1; w < NW; ++w) a += pr[w * p.n_groups * 32];
    p.y[r0 + r] = a;
  }
}

// ---------------------------------------------------------------------------
// The lane-row kernel for a few tokens (the small-N decode: 2 .. LR_TOKENS_MAX
// tokens, e.g. several sequences or speculative tokens at once). Same staging
// and arithmetic as the kernel above (staged form only); y is [n_tok][M]. The
// tokens' Q8_1 codes and {d8, s} pairs are made once per call by
// quantize_split_kernel (below) in exactly the shared-memory layout, and a pass
// pulls up to NT tokens of them with two bulk copies. Warp w takes every 16th
// work item of the CTA, unpacks the item's codes
// once and multiplies them with every token of the pass, keeping one set of
// row-group sums per token. The weights are read from HBM once whatever the
// number of tokens; later passes reuse them.
// ---------------------------------------------------------------------------
template <int NT, int WT = KQ_Q4_K>
__global__ void __launch_bounds__((LR_NW_TOK + 1) * 32, 1)
    matvec_q4k_lanerow_tokens_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT,
                                     const MatvecLaneRowParams p) {
  static_assert(WT == KQ_Q4_K || WT == KQ_Q5_K, "Q4_K or Q5_K super-blocks");
  constexpr int BB = (WT == KQ_Q5_K) ? Q5K_BYTES : Q4K_BYTES;  // bytes per super-block
  constexpr int QS = (WT == KQ_Q5_K) ? 48 : 16;                // byte offset of the nibbles
  constexpr int NW = LR_NW_TOK;
  static_assert(NT >= 1 && NT <= 4, "tokens per pass");
  constexpr int LR_CT = NW * 32;
  extern __shared__ __align__(1024) uint8_t smem[];
  int8_t* xq = reinterpret_cast<int8_t*>(smem + p.xq_off);           // [NT][xq_tok]
  uint8_t* xsb = smem + p.xs_off;                                     // [NT][xs_tok]: per 32-block {d8, d8 * Sum q}
  float* part = reinterpret_cast<float*>(smem + p.part_off);         // [warp][row group][lane]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);    // one per chunk
  uint64_t* x_full = full + p.S;                                     // the activations of a pass
  volatile int* abort = reinterpret_cast<volatile int*>(x_full + 1);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * p.R;
  const int rows = min(p.R, p.M - r0);
  const int per_chunk = p.n_groups * p.cb;  // work items per chunk
  if (threadIdx.x == 0) {
    for (int c = 0; c < p.n_chunks; ++c) mbar_init(&full[c], 1);
    mbar_init(x_full, 1);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmT);
      // The last chunk comes through tmT, whose box holds only its tail_cb
      // super-blocks (its slot is sized for them).
      for (int c = 0; c < p.n_chunks; ++c) {
        const bool last = c == p.n_chunks - 1;
        mbar_expect_tx(&full[c], static_cast<uint32_t>(p.R * (last ? p.tail_cb : p.cb) * BB));
        tma_load_2d(smem + static_cast<size_t>(c) * p.chunk_bytes, last ? &tmT : &tmW, &full[c], c * p.cb * (BB / 4),
                    r0);
      }
      // Every copy lands before the CTA may exit (also when the consumers gave up).
      for (int c = 0; c < p.n_chunks; ++c)
        if (!mbar_wait_bounded(&full[c], 0)) report_error(p.err, ERR_WAIT_TIMEOUT);
    }
    return;
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel

  const int pitch = p.cb * BB;  // row stride of a chunk; the last chunk's is tail_cb * BB
  const int items = p.n_chunks * per_chunk;
  for (int t0 = 0, pass = 0; t0 < p.n_tok; t0 += NT, ++pass) {
    const int tn = min(NT, p.n_tok - t0);  // tokens of this pass
    if (t0 > 0) asm volatile("bar.sync 1, %0;" ::"r"(LR_CT) : "memory");  // the last pass's reads are done
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();  // those reads come before the copies' writes
      mbar_expect_tx(x_full, static_cast<uint32_t>(tn * (p.xq_tok + p.xs_tok)));
      bulk_g2s(xq, p.xq_g + static_cast<size_t>(t0) * p.xq_tok, static_cast<uint32_t>(tn * p.xq_tok), x_full);
      bulk_g2s(xsb, p.xs_g + static_cast<size_t>(t0) * p.xs_tok, static_cast<uint32_t>(tn * p.xs_tok), x_full);
    }
    if (!mbar_wait(x_full, pass & 1, abort, p.err)) break;

    // Warp w takes every NW-th work item and multiplies the item's codes with
    // each token of the pass: a block's nibbles (and Q5_K high bits) are
    // unpacked once per pass, then each token costs its activation loads, 16
    // dp4a per 64 weights and the scale arithmetic.
    int ready = -1;  // last chunk this warp has seen land (later passes: at once)
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[t][k] = 0.f;
    for (int i = warp; i < items; i += NW) {
      const int c = static_cast<int>(__umulhi(static_cast<uint32_t>(i), p.inv_per_chunk));
      const int rem = i - c * per_chunk;
      const int g = static_cast<int>(__umulhi(static_cast<uint32_t>(rem), p.inv_cb));
      const int j = rem - g * p.cb;
      const int b = c * p.cb + j;
      if (b >= p.nb) continue;  // zero-filled tail of the last chunk
      if (c != ready) {
        if (!mbar_wait(&full[c], 0, abort, p.err)) break;
        ready = c;
      }
      const int srow = min(32 * g + lane, p.R - 1);  // lanes past the last row repeat it; dropped
      const int rp = (c == p.n_chunks - 1) ? p.tail_cb * BB : pitch;
      const uint8_t* blk = smem + static_cast<size_t>(c) * p.chunk_bytes + srow * rp + j * BB;
      const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
      const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
      const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
      const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
      const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
      const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
      float lo[NT], mn[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) lo[t] = mn[t] = 0.f;
      uint4 ha, hb;  // Q5_K: qh[0..15], qh[16..31]
      if (WT == KQ_Q5_K) {
        ha = *reinterpret_cast<const uint4*>(blk + 16);
        hb = *reinterpret_cast<const uint4*>(blk + 32);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 qa = *reinterpret_cast<const uint4*>(blk + QS + 32 * q);
        const uint4 qb = *reinterpret_cast<const uint4*>(blk + QS + 16 + 32 * q);
        const uint32_t scw = (q < 2) ? sc_lo : sc_hi;
        const uint32_t mw = (q < 2) ? m_lo : m_hi;
        const int sh = (q & 1) * 16;
        const int scA = (scw >> sh) & 0xFF, scB = (scw >> (sh + 8)) & 0xFF;
        const int mA = (mw >> sh) & 0xFF, mB = (mw >> (sh + 8)) & 0xFF;
        // codes of sub-block 2q (cl, against x[64q .. 64q+31]) and 2q+1 (ch,
        // against x[64q+32 .. 64q+63]); Q4_K keeps the high nibbles in place
        // (their dots are 16x the code dots)
        uint32_t cl[8], ch[8];
        if (WT == KQ_Q5_K) {
          const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
          const uint32_t h[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (q == 0) { cl[e] = q5_codes<true, 0>(w[e], h[e]); ch[e] = q5_codes<false, 1>(w[e], h[e]); }
            else if (q == 1) { cl[e] = q5_codes<true, 2>(w[e], h[e]); ch[e] = q5_codes<false, 3>(w[e], h[e]); }
            else if (q == 2) { cl[e] = q5_codes<true, 4>(w[e], h[e]); ch[e] = q5_codes<false, 5>(w[e], h[e]); }
            else { cl[e] = q5_codes<true, 6>(w[e], h[e]); ch[e] = q5_codes<false, 7>(w[e], h[e]); }
          }
        } else {
          const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            cl[e] = w[e] & 0x0F0F0F0Fu;
            ch[e] = w[e] & 0xF0F0F0F0u;
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t >= tn) break;
          const int8_t* xb = xq + t * p.xq_tok + (b << 8) + 64 * q;
          const int4 x0 = *reinterpret_cast<const int4*>(xb);
          const int4 x1 = *reinterpret_cast<const int4*>(xb + 16);
          const int4 x2 = *reinterpret_cast<const int4*>(xb + 32);
          const int4 x3 = *reinterpret_cast<const int4*>(xb + 48);
          const float4 ds = reinterpret_cast<const float4*>(xsb + t * p.xs_tok)[(b << 2) + q];  // {d8, s} of 2q, 2q+1
          int dA, dB;
          if (WT == KQ_Q5_K) {
            dA = __dp4a(static_cast<int>(cl[0]), x0.x, 0);
            dA = __dp4a(static_cast<int>(cl[1]), x0.y, dA);
            dA = __dp4a(static_cast<int>(cl[2]), x0.z, dA);
            dA = __dp4a(static_cast<int>(cl[3]), x0.w, dA);
            dA = __dp4a(static_cast<int>(cl[4]), x1.x, dA);
            dA = __dp4a(static_cast<int>(cl[5]), x1.y, dA);
            dA = __dp4a(static_cast<int>(cl[6]), x1.z, dA);
            dA = __dp4a(static_cast<int>(cl[7]), x1.w, dA);
            dB = __dp4a(static_cast<int>(ch[0]), x2.x, 0);
            dB = __dp4a(static_cast<int>(ch[1]), x2.y, dB);
            dB = __dp4a(static_cast<int>(ch[2]), x2.z, dB);
            dB = __dp4a(static_cast<int>(ch[3]), x2.w, dB);
            dB = __dp4a(static_cast<int>(ch[4]), x3.x, dB);
            dB = __dp4a(static_cast<int>(ch[5]), x3.y, dB);
            dB = __dp4a(static_cast<int>(ch[6]), x3.z, dB);
            dB = __dp4a(static_cast<int>(ch[7]), x3.w, dB);
          } else {
            int a0 = __dp4a(static_cast<int>(cl[0]), x0.x, 0);
            int a1 = __dp4a(static_cast<int>(cl[4]), x1.x, 0);
            int h0 = dp4a_us(ch[0], x2.x, 0);
            int h1 = dp4a_us(ch[4], x3.x, 0);
            a0 = __dp4a(static_cast<int>(cl[1]), x0.y, a0);
            a1 = __dp4a(static_cast<int>(cl[5]), x1.y, a1);
            h0 = dp4a_us(ch[1], x2.y, h0);
            h1 = dp4a_us(ch[5], x3.y, h1);
            a0 = __dp4a(static_cast<int>(cl[2]), x0.z, a0);
            a1 = __dp4a(static_cast<int>(cl[6]), x1.z, a1);
            h0 = dp4a_us(ch[2], x2.z, h0);
            h1 = dp4a_us(ch[6], x3.z, h1);
            a0 = __dp4a(static_cast<int>(cl[3]), x0.w, a0);
            a1 = __dp4a(static_cast<int>(cl[7]), x1.w, a1);
            h0 = dp4a_us(ch[3], x2.w, h0);
            h1 = dp4a_us(ch[7], x3.w, h1);
            dA = a0 + a1;
            dB = (h0 + h1) >> 4;
          }
          lo[t] = fmaf(ds.x, i2f(scA * dA), lo[t]);
          lo[t] = fmaf(ds.z, i2f(scB * dB), lo[t]);
          mn[t] = fmaf(ds.y, i2f(mA), mn[t]);
          mn[t] = fmaf(ds.w, i2f(mB), mn[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = fmaf(-dmin, mn[t], d * lo[t]);
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[t][k] += (g == k) ? v : 0.f;
      }
    }
    // part: [token][warp][row group][lane]
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (t < tn && k < p.n_groups) part[((t * NW + warp) * p.n_groups + k) * 32 + lane] = acc[t][k];
    asm volatile("bar.sync 1, %0;" ::"r"(LR_CT) : "memory");
    // y[token][row] = Sum over the warps, in warp order
    for (int u = threadIdx.x; u < tn * rows; u += LR_CT) {
      const int t = u / rows, r = u - t * rows;
      const float* pr = part + t * NW * p.n_groups * 32 + (r >> 5) * 32 + (r & 31);
      float a = pr[0];
      for (int w = 1; w < NW; ++w) a += pr[w * p.n_groups * 32];
      p.y[static_cast<int64_t>(t0 + t) * p.M + r0 + r] = a;
    }
  }
}

static inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Launch plan of the lane-row kernel with nw consumer warps and room for the
// activations of nt tokens in at most `budget` bytes of shared memory; `ring`
// allows fewer chunk slots than chunks (at least two). False when the rows do
// not fit (then the item kernel above runs).
static bool plan_lanerow(int64_t M, int64_t K, int num_sms, int nw, int nt, int budget, bool ring,
                         MatvecLaneRowParams* p, int* grid, size_t* smem, int bb = Q4K_BYTES, bool trim_tail = false) {
  if (K > (int64_t(1) << 20)) return false;
  p->M = static_cast<int>(M);
  p->K = static_cast<int>(K);
  p->nb = static_cast<int>(K / QK_K);
  const int64_t G0 = std::min<int64_t>(M, num_sms);
  const int64_t R = (M + G0 - 1) / G0;
  if (R > LR_MAX_ROWS) return false;
  p->R = static_cast<int>(R);
  *grid = static_cast<int>((M + R - 1) / R);
  p->n_groups = (p->R + 31) / 32;
  const int part_bytes = nt * nw * p->n_groups * 32 * 4;  // per token: [warp][row group][lane]
  p->xq_tok = round_up(p->K, 128);                      // activation codes of a token
  p->xs_tok = round_up((p->K / 32) * 8, 128);           // {d8, d8 * Sum q} per 32-block
  const int fixed = nt * (p->xq_tok + p->xs_tok) + part_bytes;  // + per-warp partials
  // Widest odd chunk that fits (the TMA box row, cb * bb bytes, is at most 256
  // words: cb <= 7 for Q4_K, 5 for Q5_K). cb >= 3 keeps both divisors of the item
  // index (cb and n_groups * cb) at least 3, so their reciprocals fit in 32 bits.
  for (int cb = (bb == Q5K_BYTES ? 5 : 7); cb >= 3; cb -= 2) {
    const int n_chunks = (p->nb + cb - 1) / cb;
    const int chunk_bytes = round_up(p->R * cb * bb, 128);
    // trim_tail (staged form): the last chunk's slot holds only its own
    // super-blocks, loaded through a second tensor map with a narrower box
    const int tail_cb = trim_tail ? p->nb - (n_chunks - 1) * cb : cb;
    const int trim = trim_tail ? chunk_bytes - round_up(p->R * tail_cb * bb, 128) : 0;
    int S = n_chunks;
    auto total = [&](int slots) {
      return static_cast<size_t>(slots) * chunk_bytes - trim + fixed + slots * 16 + 16;
    };
    while (ring && S > 2 && total(S) > static_cast<size_t>(budget)) --S;
    if (total(S) > static_cast<size_t>(budget)) continue;
    // i / d == umulhi(i, ceil(2^32 / d)) holds while i * d < 2^32
    if (static_cast<int64_t>(n_chunks) * p->n_groups * cb * p->n_groups * cb >= (int64_t(1) << 32)) return false;
    p->cb = cb;
    p->tail_cb = tail_cb;
    p->n_chunks = n_chunks;
    p->chunk_bytes = chunk_bytes;
    p->S = S;
    p->inv_per_chunk = static_cast<uint32_t>(((uint64_t(1) << 32) + p->n_groups * cb - 1) / (p->n_groups * cb));
    p->inv_cb = static_cast<uint32_t>(((uint64_t(1) << 32) + cb - 1) / cb);
    size_t off = static_cast<size_t>(S) * chunk_bytes - trim;
    p->xq_off = static_cast<int>(off);
    off += static_cast<size_t>(nt) * p->xq_tok;
    p->xs_off = static_cast<int>(off);
    off += static_cast<size_t>(nt) * p->xs_tok;
    p->part_off = static_cast<int>(off);
    off += part_bytes;
    p->bar_off = static_cast<int>(off);
    *smem = total(S);
    return true;
  }
  return false;
}

// Shared-memory attribute slot of a kernel instantiation (allow_max_smem).
constexpr int smem_slot(int base_x, int base_prod, int prod) { return prod == PROD_X ? base_x : base_prod + prod - 1; }

// Shared-memory attribute slots of the lane-row instantiations: full, ring.
constexpr int lanerow_slot(int wt, bool ring, int prod) {
  return wt == KQ_Q5_K ? smem_slot(ring ? 29 : 26, ring ? 30 : 27, prod) : smem_slot(ring ? 10 : 9, ring ? 18 : 16, prod);
}

template <int WT, int PROD>
static cudaError_t launch_lanerow(bool ring, const CUtensorMap& tmW, const MatvecLaneRowParams& lp, int grid,
                                  size_t smem, cudaStream_t s) {
  if (ring) {
    cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(matvec_q4k_lanerow_kernel<LR_NW_RING, true, PROD, WT>),
                                   lanerow_slot(WT, true, PROD));
    if (e != cudaSuccess) return e;
    return launch_pdl(matvec_q4k_lanerow_kernel<LR_NW_RING, true, PROD, WT>, dim3(grid), dim3((LR_NW_RING + 1) * 32),
                      smem, s, tmW, lp);
  }
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(matvec_q4k_lanerow_kernel<LR_NW_FULL, false, PROD, WT>),
                                 lanerow_slot(WT, false, PROD));
  if (e != cudaSuccess) return e;
  return launch_pdl(matvec_q4k_lanerow_kernel<LR_NW_FULL, false, PROD, WT>, dim3(grid), dim3((LR_NW_FULL + 1) * 32),
                    smem, s, tmW, lp);
}

template <int PROD>
static cudaError_t launch_matvec_p(int wtype, const void* W, const float* x, const float* aux, float eps, float* y,
                                   int64_t M, int64_t K, const void* pf, uint64_t pf_bytes, int* err, int num_sms,
                                   cudaStream_t s, int* status) {
  *status = KQ_OK;
  // Q4_K and Q5_K: the lane-row kernel with all rows staged at once when they
  // fit (measured faster at the decode sizes: the ring's refills wait for the
  // activations and then for HBM), else its ring form.
  if (wtype == KQ_Q4_K || wtype == KQ_Q5_K) {
    const int bb = wtype == KQ_Q5_K ? Q5K_BYTES : Q4K_BYTES;
    MatvecLaneRowParams lp{};
    size_t smem = 0;
    int grid = 0;
    const bool full = plan_lanerow(M, K, num_sms, LR_NW_FULL, 1, MV_SMEM_LIMIT, false, &lp, &grid, &smem, bb);
    const bool ring = !full && plan_lanerow(M, K, num_sms, LR_NW_RING, 1, LR_RING_SMEM, true, &lp, &grid, &smem, bb);
    if (full || ring) {
      CUtensorMap tmW;
      const uint64_t rs = static_cast<uint64_t>(lp.nb) * bb;
      if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rs / 4, static_cast<uint64_t>(M), rs,
                          static_cast<uint32_t>(lp.cb * bb / 4), static_cast<uint32_t>(lp.R),
                          CU_TENSOR_MAP_SWIZZLE_NONE)) {
        *status = KQ_ERR_CUDA;
        return cudaSuccess;
      }
      lp.x = x;
      lp.aux = aux;
      lp.eps = eps;
      lp.y = y;
      lp.n_tok = 1;
      lp.pf = static_cast<const uint8_t*>(pf);
      lp.pf_bytes = pf_bytes;
      lp.err = err;
      lp.hold = test_hold_copies();
      if (wtype == KQ_Q5_K) return launch_lanerow<KQ_Q5_K, PROD>(ring, tmW, lp, grid, smem, s);
      return launch_lanerow<KQ_Q4_K, PROD>(ring, tmW, lp, grid, smem, s);
    }
  }
  MatvecParams p{};
  p.W = static_cast<const uint8_t*>(W);
  p.x = x;
  p.aux = aux;
  p.eps = eps;
  p.y = y;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.nb = static_cast<int>(K / QK_K);
  p.bb = wtype == KQ_Q4_K ? Q4K_BYTES : wtype == KQ_Q5_K ? Q5K_BYTES : Q6K_BYTES;
  p.rs = p.nb * p.bb;
  p.w_bytes = static_cast<int64_t>(M) * p.rs;
  p.chunk_blocks = wtype == KQ_Q4_K   ? MV_CHUNK_BLOCKS_Q4K
                   : wtype == KQ_Q5_K ? MV_CHUNK_BLOCKS_Q5K
                   : K < MV_Q6K_LONG_K ? MV_CHUNK_BLOCKS_Q6K_SHORT_K
                                       : MV_CHUNK_BLOCKS_Q6K;
  p.chunk_bytes = p.chunk_blocks * p.bb;
  // room for a copy that starts up to 15 bytes before a CTA's first row
  p.slot_bytes = round_up(p.chunk_bytes + (p.rs % 16 ? 16 : 0), 128);
  p.rows_per_group = MV_PART_MAX / p.nb;
  p.xq_bytes = round_up(p.K, 128);
  p.xds_bytes = round_up((p.K / QK_K) * 8 * 16, 128);
  p.pf = static_cast<const uint8_t*>(pf);
  p.pf_bytes = pf_bytes;
  p.err = err;
  p.hold = test_hold_copies();
  if (p.rows_per_group < 1) {
    *status = KQ_ERR_SHAPE;
    return cudaSuccess;
  }
  const int fixed = p.xq_bytes + p.xds_bytes + MV_PART_MAX * 4 + 1024;
  int n_ring = (MV_SMEM_LIMIT - fixed) / (p.slot_bytes + 16);
  if (n_ring > MV_MAX_RING) n_ring = MV_MAX_RING;
  if (n_ring < 2) {
    *status = KQ_ERR_SHAPE;
    return cudaSuccess;
  }
  const int G = M < num_sms ? static_cast<int>(M) : num_sms;
  // a ring deeper than the largest CTA range buys nothing
  const int64_t max_rows = (M + G - 1) / G;
  const int64_t need = (max_rows * p.nb + p.chunk_blocks - 1) / p.chunk_blocks;
  if (n_ring > need) n_ring = static_cast<int>(need < 1 ? 1 : need);
  p.n_ring = n_ring;
  const size_t smem = static_cast<size_t>(p.xq_bytes + p.xds_bytes + MV_PART_MAX * 4) +
                      static_cast<size_t>(n_ring) * p.slot_bytes + 2 * n_ring * sizeof(uint64_t) + 16;  // + abort, issued
  cudaError_t e;
  if (wtype == KQ_Q4_K) {
    e = allow_max_smem(reinterpret_cast<const void*>(matvec_kernel<KQ_Q4_K, PROD>), smem_slot(0, 20, PROD));
    if (e != cudaSuccess) return e;
    e = launch_pdl(matvec_kernel<KQ_Q4_K, PROD>, dim3(G), dim3(MV_THREADS), smem, s, p);
  } else if (wtype == KQ_Q5_K) {
    e = allow_max_smem(reinterpret_cast<const void*>(matvec_kernel<KQ_Q5_K, PROD>), smem_slot(32, 33, PROD));
    if (e != cudaSuccess) return e;
    e = launch_pdl(matvec_kernel<KQ_Q5_K, PROD>, dim3(G), dim3(MV_THREADS), smem, s, p);
  } else {
    e = allow_max_smem(reinterpret_cast<const void*>(matvec_kernel<KQ_Q6_K, PROD>), smem_slot(1, 22, PROD));
    if (e != cudaSuccess) return e;
    e = launch_pdl(matvec_kernel<KQ_Q6_K, PROD>, dim3(G), dim3(MV_THREADS), smem, s, p);
  }
  return e;
}

cudaError_t launch_matvec(int wtype, const void* W, const float* x, const float* aux, float eps, int prod, float* y,
                          int64_t M, int64_t K, const void* pf, uint64_t pf_bytes, int* err, int num_sms, cudaStream_t s,
                          int* status) {
  switch (prod) {
    case PROD_SWIGLU:
      return launch_matvec_p<PROD_SWIGLU>(wtype, W, x, aux, eps, y, M, K, pf, pf_bytes, err, num_sms, s, status);
    case PROD_RMSNORM:
      return launch_matvec_p<PROD_RMSNORM>(wtype, W, x, aux, eps, y, M, K, pf, pf_bytes, err, num_sms, s, status);
    default:
      return launch_matvec_p<PROD_X>(wtype, W, x, aux, eps, y, M, K, pf, pf_bytes, err, num_sms, s, status);
  }
}

// Q8_1 of n_tok tokens in the layout the several-token kernel copies into
// shared memory: codes [n_tok][xq_tok] (x's order) and per 32-block
// {d8, d8 * Sum q} [n_tok][xs_tok]; the arithmetic of the one-token kernel's own
// quantiser (quantize_oct), so the codes are the same. Task t quantises eight
// values of token t / (K / 8); a warp's 32 tasks share one token.
__global__ void __launch_bounds__(256) quantize_split_kernel(const float* __restrict__ X, int n_tok, int K, int xq_tok,
                                                             int xs_tok, uint8_t* __restrict__ xq_g,
                                                             uint8_t* __restrict__ xs_g) {
  pdl_enter();
  const int nt = K >> 3;
  const int64_t total = static_cast<int64_t>(n_tok) * nt;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * 256) {
    const int tok = static_cast<int>(t / nt), tl = static_cast<int>(t - static_cast<int64_t>(tok) * nt);
    const float4* src = reinterpret_cast<const float4*>(X + static_cast<int64_t>(tok) * K) + 2 * tl;
    const float4 a = __ldg(src), c = __ldg(src + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    const Q8Oct r = quantize_oct(v);
    *reinterpret_cast<uint2*>(xq_g + static_cast<int64_t>(tok) * xq_tok + 8 * tl) = make_uint2(r.q[0], r.q[1]);
    if ((threadIdx.x & 3) == 0)
      reinterpret_cast<float2*>(xs_g + static_cast<int64_t>(tok) * xs_tok)[tl >> 2] =
          make_float2(r.dh, __fmul_rn(r.dh, static_cast<float>(r.sumq)));  // exact
  }
}

// Q4_K and Q5_K for N = 2 .. LR_TOKENS_MAX tokens: the staged lane-row kernel
// with LR_NT (else two) tokens per pass. *handled = false (nothing queued) when
// the rows do not fit staged next to the activations of two tokens.
template <int NT, int WT>
static cudaError_t launch_tokens_kernel(const CUtensorMap& tmW, const CUtensorMap& tmT, const MatvecLaneRowParams& lp,
                                        int grid, size_t smem, cudaStream_t s) {
  const int slot = WT == KQ_Q5_K ? (NT == LR_NT ? 35 : 36) : (NT == LR_NT ? 11 : 14);
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(matvec_q4k_lanerow_tokens_kernel<NT, WT>), slot);
  if (e != cudaSuccess) return e;
  return launch_pdl(matvec_q4k_lanerow_tokens_kernel<NT, WT>, dim3(grid), dim3((LR_NW_TOK + 1) * 32), smem, s, tmW,
                    tmT, lp);
}

cudaError_t launch_matvec_tokens(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K, int64_t N,
                                 void* scratch, size_t scratch_bytes, int* err, int num_sms, cudaStream_t s,
                                 bool* handled) {
  *handled = false;
  if (N < 2 || N > LR_TOKENS_MAX || (wtype != KQ_Q4_K && wtype != KQ_Q5_K)) return cudaSuccess;
  const int bb = wtype == KQ_Q5_K ? Q5K_BYTES : Q4K_BYTES;
  MatvecLaneRowParams lp{};
  size_t smem = 0;
  int grid = 0;
  int nt = LR_NT;
  if (!plan_lanerow(M, K, num_sms, LR_NW_TOK, nt, MV_SMEM_LIMIT, false, &lp, &grid, &smem, bb, true)) {
    nt = 2;
    if (!plan_lanerow(M, K, num_sms, LR_NW_TOK, nt, MV_SMEM_LIMIT, false, &lp, &grid, &smem, bb, true))
      return cudaSuccess;
  }
  CUtensorMap tmW, tmT;  // chunks of cb super-blocks; the last chunk's tail_cb
  const uint64_t rs = static_cast<uint64_t>(lp.nb) * bb;
  if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rs / 4, static_cast<uint64_t>(M), rs,
                      static_cast<uint32_t>(lp.cb * bb / 4), static_cast<uint32_t>(lp.R), CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap_2d(&tmT, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rs / 4, static_cast<uint64_t>(M), rs,
                      static_cast<uint32_t>(lp.tail_cb * bb / 4), static_cast<uint32_t>(lp.R),
                      CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaSuccess;
  const size_t xq_bytes = static_cast<size_t>(N) * lp.xq_tok, xs_bytes = static_cast<size_t>(N) * lp.xs_tok;
  if (xq_bytes + xs_bytes > scratch_bytes) return cudaSuccess;
  uint8_t* xq_g = static_cast<uint8_t*>(scratch);
  uint8_t* xs_g = xq_g + xq_bytes;  // xq_tok is a multiple of 128: 16-byte aligned
  lp.x = X;
  lp.y = Y;
  lp.n_tok = static_cast<int>(N);
  lp.xq_g = xq_g;
  lp.xs_g = xs_g;
  lp.err = err;
  smem += 16;  // the activations' barrier
  *handled = true;
  {
    const int64_t tasks = N * (K / 8);
    const int64_t blocks = std::min<int64_t>((tasks + 255) / 256, static_cast<int64_t>(num_sms) * 4);
    cudaError_t e = launch_pdl(quantize_split_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, X,
                               static_cast<int>(N), static_cast<int>(K), lp.xq_tok, lp.xs_tok, xq_g, xs_g);
    if (e != cudaSuccess) return e;
  }
  if (wtype == KQ_Q5_K)
    return nt == LR_NT ? launch_tokens_kernel<LR_NT, KQ_Q5_K>(tmW, tmT, lp, grid, smem, s)
                       : launch_tokens_kernel<2, KQ_Q5_K>(tmW, tmT, lp, grid, smem, s);
  return nt == LR_NT ? launch_tokens_kernel<LR_NT, KQ_Q4_K>(tmW, tmT, lp, grid, smem, s)
                     : launch_tokens_kernel<2, KQ_Q4_K>(tmW, tmT, lp, grid, smem, s);
}
}  // namespace kq
