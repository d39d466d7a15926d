// TQ4_1S decode matvec y = W . x ("TQ4_1S Weight Kernel Optimization":
// Architecture Overview, Block Layout, Centroid Table).
//
// A TQ4_1S block holds 32 weights in the Walsh-Hadamard-rotated space: two fp16
// half-block scales (d0 for elements 0..15, d1 for 16..31) and a 4-bit index
// per element into a 16-entry Lloyd-Max centroid table (20 bytes). The weights
// are w_b = H^-1 r_b with r_b[j] = centroid[idx_j] * d_half(j) and H the
// orthonormal 32-point Walsh-Hadamard transform in natural order (symmetric,
// its own inverse). Since H is orthogonal, w_b . x_b = r_b . (H x_b): the
// kernels rotate each 32-block of the activation once (forward WHT, fp32
// butterflies) and then dot the stored rotated weights against it, so no
// weight is ever transformed back. Arithmetic is fp32 throughout: the centroid
// table is fp32 (exactly the printed values rounded to fp32), the activation
// stays fp32 (no int8 codes, which the WHT would amplify), products and sums are
// fp32, and the orthonormal 1/sqrt(32) is applied once per output.
//
// Hot kernel (tq4_lanerow_kernel): a CTA owns R consecutive rows. A producer
// warp streams the rows' bytes through a ring of shared-memory chunk slots by
// TMA, one copy per group of four blocks (a "quad", 80 bytes per row), so a slot
// holds [quad][row][80 bytes]: the row pitch is 5 sixteen-byte units (odd), and
// 32 lanes reading one offset of 32 consecutive (row, quad) records touch
// distinct bank groups. Consumer warps first rotate x into shared memory (a
// thread per 32-block), then take work items of 32 lanes x one quad each: lane
// l handles the pair p = 32 g + l, i.e. row p mod R of quad slice p / R (F
// slices per row, so that R * F fills whole warps even when R < 32). Per
// element, the centroid comes from a 16-word table in shared memory (16
// distinct words sit in 16 distinct banks, so lookups never conflict) and one
// fp32 FMA adds it times the rotated activation; each half block's sum is
// scaled by its d once. Rotated activations are stored per quad with 16 bytes
// of padding, so lanes of different slices reading the same offset of
// different quads fall on different banks. Every lane adds its items in item
// order; the final sums run over warps and slices in a fixed order
// (deterministic results).
//
// Fallback (tq4_direct_kernel): any K that is a multiple of 32 (the TMA row
// pitch needs K % 128 == 0) and shapes the plan above does not cover: a warp
// per row, lanes over blocks read straight from global memory, x rotated into
// shared memory per K segment, a fixed shuffle-tree reduction.
#include <algorithm>

#include "kq_common.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int TQ_BLOCK = 32;           // weights per block
constexpr int TQ_BYTES = 20;           // fp16 d0, fp16 d1, qs[16]
constexpr int TQ_QUAD = 4;             // blocks per quad
constexpr int TQ_QUAD_BYTES = 80;      // bytes of one row's quad
constexpr int TQ_XR_QUAD = 132;        // floats per quad of rotated activations (128 + 4 padding)
constexpr int TQ_NW = 16;              // consumer warps of the lane-row kernel
constexpr int TQ_MAX_PAIRS = 128;      // (row, slice) pairs per CTA: at most four groups of 32 lanes
constexpr int TQ_SMEM_LIMIT = 227 * 1024;
constexpr int TQ_CHUNK_TARGET = 24 * 1024;
constexpr int TQD_WARPS = 8;           // rows per CTA of the fallback kernel
constexpr int TQD_SEG = 512;           // blocks of x rotated per pass of the fallback kernel (64 KB)
constexpr float TQ_INV_SQRT32 = 0.17677669529663688f;
constexpr int TQ_CODE_BIAS = 4096;              // pair-table codes are 1000 * centroid + 4096 (13 bits)
constexpr float TQ_MAGIC = 8388608.0f + 4096.0f;  // float bits 0x4B000000 | code equal 2^23 + code
constexpr int TQ_PAIR_TABLE_BYTES = 256 * 64 * 4;  // a word per index byte and lane, rows of 256 bytes

// Lloyd-Max centroids of N(0, 1), index order, as printed on the page, and
// the same values times 1000 (integers, since the page prints three decimals).
__constant__ int c_tq_centroids_milli[16] = {-2733, -2069, -1618, -1256, -942, -657, -388, -128,
                                             128,   388,   657,   942,   1256, 1618, 2069, 2733};
__constant__ float c_tq_centroids[16] = {-2.733f, -2.069f, -1.618f, -1.256f, -0.942f, -0.657f, -0.388f, -0.128f,
                                         0.128f,  0.388f,  0.657f,  0.942f,  1.256f,  1.618f,  2.069f,  2.733f};

// v <- H v with the unnormalised Walsh-Hadamard matrix H[i][j] = (-1)^popcount(i & j):
// butterflies of widths 1, 2, 4, 8, 16 (natural order).
__device__ __forceinline__ void wht32(float (&v)[TQ_BLOCK]) {
#pragma unroll
  for (int h = 1; h < TQ_BLOCK; h <<= 1)
#pragma unroll
    for (int i = 0; i < TQ_BLOCK; ++i)
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
}

// Loads x[32b .. 32b+32) (16-byte aligned) and rotates it.
__device__ __forceinline__ void load_rotate(const float* __restrict__ x, int b, float (&v)[TQ_BLOCK]) {
  const float4* src = reinterpret_cast<const float4*>(x) + static_cast<size_t>(b) * 8;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float4 t = __ldg(src + k);
    v[4 * k] = t.x;
    v[4 * k + 1] = t.y;
    v[4 * k + 2] = t.z;
    v[4 * k + 3] = t.w;
  }
  wht32(v);
}

__device__ __forceinline__ void load_block(const float* src, float (&v)[TQ_BLOCK]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float4 t = s4[k];
    v[4 * k] = t.x;
    v[4 * k + 1] = t.y;
    v[4 * k + 2] = t.z;
    v[4 * k + 3] = t.w;
  }
}

__device__ __forceinline__ void store_block(float* dst, const float (&v)[TQ_BLOCK]) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int k = 0; k < 8; ++k) d[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

// The centroid whose byte offset in the table is `off` (= 4 * index).
__device__ __forceinline__ float lut_at(const float* lut, uint32_t off) {
  return *reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(lut) + off);
}

// r_b . xr_b for one block: `dw` = {d0, d1} (fp16 pair), q[0..3] = qs as four
// words (word k holds elements 8k .. 8k+7: byte m has element 8k+2m in its low
// nibble and 8k+2m+1 in its high nibble), xr = the block's 32 rotated
// activations (16-byte aligned).
__device__ __forceinline__ float block_dot(uint32_t dw, const uint32_t (&q)[4], const float* xr, const float* lut) {
  const float4* x4 = reinterpret_cast<const float4*>(xr);
  float2 s[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // per half block: even / odd elements
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w = q[k];
    const uint32_t e4 = (w << 2) & 0x3C3C3C3Cu;  // 4 * index of elements 8k, 8k+2, 8k+4, 8k+6 (one per byte)
    const uint32_t o4 = (w >> 2) & 0x3C3C3C3Cu;  // 4 * index of elements 8k+1, 8k+3, 8k+5, 8k+7
    const float4 xa = x4[2 * k], xb = x4[2 * k + 1];
    float2 a = s[k >> 1];
    a = __ffma2_rn(make_float2(lut_at(lut, e4 & 0xFFu), lut_at(lut, o4 & 0xFFu)), make_float2(xa.x, xa.y), a);
    a = __ffma2_rn(make_float2(lut_at(lut, __byte_perm(e4, 0u, 0x4441u)), lut_at(lut, __byte_perm(o4, 0u, 0x4441u))),
                   make_float2(xa.z, xa.w), a);
    a = __ffma2_rn(make_float2(lut_at(lut, __byte_perm(e4, 0u, 0x4442u)), lut_at(lut, __byte_perm(o4, 0u, 0x4442u))),
                   make_float2(xb.x, xb.y), a);
    a = __ffma2_rn(make_float2(lut_at(lut, e4 >> 24), lut_at(lut, o4 >> 24)), make_float2(xb.z, xb.w), a);
    s[k >> 1] = a;
  }
  const float d0 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw & 0xFFFFu)));
  const float d1 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw >> 16)));
  return fmaf(d1, s[1].x + s[1].y, d0 * (s[0].x + s[0].y));
}

// The same dot product with the pair table, added into acc: word (b, lane) of
// `tbl`, at byte 256 b + 4 lane, holds the codes of both centroids of index
// byte b, 1000 c[b & 15] + 4096 in its low half and 1000 c[b >> 4] + 4096 in its
// high half. Each lane reads its own copy (bank = lane), so the 32 lanes never
// conflict, one 4-byte read serves two elements, and one byte permute of the
// index word and the lane's offset forms the address. A code placed in the
// mantissa of 2^23 minus 2^23 + 4096 gives 1000 c exactly in fp32. acc gets
// d0 * (r . x) over elements 0..15 plus d1 * (r . x) over 16..31 (as an even /
// odd pair), with the table's factor 1000 left in.
__device__ __forceinline__ void block_dot_pairs(uint32_t dw, const uint32_t (&q)[4], const float* xr,
                                                const uint8_t* tbl, uint32_t laneoff, float2& acc) {
  const float4* x4 = reinterpret_cast<const float4*>(xr);
  const float2 neg_magic = make_float2(-TQ_MAGIC, -TQ_MAGIC);
  float2 s[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // per half block: even / odd elements
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w = q[k];
    const float4 xa = x4[2 * k], xb = x4[2 * k + 1];
    float2 a = s[k >> 1];
#pragma unroll
    for (int m = 0; m < 4; ++m) {  // byte m: elements 8k + 2m (low nibble) and 8k + 2m + 1
      const uint32_t t = *reinterpret_cast<const uint32_t*>(tbl + __byte_perm(w, laneoff, 0x5504u + 16u * m));
      const float2 f = make_float2(__uint_as_float(__byte_perm(t, 0x4B000000u, 0x7610u)),
                                   __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7632u)));
      const float2 c = __fadd2_rn(f, neg_magic);  // exact: 1000 * centroid
      const float2 xv = m == 0 ? make_float2(xa.x, xa.y)
                        : m == 1 ? make_float2(xa.z, xa.w)
                        : m == 2 ? make_float2(xb.x, xb.y)
                                 : make_float2(xb.z, xb.w);
      a = __ffma2_rn(c, xv, a);
    }
    s[k >> 1] = a;
  }
  const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&dw));
  acc = __ffma2_rn(s[0], make_float2(d.x, d.x), acc);
  acc = __ffma2_rn(s[1], make_float2(d.y, d.y), acc);
}

// i / d for d >= 1, with inv = ceil(2^32 / d) when d >= 2 (exact while i * d < 2^32).
__device__ __forceinline__ int fdiv(int i, int d, uint32_t inv) {
  return d == 1 ? i : static_cast<int>(__umulhi(static_cast<uint32_t>(i), inv));
}

}  // namespace

struct TqLaneRowParams {
  const float* x;
  float* y;
  int M, nq;           // rows; quads per row (K / 128)
  int R;               // rows per CTA
  int F;               // quad slices per row
  int RF;              // R * F (row, slice) pairs
  int n_groups;        // ceil(RF / 32)
  int Qc;              // quads per chunk (a multiple of F)
  int steps;           // Qc / F: quads of one slice in a chunk
  int n_chunks;        // ceil(nq / Qc)
  int qpad;            // shared-memory bytes of one quad of R rows (R * 80 rounded up to 128)
  int chunk_bytes;     // Qc * qpad
  int S;               // chunk slots
  uint32_t inv_per_chunk, inv_steps, inv_R;  // ceil(2^32 / d) for d = n_groups * steps, steps, R (d >= 2)
  int slot_off, xr_off, part_off, bar_off;   // shared-memory layout (bytes); the pair table sits at 0
  const uint8_t* pf;                         // the next call's weights, prefetched into L2 (or null)
  uint64_t pf_bytes;                         // a multiple of 16
  int* err;
};

template <int NW>
__global__ void __launch_bounds__((NW + 1) * 32, 1)
    tq4_lanerow_kernel(const __grid_constant__ CUtensorMap tmW, const TqLaneRowParams p) {
  constexpr int CT = NW * 32;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint8_t* tbl = smem;                                     // pair table at offset 0 (a constant address)
  float* xr = reinterpret_cast<float*>(smem + p.xr_off);        // [quad][132]
  float* part = reinterpret_cast<float*>(smem + p.part_off);    // [warp][group][lane]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);  // one per slot
  uint64_t* empty = full + p.S;
  volatile int* abort = reinterpret_cast<volatile int*>(empty + p.S);
  volatile int* chunks_issued = abort + 1;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * p.R;
  const int rows = min(p.R, p.M - r0);
  const int per_chunk = p.n_groups * p.steps;  // work items per chunk
  if (threadIdx.x == 0) {
    for (int sl = 0; sl < p.S; ++sl) {
      mbar_init(&full[sl], 1);
      mbar_init(&empty[sl], per_chunk);  // every item of a chunk arrives once
    }
    *abort = 0;
    *chunks_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      const uint32_t qbytes = static_cast<uint32_t>(p.R * TQ_QUAD_BYTES);
      int issued = 0;
      for (int c = 0; c < p.n_chunks; ++c) {
        const int sl = c % p.S;
        if (c == p.S) prefetch_share_l2(p.pf, p.pf_bytes);  // once the ring is primed
        if (c >= p.S && !mbar_wait(&empty[sl], ((c / p.S) - 1) & 1, abort, p.err)) break;
        const int q0 = c * p.Qc;
        const int nqc = min(p.Qc, p.nq - q0);  // quads past the row end are not copied (never used)
        mbar_expect_tx(&full[sl], static_cast<uint32_t>(nqc) * qbytes);
        uint8_t* dst = smem + p.slot_off + static_cast<size_t>(sl) * p.chunk_bytes;
        for (int k = 0; k < nqc; ++k)
          tma_load_2d(dst + static_cast<size_t>(k) * p.qpad, &tmW, &full[sl], (q0 + k) * (TQ_QUAD_BYTES / 4), r0);
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
    return;
  }

  // Pair table: word (b, l) at byte 256 b + 4 l holds the codes of index byte b
  // (the other half of each 256-byte row is unused).
  for (int e = threadIdx.x; e < 256 * 32; e += CT) {
    const int b = e >> 5;
    const uint32_t lo = static_cast<uint32_t>(c_tq_centroids_milli[b & 15] + TQ_CODE_BIAS);
    const uint32_t hi = static_cast<uint32_t>(c_tq_centroids_milli[b >> 4] + TQ_CODE_BIAS);
    reinterpret_cast<uint32_t*>(smem)[(b << 6) | (e & 31)] = lo | (hi << 16);
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel

  // x -> xr, a warp per 512-byte quad (coalesced), then each 32-block rotated
  // in place: block b sits at xr[(b / 4) * 132 + (b % 4) * 32 ...].
  for (int q0 = warp; q0 < p.nq; q0 += 8 * NW) {  // up to eight loads in flight per lane
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = q0 + i * NW;
      if (q < p.nq) v[i] = __ldg(reinterpret_cast<const float4*>(p.x) + static_cast<size_t>(q) * 32 + lane);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = q0 + i * NW;
      if (q < p.nq) *reinterpret_cast<float4*>(xr + q * TQ_XR_QUAD + 4 * lane) = v[i];
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(CT) : "memory");
  const int nbt = p.nq * TQ_QUAD;
  for (int b = threadIdx.x; b < nbt; b += CT) {
    float* blk = xr + (b >> 2) * TQ_XR_QUAD + (b & 3) * TQ_BLOCK;
    float v[TQ_BLOCK];
    load_block(blk, v);
    wht32(v);
    store_block(blk, v);
  }
  asm volatile("bar.sync 1, %0;" ::"r"(CT) : "memory");

  const int items = p.n_chunks * per_chunk;
  int ready = -1, sl = -1, phase = 0;  // last chunk seen, its slot and the slot's fill parity
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // this warp's sums for lane groups 0..3
  for (int i = warp; i < items; i += NW) {
    // i = (c * n_groups + g) * steps + t
    const int c = fdiv(i, per_chunk, p.inv_per_chunk);
    const int rem = i - c * per_chunk;
    const int g = fdiv(rem, p.steps, p.inv_steps);
    const int t = rem - g * p.steps;
    if (c != ready) {
      while (ready < c) {  // chunks only move forward: slot c % S, parity (c / S) & 1
        ++ready;
        if (++sl == p.S) {
          sl = 0;
          phase ^= 1;
        }
      }
      // chunk c issued first: the parity wait cannot take an older fill of the slot
      if (!wait_counter_above(chunks_issued, c, abort, p.err) || !mbar_wait(&full[sl], phase, abort, p.err)) break;
    }
    const int pr = min(32 * g + lane, p.RF - 1);  // lanes past the last pair repeat it; their result is dropped
    const int s = fdiv(pr, p.R, p.inv_R);
    const int row = pr - s * p.R;
    const int ql = s + p.F * t;  // quad within the chunk
    const int q = c * p.Qc + ql;  // quad within the row
    const bool valid = q < p.nq;
    const int qx = valid ? q : p.nq - 1;  // past the row end: read a valid quad, drop the result
    const uint4* wq = reinterpret_cast<const uint4*>(smem + p.slot_off + static_cast<size_t>(sl) * p.chunk_bytes +
                                                     static_cast<size_t>(ql) * p.qpad + row * TQ_QUAD_BYTES);
    const uint4 u0 = wq[0], u1 = wq[1], u2 = wq[2], u3 = wq[3], u4 = wq[4];
    // block 0: words 0..4, block 1: 5..9, block 2: 10..14, block 3: 15..19
    const uint32_t qa[4] = {u0.y, u0.z, u0.w, u1.x};
    const uint32_t qb[4] = {u1.z, u1.w, u2.x, u2.y};
    const uint32_t qc[4] = {u2.w, u3.x, u3.y, u3.z};
    const uint32_t qd[4] = {u4.x, u4.y, u4.z, u4.w};
    const float* xq = xr + qx * TQ_XR_QUAD;
    const uint32_t laneoff = static_cast<uint32_t>(lane) * 4u;
    float2 a2 = make_float2(0.f, 0.f);
    block_dot_pairs(u0.x, qa, xq, tbl, laneoff, a2);
    block_dot_pairs(u1.y, qb, xq + TQ_BLOCK, tbl, laneoff, a2);
    block_dot_pairs(u2.z, qc, xq + 2 * TQ_BLOCK, tbl, laneoff, a2);
    block_dot_pairs(u3.w, qd, xq + 3 * TQ_BLOCK, tbl, laneoff, a2);
    float v = a2.x + a2.y;
    v = valid ? v : 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] += (g == k) ? v : 0.f;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[sl]);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (k < p.n_groups) part[(warp * p.n_groups + k) * 32 + lane] = acc[k];
  asm volatile("bar.sync 1, %0;" ::"r"(CT) : "memory");
  // y[row] = (Sum over warps, then over slices, in that order) / sqrt(32)
  for (int r = threadIdx.x; r < rows; r += CT) {
    float a = 0.f;
    for (int w = 0; w < NW; ++w)
      for (int s = 0; s < p.F; ++s) {
        const int pidx = s * p.R + r;
        a += part[(w * p.n_groups + (pidx >> 5)) * 32 + (pidx & 31)];
      }
    p.y[r0 + r] = a * (0.001f * TQ_INV_SQRT32);  // the pair table's codes are 1000 c
  }
}

// Fallback: warp per row; lane j takes blocks j, j + 32, ... of each K segment.
__global__ void __launch_bounds__(TQD_WARPS * 32) tq4_direct_kernel(const uint8_t* __restrict__ W,
                                                                    const float* __restrict__ x, float* __restrict__ y,
                                                                    int M, int nbt) {
  extern __shared__ __align__(128) float tq_direct_smem[];  // the table (32 floats reserved), then the segment
  float* lut = tq_direct_smem;
  float* xs = tq_direct_smem + 32;  // [seg][32] rotated activations of the segment
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * TQD_WARPS + warp;
  if (threadIdx.x < 16) lut[threadIdx.x] = c_tq_centroids[threadIdx.x];
  const size_t rs = static_cast<size_t>(nbt) * TQ_BYTES;
  float acc = 0.f;
  for (int b0 = 0; b0 < nbt; b0 += TQD_SEG) {
    const int nb = min(TQD_SEG, nbt - b0);
    __syncthreads();  // the previous segment is consumed (and the table is written)
    for (int b = threadIdx.x; b < nb; b += TQD_WARPS * 32) {
      float v[TQ_BLOCK];
      load_rotate(x, b0 + b, v);
      store_block(xs + b * TQ_BLOCK, v);
    }
    __syncthreads();
    if (row < M) {
      const uint8_t* wr = W + static_cast<size_t>(row) * rs;
      for (int b = lane; b < nb; b += 32) {
        const uint32_t* w4 = reinterpret_cast<const uint32_t*>(wr + static_cast<size_t>(b0 + b) * TQ_BYTES);
        const uint32_t q[4] = {__ldg(w4 + 1), __ldg(w4 + 2), __ldg(w4 + 3), __ldg(w4 + 4)};
        acc += block_dot(__ldg(w4), q, xs + b * TQ_BLOCK, lut);
      }
    }
  }
  acc = warp_sum_f(acc);
  if (row < M && lane == 0) y[row] = acc * TQ_INV_SQRT32;
}

namespace {

inline int round_up_i(int v, int a) { return (v + a - 1) / a * a; }
inline uint32_t recip32(int d) { return static_cast<uint32_t>(((uint64_t(1) << 32) + d - 1) / d); }

// Plan of the lane-row kernel; false when the shape does not suit it.
bool plan_tq_lanerow(int64_t M, int64_t K, int num_sms, TqLaneRowParams* p, int* grid, size_t* smem) {
  if (K % (TQ_QUAD * TQ_BLOCK) != 0 || K > (int64_t(1) << 22)) return false;  // TMA row pitch: K % 128 == 0
  const int nq = static_cast<int>(K / (TQ_QUAD * TQ_BLOCK));
  const int64_t G0 = std::min<int64_t>(M, num_sms);
  const int64_t R = (M + G0 - 1) / G0;
  if (R > TQ_MAX_PAIRS) return false;
  p->M = static_cast<int>(M);
  p->nq = nq;
  p->R = static_cast<int>(R);
  *grid = static_cast<int>((M + R - 1) / R);
  // Slices per row: the fewest that waste the fewest lanes.
  int best_f = 1;
  double best_waste = 2.0;
  for (int f = 1; f <= 32 && p->R * f <= TQ_MAX_PAIRS; f <<= 1) {
    const int pairs = p->R * f;
    const double waste = 1.0 - static_cast<double>(pairs) / round_up_i(pairs, 32);
    if (waste < best_waste - 1e-9) {
      best_waste = waste;
      best_f = f;
    }
  }
  p->F = best_f;
  p->RF = p->R * p->F;
  p->n_groups = (p->RF + 31) / 32;
  p->qpad = round_up_i(p->R * TQ_QUAD_BYTES, 128);
  const int per_slot_quads = std::max(1, TQ_CHUNK_TARGET / (p->F * p->qpad)) * p->F;
  p->Qc = std::min(per_slot_quads, round_up_i(nq, p->F));
  p->steps = p->Qc / p->F;
  p->chunk_bytes = p->Qc * p->qpad;
  p->n_chunks = (nq + p->Qc - 1) / p->Qc;
  const int xr_bytes = round_up_i(nq * TQ_XR_QUAD * 4, 128);
  const int part_bytes = TQ_NW * p->n_groups * 32 * 4;
  const size_t fixed = static_cast<size_t>(xr_bytes) + part_bytes + TQ_PAIR_TABLE_BYTES + 16;
  if (fixed + p->chunk_bytes + 16 > static_cast<size_t>(TQ_SMEM_LIMIT)) return false;
  const int S = static_cast<int>((TQ_SMEM_LIMIT - fixed) / (p->chunk_bytes + 16));
  p->S = std::min(S, p->n_chunks);
  if (p->S < 2 && p->n_chunks > 1) return false;
  const int per_chunk = p->n_groups * p->steps;
  if (static_cast<int64_t>(p->n_chunks) * per_chunk * per_chunk >= (int64_t(1) << 32)) return false;
  p->inv_per_chunk = per_chunk >= 2 ? recip32(per_chunk) : 0u;
  p->inv_steps = p->steps >= 2 ? recip32(p->steps) : 0u;
  p->inv_R = p->R >= 2 ? recip32(p->R) : 0u;
  size_t off = TQ_PAIR_TABLE_BYTES;  // the pair table
  p->slot_off = static_cast<int>(off);
  off += static_cast<size_t>(p->S) * p->chunk_bytes;
  p->xr_off = static_cast<int>(off);
  off += xr_bytes;
  p->part_off = static_cast<int>(off);
  off += part_bytes;
  p->bar_off = static_cast<int>(off);
  off += static_cast<size_t>(2 * p->S) * sizeof(uint64_t) + 16;  // + abort, chunks issued
  *smem = off;
  return *smem <= static_cast<size_t>(TQ_SMEM_LIMIT);
}

}  // namespace

cudaError_t launch_tq4_matvec(const void* W, const float* x, float* y, int64_t M, int64_t K, const void* pf,
                              uint64_t pf_bytes, int* err, int num_sms, cudaStream_t s, int* status) {
  *status = KQ_OK;
  TqLaneRowParams lp{};
  int grid = 0;
  size_t smem = 0;
  if (plan_tq_lanerow(M, K, num_sms, &lp, &grid, &smem)) {
    CUtensorMap tmW;
    const uint64_t rs = static_cast<uint64_t>(K / TQ_BLOCK) * TQ_BYTES;  // a multiple of 16 here
    if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, rs / 4, static_cast<uint64_t>(M), rs,
                        static_cast<uint32_t>(TQ_QUAD_BYTES / 4), static_cast<uint32_t>(lp.R),
                        CU_TENSOR_MAP_SWIZZLE_NONE)) {
      *status = KQ_ERR_CUDA;
      return cudaSuccess;
    }
    lp.x = x;
    lp.y = y;
    lp.pf = static_cast<const uint8_t*>(pf);
    lp.pf_bytes = pf_bytes;
    lp.err = err;
    cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(tq4_lanerow_kernel<TQ_NW>), 24);
    if (e != cudaSuccess) return e;
    return launch_pdl(tq4_lanerow_kernel<TQ_NW>, dim3(grid), dim3((TQ_NW + 1) * 32), smem, s, tmW, lp);
  }
  const int nbt = static_cast<int>(K / TQ_BLOCK);
  const size_t dsmem = static_cast<size_t>(std::min(nbt, TQD_SEG) + 1) * TQ_BLOCK * sizeof(float);
  const int64_t blocks = (M + TQD_WARPS - 1) / TQD_WARPS;
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(tq4_direct_kernel), 25);
  if (e != cudaSuccess) return e;
  return launch_pdl(tq4_direct_kernel, dim3(static_cast<unsigned>(blocks)), dim3(TQD_WARPS * 32), dsmem, s,
                    static_cast<const uint8_t*>(W), x, y, static_cast<int>(M), nbt);
}

}  // namespace kq
