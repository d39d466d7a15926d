// Prefill GEMM and MoE grouped GEMM on the fifth-generation tensor cores.
//
// Y[n, m] = Sum_k dequant(W)[m, k] * x_hat[n, k], x_hat = fp16(d_h * q) of the
// Q8_1 activations.
//
// Method: "ZINC MMQ v2 — Fused Q4_K×Q8_1 Tensor-Core GEMM" (Kernel
// architecture: weight tiles unpacked once in shared memory and fed to the
// tensor cores; Persistent kernel + atomic work queue; MoE routing: the
// expert's weight tile is loaded once for all of its tokens) and "Prefill Gap
// Closure Plan" (T1 fused dequant GEMM; T2 grouped expert GEMM with histogram,
// prefix sum and scatter). The pages' kernels target sm_89/sm_120 with
// mma.sync and cp.async; this one is built for sm_103a:
//
//  * warp 20 streams raw weight super-blocks (128 rows x 1 super-block per
//    stage) with 2-D TMA, warp 22 streams x_hat tiles (128-byte swizzle) with
//    2-D TMA, each into its own mbarrier ring;
//  * warps 0-15 (two groups of 8 taking alternate K steps, so two steps are
//    unpacked at once) unpack Q4_K / Q5_K / Q6_K to fp16 and store the A operand straight
//    into tensor memory (tcgen05.st; the page unpacks into shared memory), four
//    64-wide K steps per super-block: the weights never pass through shared
//    memory as fp16, which leaves its bandwidth to the x_hat tiles the MMA
//    reads from there;
//  * one thread of warp 21 issues tcgen05.mma (M=128, N<=256, K=16, A from
//    tensor memory, B from shared memory) into a tensor-memory accumulator;
//  * warps 16-19 drain finished accumulators (tcgen05.ld) to global memory
//    (with two accumulators, while the next tile is being computed).
//
// The grid is persistent (one CTA per SM). The raw producer picks each CTA's
// next tile and hands its index to the other roles through a small ring in
// shared memory: dense tiles (all the same cost) are strided statically; MoE
// tiles come from an atomic tile queue in the workspace ("ZINC MMQ v2",
// Persistent kernel + atomic work queue). Every output element is computed
// inside one tile, so results do not depend on which CTA takes which tile; a
// split K range is summed afterwards in a fixed order. Every wait is bounded
// (ERR_WAIT_TIMEOUT, no hang).
#include <algorithm>
#include <climits>
#include <mutex>

#include "kq_internal.h"
#include "kq_common.cuh"

namespace kq {

constexpr int GM_BM = 128;            // weight rows per tile (MMA M)
constexpr int GM_BNMAX = 256;         // largest token tile (MMA N)
constexpr int GM_BK = 64;             // K per A/B stage: one 128-byte swizzled row of fp16
constexpr int GM_A_COLS = GM_BK / 2;  // tensor-memory columns of one A stage (two fp16 per column)
constexpr int GM_A_MAX_STAGES = 8;
constexpr int GM_BBOX = 64;           // token rows per x_hat TMA box
constexpr int GM_BBOX_BYTES = GM_BBOX * GM_BK * 2;
constexpr int GM_DQ_WARPS = 16;       // warps 0..15: two groups of 8, alternate K steps
constexpr int GM_DQ_GROUP = 8;        // unpacking warps per K step (4 lane quarters x 2 halves)
constexpr int GM_EPI_WARP0 = 16;      // warps 16..19
constexpr int GM_RAW_WARP = 20;
constexpr int GM_MMA_WARP = 21;
constexpr int GM_B_WARP = 22;
constexpr int GM_THREADS = 23 * 32;
constexpr int GM_TMEM_COLS = 512;     // accumulators, then the A stages
constexpr int GM_SMEM_LIMIT = 227 * 1024;
constexpr int MOE_MAX_EXPERTS = 512;
constexpr int GM_TQ = 4;              // tile-index ring slots
// Warps that read each tile index: the x_hat producer, the MMA issuer, the
// unpackers and the epilogue (one arrival per warp on the slot's empty barrier).
constexpr int GM_TQ_READERS = 1 + 1 + GM_DQ_WARPS + 4;

template <int WT>
struct RawBox;
template <>
struct RawBox<KQ_Q4_K> {
  static constexpr int BYTES = 144;  // one Q4_K super-block per row, 16-byte aligned in a row
};
template <>
struct RawBox<KQ_Q5_K> {
  static constexpr int BYTES = 176;  // one Q5_K super-block per row, 16-byte aligned in a row
};
template <>
struct RawBox<KQ_Q6_K> {
  // A 16-byte aligned window covering one 210-byte Q6_K block (which starts up
  // to 14 bytes in). 240 bytes = 60 words: the unpackers' 32-bit loads of 32
  // consecutive rows then fall on 8 distinct banks per 8 rows (4-way at most),
  // where a 224-byte pitch gives 8-way conflicts.
  static constexpr int BYTES = 240;
};

struct GemmArgs {
  int M;            // output rows (per expert for MoE)
  int N;            // token rows of x_hat
  int nb;           // super-blocks per weight row
  int m_tiles, n_tiles, splits, bn;
  int k_stages, raw_stages;  // K-step stages (A in tensor memory + B in shared memory), raw rings
  int b_stage_bytes;
  int n_acc;        // tensor-memory accumulators (1 or 2)
  int acc_cols;     // columns per accumulator
  int a_col0;       // first tensor-memory column of the A stages
  float* Y;
  float* partial;   // split-K partial sums [splits][N][M]
  // MoE
  int n_experts;
  const int* counts;
  const int* offsets;
  const int* tile_start;
  const int* entries;
  int* tile_queue;  // MoE: next tile index minus gridDim.x (zeroed by the routing kernel)
  int* err;
  int hold;         // kq_test_hold_copies: the raw producer issues nothing and hands out no tile
};

struct Tile {
  int wrow0;   // first weight row (global row of the concatenated matrix)
  int m0;      // first output row
  int xrow0;   // first x_hat row
  int ncols;   // valid tokens in the tile
  int kb0, kb1;
  int split;
  int e;       // expert (MoE)
  int nbase;   // entries index of column 0 (MoE)
};

// Dense tiles: t = (m_tile * n_tiles + n_tile) * splits + split. A CTA pair
// takes 256 weight rows (m_tiles counts pairs of 128-row tiles); the CTA of
// rank r computes rows 128 r .. 128 r + 127 of them.
template <bool MOE, bool PAIR>
__device__ __forceinline__ Tile decode_tile(const GemmArgs& a, int t, int rank, const int* s_tile_start,
                                            const int* s_counts, const int* s_offsets) {
  Tile T;
  if (!MOE) {
    const int split = t % a.splits;
    const int mn = t / a.splits;
    const int nt = mn % a.n_tiles, mt = mn / a.n_tiles;
    T.m0 = (PAIR ? 2 * mt + rank : mt) * GM_BM;
    T.wrow0 = T.m0;
    T.xrow0 = nt * a.bn;
    T.ncols = min(a.bn, a.N - T.xrow0);
    T.split = split;
    T.kb0 = static_cast<int>(static_cast<int64_t>(split) * a.nb / a.splits);
    T.kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * a.nb / a.splits);
    T.e = 0;
    T.nbase = 0;
  } else {
    int lo = 0, hi = a.n_experts;  // find e with tile_start[e] <= t < tile_start[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int local = t - s_tile_start[e];
    const int nch = (s_counts[e] + a.bn - 1) / a.bn;
    const int mt = local / nch, nc = local % nch;
    T.e = e;
    T.m0 = mt * GM_BM;
    T.wrow0 = e * a.M + T.m0;
    T.nbase = s_offsets[e] + nc * a.bn;
    T.xrow0 = T.nbase;
    T.ncols = min(a.bn, s_counts[e] - nc * a.bn);
    T.kb0 = 0;
    T.kb1 = a.nb;
    T.split = 0;
  }
  return T;
}

// Next tile index from the ring (called by a whole warp, or by one lane when
// `one_lane`). Returns INT_MAX when a wait gave up.
__device__ __forceinline__ int tq_pop(uint64_t* full, uint64_t* empty, const int* ids, int& qi, uint32_t& qph,
                                      bool one_lane, volatile int* abort, int* err) {
  if (!mbar_wait(&full[qi], qph, abort, err)) return INT_MAX;
  const int t = *reinterpret_cast<const volatile int*>(&ids[qi]);
  if (one_lane) {
    mbar_arrive(&empty[qi]);
  } else {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[qi]);
  }
  if (++qi == GM_TQ) {
    qi = 0;
    qph ^= 1;
  }
  return t;
}

// --- weight unpacking into the fp16 A operand ---------------------------------
// A stage: 128 rows (tensor-memory lanes) x 64 K of fp16, two per 32-bit
// column, lower k in the low half. The thread of row r and half hf produces
// the 32 weights k = 16hf .. 16hf+15 (columns 8hf .. 8hf+7, lo[]) and
// k = 32+16hf .. 32+16hf+15 (columns 16+8hf .. 16+8hf+7, hi[]) of the step,
// so that each byte of the weight codes is read from shared memory once.

// Q4_K, K step s (0..3) of a super-block covers sub-blocks 2s (the low
// nibbles of qs[32s..32s+31]) and 2s+1 (their high nibbles). Half hf reads the
// 16 bytes qs[32s+16hf ..]: their low nibbles are weights 16hf.. of sub-block
// 2s, their high nibbles weights 16hf.. of sub-block 2s+1. Every weight
// w = d*sc*nib - dmin*m is one fp16 fma on the exact nibble. hdr is the
// block's first 16 bytes (d, dmin, packed 6-bit scales and mins).
__device__ __forceinline__ void dequant_q4k(const uint4& hdr, const uint8_t* __restrict__ raw, int s, int r, int hf,
                                            uint32_t (&lo)[8], uint32_t (&hi)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(raw + r * Q4K_BYTES + 16 + 32 * s + 16 * hf);
  uint32_t scw, mw;  // 6-bit scales / mins of sub-blocks 0-3 (s < 2) or 4-7, one per byte
  if (s < 2) {
    scw = hdr.y & 0x3F3F3F3Fu;
    mw = hdr.z & 0x3F3F3F3Fu;
  } else {
    scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    mw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
  }
  const int b0 = (s & 1) * 16;  // byte of sub-block 2s; 2s+1 is the next byte
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
  const __half2 sc_lo = __float2half2_rn(d * static_cast<float>((scw >> b0) & 0xFFu));
  const __half2 mn_lo = __float2half2_rn(-(dmin * static_cast<float>((mw >> b0) & 0xFFu)));
  const __half2 sc_hi = __float2half2_rn(d * static_cast<float>((scw >> (b0 + 8)) & 0xFFu));
  const __half2 mn_hi = __float2half2_rn(-(dmin * static_cast<float>((mw >> (b0 + 8)) & 0xFFu)));
  const __half2 k1024 = __float2half2_rn(1024.f);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // bytes 0,1 (and 2,3) -> fp16 (1024 + nibble) pairs, low then high nibbles
    const uint32_t l0 = __byte_perm(w[i], 0x64646464u, 0x5140) & 0xFF0FFF0Fu;
    const uint32_t l1 = __byte_perm(w[i], 0x64646464u, 0x7362) & 0xFF0FFF0Fu;
    const uint32_t h0 = __byte_perm(w[i] >> 4, 0x64646464u, 0x5140) & 0xFF0FFF0Fu;
    const uint32_t h1 = __byte_perm(w[i] >> 4, 0x64646464u, 0x7362) & 0xFF0FFF0Fu;
    lo[2 * i] = half2_bits(__hfma2(__hsub2(bits_half2(l0), k1024), sc_lo, mn_lo));
    lo[2 * i + 1] = half2_bits(__hfma2(__hsub2(bits_half2(l1), k1024), sc_lo, mn_lo));
    hi[2 * i] = half2_bits(__hfma2(__hsub2(bits_half2(h0), k1024), sc_hi, mn_hi));
    hi[2 * i + 1] = half2_bits(__hfma2(__hsub2(bits_half2(h1), k1024), sc_hi, mn_hi));
  }
}

// Q5_K K step s, the Q4_K unpack with 5-bit codes: the 16 nibble bytes of half
// hf of sub-blocks 2s (low nibbles) and 2s+1 (high nibbles) take their fifth
// bits from bits 2s and 2s+1 of the matching qh bytes (qh[16 hf ..]); a code q
// (0..31) becomes fp16 1024 + q in one byte permute, as in dequant_q4k.
__device__ __forceinline__ void dequant_q5k(const uint4& hdr, const uint8_t* __restrict__ raw, int s, int r, int hf,
                                            uint32_t (&lo)[8], uint32_t (&hi)[8]) {
  const uint8_t* row = raw + r * Q5K_BYTES;
  const uint4 q = *reinterpret_cast<const uint4*>(row + 48 + 32 * s + 16 * hf);
  const uint4 qh = *reinterpret_cast<const uint4*>(row + 16 + 16 * hf);
  uint32_t scw, mw;
  if (s < 2) {
    scw = hdr.y & 0x3F3F3F3Fu;
    mw = hdr.z & 0x3F3F3F3Fu;
  } else {
    scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    mw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
  }
  const int b0 = (s & 1) * 16;
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
  const __half2 sc_lo = __float2half2_rn(d * static_cast<float>((scw >> b0) & 0xFFu));
  const __half2 mn_lo = __float2half2_rn(-(dmin * static_cast<float>((mw >> b0) & 0xFFu)));
  const __half2 sc_hi = __float2half2_rn(d * static_cast<float>((scw >> (b0 + 8)) & 0xFFu));
  const __half2 mn_hi = __float2half2_rn(-(dmin * static_cast<float>((mw >> (b0 + 8)) & 0xFFu)));
  const __half2 k1024 = __float2half2_rn(1024.f);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  const uint32_t h[4] = {qh.x, qh.y, qh.z, qh.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t cl = (w[i] & 0x0F0F0F0Fu) | (((h[i] >> (2 * s)) & 0x01010101u) << 4);
    const uint32_t ch = ((w[i] >> 4) & 0x0F0F0F0Fu) | (((h[i] >> (2 * s + 1)) & 0x01010101u) << 4);
    const uint32_t l0 = __byte_perm(cl, 0x64646464u, 0x5140);
    const uint32_t l1 = __byte_perm(cl, 0x64646464u, 0x7362);
    const uint32_t h0 = __byte_perm(ch, 0x64646464u, 0x5140);
    const uint32_t h1 = __byte_perm(ch, 0x64646464u, 0x7362);
    lo[2 * i] = half2_bits(__hfma2(__hsub2(bits_half2(l0), k1024), sc_lo, mn_lo));
    lo[2 * i + 1] = half2_bits(__hfma2(__hsub2(bits_half2(l1), k1024), sc_lo, mn_lo));
    hi[2 * i] = half2_bits(__hfma2(__hsub2(bits_half2(h0), k1024), sc_hi, mn_hi));
    hi[2 * i + 1] = half2_bits(__hfma2(__hsub2(bits_half2(h1), k1024), sc_hi, mn_hi));
  }
}

// The 4 words that start d bytes into the 32-byte window w (d even, < 16; the
// same d for every thread of a K-block, so the branch does not diverge).
__device__ __forceinline__ void window4(const uint4& a, const uint4& b, int d, uint32_t (&out)[4]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const int sh = (d & 3) * 8;
  switch (d >> 2) {
    case 0:
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
      break;
    case 1:
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = __funnelshift_r(w[i + 1], w[i + 2], sh);
      break;
    case 2:
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = __funnelshift_r(w[i + 2], w[i + 3], sh);
      break;
    default:
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = __funnelshift_r(w[i + 3], w[i + 4], sh);
      break;
  }
}

// Q6_K half h (weights 128h .. 128h+127) of a block, for the 16 positions
// l = 16hf .. 16hf+15 of its four quarters: ql[64h + l] (quarters 0 and 2),
// ql[64h + 32 + l] (quarters 1 and 3) and qh[32h + l] (2 bits of each
// quarter). The block starts `rem` bytes into the row's 16-byte aligned window,
// so each 16 bytes come from two aligned 16-byte loads.
struct Q6Half {
  uint32_t qa[4], qb[4], qh[4];
};
__device__ __forceinline__ void load_q6k_half(const uint8_t* __restrict__ raw, int rem, int h, int r, int hf,
                                              Q6Half& q) {
  const uint8_t* row = raw + r * RawBox<KQ_Q6_K>::BYTES;
  const uint4* pa = reinterpret_cast<const uint4*>(row + 64 * h + 16 * hf);
  const uint4* pb = reinterpret_cast<const uint4*>(row + 64 * h + 32 + 16 * hf);
  const uint4* ph = reinterpret_cast<const uint4*>(row + 128 + 32 * h + 16 * hf);
  window4(pa[0], pa[1], rem, q.qa);
  window4(pb[0], pb[1], rem, q.qb);
  window4(ph[0], ph[1], rem, q.qh);
}

// Q6_K K step s: half h = s/2, quarters g0 = 2(s&1) (k = l of the step) and
// g0+1 (k = 32 + l). Weight d*sc*(q-32), q = 4 bits of ql | 2 bits of qh, sc the
// int8 scale of the 16 positions l = 16hf.. of the quarter.
__device__ __forceinline__ void dequant_q6k(const uint8_t* __restrict__ raw, int rem, const Q6Half& q, int s, int r,
                                            int hf, uint32_t (&lo)[8], uint32_t (&hi)[8]) {
  const uint8_t* blk = raw + r * RawBox<KQ_Q6_K>::BYTES + rem;
  const int h = s >> 1, g0 = 2 * (s & 1);
  const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
  const int8_t* scp = reinterpret_cast<const int8_t*>(blk + 192 + 8 * h + hf);
  const __half2 s0 = __float2half2_rn(d * static_cast<float>(scp[2 * g0]));
  const __half2 s1 = __float2half2_rn(d * static_cast<float>(scp[2 * g0 + 2]));
  const __half2 k1056 = __float2half2_rn(1056.f);
  const bool low = (s & 1) == 0;  // quarters 0,1 use low nibbles, 2,3 high
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t la = low ? (q.qa[i] & 0x0F0F0F0Fu) : ((q.qa[i] >> 4) & 0x0F0F0F0Fu);
    const uint32_t lb = low ? (q.qb[i] & 0x0F0F0F0Fu) : ((q.qb[i] >> 4) & 0x0F0F0F0Fu);
    const uint32_t va = la | (((q.qh[i] >> (2 * g0)) & 0x03030303u) << 4);
    const uint32_t vb = lb | (((q.qh[i] >> (2 * g0 + 2)) & 0x03030303u) << 4);
    lo[2 * i] = half2_bits(__hmul2(__hsub2(bits_half2(__byte_perm(va, 0x64646464u, 0x5140)), k1056), s0));
    lo[2 * i + 1] = half2_bits(__hmul2(__hsub2(bits_half2(__byte_perm(va, 0x64646464u, 0x7362)), k1056), s0));
    hi[2 * i] = half2_bits(__hmul2(__hsub2(bits_half2(__byte_perm(vb, 0x64646464u, 0x5140)), k1056), s1));
    hi[2 * i + 1] = half2_bits(__hmul2(__hsub2(bits_half2(__byte_perm(vb, 0x64646464u, 0x7362)), k1056), s1));
  }
}

// PAIR (dense only): the kernel runs in clusters of two CTAs on neighbouring
// SMs. Both CTAs stream and unpack their own 128 weight rows into their own
// tensor memory and load half of the tile's x_hat rows; one thread of the even
// CTA issues M = 256 MMAs (cta_group::2) that read both CTAs' operands and
// write each CTA's accumulator. Each SM then holds, and pulls from L2, only
// half of every B stage. Barrier roles in a pair: k_full and acc_empty of the
// even CTA collect both CTAs' arrivals (and both x_hat halves' bytes); the MMA
// commits arrive on k_empty and acc_full of both CTAs.
template <int WT, bool MOE, bool PAIR>
__global__ void __launch_bounds__(GM_THREADS, 1)
    kq_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmArgs a) {
  static_assert(!(MOE && PAIR), "the MoE kernel runs unpaired");
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  constexpr int RAW_BYTES = RawBox<WT>::BYTES * GM_BM;
  uint8_t* sB = smem;
  uint8_t* sRaw = sB + a.k_stages * a.b_stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + a.raw_stages * RAW_BYTES);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + a.raw_stages;
  // One full/empty barrier pair per K step: the x_hat TMA (its transaction
  // bytes and the producer's arrival) and the eight unpacking warps of the
  // step complete `full`; one MMA commit frees both operands through `empty`.
  uint64_t* k_full = raw_empty + a.raw_stages;
  uint64_t* k_empty = k_full + a.k_stages;
  uint64_t* acc_full = k_empty + a.k_stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* tq_full = acc_empty + 2;
  uint64_t* tq_empty = tq_full + GM_TQ;
  int* tq_ids = reinterpret_cast<int*>(tq_empty + GM_TQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tq_ids + GM_TQ);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_tile_start = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_counts = s_tile_start + (a.n_experts + 1);
  int* s_offsets = s_counts + a.n_experts;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_stride = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.raw_stages; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], GM_DQ_WARPS);
    }
    for (int i = 0; i < a.k_stages; ++i) {
      mbar_init(&k_full[i], 1 + (PAIR ? 2 : 1) * GM_DQ_GROUP);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], PAIR ? 8 : 4);
    }
    for (int i = 0; i < GM_TQ; ++i) {
      mbar_init(&tq_full[i], 1);
      mbar_init(&tq_empty[i], GM_TQ_READERS);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == GM_MMA_WARP) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, GM_TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, GM_TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (warp == GM_RAW_WARP && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  // Programmatic dependent launch: the dense GEMM's weight stream does not
  // depend on the previous kernel (W is read-only; the caller's contract), so
  // the raw producer starts at once; the x_hat producer and the epilogue wait
  // for the previous grid below. The MoE tile tables come from the routing
  // kernel, so every role of the MoE kernel waits here.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (MOE) asm volatile("griddepcontrol.wait;" ::: "memory");
  int total_tiles;
  if (MOE) {
    for (int i = threadIdx.x; i <= a.n_experts; i += GM_THREADS) s_tile_start[i] = a.tile_start[i];
    for (int i = threadIdx.x; i < a.n_experts; i += GM_THREADS) {
      s_counts[i] = a.counts[i];
      s_offsets[i] = a.offsets[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the other CTA's barriers and tensor memory are ready too
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (MOE)
    total_tiles = s_tile_start[a.n_experts];
  else
    total_tiles = a.m_tiles * a.n_tiles * a.splits;

  if (warp == GM_RAW_WARP) {
    // ---- raw weight producer -------------------------------------------------
    // It also picks the CTA's tiles: the first is its CTA (pair) index, later
    // ones come from the MoE tile queue or, for the dense GEMM, a fixed stride.
    if (lane == 0 && !a.hold) {
      int st = 0, qi = 0;
      uint32_t ph = 0, qph = 0;
      for (int t = tile0;;) {
        if (!mbar_wait(&tq_empty[qi], qph ^ 1, abort, a.err)) break;
        tq_ids[qi] = t;
        mbar_arrive(&tq_full[qi]);
        if (++qi == GM_TQ) {
          qi = 0;
          qph ^= 1;
        }
        if (t >= total_tiles || *abort) break;
        const Tile T = decode_tile<MOE, PAIR>(a, t, rank, s_tile_start, s_counts, s_offsets);
        for (int kb = T.kb0; kb < T.kb1; ++kb) {
          if (!mbar_wait(&raw_empty[st], ph ^ 1, abort, a.err)) break;
          mbar_expect_tx(&raw_full[st], RAW_BYTES);
          const int x = (WT == KQ_Q4_K) ? kb * Q4K_BYTES : (WT == KQ_Q5_K) ? kb * Q5K_BYTES : ((kb * Q6K_BYTES) & ~15);
          tma_load_2d(sRaw + st * RAW_BYTES, &tmW, &raw_full[st], x, T.wrow0);
          if (++st == a.raw_stages) {
            st = 0;
            ph ^= 1;
          }
        }
        t = MOE ? static_cast<int>(gridDim.x) + atomicAdd(a.tile_queue, 1) : t + tile_stride;
      }
    }
  } else if (warp == GM_B_WARP) {
    // ---- activation producer -------------------------------------------------
    if (!MOE) asm volatile("griddepcontrol.wait;" ::: "memory");  // x_hat comes from the previous kernel
    if (lane == 0) {
      int st = 0, qi = 0;
      uint32_t ph = 0, qph = 0;
      for (;;) {
        const int t = tq_pop(tq_full, tq_empty, tq_ids, qi, qph, true, abort, a.err);
        if (t >= total_tiles || *abort) break;
        const Tile T = decode_tile<MOE, PAIR>(a, t, rank, s_tile_start, s_counts, s_offsets);
        // Boxes of 64 token rows that hold at least one valid token. A pair
        // splits the tile's bn rows in halves; the even CTA's barrier expects
        // the bytes of both halves.
        int nbox, xrow, expect;
        if (PAIR) {
          const int hb = a.bn / (2 * GM_BBOX);
          const int n0 = min(hb, (T.ncols + GM_BBOX - 1) / GM_BBOX);
          const int n1 = max(0, min(hb, (T.ncols - hb * GM_BBOX + GM_BBOX - 1) / GM_BBOX));
          nbox = rank ? n1 : n0;
          xrow = T.xrow0 + rank * hb * GM_BBOX;
          expect = (n0 + n1) * GM_BBOX_BYTES;
        } else {
          nbox = (T.ncols + GM_BBOX - 1) / GM_BBOX;
          xrow = T.xrow0;
          expect = nbox * GM_BBOX_BYTES;
        }
        for (int kb = T.kb0; kb < T.kb1 && !*abort; ++kb) {
          if (!PAIR) {
            // Two K steps per round: the round's fixed cost (waits, arming,
            // bookkeeping) set the step of 64-token tiles (MoE 86 -> 81 us).
            // Stage n + 1 is freed by the MMAs of a step before n, so waiting
            // for both before arming either cannot stall the issuer.
            for (int s = 0; s < 4; s += 2) {
              const int st1 = (st + 1 == a.k_stages) ? 0 : st + 1;
              const uint32_t ph1 = (st + 1 == a.k_stages) ? (ph ^ 1) : ph;
              if (!mbar_wait(&k_empty[st], ph ^ 1, abort, a.err) || !mbar_wait(&k_empty[st1], ph1 ^ 1, abort, a.err))
                break;
              mbar_expect_tx(&k_full[st], expect);
              mbar_expect_tx(&k_full[st1], expect);
              for (int j = 0; j < nbox; ++j) {
                tma_load_2d(sB + st * a.b_stage_bytes + j * GM_BBOX_BYTES, &tmX, &k_full[st], kb * QK_K + s * GM_BK,
                            xrow + j * GM_BBOX);
                tma_load_2d(sB + st1 * a.b_stage_bytes + j * GM_BBOX_BYTES, &tmX, &k_full[st1],
                            kb * QK_K + (s + 1) * GM_BK, xrow + j * GM_BBOX);
              }
              st = (st1 + 1 == a.k_stages) ? 0 : st1 + 1;
              ph = (st1 + 1 == a.k_stages) ? (ph1 ^ 1) : ph1;
            }
            continue;
          }
          for (int s = 0; s < 4; ++s) {  // pairs: one K step per round
            if (!mbar_wait(&k_empty[st], ph ^ 1, abort, a.err)) break;
            const uint32_t full_cl = mapa_shared(&k_full[st], 0);
            if (rank == 0) mbar_expect_tx(&k_full[st], expect);
            for (int j = 0; j < nbox; ++j)
              tma_load_2d_pair(sB + st * a.b_stage_bytes + j * GM_BBOX_BYTES, &tmX, full_cl, kb * QK_K + s * GM_BK,
                               xrow + j * GM_BBOX);
            if (++st == a.k_stages) {
              st = 0;
              ph ^= 1;
            }
          }
        }
      }
      // A pair's MMA commits arrive on this CTA's k_empty from the other SM:
      // wait until every stage filled here has been released, so that none is
      // still in flight when the CTA exits.
      if (PAIR && !*abort) {
        for (int i = 0; i < a.k_stages; ++i) {
          if (!mbar_wait_bounded(&k_empty[st], ph ^ 1)) break;
          if (++st == a.k_stages) {
            st = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else if (warp == GM_MMA_WARP && PAIR && rank != 0) {
    // The odd CTA of a pair issues no MMAs: this warp only follows the tile ring.
    int qi = 0;
    uint32_t qph = 0;
    for (;;) {
      const int t = tq_pop(tq_full, tq_empty, tq_ids, qi, qph, false, abort, a.err);
      if (t >= total_tiles || *abort) break;
    }
  } else if (warp == GM_MMA_WARP) {
    // ---- tensor-core issuer --------------------------------------------------
    // The whole warp runs the loop converged, so descriptors and counters stay
    // warp-uniform; one elected lane issues the MMAs and commits.
    int kst = 0, qi = 0;
    uint32_t kph = 0, qph = 0;
    const uint32_t a_tmem0 = tmem_base + a.a_col0;
    const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB));
    int it = 0;
    for (;; ++it) {
      const int t = tq_pop(tq_full, tq_empty, tq_ids, qi, qph, false, abort, a.err);
      if (t >= total_tiles || *abort) break;
      const Tile T = decode_tile<MOE, PAIR>(a, t, rank, s_tile_start, s_counts, s_offsets);
      const int acc = (a.n_acc == 2) ? (it & 1) : 0;
      const uint32_t acc_ph = (a.n_acc == 2) ? ((it >> 1) & 1) : (it & 1);
      if (!mbar_wait(&acc_empty[acc], acc_ph ^ 1, abort, a.err)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * a.acc_cols;
      // a pair always multiplies the full bn rows of B (each CTA holds bn / 2)
      const uint32_t idesc =
          PAIR ? idesc_f16_f32(2 * GM_BM, a.bn) : idesc_f16_f32(GM_BM, (T.ncols + 15) & ~15);
      const int nsteps = (T.kb1 - T.kb0) * 4;
      bool ok = true;
      for (int ks = 0; ks < nsteps; ++ks) {
        if (!mbar_wait(&k_full[kst], kph, abort, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // B: the start address field advances by bytes / 16; A: 8 columns per K=16
        const uint32_t at = a_tmem0 + kst * GM_A_COLS;
        const uint64_t bd = b_desc0 + static_cast<uint64_t>((kst * a.b_stage_bytes) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < GM_BK / 16; ++k) {  // +32 bytes per K=16 step inside the 128-byte row
            if (PAIR)
              umma_f16_ta_pair(d_tmem, at + 8 * k, bd + 2 * k, idesc, (ks == 0 && k == 0) ? 0u : 1u);
            else
              umma_f16_ta(d_tmem, at + 8 * k, bd + 2 * k, idesc, (ks == 0 && k == 0) ? 0u : 1u);
          }
          if (PAIR)
            umma_commit_pair(&k_empty[kst], 0x3);
          else
            umma_commit(&k_empty[kst]);
        }
        __syncwarp();
        if (++kst == a.k_stages) {
          kst = 0;
          kph ^= 1;
        }
      }
      if (elect_one()) {
        if (PAIR)
          umma_commit_pair(&acc_full[acc], 0x3);
        else
          umma_commit(&acc_full[acc]);
      }
      __syncwarp();
      if (!ok) break;
    }
    // A pair: the other CTA's epilogue arrives on acc_empty here; wait for the
    // releases of the last accumulators before the CTA exits.
    if (PAIR && !*abort) {
      for (int j = 0; j < a.n_acc; ++j, ++it) {
        const int acc = (a.n_acc == 2) ? (it & 1) : 0;
        const uint32_t acc_ph = (a.n_acc == 2) ? ((it >> 1) & 1) : (it & 1);
        if (!mbar_wait_bounded(&acc_empty[acc], acc_ph ^ 1)) break;
      }
    }
  } else if (warp < GM_DQ_WARPS) {
    // ---- weight unpackers ----------------------------------------------------
    // warp w owns tensor-memory lanes 32 (w % 4) .. +31 (rows of the tile) and
    // the half (w / 4) % 2 of each K step; the two groups of eight warps
    // (w / 8) take alternate steps of a super-block (Q4_K: steps 0, 2 and 1, 3;
    // Q6_K: the two steps of one half of the block, which share their loads)
    const int r = 32 * (warp & 3) + lane, hf = (warp >> 2) & 1, grp = warp >> 3;
    const uint32_t a_lane = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + a.a_col0;
    int rst = 0, ast = 0, qi = 0;
    uint32_t rph = 0, aph = 0, qph = 0;
    for (;;) {
      const int t = tq_pop(tq_full, tq_empty, tq_ids, qi, qph, false, abort, a.err);
      if (t >= total_tiles || *abort) break;
      const Tile T = decode_tile<MOE, PAIR>(a, t, rank, s_tile_start, s_counts, s_offsets);
      for (int kb = T.kb0; kb < T.kb1 && !*abort; ++kb) {
        if (!mbar_wait(&raw_full[rst], rph, abort, a.err)) break;
        const uint8_t* raw = sRaw + rst * RAW_BYTES;
        const int rem = (WT == KQ_Q6_K) ? ((kb * Q6K_BYTES) & 15) : 0;
        uint4 hdr = make_uint4(0u, 0u, 0u, 0u);
        Q6Half q6;
        for (int s = 0; s < 4; ++s) {
          const bool mine = (WT != KQ_Q6_K) ? ((s & 1) == grp) : ((s >> 1) == grp);
          if (mine) {
            if (!mbar_wait(&k_empty[ast], aph ^ 1, abort, a.err)) break;
            tc_fence_after();
            uint32_t lo[8], hi[8];
            if (WT == KQ_Q4_K) {
              if (s < 2) hdr = *reinterpret_cast<const uint4*>(raw + r * Q4K_BYTES);
              dequant_q4k(hdr, raw, s, r, hf, lo, hi);
            } else if (WT == KQ_Q5_K) {
              if (s < 2) hdr = *reinterpret_cast<const uint4*>(raw + r * Q5K_BYTES);
              dequant_q5k(hdr, raw, s, r, hf, lo, hi);
            } else {
              if ((s & 1) == 0) load_q6k_half(raw, rem, s >> 1, r, hf, q6);
              dequant_q6k(raw, rem, q6, s, r, hf, lo, hi);
            }
            const uint32_t col = a_lane + ast * GM_A_COLS + 8 * hf;
            tmem_st_32x32b_x8(col, lo);
            tmem_st_32x32b_x8(col + 16, hi);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (PAIR)
                mbar_arrive_cluster(mapa_shared(&k_full[ast], 0));
              else
                mbar_arrive(&k_full[ast]);
            }
          }
          if (++ast == a.k_stages) {
            ast = 0;
            aph ^= 1;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rst]);
        if (++rst == a.raw_stages) {
          rst = 0;
          rph ^= 1;
        }
      }
    }
  } else {
    // ---- epilogue: tensor memory -> fp32 Y -----------------------------------
    if (!MOE) asm volatile("griddepcontrol.wait;" ::: "memory");  // Y may still be read by the previous kernel
    const int wq = warp - GM_EPI_WARP0;  // == warp % 4: this warp's 32 TMEM lanes
    int qi = 0;
    uint32_t qph = 0;
    for (int it = 0;; ++it) {
      const int t = tq_pop(tq_full, tq_empty, tq_ids, qi, qph, false, abort, a.err);
      if (t >= total_tiles || *abort) break;
      const Tile T = decode_tile<MOE, PAIR>(a, t, rank, s_tile_start, s_counts, s_offsets);
      const int acc = (a.n_acc == 2) ? (it & 1) : 0;
      const uint32_t acc_ph = (a.n_acc == 2) ? ((it >> 1) & 1) : (it & 1);
      if (!mbar_wait(&acc_full[acc], acc_ph, abort, a.err)) break;
      tc_fence_after();
      const int m = T.m0 + 32 * wq + lane;
      const bool mok = m < a.M;
      for (int c0 = 0; c0 < T.ncols; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + acc * a.acc_cols + (static_cast<uint32_t>(32 * wq) << 16) + c0, r);
        tmem_ld_wait();
        if (MOE) {
          const int my_slot = (c0 + lane < T.ncols) ? __ldg(a.entries + T.nbase + c0 + lane) : 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int slot = __shfl_sync(0xffffffffu, my_slot, j);
            if (c0 + j < T.ncols && mok) a.Y[static_cast<int64_t>(slot) * a.M + m] = __uint_as_float(r[j]);
          }
        } else {
          float* out = (a.splits == 1)
                           ? a.Y + static_cast<int64_t>(T.xrow0) * a.M
                           : a.partial + (static_cast<int64_t>(T.split) * a.N + T.xrow0) * a.M;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < T.ncols && mok) out[static_cast<int64_t>(c0 + j) * a.M + m] = __uint_as_float(r[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(mapa_shared(&acc_empty[acc], 0));
        else
          mbar_arrive(&acc_empty[acc]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA of the pair frees its memory while the other may still use it
  if (warp == GM_MMA_WARP) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, GM_TMEM_COLS);
    else
      tmem_dealloc(tmem_base, GM_TMEM_COLS);
  }
}

// Fixed-order sum of the split-K partials: Y[i] = Sum_s P[s][i] (n elements).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ P, float* __restrict__ Y,
                                                            int64_t n, int splits) {
  pdl_enter();
  const int64_t i4 = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) * 4;
  if (i4 >= n) return;
  if (i4 + 4 <= n && (n & 3) == 0) {
    float4 acc = __ldg(reinterpret_cast<const float4*>(P + i4));
    for (int s = 1; s < splits; ++s) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(P + static_cast<int64_t>(s) * n + i4));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<float4*>(Y + i4) = acc;
  } else {
    for (int64_t i = i4; i < n && i < i4 + 4; ++i) {
      float acc = __ldg(P + i);
      for (int s = 1; s < splits; ++s) acc += __ldg(P + static_cast<int64_t>(s) * n + i);
      Y[i] = acc;
    }
  }
}

// ---------------------------------------------------------------------------
// MoE routing ("Prefill Gap Closure Plan", T2 step 1; "ZINC MMQ v2", MoE
// routing): histogram of expert ids -> exclusive prefix sum -> a bucket
// position for every (token, slot) id. One CTA, shared-memory atomics; the
// positions are written in slot order (coalesced) and the gather kernel that
// follows scatters the rows and the slot ids. The order of slots inside a
// bucket depends on the atomics, but no result does: a slot's output row is
// the same dot products wherever it sits in its expert's tile. Also lays out
// the tile list: expert e owns m_tiles * ceil(count_e / bn) consecutive tiles
// starting at tile_start[e].
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_excl_scan_1024(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? wsum[warp - 1] : 0);
  *total = wsum[31];
  __syncthreads();
  return excl;
}

constexpr int ROUTE_IDS_PER_THREAD = 16;  // ids held in registers between the two passes

__global__ void __launch_bounds__(1024) moe_route_kernel(const int* __restrict__ ids, int n, int top_k, int E,
                                                         int m_tiles, int bn, int* counts, int* offsets,
                                                         int* tile_start, int* tile_queue, int* slot_pos, float* Y,
                                                         int M, int* err) {
  extern __shared__ int rsm[];
  int* cnt = rsm;        // [E]: histogram, then the scatter cursor of each bucket
  int* wsum = cnt + E;   // [32]
  pdl_enter();
  for (int i = threadIdx.x; i < E; i += 1024) cnt[i] = 0;
  __syncthreads();
  // pass 1: histogram (ids beyond 16 per thread are re-read in pass 2)
  int e_reg[ROUTE_IDS_PER_THREAD];
#pragma unroll
  for (int j = 0; j < ROUTE_IDS_PER_THREAD; ++j) {
    const int i = threadIdx.x + 1024 * j;
    e_reg[j] = (i < n) ? __ldg(ids + i) : -1;
  }
  for (int i0 = 0; i0 < n; i0 += 1024 * ROUTE_IDS_PER_THREAD) {
#pragma unroll
    for (int j = 0; j < ROUTE_IDS_PER_THREAD; ++j) {
      const int i = i0 + threadIdx.x + 1024 * j;
      if (i >= n) continue;
      const int e = (i0 == 0) ? e_reg[j] : __ldg(ids + i);
      if (e < 0 || e >= E)
        report_error(err, ERR_EXPERT_ID);
      else
        atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  const int tot = threadIdx.x < E ? cnt[threadIdx.x] : 0;
  int n_valid, n_tiles;
  const int off = block_excl_scan_1024(tot, wsum, &n_valid);
  const int my_tiles = threadIdx.x < E ? m_tiles * ((tot + bn - 1) / bn) : 0;
  const int toff = block_excl_scan_1024(my_tiles, wsum, &n_tiles);
  if (threadIdx.x < E) {
    counts[threadIdx.x] = tot;
    offsets[threadIdx.x] = off;
    tile_start[threadIdx.x] = toff;
    cnt[threadIdx.x] = off;  // scatter cursor
  }
  if (threadIdx.x == 0) {
    offsets[E] = n_valid;
    tile_start[E] = n_tiles;
    *tile_queue = 0;  // the grouped GEMM's atomic tile queue starts empty
  }
  __syncthreads();
  // pass 2: bucket positions (-1 for an invalid id, whose output row is zeroed)
  for (int i0 = 0; i0 < n; i0 += 1024 * ROUTE_IDS_PER_THREAD) {
#pragma unroll
    for (int j = 0; j < ROUTE_IDS_PER_THREAD; ++j) {
      const int i = i0 + threadIdx.x + 1024 * j;
      if (i >= n) continue;
      const int e = (i0 == 0) ? e_reg[j] : __ldg(ids + i);
      if (e < 0 || e >= E) {
        slot_pos[i] = -1;
        for (int m = 0; m < M; ++m) Y[static_cast<int64_t>(i) * M + m] = 0.f;
        continue;
      }
      slot_pos[i] = atomicAdd(&cnt[e], 1);
    }
  }
  (void)top_k;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static inline int64_t round_up64(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

bool encode_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return false;
    fn = reinterpret_cast<EncodeFn>(p);
  }
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int raw_box_bytes(int wtype) {
  return wtype == KQ_Q4_K ? RawBox<KQ_Q4_K>::BYTES : wtype == KQ_Q5_K ? RawBox<KQ_Q5_K>::BYTES : RawBox<KQ_Q6_K>::BYTES;
}

// Shared-memory attribute slots of the GEMM instantiations.
constexpr int gemm_slot(int wt, bool moe) { return wt == KQ_Q5_K ? (moe ? 3 : 2) : 2 + 2 * wt + (moe ? 1 : 0); }
constexpr int pair_slot(int wt) { return wt == KQ_Q5_K ? 15 : 11 + wt; }

// Tensor memory: the accumulators (two when that leaves room for four A stages,
// so the epilogue of one tile overlaps the next tile's MMAs), then up to eight
// 64-K A stages of 32 columns. Shared memory: the x_hat (B) ring, whose L2 ->
// shared memory round trip (1-2k cycles) the stages in flight must cover, and
// the raw weight ring (each super-block feeds four K steps; they come from HBM).
static bool choose_stages(int wtype, int bn, int n_experts, bool pair, GemmArgs* a, size_t* smem) {
  const int acc_cols = (bn + 15) & ~15;
  a->n_acc = (2 * acc_cols + 4 * GM_A_COLS <= GM_TMEM_COLS) ? 2 : 1;
  a->acc_cols = acc_cols;
  a->a_col0 = a->n_acc * acc_cols;
  const int a_max = std::min(GM_A_MAX_STAGES, (GM_TMEM_COLS - a->a_col0) / GM_A_COLS);
  if (a_max < 2) return false;
  // a CTA of a pair holds half of the bn x_hat rows of a stage
  const int b_bytes = (pair ? bn / (2 * GM_BBOX) : (bn + GM_BBOX - 1) / GM_BBOX) * GM_BBOX_BYTES;
  const int raw_bytes = raw_box_bytes(wtype) * GM_BM;
  const int tables = (n_experts > 0 ? 3 * (n_experts + 1) * 4 : 0) + 64 + GM_TQ * 20;
  const int budget = GM_SMEM_LIMIT - (1024 + tables + 512);
  auto bytes = [&](int bs, int rs) { return bs * b_bytes + rs * raw_bytes; };
  // The B ring gets priority: an x_hat stage takes ~1.4k cycles from issue to
  // arrival under load while the MMAs consume one every ~560 cycles (N = 256),
  // so about five must be in flight; two raw stages already cover eight K steps.
  int bs = 2, rs = 2;
  if (bytes(bs, rs) > budget) return false;
  while (bs < a_max && bytes(bs + 1, rs) <= budget) ++bs;
  while (rs < 4 && bytes(bs, rs + 1) <= budget) ++rs;
  a->k_stages = bs;
  a->raw_stages = rs;
  a->b_stage_bytes = b_bytes;
  *smem = static_cast<size_t>(bytes(bs, rs) + 1024 + tables + 512);
  return true;
}

// CTA pairs need bn = 128 or 256 (two whole 64-row x_hat boxes per half or
// one) and an even number of 128-row tiles (no pair half lies wholly past M).
GemmPlan plan_gemm(int wtype, int64_t M, int64_t K, int64_t N, int num_sms) {
  (void)wtype;
  GemmPlan p{};
  p.bn = static_cast<int>(N >= GM_BNMAX ? GM_BNMAX : round_up64(N, GM_BBOX));
  p.m_tiles = static_cast<int>((M + GM_BM - 1) / GM_BM);
  p.n_tiles = static_cast<int>((N + p.bn - 1) / p.bn);
  p.pair = (p.bn == 128 || p.bn == 256) && p.m_tiles % 2 == 0 && num_sms >= 2;
  const int nb = static_cast<int>(K / QK_K);
  const int slots = p.pair ? num_sms / 2 : num_sms;
  const int tiles = (p.pair ? p.m_tiles / 2 : p.m_tiles) * p.n_tiles;
  int splits = 1;
  if (tiles < slots) {
    splits = slots / tiles;
    if (splits > nb) splits = nb;
    if (splits > 16) splits = 16;
    if (splits < 1) splits = 1;
  }
  p.splits = splits;
  const int64_t units = static_cast<int64_t>(p.m_tiles) * p.n_tiles * splits;
  p.grid = static_cast<int>(units < num_sms ? units : num_sms);
  p.num_sms = num_sms;
  p.xhat_bytes = static_cast<size_t>(round_up64(N * K * 2, 1024));
  p.partial_bytes = splits > 1 ? static_cast<size_t>(round_up64(static_cast<int64_t>(splits) * N * M * 4, 1024)) : 0;
  p.total_bytes = p.xhat_bytes + p.partial_bytes;
  return p;
}

template <int WT, bool MOE>
static cudaError_t launch_kernel(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a, int grid,
                                 size_t smem, cudaStream_t s) {
  cudaError_t e =
      allow_max_smem(reinterpret_cast<const void*>(kq_gemm_kernel<WT, MOE, false>), gemm_slot(WT, MOE));
  if (e != cudaSuccess) return e;
  return launch_pdl(kq_gemm_kernel<WT, MOE, false>, dim3(grid), dim3(GM_THREADS), smem, s, tmW, tmX, a);
}

// Clusters of two CTAs (one per SM) that can be resident at once on the
// current device, looked up once per device and weight type; 0 when pairs
// cannot run.
template <int WT>
static int pair_clusters(cudaLaunchConfig_t cfg) {
  static std::mutex mu;
  static int cached[3][64];
  static bool known[3][64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  const int w = WT == KQ_Q4_K ? 0 : WT == KQ_Q5_K ? 1 : 2;
  if (!known[w][dev]) {
    int n = 0;
    cfg.gridDim = dim3(2);
    if (cudaOccupancyMaxActiveClusters(&n, kq_gemm_kernel<WT, false, true>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    cached[w][dev] = n;
    known[w][dev] = true;
  }
  return cached[w][dev];
}

// Launches the paired dense kernel over `units` pair tiles; *launched = false
// (and nothing queued) when the device cannot run CTA pairs.
template <int WT>
static cudaError_t launch_pair(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a, int units,
                               size_t smem, cudaStream_t s, bool* launched) {
  *launched = false;
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(kq_gemm_kernel<WT, false, true>), pair_slot(WT));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(GM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const int clusters = pair_clusters<WT>(cfg);
  if (clusters < 1) return cudaSuccess;
  cfg.gridDim = dim3(2 * std::min(units, clusters));
  *launched = true;
  return cudaLaunchKernelEx(&cfg, kq_gemm_kernel<WT, false, true>, tmW, tmX, a);
}

static cudaError_t dispatch(int wtype, bool moe, const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                            int grid, size_t smem, cudaStream_t s) {
  if (wtype == KQ_Q4_K)
    return moe ? launch_kernel<KQ_Q4_K, true>(tmW, tmX, a, grid, smem, s)
               : launch_kernel<KQ_Q4_K, false>(tmW, tmX, a, grid, smem, s);
  if (wtype == KQ_Q5_K)
    return moe ? launch_kernel<KQ_Q5_K, true>(tmW, tmX, a, grid, smem, s)
               : launch_kernel<KQ_Q5_K, false>(tmW, tmX, a, grid, smem, s);
  return moe ? launch_kernel<KQ_Q6_K, true>(tmW, tmX, a, grid, smem, s)
             : launch_kernel<KQ_Q6_K, false>(tmW, tmX, a, grid, smem, s);
}

static bool weight_tmap(CUtensorMap* tm, int wtype, const void* W, int64_t rows, int64_t K) {
  const int64_t rs = (K / QK_K) * (wtype == KQ_Q4_K ? Q4K_BYTES : wtype == KQ_Q5_K ? Q5K_BYTES : Q6K_BYTES);
  return encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, static_cast<uint64_t>(rs), static_cast<uint64_t>(rows),
                        static_cast<uint64_t>(rs), static_cast<uint32_t>(raw_box_bytes(wtype)), GM_BM,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

static bool xhat_tmap(CUtensorMap* tm, const void* Xh, int64_t rows, int64_t K) {
  return encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xh, static_cast<uint64_t>(K),
                        static_cast<uint64_t>(rows), static_cast<uint64_t>(K * 2), GM_BK, GM_BBOX,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_gemm(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K, int64_t N,
                        void* ws, const GemmPlan& plan, int* err, cudaStream_t s, int* status) {
  *status = KQ_OK;
  // A few tokens are a decode, not a GEMM: the tensor-core tiles would be
  // nearly empty, so Q4_K and Q5_K run on the matvec path, which streams the
  // weights once and multiplies each staged block with every token.
  if ((wtype == KQ_Q4_K || wtype == KQ_Q5_K) && N <= LR_TOKENS_MAX) {
    bool handled = false;
    cudaError_t e = launch_matvec_tokens(wtype, W, X, Y, M, K, N, ws, plan.xhat_bytes, err, plan.num_sms, s, &handled);
    if (e != cudaSuccess || handled) return e;
  }
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  __half* xh = reinterpret_cast<__half*>(wsb);
  float* partial = reinterpret_cast<float*>(wsb + plan.xhat_bytes);
  cudaError_t e = launch_quantize_xhat(X, xh, K, N, plan.grid, s);
  if (e != cudaSuccess) return e;
  CUtensorMap tmW, tmX;
  if (!weight_tmap(&tmW, wtype, W, M, K) || !xhat_tmap(&tmX, xh, N, K)) {
    *status = KQ_ERR_CUDA;
    return cudaSuccess;
  }
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.nb = static_cast<int>(K / QK_K);
  a.n_tiles = plan.n_tiles;
  a.splits = plan.splits;
  a.bn = plan.bn;
  a.Y = Y;
  a.partial = partial;
  a.n_experts = 0;
  a.err = err;
  a.hold = test_hold_copies();
  bool launched = false;
  if (plan.pair) {
    GemmArgs ap = a;
    ap.m_tiles = plan.m_tiles / 2;
    size_t smem = 0;
    if (choose_stages(wtype, plan.bn, 0, true, &ap, &smem)) {
      const int units = ap.m_tiles * plan.n_tiles * plan.splits;
      e = wtype == KQ_Q4_K   ? launch_pair<KQ_Q4_K>(tmW, tmX, ap, units, smem, s, &launched)
          : wtype == KQ_Q5_K ? launch_pair<KQ_Q5_K>(tmW, tmX, ap, units, smem, s, &launched)
                             : launch_pair<KQ_Q6_K>(tmW, tmX, ap, units, smem, s, &launched);
      if (e != cudaSuccess) return e;
    }
  }
  if (!launched) {
    a.m_tiles = plan.m_tiles;
    size_t smem = 0;
    if (!choose_stages(wtype, plan.bn, 0, false, &a, &smem)) {
      *status = KQ_ERR_SHAPE;
      return cudaSuccess;
    }
    e = dispatch(wtype, false, tmW, tmX, a, plan.grid, smem, s);
    if (e != cudaSuccess) return e;
  }
  if (plan.splits > 1) {
    const int64_t n = N * M;
    const int64_t threads = (n + 3) / 4;
    e = launch_pdl(splitk_reduce_kernel, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0, s,
                   partial, Y, n, plan.splits);
  }
  return e;
}

// MoE workspace: counts[E] | offsets[E+1] | tile_start[E+1] | tile queue counter | entries[n] (slot of each bucket row) |
// slot_pos[n] (bucket row of each slot) | x_hat[n][K] fp16 (bucket order)
MoePlan plan_moe(int wtype, int64_t M, int64_t K, int64_t T, int n_experts, int top_k) {
  (void)wtype;
  MoePlan p{};
  const int64_t n = T * top_k;
  p.m_tiles = static_cast<int>((M + GM_BM - 1) / GM_BM);
  size_t o = 0;
  p.off_counts = o;
  o += round_up64(4 * n_experts, 256);
  p.off_offsets = o;
  o += round_up64(4 * (n_experts + 1), 256);
  p.off_tiles = o;
  o += round_up64(4 * (n_experts + 1), 256);
  p.off_queue = o;
  o += 256;
  p.off_entries = o;
  o += round_up64(4 * n, 256);
  p.off_src = o;
  o += round_up64(4 * n, 1024);
  p.off_xhat = o;
  o += round_up64(n * K * 2, 1024);
  p.total_bytes = o;
  return p;
}

constexpr int MOE_BN = 128;  // tokens per MoE tile (one tile covers a typical expert bucket)

cudaError_t launch_moe(int wtype, const void* W, int n_experts, const int32_t* ids, int top_k, const float* X,
                       float* Y, int64_t M, int64_t K, int64_t T, void* ws, const MoePlan& plan, int* err,
                       int num_sms, cudaStream_t s, int* status) {
  *status = KQ_OK;
  if (n_experts > MOE_MAX_EXPERTS) {
    *status = KQ_ERR_SHAPE;
    return cudaSuccess;
  }
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int* counts = reinterpret_cast<int*>(wsb + plan.off_counts);
  int* offsets = reinterpret_cast<int*>(wsb + plan.off_offsets);
  int* tile_start = reinterpret_cast<int*>(wsb + plan.off_tiles);
  int* tile_queue = reinterpret_cast<int*>(wsb + plan.off_queue);
  int* entries = reinterpret_cast<int*>(wsb + plan.off_entries);
  int* slot_pos = reinterpret_cast<int*>(wsb + plan.off_src);
  __half* xh = reinterpret_cast<__half*>(wsb + plan.off_xhat);
  const int64_t n = T * top_k;

  // Routing first (bucket tables, the bucket row of every slot); then each
  // token's x_hat row is made once and written to all of its bucket rows.
  const size_t rsmem = static_cast<size_t>(n_experts + 32) * sizeof(int);
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(moe_route_kernel), 8);
  if (e != cudaSuccess) return e;
  e = launch_pdl(moe_route_kernel, dim3(1), dim3(1024), rsmem, s, ids, static_cast<int>(n), top_k, n_experts,
                 plan.m_tiles, MOE_BN, counts, offsets, tile_start, tile_queue, slot_pos, Y, static_cast<int>(M),
                 err);
  if (e != cudaSuccess) return e;
  e = launch_quantize_scatter(X, xh, K, T, top_k, slot_pos, entries, s);
  if (e != cudaSuccess) return e;

  CUtensorMap tmW, tmX;
  if (!weight_tmap(&tmW, wtype, W, static_cast<int64_t>(n_experts) * M, K) || !xhat_tmap(&tmX, xh, n, K)) {
    *status = KQ_ERR_CUDA;
    return cudaSuccess;
  }
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(n);
  a.nb = static_cast<int>(K / QK_K);
  a.m_tiles = plan.m_tiles;
  a.n_tiles = 0;
  a.splits = 1;
  a.bn = MOE_BN;
  a.Y = Y;
  a.partial = nullptr;
  a.n_experts = n_experts;
  a.counts = counts;
  a.offsets = offsets;
  a.tile_start = tile_start;
  a.entries = entries;
  a.tile_queue = tile_queue;
  a.err = err;
  a.hold = test_hold_copies();
  size_t smem = 0;
  if (!choose_stages(wtype, MOE_BN, n_experts, false, &a, &smem)) {
    *status = KQ_ERR_SHAPE;
    return cudaSuccess;
  }
  return dispatch(wtype, true, tmW, tmX, a, num_sms, smem, s);
}

}  // namespace kq
