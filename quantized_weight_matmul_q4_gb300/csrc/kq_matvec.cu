// Decode matvec y[M] = dequant(W)[M,K] . x[K] for Q4_K and Q6_K weights, with
// the fp32 -> Q8_1 quantisation of x fused in.
//
// Method: "06 · 8e/8e② — decode MMVQ: dp4a integer dot products + the
// llama.cpp launch table", §2 Principle and §3.2 Key code: per 32-weight
// sub-block an exact integer dot of the 4-bit codes with the int8 activation
// codes (dp4a), the min term taken from the activation block sum
// (W.x = Sum_sub [d*sc*d8*Sum(nib*q) - dmin*m*d8*Sum(q)]), and a warp-shuffle
// reduction per row. The page's launch geometry (one 256-thread block per row,
// plain loads) was made for a 273 GB/s LPDDR part; here the rows of the
// row-major matrix are contiguous, so each CTA owns a balanced contiguous range
// of rows and streams it through a shared-memory ring with 1-D bulk copies
// (one elected producer thread, mbarrier completion). Every byte of W is read
// from HBM once, in large coalesced transfers, with up to ~200 KB per SM in
// flight; the consumer warps quantise x into shared memory while the first
// copies land, then each warp reduces one row (or a share of one row).
#include "kq_internal.h"
#include "kq_quant.cuh"

namespace kq {

constexpr int MV_CWARPS = 16;                       // consumer warps
constexpr int MV_THREADS = (MV_CWARPS + 1) * 32;    // + one producer warp
constexpr int MV_SMEM_LIMIT = 227 * 1024;
constexpr int MV_STAGE_LIMIT = 100 * 1024;          // largest ring stage (two must fit)

struct MatvecParams {
  const uint8_t* W;
  const float* x;
  float* y;
  int M, K, nb;
  int rs;               // bytes per weight row
  int unit_rows;        // CTA row ranges start at multiples of this (16-byte aligned copies)
  int n_units;          // ceil(M / unit_rows)
  int stage_rows;       // rows per ring stage
  int warps_per_row;    // MV_CWARPS / stage_rows
  int n_ring;           // ring depth (stages)
  int stage_bytes;      // bytes per ring slot (multiple of 128)
  int xq_bytes;         // bytes reserved for the int8 activation codes
  int xds_bytes;        // bytes reserved for the per-32 (d8, d8*Sum q) pairs
  int* err;
};

// Position of activation k inside the shared int8 buffer. For Q4_K the four
// 16-byte pieces of every 64-element group (block b, chunk c) are permuted by
// h = 2(b&1) + (c>>1) so that the eight lanes of a 128-bit load phase, which
// read (two blocks) x (four chunks) at the same piece, hit distinct banks.
template <int WT>
__device__ __forceinline__ int xq_offset(int k) {
  if (WT == KQ_Q4_K) {
    const int b = k >> 8, c = (k >> 6) & 3, v = (k >> 4) & 3;
    const int h = ((b & 1) << 1) | (c >> 1);
    return (b << 8) | (c << 6) | ((v ^ h) << 4) | (k & 15);
  }
  return k;
}

// One lane's share of a Q4_K row: units (block, 32-byte chunk c) with
// u = first, first + stride, ... Chunk c of a block holds sub-block 2c in its
// low nibbles and sub-block 2c+1 in its high nibbles.
__device__ __forceinline__ float row_dot_q4k(const uint8_t* __restrict__ rowp, const uint8_t* __restrict__ xq,
                                             const float2* __restrict__ xds, int n_units, int first, int stride) {
  float acc = 0.f;
  const int c = first & 3;  // stride is a multiple of 4, so c is fixed per lane
  const int sh = (c & 1) * 16;
  for (int u = first; u < n_units; u += stride) {
    const int b = u >> 2;
    const uint8_t* blk = rowp + b * Q4K_BYTES;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
    const int h = ((b & 1) << 1) | (c >> 1);
    const uint8_t* xb = xq + (b << 8) + (c << 6);
    const int4 x0 = *reinterpret_cast<const int4*>(xb + ((0 ^ h) << 4));
    const int4 x1 = *reinterpret_cast<const int4*>(xb + ((1 ^ h) << 4));
    const int4 x2 = *reinterpret_cast<const int4*>(xb + ((2 ^ h) << 4));
    const int4 x3 = *reinterpret_cast<const int4*>(xb + ((3 ^ h) << 4));
    const float4 ds = *reinterpret_cast<const float4*>(xds + 8 * b + 2 * c);  // d8A, sA, d8B, sB

    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
    // 6-bit scales/mins of sub-blocks 0..3 (c < 2) or 4..7 (c >= 2), one per byte.
    uint32_t scw, mw;
    if (c < 2) {
      scw = hdr.y & 0x3F3F3F3Fu;
      mw = hdr.z & 0x3F3F3F3Fu;
    } else {
      scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
      mw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    }
    const float scA = static_cast<float>((scw >> sh) & 0xFFu);
    const float scB = static_cast<float>((scw >> (sh + 8)) & 0xFFu);
    const float mA = static_cast<float>((mw >> sh) & 0xFFu);
    const float mB = static_cast<float>((mw >> (sh + 8)) & 0xFFu);

    int dA = 0, dB = 0;
    dA = __dp4a(static_cast<int>(qa.x & 0x0F0F0F0Fu), x0.x, dA);
    dA = __dp4a(static_cast<int>(qa.y & 0x0F0F0F0Fu), x0.y, dA);
    dA = __dp4a(static_cast<int>(qa.z & 0x0F0F0F0Fu), x0.z, dA);
    dA = __dp4a(static_cast<int>(qa.w & 0x0F0F0F0Fu), x0.w, dA);
    dA = __dp4a(static_cast<int>(qb.x & 0x0F0F0F0Fu), x1.x, dA);
    dA = __dp4a(static_cast<int>(qb.y & 0x0F0F0F0Fu), x1.y, dA);
    dA = __dp4a(static_cast<int>(qb.z & 0x0F0F0F0Fu), x1.z, dA);
    dA = __dp4a(static_cast<int>(qb.w & 0x0F0F0F0Fu), x1.w, dA);
    dB = __dp4a(static_cast<int>((qa.x >> 4) & 0x0F0F0F0Fu), x2.x, dB);
    dB = __dp4a(static_cast<int>((qa.y >> 4) & 0x0F0F0F0Fu), x2.y, dB);
    dB = __dp4a(static_cast<int>((qa.z >> 4) & 0x0F0F0F0Fu), x2.z, dB);
    dB = __dp4a(static_cast<int>((qa.w >> 4) & 0x0F0F0F0Fu), x2.w, dB);
    dB = __dp4a(static_cast<int>((qb.x >> 4) & 0x0F0F0F0Fu), x3.x, dB);
    dB = __dp4a(static_cast<int>((qb.y >> 4) & 0x0F0F0F0Fu), x3.y, dB);
    dB = __dp4a(static_cast<int>((qb.z >> 4) & 0x0F0F0F0Fu), x3.z, dB);
    dB = __dp4a(static_cast<int>((qb.w >> 4) & 0x0F0F0F0Fu), x3.w, dB);

    acc = fmaf(ds.x * (d * scA), static_cast<float>(dA), acc);
    acc = fmaf(-(dmin * mA), ds.y, acc);
    acc = fmaf(ds.z * (d * scB), static_cast<float>(dB), acc);
    acc = fmaf(-(dmin * mB), ds.w, acc);
  }
  return acc;
}

__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) {  // 2-byte aligned 32-bit load
  const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
  return static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 16);
}

// One lane's share of a Q6_K row: units (block, half h, r-range of 8); unit
// covers weights 128h + 32g + r for g = 0..3 and r in [8*qr, 8*qr + 8).
__device__ __forceinline__ float row_dot_q6k(const uint8_t* __restrict__ rowp, const uint8_t* __restrict__ xq,
                                             const float2* __restrict__ xds, int n_units, int first, int stride) {
  float acc = 0.f;
  for (int u = first; u < n_units; u += stride) {
    const int b = u >> 3, h = (u >> 2) & 1, qr = u & 3;
    const uint8_t* blk = rowp + b * Q6K_BYTES;
    const uint8_t* pa = blk + 64 * h + 8 * qr;       // ql, quarters g = 0 (low) and 2 (high)
    const uint8_t* pb = pa + 32;                     // ql, quarters g = 1 (low) and 3 (high)
    const uint8_t* ph = blk + 128 + 32 * h + 8 * qr; // qh, two bits per quarter
    const uint32_t a0 = ld_u32_a2(pa), a1 = ld_u32_a2(pa + 4);
    const uint32_t b0 = ld_u32_a2(pb), b1 = ld_u32_a2(pb + 4);
    const uint32_t h0 = ld_u32_a2(ph), h1 = ld_u32_a2(ph + 4);
    const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk + 208)));
    const int8_t* sc = reinterpret_cast<const int8_t*>(blk + 192 + 8 * h + (qr >> 1));
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t s0 = (g & 1) ? b0 : a0, s1 = (g & 1) ? b1 : a1;
      const uint32_t l0 = (g < 2) ? (s0 & 0x0F0F0F0Fu) : ((s0 >> 4) & 0x0F0F0F0Fu);
      const uint32_t l1 = (g < 2) ? (s1 & 0x0F0F0F0Fu) : ((s1 >> 4) & 0x0F0F0F0Fu);
      const uint32_t q0 = l0 | (((h0 >> (2 * g)) & 0x03030303u) << 4);
      const uint32_t q1 = l1 | (((h1 >> (2 * g)) & 0x03030303u) << 4);
      const int k = (b << 8) + 128 * h + 32 * g + 8 * qr;
      const int2 xw = *reinterpret_cast<const int2*>(xq + k);
      int dot = dp4a_us(q0, xw.x, 0);
      dot = dp4a_us(q1, xw.y, dot);
      int sx = __dp4a(0x01010101, xw.x, 0);
      sx = __dp4a(0x01010101, xw.y, sx);
      const float d8 = xds[k >> 5].x;
      acc = fmaf(d * static_cast<float>(sc[2 * g]) * d8, static_cast<float>(dot - 32 * sx), acc);
    }
  }
  return acc;
}

template <int WT>
__global__ void __launch_bounds__(MV_THREADS, 1) matvec_kernel(const MatvecParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* xq = smem;
  float2* xds = reinterpret_cast<float2*>(smem + p.xq_bytes);
  uint8_t* ring = smem + p.xq_bytes + p.xds_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(p.n_ring) * p.stage_bytes);
  uint64_t* empty = full + p.n_ring;
  float* red = reinterpret_cast<float*>(empty + p.n_ring);  // [MV_CWARPS] partial row sums
  volatile int* abort = reinterpret_cast<volatile int*>(red + MV_CWARPS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * p.n_units / gridDim.x;
  const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * p.n_units / gridDim.x;
  const int r0 = static_cast<int>(u0 * p.unit_rows);
  const int r1 = static_cast<int>(min(static_cast<int64_t>(p.M), u1 * p.unit_rows));
  const int n_stages = (r1 - r0 + p.stage_rows - 1) / p.stage_rows;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_ring; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], MV_CWARPS);
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == MV_CWARPS) {
    // Producer: stream this CTA's rows, stage by stage, through the ring.
    if (lane == 0) {
      for (int s = 0; s < n_stages; ++s) {
        const int slot = s % p.n_ring;
        const uint32_t ph = (s / p.n_ring) & 1;
        if (!mbar_wait(&empty[slot], ph ^ 1, abort, p.err)) break;
        const int row_a = r0 + s * p.stage_rows;
        const int rows = min(p.stage_rows, r1 - row_a);
        const uint32_t bytes = static_cast<uint32_t>(rows) * p.rs;
        const uint32_t main_bytes = bytes & ~15u;
        const uint8_t* src = p.W + static_cast<int64_t>(row_a) * p.rs;
        uint8_t* dst = ring + static_cast<size_t>(slot) * p.stage_bytes;
        for (uint32_t i = main_bytes; i < bytes; ++i) dst[i] = src[i];  // ragged end of W (< 16 bytes)
        mbar_expect_tx(&full[slot], main_bytes);
        if (main_bytes) bulk_g2s(dst, src, main_bytes, &full[slot]);
      }
    }
    return;
  }

  // Consumers: quantise x to Q8_1 codes in shared memory while the first
  // stages are in flight.
  const int ctid = threadIdx.x;
  const int nq = p.K >> 2;
  for (int base = 0; base < nq; base += MV_CWARPS * 32) {
    const int qd = base + ctid;
    const bool v = qd < nq;
    float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (v) xv = __ldg(reinterpret_cast<const float4*>(p.x) + qd);
    const Q8Quad r = quantize_quad(xv);
    if (v) {
      const int k = qd << 2;
      *reinterpret_cast<uint32_t*>(xq + xq_offset<WT>(k)) = pack_q4(r.q);
      if ((qd & 7) == 0) xds[k >> 5] = make_float2(r.dh, __fmul_rn(r.dh, static_cast<float>(r.sumq)));
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(MV_CWARPS * 32) : "memory");

  const int wpr = p.warps_per_row;
  const int row_in_stage = warp / wpr, part = warp % wpr;
  const int units = (WT == KQ_Q4_K) ? p.nb * 4 : p.nb * 8;
  for (int s = 0; s < n_stages; ++s) {
    const int slot = s % p.n_ring;
    const uint32_t ph = (s / p.n_ring) & 1;
    if (!mbar_wait(&full[slot], ph, abort, p.err)) break;
    const int row = r0 + s * p.stage_rows + row_in_stage;
    float acc = 0.f;
    if (row < r1) {
      const uint8_t* rowp = ring + static_cast<size_t>(slot) * p.stage_bytes +
                            static_cast<size_t>(row_in_stage) * p.rs;
      if (WT == KQ_Q4_K)
        acc = row_dot_q4k(rowp, xq, xds, units, lane + 32 * part, 32 * wpr);
      else
        acc = row_dot_q6k(rowp, xq, xds, units, lane + 32 * part, 32 * wpr);
      acc = warp_sum_f(acc);
    }
    if (wpr == 1) {
      if (row < r1 && lane == 0) p.y[row] = acc;
    } else {
      if (lane == 0) red[warp] = acc;
      asm volatile("bar.sync 1, %0;" ::"r"(MV_CWARPS * 32) : "memory");
      if (part == 0 && lane == 0 && row < r1) {
        float t = red[warp];
        for (int i = 1; i < wpr; ++i) t += red[warp + i];
        p.y[row] = t;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(MV_CWARPS * 32) : "memory");
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
}

static inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

cudaError_t launch_matvec(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t K, int* err,
                          int num_sms, cudaStream_t s, int* status) {
  *status = KQ_OK;
  MatvecParams p{};
  p.W = static_cast<const uint8_t*>(W);
  p.x = x;
  p.y = y;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.nb = static_cast<int>(K / QK_K);
  p.rs = p.nb * (wtype == KQ_Q4_K ? Q4K_BYTES : Q6K_BYTES);
  p.unit_rows = (p.rs % 16 == 0) ? 1 : 8;
  p.err = err;
  int R = 0;
  for (int r = MV_CWARPS; r >= p.unit_rows && r >= 1; r >>= 1) {
    if (static_cast<int64_t>(r) * p.rs <= MV_STAGE_LIMIT) {
      R = r;
      break;
    }
  }
  if (R == 0) {
    *status = KQ_ERR_SHAPE;
    return cudaSuccess;
  }
  p.stage_rows = R;
  p.warps_per_row = MV_CWARPS / R;
  p.stage_bytes = round_up(R * p.rs, 128);
  p.xq_bytes = round_up(p.K, 128);
  p.xds_bytes = round_up((p.K / QK8_1) * 8, 128);
  const int fixed = p.xq_bytes + p.xds_bytes;
  const int tail = 0;
  int n_ring = (MV_SMEM_LIMIT - fixed - 1024 - tail) / (p.stage_bytes + 16);
  if (n_ring > 16) n_ring = 16;
  if (n_ring < 2) {
    *status = KQ_ERR_SHAPE;
    return cudaSuccess;
  }
  p.n_units = static_cast<int>((M + p.unit_rows - 1) / p.unit_rows);
  const int G = p.n_units < num_sms ? p.n_units : num_sms;
  // ring depth beyond what the largest CTA range needs buys nothing
  const int64_t max_rows = (static_cast<int64_t>(p.n_units + G - 1) / G) * p.unit_rows;
  const int need = static_cast<int>((max_rows + R - 1) / R);
  if (n_ring > need) n_ring = need < 2 ? 2 : need;
  p.n_ring = n_ring;
  const size_t smem = static_cast<size_t>(fixed) + static_cast<size_t>(n_ring) * p.stage_bytes +
                      2 * n_ring * sizeof(uint64_t) + MV_CWARPS * sizeof(float) + 16;
  cudaError_t e;
  if (wtype == KQ_Q4_K) {
    e = cudaFuncSetAttribute(matvec_kernel<KQ_Q4_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    matvec_kernel<KQ_Q4_K><<<G, MV_THREADS, smem, s>>>(p);
  } else {
    e = cudaFuncSetAttribute(matvec_kernel<KQ_Q6_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    matvec_kernel<KQ_Q6_K><<<G, MV_THREADS, smem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kq
