// Shared device helpers for the k-quant matmul kernels (sm_103a only).
//
// Inline-PTX wrappers for mbarriers, bulk/tensor copies (TMA) and the fifth
// generation tensor cores (tcgen05 + tensor memory), written from the PTX ISA
// description of those instructions. Also the block-format constants of
// Q4_K, Q6_K and Q8_1 as laid out by "06 · 8e/8e② — decode MMVQ" (§3.2 Key
// code, §3.3 Pitfalls).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "kq kernels target sm_103a (tcgen05, TMA); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace kq {

constexpr int QK_K = 256;          // weights per super-block
constexpr int Q4K_BYTES = 144;     // fp16 d, fp16 dmin, 12 B scales, 128 B nibbles
constexpr int Q6K_BYTES = 210;     // ql[128], qh[64], int8 scales[16], fp16 d @208
constexpr int Q5K_BYTES = 176;     // fp16 d, fp16 dmin, 12 B scales, qh[32] @16, 128 B nibbles @48
constexpr int QK8_1 = 32;          // activations per Q8_1 block
constexpr int Q8_1_BYTES = 36;     // fp16 d, fp16 s, int8 q[32]

// Device error codes (written to the library's error word; first one wins).
constexpr int ERR_WAIT_TIMEOUT = 1;     // a pipeline wait gave up
constexpr int ERR_EXPERT_ID = 2;        // an expert id outside [0, n_experts)

// A wait gives up after this long (ns of %globaltimer) and reports
// ERR_WAIT_TIMEOUT; a healthy pipeline waits microseconds.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: every kernel of the library is launched so
// that it may start while the previous kernel in the stream drains. It first
// lets its own dependents be scheduled, then waits until the previous grid has
// completed and its memory is visible, before touching any global memory.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// One lane of a converged warp (the same lane on every call) is elected.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void report_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// The waiting thread is suspended (it does not spin on the issue slots) until
// the phase completes or about 0.2 ms pass.
constexpr uint32_t WAIT_SUSPEND_HINT_NS = 200000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(WAIT_SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up after
// WAIT_LIMIT_NS, records ERR_WAIT_TIMEOUT, raises *abort and returns false.
// Also returns false at once when another thread of the CTA raised *abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        report_error(err, ERR_WAIT_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// Waits for the phase with the given parity, ignoring the abort flag (used to
// let copies already in flight land before a CTA exits). Returns false after
// WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7) == 0 && globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
}

// Waits until *counter > c, where the counter is a shared-memory word that one
// thread raises (the number of ring chunks a producer has issued). A consumer
// that waits for this before waiting on the chunk's slot barrier never takes
// an older phase of the same parity for its chunk, however far ahead of the
// other consumers it runs. Bounded like mbar_wait.
__device__ __forceinline__ bool wait_counter_above(const volatile int* counter, int c, volatile int* abort, int* err) {
  if (*counter > c) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (*counter > c) return true;
    if ((it & 7) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        report_error(err, ERR_WAIT_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Thread-block clusters (CTA pairs)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; orders earlier memory operations
// (including mbarrier initialisation) before everything after the barrier.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrives on an mbarrier given by its shared::cluster address (this CTA's or
// the other CTA's of a pair). The arrival carries the default CTA-scope
// release only: what it announces is tensor-memory data (ordered by the
// tcgen05 wait and fence before it) or the end of tensor-memory reads, never
// generic memory, and a cluster-scope release costs several hundred cycles.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}

// ---------------------------------------------------------------------------
// Bulk and tensor copies (TMA)
// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared; src, dst 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Asks L2 to fetch [src, src + bytes) from global memory (a hint: nothing
// waits for it; src 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// This CTA's share of an L2 prefetch of pf[0, bytes): one slice per CTA, in
// pieces of at most 64 KB (issued by one thread; nothing waits for them).
__device__ __forceinline__ void prefetch_share_l2(const uint8_t* pf, uint64_t bytes) {
  if (!pf || bytes == 0) return;
  const uint64_t share = (bytes / gridDim.x + 15) & ~uint64_t(15);
  const uint64_t begin = static_cast<uint64_t>(blockIdx.x) * share;
  const uint64_t end = min(begin + share, bytes);
  for (uint64_t off = begin; off < end; off += 65536)
    bulk_prefetch_l2(pf + off, static_cast<uint32_t>(min(static_cast<uint64_t>(65536), end - off)));
}

// Slice `part` of `parts` equal slices of [pf, pf + bytes), itself shared over
// the grid's CTAs as prefetch_share_l2 does: several threads of a CTA issue
// their slices at once.
__device__ __forceinline__ void prefetch_slice_l2(const uint8_t* pf, uint64_t bytes, int part, int parts) {
  if (!pf || bytes == 0) return;
  const uint64_t slice = (bytes / parts) & ~uint64_t(15);
  const uint64_t off = static_cast<uint64_t>(part) * slice;
  prefetch_share_l2(pf + off, part == parts - 1 ? bytes - off : slice);
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled tensor copy global -> shared. x (innermost) * element size must be a
// multiple of 16 bytes; out-of-range elements are filled with zeros.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 2-D tiled tensor copy into this CTA's shared memory whose completion
// (transaction bytes) is signalled on an mbarrier of either CTA of the pair,
// given by its shared::cluster address. Same alignment rule as tma_load_2d.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* tm, uint32_t bar_cl, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar_cl), "r"(x), "r"(y)
      : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (tensor core / TMA) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and MMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, fp16 operands, fp32 accumulator.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, fp16 operands, fp32 accumulator. A is M
// lanes x 16 fp16 (8 columns, two fp16 per 32-bit column, lower k in the low
// half) starting at column a_tmem.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier when all previously issued MMAs of this thread
// have completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// CTA-pair forms (cta_group::2). Tensor memory is allocated by one warp of
// each CTA of the pair, with the same number of columns; the MMA, issued by
// one thread of the even CTA, computes M = 256 rows: each CTA's tensor memory
// holds its 128 rows of A and of D, each CTA's shared memory half of B's N
// rows (at the same offset). A kernel uses either these forms or the
// cta_group::1 ones, never both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_f16_ta_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the mbarrier at the same offset in every CTA of `mask` when
// all previously issued MMAs of this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 64 fp16 (128 B), 8-row groups 1024 B apart, the
// 16-byte chunk c of row r stored at chunk position c ^ (r % 8). The tile base
// must be 1024-byte aligned; a K offset inside the 128-byte row is applied by
// advancing the start address.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);          // start address
  d |= static_cast<uint64_t>(1) << 16;                          // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A and B fp16, K-major, D fp32, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                                   // D format f32
         | (0u << 7) | (0u << 10)                    // A, B format f16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (32 * (warp % 4) + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Thread i of the warp writes r[0..15] to lane (32 * (warp % 4) + i), columns
// [col, col + 16) of taddr (whose lane field is the warp's lane quarter).
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// As tmem_st_32x32b_x16 with 8 columns.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
      "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Small integer / fp16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t half2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_half2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// dot of four unsigned bytes of a with four signed bytes of b, plus c.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace kq
