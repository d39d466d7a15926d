// Measurement aid, not part of libkq: the issue rate of fifth-generation
// tensor-core MMAs of kind::f16 on this GPU, as a function of N and of where
// the A operand lives, to see what bounds the library's GEMM at small token
// counts ("Prefill Gap Closure Plan — ZINC CUDA vs llama.cpp": the fused
// dequant GEMM; the alternative there, int8 codes with a per-32-K rescale
// epilogue, has no tcgen05 form on this target: the assembler refuses
// tcgen05.mma .kind::i8 for sm_103a).
//
// Every CTA (one per SM) issues `iters` back-to-back MMAs with M = 128, K = 16
// and the given N into one tensor-memory accumulator (fp32), B from shared
// memory (zeros: the rate does not depend on the values), and records the
// clock64 cycles from the first issue to the commit of the last. Kinds:
//   0: A fp16 in shared memory (128-byte swizzle, K-major)
//   2: A fp16 in tensor memory (as the library's GEMM issues them)
//   3: as 2, with a commit to a second mbarrier after every 4 MMAs (as the
//      GEMM frees one K step's stage), nothing waiting on it
//   4: as 3, and the issuing thread waits for each of those commits before
//      issuing the next 4 MMAs (the round trip of one K step)
// Built into its own library (libkqprobe.so) by the package's build step.
#include "kq_common.cuh"

using namespace kq;

namespace {

constexpr int A_BYTES = 128 * 128;  // 128 rows x 128 bytes, 128-byte swizzle
constexpr int B_BYTES = 256 * 128;  // up to 256 rows
// More than half of an SM's shared memory, so that one CTA runs per SM and the
// tensor-memory allocations of two CTAs never meet on one SM.
constexpr int SMEM_BYTES = 120 * 1024;

__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int kind, int n, int iters,
                                                          unsigned long long* __restrict__ cycles) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + A_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + A_BYTES + B_BYTES);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(bar + 2);
  uint64_t* bar2 = bar + 3;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(bar2, 1);
    *abort = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zeros before the tensor cores read them
  if (warp == 0) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (warp == 0) {
    if (kind >= 2) {  // A operand in tensor memory: columns 256.. (zeros)
      uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      tmem_st_32x32b_x8(tmem + 256, z);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    const uint32_t idesc = idesc_f16_f32(128, n);
    const uint64_t adesc = smem_desc_sw128(smem_u32(sA));
    const uint64_t bdesc = smem_desc_sw128(smem_u32(sB));
    unsigned long long t0 = 0;
    bool ok2 = true;
    if (kind == 4) {
      // the whole warp waits (bounded), one elected lane issues
      t0 = clock64();
      for (int i = 0; i < iters && ok2; i += 4) {
        if (elect_one()) {
          for (int k = 0; k < 4; ++k) umma_f16_ta(tmem, tmem + 256, bdesc + 2 * k, idesc, (i + k) > 0 ? 1u : 0u);
          umma_commit(bar2);
        }
        __syncwarp();
        ok2 = __all_sync(0xffffffffu, mbar_wait(bar2, (i >> 2) & 1, abort, nullptr));
      }
      if (elect_one()) umma_commit(bar);
    } else if (elect_one()) {
      t0 = clock64();
      for (int i = 0; i < iters; ++i) {
        const int k = i & 3;  // the four 32-byte K slices of the 128-byte rows
        if (kind == 0)
          umma_f16(tmem, adesc + 2 * k, bdesc + 2 * k, idesc, i > 0 ? 1u : 0u);
        else
          umma_f16_ta(tmem, tmem + 256, bdesc + 2 * k, idesc, i > 0 ? 1u : 0u);
        if (kind == 3 && k == 3) umma_commit(bar2);
      }
      umma_commit(bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(bar, 0, abort, nullptr);
    if (elect_one()) cycles[blockIdx.x] = (ok && ok2) ? clock64() - t0 : 0ull;
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int kqprobe_mma(int kind, int n, int iters,
                                                                   unsigned long long* cycles, int grid,
                                                                   void* stream) {
  if ((kind != 0 && kind != 2 && kind != 3 && kind != 4) || n < 16 || n > 256 || n % 16 != 0 || iters < 1 || grid < 1 || !cycles) return -1;
  cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return static_cast<int>(e);
  mma_rate_kernel<<<grid, 128, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(kind, n, iters, cycles);
  return static_cast<int>(cudaGetLastError());
}
