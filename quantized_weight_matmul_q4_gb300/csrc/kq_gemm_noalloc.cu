// kq_gemm_noalloc: the prefill GEMM of kq_gemm with its scratch (the fp16
// x_hat copy of X and the split-K partial sums) in a fixed device array of
// this file instead of a caller-provided workspace. Contract: include/kq.h.
//
// The array lives in this translation unit's own module. Under CUDA's default
// lazy module loading, a process that never calls kq_gemm_noalloc never loads
// the module and never pays its device memory; with eager loading
// (CUDA_MODULE_LOADING=EAGER) every context that loads the library reserves it.
#include <mutex>

#include "kq_common.cuh"
#include "kq_internal.h"

namespace kq {

// Scratch of kq_gemm_noalloc, one copy per device. Nothing in it has to start
// at zero: the quantiser writes every x_hat element the GEMM reads, and every
// split writes its whole partial-sum slice before the reduction reads it.
static __device__ __align__(256) uint8_t g_gemm_scratch[KQ_GEMM_STATIC_WS_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint8_t* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array. The first call on a device
// (with that device current) looks it up, which loads this module; later calls
// read the cached pointer.
cudaError_t scratch_for(int dev, uint8_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    uint8_t* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_gemm_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

}  // namespace
}  // namespace kq

using namespace kq;

extern "C" kq_status kq_gemm_noalloc(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K,
                                     int64_t N, kq_stream_t stream) {
  if (wtype != KQ_Q4_K && wtype != KQ_Q6_K && wtype != KQ_Q5_K) return KQ_ERR_TYPE;
  if (!W || !X || !Y) return KQ_ERR_NULL;
  if (M <= 0 || K <= 0 || N <= 0 || K % QK_K != 0 || M > kMaxDim || K > kMaxDim || N > kMaxDim ||
      M * N > (int64_t(1) << 40) || N * K > (int64_t(1) << 40))
    return KQ_ERR_SHAPE;
  if (wtype == KQ_Q6_K && K % 2048 != 0) return KQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(X) || !aligned16(Y)) return KQ_ERR_ALIGN;
  int dev, sms;
  int* err;
  if (device_context(&dev, &sms, &err) != cudaSuccess) return KQ_ERR_CUDA;
  const GemmPlan plan = plan_gemm(wtype, M, K, N, sms);
  if (plan.total_bytes > KQ_GEMM_STATIC_WS_BYTES) return KQ_ERR_WORKSPACE;
  uint8_t* ws = nullptr;
  if (scratch_for(dev, &ws) != cudaSuccess) return KQ_ERR_CUDA;
  int status = KQ_OK;
  const cudaError_t e =
      launch_gemm(wtype, W, X, Y, M, K, N, ws, plan, err, reinterpret_cast<cudaStream_t>(stream), &status);
  if (status != KQ_OK) return static_cast<kq_status>(status);
  return e == cudaSuccess ? KQ_OK : KQ_ERR_CUDA;
}
