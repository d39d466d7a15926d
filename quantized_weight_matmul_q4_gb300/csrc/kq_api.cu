// C ABI of libkq: argument checks, workspace sizing, device error word, and
// dispatch to the kernels. Declarations and contracts: include/kq.h.
#include <atomic>
#include <mutex>

#include "kq_common.cuh"
#include "kq_internal.h"

namespace kq {

// First device error recorded by any kernel since the last kq_get_device_error
// (one word per device that loads the library). Kernels receive its device
// address as an argument.
__device__ int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_addr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Current device, its SM count and the device address of its error word.
cudaError_t device_state(int* dev, int* num_sms, int** err) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_addr[*dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
    if (e != cudaSuccess) return e;
    g_err_addr[*dev] = static_cast<int*>(p);
    g_num_sms[*dev] = n;
  }
  *num_sms = g_num_sms[*dev];
  *err = g_err_addr[*dev];
  return cudaSuccess;
}

// SM count for workspace sizing without touching the device when there is none.
int sm_count_or_default() {
  int dev = 0, n = 0;
  int* err = nullptr;
  if (device_state(&dev, &n, &err) == cudaSuccess && n > 0) return n;
  return 152;
}

std::atomic<uint8_t> g_smem_set[kSmemSlots][kMaxDevices];

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_wtype(int t) { return t == KQ_Q4_K || t == KQ_Q6_K || t == KQ_Q5_K; }  // the k-quants
inline bool valid_matvec_wtype(int t) { return valid_wtype(t); }
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

kq_status finish(cudaError_t e, int status) {
  if (status != KQ_OK) return static_cast<kq_status>(status);
  return e == cudaSuccess ? KQ_OK : KQ_ERR_CUDA;
}

}  // namespace

cudaError_t device_context(int* dev, int* num_sms, int** err) { return device_state(dev, num_sms, err); }

namespace {
std::atomic<int> g_hold_copies{0};
}  // namespace

int test_hold_copies() { return g_hold_copies.load(std::memory_order_relaxed); }

cudaError_t allow_max_smem(const void* kernel, int slot) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (slot < 0 || slot >= kSmemSlots || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidValue;
  if (g_smem_set[slot][dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e == cudaSuccess) g_smem_set[slot][dev].store(1, std::memory_order_release);
  return e;
}

}  // namespace kq

using namespace kq;

extern "C" {

const char* kq_status_str(int status) {
  switch (status) {
    case KQ_OK: return "KQ_OK";
    case KQ_ERR_NULL: return "KQ_ERR_NULL: a required pointer is NULL";
    case KQ_ERR_SHAPE: return "KQ_ERR_SHAPE: a size is out of range or not a multiple of its block";
    case KQ_ERR_ALIGN: return "KQ_ERR_ALIGN: a pointer is not 16-byte aligned";
    case KQ_ERR_TYPE: return "KQ_ERR_TYPE: unknown weight type";
    case KQ_ERR_WORKSPACE: return "KQ_ERR_WORKSPACE: workspace too small";
    case KQ_ERR_CUDA: return "KQ_ERR_CUDA: a CUDA runtime call failed";
    case KQ_ERR_DEVICE: return "KQ_ERR_DEVICE: a kernel recorded an error";
    default: return "unknown kq_status";
  }
}

kq_status kq_quantize_q8_1(const float* X, void* Xq, int64_t K, int64_t N, kq_stream_t stream) {
  if (!X || !Xq) return KQ_ERR_NULL;
  if (K <= 0 || N <= 0 || K % QK8_1 != 0 || K > kMaxDim || N > kMaxDim || K * N > (int64_t(1) << 40))
    return KQ_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(Xq)) return KQ_ERR_ALIGN;
  int dev, sms;
  int* err;
  cudaError_t e = device_state(&dev, &sms, &err);
  if (e != cudaSuccess) return KQ_ERR_CUDA;
  return finish(launch_quantize_q8_1(X, Xq, K, N, reinterpret_cast<cudaStream_t>(stream)), KQ_OK);
}

static kq_status matvec_entry(int wtype, const void* W, const float* x, const float* aux, float eps, int prod,
                              float* y, int64_t M, int64_t K, kq_stream_t stream, const void* W_next = nullptr,
                              size_t W_next_bytes = 0) {
  if (W_next && !aligned16(W_next)) return KQ_ERR_ALIGN;
  if (wtype == KQ_TQ4_1S && prod == PROD_X) {
    if (!W || !x || !y) return KQ_ERR_NULL;
    if (M <= 0 || K <= 0 || K % 32 != 0 || M > kMaxDim || K > kMaxDim) return KQ_ERR_SHAPE;
    if (!aligned16(W) || !aligned16(x) || !aligned16(y)) return KQ_ERR_ALIGN;
    int dev, sms;
    int* err;
    cudaError_t e = device_state(&dev, &sms, &err);
    if (e != cudaSuccess) return KQ_ERR_CUDA;
    int status = KQ_OK;
    const uint64_t pf_bytes = W_next ? (static_cast<uint64_t>(W_next_bytes) & ~uint64_t(15)) : 0;
    e = launch_tq4_matvec(W, x, y, M, K, W_next, pf_bytes, err, sms, reinterpret_cast<cudaStream_t>(stream), &status);
    return finish(e, status);
  }
  if (!valid_matvec_wtype(wtype)) return KQ_ERR_TYPE;
  if (!W || !x || !y || (prod != PROD_X && !aux)) return KQ_ERR_NULL;
  if (M <= 0 || K <= 0 || K % QK_K != 0 || M > kMaxDim || K > kMaxDim) return KQ_ERR_SHAPE;
  if (prod == PROD_RMSNORM && !(eps >= 0.f && eps < 1e30f)) return KQ_ERR_SHAPE;  // also rejects NaN
  if (!aligned16(W) || !aligned16(x) || !aligned16(y) || (prod != PROD_X && !aligned16(aux))) return KQ_ERR_ALIGN;
  int dev, sms;
  int* err;
  cudaError_t e = device_state(&dev, &sms, &err);
  if (e != cudaSuccess) return KQ_ERR_CUDA;
  int status = KQ_OK;
  const uint64_t pf_bytes = W_next ? (static_cast<uint64_t>(W_next_bytes) & ~uint64_t(15)) : 0;
  e = launch_matvec(wtype, W, x, aux, eps, prod, y, M, K, W_next, pf_bytes, err, sms,
                    reinterpret_cast<cudaStream_t>(stream), &status);
  return finish(e, status);
}

kq_status kq_matvec(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t K, kq_stream_t stream) {
  return matvec_entry(wtype, W, x, nullptr, 0.f, PROD_X, y, M, K, stream);
}

kq_status kq_matvec_prefetch(int wtype, const void* W, const float* x, float* y, int64_t M, int64_t K,
                             const void* W_next, size_t W_next_bytes, kq_stream_t stream) {
  return matvec_entry(wtype, W, x, nullptr, 0.f, PROD_X, y, M, K, stream, W_next, W_next_bytes);
}

kq_status kq_matvec_swiglu(int wtype, const void* W, const float* gate, const float* up, float* y, int64_t M,
                           int64_t K, kq_stream_t stream) {
  return matvec_entry(wtype, W, gate, up, 0.f, PROD_SWIGLU, y, M, K, stream);
}

kq_status kq_matvec_rmsnorm(int wtype, const void* W, const float* x, const float* gamma, float eps, float* y,
                            int64_t M, int64_t K, kq_stream_t stream) {
  return matvec_entry(wtype, W, x, gamma, eps, PROD_RMSNORM, y, M, K, stream);
}

kq_status kq_moe_combine(const float* Y, const float* probs, float* out, int64_t M, int64_t T, int32_t top_k,
                         kq_stream_t stream) {
  if (!Y || !probs || !out) return KQ_ERR_NULL;
  if (M <= 0 || T <= 0 || top_k <= 0 || top_k > 512 || M > kMaxDim || T * top_k > kMaxDim ||
      T * top_k * M > (int64_t(1) << 40))
    return KQ_ERR_SHAPE;
  if (!aligned16(Y) || !aligned16(probs) || !aligned16(out)) return KQ_ERR_ALIGN;
  int dev, sms;
  int* err;
  cudaError_t e = device_state(&dev, &sms, &err);
  if (e != cudaSuccess) return KQ_ERR_CUDA;
  e = launch_moe_combine(Y, probs, out, M, T, top_k, sms, reinterpret_cast<cudaStream_t>(stream));
  return finish(e, KQ_OK);
}

size_t kq_workspace_bytes(int op, int wtype, int64_t M, int64_t K, int64_t N_or_T, int32_t n_experts,
                          int32_t top_k) {
  if (!valid_wtype(wtype) || M <= 0 || K <= 0 || K % QK_K != 0 || N_or_T <= 0) return 0;
  if (op == KQ_OP_MATVEC) return 0;
  if (op == KQ_OP_GEMM) return plan_gemm(wtype, M, K, N_or_T, sm_count_or_default()).total_bytes;
  if (op == KQ_OP_MOE) {
    if (n_experts <= 0 || top_k <= 0 || top_k > n_experts) return 0;
    return plan_moe(wtype, M, K, N_or_T, n_experts, top_k).total_bytes;
  }
  return 0;
}

kq_status kq_gemm(int wtype, const void* W, const float* X, float* Y, int64_t M, int64_t K, int64_t N, void* ws,
                  size_t ws_bytes, kq_stream_t stream) {
  if (!valid_wtype(wtype)) return KQ_ERR_TYPE;
  if (!W || !X || !Y || !ws) return KQ_ERR_NULL;
  if (M <= 0 || K <= 0 || N <= 0 || K % QK_K != 0 || M > kMaxDim || K > kMaxDim || N > kMaxDim ||
      M * N > (int64_t(1) << 40) || N * K > (int64_t(1) << 40))
    return KQ_ERR_SHAPE;
  if (wtype == KQ_Q6_K && K % 2048 != 0) return KQ_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(X) || !aligned16(Y) || !aligned16(ws)) return KQ_ERR_ALIGN;
  int dev, sms;
  int* err;
  cudaError_t e = device_state(&dev, &sms, &err);
  if (e != cudaSuccess) return KQ_ERR_CUDA;
  const GemmPlan plan = plan_gemm(wtype, M, K, N, sms);
  if (ws_bytes < plan.total_bytes) return KQ_ERR_WORKSPACE;
  int status = KQ_OK;
  e = launch_gemm(wtype, W, X, Y, M, K, N, ws, plan, err, reinterpret_cast<cudaStream_t>(stream), &status);
  return finish(e, status);
}

kq_status kq_moe_grouped_gemm(int wtype, const void* W_experts, int32_t n_experts, const int32_t* expert_ids,
                              int32_t top_k, const float* X, float* Y, int64_t M, int64_t K, int64_t T, void* ws,
                              size_t ws_bytes, kq_stream_t stream) {
  if (!valid_wtype(wtype)) return KQ_ERR_TYPE;
  if (!W_experts || !expert_ids || !X || !Y || !ws) return KQ_ERR_NULL;
  if (M <= 0 || K <= 0 || T <= 0 || K % QK_K != 0 || n_experts <= 0 || n_experts > 512 || top_k <= 0 ||
      top_k > n_experts || M > kMaxDim || K > kMaxDim || T * top_k > kMaxDim ||
      static_cast<int64_t>(n_experts) * M > kMaxDim || T * top_k * K > (int64_t(1) << 40))
    return KQ_ERR_SHAPE;
  if (wtype == KQ_Q6_K && K % 2048 != 0) return KQ_ERR_SHAPE;
  if (!aligned16(W_experts) || !aligned16(expert_ids) || !aligned16(X) || !aligned16(Y) || !aligned16(ws))
    return KQ_ERR_ALIGN;
  int dev, sms;
  int* err;
  cudaError_t e = device_state(&dev, &sms, &err);
  if (e != cudaSuccess) return KQ_ERR_CUDA;
  const MoePlan plan = plan_moe(wtype, M, K, T, n_experts, top_k);
  if (ws_bytes < plan.total_bytes) return KQ_ERR_WORKSPACE;
  int status = KQ_OK;
  e = launch_moe(wtype, W_experts, n_experts, expert_ids, top_k, X, Y, M, K, T, ws, plan, err, sms,
                 reinterpret_cast<cudaStream_t>(stream), &status);
  return finish(e, status);
}

kq_status kq_test_hold_copies(int hold) {
  g_hold_copies.store(hold ? 1 : 0, std::memory_order_relaxed);
  return KQ_OK;
}

kq_status kq_get_device_error(int32_t* code, kq_stream_t stream) {
  if (!code) return KQ_ERR_NULL;
  int dev, sms;
  int* err;
  if (device_state(&dev, &sms, &err) != cudaSuccess) return KQ_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KQ_ERR_CUDA;
  if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KQ_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return KQ_ERR_CUDA;
  *code = host;
  return host == 0 ? KQ_OK : KQ_ERR_DEVICE;
}

}  // extern "C"
