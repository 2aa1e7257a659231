// Library-wide C ABI entry points: the device error word, status strings and the
// diagnostic Philox kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/vas.h"
#include "philox.cuh"
#include "vas_internal.h"

namespace vas {

// One error word per device; kernels OR bits into it, vas_last_device_error clears it.
__device__ int32_t g_error_word;

namespace {
constexpr int kMaxDevices = kMaxCachedDevices;
int g_sms[kMaxDevices];
SymbolCache g_error_cache;
std::mutex g_mu;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Driver entry points, found through the runtime (the library does not link libcuda).
template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}
}  // namespace

unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

void* cached_symbol_address(SymbolCache& cache, const void* symbol) {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (id == 0 || cache.ctx[dev] != id || !cache.ptr[dev]) {
    // No context yet (the lookup below makes the device's primary context current), or
    // a different one from the cached lookup's: resolve the address again.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
    cache.ptr[dev] = p;
    cache.ctx[dev] = current_context_id();
  }
  return cache.ptr[dev];
}

int32_t* device_error_word() {
  return static_cast<int32_t*>(cached_symbol_address(g_error_cache, &g_error_word));
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

__global__ void philox_fill_kernel(const uint4* ctr, uint32_t k0, uint32_t k1, uint4* out,
                                   int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = philox4x32_10(ctr[i], k0, k1);
}

}  // namespace vas

extern "C" {

int vas_last_device_error(int32_t* bits, vas_stream_t stream) {
  if (!bits) return VAS_E_INVALID_ARG;
  int32_t* word = vas::device_error_word();
  if (!word) return VAS_E_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return VAS_E_CUDA;
  if (cudaMemsetAsync(word, 0, sizeof host, s) != cudaSuccess) return VAS_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return VAS_E_CUDA;
  *bits = host;
  return VAS_OK;
}

int vas_philox4x32_10(const uint32_t* counters, uint32_t key0, uint32_t key1, uint32_t* out,
                      int64_t n, vas_stream_t stream) {
  if (n < 0 || (n > 0 && (!counters || !out))) return VAS_E_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(counters) | reinterpret_cast<uintptr_t>(out)) & 15)
    return VAS_E_INVALID_ARG;
  if (n == 0) return VAS_OK;
  const int sms = vas::num_sms();
  if (!sms) return VAS_E_CUDA;
  const int64_t blocks64 = (n + 255) / 256;
  const int blocks = static_cast<int>(blocks64 < 8 * sms ? blocks64 : 8 * sms);
  vas::philox_fill_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(counters), key0, key1, reinterpret_cast<uint4*>(out), n);
  return cudaGetLastError() == cudaSuccess ? VAS_OK : VAS_E_CUDA;
}

const char* vas_status_string(int status) {
  switch (status) {
    case VAS_OK: return "ok";
    case VAS_E_INVALID_ARG: return "invalid argument";
    case VAS_E_UNSUPPORTED: return "unsupported dtype, head_dim or page_size";
    case VAS_E_WORKSPACE: return "workspace too small";
    case VAS_E_CUDA: return "CUDA error";
    case VAS_E_NOMEM: return "not enough free pages";
    case VAS_E_NOT_FOUND: return "unknown sequence id";
    case VAS_E_EXISTS: return "sequence id already present";
    default: return "unknown status";
  }
}

}  // extern "C"
