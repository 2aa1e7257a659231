// paged_attn_fwd for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code running inside a CUDA graph that
// is being captured (cudaMalloc is not allowed there), plug-in hosts that own every
// allocation and hand out only the tensors of a call, or allocators with no free memory
// left at the moment of the call.  This entry point gives them the same attention with
// scratch memory that the library reserves itself: a fixed array in device global memory,
// created when the library's device code is loaded on a GPU and held until the process
// exits.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/vas.h"
#include "vas_internal.h"

namespace vas {
namespace {

// 32 MiB per device: the work list of several thousand sequences plus room for tens of
// thousands of split partial rows.  When a batch needs more partial rows than fit, the
// planner simply splits long sequences less finely.
constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;

static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

SymbolCache g_static_cache;

// Device address of this device's copy of the array.  In host code the array's name is
// only a stand-in for the symbol, so the address comes from the runtime: looked up with
// that device current on the first call, and again whenever the device's context has
// changed since (a context destroyed by cudaDeviceReset and created anew holds the
// array at a new address).
void* static_workspace_address() {
  return cached_symbol_address(g_static_cache, &g_static_workspace);
}

}  // namespace
}  // namespace vas

extern "C" int paged_attn_fwd_static(const void* q, const void* k_pages, const void* v_pages,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     const int32_t* query_lens, void* out, float* lse,
                                     const vas_attn_dims* dims, vas_stream_t stream) {
  const size_t need = paged_attn_workspace_min(dims);
  if (need == 0) {
    // Invalid or unsupported dimensions: let the main entry point name the error.
    return paged_attn_fwd(q, k_pages, v_pages, block_table, seq_lens, query_lens, out, lse,
                          dims, nullptr, 0, stream);
  }
  if (need > vas::kStaticWorkspaceBytes) return VAS_E_WORKSPACE;  // batch too large
  void* ws = vas::static_workspace_address();
  if (!ws) return VAS_E_CUDA;
  return paged_attn_fwd(q, k_pages, v_pages, block_table, seq_lens, query_lens, out, lse, dims,
                        ws, vas::kStaticWorkspaceBytes, stream);
}
