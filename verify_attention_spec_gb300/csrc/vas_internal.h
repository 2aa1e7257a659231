// Internal host-side helpers shared by the library's translation units.
#pragma once

#include <cstdint>

namespace vas {

// Device address of the current device's error word (nullptr if CUDA fails).
int32_t* device_error_word();

// Number of SMs of the current device (0 if CUDA fails).
int num_sms();

// Process-unique id of the CUDA context current on this thread, 0 when none is current
// or the driver cannot say.  Ids are never reused within a process, so a cache of device
// addresses keyed on it notices a context that was destroyed and created again (after
// cudaDeviceReset, say) even when the new context's handle has the old value.
unsigned long long current_context_id();

// Device address of a __device__ variable in the current device's context, looked up
// with cudaGetSymbolAddress and cached per device against current_context_id(); nullptr
// if CUDA fails.  `cache` holds one entry per device index below kMaxCachedDevices.
constexpr int kMaxCachedDevices = 64;
struct SymbolCache {
  void* ptr[kMaxCachedDevices];
  unsigned long long ctx[kMaxCachedDevices];
};
void* cached_symbol_address(SymbolCache& cache, const void* symbol);

}  // namespace vas
