// Internal host-side helpers shared by the library's translation units.
#pragma once

#include <cstdint>

namespace vas {

// Device address of the current device's error word (nullptr if CUDA fails).
int32_t* device_error_word();

// Number of SMs of the current device (0 if CUDA fails).
int num_sms();

}  // namespace vas
