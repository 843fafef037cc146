// api_internal.h -- host-side helpers shared by the translation units of libmoe.so (not part of the C ABI).
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/moe.h"

namespace moe_internal {

// true if the environment variable MOE_FAULT names `site` (host-side fault injection for tests)
bool fault(const char* site);
// H, I multiples of 256 within [256, 4096]
bool shape_ok(int64_t H, int64_t I);
// number of SMs of the current device (cached per device)
int num_sms();

}  // namespace moe_internal
