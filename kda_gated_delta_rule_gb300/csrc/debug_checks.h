// Debug-mode slot-id checks (debug_checks.cu) used by the C ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {
// With the debug checks on: the n ids at dev_ids are distinct, and none of them is among the n_other ids
// at dev_other (when dev_other is not null).  KDA_OK when the checks are off.
kda_status debug_check_slots(const int32_t* dev_ids, int32_t n, const int32_t* dev_other, int32_t n_other,
                             cudaStream_t s);
}  // namespace kda
