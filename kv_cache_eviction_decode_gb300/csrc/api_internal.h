// api_internal.h -- helpers shared by the host translation units of the
// library (not part of the C ABI: hidden from the shared library's exports).
#pragma once

#include "kvevict.h"

#define KVEVICT_INTERNAL __attribute__((visibility("hidden")))

extern "C" {

// The CUDA device that holds the handle's state buffer (found once, at
// kvevict_create).
KVEVICT_INTERNAL int kvevict_handle_device(kvevict_t h);

// Every check kvevict_prefill_scored makes before it looks at the workspace:
// policy and dtype, the layer and its state, the prompt length, the Q/K/V
// pointers and their alignment, the launch limits. KVEVICT_OK or the status
// that call would return.
KVEVICT_INTERNAL int kvevict_prefill_scored_check(kvevict_t h, int layer, const void *Q, const void *K,
                                                  const void *V, int prompt_len);

// The device address of the allocation-free prefill's fixed scratch array on
// `device`, looked up once per device and cached; the lookup makes `device`
// current for its duration and restores the caller's device.
KVEVICT_INTERNAL int kvevict_static_scratch_address(int device, void **out);

}  // extern "C"
