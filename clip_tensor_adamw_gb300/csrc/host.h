// Host-side helpers shared by the C ABI's translation units (api.cpp, noalloc.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include "mica_optim.h"

namespace mica {

// `p` must be device (or managed) memory of `device`, aligned to `align`, and [p, p + bytes) must lie inside the
// allocation that holds p when the driver can tell its extent; on failure the call's error detail names `what`
// and `index`. MICA_OK or MICA_ERR_ADDRESS.
mica_status check_device_span(const void* p, size_t bytes, size_t align, int device, const char* what,
                              int64_t index);

// Forgets the device addresses of the no-allocation norm's scratch array, so that the next call looks each one up
// again (a device reset may move the array). Called by mica_release_cache().
void noalloc_forget_addresses();

}  // namespace mica
