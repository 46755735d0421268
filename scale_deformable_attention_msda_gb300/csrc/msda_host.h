// Host-side helpers shared by the entry points (no device code).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "msda.h"

namespace msda {

// Device address of a file-scope __device__ variable (given by its host-side
// name) in the context that is current on the calling thread. The address is
// cached per device together with the identity of the context it was looked
// up in; a call from a different context -- the primary context after
// cudaDeviceReset, or a context the caller made current -- looks it up again,
// so a stale address from a destroyed context is never handed to a kernel.
cudaError_t symbol_address(const void *symbol, void **out);

// Device word of the calling thread's current context in which the kernels
// of the range-checked build record an access outside a tensor;
// msda_device_check reads and clears it.
cudaError_t fault_word(unsigned **out);

}  // namespace msda
