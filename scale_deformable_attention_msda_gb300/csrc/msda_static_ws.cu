// msda_backward_static_workspace: the backward without a caller-provided
// workspace, for callers that cannot allocate device memory when they call.
//
// For a 16-bit dtype, msda_backward accumulates grad_value in an fp32
// workspace of B*S*M*D floats that the caller allocates. Some callers cannot
// do that at call time: an operator plugin inside an inference or training
// engine that owns all device memory through its own pool and hands the
// operator no scratch, or an application that forbids device allocation after
// start-up because cudaMalloc can synchronise the device and fragment memory
// reserved up front. This entry point gives them the same result with the
// scratch in a fixed array that belongs to the library.
//
// The array is a file-scope __device__ variable of MSDA_STATIC_WORKSPACE_BYTES
// (declared in msda.h). Host code cannot use the array's name as a device
// address (on the host it names a host-side stand-in), so each call looks up
// the real address with cudaGetSymbolAddress in the calling thread's current
// context; the address is cached together with that context's identity and
// looked up again whenever a call comes from another context (for instance
// the primary context recreated after cudaDeviceReset), so a call never adds
// through an address of a destroyed context. The first lookup in a context
// loads the library's module there; make that first call before any stream
// capture begins.
//
// Every call shares the one array and leaves its contents behind. msda_backward
// zeroes the part a call uses before accumulating into it, so stale contents
// never reach a result, but calls whose work overlaps on the GPU (different
// streams, or different host threads) race on the array and must be ordered
// by the caller. Nothing here calls cudaMalloc, cudaFree or any other
// allocating routine.
#include <cuda_runtime.h>

#include "msda.h"
#include "msda_host.h"

namespace {

constexpr size_t kStaticFloats = MSDA_STATIC_WORKSPACE_BYTES / sizeof(float);

__device__ __align__(256) float g_static_workspace[kStaticFloats];

// Device address of g_static_workspace in the current context.
msda_status_t static_workspace_address(void **out) {
    return msda::symbol_address(reinterpret_cast<const void *>(&g_static_workspace), out) ==
                   cudaSuccess
               ? MSDA_OK
               : MSDA_ERR_CUDA;
}

}  // namespace

extern "C" msda_status_t msda_backward_static_workspace(
    const void *value, const int64_t *spatial_shapes, const int64_t *level_start_index,
    const void *sampling_locations, const void *attention_weights, const int32_t *query_order,
    const void *grad_out, void *grad_value, void *grad_sampling_locations,
    void *grad_attention_weights, const msda_dims_t *dims, msda_dtype_t dtype, void *stream) {
    if (!dims) return MSDA_ERR_NULL;
    // 0 for fp32 data (no workspace needed) and for dimensions msda_backward rejects
    const size_t need = msda_backward_workspace_bytes(dims, dtype, MSDA_ACC_FP32_BUFFER);
    if (need > MSDA_STATIC_WORKSPACE_BYTES) return MSDA_ERR_WORKSPACE;
    void *ws = nullptr;
    if (need > 0) {
        const msda_status_t st = static_workspace_address(&ws);
        if (st != MSDA_OK) return st;
    }
    return msda_backward(value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, query_order, grad_out, grad_value,
                         grad_sampling_locations, grad_attention_weights, ws,
                         need > 0 ? MSDA_STATIC_WORKSPACE_BYTES : 0, MSDA_ACC_FP32_BUFFER, dims,
                         dtype, stream);
}
