// The range-checked build's fault word and its readback (libmsda_checked.so,
// compiled with -DMSDA_CHECKED; the normal libmsda.so has the same entry
// points, which then report no faults).
//
// compute-sanitizer is not available where this library is tested, so the
// checked build stands in for its memcheck: every global access of the
// operator kernels (forward, backward, corners) is checked first against the
// extent of the tensor it belongs to (in_tensor in msda_common.cuh); the
// workspace passes (zero, convert, the fp16 workspace's prepare and finish)
// each walk a flat range [0, n) of the buffer they are launched over, bounded
// by their loop conditions. An access that would leave its tensor is
// skipped and sets bit 0 of one device word per context; the host reads and
// clears that word after a synchronisation. Nothing traps, so a fault found
// this way leaves the context usable.
//
// The word is a file-scope __device__ variable (msda_runtime.cu). Its device
// address is looked up in the calling thread's current context and cached
// with that context's identity, so a new context (after cudaDeviceReset, for
// instance) gets its own address. The first lookup in a context loads the
// library's module; make it before any stream capture begins.
#include "msda_common.cuh"
#include "msda_host.h"

namespace msda {

namespace {

// One range check that must fail (a NULL tensor of extent 0); no memory access.
__global__ void bounds_self_test_kernel(const Params p) {
    if (threadIdx.x == 0) (void)in_tensor(p, static_cast<const int *>(nullptr),
                                          static_cast<const int *>(nullptr), 1, 0);
}

}  // namespace

// Params::err for a launch: the current context's fault word in the checked
// build, NULL in the normal one.
cudaError_t fault_word_for_launch(unsigned **err) {
#ifdef MSDA_CHECKED
    return fault_word(err);
#else
    *err = nullptr;
    return cudaSuccess;
#endif
}

}  // namespace msda

extern "C" {

int msda_checked_build(void) {
#ifdef MSDA_CHECKED
    return 1;
#else
    return 0;
#endif
}

msda_status_t msda_device_check(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MSDA_ERR_CUDA;
#ifdef MSDA_CHECKED
    unsigned *word = nullptr;
    if (msda::fault_word(&word) != cudaSuccess) return MSDA_ERR_CUDA;
    unsigned v = 0u;
    if (cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MSDA_ERR_CUDA;
    if (v != 0u) {
        const unsigned zero = 0u;
        if (cudaMemcpy(word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return MSDA_ERR_CUDA;
        return MSDA_ERR_DEVICE_BOUNDS;
    }
#endif
    return MSDA_OK;
}

msda_status_t msda_debug_bounds_self_test(void *stream) {
    msda::Params p = {};
    if (msda::fault_word_for_launch(&p.err) != cudaSuccess) return MSDA_ERR_CUDA;
    msda::bounds_self_test_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? MSDA_OK : MSDA_ERR_CUDA;
}

}  // extern "C"
