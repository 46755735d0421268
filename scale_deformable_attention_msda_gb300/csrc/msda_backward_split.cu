// MSDA backward: the sample-split instantiations (small problems; see
// choose_split in msda_common.cuh and the kernel in msda_backward.cuh).
#include "msda_backward.cuh"

namespace msda {

cudaError_t launch_backward_split(const Params &p, msda_dtype_t dt, bool f32acc, int lpg,
                                  bool softmax, cudaStream_t stream) {
    return softmax ? launch_backward_s<true, true>(p, dt, f32acc, lpg, stream)
                   : launch_backward_s<false, true>(p, dt, f32acc, lpg, stream);
}

}  // namespace msda
