// MSDA backward of bf16 data accumulated in the scaled fp16 workspace
// (MSDA_ACC_FP16_BUFFER; F16ACC in msda_backward.cuh): the instantiations, with
// and without the sample split, compiled in a unit of their own.
#include "msda_backward.cuh"

namespace msda {

cudaError_t launch_backward_f16acc(const Params &p0, int lpg, bool softmax, cudaStream_t stream) {
    Params p = p0;
    p.split_log2 = choose_split(p.triples, 32 / lpg, p.LK, p0.split_log2);
    if (p.split_log2 > 0)
        return softmax ? launch_backward_f16acc_s<true, true>(p, lpg, stream)
                       : launch_backward_f16acc_s<false, true>(p, lpg, stream);
    return softmax ? launch_backward_f16acc_s<true, false>(p, lpg, stream)
                   : launch_backward_f16acc_s<false, false>(p, lpg, stream);
}

}  // namespace msda
