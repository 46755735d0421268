// MSDA backward: launches. The kernel and its device helpers are in
// msda_backward.cuh; this unit holds the workspace kernels (zero, round to
// 16 bits) and the one-group-per-query-head instantiations, and
// msda_backward_split.cu the sample-split ones.
#include "msda_backward.cuh"

namespace msda {

// Zero n16 16-byte words.
__global__ void zero16_kernel(uint4 *p, int64_t n16) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// grad_value = round(workspace), 8 elements per thread.
template <typename T>
__global__ void convert8_kernel(const float4 *ws, uint4 *gv, int64_t n8) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const float4 a = ws[2 * i], b = ws[2 * i + 1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        gv[i] = pack16<T>(v);
    }
}

static unsigned stream_grid(int64_t n, int threads) {
    const int64_t want = (n + threads - 1) / threads;
    const int64_t cap = 152 * 16;  // a few waves of resident blocks on 152 SMs
    return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
}

cudaError_t launch_zero(void *p, int64_t bytes, cudaStream_t stream) {
    const int64_t n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    zero16_kernel<<<stream_grid(n16, 256), 256, 0, stream>>>(reinterpret_cast<uint4 *>(p), n16);
    return cudaGetLastError();
}

cudaError_t launch_convert(const float *ws, void *gv, int64_t n, msda_dtype_t dt, cudaStream_t stream) {
    const int64_t n8 = n / 8;
    if (n8 == 0) return cudaSuccess;
    const unsigned grid = stream_grid(n8, 256);
    if (dt == MSDA_BF16)
        convert8_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
            reinterpret_cast<const float4 *>(ws), reinterpret_cast<uint4 *>(gv), n8);
    else if (dt == MSDA_F16)
        convert8_kernel<__half><<<grid, 256, 0, stream>>>(
            reinterpret_cast<const float4 *>(ws), reinterpret_cast<uint4 *>(gv), n8);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_backward(const Params &p0, msda_dtype_t dt, bool f32acc, int lpg, bool softmax,
                            cudaStream_t stream) {
    // lanes per query-head as launch_backward_t picks them (narrow: 16-bit
    // data with the fp32 workspace)
    const bool narrow = f32acc && dt != MSDA_F32 && 2 * lpg <= 32;
    const int lanes = narrow ? 2 * lpg : lpg;
    Params p = p0;
    p.split_log2 = choose_split(p.triples, 32 / lanes, p.LK, p0.split_log2);
    if (p.split_log2 > 0) return launch_backward_split(p, dt, f32acc, lpg, softmax, stream);
    return softmax ? launch_backward_s<true, false>(p, dt, f32acc, lpg, stream)
                   : launch_backward_s<false, false>(p, dt, f32acc, lpg, stream);
}

}  // namespace msda
