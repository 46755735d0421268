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

// Scaled fp16 workspace (MSDA_ACC_FP16_BUFFER), before the adds: zero the
// workspace and record each block's largest |grad_out| (bf16, 8 per word) and,
// when attn is given, its largest |attention weight| (bf16, one at a time: the
// weights are 2-byte aligned only).
__device__ __forceinline__ float block_max_of(float m, float *warp_max) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    float b = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) b = fmaxf(b, warp_max[w]);
    __syncthreads();
    return b;
}

__global__ void zero_f16_max_kernel(uint4 *ws, int64_t n16, const uint4 *gout, int64_t ng8,
                                    const unsigned short *attn, int64_t na, float *gmax,
                                    float *amax) {
    __shared__ float warp_max[32];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = i0; i < n16; i += stride) ws[i] = make_uint4(0u, 0u, 0u, 0u);
    float m = 0.0f;
    for (int64_t i = i0; i < ng8; i += stride) {
        const uint4 w = gout[i];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)   // |bf16| as fp32: drop the sign, widen exactly
            m = fmaxf(m, fmaxf(__uint_as_float((u[k] << 16) & 0x7fffffffu),
                               __uint_as_float(u[k] & 0x7fff0000u)));
    }
    float ma = 0.0f;
    if (attn)
        for (int64_t i = i0; i < na; i += stride)
            ma = fmaxf(ma, __uint_as_float(((uint32_t)attn[i] << 16) & 0x7fffffffu));
    m = block_max_of(m, warp_max);
    ma = block_max_of(ma, warp_max);
    if (threadIdx.x == 0) {
        gmax[blockIdx.x] = m;
        amax[blockIdx.x] = ma;
    }
}

// One block: the call's scale 2^k. Every element of grad_value sums, over the
// samples that reach it, |a| * w * |g| with bilinear weight w <= 1, one sample
// per (q, l, k) at most, so |sum| <= max|g| * Q * A, where A = max over
// query-heads of sum_{l,k} |a| <= L K max|a| (A = 1 for the softmax variant,
// whose weights are probabilities). k puts that bound in [2^14, 2^15): no sum
// can pass fp16's largest finite value, 65504. Inside fp16's normal range the
// rounding of a sum does not depend on k; a sum below 2^-29 of the bound falls
// into fp16's subnormals and keeps fewer bits.
__global__ void f16_scale_kernel(const float *gmax, const float *amax, int n, int64_t Q,
                                 int64_t LK, float *scale_pair) {
    __shared__ float warp_max[32];
    float m = 0.0f, ma = 0.0f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        m = fmaxf(m, gmax[i]);
        if (amax) ma = fmaxf(ma, amax[i]);
    }
    m = block_max_of(m, warp_max);
    ma = block_max_of(ma, warp_max);
    if (threadIdx.x == 0) {
        const double a = amax ? (double)LK * (double)ma : 1.0;
        const double bound = (double)m * (double)Q * a;
        int k = 0;
        if (bound > 0.0 && bound < 1.0e300) {
            int e;
            (void)frexp(bound, &e);              // bound = f 2^e, f in [0.5, 1)
            k = min(max(15 - e, -126), 126);
        }
        scale_pair[0] = ldexpf(1.0f, k);
        scale_pair[1] = ldexpf(1.0f, -k);
    }
}

// After the adds: grad_value = round(workspace * 2^-k), 8 elements per thread.
template <typename T>
__global__ void finish_f16_kernel(const uint4 *ws, uint4 *gv, int64_t n8, const float *scale_pair) {
    const float inv = scale_pair[1];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        float v[8];
        unpack16<__half>(v, ws[i]);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] *= inv;
        gv[i] = pack16<T>(v);
    }
}

// a few waves of resident blocks on 152 SMs; the fp16 workspace's tail holds
// one maximum per block of such a grid
constexpr int64_t kStreamGridCap = 152 * 16;
static_assert(kStreamGridCap <= kF16MaxBlocks, "fp16 workspace tail");
static unsigned stream_grid(int64_t n, int threads) {
    const int64_t want = (n + threads - 1) / threads;
    const int64_t cap = kStreamGridCap;
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

// The scaled fp16 workspace: [accumulator: n halfs][tail], the tail laid out
// as kF16MaxBlocks says. Zero + maxima, scale, (adds), finish. attn NULL: the
// weights are probabilities (the softmax variant).
cudaError_t launch_f16_prepare(void *ws, int64_t n, const void *grad_out, int64_t ng,
                               const void *attn, int64_t na, int64_t Q, int64_t LK,
                               cudaStream_t stream) {
    const int64_t n16 = n * 2 / 16, ng8 = ng / 8;
    float *tail = reinterpret_cast<float *>(static_cast<char *>(ws) + n * 2);
    int64_t work = n16 > ng8 ? n16 : ng8;
    if (attn && na / 8 > work) work = na / 8;
    const unsigned grid = stream_grid(work, 256);   // <= kF16MaxBlocks
    zero_f16_max_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<uint4 *>(ws), n16,
                                                  reinterpret_cast<const uint4 *>(grad_out), ng8,
                                                  static_cast<const unsigned short *>(attn), na,
                                                  tail, tail + kF16MaxBlocks);
    f16_scale_kernel<<<1, 256, 0, stream>>>(tail, attn ? tail + kF16MaxBlocks : nullptr, (int)grid,
                                            Q, LK, tail + 2 * kF16MaxBlocks);
    return cudaGetLastError();
}
const float *f16_scale_pair(const void *ws, int64_t n) {
    return reinterpret_cast<const float *>(static_cast<const char *>(ws) + n * 2) + 2 * kF16MaxBlocks;
}
cudaError_t launch_f16_finish(const void *ws, void *gv, int64_t n, cudaStream_t stream) {
    const int64_t n8 = n / 8;
    if (n8 == 0) return cudaSuccess;
    finish_f16_kernel<__nv_bfloat16><<<stream_grid(n8, 256), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(ws), reinterpret_cast<uint4 *>(gv), n8, f16_scale_pair(ws, n));
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
