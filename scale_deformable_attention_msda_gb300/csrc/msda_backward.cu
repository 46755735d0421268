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
// when attn is given, its largest |attention weight| (bf16; 8 per word when
// the weights are 16-byte aligned, else one at a time). One block of 1024
// threads per SM at most (kF16MaxBlocks), four loads in flight per thread.
__device__ __forceinline__ float abs_max8_bf16(float m, const uint4 w) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)   // |bf16| as fp32: drop the sign, widen exactly
        m = fmaxf(m, fmaxf(__uint_as_float((u[k] << 16) & 0x7fffffffu),
                           __uint_as_float(u[k] & 0x7fff0000u)));
    return m;
}

__device__ __forceinline__ float abs_max_stream(float m, const uint4 *x, int64_t n8, int64_t i0,
                                                int64_t stride) {
    int64_t i = i0;
    for (; i + 3 * stride < n8; i += 4 * stride) {
        const uint4 a = x[i], b = x[i + stride], c = x[i + 2 * stride], d = x[i + 3 * stride];
        m = abs_max8_bf16(abs_max8_bf16(abs_max8_bf16(abs_max8_bf16(m, a), b), c), d);
    }
    for (; i < n8; i += stride) m = abs_max8_bf16(m, x[i]);
    return m;
}

__global__ void zero_f16_max_kernel(uint4 *ws, int64_t n16, const uint4 *gout, int64_t ng8,
                                    const unsigned short *attn, int64_t na, float *gmax,
                                    float *amax) {
    __shared__ float warp_max[2][32];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = i0; i < n16; i += stride) ws[i] = make_uint4(0u, 0u, 0u, 0u);
    float m = abs_max_stream(0.0f, gout, ng8, i0, stride);
    float ma = 0.0f;
    if (attn) {
        int64_t done = 0;
        if ((reinterpret_cast<uintptr_t>(attn) & 15u) == 0) {
            ma = abs_max_stream(ma, reinterpret_cast<const uint4 *>(attn), na / 8, i0, stride);
            done = na / 8 * 8;
        }
        for (int64_t i = done + i0; i < na; i += stride)
            ma = fmaxf(ma, __uint_as_float(((uint32_t)attn[i] << 16) & 0x7fffffffu));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, off));
    }
    if ((threadIdx.x & 31) == 0) {
        warp_max[0][threadIdx.x >> 5] = m;
        warp_max[1][threadIdx.x >> 5] = ma;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.0f, ba = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            b = fmaxf(b, warp_max[0][w]);
            ba = fmaxf(ba, warp_max[1][w]);
        }
        gmax[blockIdx.x] = b;
        amax[blockIdx.x] = ba;
    }
}

// After the adds: grad_value = round(workspace * 2^-k), 8 elements per thread;
// (2^k, 2^-k) as block 0 of the backward stored it.
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

// The scaled fp16 workspace: [accumulator: n halfs][tail], the tail laid out
// as kF16MaxBlocks says. Zero + maxima here; the backward derives the scale
// from the maxima (f16_block_scale) and the finish pass applies its inverse.
// attn NULL: the weights are probabilities (the softmax variant).
int f16_prepare_blocks(int64_t n, int64_t ng, const void *attn, int64_t na) {
    int64_t work = n / 8 > ng / 8 ? n / 8 : ng / 8;
    if (attn && na / 8 > work) work = na / 8;
    const int64_t want = (work + 1023) / 1024;
    return (int)(want < 1 ? 1 : (want < kF16MaxBlocks ? want : kF16MaxBlocks));
}
cudaError_t launch_f16_prepare(void *ws, int64_t n, const void *grad_out, int64_t ng,
                               const void *attn, int64_t na, cudaStream_t stream) {
    float *tail = reinterpret_cast<float *>(static_cast<char *>(ws) + n * 2);
    const int grid = f16_prepare_blocks(n, ng, attn, na);
    zero_f16_max_kernel<<<grid, 1024, 0, stream>>>(reinterpret_cast<uint4 *>(ws), n * 2 / 16,
                                                  reinterpret_cast<const uint4 *>(grad_out), ng / 8,
                                                  static_cast<const unsigned short *>(attn), na,
                                                  tail, tail + grid);
    return cudaGetLastError();
}
float *f16_scale_pair(void *ws, int64_t n) {
    return reinterpret_cast<float *>(static_cast<char *>(ws) + n * 2) + 2 * kF16MaxBlocks;
}
cudaError_t launch_f16_finish(void *ws, void *gv, int64_t n, cudaStream_t stream) {
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
