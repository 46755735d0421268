// Integer parts of every sample, computed by the same device code
// (load_level_table, level_of, sample_geometry) the forward and backward
// kernels use. For bit-exact checks against an independent definition.
#include "msda_common.cuh"

namespace msda {

template <typename T>
__global__ void __launch_bounds__(kThreads)
msda_corners_kernel(const Params p, int32_t *rows) {
    __shared__ LevelTable lt;
    load_level_table(lt, p);
    __syncthreads();
    const int64_t n = p.triples * p.LK;
    const T *loc = reinterpret_cast<const T *>(p.loc);
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n;
         s += (int64_t)gridDim.x * blockDim.x) {
        const int idx = (int)(s % p.LK);
        const int l = level_of(idx, p.inv_K);
        if (!in_tensor(p, loc, loc + 2 * s, 2, 2 * n) || !in_tensor(p, rows, rows + 4 * s, 4, 4 * n))
            continue;
        const float2 xy = load_xy<T>(loc + 2 * s);
        SampleGeom g;
        sample_geometry(g, xy.x, xy.y, lt, l);
        int4 o;
        o.x = (g.vx0 && g.vy0) ? g.row[0] : -1;
        o.y = (g.vx1 && g.vy0) ? g.row[1] : -1;
        o.z = (g.vx0 && g.vy1) ? g.row[2] : -1;
        o.w = (g.vx1 && g.vy1) ? g.row[3] : -1;
        reinterpret_cast<int4 *>(rows)[s] = o;
    }
}

cudaError_t launch_corners(const Params &p, msda_dtype_t dt, int32_t *rows, cudaStream_t stream) {
    const int64_t n = p.triples * p.LK;
    const int64_t want = (n + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(want < 4096 ? want : 4096);
    switch (dt) {
        case MSDA_F32: msda_corners_kernel<float><<<grid, kThreads, 0, stream>>>(p, rows); break;
        case MSDA_BF16: msda_corners_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(p, rows); break;
        case MSDA_F16: msda_corners_kernel<__half><<<grid, kThreads, 0, stream>>>(p, rows); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace msda
