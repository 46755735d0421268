// MSDA in float64: forward, backward (with the softmax variant) and the
// integer parts, for callers that need the operator in double precision
// (gradient checks, reference runs). Double-precision throughput is low on
// GB300, so these kernels favour plainness over speed: a group of LPG = D/2
// lanes owns one (b, q, m), each lane 16 bytes (two channels), and every lane
// computes the geometry of each sample itself.
//
// Geometry as the double-precision loop of the msda-triton course, ch. 1
// ("The simplest possible implementation"): x = loc_x*W - 0.5 with a
// rounded multiply and a rounded add (no fused multiply-add, so the integer
// parts are those of that loop bit for bit), x0 = floor(x), lx = x - x0.
#include "msda_common.cuh"

namespace msda {

struct Geom64 {
    bool inside;
    double lx, ly;
    bool vx0, vx1, vy0, vy1;
    int row[4];
};

__device__ __forceinline__ void sample_geometry64(Geom64 &g, double loc_x, double loc_y,
                                                  const LevelTable &lt, int l) {
    const double Wd = lt.Wf[l], Hd = lt.Hf[l];   // -2 for an invalid level
    const double x = __dadd_rn(__dmul_rn(loc_x, Wd), -0.5);
    const double y = __dadd_rn(__dmul_rn(loc_y, Hd), -0.5);
    g.inside = (x >= -1.0) && (x < Wd) && (y >= -1.0) && (y < Hd);
    const double x0f = g.inside ? floor(x) : 0.0, y0f = g.inside ? floor(y) : 0.0;
    const int x0 = (int)x0f, y0 = (int)y0f;
    const int W = lt.W[l], H = (int)lt.Hf[l];
    g.lx = g.inside ? x - x0f : 0.0;
    g.ly = g.inside ? y - y0f : 0.0;
    g.vx0 = g.inside && x0 >= 0;
    g.vx1 = g.inside && x0 + 1 < W;
    g.vy0 = g.inside && y0 >= 0;
    g.vy1 = g.inside && y0 + 1 < H;
    const int xa = g.vx0 ? x0 : 0, xb = g.vx1 ? x0 + 1 : 0;
    const int ya = g.vy0 ? y0 : 0, yb = g.vy1 ? y0 + 1 : 0;
    const int r0 = lt.start[l] + ya * W, r1 = lt.start[l] + yb * W;
    g.row[0] = r0 + xa;
    g.row[1] = r0 + xb;
    g.row[2] = r1 + xa;
    g.row[3] = r1 + xb;
}

// Softmax statistics of one query-head's L*K logits, computed by each lane.
__device__ __forceinline__ void softmax64(const double *z, int LK, double &mx, double &inv) {
    mx = -INFINITY;
    for (int i = 0; i < LK; ++i) mx = fmax(mx, z[i]);
    double s = 0.0;
    for (int i = 0; i < LK; ++i) s += exp(z[i] - mx);
    inv = 1.0 / s;
}

// The lane's group: (b, q, m) of triple t, with `valid` false past the end or
// for a dispatch slot outside [0, Q).
__device__ __forceinline__ Triple group_triple(const Params &p, int64_t t, bool &valid) {
    valid = t < p.triples;
    Triple tr = triple_of(valid ? t : 0, p);
    valid = valid && tr.q >= 0 && tr.q < p.Q;
    return tr;
}

template <int LPG, bool SOFTMAX>
__global__ void __launch_bounds__(kThreads) msda_forward_f64_kernel(const Params p) {
    __shared__ LevelTable lt;
    load_level_table(lt, p);
    __syncthreads();
    const int lane = threadIdx.x & 31, r = lane % LPG;
    const int64_t t = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LPG;
    bool valid;
    const Triple tr = group_triple(p, t, valid);
    if (!valid) return;   // no shuffles below: lanes may leave independently
    const double *loc0 = reinterpret_cast<const double *>(p.loc);
    const double *attn0 = reinterpret_cast<const double *>(p.attn);
    const double *value = reinterpret_cast<const double *>(p.value);
    const double *loc = loc0 + tr.bqm * p.LK * 2;
    const double *attn = attn0 + tr.bqm * p.LK;
    const double *vbase = value + ((int64_t)tr.b * p.S * p.M + tr.m) * p.D + 2 * r;
    const int64_t nv = n_value(p), ns = n_samples(p);
    if (!in_tensor(p, loc0, loc, 2 * (int64_t)p.LK, 2 * ns) ||
        !in_tensor(p, attn0, attn, p.LK, ns))
        return;
    double mx = 0.0, inv = 1.0;
    if (SOFTMAX) softmax64(attn, p.LK, mx, inv);
    double acc0 = 0.0, acc1 = 0.0;
    for (int idx = 0; idx < p.LK; ++idx) {
        const int l = level_of(idx, p.inv_K);
        const double a = SOFTMAX ? exp(attn[idx] - mx) * inv : attn[idx];
        Geom64 g;
        sample_geometry64(g, loc[2 * idx], loc[2 * idx + 1], lt, l);
        const double hx = 1.0 - g.lx, hy = 1.0 - g.ly;
        const double w[4] = {(g.vx0 && g.vy0) ? a * hx * hy : 0.0, (g.vx1 && g.vy0) ? a * g.lx * hy : 0.0,
                             (g.vx0 && g.vy1) ? a * hx * g.ly : 0.0, (g.vx1 && g.vy1) ? a * g.lx * g.ly : 0.0};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (w[c] != 0.0 && in_tensor(p, value, vbase + (int64_t)g.row[c] * p.MD, 2, nv)) {
                const double2 v = __ldg(reinterpret_cast<const double2 *>(vbase + (int64_t)g.row[c] * p.MD));
                acc0 = fma(w[c], v.x, acc0);
                acc1 = fma(w[c], v.y, acc1);
            }
        }
    }
    double *out = reinterpret_cast<double *>(p.out);
    double *o = out + tr.bqm * p.D + 2 * r;
    if (in_tensor(p, out, o, 2, n_out(p))) *reinterpret_cast<double2 *>(o) = make_double2(acc0, acc1);
}

__device__ __forceinline__ void red_add_f64(double *p, double v) {
    asm volatile("red.global.add.f64 [%0], %1;" ::"l"(p), "d"(v) : "memory");
}

// Backward. The LPG lanes of a group complete the four corner dot products
// with an xor butterfly, so all 32 lanes stay until the end; a lane of a group
// without a query works on zeros and writes nothing.
template <int LPG, bool SOFTMAX>
__global__ void __launch_bounds__(kThreads) msda_backward_f64_kernel(const Params p) {
    __shared__ LevelTable lt;
    load_level_table(lt, p);
    __syncthreads();
    const int lane = threadIdx.x & 31, r = lane % LPG;
    const int64_t t = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LPG;
    if (((int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31)) / LPG >= p.triples) return;  // whole warp
    bool valid;
    Triple tr = group_triple(p, t, valid);
    const int64_t bqm = valid ? tr.bqm : 0;
    const double *loc0 = reinterpret_cast<const double *>(p.loc);
    const double *attn0 = reinterpret_cast<const double *>(p.attn);
    const double *value = reinterpret_cast<const double *>(p.value);
    double *gv0 = reinterpret_cast<double *>(p.grad_value);
    double *gloc0 = reinterpret_cast<double *>(p.grad_loc);
    double *gattn0 = reinterpret_cast<double *>(p.grad_attn);
    const double *gout = reinterpret_cast<const double *>(p.grad_out);
    const double *loc = loc0 + bqm * p.LK * 2;
    const double *attn = attn0 + bqm * p.LK;
    const int64_t head = ((int64_t)tr.b * p.S * p.M + tr.m) * p.D + 2 * r;
    const double *vbase = value + head;
    double *gvbase = gv0 + head;
    double *gloc = gloc0 + bqm * p.LK * 2;
    double *gattn = gattn0 + bqm * p.LK;
    const int64_t nv = n_value(p), ns = n_samples(p);
    // a group's per-sample rows are contiguous blocks of L*K entries
    if (valid && (!in_tensor(p, loc0, loc, 2 * (int64_t)p.LK, 2 * ns) ||
                  !in_tensor(p, attn0, attn, p.LK, ns) ||
                  !in_tensor(p, gloc0, gloc, 2 * (int64_t)p.LK, 2 * ns) ||
                  !in_tensor(p, gattn0, gattn, p.LK, ns) ||
                  !in_tensor(p, gout, gout + tr.bqm * p.D + 2 * r, 2, n_out(p))))
        valid = false;
    double g0 = 0.0, g1 = 0.0;
    if (valid) {
        const double2 g = __ldg(reinterpret_cast<const double2 *>(gout + tr.bqm * p.D + 2 * r));
        g0 = g.x;
        g1 = g.y;
    }
    double mx = 0.0, inv = 1.0, sum_ag = 0.0;
    if (SOFTMAX && valid) softmax64(attn, p.LK, mx, inv);
    for (int idx = 0; idx < p.LK; ++idx) {
        const int l = level_of(idx, p.inv_K);
        double a = 0.0;
        Geom64 g = {};
        if (valid) {
            a = SOFTMAX ? exp(attn[idx] - mx) * inv : attn[idx];
            sample_geometry64(g, loc[2 * idx], loc[2 * idx + 1], lt, l);
        }
        const double hx = 1.0 - g.lx, hy = 1.0 - g.ly;
        const bool vc[4] = {g.vx0 && g.vy0, g.vx1 && g.vy0, g.vx0 && g.vy1, g.vx1 && g.vy1};
        const double wb[4] = {hx * hy, g.lx * hy, hx * g.ly, g.lx * g.ly};
        double s[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            s[c] = 0.0;
            if (vc[c] && in_tensor(p, value, vbase + (int64_t)g.row[c] * p.MD, 2, nv) &&
                in_tensor(p, (const double *)gv0, (const double *)gvbase + (int64_t)g.row[c] * p.MD,
                          2, nv)) {
                const int64_t off = (int64_t)g.row[c] * p.MD;
                const double2 v = __ldg(reinterpret_cast<const double2 *>(vbase + off));
                s[c] = fma(g0, v.x, g1 * v.y);
                const double aw = a * wb[c];
                if (aw != 0.0) {
                    red_add_f64(gvbase + off, aw * g0);
                    red_add_f64(gvbase + off + 1, aw * g1);
                }
            }
        }
#pragma unroll
        for (int off = LPG / 2; off > 0; off >>= 1) {
#pragma unroll
            for (int c = 0; c < 4; ++c) s[c] += __shfl_xor_sync(0xffffffffu, s[c], off);
        }
        if (valid && r == 0) {
            const double ga = wb[0] * s[0] + wb[1] * s[1] + wb[2] * s[2] + wb[3] * s[3];
            const double dlx = hy * (s[1] - s[0]) + g.ly * (s[3] - s[2]);
            const double dly = hx * (s[2] - s[0]) + g.lx * (s[3] - s[1]);
            gloc[2 * idx] = a * (double)lt.Wf[l] * dlx;
            gloc[2 * idx + 1] = a * (double)lt.Hf[l] * dly;
            gattn[idx] = ga;          // d loss / d weight; rescaled below for the softmax variant
            sum_ag += a * ga;
        }
    }
    if (SOFTMAX && valid && r == 0) {
        for (int idx = 0; idx < p.LK; ++idx) {
            const double a = exp(attn[idx] - mx) * inv;
            gattn[idx] = a * (gattn[idx] - sum_ag);
        }
    }
}

template <int LPG>
__global__ void __launch_bounds__(kThreads) msda_corners_f64_kernel(const Params p, int32_t *rows) {
    __shared__ LevelTable lt;
    load_level_table(lt, p);
    __syncthreads();
    const int64_t n = p.triples * p.LK;
    const double *loc = reinterpret_cast<const double *>(p.loc);
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n;
         s += (int64_t)gridDim.x * blockDim.x) {
        const int l = level_of((int)(s % p.LK), p.inv_K);
        if (!in_tensor(p, loc, loc + 2 * s, 2, 2 * n) || !in_tensor(p, rows, rows + 4 * s, 4, 4 * n))
            continue;
        Geom64 g;
        sample_geometry64(g, loc[2 * s], loc[2 * s + 1], lt, l);
        reinterpret_cast<int4 *>(rows)[s] =
            make_int4((g.vx0 && g.vy0) ? g.row[0] : -1, (g.vx1 && g.vy0) ? g.row[1] : -1,
                      (g.vx0 && g.vy1) ? g.row[2] : -1, (g.vx1 && g.vy1) ? g.row[3] : -1);
    }
}

static int64_t f64_blocks(const Params &p, int lpg) {
    return (p.triples * lpg + kThreads - 1) / kThreads;
}

#define MSDA_F64_LPG_SWITCH(LPG_VAR, CALL)                                  \
    switch (LPG_VAR) {                                                      \
        case 1: CALL(1); break;                                             \
        case 2: CALL(2); break;                                             \
        case 4: CALL(4); break;                                             \
        case 8: CALL(8); break;                                             \
        case 16: CALL(16); break;                                           \
        case 32: CALL(32); break;                                           \
        default: return cudaErrorInvalidValue;                              \
    }

cudaError_t launch_forward_f64(const Params &p, int lpg, bool softmax, cudaStream_t stream) {
    const int64_t blocks = f64_blocks(p, lpg);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
#define FWD(N)                                                                               \
    if (softmax) msda_forward_f64_kernel<N, true><<<(unsigned)blocks, kThreads, 0, stream>>>(p); \
    else msda_forward_f64_kernel<N, false><<<(unsigned)blocks, kThreads, 0, stream>>>(p)
    MSDA_F64_LPG_SWITCH(lpg, FWD)
#undef FWD
    return cudaGetLastError();
}

cudaError_t launch_backward_f64(const Params &p, int lpg, bool softmax, cudaStream_t stream) {
    const int64_t blocks = f64_blocks(p, lpg);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
#define BWD(N)                                                                                \
    if (softmax) msda_backward_f64_kernel<N, true><<<(unsigned)blocks, kThreads, 0, stream>>>(p); \
    else msda_backward_f64_kernel<N, false><<<(unsigned)blocks, kThreads, 0, stream>>>(p)
    MSDA_F64_LPG_SWITCH(lpg, BWD)
#undef BWD
    return cudaGetLastError();
}

cudaError_t launch_corners_f64(const Params &p, int32_t *rows, cudaStream_t stream) {
    const int64_t n = p.triples * p.LK;
    const int64_t want = (n + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(want < 4096 ? want : 4096);
    if (grid == 0) return cudaSuccess;
    msda_corners_f64_kernel<1><<<grid, kThreads, 0, stream>>>(p, rows);
    return cudaGetLastError();
}

}  // namespace msda
