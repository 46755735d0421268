// Device-side building blocks shared by the MSDA kernels (sm_103a).
//
// Coordinate conventions follow the msda-triton course, ch. 1 "Deformable
// attention, from scratch", section "Bilinear interpolation": pixel
// x = loc_x*W - 0.5 (grid_sample align_corners=False), corners of
// (floor(x), floor(y)) weighted by the fractional parts, zero outside the map.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msda.h"

namespace msda {

constexpr int kMaxLevels = 16;
constexpr int kWarpsPerBlock = 8;
constexpr int kThreads = kWarpsPerBlock * 32;
// The scaled fp16 workspace (MSDA_ACC_FP16_BUFFER) is n halfs followed by a
// tail of kF16TailBytes: per-block maxima of |grad_out| and of |attention
// weight| (kF16MaxBlocks floats each), then the pair (2^k, 2^-k).
constexpr int kF16MaxBlocks = 152;
constexpr size_t kF16TailBytes = 20480;
static_assert((2 * kF16MaxBlocks + 2) * sizeof(float) <= kF16TailBytes, "fp16 workspace tail");

// Everything a kernel needs, passed by value.
struct Params {
    const void *value;
    const int64_t *shapes;
    const int64_t *starts;
    const void *loc;
    const void *attn;
    const int32_t *order;  // NULL: linear dispatch
    const void *grad_out;
    void *out;             // forward output
    void *grad_value;      // fp32 or fp16 workspace, or the 16-bit/fp32 grad_value
    // fp16 workspace: per-block maxima of |grad_out| (f16_nmax of them, then as
    // many of |attention weight| when f16_amax), and where block 0 of the
    // backward stores the call's (2^k, 2^-k) for the finish pass
    const float *f16_max;
    float *f16_scale;
    int f16_nmax, f16_amax;
    void *grad_loc;
    void *grad_attn;
    int B, S, Q, M, D, L, K;
    int LK;                // L*K samples per (b,q,m)
    int MD;                // M*D elements per value row
    float inv_K;           // 1/K, for level = floor((idx + 0.5) / K)
    int64_t triples;       // B*Q*M
    unsigned *err;         // checked build: device word of range faults (see in_tensor)
    int split_log2;        // log2 of the lane groups sharing one (b,q,m); -1 before
                           // the launch chooses it (see choose_split)
};

// Sample split for small problems. With one group of lanes per (b, q, m), a
// problem of few query-heads (a detector decoder: B*Q*M = 4,800) fills a
// fraction of the SMs and each group walks its L*K samples one after another.
// Such a problem instead spreads each query-head's samples over 2^s groups of
// one warp (group sub takes samples sub, sub + 2^s, ...), and the groups
// combine what they share with shuffles. s grows while the launch stays
// within about four blocks per SM of a 152-SM GB300 and each warp keeps at
// least two query-heads, and stops at the sample count. On the decoder
// (measured on a GB300, CUDA graph of back-to-back calls): the bf16 forward
// takes 5.6 us at s = 2 against 6.7 us unsplit, the backward's accumulate
// step 10.4 against 10.9 us at s = 1; one query-head per warp was slower in
// both (7.7 and 13.3 us). forced >= 0 (msda_set_sample_split) replaces the
// size rule and may go down to one query-head per warp.
inline int choose_split(int64_t triples, int gpw, int LK, int forced) {
    constexpr int64_t kTargetBlocks = 152 * 4;
    const int max_groups = forced >= 0 ? gpw : gpw / 2;
    int s = 0;
    for (;;) {
        const int next = 2 << s;
        if (next > max_groups || next > LK || next > 8) break;
        if (forced >= 0) {
            if (s >= forced) break;
        } else {
            const int64_t per_warp = gpw / next;                  // query-heads per warp
            const int64_t warps = (triples + per_warp - 1) / per_warp;
            if ((warps + kWarpsPerBlock - 1) / kWarpsPerBlock > kTargetBlocks) break;
        }
        ++s;
    }
    return s;
}

// ------------------------------------------------------------ checked build
// Built with -DMSDA_CHECKED (libmsda_checked.so), every global access of the
// operator kernels is first checked against the extent of the tensor it
// belongs to:
// an access that would leave it is skipped (a load yields zeros) and bit 0 of
// the device word p.err is set, which msda_device_check reads and clears.
// No access is ever made outside a tensor and nothing traps. In the normal
// build the check is the constant true and compiles away.
#ifdef MSDA_CHECKED
template <typename E>
__device__ __forceinline__ bool in_tensor(const Params &p, const E *base, const E *at, int64_t n,
                                          int64_t extent) {
    const int64_t off = at - base;
    const bool ok = base != nullptr && off >= 0 && n >= 0 && off <= extent - n;
    if (!ok && p.err) atomicOr(p.err, 1u);
    return ok;
}
#else
template <typename E>
__device__ __forceinline__ constexpr bool in_tensor(const Params &, const E *, const E *, int64_t,
                                                    int64_t) {
    return true;
}
#endif
// element counts of the tensors the kernels touch
__device__ __forceinline__ int64_t n_value(const Params &p) {
    return (int64_t)p.B * p.S * p.M * p.D;
}
__device__ __forceinline__ int64_t n_samples(const Params &p) { return p.triples * p.LK; }
__device__ __forceinline__ int64_t n_out(const Params &p) { return p.triples * p.D; }

// Level table in shared memory. An invalid level gets W = H = -2 so that the
// range test of every sample in it fails.
struct LevelTable {
    float Wf[kMaxLevels], Hf[kMaxLevels];
    int W[kMaxLevels], start[kMaxLevels];
};

__device__ __forceinline__ void load_level_table(LevelTable &lt, const Params &p) {
    for (int l = threadIdx.x; l < p.L; l += blockDim.x) {
        int64_t H = p.shapes[2 * l], W = p.shapes[2 * l + 1], s0 = p.starts[l];
        bool ok = H >= 1 && W >= 1 && H < (1 << 22) && W < (1 << 22) && s0 >= 0 &&
                  s0 + H * W <= (int64_t)p.S;
        lt.Wf[l] = ok ? (float)W : -2.0f;
        lt.Hf[l] = ok ? (float)H : -2.0f;
        lt.W[l] = ok ? (int)W : 1;
        lt.start[l] = ok ? (int)s0 : 0;
    }
}

// ---------------------------------------------------------------- scalars

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};

// A (x, y) location pair, loaded in one access.
template <typename T> __device__ __forceinline__ float2 load_xy(const T *p);
template <> __device__ __forceinline__ float2 load_xy<float>(const float *p) {
    return __ldg(reinterpret_cast<const float2 *>(p));
}
template <> __device__ __forceinline__ float2 load_xy<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat1622float2(__ldg(reinterpret_cast<const __nv_bfloat162 *>(p)));
}
template <> __device__ __forceinline__ float2 load_xy<__half>(const __half *p) {
    return __half22float2(__ldg(reinterpret_cast<const __half2 *>(p)));
}

template <typename T> __device__ __forceinline__ float load_scalar(const T *p) {
    return Elem<T>::to_f(p[0]);
}
template <> __device__ __forceinline__ float load_scalar<float>(const float *p) { return __ldg(p); }

// ------------------------------------------------------ 16-byte vectors
// VEC channels per 16 bytes: 4 for fp32, 8 for 16-bit types.

template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
};

__device__ __forceinline__ uint4 ldg16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// acc[i] += w * v[i] over the 16 bytes in `raw`.
template <typename T> __device__ __forceinline__ void fma16(float *acc, float w, uint4 raw);
template <> __device__ __forceinline__ void fma16<float>(float *acc, float w, uint4 raw) {
    acc[0] = fmaf(w, __uint_as_float(raw.x), acc[0]);
    acc[1] = fmaf(w, __uint_as_float(raw.y), acc[1]);
    acc[2] = fmaf(w, __uint_as_float(raw.z), acc[2]);
    acc[3] = fmaf(w, __uint_as_float(raw.w), acc[3]);
}
// bf16 -> fp32 is exact: the 16 bits become the high half of the fp32 word.
__device__ __forceinline__ void fma_bf16x2(float *acc, float w, uint32_t u) {
    acc[0] = fmaf(w, __uint_as_float(u << 16), acc[0]);
    acc[1] = fmaf(w, __uint_as_float(u & 0xffff0000u), acc[1]);
}
template <> __device__ __forceinline__ void fma16<__nv_bfloat16>(float *acc, float w, uint4 raw) {
    fma_bf16x2(acc + 0, w, raw.x);
    fma_bf16x2(acc + 2, w, raw.y);
    fma_bf16x2(acc + 4, w, raw.z);
    fma_bf16x2(acc + 6, w, raw.w);
}
__device__ __forceinline__ void fma_f16x2(float *acc, float w, uint32_t u) {
    float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u));
    acc[0] = fmaf(w, f.x, acc[0]);
    acc[1] = fmaf(w, f.y, acc[1]);
}
template <> __device__ __forceinline__ void fma16<__half>(float *acc, float w, uint4 raw) {
    fma_f16x2(acc + 0, w, raw.x);
    fma_f16x2(acc + 2, w, raw.y);
    fma_f16x2(acc + 4, w, raw.z);
    fma_f16x2(acc + 6, w, raw.w);
}

// v[i] as fp32 for the 16 bytes in `raw`.
template <typename T> __device__ __forceinline__ void unpack16(float *v, uint4 raw) {
    float z[Vec16<T>::N];
#pragma unroll
    for (int i = 0; i < Vec16<T>::N; ++i) z[i] = 0.0f;
    fma16<T>(z, 1.0f, raw);
#pragma unroll
    for (int i = 0; i < Vec16<T>::N; ++i) v[i] = z[i];
}
template <> __device__ __forceinline__ void unpack16<float>(float *v, uint4 raw) {
    v[0] = __uint_as_float(raw.x); v[1] = __uint_as_float(raw.y);
    v[2] = __uint_as_float(raw.z); v[3] = __uint_as_float(raw.w);
}
template <> __device__ __forceinline__ void unpack16<__nv_bfloat16>(float *v, uint4 raw) {
    const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// 16 bytes of T from fp32 (round to nearest even for 16-bit types).
template <typename T> __device__ __forceinline__ uint4 pack16(const float *v);
template <> __device__ __forceinline__ uint4 pack16<float>(const float *v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
}
template <> __device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float *v) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        u[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}
template <> __device__ __forceinline__ uint4 pack16<__half>(const float *v) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        u[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}

// ------------------------------------------------------------ one sample
// Geometry of one sample at one level. `inside` is false when no corner can
// lie in the map (a coordinate that is not finite, or a full pixel or more
// outside it); then every weight is zero and every row is 0 (a safe row).
struct SampleGeom {
    bool inside;
    float lx, ly;          // fractional parts, in [0, 1]
    bool vx0, vx1, vy0, vy1;  // corner columns / rows inside the map
    int row[4];            // value rows of the corners (clamped into the map)
};

// x0 = floor(loc*n - 0.5) EXACTLY: fma with rounding toward -infinity never
// rounds across an integer (integers are representable), so floor of the
// rounded value is the floor of the real value. The fractional part is the
// single rounding of the exact real loc*n - 0.5 - x0.
__device__ __forceinline__ void sample_geometry(SampleGeom &g, float loc_x, float loc_y,
                                                const LevelTable &lt, int l) {
    const float Wf = lt.Wf[l], Hf = lt.Hf[l];
    const float xr = __fmaf_rd(loc_x, Wf, -0.5f);
    const float yr = __fmaf_rd(loc_y, Hf, -0.5f);
    // x0 in [-1, W-1] and y0 in [-1, H-1]; false for NaN and for invalid levels.
    g.inside = (xr >= -1.0f) && (xr < Wf) && (yr >= -1.0f) && (yr < Hf);
    const float x0f = g.inside ? floorf(xr) : 0.0f;
    const float y0f = g.inside ? floorf(yr) : 0.0f;
    const int x0 = (int)x0f, y0 = (int)y0f;
    const int W = lt.W[l];
    const int H = (int)Hf;
    g.lx = g.inside ? __fmaf_rn(loc_x, Wf, -0.5f - x0f) : 0.0f;
    g.ly = g.inside ? __fmaf_rn(loc_y, Hf, -0.5f - y0f) : 0.0f;
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

// Level of sample index idx in [0, L*K): floor((idx + 0.5) / K), exact for
// idx < 2^20 and K < 2^10 (the quotient is at least 0.5/K from an integer).
__device__ __forceinline__ int level_of(int idx, float inv_K) {
    return (int)(((float)idx + 0.5f) * inv_K);
}

// Softmax over the L*K logits of one query-head, for the variant that takes
// logits (deformops README, "Multi-scale deformable attention": the softmax
// method normalises the logits jointly over levels and points). The lanes
// that prepare one query-head are lane % GPW == const, so lane `lane` reads
// logits pj, pj + LPG, ... (pj = lane / GPW) and the partial max and sum are
// combined with xor shuffles over the lane bits above GPW.
struct SoftmaxStats {
    float max, inv_sum;
};

// Every lane of the warp must call this (it shuffles); a lane whose group has
// no query passes LK = 0 and gets a value it does not use.
template <typename T, int LPG>
__device__ __forceinline__ SoftmaxStats softmax_stats(const T *logits, int LK, int lane, int sl2 = 0) {
    constexpr int GPW = 32 / LPG;
    // the lanes preparing one query-head: lane bits above GPW, and with a
    // sample split (sl2 > 0) the low sl2 bits as well
    const int k = ((lane / GPW) << sl2) + (lane & ((1 << sl2) - 1)), step = LPG << sl2;
    float mx = -INFINITY;
    for (int i = k; i < LK; i += step) mx = fmaxf(mx, load_scalar<T>(logits + i));
    for (int off = 1; off < (1 << sl2); off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
#pragma unroll
    for (int off = GPW; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float sum = 0.0f;
    for (int i = k; i < LK; i += step) sum += expf(load_scalar<T>(logits + i) - mx);
    for (int off = 1; off < (1 << sl2); off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
#pragma unroll
    for (int off = GPW; off < 32; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    return SoftmaxStats{mx, 1.0f / sum};
}

__device__ __forceinline__ float softmax_weight(float logit, const SoftmaxStats &s) {
    return expf(logit - s.max) * s.inv_sum;
}

// (b, q, m) of triple t in dispatch order, and its linear (b*Q+q)*M+m index.
struct Triple {
    int b, q, m;
    int64_t bqm;
};
__device__ __forceinline__ Triple triple_of(int64_t t, const Params &p) {
    Triple r;
    const int64_t QM = (int64_t)p.Q * p.M;
    r.b = (int)(t / QM);
    const int64_t rem = t - (int64_t)r.b * QM;
    const int qs = (int)(rem / p.M);
    r.m = (int)(rem - (int64_t)qs * p.M);
    r.q = p.order ? (in_tensor(p, p.order, p.order + qs, 1, p.Q) ? p.order[qs] : -1) : qs;
    r.bqm = ((int64_t)r.b * p.Q + r.q) * p.M + r.m;
    return r;
}

}  // namespace msda
