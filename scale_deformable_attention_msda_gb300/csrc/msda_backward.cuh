// MSDA backward on sm_103a.
//
// The three gradients named by the msda-triton course index, chapter 5 ("The
// backward kernel"), derived from the forward by the chain rule. For a sample
// with attention weight a, bilinear weights w_c and g = grad_out[b,q,m,:]:
//   s_c        = <g, value[corner c]>            (0 for a corner off the map)
//   grad_attn  = sum_c w_c s_c
//   grad_value[corner c] += a w_c g              (vector atomics, relaxed)
//   grad_loc_x = a W ((1-ly)(s_01 - s_00) + ly (s_11 - s_10))
//   grad_loc_y = a H ((1-lx)(s_10 - s_00) + lx (s_11 - s_01))
//
// Work split as in the forward: a group of LPG lanes owns one (b,q,m), each
// lane 16 bytes of its D channels (8 bytes in NARROW mode, below). Per chunk
// of samples a warp
//  1. prepares descriptors (lane per sample): corner rows, a*w_c for the
//     scatter, and keeps lx, ly, a, W, H and the corner mask in registers;
//  2. gathers (group per sample): four corner loads of the lane's bytes,
//     per-lane partial dot products with g, vector atomic adds of a*w_c*g
//     into grad_value, and an xor-butterfly that completes the four dot
//     products across the group;
//  3. finishes (lane per sample, the lane that prepared it): grad_attn and
//     grad_loc from the four dot products, one coalesced store each.
// No per-sample buffer exists outside shared memory (deformops README,
// "Zero-buffer kernels").
//
// SPL (small problems, see choose_split): 2^s groups of a warp share one
// query-head and take every 2^s-th of its samples. Samples are independent in
// the backward, so nothing is reduced across the groups except, with the
// softmax, the sum over the query-head's samples of a * d loss / d a.
//
// Accumulation of grad_value (Efficient-MSDA summary page, "The backward pass
// is an atomics problem"; deformops README, "Backend selection"): fp32 data
// uses red.global.add.v4.f32; 16-bit data either adds natively with
// red.global.add.noftz.v4.{bf16x2,f16x2} (8 channels per instruction) or adds
// in fp32 into a workspace that a second kernel rounds into grad_value.
#pragma once

#include <type_traits>

#include "msda_common.cuh"

namespace msda {

// w * (x[i], x[i+1]) for i = 0, 2, ..., 2N-2 in packed fp32 pairs (one
// mul.rn.f32x2 per pair; products rounded as the scalar multiplies are).
template <int N> __device__ __forceinline__ void scale_pairs(float *t, float w, const float *x) {
    const float2 w2 = make_float2(w, w);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float2 y = __fmul2_rn(w2, make_float2(x[2 * i], x[2 * i + 1]));
        t[2 * i] = y.x;
        t[2 * i + 1] = y.y;
    }
}

__device__ __forceinline__ void red_add_v4_f32(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ void red_add_v4_bf16x2(void *p, uint4 v) {
    asm volatile("red.global.add.noftz.v4.bf16x2 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void red_add_v4_f16x2(void *p, uint4 v) {
    asm volatile("red.global.add.noftz.v4.f16x2 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// One lane's share of grad_value[row, 0..D) += w * g, where `row` points at
// the D channels of one head at one corner pixel. Each lane holds the grad_out
// channels it scatters (sc, loaded once per query-head by load_scatter_g), and
// every instruction of the group covers whole 32-byte sectors:
//  - fp32 data: lane r adds channels [4r, 4r+4); LPG lanes cover D floats.
//  - 16-bit data, fp32 workspace: two 16-byte adds per lane, channels
//    [4r, 4r+4) then [4 LPG + 4r, ...), so each instruction writes 16 LPG
//    contiguous bytes per group (a lane's gathered 8 channels would leave
//    every other 16 bytes of a sector untouched).
//  - 16-bit data, native: lane r adds its 8 channels [8r, 8r+8) in one
//    bf16x2/f16x2 instruction.
template <typename T, bool F32ACC, int LPG> struct Scatter;
template <int LPG> struct Scatter<float, true, LPG> {
    using Acc = float;
    static constexpr int NSC = 4;
    static __device__ __forceinline__ void add(float *row, float w, const float *sc, int r) {
        float t[4];
        scale_pairs<2>(t, w, sc);
        red_add_v4_f32(row + 4 * r, t[0], t[1], t[2], t[3]);
    }
};
template <typename T, int LPG> struct Scatter<T, true, LPG> {
    using Acc = float;
    static constexpr int NSC = 8;
    static __device__ __forceinline__ void add(float *row, float w, const float *sc, int r) {
        float t[8];
        scale_pairs<4>(t, w, sc);
        red_add_v4_f32(row + 4 * r, t[0], t[1], t[2], t[3]);
        red_add_v4_f32(row + 4 * LPG + 4 * r, t[4], t[5], t[6], t[7]);
    }
};
template <int LPG> struct Scatter<__nv_bfloat16, false, LPG> {
    using Acc = __nv_bfloat16;
    static constexpr int NSC = 8;
    static __device__ __forceinline__ void add(__nv_bfloat16 *row, float w, const float *sc, int r) {
        float t[8];
        scale_pairs<4>(t, w, sc);
        red_add_v4_bf16x2(row + 8 * r, pack16<__nv_bfloat16>(t));
    }
};
template <int LPG> struct Scatter<__half, false, LPG> {
    using Acc = __half;
    static constexpr int NSC = 8;
    static __device__ __forceinline__ void add(__half *row, float w, const float *sc, int r) {
        float t[8];
        scale_pairs<4>(t, w, sc);
        red_add_v4_f16x2(row + 8 * r, pack16<__half>(t));
    }
};

// 16-bit data accumulated in the scaled fp16 workspace (MSDA_ACC_FP16_BUFFER):
// lane r adds its 8 channels, with the call's scale folded into w by the
// kernel, in one red.noftz.v4.f16x2 (64-byte groups per query-head).
template <int LPG> struct ScatterF16 {
    using Acc = __half;
    static constexpr int NSC = 8;
    static __device__ __forceinline__ void add(__half *row, float w, const float *sc, int r) {
        float t[8];
        scale_pairs<4>(t, w, sc);
        red_add_v4_f16x2(row + 8 * r, pack16<__half>(t));
    }
};

// The scale 2^k of the fp16 workspace. Every element of grad_value sums, over
// the samples that reach it, |a| * w * |g| with bilinear weight w <= 1 and one
// sample per (q, l, k) at most, so |sum| <= max|g| * Q * A, where A = max over
// query-heads of sum_{l,k} |a| <= L K max|a| (A = 1 for the softmax variant,
// whose weights are probabilities). With each factor x < 2^e(x), k = 15 -
// sum of the e's puts that bound below 2^15, under fp16's largest finite
// value, 65504 (and, for normal inputs, at or above 2^11), for any bound up
// to 2^141. Inside fp16's normal range the rounding of a sum does not depend
// on k; a sum below 2^-25 of the bound falls into fp16's subnormals and keeps
// fewer bits. The kernel scales each corner weight first (w 2^k, then times
// g), so k also stays below 128 - e(max w) (max w <= max|a|, or 1 for softmax
// weights): w 2^k is finite even when tiny gradients alone would ask for a
// larger k. Integer arithmetic only: every thread of every block evaluates
// it. A zero or non-finite maximum gives k = 0.
__device__ __forceinline__ int exp_above(float x) {      // x < 2^e for 0 < x < inf
    return (int)((__float_as_uint(x) >> 23) & 0xffu) - 126;
}
__device__ __forceinline__ int exp_above(int64_t x) {    // x < 2^e for x >= 1
    return 64 - __clzll((long long)x);
}
__device__ __forceinline__ float f16_scale_of(float gmax, float amax, bool have_amax, int64_t Q,
                                              int64_t LK) {
    const bool finite = gmax > 0.0f && gmax <= 3.4028235e38f &&
                        (!have_amax || (amax > 0.0f && amax <= 3.4028235e38f));
    int e = exp_above(gmax) + exp_above(Q < 1 ? (int64_t)1 : Q);
    if (have_amax) e += exp_above(amax) + exp_above(LK < 1 ? (int64_t)1 : LK);
    const int kw = 127 - (have_amax ? exp_above(amax) : 1);   // w 2^k < 2^127
    const int k = finite ? min(max(min(15 - e, kw), -126), 126) : 0;
    return __uint_as_float((uint32_t)(k + 127) << 23);  // 2^k, a normal float
}

// Each warp's maximum over the prepare pass's block maxima (at most
// 2 * kF16MaxBlocks values, read in flight with the level table's) into s[warp]
// (of |grad_out|) and s[WPB + warp] (of |attention weight|), WPB warps a block.
template <int WPB> __device__ __forceinline__ void f16_warp_maxima(const Params &p, float *s) {
    const int n = p.f16_nmax, total = p.f16_amax ? 2 * n : n;
    float m = 0.0f, ma = 0.0f;
    for (int j = threadIdx.x; j < total; j += WPB * 32) {
        const float v = p.f16_max[j];
        if (j < n) m = fmaxf(m, v); else ma = fmaxf(ma, v);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, off));
    }
    if ((threadIdx.x & 31) == 0) {
        s[threadIdx.x >> 5] = m;
        s[WPB + (threadIdx.x >> 5)] = ma;
    }
}

// After a __syncthreads that follows f16_warp_maxima: the call's 2^k; block 0
// stores (2^k, 2^-k) for the finish pass.
template <int WPB> __device__ __forceinline__ float f16_block_scale(const Params &p, const float *s) {
    float m = 0.0f, ma = 0.0f;
#pragma unroll
    for (int w = 0; w < WPB; ++w) {
        m = fmaxf(m, s[w]);
        ma = fmaxf(ma, s[WPB + w]);
    }
    const float scale = f16_scale_of(m, ma, p.f16_amax != 0, p.Q, p.LK);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        p.f16_scale[0] = scale;
        p.f16_scale[1] = __uint_as_float((uint32_t)(254 - ((__float_as_uint(scale) >> 23) & 0xffu))
                                         << 23);  // 2^-k
    }
    return scale;
}

// 8 bytes of T (4 channels) as fp32.
template <typename T> __device__ __forceinline__ void load4(float *v, const T *p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    float x[8];
    unpack16<T>(x, make_uint4(u.x, u.y, 0u, 0u));
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = x[i];
}

// The grad_out channels lane r scatters (see Scatter).
template <typename T, bool F32ACC, int LPG>
__device__ __forceinline__ void load_scatter_g(float *sc, const float *go, const T *grow, int r) {
    if constexpr (F32ACC && sizeof(T) == 2) {
        load4<T>(sc, grow + 4 * r);
        load4<T>(sc + 4, grow + 4 * LPG + 4 * r);
    } else {
#pragma unroll
        for (int i = 0; i < Vec16<T>::N; ++i) sc[i] = go[i];
    }
}

template <typename T> __device__ __forceinline__ void store_xy(T *p, float x, float y);
template <> __device__ __forceinline__ void store_xy<float>(float *p, float x, float y) {
    *reinterpret_cast<float2 *>(p) = make_float2(x, y);
}
template <> __device__ __forceinline__ void store_xy<__nv_bfloat16>(__nv_bfloat16 *p, float x, float y) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x, y);
}
template <> __device__ __forceinline__ void store_xy<__half>(__half *p, float x, float y) {
    *reinterpret_cast<__half2 *>(p) = __floats2half2_rn(x, y);
}

// Per-warp fp32 slots that hold d loss / d weight of every sample of the
// warp's query-heads until the softmax backward can combine them: GPW
// query-heads x at most kSoftmaxSlots / GPW samples each.
constexpr int kSoftmaxSlots = 512;

// A lane's share of one corner vector: 16 bytes, or 8 bytes in NARROW mode.
template <typename T, int NB> __device__ __forceinline__ uint4 ldg_lane(const T *p) {
    if constexpr (NB == 16) {
        return ldg16(p);
    } else {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        return make_uint4(u.x, u.y, 0u, 0u);
    }
}
template <typename T, int N> __device__ __forceinline__ void unpack_n(float *v, uint4 raw) {
    float t[Vec16<T>::N];
    unpack16<T>(t, raw);
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = t[i];
}

// Corners of one query-head that land on the same value row add the same
// grad_out vector, so their weights can be summed before the scatter: one add
// instead of several. Points of one head and level sit a few pixels apart and
// often share corner pixels (about one corner in ten for offsets of 2 px).
// The P samples compared are those of the lanes pj ^ d (d < P) of one group
// in one round of phase 1, an aligned block of P consecutive samples (one
// level when K = P). Of the live entries (nonzero weight) with one row, the
// one of the lowest pj takes the sum of their weights and the others get
// weight 0, which the scatter skips; an entry's corners have distinct rows.
template <int P, int GPW>
__device__ __forceinline__ void merge_shared_rows(float4 &w, const int4 &o, int pj) {
    const float wc[4] = {w.x, w.y, w.z, w.w};
    const int oc[4] = {o.x, o.y, o.z, o.w};
    float sum[4] = {wc[0], wc[1], wc[2], wc[3]};
    bool dup[4] = {false, false, false, false};
#pragma unroll
    for (int d = 1; d < P; ++d) {
        const int po[4] = {__shfl_xor_sync(0xffffffffu, o.x, d * GPW),
                           __shfl_xor_sync(0xffffffffu, o.y, d * GPW),
                           __shfl_xor_sync(0xffffffffu, o.z, d * GPW),
                           __shfl_xor_sync(0xffffffffu, o.w, d * GPW)};
        const float pw[4] = {__shfl_xor_sync(0xffffffffu, w.x, d * GPW),
                             __shfl_xor_sync(0xffffffffu, w.y, d * GPW),
                             __shfl_xor_sync(0xffffffffu, w.z, d * GPW),
                             __shfl_xor_sync(0xffffffffu, w.w, d * GPW)};
        const bool lower = (pj ^ d) < pj;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (pw[e] == 0.0f) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (po[e] != oc[c]) continue;
                if (lower) dup[c] = true;
                else sum[c] += pw[e];
            }
        }
    }
    w.x = (wc[0] != 0.0f && !dup[0]) ? sum[0] : 0.0f;
    w.y = (wc[1] != 0.0f && !dup[1]) ? sum[1] : 0.0f;
    w.z = (wc[2] != 0.0f && !dup[2]) ? sum[2] : 0.0f;
    w.w = (wc[3] != 0.0f && !dup[3]) ? sum[3] : 0.0f;
}

// NARROW (16-bit data with the fp32 workspace): 8 lanes of 8 bytes per
// D = 32 query-head instead of 4 lanes of 16 bytes, so that each lane's
// 16-byte fp32 add covers its 4 channels and one add instruction writes a
// whole 128-byte workspace row per query-head (L2 reduces 128-byte groups
// about 1.2x faster than 64-byte ones); the extra per-lane work fits in the
// kernel's idle issue slots.
// Every instantiation is held to 4 resident blocks per SM (64 registers).
// The narrow ones gather two samples at a time and fit; the 16-byte-lane
// ones (fp32 data, native 16-bit adds) gather one at a time to fit. Measured
// on the encoder (GB300): the narrow softmax backward would take 74
// registers and run at 3 blocks (436.9 against 422.5 us); native bf16
// accumulation took 96 registers at 2 blocks (332 us), 80 at 3 (291 us),
// and takes 285 us here; the fp32 softmax one 461 against 449 us.
//
// F16ACC (bf16 data, MSDA_ACC_FP16_BUFFER): the 16-byte-lane kernel of native
// accumulation, adding into an fp16 workspace instead of grad_value, with every
// contribution multiplied by 2^k (f16_scale_of; each block derives it from the
// prepare pass's block maxima while it loads the level table): fp16 keeps 11
// bits where bf16 keeps 8, at the same 64 bytes per add.
//
// Warps per block: 2 for the 16-byte-lane kernels of ordinary launches, so
// that the last wave ends in smaller pieces at the same 32 resident warps per
// SM (GB300, cold, against 8-warp blocks: Mask2Former native 390.8 -> 378.5
// us, fp16 workspace 430.7 -> 421.5 us, encoder native 287.4 -> 283.3 us,
// the 4x4 contention sweep native 113.8 -> 105.6 us); the narrow
// fp32-workspace kernel (404.1 -> 408.2 us with 2) and the split launches
// keep 8.
template <bool NARROW, bool SPL> __host__ __device__ constexpr int bwd_warps() {
    return (NARROW || SPL) ? kWarpsPerBlock : 2;
}

template <typename T, int LPG, bool F32ACC, bool SOFTMAX, bool NARROW, bool SPL, bool F16ACC = false>
__global__ void __launch_bounds__(bwd_warps<NARROW, SPL>() * 32,
                                  bwd_warps<NARROW, SPL>() == 2 ? 16 : 4)
msda_backward_kernel(const Params p) {
    constexpr int WPB = bwd_warps<NARROW, SPL>();   // warps per block
    static_assert(!NARROW || (F32ACC && sizeof(T) == 2), "narrow lanes: 16-bit data, fp32 workspace");
    static_assert(!F16ACC || (!F32ACC && !NARROW && sizeof(T) == 2), "fp16 workspace: 16-bit data");
    constexpr int LB = NARROW ? 8 : 16;      // bytes of one corner vector per lane
    constexpr int VEC = LB / (int)sizeof(T);
    constexpr int GPW = 32 / LPG;
    constexpr int SPW = 64;
    constexpr int CH = SPW / GPW;
    constexpr int NP = SPW / 32;             // samples each lane prepares per chunk
    constexpr int UW = NARROW ? 2 : 1;       // samples gathered at a time
    constexpr int U = CH < UW ? CH : UW;
    using S = std::conditional_t<F16ACC, ScatterF16<LPG>, Scatter<T, F32ACC, LPG>>;
    using Acc = typename S::Acc;
    constexpr int NSC = NARROW ? VEC : S::NSC;

    __shared__ LevelTable lt;
    __shared__ float4 s_w[WPB][SPW];
    __shared__ int4 s_o[WPB][SPW];
    __shared__ float4 s_dot[WPB][SPW];
    __shared__ float s_ga[WPB][SOFTMAX ? kSoftmaxSlots : 1];
    __shared__ float s_f16max[F16ACC ? 2 * WPB : 1];
    constexpr int SLOTS = SOFTMAX ? kSoftmaxSlots / GPW : 1;   // samples per query-head

    load_level_table(lt, p);
    if constexpr (F16ACC) f16_warp_maxima<WPB>(p, s_f16max);
    __syncthreads();
    // fp16 workspace: the call's scale, folded into each corner's weight
    const float acc_scale = F16ACC ? f16_block_scale<WPB>(p, s_f16max) : 1.0f;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / LPG, r = lane % LPG;
    // sl2: log2 of the groups per query-head (0 unless SPL)
    const int sl2 = SPL ? p.split_log2 : 0;
    const int64_t t0 = ((int64_t)blockIdx.x * WPB + warp) * (GPW >> sl2);
    if (t0 >= p.triples) return;

    const int64_t t = t0 + (g >> sl2);
    const bool active = t < p.triples;
    const Triple tr = triple_of(active ? t : t0, p);
    const bool valid_q = active && tr.q >= 0 && tr.q < p.Q;
    const int64_t head = ((int64_t)tr.b * p.S * p.M + tr.m) * p.D;    // row 0 of this head
    const T *value = reinterpret_cast<const T *>(p.value);
    const T *vbase = value + head + r * VEC;
    Acc *gvbase = reinterpret_cast<Acc *>(p.grad_value);
    Acc *gvhead = gvbase + head;
    const int64_t nv = n_value(p), ns = n_samples(p);

    // grad_out of this query-head: the lane's gathered channels (for the dot
    // products) and the channels it scatters (zero for a group with no work)
    float go[VEC], sc[NSC];
    const T *gout = reinterpret_cast<const T *>(p.grad_out);
    if (valid_q && in_tensor(p, gout, gout + tr.bqm * p.D, p.D, n_out(p))) {
        const T *grow = gout + tr.bqm * p.D;
        unpack_n<T, VEC>(go, ldg_lane<T, LB>(grow + r * VEC));
        if constexpr (NARROW) {
#pragma unroll
            for (int i = 0; i < NSC; ++i) sc[i] = go[i];
        } else {
            load_scatter_g<T, F32ACC, LPG>(sc, go, grow, r);
        }
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) go[i] = 0.0f;
#pragma unroll
        for (int i = 0; i < NSC; ++i) sc[i] = 0.0f;
    }
    // phase-1/3 mapping as in the forward: slot lane + 32*i is chunk sample
    // pj + i*LPG of group pg = lane % GPW, i.e. sample ((pj + i*LPG) << sl2)
    // + psub of the chunk of query-head t0 + (pg >> sl2)
    const int pg = lane % GPW, pj = lane / GPW;
    const int psub = pg & ((1 << sl2) - 1);
    const int64_t tp = t0 + (pg >> sl2);
    bool prep_ok = tp < p.triples;
    const Triple trp = triple_of(prep_ok ? tp : t0, p);
    prep_ok = prep_ok && trp.q >= 0 && trp.q < p.Q;

    const T *loc = reinterpret_cast<const T *>(p.loc);
    const T *attn = reinterpret_cast<const T *>(p.attn);
    T *gloc = reinterpret_cast<T *>(p.grad_loc);
    T *gattn = reinterpret_cast<T *>(p.grad_attn);

    // With SOFTMAX, attn holds logits and grad_attn receives d loss / d logit:
    // a = softmax(logits), g_logit = a * (g_a - sum_j a_j g_a_j).
    SoftmaxStats sm = {0.0f, 1.0f};
    const bool logits_ok = prep_ok && in_tensor(p, attn, attn + trp.bqm * p.LK, p.LK, ns);
    if (SOFTMAX) sm = softmax_stats<T, LPG>(attn + trp.bqm * p.LK, logits_ok ? p.LK : 0, lane, sl2);
    // softmax slots of the prepared query-head: SLOTS << sl2 of them
    const int slot0 = (pg >> sl2) * (SLOTS << sl2);
    float sum_ag = 0.0f;

    for (int base = 0; base < p.LK; base += CH << sl2) {
        // ---- phase 1: descriptors, and the finishing state of each sample
        float f_lx[NP], f_ly[NP], f_a[NP], f_W[NP], f_H[NP];
        unsigned f_mask[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int idx = base + ((pj + i * LPG) << sl2) + psub;
            float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
            int4 o = make_int4(0, 0, 0, 0);
            f_lx[i] = f_ly[i] = f_a[i] = f_W[i] = f_H[i] = 0.0f;
            f_mask[i] = 0u;
            if (prep_ok && idx < p.LK) {
                const int64_t e = trp.bqm * p.LK + idx;
                const float2 xy = in_tensor(p, loc, loc + 2 * e, 2, 2 * ns)
                                      ? load_xy<T>(loc + 2 * e) : make_float2(0.f, 0.f);
                const float z = in_tensor(p, attn, attn + e, 1, ns) ? load_scalar<T>(attn + e)
                                                                     : 0.0f;
                const float a = SOFTMAX ? softmax_weight(z, sm) : z;
                const int l = level_of(idx, p.inv_K);
                SampleGeom sg;
                sample_geometry(sg, xy.x, xy.y, lt, l);
                const unsigned m = (sg.vx0 && sg.vy0 ? 1u : 0u) | (sg.vx1 && sg.vy0 ? 2u : 0u) |
                                   (sg.vx0 && sg.vy1 ? 4u : 0u) | (sg.vx1 && sg.vy1 ? 8u : 0u);
                const float hx = 1.0f - sg.lx, hy = 1.0f - sg.ly;
                const float ahy = a * hy, aly = a * sg.ly;
                w.x = (m & 1u) ? ahy * hx : 0.0f;
                w.y = (m & 2u) ? ahy * sg.lx : 0.0f;
                w.z = (m & 4u) ? aly * hx : 0.0f;
                w.w = (m & 8u) ? aly * sg.lx : 0.0f;
                o = make_int4(sg.row[0] * p.MD, sg.row[1] * p.MD, sg.row[2] * p.MD,
                              sg.row[3] * p.MD);
                f_lx[i] = sg.lx;
                f_ly[i] = sg.ly;
                f_a[i] = a;
                f_W[i] = lt.Wf[l];
                f_H[i] = lt.Hf[l];
                f_mask[i] = m;
            }
            merge_shared_rows<(LPG < 4 ? LPG : 4), GPW>(w, o, pj);
            s_w[warp][lane + 32 * i] = w;
            s_o[warp][lane + 32 * i] = o;
        }
        __syncwarp();

        // ---- phase 2: gather, dot products, scatter
        const int n = min(CH, (p.LK - base + (1 << sl2) - 1) >> sl2);
        for (int j = 0; j < n; j += U) {
            float4 w[U];
            int4 o[U];
            uint4 v[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                w[u] = s_w[warp][(j + u) * GPW + g];
                o[u] = s_o[warp][(j + u) * GPW + g];
                const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
                if (SPL && j + u >= n) {   // an empty slot: zero weights, nothing to load
                    v[u][0] = v[u][1] = v[u][2] = v[u][3] = zero;
                    continue;
                }
                v[u][0] = in_tensor(p, value, vbase + o[u].x, VEC, nv)
                              ? ldg_lane<T, LB>(vbase + o[u].x) : zero;
                v[u][1] = in_tensor(p, value, vbase + o[u].y, VEC, nv)
                              ? ldg_lane<T, LB>(vbase + o[u].y) : zero;
                v[u][2] = in_tensor(p, value, vbase + o[u].z, VEC, nv)
                              ? ldg_lane<T, LB>(vbase + o[u].z) : zero;
                v[u][3] = in_tensor(p, value, vbase + o[u].w, VEC, nv)
                              ? ldg_lane<T, LB>(vbase + o[u].w) : zero;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float d[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float x[VEC];
                    unpack_n<T, VEC>(x, v[u][c]);
                    if constexpr (NARROW) {
                        float acc = 0.0f;
#pragma unroll
                        for (int i = 0; i < VEC; ++i) acc = fmaf(go[i], x[i], acc);
                        d[c] = acc;
                    } else {   // packed fp32 pairs: even and odd channels summed apart
                        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int i = 0; i < VEC; i += 2)
                            acc = __ffma2_rn(make_float2(go[i], go[i + 1]),
                                             make_float2(x[i], x[i + 1]), acc);
                        d[c] = acc.x + acc.y;
                    }
                }
                const float wc[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                const int oc[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // the group adds within the D channels of one head's row
                    if (wc[c] == 0.0f || !in_tensor(p, gvbase, gvhead + oc[c], p.D, nv)) continue;
                    if constexpr (NARROW) {
                        float *dst = reinterpret_cast<float *>(gvhead) + oc[c] + 4 * r;
                        red_add_v4_f32(dst, wc[c] * sc[0], wc[c] * sc[1], wc[c] * sc[2], wc[c] * sc[3]);
                    } else {
                        S::add(gvhead + oc[c], F16ACC ? wc[c] * acc_scale : wc[c], sc, r);
                    }
                }
#pragma unroll
                for (int off = LPG / 2; off > 0; off >>= 1) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) d[c] += __shfl_xor_sync(0xffffffffu, d[c], off);
                }
                if (r == 0) s_dot[warp][(j + u) * GPW + g] = make_float4(d[0], d[1], d[2], d[3]);
            }
        }
        __syncwarp();

        // ---- phase 3: grad_attn and grad_loc of the samples this lane prepared
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int idx = base + ((pj + i * LPG) << sl2) + psub;
            if (prep_ok && idx < p.LK) {
                const float4 dd = s_dot[warp][lane + 32 * i];
                const unsigned m = f_mask[i];
                const float s00 = (m & 1u) ? dd.x : 0.0f, s01 = (m & 2u) ? dd.y : 0.0f;
                const float s10 = (m & 4u) ? dd.z : 0.0f, s11 = (m & 8u) ? dd.w : 0.0f;
                const float lx = f_lx[i], ly = f_ly[i], hx = 1.0f - lx, hy = 1.0f - ly;
                const float ga = hy * (hx * s00 + lx * s01) + ly * (hx * s10 + lx * s11);
                const float dlx = hy * (s01 - s00) + ly * (s11 - s10);
                const float dly = hx * (s10 - s00) + lx * (s11 - s01);
                const int64_t e = trp.bqm * p.LK + idx;
                if (SOFTMAX) {
                    float *slot = &s_ga[warp][slot0 + idx];
                    if (in_tensor(p, &s_ga[warp][0], slot, 1, SOFTMAX ? kSoftmaxSlots : 1))
                        *slot = ga;
                    sum_ag += f_a[i] * ga;
                } else if (in_tensor(p, gattn, gattn + e, 1, ns)) {
                    gattn[e] = Elem<T>::from_f(ga);
                }
                if (in_tensor(p, gloc, gloc + 2 * e, 2, 2 * ns))
                    store_xy<T>(gloc + 2 * e, f_a[i] * f_W[i] * dlx, f_a[i] * f_H[i] * dly);
            }
        }
        __syncwarp();
    }

    if (SOFTMAX) {
        // the lanes of one query-head differ in the lane bits above GPW, and
        // with a split in the low sl2 bits
        for (int off = 1; off < (1 << sl2); off <<= 1)
            sum_ag += __shfl_xor_sync(0xffffffffu, sum_ag, off);
#pragma unroll
        for (int off = GPW; off < 32; off <<= 1) sum_ag += __shfl_xor_sync(0xffffffffu, sum_ag, off);
        __syncwarp();
        if (prep_ok) {
            for (int idx = (pj << sl2) + psub; idx < p.LK; idx += LPG << sl2) {
                const int64_t e = trp.bqm * p.LK + idx;
                if (!in_tensor(p, gattn, gattn + e, 1, ns) || !in_tensor(p, attn, attn + e, 1, ns) ||
                    !in_tensor(p, &s_ga[warp][0], &s_ga[warp][slot0 + idx], 1,
                               SOFTMAX ? kSoftmaxSlots : 1))
                    continue;
                const float a = softmax_weight(load_scalar<T>(attn + e), sm);
                gattn[e] = Elem<T>::from_f(a * (s_ga[warp][slot0 + idx] - sum_ag));
            }
        }
    }
}

template <typename T, bool F32ACC, bool SOFTMAX, bool SPL, bool F16ACC = false>
static cudaError_t launch_backward_t(const Params &p, int lpg, cudaStream_t stream) {
    // 16-bit data with the fp32 workspace: twice the lanes, 8 bytes each
    constexpr bool kNarrowable = F32ACC && sizeof(T) == 2;
    const bool narrow = kNarrowable && 2 * lpg <= 32;
    const int lanes = narrow ? 2 * lpg : lpg;
    const int64_t per_warp = (32 / lanes) >> p.split_log2;    // query-heads per warp
    const int64_t warps = (p.triples + per_warp - 1) / per_warp;
    if (warps == 0) return cudaSuccess;
    // blocks of bwd_warps<NAR, SPL>() warps
#define MSDA_BWD(N, NAR)                                                                          \
    do {                                                                                          \
        constexpr int wpb = bwd_warps<NAR, SPL>();                                                \
        const int64_t blocks = (warps + wpb - 1) / wpb;                                           \
        if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;                           \
        msda_backward_kernel<T, N, F32ACC, SOFTMAX, NAR, SPL, F16ACC>                             \
            <<<dim3((unsigned)blocks), wpb * 32, 0, stream>>>(p);                                 \
    } while (0)
    if constexpr (kNarrowable) {
        if (narrow) {
            switch (lanes) {
                case 2: MSDA_BWD(2, true); break;
                case 4: MSDA_BWD(4, true); break;
                case 8: MSDA_BWD(8, true); break;
                case 16: MSDA_BWD(16, true); break;
                case 32: MSDA_BWD(32, true); break;
                default: return cudaErrorInvalidValue;
            }
            return cudaGetLastError();
        }
    }
    switch (lanes) {
        case 1: MSDA_BWD(1, false); break;
        case 2: MSDA_BWD(2, false); break;
        case 4: MSDA_BWD(4, false); break;
        case 8: MSDA_BWD(8, false); break;
        case 16: MSDA_BWD(16, false); break;
        case 32: MSDA_BWD(32, false); break;
        default: return cudaErrorInvalidValue;
    }
#undef MSDA_BWD
    return cudaGetLastError();
}

template <bool SOFTMAX, bool SPL>
static cudaError_t launch_backward_s(const Params &p, msda_dtype_t dt, bool f32acc, int lpg,
                                     cudaStream_t stream) {
    switch (dt) {
        case MSDA_F32: return launch_backward_t<float, true, SOFTMAX, SPL>(p, lpg, stream);
        case MSDA_BF16:
            return f32acc ? launch_backward_t<__nv_bfloat16, true, SOFTMAX, SPL>(p, lpg, stream)
                          : launch_backward_t<__nv_bfloat16, false, SOFTMAX, SPL>(p, lpg, stream);
        case MSDA_F16:
            return f32acc ? launch_backward_t<__half, true, SOFTMAX, SPL>(p, lpg, stream)
                          : launch_backward_t<__half, false, SOFTMAX, SPL>(p, lpg, stream);
    }
    return cudaErrorInvalidValue;
}

// bf16 data with the scaled fp16 workspace (msda_backward_f16acc.cu): the
// native kernel's lanes adding fp16; p.split_log2 already chosen.
template <bool SOFTMAX, bool SPL>
static cudaError_t launch_backward_f16acc_s(const Params &p, int lpg, cudaStream_t stream) {
    return launch_backward_t<__nv_bfloat16, false, SOFTMAX, SPL, true>(p, lpg, stream);
}
cudaError_t launch_backward_f16acc(const Params &p, int lpg, bool softmax, cudaStream_t stream);

// The split instantiations (msda_backward_split.cu), compiled apart so that
// the two halves build in parallel.
cudaError_t launch_backward_split(const Params &p, msda_dtype_t dt, bool f32acc, int lpg,
                                  bool softmax, cudaStream_t stream);

}  // namespace msda
