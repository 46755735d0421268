// MSDA forward on sm_103a: gather-and-weight over L levels x K points.
//
// Work split. A "group" of LPG lanes owns one (b, q, m) query-head; each lane
// owns 16 bytes (VEC channels) of the head's D channels, so one 16-byte load
// per lane moves a whole D-channel corner vector per group. A warp holds
// GPW = 32/LPG groups (consecutive heads of one query for the detector sizes),
// and consecutive warps take consecutive queries: the query-block tiling of
// the Efficient-MSDA summary page ("Two heuristics that do not apply": the
// locality that matters comes from the tiling inside a query block).
//
// Per chunk of samples a warp runs two phases, separated by __syncwarp():
//  1. prepare: each lane turns its own samples (2 per lane) into a descriptor
//     -- four corner weights with the attention weight folded in (zero for a
//     corner outside the map) and four corner row offsets -- from coalesced
//     loads of sampling_locations and attention_weights, and stages it in
//     shared memory. The coordinate arithmetic runs once per sample instead
//     of once per lane of the group.
//  2. gather: every lane of a group reads its group's descriptors (a
//     broadcast) and issues four 16-byte loads per sample, U samples at a
//     time so that 4U loads are in flight, accumulating in fp32 registers.
// The group then writes its D output channels once (16 bytes per lane).
//
// SPL (small problems, see choose_split): 2^s groups of a warp share one
// query-head, each gathering every 2^s-th of its samples, and reduce their
// partial sums with xor shuffles across the group bits of the lane index
// before the first of them writes the output (a warp-level reduction across
// the L x K samples).
#include "msda_common.cuh"

namespace msda {

// UMAX: samples per gather step, 8 (32 loads in flight) or 4. A query-head
// whose L*K leaves a last chunk of 1 to 4 samples (L*K = 12: chunks of 8 and
// 4) takes 4, so that no step gathers empty slots.
//
// Warps per block: 2 for the ordinary launch, so that the last wave of blocks
// ends in smaller pieces (GB300, cold, against 8-warp blocks: encoder bf16
// 103.0 -> 101.0 us, fp32 148.1 -> 146.0 us, Mask2Former bf16 160.4 -> 148.1
// us); the split launches of small problems keep 8 (the decoder took 15.0 us
// with 2-warp blocks against 13.0 us). The bound of 20 resident 2-warp blocks
// per SM (at most 51 registers) makes the compiler take 48 registers in every
// instantiation with no spill; left free it chose 40 for some and spilled
// (fp32 Mask2Former 221.8 us against 213.6 us).
template <bool SPL> __host__ __device__ constexpr int fwd_warps() { return SPL ? kWarpsPerBlock : 2; }

template <typename T, int LPG, bool SOFTMAX, bool SPL, int UMAX = 8>
__global__ void __launch_bounds__(fwd_warps<SPL>() * 32, SPL ? 1 : 20)
msda_forward_kernel(const Params p) {
    constexpr int WPB = fwd_warps<SPL>();    // warps per block
    constexpr int VEC = Vec16<T>::N;
    constexpr int GPW = 32 / LPG;            // groups per warp
    constexpr int SPW = 64;                  // descriptors per warp per chunk
    constexpr int CH = SPW / GPW;            // samples per group per chunk
    constexpr int U = CH < UMAX ? CH : UMAX; // samples per gather step

    __shared__ LevelTable lt;
    __shared__ float4 s_w[WPB][SPW];
    __shared__ int4 s_o[WPB][SPW];

    load_level_table(lt, p);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / LPG, r = lane % LPG;
    // sl2: log2 of the groups per query-head (0 unless SPL)
    const int sl2 = SPL ? p.split_log2 : 0;
    // Warp task gw: the warps of one block take tasks n apart (task w*n + b
    // for warp w of block b, n = tasks / WPB), so that they do not gather the
    // same corners at the same moment; neighbouring blocks keep neighbouring
    // tasks. A bijection of the first WPB*n tasks; the rest keep their index.
    int64_t gw = (int64_t)blockIdx.x * WPB + warp;
    if (!SPL) {
        const int64_t tasks = (p.triples + GPW - 1) / GPW;
        const int64_t n = tasks / WPB;
        if (gw < n * WPB) gw = (gw % WPB) * n + gw / WPB;
    }
    const int64_t t0 = gw * (GPW >> sl2);
    if (t0 >= p.triples) return;

    // this lane's group: query-head t0 + (g >> sl2), sample subset sub
    const int sub = g & ((1 << sl2) - 1);
    const int64_t t = t0 + (g >> sl2);
    const bool active = t < p.triples;
    Triple tr = triple_of(active ? t : t0, p);
    const bool valid_q = active && tr.q >= 0 && tr.q < p.Q;
    const T *value = reinterpret_cast<const T *>(p.value);
    const T *vbase = value + ((int64_t)tr.b * p.S * p.M + tr.m) * p.D + r * VEC;
    const int64_t nv = n_value(p), ns = n_samples(p);

    // Phase 1 fills descriptor slot lane + 32*i, stored in [sample][group]
    // order, so consecutive lanes write consecutive 16-byte words (no bank
    // conflicts). Slot lane + 32*i belongs to group lane % GPW and sample
    // lane / GPW + i*LPG of the chunk: each lane prepares one triple's samples.
    // With a split, group pg's chunk sample j is sample (j << sl2) + psub of
    // its query-head's chunk.
    const int pg = lane % GPW, pj = lane / GPW;
    const int psub = pg & ((1 << sl2) - 1);
    const int64_t tp = t0 + (pg >> sl2);
    bool prep_ok = tp < p.triples;
    const Triple trp = triple_of(prep_ok ? tp : t0, p);
    prep_ok = prep_ok && trp.q >= 0 && trp.q < p.Q;

    const T *loc = reinterpret_cast<const T *>(p.loc);
    const T *attn = reinterpret_cast<const T *>(p.attn);

    // With SOFTMAX, attn holds logits: the weight of sample idx is
    // exp(logit - max) / sum over the L*K logits of the prepared query-head.
    SoftmaxStats sm = {0.0f, 1.0f};
    const bool logits_ok = prep_ok && in_tensor(p, attn, attn + trp.bqm * p.LK, p.LK, ns);
    if (SOFTMAX) sm = softmax_stats<T, LPG>(attn + trp.bqm * p.LK, logits_ok ? p.LK : 0, lane, sl2);

    float acc[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] = 0.0f;

    for (int base = 0; base < p.LK; base += CH << sl2) {
        // ---- phase 1: descriptors
#pragma unroll
        for (int i = 0; i < SPW / 32; ++i) {
            const int j = pj + i * LPG;
            const int idx = base + (j << sl2) + psub;
            float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
            int4 o = make_int4(0, 0, 0, 0);
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
                const float hx = 1.0f - sg.lx, hy = 1.0f - sg.ly;
                const float ahy = a * hy, aly = a * sg.ly;
                w.x = (sg.vx0 && sg.vy0) ? ahy * hx : 0.0f;
                w.y = (sg.vx1 && sg.vy0) ? ahy * sg.lx : 0.0f;
                w.z = (sg.vx0 && sg.vy1) ? aly * hx : 0.0f;
                w.w = (sg.vx1 && sg.vy1) ? aly * sg.lx : 0.0f;
                o = make_int4(sg.row[0] * p.MD, sg.row[1] * p.MD, sg.row[2] * p.MD,
                              sg.row[3] * p.MD);
            }
            s_w[warp][lane + 32 * i] = w;     // == [j * GPW + pg]
            s_o[warp][lane + 32 * i] = o;
        }
        __syncwarp();

        // ---- phase 2: gather
        const int n = min(CH, (p.LK - base + (1 << sl2) - 1) >> sl2);
        for (int j = 0; j < n; j += U) {
            float4 w[U];
            uint4 v[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                w[u] = s_w[warp][(j + u) * GPW + g];
                const int4 o = s_o[warp][(j + u) * GPW + g];
                const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
                if (SPL && j + u >= n) {   // a split group's chunk is mostly empty slots
                    v[u][0] = v[u][1] = v[u][2] = v[u][3] = zero;
                    continue;
                }
                v[u][0] = in_tensor(p, value, vbase + o.x, VEC, nv) ? ldg16(vbase + o.x) : zero;
                v[u][1] = in_tensor(p, value, vbase + o.y, VEC, nv) ? ldg16(vbase + o.y) : zero;
                v[u][2] = in_tensor(p, value, vbase + o.z, VEC, nv) ? ldg16(vbase + o.z) : zero;
                v[u][3] = in_tensor(p, value, vbase + o.w, VEC, nv) ? ldg16(vbase + o.w) : zero;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                fma16<T>(acc, w[u].x, v[u][0]);
                fma16<T>(acc, w[u].y, v[u][1]);
                fma16<T>(acc, w[u].z, v[u][2]);
                fma16<T>(acc, w[u].w, v[u][3]);
            }
        }
        __syncwarp();
    }

    if (SPL) {
        for (int off = LPG; off < (LPG << sl2); off <<= 1) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
        }
    }
    if (valid_q && sub == 0) {
        T *out = reinterpret_cast<T *>(p.out);
        T *o = out + tr.bqm * p.D + r * VEC;
        if (in_tensor(p, out, o, VEC, n_out(p))) *reinterpret_cast<uint4 *>(o) = pack16<T>(acc);
    }
}

template <typename T, bool SOFTMAX, bool SPL, int UMAX = 8>
static cudaError_t launch_forward_t(const Params &p, int lpg, cudaStream_t stream) {
    const int gpw = 32 / lpg;
    const int64_t per_warp = gpw >> p.split_log2;     // query-heads per warp
    const int64_t warps = (p.triples + per_warp - 1) / per_warp;
    constexpr int wpb = fwd_warps<SPL>();
    const int64_t blocks = (warps + wpb - 1) / wpb;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks);
    switch (lpg) {
        case 1: msda_forward_kernel<T, 1, SOFTMAX, SPL, UMAX><<<grid, wpb * 32, 0, stream>>>(p); break;
        case 2: msda_forward_kernel<T, 2, SOFTMAX, SPL, UMAX><<<grid, wpb * 32, 0, stream>>>(p); break;
        case 4: msda_forward_kernel<T, 4, SOFTMAX, SPL, UMAX><<<grid, wpb * 32, 0, stream>>>(p); break;
        case 8: msda_forward_kernel<T, 8, SOFTMAX, SPL, UMAX><<<grid, wpb * 32, 0, stream>>>(p); break;
        case 16: msda_forward_kernel<T, 16, SOFTMAX, SPL, UMAX><<<grid, wpb * 32, 0, stream>>>(p); break;
        case 32: msda_forward_kernel<T, 32, SOFTMAX, SPL, UMAX><<<grid, wpb * 32, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_forward_d(const Params &p0, int lpg, bool softmax, cudaStream_t stream) {
    Params p = p0;
    p.split_log2 = choose_split(p.triples, 32 / lpg, p.LK, p0.split_log2);
    if (p.split_log2 > 0)
        return softmax ? launch_forward_t<T, true, true>(p, lpg, stream)
                       : launch_forward_t<T, false, true>(p, lpg, stream);
    // the chunk of CH samples per group: 8 for 16-byte lanes of a 64-byte
    // head or wider; a last chunk of 1 to 4 samples takes 4-sample steps
    const int last = p.LK % 8;
    if (last >= 1 && last <= 4)
        return softmax ? launch_forward_t<T, true, false, 4>(p, lpg, stream)
                       : launch_forward_t<T, false, false, 4>(p, lpg, stream);
    return softmax ? launch_forward_t<T, true, false>(p, lpg, stream)
                   : launch_forward_t<T, false, false>(p, lpg, stream);
}

cudaError_t launch_forward(const Params &p, msda_dtype_t dt, int lpg, bool softmax,
                           cudaStream_t stream) {
    switch (dt) {
        case MSDA_F32: return launch_forward_d<float>(p, lpg, softmax, stream);
        case MSDA_BF16: return launch_forward_d<__nv_bfloat16>(p, lpg, softmax, stream);
        case MSDA_F16: return launch_forward_d<__half>(p, lpg, softmax, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace msda
