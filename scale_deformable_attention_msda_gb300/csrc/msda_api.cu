// libmsda C ABI: argument validation and kernel dispatch (host code).
// The entry points and their contracts are declared in include/msda.h.
#include <stdint.h>

#include <atomic>

#include "msda_common.cuh"

namespace msda {
cudaError_t launch_forward(const Params &p, msda_dtype_t dt, int lpg, bool softmax,
                           cudaStream_t stream);
cudaError_t launch_backward(const Params &p, msda_dtype_t dt, bool f32acc, int lpg, bool softmax,
                            cudaStream_t stream);
cudaError_t launch_zero(void *p, int64_t bytes, cudaStream_t stream);
cudaError_t launch_convert(const float *ws, void *gv, int64_t n, msda_dtype_t dt,
                           cudaStream_t stream);
int f16_prepare_blocks(int64_t n, int64_t ng, const void *attn, int64_t na);
cudaError_t launch_f16_prepare(void *ws, int64_t n, const void *grad_out, int64_t ng,
                               const void *attn, int64_t na, cudaStream_t stream);
float *f16_scale_pair(void *ws, int64_t n);
cudaError_t launch_f16_finish(void *ws, void *gv, int64_t n, cudaStream_t stream);
cudaError_t launch_backward_f16acc(const Params &p, int lpg, bool softmax, cudaStream_t stream);
cudaError_t launch_corners(const Params &p, msda_dtype_t dt, int32_t *rows, cudaStream_t stream);
cudaError_t launch_forward_f64(const Params &p, int lpg, bool softmax, cudaStream_t stream);
cudaError_t launch_backward_f64(const Params &p, int lpg, bool softmax, cudaStream_t stream);
cudaError_t launch_corners_f64(const Params &p, int32_t *rows, cudaStream_t stream);
cudaError_t fault_word_for_launch(unsigned **err);
}  // namespace msda

namespace {

using msda::Params;

bool dtype_ok(msda_dtype_t dt) {
    return dt == MSDA_F32 || dt == MSDA_BF16 || dt == MSDA_F16 || dt == MSDA_F64;
}
bool is_16bit(msda_dtype_t dt) { return dt == MSDA_BF16 || dt == MSDA_F16; }
int elem_bytes(msda_dtype_t dt) { return dt == MSDA_F64 ? 8 : (dt == MSDA_F32 ? 4 : 2); }

// MSDA_ACC_AUTO, resolved on the host from the sizes alone: native
// accumulation when the value rows receive on average at most kAutoMeanAdds
// corner adds per head (4 Q K L <= kAutoMeanAdds S), the fp32 workspace
// otherwise. Other modes are returned unchanged.
// MSDA_ACC_FP16_BUFFER applies to bf16 data; other dtypes accumulate natively
// (fp16 data already adds in fp16, fp32 and fp64 in their own type).
constexpr int64_t kAutoMeanAdds = 4;
msda_accum_t resolve_accum(const msda_dims_t &d, msda_dtype_t dt, msda_accum_t accum) {
    if (accum == MSDA_ACC_FP16_BUFFER) return dt == MSDA_BF16 ? accum : MSDA_ACC_NATIVE;
    if (accum != MSDA_ACC_AUTO) return accum;
    const double adds = 4.0 * (double)d.Q * (double)d.K * (double)d.L;
    return adds <= (double)kAutoMeanAdds * (double)d.S ? MSDA_ACC_NATIVE : MSDA_ACC_FP32_BUFFER;
}
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Lanes per (b,q,m) group: D / (channels per 16 bytes), a power of two <= 32.
int lanes_per_group(const msda_dims_t &d, msda_dtype_t dt) {
    const int vec = 16 / elem_bytes(dt);
    if (d.D % vec != 0) return 0;
    const int64_t lpg = d.D / vec;
    if (lpg < 1 || lpg > 32 || (lpg & (lpg - 1)) != 0) return 0;
    return (int)lpg;
}

// Sizes the kernels support (see msda_dims_t in msda.h).
msda_status_t check_dims(const msda_dims_t *d, msda_dtype_t dt, int *lpg) {
    if (!d) return MSDA_ERR_NULL;
    if (!dtype_ok(dt)) return MSDA_ERR_DTYPE;
    if (d->B < 0 || d->Q < 0 || d->S < 1 || d->M < 1 || d->D < 1 || d->L < 1 ||
        d->L > msda::kMaxLevels || d->K < 1)
        return MSDA_ERR_SHAPE;
    if (d->S > INT32_MAX || d->M > INT32_MAX || d->D > INT32_MAX || d->K > (1 << 10) ||
        d->B > INT32_MAX || d->Q > INT32_MAX)
        return MSDA_ERR_SHAPE;
    if (d->S * d->M * d->D > INT32_MAX) return MSDA_ERR_SHAPE;     // 32-bit row offsets
    // value-sized tensors (and the fp32 workspace, 4 bytes per element) must
    // have byte counts that fit in int64: B*S*M*D <= 2^60
    if (d->B > ((int64_t)1 << 60) / (d->S * d->M * d->D)) return MSDA_ERR_SHAPE;
    const int64_t lk = d->L * d->K;
    if (lk > (1 << 20)) return MSDA_ERR_SHAPE;
    // every element count must fit comfortably in int64
    const double samples = (double)d->B * d->Q * d->M * lk;
    if (samples * 2.0 > 9.0e18) return MSDA_ERR_SHAPE;
    const int l = lanes_per_group(*d, dt);
    if (!l) return MSDA_ERR_SHAPE;
    if (lpg) *lpg = l;
    return MSDA_OK;
}

// msda_set_sample_split: -1 chooses the split per launch, 0..3 force it.
std::atomic<int> g_sample_split{-1};

Params make_params(const msda_dims_t &d) {
    Params p = {};
    p.split_log2 = g_sample_split.load(std::memory_order_relaxed);
    p.B = (int)d.B;
    p.S = (int)d.S;
    p.Q = (int)d.Q;
    p.M = (int)d.M;
    p.D = (int)d.D;
    p.L = (int)d.L;
    p.K = (int)d.K;
    p.LK = (int)(d.L * d.K);
    p.MD = (int)(d.M * d.D);
    p.inv_K = 1.0f / (float)d.K;
    p.triples = d.B * d.Q * d.M;
    return p;
}

msda_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MSDA_OK : MSDA_ERR_CUDA; }

// The softmax variant keeps d loss / d weight of a warp's query-heads in 512
// fp32 shared-memory slots: L*K <= 512 / (32 / lanes per group).
bool softmax_fits(const msda_dims_t &d, msda_dtype_t dt, int lpg) {
    return dt == MSDA_F64 || d.L * d.K <= 16 * (int64_t)lpg;   // fp64 keeps no slots
}

// Pointers shared by the forward and the backward.
msda_status_t check_common(const void *value, const int64_t *shapes, const int64_t *starts,
                           const void *loc, const void *attn, const msda_dims_t &d,
                           msda_dtype_t dt) {
    const int e = elem_bytes(dt);
    const bool has_q = d.B > 0 && d.Q > 0;
    if (!shapes || !starts) return MSDA_ERR_NULL;
    if (d.B > 0 && !value) return MSDA_ERR_NULL;
    if (has_q && (!loc || !attn)) return MSDA_ERR_NULL;
    if (!aligned(shapes, 8) || !aligned(starts, 8)) return MSDA_ERR_ALIGN;
    if (value && !aligned(value, 16)) return MSDA_ERR_ALIGN;
    if (loc && !aligned(loc, 2 * e)) return MSDA_ERR_ALIGN;
    if (attn && !aligned(attn, e)) return MSDA_ERR_ALIGN;
    return MSDA_OK;
}

}  // namespace

extern "C" {

int msda_version(void) { return 200; }

msda_status_t msda_set_sample_split(int log2_groups) {
    if (log2_groups < -1 || log2_groups > 3) return MSDA_ERR_SHAPE;
    g_sample_split.store(log2_groups, std::memory_order_relaxed);
    return MSDA_OK;
}

const char *msda_status_string(msda_status_t s) {
    switch (s) {
        case MSDA_OK: return "ok";
        case MSDA_ERR_NULL: return "a required pointer is NULL";
        case MSDA_ERR_SHAPE: return "a dimension is outside the supported range";
        case MSDA_ERR_DTYPE: return "unknown dtype or accumulation mode";
        case MSDA_ERR_ALIGN: return "a pointer is not aligned as required";
        case MSDA_ERR_WORKSPACE: return "workspace missing or too small";
        case MSDA_ERR_CUDA: return "the CUDA runtime rejected a launch";
        case MSDA_ERR_DEVICE_BOUNDS:
            return "checked build: a kernel access fell outside its tensor";
    }
    return "unknown status";
}

static msda_status_t forward_impl(const void *value, const int64_t *spatial_shapes,
                                  const int64_t *level_start_index,
                                  const void *sampling_locations, const void *attention_weights,
                                  const int32_t *query_order, void *out, const msda_dims_t *dims,
                                  msda_dtype_t dtype, bool softmax, void *stream) {
    int lpg = 0;
    msda_status_t st = check_dims(dims, dtype, &lpg);
    if (st != MSDA_OK) return st;
    const msda_dims_t &d = *dims;
    if (softmax && !softmax_fits(d, dtype, lpg)) return MSDA_ERR_SHAPE;
    st = check_common(value, spatial_shapes, level_start_index, sampling_locations,
                      attention_weights, d, dtype);
    if (st != MSDA_OK) return st;
    if (d.B == 0 || d.Q == 0) return MSDA_OK;
    if (!out) return MSDA_ERR_NULL;
    if (!aligned(out, 16) || (query_order && !aligned(query_order, 4))) return MSDA_ERR_ALIGN;
    Params p = make_params(d);
    if (msda::fault_word_for_launch(&p.err) != cudaSuccess) return MSDA_ERR_CUDA;
    p.value = value;
    p.shapes = spatial_shapes;
    p.starts = level_start_index;
    p.loc = sampling_locations;
    p.attn = attention_weights;
    p.order = query_order;
    p.out = out;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(dtype == MSDA_F64 ? msda::launch_forward_f64(p, lpg, softmax, s)
                                       : msda::launch_forward(p, dtype, lpg, softmax, s));
}

msda_status_t msda_forward(const void *value, const int64_t *spatial_shapes,
                           const int64_t *level_start_index, const void *sampling_locations,
                           const void *attention_weights, const int32_t *query_order,
                           void *out, const msda_dims_t *dims, msda_dtype_t dtype,
                           void *stream) {
    return forward_impl(value, spatial_shapes, level_start_index, sampling_locations,
                        attention_weights, query_order, out, dims, dtype, false, stream);
}

msda_status_t msda_forward_softmax(const void *value, const int64_t *spatial_shapes,
                                   const int64_t *level_start_index,
                                   const void *sampling_locations, const void *attention_logits,
                                   const int32_t *query_order, void *out,
                                   const msda_dims_t *dims, msda_dtype_t dtype, void *stream) {
    return forward_impl(value, spatial_shapes, level_start_index, sampling_locations,
                        attention_logits, query_order, out, dims, dtype, true, stream);
}

size_t msda_backward_workspace_bytes(const msda_dims_t *dims, msda_dtype_t dtype,
                                     msda_accum_t accum) {
    if (check_dims(dims, dtype, nullptr) != MSDA_OK) return 0;
    const msda_accum_t acc = resolve_accum(*dims, dtype, accum);
    const size_t n = (size_t)(dims->B * dims->S * dims->M * dims->D);
    if (acc == MSDA_ACC_FP16_BUFFER) return n * 2 + msda::kF16TailBytes;
    if (!is_16bit(dtype) || acc != MSDA_ACC_FP32_BUFFER) return 0;
    return n * sizeof(float);
}

namespace {

// Validation shared by the backward entry points; fills the launch parameters.
struct BackwardPlan {
    int lpg;
    bool f32acc;      // 16-bit data accumulated in the fp32 workspace
    bool f16acc;      // bf16 data accumulated in the scaled fp16 workspace
    void *target;     // what the atomics add into
    int64_t nval;     // B*S*M*D
    int64_t target_bytes;
};

// one_call: the scaled fp16 workspace needs grad_out in its zero step, so only
// msda_backward and msda_backward_softmax accept it for bf16 data.
msda_status_t plan_target(void *grad_value, void *workspace, size_t workspace_bytes,
                          msda_accum_t accum, const msda_dims_t *dims, msda_dtype_t dtype,
                          BackwardPlan *bp, bool one_call = false) {
    msda_status_t st = check_dims(dims, dtype, &bp->lpg);
    if (st != MSDA_OK) return st;
    if (accum != MSDA_ACC_NATIVE && accum != MSDA_ACC_FP32_BUFFER && accum != MSDA_ACC_AUTO &&
        accum != MSDA_ACC_FP16_BUFFER)
        return MSDA_ERR_DTYPE;
    const msda_dims_t &d = *dims;
    accum = resolve_accum(d, dtype, accum);
    if (accum == MSDA_ACC_FP16_BUFFER && !one_call) return MSDA_ERR_DTYPE;
    bp->f32acc = is_16bit(dtype) && accum == MSDA_ACC_FP32_BUFFER;
    bp->f16acc = accum == MSDA_ACC_FP16_BUFFER;
    bp->nval = d.B * d.S * d.M * d.D;
    bp->target = (bp->f32acc || bp->f16acc) ? workspace : grad_value;
    bp->target_bytes = bp->nval * (bp->f32acc ? 4 : elem_bytes(dtype));
    if (d.B == 0) return MSDA_OK;
    if (bp->f32acc || bp->f16acc) {
        const size_t need = msda_backward_workspace_bytes(dims, dtype, accum);
        if (!workspace || workspace_bytes < need) return MSDA_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return MSDA_ERR_ALIGN;
    }
    return MSDA_OK;
}

}  // namespace

msda_status_t msda_backward_zero(void *grad_value, void *workspace, size_t workspace_bytes,
                                 msda_accum_t accum, const msda_dims_t *dims,
                                 msda_dtype_t dtype, void *stream) {
    BackwardPlan bp;
    msda_status_t st = plan_target(grad_value, workspace, workspace_bytes, accum, dims, dtype, &bp);
    if (st != MSDA_OK) return st;
    if (dims->B == 0) return MSDA_OK;
    if (!bp.target) return MSDA_ERR_NULL;
    if (!aligned(bp.target, 16)) return MSDA_ERR_ALIGN;
    return from_cuda(msda::launch_zero(bp.target, bp.target_bytes, static_cast<cudaStream_t>(stream)));
}

static msda_status_t accumulate_impl(const void *value, const int64_t *spatial_shapes,
                                     const int64_t *level_start_index,
                                     const void *sampling_locations,
                                     const void *attention_weights, const int32_t *query_order,
                                     const void *grad_out, void *grad_value,
                                     void *grad_sampling_locations, void *grad_attention_weights,
                                     void *workspace, size_t workspace_bytes, msda_accum_t accum,
                                     const msda_dims_t *dims, msda_dtype_t dtype, bool softmax,
                                     void *stream) {
    BackwardPlan bp;
    msda_status_t st = plan_target(grad_value, workspace, workspace_bytes, accum, dims, dtype, &bp);
    if (st != MSDA_OK) return st;
    const msda_dims_t &d = *dims;
    if (softmax && !softmax_fits(d, dtype, bp.lpg)) return MSDA_ERR_SHAPE;
    st = check_common(value, spatial_shapes, level_start_index, sampling_locations,
                      attention_weights, d, dtype);
    if (st != MSDA_OK) return st;
    if (d.B == 0 || d.Q == 0) return MSDA_OK;
    const int e = elem_bytes(dtype);
    if (!grad_value || !grad_out || !grad_sampling_locations || !grad_attention_weights)
        return MSDA_ERR_NULL;
    if (!aligned(grad_value, 16) || !aligned(grad_out, 16) ||
        !aligned(grad_sampling_locations, 2 * e) || !aligned(grad_attention_weights, e) ||
        (query_order && !aligned(query_order, 4)))
        return MSDA_ERR_ALIGN;
    Params p = make_params(d);
    if (msda::fault_word_for_launch(&p.err) != cudaSuccess) return MSDA_ERR_CUDA;
    p.value = value;
    p.shapes = spatial_shapes;
    p.starts = level_start_index;
    p.loc = sampling_locations;
    p.attn = attention_weights;
    p.order = query_order;
    p.grad_out = grad_out;
    p.grad_value = bp.target;
    p.grad_loc = grad_sampling_locations;
    p.grad_attn = grad_attention_weights;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(dtype == MSDA_F64
                         ? msda::launch_backward_f64(p, bp.lpg, softmax, s)
                         : msda::launch_backward(p, dtype, bp.f32acc, bp.lpg, softmax, s));
}

msda_status_t msda_backward_accumulate(const void *value, const int64_t *spatial_shapes,
                                       const int64_t *level_start_index,
                                       const void *sampling_locations,
                                       const void *attention_weights,
                                       const int32_t *query_order, const void *grad_out,
                                       void *grad_value, void *grad_sampling_locations,
                                       void *grad_attention_weights, void *workspace,
                                       size_t workspace_bytes, msda_accum_t accum,
                                       const msda_dims_t *dims, msda_dtype_t dtype,
                                       void *stream) {
    return accumulate_impl(value, spatial_shapes, level_start_index, sampling_locations,
                           attention_weights, query_order, grad_out, grad_value,
                           grad_sampling_locations, grad_attention_weights, workspace,
                           workspace_bytes, accum, dims, dtype, false, stream);
}

msda_status_t msda_backward_finish(const void *workspace, size_t workspace_bytes,
                                   void *grad_value, msda_accum_t accum,
                                   const msda_dims_t *dims, msda_dtype_t dtype, void *stream) {
    BackwardPlan bp;
    msda_status_t st = plan_target(grad_value, const_cast<void *>(workspace), workspace_bytes,
                                   accum, dims, dtype, &bp);
    if (st != MSDA_OK) return st;
    if (dims->B == 0 || !bp.f32acc) return MSDA_OK;
    if (!grad_value) return MSDA_ERR_NULL;
    if (!aligned(grad_value, 16)) return MSDA_ERR_ALIGN;
    return from_cuda(msda::launch_convert(static_cast<const float *>(workspace), grad_value,
                                          bp.nval, dtype, static_cast<cudaStream_t>(stream)));
}

static msda_status_t backward_impl(const void *value, const int64_t *spatial_shapes,
                                   const int64_t *level_start_index,
                                   const void *sampling_locations, const void *attention_weights,
                                   const int32_t *query_order, const void *grad_out,
                                   void *grad_value, void *grad_sampling_locations,
                                   void *grad_attention_weights, void *workspace,
                                   size_t workspace_bytes, msda_accum_t accum,
                                   const msda_dims_t *dims, msda_dtype_t dtype, bool softmax,
                                   void *stream) {
    // Validate everything before the first launch, so that an error enqueues nothing.
    BackwardPlan bp;
    msda_status_t st = plan_target(grad_value, workspace, workspace_bytes, accum, dims, dtype, &bp,
                                   true);
    if (st != MSDA_OK) return st;
    const msda_dims_t &d = *dims;
    if (softmax && !softmax_fits(d, dtype, bp.lpg)) return MSDA_ERR_SHAPE;
    st = check_common(value, spatial_shapes, level_start_index, sampling_locations,
                      attention_weights, d, dtype);
    if (st != MSDA_OK) return st;
    if (d.B == 0) return MSDA_OK;
    const int e = elem_bytes(dtype);
    if (!grad_value) return MSDA_ERR_NULL;
    if (d.Q > 0 && (!grad_out || !grad_sampling_locations || !grad_attention_weights))
        return MSDA_ERR_NULL;
    if (!aligned(grad_value, 16) || (grad_out && !aligned(grad_out, 16)) ||
        (grad_sampling_locations && !aligned(grad_sampling_locations, 2 * e)) ||
        (grad_attention_weights && !aligned(grad_attention_weights, e)) ||
        (query_order && !aligned(query_order, 4)))
        return MSDA_ERR_ALIGN;
    if (bp.f16acc) {
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (d.Q == 0)   // nothing to add: grad_value is zero
            return msda_backward_zero(grad_value, nullptr, 0, MSDA_ACC_NATIVE, dims, dtype, stream);
        Params p = make_params(d);
        if (msda::fault_word_for_launch(&p.err) != cudaSuccess) return MSDA_ERR_CUDA;
        p.value = value;
        p.shapes = spatial_shapes;
        p.starts = level_start_index;
        p.loc = sampling_locations;
        p.attn = attention_weights;
        p.order = query_order;
        p.grad_out = grad_out;
        p.grad_value = workspace;
        // the softmax variant's weights are probabilities: no pass over the logits
        const void *amax_of = softmax ? nullptr : attention_weights;
        const int64_t ng = d.B * d.Q * d.M * d.D, na = d.B * d.Q * d.M * d.L * d.K;
        p.f16_nmax = msda::f16_prepare_blocks(bp.nval, ng, amax_of, na);
        p.f16_amax = amax_of != nullptr;
        p.f16_max = reinterpret_cast<const float *>(static_cast<char *>(workspace) + bp.nval * 2);
        p.f16_scale = msda::f16_scale_pair(workspace, bp.nval);
        p.grad_loc = grad_sampling_locations;
        p.grad_attn = grad_attention_weights;
        cudaError_t e = msda::launch_f16_prepare(workspace, bp.nval, grad_out, ng, amax_of, na, s);
        if (e == cudaSuccess) e = msda::launch_backward_f16acc(p, bp.lpg, softmax, s);
        if (e == cudaSuccess) e = msda::launch_f16_finish(workspace, grad_value, bp.nval, s);
        return from_cuda(e);
    }
    st = msda_backward_zero(grad_value, workspace, workspace_bytes, accum, dims, dtype, stream);
    if (st != MSDA_OK) return st;
    st = accumulate_impl(value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, query_order, grad_out, grad_value,
                         grad_sampling_locations, grad_attention_weights, workspace,
                         workspace_bytes, accum, dims, dtype, softmax, stream);
    if (st != MSDA_OK) return st;
    return msda_backward_finish(workspace, workspace_bytes, grad_value, accum, dims, dtype, stream);
}

msda_status_t msda_backward(const void *value, const int64_t *spatial_shapes,
                            const int64_t *level_start_index, const void *sampling_locations,
                            const void *attention_weights, const int32_t *query_order,
                            const void *grad_out, void *grad_value,
                            void *grad_sampling_locations, void *grad_attention_weights,
                            void *workspace, size_t workspace_bytes, msda_accum_t accum,
                            const msda_dims_t *dims, msda_dtype_t dtype, void *stream) {
    return backward_impl(value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, query_order, grad_out, grad_value,
                         grad_sampling_locations, grad_attention_weights, workspace,
                         workspace_bytes, accum, dims, dtype, false, stream);
}

msda_status_t msda_backward_softmax(const void *value, const int64_t *spatial_shapes,
                                    const int64_t *level_start_index,
                                    const void *sampling_locations, const void *attention_logits,
                                    const int32_t *query_order, const void *grad_out,
                                    void *grad_value, void *grad_sampling_locations,
                                    void *grad_attention_logits, void *workspace,
                                    size_t workspace_bytes, msda_accum_t accum,
                                    const msda_dims_t *dims, msda_dtype_t dtype, void *stream) {
    return backward_impl(value, spatial_shapes, level_start_index, sampling_locations,
                         attention_logits, query_order, grad_out, grad_value,
                         grad_sampling_locations, grad_attention_logits, workspace,
                         workspace_bytes, accum, dims, dtype, true, stream);
}

msda_status_t msda_debug_corners(const int64_t *spatial_shapes, const int64_t *level_start_index,
                                 const void *sampling_locations, int32_t *corner_rows,
                                 const msda_dims_t *dims, msda_dtype_t dtype, void *stream) {
    if (!dims) return MSDA_ERR_NULL;
    if (!dtype_ok(dtype)) return MSDA_ERR_DTYPE;
    const msda_dims_t &d = *dims;
    if (d.B < 0 || d.Q < 0 || d.S < 1 || d.M < 1 || d.L < 1 || d.L > msda::kMaxLevels ||
        d.K < 1 || d.K > (1 << 10) || d.S > INT32_MAX)
        return MSDA_ERR_SHAPE;
    if (!spatial_shapes || !level_start_index) return MSDA_ERR_NULL;
    const int64_t n = d.B * d.Q * d.M * d.L * d.K;
    if (n == 0) return MSDA_OK;
    if (!sampling_locations || !corner_rows) return MSDA_ERR_NULL;
    if (!aligned(sampling_locations, 2 * elem_bytes(dtype)) || !aligned(corner_rows, 16) ||
        !aligned(spatial_shapes, 8) || !aligned(level_start_index, 8))
        return MSDA_ERR_ALIGN;
    Params p = {};
    p.shapes = spatial_shapes;
    p.starts = level_start_index;
    p.loc = sampling_locations;
    p.B = (int)d.B;
    p.S = (int)d.S;
    p.Q = (int)d.Q;
    p.M = (int)d.M;
    p.L = (int)d.L;
    p.K = (int)d.K;
    p.LK = (int)(d.L * d.K);
    p.inv_K = 1.0f / (float)d.K;
    p.triples = d.B * d.Q * d.M;
    if (msda::fault_word_for_launch(&p.err) != cudaSuccess) return MSDA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(dtype == MSDA_F64 ? msda::launch_corners_f64(p, corner_rows, s)
                                       : msda::launch_corners(p, dtype, corner_rows, s));
}

}  // extern "C"
