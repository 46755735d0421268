/*
 * libmsda -- multi-scale deformable attention (MSDA) for GB300 (sm_103a).
 *
 * C ABI. Every pointer argument named as a tensor is a DEVICE pointer to a
 * dense, row-major (C-contiguous) array; the library allocates nothing, frees
 * nothing and keeps no state between calls. Every call is asynchronous: it
 * validates its arguments on the host, enqueues its kernels on `stream` (a
 * cudaStream_t passed as void*; NULL is the legacy default stream) and returns.
 * A non-OK status means nothing was enqueued, except MSDA_ERR_CUDA, which
 * reports the error of a launch that the runtime rejected.
 *
 * The operator is the bracketed term of Eq. 1 of Deformable DETR as the
 * msda-triton course, ch. 1 "Deformable attention, from scratch" states it
 * (sections "The equation, term by term" and "Bilinear interpolation"):
 *
 *   out[b,q,m*D+d] = sum_{l<L} sum_{k<K} A[b,q,m,l,k] *
 *                    bilinear(value[b, level l, m, d], loc[b,q,m,l,k,:])
 *
 * with pixel coordinates x = loc_x*W_l - 0.5, y = loc_y*H_l - 0.5 (the
 * grid_sample align_corners=False convention), the four corners
 * (y0,x0), (y0,x0+1), (y0+1,x0), (y0+1,x0+1) of x0 = floor(x), y0 = floor(y)
 * weighted (1-lx)(1-ly), lx(1-ly), (1-lx)ly, lx*ly, and zero for a corner
 * outside [0,W_l) x [0,H_l). Level l occupies value rows
 * [level_start_index[l], level_start_index[l] + H_l*W_l), pixel (y, x) at
 * row level_start_index[l] + y*W_l + x.
 *
 * Operands (shapes use B batch, S = sum_l H_l*W_l value rows, Q queries,
 * M heads, D channels per head, L levels, K points per level):
 *   value                (B, S, M, D)        float type `dtype`
 *   spatial_shapes       (L, 2) int64        rows (H_l, W_l)
 *   level_start_index    (L,)   int64        exclusive prefix sum of H_l*W_l
 *   sampling_locations   (B, Q, M, L, K, 2)  `dtype`, last dim (x, y), normalised
 *   attention_weights    (B, Q, M, L, K)     `dtype`, used as given
 *   out                  (B, Q, M*D)         `dtype`
 * Sampling locations may be anything, including off the map, infinite or
 * NaN: a sample none of whose corners is inside the map contributes zero and
 * receives zero gradient. The integer parts (x0, y0) are the exact floor of
 * the real number loc*W - 0.5 for the stored loc. value and grad_out must be
 * finite: a corner outside the map is read from a clamped in-map row with
 * weight zero, so a non-finite value there would leak into the result.
 * A level whose table entry is not a non-empty rectangle inside [0, S)
 * (H_l < 1, W_l < 1, start < 0 or start + H_l*W_l > S) is treated as empty.
 *
 * Arithmetic: products and sums in fp32 for fp32 and 16-bit storage (a 16-bit
 * result is rounded once, to nearest even, when it is stored); in fp64 for
 * MSDA_F64, whose integer parts follow x = loc*W - 0.5 computed with a
 * rounded multiply and a rounded add in double.
 */
#ifndef MSDA_H
#define MSDA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSDA_API __attribute__((visibility("default")))
#else
#define MSDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type of every float operand of one call. */
typedef enum {
    MSDA_F32 = 0,
    MSDA_BF16 = 1,
    MSDA_F16 = 2,
    MSDA_F64 = 3   /* double throughout: geometry, arithmetic and atomics */
} msda_dtype_t;

/* How msda_backward accumulates grad_value for a 16-bit dtype.
 * NATIVE: vector atomic adds straight into the 16-bit grad_value (each add
 *   rounds to the 16-bit format, so the result depends on contention).
 *   Measured grad_value error against an fp64 reference (relative L2, bf16,
 *   GB300): decoder shape 3.3e-3, Mask2Former encoder 1.2e-2, Deformable-DETR
 *   encoder 1.9e-2 (at the 2e-2 bar: a level-3 pixel receives about 1,300
 *   adds per head), and 5.5e-2 when every point of 5,000 queries falls in one
 *   4x4 patch per level: NATIVE misses 2e-2 on contended maps. fp16 keeps 3
 *   more mantissa bits (decoder 4.1e-4). FP32_BUFFER stays at the 16-bit
 *   rounding of the result (1.7e-3 bf16) on every one of them, and
 *   FP16_BUFFER (below) within 2e-2 on each at close to NATIVE's speed.
 * FP32_BUFFER: atomic adds into a caller-provided fp32 workspace, then one
 *   rounding pass into grad_value. For MSDA_F32 and MSDA_F64 both modes are
 *   the same (atomics of that type into grad_value) and no workspace is needed.
 * The pages motivate the switch: the Efficient-MSDA summary page, section
 * "The backward pass is an atomics problem", and the deformops README,
 * section "Backend selection" (fp32 accumulator vs native half atomics). */
typedef enum {
    MSDA_ACC_NATIVE = 0,
    MSDA_ACC_FP32_BUFFER = 1,
    MSDA_ACC_AUTO = 2,
    MSDA_ACC_FP16_BUFFER = 3
} msda_accum_t;
/* MSDA_ACC_FP16_BUFFER (bf16 data; msda_backward and msda_backward_softmax
 * only -- the three-step calls below refuse it with MSDA_ERR_DTYPE, since its
 * zero step reads grad_out): native 16-bit atomic adds, but into an fp16
 * workspace, which keeps 11 significant bits where bf16 keeps 8, with every
 * contribution multiplied by a power of two 2^k chosen per call; grad_value is
 * then round(ws * 2^-k). Each element of grad_value sums |a| w |g| over the
 * samples that reach it (bilinear weight w <= 1, one sample per query, level
 * and point at most), so no sum exceeds max|grad_out| * Q * A, with A = 1 for
 * msda_backward_softmax (probabilities) and L * K * max|attention weight|
 * otherwise; 2^k puts that bound below 2^15 (and, for normal inputs, at or
 * above 2^11), under fp16's largest finite value, for any bound up to 2^141,
 * and keeps every weight times 2^k finite in fp32.
 * Sums far below the bound (2^-25 of it and less) fall into fp16's subnormals
 * and keep fewer bits. The adds move 64 bytes per corner and head,
 * as native accumulation does (half the fp32 buffer's).
 * Measured (relative L2 against an fp64 reference, GB300): grad_value 1.7e-3
 * on the decoder shape, 3.1e-3 on the Deformable-DETR encoder, 2.3e-3 on the
 * Mask2Former encoder, 7.8e-3 with 5,000 queries in one 4x4 patch per level
 * (NATIVE 5.5e-2); the encoder backward takes 306 us against 277 us NATIVE and
 * 383 us with FP32_BUFFER. Limit: a 16-bit running sum stagnates once it is
 * 2^11 times its addends, so thousands of same-sign adds into one element
 * (all-positive grad_out with every query on one small patch) lose most of
 * their sum; FP32_BUFFER is the mode for such inputs.
 * Workspace: B*S*M*D*2 + 20480 bytes (msda_backward_workspace_bytes). For
 * fp16, fp32 and fp64 data it is the same as MSDA_ACC_NATIVE. */
/* MSDA_ACC_AUTO (16-bit data): NATIVE or FP32_BUFFER, chosen on the host from
 * the sizes alone. The call adds natively when the value rows receive on
 * average at most 4 corner adds per head, 4*Q*K*L <= 4*S, and uses the fp32
 * workspace otherwise. A detector decoder (300 queries over the 22,223 rows of
 * an 800x1333 pyramid: 0.9 adds per row) then needs no workspace and no pass
 * over one; encoder shapes (Q = S: 4*K*L adds per row) keep the workspace.
 * msda_backward_workspace_bytes and every backward call resolve it the same
 * way, so the three-step calls accept it too.
 * Accuracy: native adds round at every add, so their error grows with the adds
 * a row actually receives. The mean over the pyramid does not see a level much
 * smaller than S/L, nor samples concentrated on a few pixels; either can give
 * a native call an error above 2e-2 relative L2 that FP32_BUFFER would not. */

typedef enum {
    MSDA_OK = 0,
    MSDA_ERR_NULL = 1,      /* a required pointer is NULL                      */
    MSDA_ERR_SHAPE = 2,     /* a dimension is out of the supported range       */
    MSDA_ERR_DTYPE = 3,     /* unknown dtype or accumulation mode              */
    MSDA_ERR_ALIGN = 4,     /* a pointer is not aligned as required            */
    MSDA_ERR_WORKSPACE = 5, /* workspace missing or smaller than required      */
    MSDA_ERR_CUDA = 6,      /* the CUDA runtime rejected a launch              */
    MSDA_ERR_DEVICE_BOUNDS = 7  /* checked build: a kernel access left its tensor */
} msda_status_t;

/* Problem sizes. Supported: B >= 0, Q >= 0 (zero is a valid empty call),
 * S >= 1, M >= 1, 1 <= L <= 16, K >= 1, S*M*D < 2^31, and D a power-of-two
 * multiple of the 16-byte vector width: D/4 in {1,2,4,...,32} for MSDA_F32,
 * D/8 in {1,2,4,...,32} for 16-bit dtypes, D/2 in {1,2,4,...,32} for
 * MSDA_F64 (D = 32 is the detector case). */
typedef struct {
    int64_t B, S, Q, M, D, L, K;
} msda_dims_t;

/* Forward: writes out (B, Q, M*D). The bracketed term of Eq. 1 (see top).
 * query_order: NULL for linear dispatch, else a device int32 permutation of
 *   [0, Q) shared by every batch; dispatch slot i computes query
 *   query_order[i]. The result does not depend on it (Efficient-MSDA page,
 *   "Two heuristics that do not apply": dispatch order is a scheduling knob).
 *   A slot whose entry lies outside [0, Q) computes nothing; an array that is
 *   not a permutation leaves some outputs unwritten.
 * Alignment: value and out 16 bytes; sampling_locations 2*element size;
 *   attention_weights element size; spatial_shapes, level_start_index 8.
 * Errors: MSDA_ERR_NULL, _SHAPE, _DTYPE, _ALIGN before any launch;
 *   MSDA_ERR_CUDA if the launch is rejected. */
MSDA_API msda_status_t msda_forward(const void *value, const int64_t *spatial_shapes,
                           const int64_t *level_start_index,
                           const void *sampling_locations,
                           const void *attention_weights,
                           const int32_t *query_order, void *out,
                           const msda_dims_t *dims, msda_dtype_t dtype,
                           void *stream);

/* Bytes of device workspace msda_backward needs: B*S*M*D*4 for a 16-bit
 * dtype with MSDA_ACC_FP32_BUFFER, or MSDA_ACC_AUTO where it resolves to the
 * fp32 buffer; B*S*M*D*2 + 20480 for bf16 with MSDA_ACC_FP16_BUFFER; else 0.
 * Returns 0 for
 * invalid dims. */
MSDA_API size_t msda_backward_workspace_bytes(const msda_dims_t *dims,
                                     msda_dtype_t dtype, msda_accum_t accum);

/* Backward: given grad_out (B, Q, M*D), OVERWRITES
 *   grad_value               (B, S, M, D)       d loss / d value
 *   grad_sampling_locations  (B, Q, M, L, K, 2) d loss / d loc
 *   grad_attention_weights   (B, Q, M, L, K)    d loss / d attention weight
 * The three gradients the msda-triton course index names for chapter 5
 * ("The backward kernel"), derived from the forward by the chain rule: with
 * g = grad_out[b,q,m,:] and s_c = <g, value[corner c]> (0 outside the map),
 *   grad_attn = sum_c w_c s_c,   grad_value[corner c] += a w_c g,
 *   grad_loc_x = a W_l ((1-ly)(s_01-s_00) + ly(s_11-s_10)),
 *   grad_loc_y = a H_l ((1-lx)(s_10-s_00) + lx(s_11-s_01)).
 * No per-sample intermediate buffer is used (deformops README, "Zero-buffer
 * kernels"). grad_value is accumulated with atomics, so its rounding order is
 * not deterministic; the other two gradients are.
 * workspace: device memory of at least msda_backward_workspace_bytes(...)
 *   bytes, 16-byte aligned, owned by the caller (may be NULL when 0 bytes
 *   are needed). Its contents are overwritten.
 * Alignment: value, grad_out, grad_value 16 bytes; sampling_locations and
 *   grad_sampling_locations 2*element size; attention weights and their
 *   gradient element size.
 * Errors: as msda_forward, plus MSDA_ERR_WORKSPACE. */
MSDA_API msda_status_t msda_backward(const void *value, const int64_t *spatial_shapes,
                            const int64_t *level_start_index,
                            const void *sampling_locations,
                            const void *attention_weights,
                            const int32_t *query_order, const void *grad_out,
                            void *grad_value, void *grad_sampling_locations,
                            void *grad_attention_weights, void *workspace,
                            size_t workspace_bytes, msda_accum_t accum,
                            const msda_dims_t *dims, msda_dtype_t dtype,
                            void *stream);

/* The softmax variant: attention_logits (B, Q, M, L, K) are raw logits and
 * the operator uses a = softmax over the L*K logits of each (b,q,m) -- the
 * method the deformops README ("Multi-scale deformable attention") describes
 * for normalising logits jointly over levels and points inside the kernel.
 * msda_forward_softmax: as msda_forward with a in place of the weights.
 * msda_backward_softmax: as msda_backward, writing d loss / d logit to
 *   grad_attention_logits: a * (g_a - sum_j a_j g_a_j), g_a = d loss / d a.
 * Logits must be finite. Supported: L*K <= 16 * D / (16 / element size), i.e.
 * L*K <= 64 for 16-bit D = 32 and <= 128 for fp32 D = 32 (MSDA_ERR_SHAPE
 * otherwise). Errors and alignment as msda_forward / msda_backward. */
MSDA_API msda_status_t msda_forward_softmax(const void *value, const int64_t *spatial_shapes,
                                            const int64_t *level_start_index,
                                            const void *sampling_locations,
                                            const void *attention_logits,
                                            const int32_t *query_order, void *out,
                                            const msda_dims_t *dims, msda_dtype_t dtype,
                                            void *stream);
MSDA_API msda_status_t msda_backward_softmax(
    const void *value, const int64_t *spatial_shapes, const int64_t *level_start_index,
    const void *sampling_locations, const void *attention_logits, const int32_t *query_order,
    const void *grad_out, void *grad_value, void *grad_sampling_locations,
    void *grad_attention_logits, void *workspace, size_t workspace_bytes, msda_accum_t accum,
    const msda_dims_t *dims, msda_dtype_t dtype, void *stream);

/* The same backward in three steps, for callers that sum grad_value over
 * several calls sharing one value tensor (or that time the kernels apart).
 * msda_backward(...) is exactly zero + accumulate + finish on one stream.
 *
 * msda_backward_zero: zeroes the accumulation target -- the fp32 workspace
 *   for a 16-bit dtype with MSDA_ACC_FP32_BUFFER, else grad_value.
 * msda_backward_accumulate: ADDS this call's contribution into that target
 *   and overwrites grad_sampling_locations and grad_attention_weights.
 *   Arguments as msda_backward.
 * msda_backward_finish: rounds the fp32 workspace into grad_value (16-bit
 *   dtype with MSDA_ACC_FP32_BUFFER); does nothing in the other modes.
 * Errors: as msda_backward. */
MSDA_API msda_status_t msda_backward_zero(void *grad_value, void *workspace,
                                          size_t workspace_bytes, msda_accum_t accum,
                                          const msda_dims_t *dims, msda_dtype_t dtype,
                                          void *stream);
MSDA_API msda_status_t msda_backward_accumulate(
    const void *value, const int64_t *spatial_shapes, const int64_t *level_start_index,
    const void *sampling_locations, const void *attention_weights,
    const int32_t *query_order, const void *grad_out, void *grad_value,
    void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
    size_t workspace_bytes, msda_accum_t accum, const msda_dims_t *dims,
    msda_dtype_t dtype, void *stream);
MSDA_API msda_status_t msda_backward_finish(const void *workspace, size_t workspace_bytes,
                                            void *grad_value, msda_accum_t accum,
                                            const msda_dims_t *dims, msda_dtype_t dtype,
                                            void *stream);

/* Size of the fp32 accumulator that msda_backward_static_workspace keeps
 * inside the library: 64 MiB, enough for B*S*M*D <= 16,777,216 (for example
 * the Deformable-DETR encoder shape with B = 2). */
#define MSDA_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)

/* msda_backward for callers that cannot allocate device memory when they call
 * (an operator plugin whose engine owns all device memory and offers no
 * scratch, or an application that allows no device allocation after start-up).
 * The pages describe no such entry point; it exists for those callers only.
 * It computes what msda_backward computes with MSDA_ACC_FP32_BUFFER, using as
 * its fp32 workspace a fixed MSDA_STATIC_WORKSPACE_BYTES array that belongs to
 * the library, and it allocates nothing. Arguments as msda_backward, without
 * the workspace and the accumulation mode.
 * - Returns MSDA_ERR_WORKSPACE, before any launch, when a 16-bit problem needs
 *   more than MSDA_STATIC_WORKSPACE_BYTES (B*S*M*D*4 bytes). fp32 data needs no
 *   workspace and has no such limit.
 * - Each call finds the array's device address in the calling thread's
 *   current context (MSDA_ERR_CUDA if that fails). The address is cached per
 *   context and looked up again when the context changes (for instance after
 *   cudaDeviceReset), never reused across contexts. The first call in a
 *   context may load the library's module; make it before any stream capture
 *   begins.
 * - Every call shares the one array. Each call clears the part it uses, but
 *   calls that overlap on the GPU (other streams, other host threads) race on
 *   it: the caller must order them.
 * - The array occupies device memory in every context that has loaded the
 *   library's module, until the process exits: under the default lazy module
 *   loading that is the first call of any libmsda entry point that runs a
 *   kernel on that device; with CUDA_MODULE_LOADING=EAGER it is every device
 *   the process initialises, as soon as it does. */
MSDA_API msda_status_t msda_backward_static_workspace(
    const void *value, const int64_t *spatial_shapes, const int64_t *level_start_index,
    const void *sampling_locations, const void *attention_weights,
    const int32_t *query_order, const void *grad_out, void *grad_value,
    void *grad_sampling_locations, void *grad_attention_weights, const msda_dims_t *dims,
    msda_dtype_t dtype, void *stream);

/* The integer parts every kernel uses, for bit-exact checks (same device
 * code as the forward and backward kernels). For each sample s (flattened
 * (b,q,m,l,k)) and corner c in order 00, 01, 10, 11, writes to the device
 * array corner_rows (B*Q*M*L*K*4 int32) the value row
 * level_start_index[l] + yy*W_l + xx of a corner inside the map, -1 for a
 * corner outside it -- the row the loop of the msda-triton course, ch. 1
 * "The simplest possible implementation", reads for that corner after its
 * bounds test. One int32 per corner carries both the corner index and its
 * in-map mask (-1), in place of a separate (x0, y0) pair and 4-bit mask.
 * D of dims is not used. Errors: MSDA_ERR_NULL, _SHAPE, _DTYPE, _ALIGN before
 * any launch (corner_rows 16-byte aligned); MSDA_ERR_CUDA on a rejected launch. */
MSDA_API msda_status_t msda_debug_corners(const int64_t *spatial_shapes,
                                 const int64_t *level_start_index,
                                 const void *sampling_locations,
                                 int32_t *corner_rows, const msda_dims_t *dims,
                                 msda_dtype_t dtype, void *stream);

/* Range-checked build. libmsda_checked.so is built from the same sources
 * with every global access of the forward, backward and corner kernels first
 * checked against the extent of its tensor (derived from dims): an access
 * that would leave its tensor is skipped -- a load yields zeros, a store or
 * add does nothing -- and a per-context fault word is set; nothing traps. The
 * workspace passes (zero, convert, the fp16 workspace's prepare and finish)
 * walk a flat range of the buffer they are given, bounded by their loops. It is a debugging stand-in for
 * a memory checker, much slower than libmsda.so. The normal library exports
 * the same three entry points and never sets the word.
 * msda_checked_build: 1 in libmsda_checked.so, 0 in libmsda.so.
 * msda_device_check: synchronizes `stream`, then reads and clears the fault
 *   word of the calling thread's current context: MSDA_ERR_DEVICE_BOUNDS if
 *   any checked access was out of range since the last call, MSDA_OK
 *   otherwise (always in the normal build); MSDA_ERR_CUDA if the
 *   synchronization or the readback fails.
 * msda_debug_bounds_self_test: enqueues one range check that must fail (no
 *   memory is accessed), so that the next msda_device_check of the checked
 *   build returns MSDA_ERR_DEVICE_BOUNDS; a no-op check in the normal build.
 * The word's address is looked up per context and cached with the context's
 * identity (a new context, e.g. after cudaDeviceReset, gets its own); the
 * first lookup in a context may load the library's module, so make it before
 * any stream capture begins. */
MSDA_API int msda_checked_build(void);
MSDA_API msda_status_t msda_device_check(void *stream);
MSDA_API msda_status_t msda_debug_bounds_self_test(void *stream);


/* Sample split (launch tuning; process-wide). With one lane group per
 * (b, q, m), a problem with few query-heads -- a detector decoder's B*Q*M =
 * 4,800 -- occupies a fraction of the SMs. The kernels then spread each
 * query-head's L*K samples over 2^s lane groups of one warp, which combine
 * their partial results with warp shuffles. Results agree with s = 0 up to
 * the fp32 summation order. By default (log2_groups = -1) s is chosen per
 * launch from the problem size; 0 to 3 force s, clamped per launch to the
 * groups of a warp and to L*K. Applies to the 16-bit and fp32 kernels (fp64
 * kernels never split). Meant for tests and tuning: set it when no other
 * thread is launching. MSDA_ERR_SHAPE for a value outside -1..3, which
 * leaves the setting unchanged. */
MSDA_API msda_status_t msda_set_sample_split(int log2_groups);

/* Static description of a status code (never NULL). Host only; the pages
 * define no such call: it names the statuses above for error messages. */
MSDA_API const char *msda_status_string(msda_status_t status);

/* Library version, major*10000 + minor*100 + patch. Host only. */
MSDA_API int msda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSDA_H */
