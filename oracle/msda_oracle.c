/*
 * Multi-scale deformable attention (MSDA): the ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY. This file is a plain, slow, fp64 CPU statement of
 * what the operator computes, used to check the CUDA library. Only the tests,
 * the smoke check and the CPU-baseline leg of the benchmark may load it. The
 * CUDA library neither links nor calls it, and the two share no code.
 *
 * Sources (the operator has no printed formula that survived; it is restated
 * here from the prose and the loop the pages give):
 *   [C1-eq]   msda-triton course, ch. 1 "Deformable attention, from scratch",
 *             section "The equation, term by term": the bracketed term of Eq. 1
 *             of Deformable DETR -- per query q and head m, the sum over levels
 *             l and points k of A_mlqk times the feature map x_l read at
 *             phi_l(p_q) + dp_mlqk. Operand layouts are listed right after it:
 *             value (B,S,M,D), spatial_shapes (L,2) as (H_l,W_l),
 *             sampling_locations (B,Q,M,L,K,2), attention_weights (B,Q,M,L,K),
 *             output (B,Q,M*D).
 *   [C1-bil]  same chapter, section "Bilinear interpolation: reading between
 *             the pixels": x0 = floor(x), y0 = floor(y), lx = x-x0, ly = y-y0,
 *             corners (y0,x0), (y0,x0+1), (y0+1,x0), (y0+1,x0+1) weighted
 *             (1-lx)(1-ly), lx(1-ly), (1-lx)ly, lx*ly. Pixel mapping as
 *             grid_sample(align_corners=False): x = loc_x*W_l - 0.5,
 *             y = loc_y*H_l - 0.5. A corner outside the map contributes zero.
 *   [C1-loop] same chapter, section "The simplest possible implementation":
 *             the loop nest b, q, m, level, k, corners, in that order; value row
 *             index start_l + yy*W_l + xx. The pages state its arithmetic in
 *             double precision (Python floats), which this file keeps.
 *   [C1-ch5]  msda-triton course index, chapter 5 "The backward kernel":
 *             three gradients (value, sampling locations, attention weights).
 *             The pages do not print them; they are derived below from the
 *             forward by the chain rule.
 *
 * Every function returns 0 on success and -1 on an invalid argument.
 * Arrays are dense, row-major, fp64 (shapes and starts int64).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_LEVELS 64

static int dims_ok(int64_t B, int64_t S, int64_t Q, int64_t M, int64_t D,
                   int64_t L, int64_t K) {
    return B >= 0 && S >= 1 && Q >= 0 && M >= 1 && D >= 1 && L >= 1 &&
           L <= ORACLE_MAX_LEVELS && K >= 1;
}

/* nthreads > 0: that many OpenMP threads; 0: every processor (set each call,
 * since the OpenMP thread count persists between calls). */
static void set_threads(int nthreads) {
#ifdef _OPENMP
    omp_set_num_threads(nthreads > 0 ? nthreads : omp_get_num_procs());
#else
    (void)nthreads;
#endif
}

/* Pixel-space coordinates of one sample and its four bilinear corners [C1-bil].
 * Returns 0 when no corner can be inside the map (the coordinate is not a
 * finite number, or it lies a full pixel or more outside the map). Skipping
 * such a sample is what the definition does anyway -- every corner fails the
 * zero-padding test -- and it avoids converting a huge or NaN double to an
 * integer. */
typedef struct {
    int64_t yy[4], xx[4]; /* corner pixel coordinates, order 00, 01, 10, 11 */
    double wgt[4];        /* bilinear weights of the four corners           */
    int inside[4];        /* 1 if the corner lies in [0,W) x [0,H)         */
    double lx, ly;        /* fractional parts                               */
} corners_t;

static int sample_corners(double loc_x, double loc_y, int64_t H, int64_t W,
                          corners_t *c) {
    double x = loc_x * (double)W - 0.5; /* grid_sample(align_corners=False) */
    double y = loc_y * (double)H - 0.5;
    if (!(x > -2.0 && x < (double)W + 1.0 && y > -2.0 && y < (double)H + 1.0))
        return 0;
    double x0 = floor(x), y0 = floor(y);
    double lx = x - x0, ly = y - y0;
    int64_t ix = (int64_t)x0, iy = (int64_t)y0;
    c->lx = lx;
    c->ly = ly;
    c->yy[0] = iy;     c->xx[0] = ix;     c->wgt[0] = (1.0 - lx) * (1.0 - ly);
    c->yy[1] = iy;     c->xx[1] = ix + 1; c->wgt[1] = lx * (1.0 - ly);
    c->yy[2] = iy + 1; c->xx[2] = ix;     c->wgt[2] = (1.0 - lx) * ly;
    c->yy[3] = iy + 1; c->xx[3] = ix + 1; c->wgt[3] = lx * ly;
    int any = 0;
    for (int i = 0; i < 4; ++i) {
        c->inside[i] = (0 <= c->xx[i] && c->xx[i] < W && 0 <= c->yy[i] && c->yy[i] < H);
        any |= c->inside[i];
    }
    return any;
}

/* Forward: out[b,q,m*D+d] = sum_{l,k} a * sum_{corners inside} wgt * value[b, start_l+yy*W+xx, m, d]
 * [C1-eq], [C1-bil], [C1-loop]. Parallel over (b,q); each output row is
 * written by one thread, so the result does not depend on the thread count. */
int msda_oracle_forward(const double *value, const int64_t *shapes,
                        const int64_t *starts, const double *loc,
                        const double *attn, double *out, int64_t B, int64_t S,
                        int64_t Q, int64_t M, int64_t D, int64_t L, int64_t K,
                        int nthreads) {
    if (!dims_ok(B, S, Q, M, D, L, K)) return -1;
    set_threads(nthreads);
    int64_t BQ = B * Q;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t bq = 0; bq < BQ; ++bq) {
        int64_t b = bq / Q;
        double *o = out + bq * M * D;
        memset(o, 0, sizeof(double) * (size_t)(M * D));
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t l = 0; l < L; ++l) {
                int64_t H = shapes[2 * l], W = shapes[2 * l + 1];
                for (int64_t k = 0; k < K; ++k) {
                    int64_t s = ((bq * M + m) * L + l) * K + k;
                    double a = attn[s];
                    corners_t c;
                    if (!sample_corners(loc[2 * s], loc[2 * s + 1], H, W, &c)) continue;
                    for (int i = 0; i < 4; ++i) {
                        if (!c.inside[i]) continue; /* zeros padding */
                        const double *v =
                            value + ((b * S + starts[l] + c.yy[i] * W + c.xx[i]) * M + m) * D;
                        for (int64_t d = 0; d < D; ++d) o[m * D + d] += a * c.wgt[i] * v[d];
                    }
                }
            }
        }
    }
    return 0;
}

/* Backward [C1-ch5], derived from the forward above. For one sample with
 * g = grad_out[b,q,m,:] and s_c = <g, value[corner c]> (0 for a corner outside
 * the map):
 *   d out/d a          -> grad_attn = sum_c wgt_c * s_c
 *   d out/d value[c]   -> grad_value[c] += a * wgt_c * g
 *   d/d lx             =  a * ((1-ly)(s_01 - s_00) + ly (s_11 - s_10))
 *   d/d ly             =  a * ((1-lx)(s_10 - s_00) + lx (s_11 - s_01))
 *   x = loc_x*W - 0.5  -> grad_loc_x = W * d/d lx,  grad_loc_y = H * d/d ly
 * (lx = x - floor(x) has derivative 1 away from integer x; at an integer the
 * floor picks the cell, so the derivative is the one-sided one from above.)
 * Parallel over (b,m): grad_value[b,:,m,:] and the (b,.,m) rows of grad_loc
 * and grad_attn belong to exactly one (b,m), so every sum runs in one fixed
 * serial order and the result is deterministic. */
int msda_oracle_backward(const double *value, const int64_t *shapes,
                         const int64_t *starts, const double *loc,
                         const double *attn, const double *grad_out,
                         double *grad_value, double *grad_loc,
                         double *grad_attn, int64_t B, int64_t S, int64_t Q,
                         int64_t M, int64_t D, int64_t L, int64_t K,
                         int nthreads) {
    if (!dims_ok(B, S, Q, M, D, L, K)) return -1;
    set_threads(nthreads);
    memset(grad_value, 0, sizeof(double) * (size_t)(B * S * M * D));
    int64_t BM = B * M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bm = 0; bm < BM; ++bm) {
        int64_t b = bm / M, m = bm % M;
        for (int64_t q = 0; q < Q; ++q) {
            const double *g = grad_out + ((b * Q + q) * M + m) * D;
            for (int64_t l = 0; l < L; ++l) {
                int64_t H = shapes[2 * l], W = shapes[2 * l + 1];
                for (int64_t k = 0; k < K; ++k) {
                    int64_t s = (((b * Q + q) * M + m) * L + l) * K + k;
                    double a = attn[s];
                    corners_t c;
                    grad_attn[s] = 0.0;
                    grad_loc[2 * s] = 0.0;
                    grad_loc[2 * s + 1] = 0.0;
                    if (!sample_corners(loc[2 * s], loc[2 * s + 1], H, W, &c)) continue;
                    double sc[4] = {0.0, 0.0, 0.0, 0.0};
                    for (int i = 0; i < 4; ++i) {
                        if (!c.inside[i]) continue;
                        int64_t row = (b * S + starts[l] + c.yy[i] * W + c.xx[i]) * M + m;
                        const double *v = value + row * D;
                        double *gv = grad_value + row * D;
                        double dot = 0.0;
                        for (int64_t d = 0; d < D; ++d) {
                            dot += g[d] * v[d];
                            gv[d] += a * c.wgt[i] * g[d];
                        }
                        sc[i] = dot;
                    }
                    double ga = 0.0;
                    for (int i = 0; i < 4; ++i) ga += c.wgt[i] * sc[i];
                    grad_attn[s] = ga;
                    double dlx = (1.0 - c.ly) * (sc[1] - sc[0]) + c.ly * (sc[3] - sc[2]);
                    double dly = (1.0 - c.lx) * (sc[2] - sc[0]) + c.lx * (sc[3] - sc[1]);
                    grad_loc[2 * s] = a * (double)W * dlx;
                    grad_loc[2 * s + 1] = a * (double)H * dly;
                }
            }
        }
    }
    return 0;
}

/* Integer parts of every sample [C1-bil], [C1-loop]: for sample s (flattened
 * (b,q,m,l,k)) and corner c in order 00, 01, 10, 11, idx[4*s+c] is the value
 * row start_l + yy*W + xx of a corner inside the map and -1 for a corner
 * outside it. These are the integers the kernels must reproduce bit for bit. */
int msda_oracle_corners(const int64_t *shapes, const int64_t *starts,
                        const double *loc, int64_t BQM, int64_t L, int64_t K,
                        int32_t *idx) {
    if (BQM < 0 || L < 1 || L > ORACLE_MAX_LEVELS || K < 1) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < BQM; ++t) {
        for (int64_t l = 0; l < L; ++l) {
            int64_t H = shapes[2 * l], W = shapes[2 * l + 1];
            for (int64_t k = 0; k < K; ++k) {
                int64_t s = (t * L + l) * K + k;
                corners_t c;
                int any = sample_corners(loc[2 * s], loc[2 * s + 1], H, W, &c);
                for (int i = 0; i < 4; ++i)
                    idx[4 * s + i] = (any && c.inside[i])
                                         ? (int32_t)(starts[l] + c.yy[i] * W + c.xx[i])
                                         : -1;
            }
        }
    }
    return 0;
}
