/*
 * Multi-scale deformable attention: slow, plain CPU oracle in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call this file.  It shares
 * no code, header, table or helper with the CUDA library, and the library
 * never calls it.
 *
 * What it computes (Deformable DETR walk-through, "2.2.4 源码分析",
 * ms_deform_attn_core_pytorch; MSDeformAttn.forward for the (W, H)
 * normaliser; Ascend DrivingSDK page "multi_scale_deformable_attn" for the
 * argument shapes):
 *
 *   out[b, q, m*D + d] = sum_l sum_p a[b,q,m,l,p] *
 *                        bilinear_zero(V_{b,l,m}(., ., d), x, y)
 *
 *   V_{b,l,m}(y, x, d) = value[b, lsi[l] + y*W_l + x, m, d]   (row-major levels)
 *   x = loc_x * W_l - 0.5,  y = loc_y * H_l - 0.5
 *
 * which is grid_sample(mode=bilinear, padding_mode=zeros,
 * align_corners=False) at grid = 2*loc - 1: the sample is the weighted sum
 * of the four pixels around (x, y), each weighted by the product of its
 * 1-D distances' complements, and a pixel outside the map counts as 0.
 *
 * Readings the pages leave open (all shared with the CUDA side by contract,
 * not by code):
 *  - coord_mode 0: x and y are rounded once to binary32, i.e. the
 *    correctly rounded fused multiply-add fmaf(loc, W, -0.5f); the cell
 *    (floor) and the fractions then come out bit-identical to a GPU that
 *    uses one fp32 FMA.  coord_mode 1 keeps them exact in fp64 (used by the
 *    finite-difference and library cross-checks).
 *  - a sample contributes (and receives gradient) only when
 *    -1 < x < W and -1 < y < H; at those bounds every pixel weight is 0.
 *  - the gradient at integer x (or y) is the one of the cell
 *    [floor(x), floor(x) + 1], i.e. the right derivative.
 *  - attention weights are used as given (the softmax belongs to the caller).
 *
 * Backward (the analytic derivative of the sum above):
 *   grad_value[b, key_c, m, d] += a * w_c * g[d]
 *   grad_attn[b,q,m,l,p]        = sum_d g[d] * s[d],  s = sum_c w_c v_c
 *   grad_loc_x = W * a * sum_d g[d] ((1-fy)(v01-v00) + fy (v11-v10))
 *   grad_loc_y = H * a * sum_d g[d] ((1-fx)(v10-v00) + fx (v11-v01))
 * with v_yx the pixel at (y0+y, x0+x) (0 outside the map).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1 };

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Position of a sample along one axis in pixel units of its level. */
static double pixel_coord(double loc, int64_t size, int coord_mode) {
    if (coord_mode == 0)
        return (double)fmaf((float)loc, (float)size, -0.5f);
    return loc * (double)size - 0.5;
}

static int check_dims(int bs, int num_keys, int num_heads, int head_dim, int num_levels,
                      int num_points, int num_queries) {
    if (bs < 0 || num_keys < 0 || num_heads < 0 || head_dim < 0 || num_levels < 0 ||
        num_points < 0 || num_queries < 0)
        return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/* One sample's bilinear footprint: up to four pixels with their keys and weights. */
typedef struct {
    int in_range;
    double fx, fy;         /* fractions inside the cell */
    int64_t key[4];        /* order: (y0,x0), (y0,x0+1), (y0+1,x0), (y0+1,x0+1) */
    int valid[4];
    double w[4];           /* bilinear weights (without the attention weight) */
} footprint;

static void make_footprint(double loc_x, double loc_y, int64_t H, int64_t W, int64_t start,
                           int coord_mode, footprint* f) {
    double x = pixel_coord(loc_x, W, coord_mode);
    double y = pixel_coord(loc_y, H, coord_mode);
    f->in_range = (x > -1.0 && x < (double)W && y > -1.0 && y < (double)H);
    if (!f->in_range) return;
    double x0 = floor(x), y0 = floor(y);
    f->fx = x - x0;
    f->fy = y - y0;
    for (int c = 0; c < 4; ++c) {
        int64_t xc = (int64_t)x0 + (c & 1);
        int64_t yc = (int64_t)y0 + (c >> 1);
        double wx = (c & 1) ? f->fx : 1.0 - f->fx;
        double wy = (c >> 1) ? f->fy : 1.0 - f->fy;
        f->w[c] = wx * wy;
        f->valid[c] = (xc >= 0 && xc < W && yc >= 0 && yc < H);
        f->key[c] = f->valid[c] ? start + yc * W + xc : -1;
    }
}

int oracle_forward(const double* value, const int64_t* spatial_shapes,
                   const int64_t* level_start_index, const double* sampling_locations,
                   const double* attention_weights, double* output, int bs, int num_keys,
                   int num_heads, int head_dim, int num_levels, int num_points, int num_queries,
                   int coord_mode, int threads) {
    if (check_dims(bs, num_keys, num_heads, head_dim, num_levels, num_points, num_queries))
        return ORACLE_ERR_ARG;
    const int64_t M = num_heads, D = head_dim, L = num_levels, P = num_points;
    const int64_t K = num_keys, Q = num_queries;
    const int64_t rows = (int64_t)bs * Q;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t bq = 0; bq < rows; ++bq) {
        const int64_t b = bq / Q;
        for (int64_t m = 0; m < M; ++m) {
            double* o = output + (bq * M + m) * D;
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t l = 0; l < L; ++l) {
                const int64_t H = spatial_shapes[2 * l], W = spatial_shapes[2 * l + 1];
                for (int64_t p = 0; p < P; ++p) {
                    const int64_t pt = ((bq * M + m) * L + l) * P + p;
                    footprint f;
                    make_footprint(sampling_locations[2 * pt], sampling_locations[2 * pt + 1], H,
                                   W, level_start_index[l], coord_mode, &f);
                    if (!f.in_range) continue;
                    const double a = attention_weights[pt];
                    for (int c = 0; c < 4; ++c) {
                        if (!f.valid[c]) continue;
                        if (f.key[c] < 0 || f.key[c] >= K) continue; /* inconsistent shapes: skip */
                        const double* v = value + ((b * K + f.key[c]) * M + m) * D;
                        const double s = a * f.w[c];
                        for (int64_t d = 0; d < D; ++d) o[d] += s * v[d];
                    }
                }
            }
        }
    }
    return ORACLE_OK;
}

int oracle_backward(const double* value, const int64_t* spatial_shapes,
                    const int64_t* level_start_index, const double* sampling_locations,
                    const double* attention_weights, const double* grad_output,
                    double* grad_value, double* grad_sampling_loc, double* grad_attention_weights,
                    int bs, int num_keys, int num_heads, int head_dim, int num_levels,
                    int num_points, int num_queries, int coord_mode, int threads) {
    if (check_dims(bs, num_keys, num_heads, head_dim, num_levels, num_points, num_queries))
        return ORACLE_ERR_ARG;
    const int64_t M = num_heads, D = head_dim, L = num_levels, P = num_points;
    const int64_t K = num_keys, Q = num_queries;
    memset(grad_value, 0, sizeof(double) * (size_t)(bs * K * M * D));
    /* One (b, m) slice per task: each task owns grad_value[b, :, m, :] alone,
       so the sums are race-free and in a fixed order (deterministic). */
    const int64_t tasks = (int64_t)bs * M;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t t = 0; t < tasks; ++t) {
        const int64_t b = t / M, m = t % M;
        double* corner = (double*)malloc(sizeof(double) * (size_t)(4 * (D > 0 ? D : 1)));
        for (int64_t q = 0; q < Q; ++q) {
            const int64_t bq = b * Q + q;
            const double* g = grad_output + (bq * M + m) * D;
            for (int64_t l = 0; l < L; ++l) {
                const int64_t H = spatial_shapes[2 * l], W = spatial_shapes[2 * l + 1];
                for (int64_t p = 0; p < P; ++p) {
                    const int64_t pt = ((bq * M + m) * L + l) * P + p;
                    footprint f;
                    make_footprint(sampling_locations[2 * pt], sampling_locations[2 * pt + 1], H,
                                   W, level_start_index[l], coord_mode, &f);
                    if (!f.in_range) {
                        grad_sampling_loc[2 * pt] = 0.0;
                        grad_sampling_loc[2 * pt + 1] = 0.0;
                        grad_attention_weights[pt] = 0.0;
                        continue;
                    }
                    const double a = attention_weights[pt];
                    for (int c = 0; c < 4; ++c) {
                        const int ok = f.valid[c] && f.key[c] >= 0 && f.key[c] < K;
                        const double* v = ok ? value + ((b * K + f.key[c]) * M + m) * D : NULL;
                        for (int64_t d = 0; d < D; ++d) corner[c * D + d] = ok ? v[d] : 0.0;
                    }
                    double ga = 0.0, gx = 0.0, gy = 0.0;
                    for (int64_t d = 0; d < D; ++d) {
                        const double v00 = corner[d], v01 = corner[D + d];
                        const double v10 = corner[2 * D + d], v11 = corner[3 * D + d];
                        const double s = f.w[0] * v00 + f.w[1] * v01 + f.w[2] * v10 + f.w[3] * v11;
                        ga += g[d] * s;
                        gx += g[d] * ((1.0 - f.fy) * (v01 - v00) + f.fy * (v11 - v10));
                        gy += g[d] * ((1.0 - f.fx) * (v10 - v00) + f.fx * (v11 - v01));
                    }
                    grad_attention_weights[pt] = ga;
                    grad_sampling_loc[2 * pt] = (double)W * a * gx;
                    grad_sampling_loc[2 * pt + 1] = (double)H * a * gy;
                    for (int c = 0; c < 4; ++c) {
                        if (!f.valid[c] || f.key[c] < 0 || f.key[c] >= K) continue;
                        double* gv = grad_value + ((b * K + f.key[c]) * M + m) * D;
                        const double s = a * f.w[c];
                        for (int64_t d = 0; d < D; ++d) gv[d] += s * g[d];
                    }
                }
            }
        }
        free(corner);
    }
    return ORACLE_OK;
}

/*
 * Rows of value that a forward pass reads with a non-zero pixel weight,
 * counted once each: distinct (b, key, m) triples.  Used to report the
 * decoder workload's "touched bytes" roofline.  mark must hold bs*K*M bytes.
 */
int64_t oracle_touched_rows(const int64_t* spatial_shapes, const int64_t* level_start_index,
                            const double* sampling_locations, const double* attention_weights,
                            unsigned char* mark, int bs, int num_keys, int num_heads,
                            int num_levels, int num_points, int num_queries, int coord_mode) {
    const int64_t M = num_heads, L = num_levels, P = num_points, K = num_keys, Q = num_queries;
    memset(mark, 0, (size_t)(bs * K * M));
    int64_t count = 0;
    for (int64_t bq = 0; bq < (int64_t)bs * Q; ++bq) {
        const int64_t b = bq / Q;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t l = 0; l < L; ++l) {
                const int64_t H = spatial_shapes[2 * l], W = spatial_shapes[2 * l + 1];
                for (int64_t p = 0; p < P; ++p) {
                    const int64_t pt = ((bq * M + m) * L + l) * P + p;
                    footprint f;
                    make_footprint(sampling_locations[2 * pt], sampling_locations[2 * pt + 1], H,
                                   W, level_start_index[l], coord_mode, &f);
                    if (!f.in_range || attention_weights[pt] == 0.0) continue;
                    for (int c = 0; c < 4; ++c) {
                        if (!f.valid[c] || f.key[c] < 0 || f.key[c] >= K || f.w[c] == 0.0) continue;
                        unsigned char* mk = mark + (b * K + f.key[c]) * M + m;
                        if (!*mk) { *mk = 1; ++count; }
                    }
                }
            }
    }
    return count;
}
