// Backward gather/scatter kernel of multi-scale deformable attention.
//
// For every sample (b, q, m, l, p) with attention weight a, fractions
// (fx, fy), corner weights w_c and corner rows v_c (zero off the map), and
// grad_output row g (DQ-DETR ops page, MSDeformAttnFunction.backward returns
// these three gradients; the formulas are the derivative of the walk-through's
// ms_deform_attn_core_pytorch sum):
//   grad_attn[pt]       = sum_d g_d * sum_c w_c v_c,d
//   grad_loc[pt].x      = W * a * sum_d g_d ((1-fy)(v01-v00) + fy (v11-v10))_d
//   grad_loc[pt].y      = H * a * sum_d g_d ((1-fx)(v10-v00) + fx (v11-v01))_d
//   grad_value[b,key_c,m,d] += a * w_c * g_d          (fp32 vector red to global)
//
// Decomposition as in the forward (one row per lane group, 16-byte vectors per
// lane).  The channel sums for the three per-sample gradients are reduced
// across the group's lanes with xor shuffles; the per-sample results are
// staged in shared memory and written back coalesced once the group's rows
// are done.  grad_value is accumulated in fp32 (the caller's fp32 grad_value,
// or the fp32 workspace for bf16) with red.global.add.v4.f32.
#pragma once

#include "msda_device.cuh"

namespace msda {

template <typename T, int kLanes, int kVPL>
__global__ void __launch_bounds__(kThreadsPerCta)
    backward_kernel(const T* __restrict__ value, const int64_t* __restrict__ spatial_shapes,
                    const int64_t* __restrict__ level_start_index, const T* __restrict__ loc,
                    const T* __restrict__ attn, const T* __restrict__ grad_out,
                    float* __restrict__ grad_value_f32, T* __restrict__ grad_loc,
                    T* __restrict__ grad_attn, int num_keys, int num_heads, int head_dim,
                    int num_levels, int num_points, int num_queries, int rows,
                    int rows_per_warp) {
    constexpr int kGroups = 32 / kLanes;
    constexpr int V = IO<T>::kVec;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    LevelInfo* s_levels = reinterpret_cast<LevelInfo*>(smem_raw);
    const int LP = num_levels * num_points;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / kLanes, li = lane % kLanes;
    const int pts_per_iter = kGroups * LP;
    const size_t per_warp = (size_t)pts_per_iter;
    unsigned char* base = smem_raw + sizeof(LevelInfo) * kMaxLevels;
    float4* s_w = reinterpret_cast<float4*>(base) + warp * per_warp;
    float4* s_aux = reinterpret_cast<float4*>(base) + (kWarpsPerCta + warp) * per_warp;
    float4* s_res = reinterpret_cast<float4*>(base) + (2 * kWarpsPerCta + warp) * per_warp;
    int2* s_k = reinterpret_cast<int2*>(reinterpret_cast<float4*>(base) +
                                        3 * kWarpsPerCta * per_warp) +
                warp * per_warp;

    load_level_table(s_levels, spatial_shapes, level_start_index, num_levels, num_keys);
    __syncthreads();

    const int64_t MD = (int64_t)num_heads * head_dim;
    const int nvec = head_dim / V;
    const int row0 = (blockIdx.x * kWarpsPerCta + warp) * rows_per_warp;

    for (int it = 0; it < rows_per_warp; it += kGroups) {
        const int rbase = row0 + it;
        if (rbase >= rows) break;
        const int64_t pt0 = (int64_t)rbase * LP;
        // ---- phase 1: footprints (bilinear weights without a; validity mask)
        for (int t = lane; t < pts_per_iter; t += 32) {
            const int rl = t / LP;
            float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 aux = make_float4(0.f, 0.f, 0.f, 0.f);
            int2 k2 = make_int2(0, 0);
            if (rbase + rl < rows) {
                const int j = t - rl * LP;
                const LevelInfo lv = s_levels[j / num_points];
                const float2 xy = IO<T>::load_xy(loc + 2 * (pt0 + t));
                const float a = IO<T>::load_one(attn + pt0 + t);
                const float x = fmaf(xy.x, (float)lv.W, -0.5f);
                const float y = fmaf(xy.y, (float)lv.H, -0.5f);
                const Footprint f = make_footprint(x, y, lv);
                w4 = make_float4(f.w[0], f.w[1], f.w[2], f.w[3]);
                aux = make_float4(a, f.fx, f.fy, 0.f);
                k2 = make_int2(f.key00, (int)f.info);
            }
            s_w[t] = w4;
            s_aux[t] = aux;
            s_k[t] = k2;
        }
        __syncwarp();

        // ---- phase 2: gather corners, reduce per-sample grads, scatter grad_value.
        // Every lane runs the sample loop (the group sums shuffle across the
        // whole warp); a group past the last row has all-zero footprints, so
        // it reads and writes nothing.
        const bool active = rbase + g < rows;
        const int r = active ? rbase + g : rbase;
        {
            const int m = r % num_heads;
            const int b = (r / num_heads) / num_queries;
            const int64_t vrow = ((int64_t)b * num_keys * num_heads + m) * head_dim;
            const T* vb = value + vrow;
            float* gvb = grad_value_f32 + vrow;
            float gr[kVPL][V];
#pragma unroll
            for (int k = 0; k < kVPL; ++k) {
                const int vi = li + k * kLanes;
                if (active && vi < nvec) {
                    IO<T>::load_vec_stream(grad_out + (int64_t)r * head_dim + vi * V, gr[k]);
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e) gr[k][e] = 0.f;
                }
            }
            const float4* sw = s_w + g * LP;
            const float4* sa = s_aux + g * LP;
            const int2* sk = s_k + g * LP;
            for (int j = 0; j < LP; ++j) {
                const float4 w4 = sw[j];
                const float4 ax = sa[j];
                const int2 k2 = sk[j];
                const unsigned mask = (unsigned)k2.y & 15u;
                const int W = (int)((unsigned)k2.y >> 4);
                const float a = ax.x, fx = ax.y, fy = ax.z;
                float v[4][kVPL][V];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const T* p = vb + (int64_t)corner_key(k2.x, W, c) * MD;
#pragma unroll
                    for (int k = 0; k < kVPL; ++k) {
                        const int vi = li + k * kLanes;
                        if ((mask >> c & 1u) && vi < nvec) {
                            IO<T>::load_vec(p + vi * V, v[c][k]);
                        } else {
#pragma unroll
                            for (int e = 0; e < V; ++e) v[c][k][e] = 0.f;
                        }
                    }
                }
                float pa = 0.f, px = 0.f, py = 0.f;
                const float gy0 = 1.f - fy, gx0 = 1.f - fx;
#pragma unroll
                for (int k = 0; k < kVPL; ++k)
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float v00 = v[0][k][e], v01 = v[1][k][e];
                        const float v10 = v[2][k][e], v11 = v[3][k][e];
                        const float s = w4.x * v00 + w4.y * v01 + w4.z * v10 + w4.w * v11;
                        const float gd = gr[k][e];
                        pa = fmaf(gd, s, pa);
                        px = fmaf(gd, gy0 * (v01 - v00) + fy * (v11 - v10), px);
                        py = fmaf(gd, gx0 * (v10 - v00) + fx * (v11 - v01), py);
                    }
                // scatter a * w_c * g into grad_value for every corner on the map
                const float aw[4] = {a * w4.x, a * w4.y, a * w4.z, a * w4.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (!(mask >> c & 1u)) continue;
                    float* q = gvb + (int64_t)corner_key(k2.x, W, c) * MD;
#pragma unroll
                    for (int k = 0; k < kVPL; ++k) {
                        const int vi = li + k * kLanes;
                        if (vi < nvec) {
#pragma unroll
                            for (int e = 0; e < V; e += 4)
                                red_add_v4(q + vi * V + e, aw[c] * gr[k][e], aw[c] * gr[k][e + 1],
                                           aw[c] * gr[k][e + 2], aw[c] * gr[k][e + 3]);
                        }
                    }
                }
                pa = group_sum<kLanes>(pa);
                px = group_sum<kLanes>(px);
                py = group_sum<kLanes>(py);
                if (li == 0) {
                    const LevelInfo lv = s_levels[j / num_points];
                    s_res[g * LP + j] = make_float4((float)lv.W * (a * px), (float)lv.H * (a * py),
                                                    pa, 0.f);
                }
            }
        }
        __syncwarp();
        // ---- write back the per-sample gradients of the iteration, coalesced
        for (int t = lane; t < pts_per_iter; t += 32) {
            if (rbase + t / LP < rows) {
                const float4 res = s_res[t];
                IO<T>::store_xy(grad_loc + 2 * (pt0 + t), res.x, res.y);
                IO<T>::store_one(grad_attn + pt0 + t, res.z);
            }
        }
        __syncwarp();
    }
}

}  // namespace msda
