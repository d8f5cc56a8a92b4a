// Forward gather kernel of multi-scale deformable attention.
//
// Computes (Deformable DETR walk-through, "2.2.4 源码分析",
// ms_deform_attn_core_pytorch):
//   out[b, q, m*D + d] = sum_{l,p} a[b,q,m,l,p] * sum_c w_c * value[b, key_c, m, d]
//
// Work decomposition.  A "row" is one (b, q, m) triple: its L*P samples are
// contiguous in sampling_locations / attention_weights and its D outputs are
// contiguous in output.  A warp is split into 32/kLanes lane groups; each
// group owns one row at a time and each lane owns kVPL 16-byte vectors of
// the head's D channels, so one corner row of value (D*e bytes) is read by
// the group as coalesced 128-bit loads.
//
// Each warp iteration has two phases:
//   1. footprint: the warp's lanes take the iteration's samples one per lane
//      (coalesced loads of locations and weights), compute the pixel
//      coordinates, cell, corner validity and the four corner weights with
//      the attention weight folded in, once per sample, into shared memory;
//   2. gather: every group walks its row's samples, reads each footprint
//      as a shared-memory broadcast and issues one 128-bit load per live
//      corner and vector, accumulating 4 FMAs per channel per sample in fp32.
// Corners off the map or with weight 0 are not read at all.
#pragma once

#include "msda_device.cuh"

namespace msda {

template <typename T, int kLanes, int kVPL>
__global__ void __launch_bounds__(kThreadsPerCta)
    forward_kernel(const T* __restrict__ value, const int64_t* __restrict__ spatial_shapes,
                   const int64_t* __restrict__ level_start_index, const T* __restrict__ loc,
                   const T* __restrict__ attn, T* __restrict__ out, int num_keys, int num_heads,
                   int head_dim, int num_levels, int num_points, int num_queries, int rows,
                   int rows_per_warp) {
    constexpr int kGroups = 32 / kLanes;
    constexpr int V = IO<T>::kVec;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    LevelInfo* s_levels = reinterpret_cast<LevelInfo*>(smem_raw);
    const int LP = num_levels * num_points;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / kLanes, li = lane % kLanes;
    const int pts_per_iter = kGroups * LP;
    float4* s_w = reinterpret_cast<float4*>(smem_raw + sizeof(LevelInfo) * kMaxLevels) +
                  (size_t)warp * pts_per_iter;
    int2* s_k = reinterpret_cast<int2*>(
                    smem_raw + sizeof(LevelInfo) * kMaxLevels +
                    sizeof(float4) * (size_t)kWarpsPerCta * pts_per_iter) +
                (size_t)warp * pts_per_iter;

    load_level_table(s_levels, spatial_shapes, level_start_index, num_levels, num_keys);
    __syncthreads();

    const int64_t MD = (int64_t)num_heads * head_dim;
    const int nvec = head_dim / V;
    const int row0 = (blockIdx.x * kWarpsPerCta + warp) * rows_per_warp;

    for (int it = 0; it < rows_per_warp; it += kGroups) {
        const int rbase = row0 + it;
        if (rbase >= rows) break;
        // ---- phase 1: one footprint per sample, one sample per lane
        const int64_t pt0 = (int64_t)rbase * LP;
        for (int t = lane; t < pts_per_iter; t += 32) {
            const int rl = t / LP;
            float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f);
            int2 k2 = make_int2(0, 0);
            if (rbase + rl < rows) {
                const int j = t - rl * LP;
                const LevelInfo lv = s_levels[j / num_points];
                const float2 xy = IO<T>::load_xy(loc + 2 * (pt0 + t));
                const float a = IO<T>::load_one(attn + pt0 + t);
                const float x = fmaf(xy.x, (float)lv.W, -0.5f);
                const float y = fmaf(xy.y, (float)lv.H, -0.5f);
                Footprint f = make_footprint(x, y, lv);
                w4 = make_float4(a * f.w[0], a * f.w[1], a * f.w[2], a * f.w[3]);
                unsigned mask = f.info & 15u;
                mask &= (w4.x != 0.f ? 1u : 0u) | (w4.y != 0.f ? 2u : 0u) |
                        (w4.z != 0.f ? 4u : 0u) | (w4.w != 0.f ? 8u : 0u);
                k2 = make_int2(f.key00, (int)((f.info & ~15u) | mask));
            }
            s_w[t] = w4;
            s_k[t] = k2;
        }
        __syncwarp();

        // ---- phase 2: gather, one row per lane group
        const int r = rbase + g;
        if (r < rows) {
            const int m = r % num_heads;
            const int b = (r / num_heads) / num_queries;
            const T* vb = value + ((int64_t)b * num_keys * num_heads + m) * head_dim;
            float acc[kVPL][V];
#pragma unroll
            for (int k = 0; k < kVPL; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[k][e] = 0.f;
            const float4* sw = s_w + g * LP;
            const int2* sk = s_k + g * LP;
#pragma unroll 2
            for (int j = 0; j < LP; ++j) {
                const float4 w4 = sw[j];
                const int2 k2 = sk[j];
                const unsigned mask = (unsigned)k2.y & 15u;
                const int W = (int)((unsigned)k2.y >> 4);
                const float wc[4] = {w4.x, w4.y, w4.z, w4.w};
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
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < kVPL; ++k)
#pragma unroll
                        for (int e = 0; e < V; ++e) acc[k][e] = fmaf(wc[c], v[c][k][e], acc[k][e]);
            }
            T* o = out + (int64_t)r * head_dim;
#pragma unroll
            for (int k = 0; k < kVPL; ++k) {
                const int vi = li + k * kLanes;
                if (vi < nvec) IO<T>::store_vec(o + vi * V, acc[k]);
            }
        }
        __syncwarp();
    }
}

}  // namespace msda
