// Forward gather kernel of multi-scale deformable attention.
//
// Computes (Deformable DETR walk-through, "2.2.4 源码分析",
// ms_deform_attn_core_pytorch):
//   out[b, q, m*D + d] = sum_{l,p} a[b,q,m,l,p] * sum_c w_c * value[b, key_c, m, d]
//
// One warp tile = kGroups consecutive queries of one (b, m) (see
// msda_device.cuh); a CTA's warps take consecutive tiles of a contiguous
// range.  The tile's samples are handled in rounds of kSamplesPerWarp, and
// the locations and weights of the next round are loaded while the current
// round gathers:
//   1. footprint: each lane takes two samples (coalesced loads of locations
//      and weights), computes the cell, the four corner keys (-1 when off
//      the map) and the four corner weights with the attention weight folded
//      in, and stores them as two 16-byte records in shared memory (per-group
//      stride padded so the four groups' reads never share a bank);
//   2. gather: each group walks its query's samples; per sample one 16-byte
//      broadcast read of keys and of weights, one 128-bit load per lane and
//      live corner, and 4 FMAs per channel, accumulated in fp32 registers.
// The group writes its query's head_dim outputs once, as 128-bit stores.
#pragma once

#include "msda_device.cuh"

namespace msda {

// Unroll of the gather loop over a group's samples: 2, and 4 for fp32 rows of
// 128 bytes in 8-lane groups (the encoder shape: 2% faster there; 4 was 5%
// slower for bf16).
#ifndef MSDA_FWD_UNROLL
#define MSDA_FWD_UNROLL 2
#endif
#ifndef MSDA_FWD_UNROLL_F32_128
#define MSDA_FWD_UNROLL_F32_128 4
#endif
#ifndef MSDA_FWD_MIN_BLOCKS
#define MSDA_FWD_MIN_BLOCKS 4
#endif
// Packed fp32 FMA (two channels per instruction) in the gather's accumulation of
// 16-bit rows: bf16 encoder forward 303 -> 287 us; fp32 rows measured slower
// (164.6 -> 166.3 us, the 64-register build spilled), so they keep scalar FMAs.
#ifndef MSDA_FWD_PACKED
#define MSDA_FWD_PACKED 1
#endif
// Plain 16-bit rows in groups of at most 8 lanes: dead corners and idle lanes
// load the zero row (g_zero_row) instead of a predicated load into zero-filled
// registers, which the ALU-bound widening of those rows felt (encoder forward
// bf16 274 -> 262 us, fp16 283 -> 274 us).  Measured slower elsewhere: fp32 rows
// (158 -> 162 us), the fused 16-bit forward (345 -> 367 us) and the backward
// (fp32 393 -> 397 us, bf16 741 -> 805 us with 180 bytes of spills).
#ifndef MSDA_FWD_ZERO_ROW
#define MSDA_FWD_ZERO_ROW 1
#endif
// The instantiations that take the zero row: plain 16-bit rows, one vector per
// lane, groups of at most 8 lanes of at most 16 bytes.
template <typename T, int kLanes, int kVPL, int kVB, int kRef>
__host__ __device__ constexpr bool forward_zero_row() {
    return MSDA_FWD_ZERO_ROW != 0 && sizeof(T) == 2 && kRef == 0 && kVPL == 1 && kLanes <= 8 &&
           kLanes * kVB <= 128;
}
#define MSDA_PRAGMA(x) _Pragma(#x)
#define MSDA_UNROLL(n) MSDA_PRAGMA(unroll n)

// Stores the footprint records of the round fetched in f.
// kRef: 0 on the plain path; 2 or 4, the width of the reference points, on the
// fused entry points, where the round holds offsets and softmax weights;
// the location is formed from pf's reference point first.
template <int kSPG, int kStride, int kRef>
__device__ __forceinline__ void forward_records(int4* wk, float4* ww, const SampleFetch& f,
                                                const PrepFetch& pf, float points_f,
                                                const unsigned char* __restrict__ mrow,
                                                const LevelInfo* s_levels,
                                                const unsigned char* s_level_of, int r0,
                                                int lane) {
#pragma unroll
    for (int h = 0; h < kSamplesPerWarp / 32; ++h) {
        const int s = lane + 32 * h;
        const int sg = s / kSPG, sj = s % kSPG;
        int4 key = make_int4(-1, -1, -1, -1);
        float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
        if (f.ok[h]) {
            const LevelInfo lv = s_levels[s_level_of[r0 + sj]];
            const float a = f.a[h];
            float2 xy = f.xy[h];
            if constexpr (kRef != 0) {
                xy = prep_location<kRef>(pf.rxy[h], pf.rwh[h], xy, (float)lv.W, (float)lv.H,
                                         points_f);
            }
            Footprint fp = make_footprint(fmaf(xy.x, (float)lv.W, -0.5f),
                                          fmaf(xy.y, (float)lv.H, -0.5f), lv);
            if constexpr (kRef != 0)
                if (mrow != nullptr) mask_corners(fp, mrow);
            key = make_int4(fp.key[0], fp.key[1], fp.key[2], fp.key[3]);
            w = make_float4(fp.key[0] >= 0 ? a * fp.w[0] : 0.f, fp.key[1] >= 0 ? a * fp.w[1] : 0.f,
                            fp.key[2] >= 0 ? a * fp.w[2] : 0.f, fp.key[3] >= 0 ? a * fp.w[3] : 0.f);
        }
        wk[sg * kStride + sj] = key;
        ww[sg * kStride + sj] = w;
    }
}

// tiles_per_cta: CTA c runs tiles [c * tiles_per_cta, (c + 1) * tiles_per_cta).
#ifndef MSDA_FWD_MIN_BLOCKS8
#define MSDA_FWD_MIN_BLOCKS8 3
#endif

// Resident warps per SM the register budget is sized for, by the number of
// channels a lane holds (each corner's loaded vector is that many registers);
// __launch_bounds__ takes it as CTAs of MSDA_FWD_WARPS warps.
constexpr int forward_warps_per_sm(int channels_per_lane) {
    return 8 * (channels_per_lane <= 4   ? MSDA_FWD_MIN_BLOCKS
                : channels_per_lane <= 8 ? MSDA_FWD_MIN_BLOCKS8
                : channels_per_lane <= 16 ? 2
                                          : 1);
}
// The zero-row 16-bit instantiations with eight channels a lane hold fewer live
// registers and take 7 CTAs (72 registers, no spills): bf16 encoder forward
// 263 -> 248 us, fp16 274 -> 258 us.
#ifndef MSDA_FWD_CTAS16
#define MSDA_FWD_CTAS16 7
#endif
constexpr int forward_min_blocks(int channels_per_lane, bool zero_row) {
    if (zero_row && channels_per_lane > 4 && channels_per_lane <= 8) return MSDA_FWD_CTAS16;
    return forward_warps_per_sm(channels_per_lane) >= MSDA_FWD_WARPS
               ? forward_warps_per_sm(channels_per_lane) / MSDA_FWD_WARPS
               : 1;
}

// kVB: bytes per row vector and lane (16, or 32 with 256-bit loads).
// kRef != 0: fused entry point -- loc holds sampling offsets, attn the attention
// logits, ref the reference points [bs, Q, L, kRef]; requires L*P <= kSPG.
template <typename T, int kLanes, int kVPL, int kVB, int kRef>
__global__ void __launch_bounds__(
    MSDA_FWD_WARPS * 32,
    forward_min_blocks(kVPL * kVB / (int)sizeof(T), forward_zero_row<T, kLanes, kVPL, kVB, kRef>()))
    forward_kernel(const T* __restrict__ value, const void* __restrict__ spatial_shapes,
                   const void* __restrict__ level_start_index, int idx32, const T* __restrict__ loc,
                   const T* __restrict__ attn, T* __restrict__ out, int num_keys, int num_heads,
                   int head_dim, int num_levels, int num_points, int num_queries,
                   int num_qtiles, int num_tiles, int tiles_per_cta, const T* __restrict__ ref,
                   const unsigned char* __restrict__ mask) {
    constexpr bool kPrep = kRef != 0;
    using Geom = TileGeom<kLanes>;
    using VIO = VecIO<T, kVB>;
    constexpr int kGroups = Geom::kGroups, kSPG = Geom::kSPG, kStride = Geom::kStride;
    constexpr int V = VIO::kVec;
    constexpr int kUnroll = (sizeof(T) == 4 && kVB == 16 && kLanes == 8 && kVPL == 1)
                                ? MSDA_FWD_UNROLL_F32_128
                                : MSDA_FWD_UNROLL;
    constexpr bool kPackedFma = MSDA_FWD_PACKED != 0 && sizeof(T) == 2;
    constexpr bool kZeroRow = forward_zero_row<T, kLanes, kVPL, kVB, kRef>();
    __shared__ LevelInfo s_levels[kMaxLevels];
    __shared__ unsigned char s_level_of[kMaxLevelPoints];
    constexpr int kWarps = MSDA_FWD_WARPS;
    __shared__ int4 s_key[kWarps][Geom::kRecords];
    __shared__ float4 s_w[kWarps][Geom::kRecords];

    load_level_table(s_levels, s_level_of, spatial_shapes, level_start_index, idx32,
                     num_levels, num_points, num_keys);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / kLanes, li = lane % kLanes;
    const float points_f = (float)num_points;
    const int LP = num_levels * num_points;
    const int nvec = head_dim / V;
    const unsigned row_bytes = (unsigned)(num_heads * head_dim) * (unsigned)sizeof(T);
    int4* wk = s_key[warp];
    float4* ww = s_w[warp];

    StepIter it;
    it.t = blockIdx.x * tiles_per_cta + warp;
    it.end = min(num_tiles, (blockIdx.x + 1) * tiles_per_cta);
    it.r0 = 0;
    it.LP = LP;
    it.spg = kSPG;
    it.stride = kWarps;
    if (!it.valid()) return;

    SampleFetch f;
    PrepFetch pf;
    TileCoord tc = tile_coord(it.t, num_heads, num_qtiles, kGroups);
    fetch_samples<T, kSPG>(f, loc, attn, tc, 0, lane, LP, num_queries, num_heads);
    PrepLane pl;
    if constexpr (kPrep) pl = prep_lane<kSPG>(lane, num_levels, LP, kRef, s_level_of);
    float acc[kVPL][V];
#pragma unroll
    for (int k = 0; k < kVPL; ++k)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[k][e] = 0.f;

    while (true) {
        // ---- 1. footprints of this round (inputs fetched, references prefetched, a round ahead)
        if constexpr (kPrep) fetch_refs<T, kRef>(pf, f, ref, tc, num_queries, num_levels, pl);
        if constexpr (kPrep) softmax_rows<kSPG>(f);
        forward_records<kSPG, kStride, kRef>(
            wk, ww, f, pf, points_f, mask ? mask + (int64_t)tc.b * num_keys : nullptr,
            s_levels, s_level_of, it.r0, lane);
        __syncwarp();
        const TileCoord cur = tc;
        const int r0 = it.r0;
        const bool last = it.last_round();
        it.next();
        const bool more = it.valid();
        if (more) {
            tc = tile_coord(it.t, num_heads, num_qtiles, kGroups);
            fetch_samples<T, kSPG>(f, loc, attn, tc, it.r0, lane, LP, num_queries, num_heads);
            if constexpr (kPrep) prefetch_refs<T, kRef>(f, ref, tc, num_queries, num_levels, pl);
        }

        // ---- 2. gather: group g walks its query's samples
        const char* vbase = reinterpret_cast<const char*>(
            value + ((int64_t)cur.b * num_keys * num_heads + cur.m) * head_dim);
        const int nj = min(kSPG, LP - r0);
        const int4* gk = wk + g * kStride;
        const float4* gw = ww + g * kStride;
        MSDA_UNROLL(kUnroll)
        for (int jj = 0; jj < nj; ++jj) {
            const int4 k4 = gk[jj];
            const float4 w4 = gw[jj];
            const int keys[4] = {k4.x, k4.y, k4.z, k4.w};
            const float wc[4] = {w4.x, w4.y, w4.z, w4.w};
            float v[4][kVPL][V];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const char* p = row_ptr(vbase, keys[c], row_bytes);
                if constexpr (kZeroRow) {
                    // dead corners and idle lanes read the zero row
                    const bool live =
                        keys[c] >= 0 && li < nvec && row_in_range(keys[c], num_keys);
                    VIO::load((live ? p : reinterpret_cast<const char*>(g_zero_row)) + li * kVB,
                              v[c][0]);
                } else {
#pragma unroll
                    for (int k = 0; k < kVPL; ++k) {
                        const int vi = li + k * kLanes;
#pragma unroll
                        for (int e = 0; e < V; ++e) v[c][k][e] = 0.f;
                        if (keys[c] >= 0 && vi < nvec && row_in_range(keys[c], num_keys))
                            VIO::load(p + vi * kVB, v[c][k]);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if constexpr (kPackedFma) {
                    // two channels per instruction (sm_100 packed fp32 FMA; each half is
                    // the same fmaf as the scalar form)
                    const float2 w2 = make_float2(wc[c], wc[c]);
#pragma unroll
                    for (int k = 0; k < kVPL; ++k)
#pragma unroll
                        for (int e = 0; e < V; e += 2) {
                            const float2 a =
                                __ffma2_rn(w2, make_float2(v[c][k][e], v[c][k][e + 1]),
                                           make_float2(acc[k][e], acc[k][e + 1]));
                            acc[k][e] = a.x;
                            acc[k][e + 1] = a.y;
                        }
                } else {
#pragma unroll
                    for (int k = 0; k < kVPL; ++k)
#pragma unroll
                        for (int e = 0; e < V; ++e)
                            acc[k][e] = fmaf(wc[c], v[c][k][e], acc[k][e]);
                }
            }
        }
        __syncwarp();

        if (last) {
            const int q = cur.q0 + g;
            if (q < num_queries) {
                T* o = out + (((int64_t)cur.b * num_queries + q) * num_heads + cur.m) * head_dim;
#pragma unroll
                for (int k = 0; k < kVPL; ++k) {
                    const int vi = li + k * kLanes;
                    if (vi < nvec) VIO::store(o + vi * V, acc[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < kVPL; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[k][e] = 0.f;
        }
        if (!more) break;
    }
}

}  // namespace msda
