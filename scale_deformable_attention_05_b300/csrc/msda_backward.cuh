// Backward gather/scatter kernel of multi-scale deformable attention.
//
// For every sample (b, q, m, l, p) with attention weight a, fractions
// (fx, fy), corner weights w_c, corner rows v_c (zero off the map) and
// grad_output row g (DQ-DETR ops page, MSDeformAttnFunction.backward returns
// these three gradients; the formulas are the derivative of the walk-through's
// ms_deform_attn_core_pytorch sum), with the corner dot products
// s_c = sum_d g_d v_c,d:
//   grad_attn[pt]       = sum_c w_c s_c
//   grad_loc[pt].x      = W * a * ((1-fy)(s_01 - s_00) + fy (s_11 - s_10))
//   grad_loc[pt].y      = H * a * ((1-fx)(s_10 - s_00) + fx (s_11 - s_01))
//   grad_value[b,key_c,m,d] += a * w_c * g_d          (fp32 vector red to global)
//
// Decomposition as in the forward (one query per lane group, kGroups
// consecutive queries of one (b, m) per warp tile, footprints in shared
// memory).  Each group walks its samples in batches of eight: per sample it
// loads the live corner rows, adds each lane's share of the four dot
// products into registers and scatters a*w_c*g into grad_value with
// red.global.add.v4.f32.  After a batch the 32 partial dot products of the
// group are transpose-reduced across its lanes (each exchange halves the
// values a lane holds), which leaves the four dot products of one sample in
// one lane (kLanes = 8); that lane forms the sample's location and weight
// gradients, so the group writes eight consecutive samples' gradients at once.
#pragma once

#include <type_traits>

#include "msda_device.cuh"

namespace msda {

// Corner dot products of 16-bit rows with sm_100's mixed-precision FMA (16-bit
// multiplicands, fp32 addend and result): the value row stays packed instead of
// being widened channel by channel.  A product of two bf16 (or fp16) values is
// exact in fp32 and each fma rounds once, so the sums equal fmaf on the widened
// values bit for bit, in the same order (low half, then high half).
// Packed fp32 multiply (two channels per instruction) for the red payload of
// 16-bit rows (with the mixed-precision dot products below: bf16 encoder
// backward 906 -> 872 us); fp32 rows measured slower with it (430 -> 434 us).
#ifndef MSDA_BWD_PACKED
#define MSDA_BWD_PACKED 1
#endif
// 16-bit rows send each corner's reds as predicated instructions instead of
// branching around them (bf16 encoder backward 768 -> 747 us, fp16 768 -> 750
// us); fp32 rows keep the branch (393 -> 397 us predicated).
#ifndef MSDA_BWD_PRED_RED
#define MSDA_BWD_PRED_RED 1
#endif
#ifndef MSDA_BWD_MIXED_DOT
#define MSDA_BWD_MIXED_DOT 1
#endif
template <typename T>
__device__ __forceinline__ float dot2_16(uint32_t a, uint32_t b, float d);
template <>
__device__ __forceinline__ float dot2_16<__nv_bfloat16>(uint32_t a, uint32_t b, float d) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(d)
        : "r"(a), "r"(b));
    return d;
}
template <>
__device__ __forceinline__ float dot2_16<__half>(uint32_t a, uint32_t b, float d) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(d)
        : "r"(a), "r"(b));
    return d;
}
// Two fp32 values that are exact in T (a widened grad_output row), packed back.
template <typename T>
__device__ __forceinline__ uint32_t repack16x2(float lo, float hi) {
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        return pack_bf16x2(lo, hi);
    }
}

// Bilinear weight of corner c and its derivatives along x_im and y_im.
__device__ __forceinline__ void corner_terms(int c, float fx, float fy, float& w, float& dwx,
                                             float& dwy) {
    const bool cx = (c & 1) != 0, cy = (c & 2) != 0;
    const float wx = cx ? fx : 1.f - fx, wy = cy ? fy : 1.f - fy;
    w = wx * wy;
    dwx = cx ? wy : -wy;
    dwy = cy ? wx : -wx;
}

// CTA shape of backward_kernel.  Lane groups of at most 8 lanes with one vector
// per lane (head_dim <= 32) run resident CTAs of 4 warps, 6 per SM for fp32
// rows (80 registers per thread) and 8 for 16-bit rows (64 registers), and load
// each round's inputs at the start of that round rather than one round ahead,
// which frees the registers the prefetch held.  (CTAs of 4 warps instead of 8
// at the same warps per SM: fp32 encoder 416 -> 413 us, decoder 34.8 -> 32.7
// us, bf16 unchanged.)  Measured (kernel-only events,
// against 3 CTAs with the prefetch on the plain path and one CTA of 16 warps
// with it on the fused one): plain encoder fp32 440 -> 417 us, bf16 877 -> 825
// us, fp16 879 -> 827 us, decoder 38.9 -> 34.8 us; fused encoder 2-d 563 -> 528
// us, 4-d 576 -> 534 us, bf16 1300 -> 1090 us (the fused decoder 36 -> 39 us);
// one CTA of 16 warps with 128 registers had been slower still on the plain
// path (fp32 452 us, bf16 1073 us).  Wider rows keep one CTA of 16 warps and
// the prefetch.
#ifndef MSDA_BWD_NARROW_WARPS
#define MSDA_BWD_NARROW_WARPS 4
#endif
#ifndef MSDA_BWD_NARROW_BLOCKS
#define MSDA_BWD_NARROW_BLOCKS 6
#endif
#ifndef MSDA_BWD_NARROW_BLOCKS16
#define MSDA_BWD_NARROW_BLOCKS16 8
#endif
// The fused entry points' 16-bit backward holds the softmax-Jacobian and offset
// state as well: at 8 CTAs (64 registers) it spilled 176 bytes per thread; 7 CTAs
// (72 registers) measured best (bf16 encoder 953 -> 898 us; 6 CTAs 939 us).
#ifndef MSDA_BWD_FUSED16_BLOCKS
#define MSDA_BWD_FUSED16_BLOCKS 7
#endif
#ifndef MSDA_BWD_NARROW_PREFETCH
#define MSDA_BWD_NARROW_PREFETCH 0
#endif
// fp32 rows also have a dense shape, 7 CTAs per SM at 72 registers, which the
// launcher takes when the grid fills 7 CTAs on every SM: encoder backward 392 ->
// 386 us; on grids of a few CTAs per SM (the decoder's 300) the 80-register
// build is the faster one (32.7 against 36.9 us).
#ifndef MSDA_BWD_NARROW_BLOCKS_DENSE
#define MSDA_BWD_NARROW_BLOCKS_DENSE 7
#endif
template <typename T, int kLanes, int kVPL, int kRef, bool kDense = false>
struct BwdShape {
    static constexpr bool kNarrow = kLanes <= 8 && kVPL == 1;
    static constexpr int kWarps = kNarrow ? MSDA_BWD_NARROW_WARPS : MSDA_BWD_WARPS;
    static constexpr int kMinBlocks = !kNarrow           ? 1
                                      : sizeof(T) == 4   ? (kDense ? MSDA_BWD_NARROW_BLOCKS_DENSE
                                                                   : MSDA_BWD_NARROW_BLOCKS)
                                      : kRef != 0        ? MSDA_BWD_FUSED16_BLOCKS
                                                         : MSDA_BWD_NARROW_BLOCKS16;
};
// backward_merge_kernel: one CTA of MSDA_MERGE_WARPS warps per SM, whose
// threads may then hold up to 255 registers.  Its 1 KB rows measured slower
// with more warps of fewer registers (kernel-only, envelope backward): one CTA
// of 16 warps at 128 registers 2481 us, one of 8 warps 2417 us, two of 8 warps
// at 128 registers (62 bytes of spills) 2493 us, three 2734 us, 24 warps of 80
// registers 10% slower.
#ifndef MSDA_MERGE_WARPS
#define MSDA_MERGE_WARPS 8
#endif

// Locations, weights and grad_output rows of the next round loaded during this
// round's gathers (1), or at the start of their round (0, fewer live registers);
// the narrow shapes above use MSDA_BWD_NARROW_PREFETCH instead.
#ifndef MSDA_BWD_PREFETCH
#define MSDA_BWD_PREFETCH 1
#endif

// Samples per transpose-reduce of the corner dot products (raised to kLanes / 4
// where a lane group is wider).  4 measured ~3% faster than 8 on the fp32 and
// bf16 encoder shapes (fewer live registers in the 128-register budget).
#ifndef MSDA_BWD_BATCH
#define MSDA_BWD_BATCH 4
#endif

// Stores the footprint records of the round fetched in f: corner keys, the
// weight each corner's grad_value red carries, and (a, fx, fy, level).
//
// Red weights are merged within aligned segments of kDedup lanes that hold
// the points of one (query, level): the samples of a query share its
// grad_output row, so when several of them touch the same pixel the lowest
// lane sends one red with the summed weight a*w_c and the others send none.
// Corners can only coincide within a pixel parity class, so each class is
// compared across the segment with xor shuffles.
// kRef: 0 on the plain path; 2 or 4, the width of the reference points, on the
// fused entry points, where the round holds offsets and softmax weights;
// the location is formed from pf's reference point first, aux.x keeps the
// softmax weight of every sample (finite by construction), and the sample's
// offset and box size (4-d references only) go to woffwh for the offset and
// reference-point gradients.
template <int kSPG, int kStride, int kRef>
__device__ __forceinline__ void backward_records(int4* wk, float4* waw, float4* wax,
                                                 float4* woffwh, const SampleFetch& f,
                                                 const PrepFetch& pf, float points_f,
                                                 const unsigned char* __restrict__ mrow,
                                                 const LevelInfo* s_levels,
                                                 const unsigned char* s_level_of, int r0,
                                                 int lane, int dedup) {
#pragma unroll
    for (int h = 0; h < kSamplesPerWarp / 32; ++h) {
        const int s = lane + 32 * h;
        const int sg = s / kSPG, sj = s % kSPG;
        int4 key = make_int4(-1, -1, -1, -1);
        float4 aux = make_float4(0.f, 0.f, 0.f, 0.f);
        ClassCorners cc;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            cc.key[t] = -1;
            cc.w[t] = 0.f;
        }
        int px = 0, py = 0;
        if (f.ok[h]) {
            const int l = s_level_of[r0 + sj];
            const LevelInfo lv = s_levels[l];
            const float a = f.a[h];
            float2 xy = f.xy[h];
            if constexpr (kRef != 0) {
                if constexpr (kRef == 4)
                    woffwh[sg * kStride + sj] = make_float4(xy.x, xy.y, pf.rwh[h].x, pf.rwh[h].y);
                xy = prep_location<kRef>(pf.rxy[h], pf.rwh[h], xy, (float)lv.W, (float)lv.H,
                                         points_f);
            }
            Footprint fp = make_footprint(fmaf(xy.x, (float)lv.W, -0.5f),
                                          fmaf(xy.y, (float)lv.H, -0.5f), lv);
            if constexpr (kRef != 0)
                if (mrow != nullptr) mask_corners(fp, mrow);
            key = make_int4(fp.key[0], fp.key[1], fp.key[2], fp.key[3]);
            aux = make_float4(fp.live || kRef != 0 ? a : 0.f, fp.fx, fp.fy, __int_as_float(l));
            cc = class_corners(fp, a);
            px = fp.x0 & 1;
            py = fp.y0 & 1;
        }
        float rw[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int k = cc.key[t];
            float A = cc.w[t];
            bool lead = k >= 0;
            // peers at xor distance 1..3 within the segment (dedup is warp-uniform);
            // selects instead of a branch on each match
#pragma unroll
            for (int i = 1; i < 4; ++i) {
                if (i < dedup) {
                    const int kp = __shfl_xor_sync(0xffffffffu, k, i);
                    const float wp = __shfl_xor_sync(0xffffffffu, cc.w[t], i);
                    const bool same = kp == k, lower = (lane ^ i) < lane;
                    lead = lead && !(same && lower);
                    A += (same && !lower) ? wp : 0.f;
                }
            }
            // class t sits at corner ((t>>1)^py, (t&1)^px)
            const int c = (((t >> 1) ^ py) << 1) | ((t & 1) ^ px);
            const float r = lead ? A : 0.f;
#pragma unroll
            for (int cc2 = 0; cc2 < 4; ++cc2)
                if (c == cc2) rw[cc2] = r;
        }
        wk[sg * kStride + sj] = key;
        waw[sg * kStride + sj] = make_float4(rw[0], rw[1], rw[2], rw[3]);
        wax[sg * kStride + sj] = aux;
    }
}

// grad_output row of query q (zeros past the last query or channel).
template <typename T, int kLanes, int kVPL, int kVB>
__device__ __forceinline__ void load_grad_row(float (&gr)[kVPL][VecIO<T, kVB>::kVec],
                                              const T* __restrict__ grad_out,
                                              const TileCoord& tc, int g, int li, int nvec,
                                              int num_queries, int num_heads, int head_dim) {
    const int q = tc.q0 + g;
    const int64_t row = ((int64_t)tc.b * num_queries + q) * num_heads + tc.m;
#pragma unroll
    for (int k = 0; k < kVPL; ++k) {
        const int vi = li + k * kLanes;
#pragma unroll
        for (int e = 0; e < VecIO<T, kVB>::kVec; ++e) gr[k][e] = 0.f;
        if (q < num_queries && vi < nvec)
            VecIO<T, kVB>::load_stream(grad_out + row * head_dim + vi * VecIO<T, kVB>::kVec,
                                       gr[k]);
    }
}

// tiles_per_cta: CTA c runs tiles [c * tiles_per_cta, (c + 1) * tiles_per_cta).
// kRef != 0: fused entry point -- loc holds sampling offsets, attn the attention
// logits, ref the reference points; grad_loc receives the offset gradient,
// grad_attn the logit gradient (softmax Jacobian), grad_ref (fp32, may be
// null) the reference-point gradient summed over heads and points.  Requires
// L*P <= kSPG (every row in one round).
// kVB: bytes per row vector and lane: 16, or 8 for 16-bit types, so that a lane
// holds four channels and its share of a corner's fp32 grad_value row is one
// 16-byte red.  (With eight 16-bit channels a lane sends two 16-byte reds,
// each covering half of every 32-byte sector of the row; the bf16 encoder
// backward measured 1298 us that way against 1207 us with 8-byte vectors.)
template <typename T, int kLanes, int kVPL, int kRef, int kVB, bool kDense = false>
__global__ void __launch_bounds__(BwdShape<T, kLanes, kVPL, kRef, kDense>::kWarps * 32,
                                  BwdShape<T, kLanes, kVPL, kRef, kDense>::kMinBlocks)
    backward_kernel(const T* __restrict__ value, const void* __restrict__ spatial_shapes,
                    const void* __restrict__ level_start_index, int idx32, const T* __restrict__ loc,
                    const T* __restrict__ attn, const T* __restrict__ grad_out,
                    float* __restrict__ grad_value_f32, T* __restrict__ grad_loc,
                    T* __restrict__ grad_attn, int num_keys, int num_heads, int head_dim,
                    int num_levels, int num_points, int num_queries, int num_qtiles,
                    int num_tiles, int tiles_per_cta, const T* __restrict__ ref,
                    const unsigned char* __restrict__ mask, float* __restrict__ grad_ref) {
    constexpr bool kPrep = kRef != 0;
    constexpr int kWarps = BwdShape<T, kLanes, kVPL, kRef, kDense>::kWarps;
    using Geom = TileGeom<kLanes>;
    using VIO = VecIO<T, kVB>;
    constexpr int kGroups = Geom::kGroups, kSPG = Geom::kSPG, kStride = Geom::kStride;
    constexpr int V = VIO::kVec;
    // samples per transpose-reduce (at least kLanes / 4, so a lane keeps >= 1 value)
    constexpr int kBatch = MSDA_BWD_BATCH > kLanes / 4 ? MSDA_BWD_BATCH : kLanes / 4;
    constexpr int kHeld = 4 * kBatch / kLanes;     // dot products a lane keeps after it
    constexpr int kSampPerLane = kHeld >= 4 ? kHeld / 4 : 1;
    constexpr int kLanesPerSamp = kHeld >= 4 ? 1 : 4 / kHeld;
    static_assert(kSPG % kBatch == 0, "round must hold whole batches");

    __shared__ LevelInfo s_levels[kMaxLevels];
    __shared__ unsigned char s_level_of[kMaxLevelPoints];
    __shared__ int4 s_key[kWarps][Geom::kRecords];
    __shared__ float4 s_aw[kWarps][Geom::kRecords];
    __shared__ float4 s_aux[kWarps][Geom::kRecords];
    // fused mode: per sample (offset, box size) for 4-d references, (grad_loc, grad_a)
    constexpr int kPrepRecords = kPrep ? Geom::kRecords : 1;
    constexpr int kBoxRecords = kRef == 4 ? Geom::kRecords : 1;
    __shared__ float4 s_offwh[kRef == 4 ? kWarps : 1][kBoxRecords];
    __shared__ float4 s_gla[kPrep ? kWarps : 1][kPrepRecords];

    load_level_table(s_levels, s_level_of, spatial_shapes, level_start_index, idx32,
                     num_levels, num_points, num_keys);
    __syncthreads();
    // 1 / (2P): the derivative of the 4-d location along the offset is ref_wh / (2P)
    const float inv_2p = kPrep ? __frcp_rn((float)(2 * num_points)) : 0.f;
    const float points_f = (float)num_points;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / kLanes, li = lane % kLanes;
    const int LP = num_levels * num_points;
    const int nvec = head_dim / V;
    const unsigned row_bytes = (unsigned)(num_heads * head_dim) * (unsigned)sizeof(T);
    const unsigned row_bytes32 = (unsigned)(num_heads * head_dim) * 4u;
    // lanes that hold the points of one (query, level): an aligned segment
    // of up to 4 lanes when the points per level tile the round
    const int dedup = (num_points % 4 == 0 && kSPG % 4 == 0) ? 4
                      : (num_points % 2 == 0 && kSPG % 2 == 0) ? 2 : 1;
    int4* wk = s_key[warp];
    float4* waw = s_aw[warp];
    float4* wax = s_aux[warp];
    float4* woffwh = s_offwh[kRef == 4 ? warp : 0];
    float4* wgla = s_gla[kPrep ? warp : 0];

    StepIter it;
    it.t = blockIdx.x * tiles_per_cta + warp;
    it.end = min(num_tiles, (blockIdx.x + 1) * tiles_per_cta);
    it.r0 = 0;
    it.LP = LP;
    it.spg = kSPG;
    it.stride = kWarps;
    if (!it.valid()) return;

    constexpr bool kPrefetch = BwdShape<T, kLanes, kVPL, kRef, kDense>::kNarrow
                                   ? MSDA_BWD_NARROW_PREFETCH != 0
                                   : MSDA_BWD_PREFETCH != 0 || kPrep;
    SampleFetch f;
    PrepFetch pf;
    TileCoord tc = tile_coord(it.t, num_heads, num_qtiles, kGroups);
    PrepLane pl;
    if constexpr (kPrep) pl = prep_lane<kSPG>(lane, num_levels, LP, kRef, s_level_of);
    float gr[kVPL][V], gnext[kVPL][V];
    if constexpr (kPrefetch) {
        fetch_samples<T, kSPG>(f, loc, attn, tc, 0, lane, LP, num_queries, num_heads);
        load_grad_row<T, kLanes, kVPL, kVB>(gnext, grad_out, tc, g, li, nvec, num_queries,
                                            num_heads, head_dim);
    }

    while (true) {
        if constexpr (!kPrefetch) {
            fetch_samples<T, kSPG>(f, loc, attn, tc, it.r0, lane, LP, num_queries, num_heads);
            if (it.r0 == 0)
                load_grad_row<T, kLanes, kVPL, kVB>(gr, grad_out, tc, g, li, nvec, num_queries,
                                                    num_heads, head_dim);
        }
        // ---- 1. footprints of this round (inputs fetched, references prefetched, a round ahead)
        if constexpr (kPrep) fetch_refs<T, kRef>(pf, f, ref, tc, num_queries, num_levels, pl);
        if constexpr (kPrep) softmax_rows<kSPG>(f);
        backward_records<kSPG, kStride, kRef>(
            wk, waw, wax, woffwh, f, pf, points_f,
            mask ? mask + (int64_t)tc.b * num_keys : nullptr, s_levels, s_level_of, it.r0, lane,
            dedup);
        __syncwarp();
        const TileCoord cur = tc;
        const int r0 = it.r0;
        if (kPrefetch && r0 == 0) {
#pragma unroll
            for (int k = 0; k < kVPL; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) gr[k][e] = gnext[k][e];
        }
        it.next();
        const bool more = it.valid();
        if (more) {
            tc = tile_coord(it.t, num_heads, num_qtiles, kGroups);
            if constexpr (kPrefetch) {
                fetch_samples<T, kSPG>(f, loc, attn, tc, it.r0, lane, LP, num_queries,
                                       num_heads);
                if constexpr (kPrep)
                    prefetch_refs<T, kRef>(f, ref, tc, num_queries, num_levels, pl);
                if (it.r0 == 0)
                    load_grad_row<T, kLanes, kVPL, kVB>(gnext, grad_out, tc, g, li, nvec,
                                                        num_queries, num_heads, head_dim);
            }
        }

        const int64_t head0 = ((int64_t)cur.b * num_keys * num_heads + cur.m) * head_dim;
        const char* vbase = reinterpret_cast<const char*>(value + head0);
        char* gvbase = reinterpret_cast<char*>(grad_value_f32 + head0);
        constexpr bool kMixedDot = MSDA_BWD_MIXED_DOT != 0 && sizeof(T) == 2 && kVB == 8;
        constexpr bool kPackedMul = MSDA_BWD_PACKED != 0 && sizeof(T) == 2;
        constexpr bool kPredRed = MSDA_BWD_PRED_RED != 0 && sizeof(T) == 2;
        uint2 grp[kVPL];                  // the grad_output row packed (16-bit rows)
        if constexpr (kMixedDot) {
#pragma unroll
            for (int k = 0; k < kVPL; ++k)
                grp[k] = make_uint2(repack16x2<T>(gr[k][0], gr[k][1]),
                                    repack16x2<T>(gr[k][2], gr[k][3]));
        }
        const int q = cur.q0 + g;
        const int64_t row = ((int64_t)cur.b * num_queries + q) * num_heads + cur.m;
        const int nj = min(kSPG, LP - r0);
        const int4* gk = wk + g * kStride;
        const float4* gaw = waw + g * kStride;
        const float4* gax = wax + g * kStride;
        for (int jb = 0; jb < nj; jb += kBatch) {
            // ---- 2. gather + scatter a batch of eight samples (records past
            //         the round's end hold dead samples)
            float dots[4 * kBatch];
#pragma unroll
            for (int s8 = 0; s8 < kBatch; ++s8) {
                const int4 k4 = gk[jb + s8];
                const float4 a4 = gaw[jb + s8];
                const int keys[4] = {k4.x, k4.y, k4.z, k4.w};
                const float awc[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const char* p = row_ptr(vbase, keys[c], row_bytes);
                    float d = 0.f;
                    if constexpr (kMixedDot) {
#pragma unroll
                        for (int k = 0; k < kVPL; ++k) {
                            const int vi = li + k * kLanes;
                            uint2 raw = make_uint2(0u, 0u);
                            if (keys[c] >= 0 && vi < nvec && row_in_range(keys[c], num_keys))
                                raw = __ldg(reinterpret_cast<const uint2*>(p + vi * kVB));
                            d = dot2_16<T>(grp[k].x, raw.x, d);
                            d = dot2_16<T>(grp[k].y, raw.y, d);
                        }
                    } else {
                        float v[kVPL][V];
#pragma unroll
                        for (int k = 0; k < kVPL; ++k) {
                            const int vi = li + k * kLanes;
#pragma unroll
                            for (int e = 0; e < V; ++e) v[k][e] = 0.f;
                            if (keys[c] >= 0 && vi < nvec && row_in_range(keys[c], num_keys))
                                VIO::load(p + vi * kVB, v[k]);
                        }
#pragma unroll
                        for (int k = 0; k < kVPL; ++k)
#pragma unroll
                            for (int e = 0; e < V; ++e) d = fmaf(gr[k][e], v[k][e], d);
                    }
                    dots[s8 * 4 + c] = d;
                    // merged duplicates and corners off the map carry red weight 0
                    // (the records zero both), so the weight alone decides the red
                    // (one test fewer per corner: fp32 encoder 397 -> 393 us)
                    if constexpr (kPredRed) {
                        // the address of a corner that sends nothing is formed, never used
                        const bool send = awc[c] != 0.f && row_in_range(keys[c], num_keys);
                        float* gp = reinterpret_cast<float*>(
                            gvbase + (size_t)(unsigned)keys[c] * row_bytes32);
#pragma unroll
                        for (int k = 0; k < kVPL; ++k) {
                            const int vi = li + k * kLanes;
                            const bool ok = send && vi < nvec;
#pragma unroll
                            for (int e = 0; e < V; e += 4) {
                                if constexpr (kPackedMul) {
                                    const float2 a2 = make_float2(awc[c], awc[c]);
                                    const float2 p01 =
                                        __fmul2_rn(a2, make_float2(gr[k][e], gr[k][e + 1]));
                                    const float2 p23 =
                                        __fmul2_rn(a2, make_float2(gr[k][e + 2], gr[k][e + 3]));
                                    red_add_v4_if(ok, gp + vi * V + e, p01.x, p01.y, p23.x,
                                                  p23.y);
                                } else {
                                    red_add_v4_if(ok, gp + vi * V + e, awc[c] * gr[k][e],
                                                  awc[c] * gr[k][e + 1], awc[c] * gr[k][e + 2],
                                                  awc[c] * gr[k][e + 3]);
                                }
                            }
                        }
                    } else if (awc[c] != 0.f && row_in_range(keys[c], num_keys)) {
                        float* gp = reinterpret_cast<float*>(
                            gvbase + (size_t)(unsigned)keys[c] * row_bytes32);
#pragma unroll
                        for (int k = 0; k < kVPL; ++k) {
                            const int vi = li + k * kLanes;
                            if (vi < nvec) {
#pragma unroll
                                for (int e = 0; e < V; e += 4) {
                                    if constexpr (kPackedMul) {
                                        // the payload two channels per instruction (sm_100
                                        // packed fp32 multiply; each half is the scalar product)
                                        const float2 a2 = make_float2(awc[c], awc[c]);
                                        const float2 p01 = __fmul2_rn(
                                            a2, make_float2(gr[k][e], gr[k][e + 1]));
                                        const float2 p23 = __fmul2_rn(
                                            a2, make_float2(gr[k][e + 2], gr[k][e + 3]));
                                        red_add_v4(gp + vi * V + e, p01.x, p01.y, p23.x, p23.y);
                                    } else {
                                        red_add_v4(gp + vi * V + e, awc[c] * gr[k][e],
                                                   awc[c] * gr[k][e + 1], awc[c] * gr[k][e + 2],
                                                   awc[c] * gr[k][e + 3]);
                                    }
                                }
                            }
                        }
                    }
                }
            }

            // ---- 3. transpose-reduce the batch's dot products across the group
#pragma unroll
            for (int rr = 0; (kLanes >> (rr + 1)) >= 1; ++rr) {
                const int o = kLanes >> (rr + 1);
                const int n = (4 * kBatch / 2) >> rr;
                const bool upper = (li & o) != 0;
#pragma unroll
                for (int k = 0; k < n; ++k) {
                    const float send = upper ? dots[k] : dots[k + n];
                    const float keep = upper ? dots[k + n] : dots[k];
                    dots[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }

            // ---- 4. per-sample location and weight gradients
#pragma unroll
            for (int u = 0; u < kSampPerLane; ++u) {
                const int s8 = kHeld >= 4 ? li * (kHeld / 4) + u : (li * kHeld) / 4;
                const float4 ax = gax[jb + s8];
                const float a = ax.x, fx = ax.y, fy = ax.z;
                float ga = 0.f, gx = 0.f, gy = 0.f;
#pragma unroll
                for (int k = 0; k < (kHeld >= 4 ? 4 : kHeld); ++k) {
                    const int c = kHeld >= 4 ? k : (li * kHeld + k) & 3;
                    float w, dwx, dwy;
                    corner_terms(c, fx, fy, w, dwx, dwy);
                    const float d = dots[(kHeld >= 4 ? u * 4 : 0) + k];
                    ga = fmaf(w, d, ga);
                    gx = fmaf(dwx, d, gx);
                    gy = fmaf(dwy, d, gy);
                }
#pragma unroll
                for (int o = 1; o < kLanesPerSamp; o <<= 1) {
                    ga += __shfl_xor_sync(0xffffffffu, ga, o);
                    gx += __shfl_xor_sync(0xffffffffu, gx, o);
                    gy += __shfl_xor_sync(0xffffffffu, gy, o);
                }
                if (li % kLanesPerSamp == 0 && jb + s8 < nj && q < num_queries) {
                    const LevelInfo lv = s_levels[__float_as_int(ax.w)];
                    const int64_t pt = row * LP + r0 + jb + s8;
                    const float glx = (float)lv.W * (a * gx), gly = (float)lv.H * (a * gy);
                    if constexpr (kPrep) {
                        // offset gradient now; weight and location gradients kept for
                        // the softmax Jacobian and the reference-point sums below
                        const int rec = g * kStride + jb + s8;
                        wgla[rec] = make_float4(glx, gly, ga, 0.f);
                        float ox = a * gx, oy = a * gy;             // grad_loc / (W, H)
                        if constexpr (kRef == 4) {
                            const float4 ow = woffwh[rec];
                            ox = glx * ow.z * inv_2p;               // grad_loc * box / (2P)
                            oy = gly * ow.w * inv_2p;
                        }
                        IO<T>::store_xy(grad_loc + 2 * pt, ox, oy);
                    } else {
                        IO<T>::store_xy(grad_loc + 2 * pt, glx, gly);
                        IO<T>::store_one(grad_attn + pt, ga);
                    }
                }
            }
        }
        if constexpr (kPrep) {
            // ---- 5. the row's logit gradients a_j (g_j - sum_i a_i g_i) and its
            //         reference-point gradient sums (the row is this round's whole tile)
            __syncwarp();
            const bool qok = q < num_queries;
            float S = 0.f;
            for (int jj = li; qok && jj < LP; jj += kLanes) {
                const int rec = g * kStride + jj;
                S = fmaf(wax[rec].x, wgla[rec].z, S);
            }
#pragma unroll
            for (int o = 1; o < kLanes; o <<= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
            for (int jj = li; qok && jj < LP; jj += kLanes) {
                const int rec = g * kStride + jj;
                IO<T>::store_one(grad_attn + row * LP + jj, wax[rec].x * (wgla[rec].z - S));
            }
            if (grad_ref != nullptr && qok) {
                for (int pi = li; pi < num_levels * kRef; pi += kLanes) {
                    const int l = pi / kRef, c = pi - l * kRef;
                    float sum = 0.f;
                    for (int p = 0; p < num_points; ++p) {
                        const int rec = g * kStride + l * num_points + p;
                        const float4 gla = wgla[rec];
                        const float glc = (c & 1) ? gla.y : gla.x;
                        if (c < 2) {
                            sum += glc;
                        } else {
                            const float4 ow = woffwh[rec];
                            sum += glc * ((c & 1) ? ow.y : ow.x) * inv_2p;
                        }
                    }
                    atomicAdd(grad_ref +
                                  (((int64_t)cur.b * num_queries + q) * num_levels + l) * kRef +
                                  c,
                              sum);
                }
            }
        }
        __syncwarp();
        if (!more) break;
    }
}

// ------------------------------------------------------------------------
// Backward with merged grad_value scatter (the fast path).
//
// The scatter of grad_value is bound by the bytes the SMs send to L2: every
// red.global.add of a corner row carries head_dim fp32 values.  Neighbouring
// queries of one head sample the same pixels, so this kernel merges them
// before sending: a warp tile is G = 32 / kLanes (<= 4) consecutive queries of
// one (b, m), and its samples are taken in rounds of 32 ordered (level, query,
// point), one sample per lane.  In a round, for each pixel parity class t
// (two corners can be the same pixel only if they have the same class), the
// lanes holding the same corner key find each other with __match_any_sync;
// the lowest lane collects the per-query weight sums A_q = sum a*w_c over its
// peers, and the round's distinct (key, A_0..A_{G-1}) entries go to a list in
// shared memory.  The groups then send one red per distinct entry with the
// payload sum_q A_q * g_q (every lane holds the grad_output rows of all G
// queries).  The location and weight gradients come from the corner dot
// products as in backward_kernel, each group handling its own query's samples.
template <typename T, int kLanes, int kVPL>
__global__ void __launch_bounds__(MSDA_MERGE_WARPS * 32, 1)
    backward_merge_kernel(const T* __restrict__ value, const void* __restrict__ spatial_shapes,
                          const void* __restrict__ level_start_index, int idx32,
                          const T* __restrict__ loc, const T* __restrict__ attn,
                          const T* __restrict__ grad_out, float* __restrict__ grad_value_f32,
                          T* __restrict__ grad_loc, T* __restrict__ grad_attn, int num_keys,
                          int num_heads, int head_dim, int num_levels, int num_points,
                          int log2_points, int num_queries, int num_qtiles, int num_tiles,
                          int tiles_per_cta) {
    constexpr int G = 32 / kLanes;                 // queries per tile (one per lane group)
    static_assert(G <= 4, "merged weights hold at most four queries");
    constexpr int V = IO<T>::kVec;
    constexpr int kBatch = 8;                      // samples per transpose-reduce
    constexpr int kHeld = 32 / kLanes;             // dot products a lane keeps after it
    constexpr int kSampPerLane = kHeld >= 4 ? kHeld / 4 : 1;
    constexpr int kLanesPerSamp = kHeld >= 4 ? 1 : 4 / kHeld;
    constexpr int kPerGroup = 32 / G;              // a group's samples in one round
    constexpr int kMaxUnique = 4 * 32;

    __shared__ LevelInfo s_levels[kMaxLevels];
    __shared__ unsigned char s_level_of[kMaxLevelPoints];
    __shared__ int4 s_key[MSDA_MERGE_WARPS][32];       // corner keys (corner order) per round sample
    __shared__ float4 s_aux[MSDA_MERGE_WARPS][32];     // (a, fx, fy, level) per round sample
    __shared__ int s_ukey[MSDA_MERGE_WARPS][kMaxUnique];
    __shared__ float4 s_uA[MSDA_MERGE_WARPS][kMaxUnique];

    load_level_table(s_levels, s_level_of, spatial_shapes, level_start_index, idx32,
                     num_levels, num_points, num_keys);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / kLanes, li = lane % kLanes;
    const int P = num_points, LP = num_levels * num_points;
    const int log2_gp = log2_points + (G == 4 ? 2 : G == 2 ? 1 : 0);
    const int S = G * LP;                          // samples per tile
    const int nvec = head_dim / V;
    const unsigned row_bytes = (unsigned)(num_heads * head_dim) * (unsigned)sizeof(T);
    const unsigned row_bytes32 = (unsigned)(num_heads * head_dim) * 4u;

    StepIter it;
    it.t = blockIdx.x * tiles_per_cta + warp;
    it.end = min(num_tiles, (blockIdx.x + 1) * tiles_per_cta);
    it.r0 = 0;
    it.LP = S;
    it.spg = 32;
    it.stride = MSDA_MERGE_WARPS;
    if (!it.valid()) return;

    // round sample s = r0 + lane  ->  (level, query, point)
    auto locate = [&](int r0, int& qo, int& j) {
        const int s = r0 + lane;
        const int l = s >> log2_gp, rem = s & ((1 << log2_gp) - 1);
        qo = rem >> log2_points;
        j = l * P + (rem & (P - 1));
        return s < S;
    };
    auto fetch = [&](const TileCoord& tc, int r0, float2& xy, float& a, bool& ok) {
        int qo, j;
        ok = locate(r0, qo, j) && tc.q0 + qo < num_queries;
        xy = make_float2(0.f, 0.f);
        a = 0.f;
        if (ok) {
            const int64_t pt =
                (((int64_t)tc.b * num_queries + tc.q0 + qo) * num_heads + tc.m) * LP + j;
            xy = IO<T>::load_xy(loc + 2 * pt);
            a = IO<T>::load_one(attn + pt);
        }
    };

    TileCoord tc = tile_coord(it.t, num_heads, num_qtiles, G);
    float2 fxy;
    float fa;
    bool fok;
    fetch(tc, 0, fxy, fa, fok);
    float gq[G][kVPL][V];
    float gown[kVPL][V];

    while (true) {
        const TileCoord cur = tc;
        const int r0 = it.r0;
        if (r0 == 0) {
            // grad_output rows of the tile's queries, in every lane
#pragma unroll
            for (int qq = 0; qq < G; ++qq) {
                const int q = cur.q0 + qq;
                const int64_t row = ((int64_t)cur.b * num_queries + q) * num_heads + cur.m;
#pragma unroll
                for (int k = 0; k < kVPL; ++k) {
                    const int vi = li + k * kLanes;
#pragma unroll
                    for (int e = 0; e < V; ++e) gq[qq][k][e] = 0.f;
                    if (q < num_queries && vi < nvec)
                        IO<T>::load_vec_stream(grad_out + row * head_dim + vi * V, gq[qq][k]);
                }
            }
#pragma unroll
            for (int k = 0; k < kVPL; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    float x = gq[0][k][e];
#pragma unroll
                    for (int qq = 1; qq < G; ++qq) x = g == qq ? gq[qq][k][e] : x;
                    gown[k][e] = x;
                }
        }

        // ---- 1. my sample's footprint
        int myq, myj;
        locate(r0, myq, myj);
        ClassCorners cc;
        {
            int4 key = make_int4(-1, -1, -1, -1);
            float4 aux = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                cc.key[t] = -1;
                cc.w[t] = 0.f;
            }
            if (fok) {
                const int l = s_level_of[myj];
                const LevelInfo lv = s_levels[l];
                const Footprint fp = make_footprint(fmaf(fxy.x, (float)lv.W, -0.5f),
                                                    fmaf(fxy.y, (float)lv.H, -0.5f), lv);
                key = make_int4(fp.key[0], fp.key[1], fp.key[2], fp.key[3]);
                aux = make_float4(fp.live ? fa : 0.f, fp.fx, fp.fy, __int_as_float(l));
                cc = class_corners(fp, fa);
            }
            s_key[warp][lane] = key;
            s_aux[warp][lane] = aux;
        }
        it.next();
        const bool more = it.valid();
        if (more) {
            tc = tile_coord(it.t, num_heads, num_qtiles, G);
            fetch(tc, it.r0, fxy, fa, fok);
        }

        // ---- 2. merge equal corner keys of the round, class by class
        int nu = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int key = cc.key[t];
            const float aw = cc.w[t];
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const bool lead = key >= 0 && (__ffs(peers) - 1) == lane;
            float A[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) A[qq] = myq == qq ? aw : 0.f;
            unsigned rem = lead ? (peers & (peers - 1u)) : 0u;
            while (__any_sync(0xffffffffu, rem != 0u)) {
                const int src = rem ? __ffs(rem) - 1 : lane;
                const float w = __shfl_sync(0xffffffffu, aw, src);
                const int qs = __shfl_sync(0xffffffffu, myq, src);
                if (rem) {
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) A[qq] += qs == qq ? w : 0.f;
                    rem &= rem - 1u;
                }
            }
            const unsigned lm = __ballot_sync(0xffffffffu, lead);
            if (lead) {
                const int pos = nu + __popc(lm & ((1u << lane) - 1u));
                s_ukey[warp][pos] = key;
                s_uA[warp][pos] = make_float4(A[0], A[1], A[2], A[3]);
            }
            nu += __popc(lm);
        }
        __syncwarp();

        // ---- 3. corner dot products and location / weight gradients of my group's samples
        const int64_t head0 = ((int64_t)cur.b * num_keys * num_heads + cur.m) * head_dim;
        const char* vbase = reinterpret_cast<const char*>(value + head0);
        char* gvbase = reinterpret_cast<char*>(grad_value_f32 + head0);
        const int q = cur.q0 + g;
        const int64_t row = ((int64_t)cur.b * num_queries + q) * num_heads + cur.m;
#pragma unroll 1
        for (int kb = 0; kb < kPerGroup; kb += kBatch) {
            float dots[4 * kBatch];
#pragma unroll
            for (int s8 = 0; s8 < kBatch; ++s8) {
                const int k = kb + s8;
                const int sl = ((k >> log2_points) << log2_gp) + (g << log2_points) + (k & (P - 1));
                const int4 k4 = s_key[warp][sl];
                const int keys[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[kVPL][V];
                    const char* p = row_ptr(vbase, keys[c], row_bytes);
#pragma unroll
                    for (int kk = 0; kk < kVPL; ++kk) {
                        const int vi = li + kk * kLanes;
#pragma unroll
                        for (int e = 0; e < V; ++e) v[kk][e] = 0.f;
                        if (keys[c] >= 0 && vi < nvec && row_in_range(keys[c], num_keys))
                            IO<T>::load_vec(p + vi * 16, v[kk]);
                    }
                    float d = 0.f;
#pragma unroll
                    for (int kk = 0; kk < kVPL; ++kk)
#pragma unroll
                        for (int e = 0; e < V; ++e) d = fmaf(gown[kk][e], v[kk][e], d);
                    dots[s8 * 4 + c] = d;
                }
            }
#pragma unroll
            for (int rr = 0; (kLanes >> (rr + 1)) >= 1; ++rr) {
                const int o = kLanes >> (rr + 1);
                const int n = (4 * kBatch / 2) >> rr;
                const bool upper = (li & o) != 0;
#pragma unroll
                for (int k = 0; k < n; ++k) {
                    const float send = upper ? dots[k] : dots[k + n];
                    const float keep = upper ? dots[k + n] : dots[k];
                    dots[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
#pragma unroll
            for (int u = 0; u < kSampPerLane; ++u) {
                const int s8 = kHeld >= 4 ? li * (kHeld / 4) + u : (li * kHeld) / 4;
                const int k = kb + s8;
                const int sl = ((k >> log2_points) << log2_gp) + (g << log2_points) + (k & (P - 1));
                const float4 ax = s_aux[warp][sl];
                const float a = ax.x, fx = ax.y, fy = ax.z;
                float ga = 0.f, gx = 0.f, gy = 0.f;
#pragma unroll
                for (int kk = 0; kk < (kHeld >= 4 ? 4 : kHeld); ++kk) {
                    const int c = kHeld >= 4 ? kk : (li * kHeld + kk) & 3;
                    float w, dwx, dwy;
                    corner_terms(c, fx, fy, w, dwx, dwy);
                    const float d = dots[(kHeld >= 4 ? u * 4 : 0) + kk];
                    ga = fmaf(w, d, ga);
                    gx = fmaf(dwx, d, gx);
                    gy = fmaf(dwy, d, gy);
                }
#pragma unroll
                for (int o = 1; o < kLanesPerSamp; o <<= 1) {
                    ga += __shfl_xor_sync(0xffffffffu, ga, o);
                    gx += __shfl_xor_sync(0xffffffffu, gx, o);
                    gy += __shfl_xor_sync(0xffffffffu, gy, o);
                }
                const int s = r0 + sl;
                const int j = (s >> log2_gp) * P + (s & (P - 1));
                if (li % kLanesPerSamp == 0 && s < S && q < num_queries) {
                    const LevelInfo lv = s_levels[__float_as_int(ax.w)];
                    const int64_t pt = row * LP + j;
                    IO<T>::store_xy(grad_loc + 2 * pt, (float)lv.W * (a * gx),
                                    (float)lv.H * (a * gy));
                    IO<T>::store_one(grad_attn + pt, ga);
                }
            }
        }

        // ---- 4. one red per distinct corner row: payload sum_q A_q * g_q
#pragma unroll 1
        for (int u = g; u < nu; u += G) {
            const int key = s_ukey[warp][u];
            if (!row_in_range(key, num_keys)) continue;
            const float4 A4 = s_uA[warp][u];
            const float A[4] = {A4.x, A4.y, A4.z, A4.w};
            float* gp = reinterpret_cast<float*>(gvbase + (size_t)(unsigned)key * row_bytes32);
#pragma unroll
            for (int k = 0; k < kVPL; ++k) {
                const int vi = li + k * kLanes;
                if (vi < nvec) {
                    float pay[V];
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        float x = A[0] * gq[0][k][e];
#pragma unroll
                        for (int qq = 1; qq < G; ++qq) x = fmaf(A[qq], gq[qq][k][e], x);
                        pay[e] = x;
                    }
#pragma unroll
                    for (int e = 0; e < V; e += 4)
                        red_add_v4(gp + vi * V + e, pay[e], pay[e + 1], pay[e + 2], pay[e + 3]);
                }
            }
        }
        __syncwarp();
        if (!more) break;
    }
}

}  // namespace msda
