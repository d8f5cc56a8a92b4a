// Device-side building blocks shared by the forward and backward kernels:
// element-type traits with 16-byte vector loads/stores, the per-CTA level
// table, the per-sample bilinear footprint, and the warp-tile geometry.
//
// Sampling semantics (Deformable DETR walk-through, "2.2.4 源码分析",
// ms_deform_attn_core_pytorch: grid_sample(bilinear, zeros,
// align_corners=False) at grid = 2*loc - 1):
//   x_im = loc_x * W - 0.5 (one fp32 FMA), y_im = loc_y * H - 0.5
//   the sample is live iff -1 < x_im < W and -1 < y_im < H
//   corners (y0,x0), (y0,x0+1), (y0+1,x0), (y0+1,x0+1) with x0 = floor(x_im),
//   weights (1-fx)(1-fy), fx(1-fy), (1-fx)fy, fx*fy; a corner off the map is 0.
//
// Work decomposition (both kernels).  A "row" is one (b, q, m) triple: its
// L*P samples are contiguous in sampling_locations / attention_weights and
// its head_dim outputs are contiguous in output.  A warp is split into
// kGroups = 32 / kLanes lane groups; each lane owns kVPL 16-byte vectors of
// the head's channels, so one corner row of value (head_dim * e bytes) is
// read by a group as coalesced 128-bit loads (one 128-byte line for fp32
// head_dim 32).  A warp tile is kGroups consecutive queries of ONE (b, m):
// group g owns query q0 + g, all groups read the same head's slice of value,
// and samples of neighbouring queries that fall on the same pixel row are
// served by one cache line in the same load instruction.
#pragma once

#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msda {

// Warps per CTA of the forward and backward kernels.  The forward runs CTAs of
// 4 warps (the same resident warps per SM as 8-warp CTAs: encoder fp32 forward
// 163.8 -> 161.8 us, bf16 286.7 -> 284.7 us, kernel-only; 16-warp CTAs were
// slower, 167.9 / 340.0 us).
#ifndef MSDA_FWD_WARPS
#define MSDA_FWD_WARPS 4
#endif
#ifndef MSDA_BWD_WARPS
#define MSDA_BWD_WARPS 16
#endif
constexpr int kMaxLevels = 16;
constexpr int kMaxLevelPoints = 256;
// Samples whose footprints one warp computes per round (two per lane).
constexpr int kSamplesPerWarp = 64;

// Set (atomicOr) by a kernel that meets a level whose pixels would fall
// outside [0, num_keys), or, in the checked build, a row index outside its
// tensor; read and cleared by msda_last_device_error().  Defined here: all
// device code is compiled as the one translation unit msda_kernels.cu (no
// relocatable device code).
__device__ unsigned int g_error_word = 0;

// 128 zero bytes: the row that dead corners and idle lanes of the narrow lane
// groups (at most 8 lanes of at most 16 bytes) read instead of a predicated load.
__device__ __align__(128) uint4 g_zero_row[8] = {};
constexpr unsigned int kErrLevelOutOfRange = 1u;
constexpr unsigned int kErrRowOutOfRange = 2u;

// Checked build (-DMSDA_BOUNDS_CHECK, the library's stand-in for a memory
// sanitizer): every data-dependent value / grad_value row access first tests
// its row index against [0, num_keys) and, outside it, records
// kErrRowOutOfRange and skips the access.  The product build compiles the
// test away.
__device__ __forceinline__ bool row_in_range(int key, int num_keys) {
#ifdef MSDA_BOUNDS_CHECK
    if ((unsigned)key < (unsigned)num_keys) return true;
    atomicOr(&g_error_word, kErrRowOutOfRange);
    return false;
#else
    (void)key;
    (void)num_keys;
    return true;
#endif
}

// ---------------------------------------------------------------- I/O traits
template <typename T>
struct IO;

template <>
struct IO<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    // Value rows: read-only, reused across samples -> keep in L1.
    __device__ __forceinline__ static void load_vec(const void* p, float (&v)[kVec]) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
    // Streamed once (grad_output): evict-first.
    __device__ __forceinline__ static void load_vec_stream(const float* p, float (&v)[kVec]) {
        const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
    __device__ __forceinline__ static float2 load_xy(const float* p) {
        return __ldcs(reinterpret_cast<const float2*>(p));
    }
    __device__ __forceinline__ static float load_one(const float* p) { return __ldcs(p); }
    __device__ __forceinline__ static float4 load_xywh(const float* p) {
        return __ldg(reinterpret_cast<const float4*>(p));
    }
    __device__ __forceinline__ static void store_vec(float* p, const float (&v)[kVec]) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    }
    __device__ __forceinline__ static void store_one(float* p, float v) { __stcs(p, v); }
    __device__ __forceinline__ static void store_xy(float* p, float x, float y) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(x, y));
    }
};

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <>
struct IO<__nv_bfloat16> {
    using T = __nv_bfloat16;
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 t, float (&v)[kVec]) {
        v[0] = bf16_lo(t.x); v[1] = bf16_hi(t.x); v[2] = bf16_lo(t.y); v[3] = bf16_hi(t.y);
        v[4] = bf16_lo(t.z); v[5] = bf16_hi(t.z); v[6] = bf16_lo(t.w); v[7] = bf16_hi(t.w);
    }
    __device__ __forceinline__ static void load_vec(const void* p, float (&v)[kVec]) {
        unpack(__ldg(reinterpret_cast<const uint4*>(p)), v);
    }
    __device__ __forceinline__ static void load_vec_stream(const T* p, float (&v)[kVec]) {
        unpack(__ldcs(reinterpret_cast<const uint4*>(p)), v);
    }
    __device__ __forceinline__ static float2 pair(uint32_t u) {
        return make_float2(bf16_lo(u), bf16_hi(u));
    }
    __device__ __forceinline__ static float2 load_xy(const T* p) {
        return pair(__ldcs(reinterpret_cast<const unsigned int*>(p)));
    }
    __device__ __forceinline__ static float load_one(const T* p) {
        const unsigned short u = __ldcs(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    }
    __device__ __forceinline__ static float4 load_xywh(const T* p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    }
    __device__ __forceinline__ static void store_vec(T* p, const float (&v)[kVec]) {
        uint4 t;
        t.x = pack_bf16x2(v[0], v[1]); t.y = pack_bf16x2(v[2], v[3]);
        t.z = pack_bf16x2(v[4], v[5]); t.w = pack_bf16x2(v[6], v[7]);
        __stcs(reinterpret_cast<uint4*>(p), t);
    }
    __device__ __forceinline__ static void store_one(T* p, float v) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        __stcs(reinterpret_cast<unsigned short*>(p), *reinterpret_cast<const unsigned short*>(&h));
    }
    __device__ __forceinline__ static void store_xy(T* p, float x, float y) {
        __stcs(reinterpret_cast<unsigned int*>(p), pack_bf16x2(x, y));
    }
};

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t u) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return __half22float2(h);
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <>
struct IO<__half> {
    using T = __half;
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 t, float (&v)[kVec]) {
        const float2 a = half2_bits_to_float2(t.x), b = half2_bits_to_float2(t.y);
        const float2 c = half2_bits_to_float2(t.z), d = half2_bits_to_float2(t.w);
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
    }
    __device__ __forceinline__ static void load_vec(const void* p, float (&v)[kVec]) {
        unpack(__ldg(reinterpret_cast<const uint4*>(p)), v);
    }
    __device__ __forceinline__ static void load_vec_stream(const T* p, float (&v)[kVec]) {
        unpack(__ldcs(reinterpret_cast<const uint4*>(p)), v);
    }
    __device__ __forceinline__ static float2 pair(uint32_t u) { return half2_bits_to_float2(u); }
    __device__ __forceinline__ static float2 load_xy(const T* p) {
        return pair(__ldcs(reinterpret_cast<const unsigned int*>(p)));
    }
    __device__ __forceinline__ static float load_one(const T* p) {
        const unsigned short u = __ldcs(reinterpret_cast<const unsigned short*>(p));
        return __half2float(__ushort_as_half(u));
    }
    __device__ __forceinline__ static float4 load_xywh(const T* p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        const float2 a = half2_bits_to_float2(u.x), b = half2_bits_to_float2(u.y);
        return make_float4(a.x, a.y, b.x, b.y);
    }
    __device__ __forceinline__ static void store_vec(T* p, const float (&v)[kVec]) {
        uint4 t;
        t.x = pack_half2(v[0], v[1]); t.y = pack_half2(v[2], v[3]);
        t.z = pack_half2(v[4], v[5]); t.w = pack_half2(v[6], v[7]);
        __stcs(reinterpret_cast<uint4*>(p), t);
    }
    __device__ __forceinline__ static void store_one(T* p, float v) {
        __stcs(reinterpret_cast<unsigned short*>(p), __half_as_ushort(__float2half_rn(v)));
    }
    __device__ __forceinline__ static void store_xy(T* p, float x, float y) {
        __stcs(reinterpret_cast<unsigned int*>(p), pack_half2(x, y));
    }
};

// 32-byte vectors (one 256-bit load per lane, sm_100+).  Value rows are read
// through the non-coherent path and kept in L1.
template <typename T>
struct IO32;

template <>
struct IO32<float> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void load(const void* p, float (&v)[kVec]) {
        asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                       "=f"(v[6]), "=f"(v[7])
                     : "l"(p));
    }
    __device__ __forceinline__ static void load_stream(const float* p, float (&v)[kVec]) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    __device__ __forceinline__ static void store(float* p, const float (&v)[kVec]) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
};

template <>
struct IO32<__nv_bfloat16> {
    using T = __nv_bfloat16;
    static constexpr int kVec = 16;
    __device__ __forceinline__ static void unpack(const uint32_t (&u)[8], float (&v)[kVec]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = bf16_lo(u[i]);
            v[2 * i + 1] = bf16_hi(u[i]);
        }
    }
    __device__ __forceinline__ static void load(const void* p, float (&v)[kVec]) {
        uint32_t u[8];
        asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]),
                       "=r"(u[6]), "=r"(u[7])
                     : "l"(p));
        unpack(u, v);
    }
    __device__ __forceinline__ static void load_stream(const T* p, float (&v)[kVec]) {
        const uint4 a = __ldcs(reinterpret_cast<const uint4*>(p));
        const uint4 b = __ldcs(reinterpret_cast<const uint4*>(p) + 1);
        const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        unpack(u, v);
    }
    __device__ __forceinline__ static void store(T* p, const float (&v)[kVec]) {
        uint4 a, b;
        a.x = pack_bf16x2(v[0], v[1]); a.y = pack_bf16x2(v[2], v[3]);
        a.z = pack_bf16x2(v[4], v[5]); a.w = pack_bf16x2(v[6], v[7]);
        b.x = pack_bf16x2(v[8], v[9]); b.y = pack_bf16x2(v[10], v[11]);
        b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
        __stcs(reinterpret_cast<uint4*>(p), a);
        __stcs(reinterpret_cast<uint4*>(p) + 1, b);
    }
};

template <>
struct IO32<__half> {
    using T = __half;
    static constexpr int kVec = 16;
    __device__ __forceinline__ static void load(const void* p, float (&v)[kVec]) {
        uint32_t u[8];
        asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]),
                       "=r"(u[6]), "=r"(u[7])
                     : "l"(p));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 f = half2_bits_to_float2(u[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ __forceinline__ static void store(T* p, const float (&v)[kVec]) {
        uint4 a, b;
        a.x = pack_half2(v[0], v[1]); a.y = pack_half2(v[2], v[3]);
        a.z = pack_half2(v[4], v[5]); a.w = pack_half2(v[6], v[7]);
        b.x = pack_half2(v[8], v[9]); b.y = pack_half2(v[10], v[11]);
        b.z = pack_half2(v[12], v[13]); b.w = pack_half2(v[14], v[15]);
        __stcs(reinterpret_cast<uint4*>(p), a);
        __stcs(reinterpret_cast<uint4*>(p) + 1, b);
    }
};

// Row vectors of kBytes (16 or 32) bytes: the loads of value rows and the
// stores of output rows in the forward kernel.
template <typename T, int kBytes>
struct VecIO;

// 8-byte vectors of a 16-bit type: four channels, whose fp32 gradient is one
// 16-byte red (the backward's layout for half types, see backward_kernel).
template <typename T>
struct VecIO<T, 8> {
    static_assert(sizeof(T) == 2, "8-byte vectors hold four 16-bit values");
    static constexpr int kVec = 4;
    __device__ __forceinline__ static void unpack(const uint2 u, float (&v)[kVec]) {
        const float2 a = IO<T>::pair(u.x), b = IO<T>::pair(u.y);
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    }
    __device__ __forceinline__ static void load(const void* p, float (&v)[kVec]) {
        unpack(__ldg(reinterpret_cast<const uint2*>(p)), v);
    }
    __device__ __forceinline__ static void load_stream(const T* p, float (&v)[kVec]) {
        unpack(__ldcs(reinterpret_cast<const uint2*>(p)), v);
    }
    // round to nearest even, as the 16-byte stores
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        if constexpr (std::is_same<T, __half>::value) return pack_half2(lo, hi);
        else return pack_bf16x2(lo, hi);
    }
    __device__ __forceinline__ static void store(T* p, const float (&v)[kVec]) {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(pack(v[0], v[1]), pack(v[2], v[3])));
    }
};

template <typename T>
struct VecIO<T, 16> {
    static constexpr int kVec = IO<T>::kVec;
    __device__ __forceinline__ static void load(const void* p, float (&v)[kVec]) {
        IO<T>::load_vec(p, v);
    }
    __device__ __forceinline__ static void load_stream(const T* p, float (&v)[kVec]) {
        IO<T>::load_vec_stream(p, v);
    }
    __device__ __forceinline__ static void store(T* p, const float (&v)[kVec]) {
        IO<T>::store_vec(p, v);
    }
};

template <typename T>
struct VecIO<T, 32> {
    static constexpr int kVec = IO32<T>::kVec;
    __device__ __forceinline__ static void load(const void* p, float (&v)[kVec]) {
        IO32<T>::load(p, v);
    }
    __device__ __forceinline__ static void store(T* p, const float (&v)[kVec]) {
        IO32<T>::store(p, v);
    }
};

// ------------------------------------------------------------- level table
// One entry per level: H, W, first key, and whether every pixel of the level
// lies inside [0, num_keys).  Built once per CTA in shared memory, together
// with the level of every flattened (level, point) index j < L*P.
struct LevelInfo {
    int H, W, start, ok;
};

// spatial_shapes / level_start_index hold int64, or int32 when idx32.
__device__ __forceinline__ int64_t index_at(const void* p, int i, int idx32) {
    return idx32 ? (int64_t) static_cast<const int32_t*>(p)[i] : static_cast<const int64_t*>(p)[i];
}

__device__ __forceinline__ void load_level_table(LevelInfo* s_levels, unsigned char* s_level_of,
                                                 const void* __restrict__ spatial_shapes,
                                                 const void* __restrict__ level_start_index,
                                                 int idx32, int num_levels, int num_points,
                                                 int num_keys) {
    if (threadIdx.x < num_levels) {
        const int l = threadIdx.x;
        const int64_t H = index_at(spatial_shapes, 2 * l, idx32);
        const int64_t W = index_at(spatial_shapes, 2 * l + 1, idx32);
        const int64_t s = index_at(level_start_index, l, idx32);
        const bool ok = H >= 0 && W >= 0 && H < (1 << 24) && W < (1 << 24) && s >= 0 &&
                        s + H * W <= (int64_t)num_keys;
        LevelInfo li;
        li.H = ok ? (int)H : 0;
        li.W = ok ? (int)W : 0;
        li.start = ok ? (int)s : 0;
        li.ok = ok;
        s_levels[l] = li;
        if (!ok && blockIdx.x == 0) atomicOr(&g_error_word, kErrLevelOutOfRange);
    }
    const int LP = num_levels * num_points;
    for (int j = threadIdx.x; j < LP; j += blockDim.x) s_level_of[j] = (unsigned char)(j / num_points);
}

// --------------------------------------------------------------- footprint
// Bilinear footprint of one sample.
//   key[c] : flattened key of corner c, or -1 when the corner is off the map
//            or the sample is not live (such corners are never read)
//   fx, fy : fractions inside the cell (0 for a dead sample)
//   w[c]   : (1-fx)(1-fy), fx(1-fy), (1-fx)fy, fx*fy
struct Footprint {
    int key[4];
    int x0, y0;  // cell (top-left pixel); 0 for a dead sample
    float fx, fy;
    float w[4];
    bool live;
};

// x, y: pixel coordinates already rounded to fp32 (one FMA each).
__device__ __forceinline__ Footprint make_footprint(float x, float y, const LevelInfo& lv) {
    Footprint f;
    const float Wf = (float)lv.W, Hf = (float)lv.H;
    f.live = lv.ok && (x > -1.f) && (x < Wf) && (y > -1.f) && (y < Hf);  // NaN -> dead
    const float xs = f.live ? x : 0.f, ys = f.live ? y : 0.f;
    const float x0f = floorf(xs), y0f = floorf(ys);
    f.fx = xs - x0f;  // exact for |x| >= 1 (Sterbenz); for x in (-1, 0) one rounding
    f.fy = ys - y0f;
    const int x0 = (int)x0f, y0 = (int)y0f;
    f.x0 = x0;
    f.y0 = y0;
    const bool vx0 = f.live && x0 >= 0, vx1 = f.live && x0 + 1 < lv.W;
    const bool vy0 = y0 >= 0, vy1 = y0 + 1 < lv.H;
    const int k00 = lv.start + y0 * lv.W + x0;
    f.key[0] = (vx0 && vy0) ? k00 : -1;
    f.key[1] = (vx1 && vy0) ? k00 + 1 : -1;
    f.key[2] = (vx0 && vy1) ? k00 + lv.W : -1;
    f.key[3] = (vx1 && vy1) ? k00 + lv.W + 1 : -1;
    const float gx = 1.f - f.fx, gy = 1.f - f.fy;
    f.w[0] = gx * gy;
    f.w[1] = f.fx * gy;
    f.w[2] = gx * f.fy;
    f.w[3] = f.fx * f.fy;
    return f;
}

// Key padding mask of the fused entry points (the module's masked_fill of
// value): a corner on a padded key reads as zero, which is what an off-map
// corner does, so it is dropped the same way.  mrow: the tile's batch row of
// the [bs, K] mask.
__device__ __forceinline__ void mask_corners(Footprint& fp, const unsigned char* __restrict__ mrow) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
        if (fp.key[c] >= 0 && __ldg(mrow + fp.key[c]) != 0) fp.key[c] = -1;
}

// Corners of a footprint reordered by pixel parity class t = (x & 1) + 2 (y & 1).
// Each sample has exactly one corner in each class, so two samples can share
// a pixel only within the same class.  kw[t] is corner weight * a (0 when off
// the map).
struct ClassCorners {
    int key[4];
    float w[4];
};

__device__ __forceinline__ ClassCorners class_corners(const Footprint& f, float a) {
    ClassCorners cc;
    const int px = f.x0 & 1, py = f.y0 & 1;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int c = (((t >> 1) ^ py) << 1) | ((t & 1) ^ px);  // corner holding class t
        const int k = c == 0 ? f.key[0] : c == 1 ? f.key[1] : c == 2 ? f.key[2] : f.key[3];
        const float w = c == 0 ? f.w[0] : c == 1 ? f.w[1] : c == 2 ? f.w[2] : f.w[3];
        cc.key[t] = k;
        cc.w[t] = k >= 0 ? a * w : 0.f;
    }
    return cc;
}

// Byte address of the row of `key` in a [*, num_keys, M, D] slice starting at base.
__device__ __forceinline__ const char* row_ptr(const char* base, int key, unsigned row_bytes) {
    return base + (size_t)(unsigned)key * row_bytes;
}

// Fire-and-forget vector fp32 add into global memory (sm_90+ vector red).
// No "memory" clobber unless MSDA_RED_CLOBBER: the kernels that call it never
// read the buffer they add into, and without the clobber the compiler may
// schedule the gathers of later samples ahead of these reds.
#ifndef MSDA_RED_CLOBBER
#define MSDA_RED_CLOBBER 0
#endif
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
#if MSDA_RED_CLOBBER
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
#else
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d));
#endif
}

// red_add_v4 under a predicate, one instruction (no branch around it).
__device__ __forceinline__ void red_add_v4_if(bool pred, float* p, float a, float b, float c,
                                              float d) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
                 "@q red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n\t}" ::"l"(p),
                 "f"(a), "f"(b), "f"(c), "f"(d), "r"((int)pred));
}

// Geometry of a warp tile for lane groups of kLanes lanes.
template <int kLanes>
struct TileGeom {
    static_assert(kLanes >= 1 && kLanes <= 32 && (kLanes & (kLanes - 1)) == 0, "lane group");
    static constexpr int kGroups = 32 / kLanes;                  // queries per warp tile
    static constexpr int kSPG = kSamplesPerWarp / kGroups;       // samples per group per round
    static constexpr int kStride = kSPG + 1;                     // padded record stride (16 B units)
    static constexpr int kRecords = kGroups * kStride;           // records per warp
};

// Warp tile t -> (b, first query, m).  Tiles are ordered (b, m, query block):
// consecutive tiles are neighbouring queries of one head, and a CTA walks a
// contiguous range of them, so the value rows its samples touch stay in L1.
struct TileCoord {
    int b, q0, m;
};
__device__ __forceinline__ TileCoord tile_coord(int t, int num_heads, int num_qtiles, int groups) {
    TileCoord c;
    const int qt = t % num_qtiles;
    const int rest = t / num_qtiles;
    c.q0 = qt * groups;
    c.m = rest % num_heads;
    c.b = rest / num_heads;
    return c;
}

// Locations and attention weights of the two samples a lane handles in one
// round of a warp tile, loaded one round ahead of their use.
struct SampleFetch {
    float2 xy[2];
    float a[2];
    bool ok[2];
};

template <typename T, int kSPG>
__device__ __forceinline__ void fetch_samples(SampleFetch& f, const T* __restrict__ loc,
                                              const T* __restrict__ attn, const TileCoord& tc,
                                              int r0, int lane, int LP, int num_queries,
                                              int num_heads) {
#pragma unroll
    for (int h = 0; h < kSamplesPerWarp / 32; ++h) {
        const int s = lane + 32 * h;
        const int sg = s / kSPG, sj = s % kSPG;
        const int j = r0 + sj, q = tc.q0 + sg;
        f.ok[h] = q < num_queries && j < LP;
        f.xy[h] = make_float2(0.f, 0.f);
        f.a[h] = 0.f;
        if (f.ok[h]) {
            const int64_t pt = (((int64_t)tc.b * num_queries + q) * num_heads + tc.m) * LP + j;
            f.xy[h] = IO<T>::load_xy(loc + 2 * pt);
            f.a[h] = IO<T>::load_one(attn + pt);
        }
    }
}

// ---------------------------------------------------------- fused preparation
// The fused entry points take, instead of locations and weights, reference
// points [bs, Q, L, ref_dim] (ref_dim 2: (x, y); 4: (x, y, w, h)), sampling
// offsets in the layout of sampling_locations and attention logits in the
// layout of attention_weights (Deformable DETR walk-through, "2.2.4 源码分析",
// MSDeformAttn.forward; 4-d references from section "2.4").  A fused round
// fetches, per sample, the offsets into SampleFetch::xy, the logit into
// SampleFetch::a, and the reference point into PrepFetch.
struct PrepFetch {
    float2 rxy[2], rwh[2];
};

// A fused tile is one round (L*P <= kSPG), so the level of each of a lane's
// two samples, and the offset of its reference point inside the tile's block
// of references, stay the same for every tile the lane visits.
struct PrepLane {
    int ref_off[2];  // (group * L + level) * ref_dim
};

template <int kSPG>
__device__ __forceinline__ PrepLane prep_lane(int lane, int num_levels, int LP, int ref_dim,
                                              const unsigned char* s_level_of) {
    PrepLane pl;
#pragma unroll
    for (int h = 0; h < kSamplesPerWarp / 32; ++h) {
        const int s = lane + 32 * h;
        const int sg = s / kSPG, sj = s % kSPG;
        const int l = sj < LP ? s_level_of[sj] : 0;
        pl.ref_off[h] = (sg * num_levels + l) * ref_dim;
    }
    return pl;
}

// Reference points are only prefetched into L1 one round ahead (prefetch_refs)
// and loaded when their round starts (fetch_refs), so they are not live in
// registers across the gather; measured faster than loading them a round ahead.
template <typename T, int kRef>
__device__ __forceinline__ void fetch_refs(PrepFetch& pf, const SampleFetch& f,
                                           const T* __restrict__ ref,
                                           const TileCoord& tc, int num_queries, int num_levels,
                                           const PrepLane& pl) {
    const T* rt = ref + ((int64_t)tc.b * num_queries + tc.q0) * (num_levels * kRef);
#pragma unroll
    for (int h = 0; h < kSamplesPerWarp / 32; ++h) {
        pf.rxy[h] = make_float2(0.f, 0.f);
        pf.rwh[h] = make_float2(0.f, 0.f);
        if (f.ok[h]) {
            if constexpr (kRef == 4) {
                const float4 r = IO<T>::load_xywh(rt + pl.ref_off[h]);
                pf.rxy[h] = make_float2(r.x, r.y);
                pf.rwh[h] = make_float2(r.z, r.w);
            } else {
                pf.rxy[h] = IO<T>::load_xy(rt + pl.ref_off[h]);
            }
        }
    }
}

template <typename T, int kRef>
__device__ __forceinline__ void prefetch_refs(const SampleFetch& f, const T* __restrict__ ref,
                                              const TileCoord& tc, int num_queries,
                                              int num_levels, const PrepLane& pl) {
    const T* rt = ref + ((int64_t)tc.b * num_queries + tc.q0) * (num_levels * kRef);
#pragma unroll
    for (int h = 0; h < kSamplesPerWarp / 32; ++h)
        if (f.ok[h]) asm volatile("prefetch.global.L1 [%0];" ::"l"(rt + pl.ref_off[h]));
}

// Sampling location of one sample: the module's expression (Deformable DETR
// walk-through, "2.2.4 源码分析", MSDeformAttn.forward; 4-d references from
// section "2.4") in binary32, one correctly rounded operation at a time, left
// to right, with IEEE division:
//   2-d: loc = ref + off / (W, H)
//   4-d: loc = ref_xy + off / P * ref_wh * 0.5
// w, h: the level's width and height; p: the number of points (exact floats).
template <int kRef>
__device__ __forceinline__ float2 prep_location(float2 rxy, float2 rwh, float2 off, float w,
                                                float h, float p) {
    if constexpr (kRef == 2)
        return make_float2(__fadd_rn(rxy.x, __fdiv_rn(off.x, w)),
                           __fadd_rn(rxy.y, __fdiv_rn(off.y, h)));
    return make_float2(__fadd_rn(rxy.x, __fmul_rn(__fmul_rn(__fdiv_rn(off.x, p), rwh.x), 0.5f)),
                       __fadd_rn(rxy.y, __fmul_rn(__fmul_rn(__fdiv_rn(off.y, p), rwh.y), 0.5f)));
}

// Replaces the logits in f.a by the softmax over each row's L*P samples.  A
// fused round holds whole rows (L*P <= kSPG): for kSPG <= 32 a row is an
// aligned segment of kSPG lanes of one half (h) of the round, for kSPG = 64 it
// is both halves of all 32 lanes.  Samples past the row's end do not count; a
// row with no sample (a query past the last) gets weights 0.
template <int kSPG>
__device__ __forceinline__ void softmax_rows(SampleFetch& f) {
    constexpr int kSeg = kSPG < 32 ? kSPG : 32;
    if constexpr (kSPG == 64) {
        float m = fmaxf(f.ok[0] ? f.a[0] : -INFINITY, f.ok[1] ? f.a[1] : -INFINITY);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float e0 = f.ok[0] && m != -INFINITY ? expf(f.a[0] - m) : 0.f;
        const float e1 = f.ok[1] && m != -INFINITY ? expf(f.a[1] - m) : 0.f;
        float sum = e0 + e1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = sum > 0.f ? __frcp_rn(sum) : 0.f;
        f.a[0] = e0 * inv;
        f.a[1] = e1 * inv;
    } else {
#pragma unroll
        for (int h = 0; h < kSamplesPerWarp / 32; ++h) {
            float m = f.ok[h] ? f.a[h] : -INFINITY;
#pragma unroll
            for (int o = 1; o < kSeg; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float e = f.ok[h] && m != -INFINITY ? expf(f.a[h] - m) : 0.f;
            float sum = e;
#pragma unroll
            for (int o = 1; o < kSeg; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            f.a[h] = sum > 0.f ? e * __frcp_rn(sum) : 0.f;
        }
    }
}

// The (tile, round) steps one warp executes: tiles begin + warp, begin + warp
// + stride, ... below end; each tile in rounds of spg samples per group.
struct StepIter {
    int t, r0, end, LP, spg, stride;  // stride: warps per CTA
    __device__ __forceinline__ bool valid() const { return t < end; }
    __device__ __forceinline__ bool last_round() const { return r0 + spg >= LP; }
    __device__ __forceinline__ void next() {
        r0 += spg;
        if (r0 >= LP) {
            r0 = 0;
            t += stride;
        }
    }
};

}  // namespace msda
