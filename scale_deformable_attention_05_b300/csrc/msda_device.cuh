// Device-side building blocks shared by the forward and backward kernels:
// element-type traits with 16-byte vector loads/stores, the per-CTA level
// table, and the per-sample "footprint" (bilinear corners of one sample).
//
// Sampling semantics (Deformable DETR walk-through, "2.2.4 源码分析",
// ms_deform_attn_core_pytorch: grid_sample(bilinear, zeros,
// align_corners=False) at grid = 2*loc - 1):
//   x_im = loc_x * W - 0.5 (one fp32 FMA), y_im = loc_y * H - 0.5
//   the sample is live iff -1 < x_im < W and -1 < y_im < H
//   corners (y0,x0), (y0,x0+1), (y0+1,x0), (y0+1,x0+1) with x0 = floor(x_im),
//   weights (1-fx)(1-fy), fx(1-fy), (1-fx)fy, fx*fy; a corner off the map is 0.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msda {

constexpr int kWarpsPerCta = 8;
constexpr int kThreadsPerCta = kWarpsPerCta * 32;
constexpr int kMaxLevels = 16;

// Set (atomicOr) by a kernel that meets a level whose pixels would fall
// outside [0, num_keys); read and cleared by msda_last_device_error().
// Defined here: all device code is compiled as the one translation unit
// msda_kernels.cu (no relocatable device code).
__device__ unsigned int g_error_word = 0;
constexpr unsigned int kErrLevelOutOfRange = 1u;

// ---------------------------------------------------------------- I/O traits
template <typename T>
struct IO;

template <>
struct IO<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    // Value rows: read-only, reused across queries -> keep in L1.
    __device__ __forceinline__ static void load_vec(const float* p, float (&v)[kVec]) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
    // Streamed once (locations, weights, grad_output): evict-first.
    __device__ __forceinline__ static void load_vec_stream(const float* p, float (&v)[kVec]) {
        const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
    __device__ __forceinline__ static float2 load_xy(const float* p) {
        return __ldcs(reinterpret_cast<const float2*>(p));
    }
    __device__ __forceinline__ static float load_one(const float* p) { return __ldcs(p); }
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
    __device__ __forceinline__ static void load_vec(const T* p, float (&v)[kVec]) {
        unpack(__ldg(reinterpret_cast<const uint4*>(p)), v);
    }
    __device__ __forceinline__ static void load_vec_stream(const T* p, float (&v)[kVec]) {
        unpack(__ldcs(reinterpret_cast<const uint4*>(p)), v);
    }
    __device__ __forceinline__ static float2 load_xy(const T* p) {
        const uint32_t u = __ldcs(reinterpret_cast<const unsigned int*>(p));
        return make_float2(bf16_lo(u), bf16_hi(u));
    }
    __device__ __forceinline__ static float load_one(const T* p) {
        const unsigned short u = __ldcs(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
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

// ------------------------------------------------------------- level table
// One entry per level: H, W, first key, and whether every pixel of the level
// lies inside [0, num_keys).  Built once per CTA in shared memory.
struct LevelInfo {
    int H, W, start, ok;
};

__device__ __forceinline__ void load_level_table(LevelInfo* s_levels,
                                                 const int64_t* __restrict__ spatial_shapes,
                                                 const int64_t* __restrict__ level_start_index,
                                                 int num_levels, int num_keys) {
    if (threadIdx.x < num_levels) {
        const int l = threadIdx.x;
        const int64_t H = spatial_shapes[2 * l], W = spatial_shapes[2 * l + 1];
        const int64_t s = level_start_index[l];
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
}

// --------------------------------------------------------------- footprint
// Bilinear footprint of one sample, as stored in shared memory.
//   key00: flattened key of corner (y0, x0) (may be off the map)
//   info : (W << 4) | mask, bit c of mask set when corner c is read
struct Footprint {
    float fx, fy;
    int key00;
    unsigned info;
    float w[4];  // bilinear corner weights (1-fx)(1-fy), fx(1-fy), (1-fx)fy, fx*fy
};

// x, y: pixel coordinates already rounded to fp32 (one FMA each).
__device__ __forceinline__ Footprint make_footprint(float x, float y, const LevelInfo& lv) {
    Footprint f;
    const float Wf = (float)lv.W, Hf = (float)lv.H;
    const bool live = lv.ok && (x > -1.f) && (x < Wf) && (y > -1.f) && (y < Hf);
    const float x0f = floorf(x), y0f = floorf(y);
    f.fx = live ? x - x0f : 0.f;  // exact (Sterbenz)
    f.fy = live ? y - y0f : 0.f;
    const int x0 = live ? (int)x0f : 0, y0 = live ? (int)y0f : 0;
    const float gx = 1.f - f.fx, gy = 1.f - f.fy;
    f.w[0] = gx * gy;
    f.w[1] = f.fx * gy;
    f.w[2] = gx * f.fy;
    f.w[3] = f.fx * f.fy;
    const bool vx0 = x0 >= 0, vx1 = x0 + 1 < lv.W, vy0 = y0 >= 0, vy1 = y0 + 1 < lv.H;
    unsigned mask = (unsigned)(vx0 && vy0) | ((unsigned)(vx1 && vy0) << 1) |
                    ((unsigned)(vx0 && vy1) << 2) | ((unsigned)(vx1 && vy1) << 3);
    if (!live) mask = 0;
    f.key00 = live ? lv.start + y0 * lv.W + x0 : 0;
    f.info = ((unsigned)lv.W << 4) | mask;
    return f;
}

__device__ __forceinline__ int corner_key(int key00, int W, int c) {
    return key00 + (c & 1) + ((c >> 1) ? W : 0);
}

// Sum over the `width` lanes of an aligned lane group (width a power of two).
template <int kWidth>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = kWidth / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Fire-and-forget vector fp32 add into global memory (sm_90+ vector red).
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

}  // namespace msda
