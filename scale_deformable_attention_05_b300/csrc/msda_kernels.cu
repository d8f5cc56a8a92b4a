// All device code of the library, in one translation unit: the forward and
// backward kernels (instantiated per element type and lane layout), the
// fill / finalize / shape-check kernels, and the host-side launchers the
// C ABI calls.
#include <algorithm>

#include "msda_backward.cuh"
#include "msda_device.cuh"
#include "msda_forward.cuh"
#include "msda_launch.h"

namespace msda {

__device__ int g_shape_check = 0;

// ------------------------------------------------------------ small kernels
// Grid-stride zero fill: n16 16-byte words, then tail_bytes (< 16) single bytes.
__global__ void zero_fill_kernel(uint4* __restrict__ p, size_t n16, int tail_bytes) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = z;
    if (blockIdx.x == 0 && threadIdx.x < tail_bytes)
        reinterpret_cast<unsigned char*>(p + n16)[threadIdx.x] = 0;
}

// Half-precision grad_value from the fp32 workspace: overwrite, or add when
// accumulating.  n8 = number of 8-element groups (head_dim % 8 == 0 makes the
// total a multiple of 8).
template <typename T>
__global__ void finalize_half_kernel(const float4* __restrict__ ws, T* __restrict__ gv,
                                     size_t n8, int accumulate) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (size_t)gridDim.x * blockDim.x) {
        const float4 a = __ldcs(ws + 2 * i), b = __ldcs(ws + 2 * i + 1);
        float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (accumulate) {
            float old[8];
            IO<T>::load_vec_stream(gv + 8 * i, old);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] += old[e];
        }
        IO<T>::store_vec(gv + 8 * i, v);
    }
}

// One thread: level_start_index must be the exclusive prefix sum of H*W and
// the levels must add up to num_keys.
__global__ void check_shapes_kernel(const int64_t* __restrict__ shapes,
                                    const int64_t* __restrict__ lsi, int num_levels,
                                    int num_keys) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    int64_t acc = 0;
    int ok = 1;
    for (int l = 0; l < num_levels; ++l) {
        const int64_t H = shapes[2 * l], W = shapes[2 * l + 1];
        if (H < 0 || W < 0 || lsi[l] != acc) ok = 0;
        acc += H * W;
    }
    if (acc != (int64_t)num_keys) ok = 0;
    g_shape_check = ok;
}

// ---------------------------------------------------------------- dispatch
namespace {

struct Layout {
    int lanes, vpl;
};

// Lanes per lane group and row vectors per lane for a head of `nvec` vectors
// (of whatever width the kernel reads): one vector per lane up to 32 vectors
// (at least 4 lanes, so a warp tile holds at most 8 queries), then 2 or 4
// vectors on 32 lanes.
Layout choose_layout(int nvec) {
    Layout ly{4, 1};
    if (nvec <= 32) {
        while (ly.lanes < nvec) ly.lanes <<= 1;
    } else {
        ly.lanes = 32;
        ly.vpl = nvec <= 64 ? 2 : 4;
    }
    return ly;
}

// Waves of resident CTAs per launch: 0 picks them from the working set
// (persistent_waves), a positive value fixes them.
#ifndef MSDA_PERSISTENT_WAVES
#define MSDA_PERSISTENT_WAVES 0
#endif

int sm_count() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

int64_t l2_bytes() {
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    return l2 > 0 ? l2 : (int64_t)126 << 20;
}

// Waves per launch from the working set: value (and, in the backward, its fp32
// gradient) over a target share of L2, rounded up to a power of two and capped.
// The CTAs resident at a time then cover that share of the (b, m)-ordered
// tiles, whose value and grad_value slices stay in L2 against the streamed
// inputs and outputs, and the shorter tile ranges of more waves even out the
// CTAs' finishing times.  Targets from sweeps of 1..64 waves (kernel-only CUDA
// events) with the current CTA shapes (4-warp CTAs): the backward wants ~L2 / 13
// of slices live, at most 16 waves (fp32 encoder 2 -> 16 waves: 412 -> 395 us,
// bf16 822 -> 766, fp16 825 -> 767; 32 and 64 slower; D = 256 envelope best at
// 8-16), the forward ~L2 / 32, at most 32 waves (fp32 encoder 4 -> 16: 162 ->
// 158 us, bf16 285 -> 274; envelope best at 32).
int persistent_waves(const Problem& pb, int elem_bytes, bool backward) {
    if (MSDA_PERSISTENT_WAVES > 0) return MSDA_PERSISTENT_WAVES;
    const double ws = (double)pb.bs * pb.K * pb.M * pb.D * (elem_bytes + (backward ? 4 : 0));
    const double target = (double)l2_bytes() * (backward ? 0.075 : 1.0 / 32.0);
    const int cap = backward ? 16 : 32;
    int w = 1;
    while (w < cap && w * target < ws) w <<= 1;
    return w;
}

#ifndef MSDA_SMEM_CARVEOUT
#define MSDA_SMEM_CARVEOUT -1
#endif

// CTAs of `Kernel` that fit on one SM at once, looked up once per kernel.  The
// cache is keyed by the kernel itself: instantiations that differ only in their
// template arguments share one function type but not their register counts.
template <auto Kernel>
int resident_ctas(int threads) {
    static const int n = [threads] {
        if (MSDA_SMEM_CARVEOUT >= 0)
            cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 MSDA_SMEM_CARVEOUT);
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, Kernel, threads, 0) != cudaSuccess ||
            v < 1)
            v = 1;
        return v;
    }();
    return n;
}

struct TileGrid {
    int num_qtiles, num_tiles, tiles_per_cta, grid;
};

// Warp tiles of `queries_per_tile` queries, ordered (b, m, query block).  The grid is
// `waves` waves of resident CTAs; each CTA takes a contiguous
// range of tiles (a multiple of its warps), so consecutive tiles of one head
// run on one SM and share its L1.
TileGrid tile_grid(const Problem& pb, int queries_per_tile, int resident, int warps, int waves) {
    TileGrid tg;
    tg.num_qtiles = (pb.Q + queries_per_tile - 1) / queries_per_tile;
    tg.num_tiles = pb.bs * pb.M * tg.num_qtiles;
    const int64_t ctas = (int64_t)sm_count() * resident * waves;
    int64_t per = (tg.num_tiles + ctas - 1) / ctas;
    per = (per + warps - 1) / warps * warps;
    tg.tiles_per_cta = (int)per;
    tg.grid = (int)((tg.num_tiles + per - 1) / per);
    return tg;
}

template <typename T, int kLanes, int kVPL, int kVB, int kRef = 0>
cudaError_t launch_forward_t(const Problem& pb, void* out, cudaStream_t st) {
    auto kernel = forward_kernel<T, kLanes, kVPL, kVB, kRef>;
    constexpr int kThreads = MSDA_FWD_WARPS * 32;
    const int resident = resident_ctas<forward_kernel<T, kLanes, kVPL, kVB, kRef>>(kThreads);
    const TileGrid tg = tile_grid(pb, 32 / kLanes, resident, MSDA_FWD_WARPS,
                                  persistent_waves(pb, (int)sizeof(T), false));
    kernel<<<tg.grid, kThreads, 0, st>>>(
        static_cast<const T*>(pb.value), pb.shapes, pb.lsi, pb.idx32, static_cast<const T*>(pb.loc),
        static_cast<const T*>(pb.attn), static_cast<T*>(out), pb.K, pb.M, pb.D, pb.L, pb.P, pb.Q,
        tg.num_qtiles, tg.num_tiles, tg.tiles_per_cta, static_cast<const T*>(pb.ref), pb.mask);
    return cudaGetLastError();
}

template <typename T, int kLanes, int kVPL, int kRef, int kVB, bool kDense>
cudaError_t launch_backward_shape(const Problem& pb, const TileGrid& tg, const void* grad_out,
                                  float* gv32, void* grad_loc, void* grad_attn, cudaStream_t st,
                                  float* grad_ref) {
    auto kernel = backward_kernel<T, kLanes, kVPL, kRef, kVB, kDense>;
    constexpr int kThreads = BwdShape<T, kLanes, kVPL, kRef, kDense>::kWarps * 32;
    kernel<<<tg.grid, kThreads, 0, st>>>(
        static_cast<const T*>(pb.value), pb.shapes, pb.lsi, pb.idx32, static_cast<const T*>(pb.loc),
        static_cast<const T*>(pb.attn), static_cast<const T*>(grad_out), gv32,
        static_cast<T*>(grad_loc), static_cast<T*>(grad_attn), pb.K, pb.M, pb.D, pb.L, pb.P,
        pb.Q, tg.num_qtiles, tg.num_tiles, tg.tiles_per_cta, static_cast<const T*>(pb.ref),
        pb.mask, grad_ref);
    return cudaGetLastError();
}

template <typename T, int kLanes, int kVPL, int kRef, int kVB>
cudaError_t launch_backward_t(const Problem& pb, const void* grad_out, float* gv32,
                              void* grad_loc, void* grad_attn, cudaStream_t st,
                              float* grad_ref = nullptr) {
    constexpr int kWarps = BwdShape<T, kLanes, kVPL, kRef>::kWarps;
    constexpr int kThreads = kWarps * 32;
    const int waves = persistent_waves(pb, (int)sizeof(T), true);
    if constexpr (sizeof(T) == 4 && BwdShape<T, kLanes, kVPL, kRef>::kNarrow) {
        // the dense shape where its grid fills every SM's slots at least once
        const int dense =
            resident_ctas<backward_kernel<T, kLanes, kVPL, kRef, kVB, true>>(kThreads);
        const TileGrid td = tile_grid(pb, 32 / kLanes, dense, kWarps, waves);
        if ((int64_t)td.grid >= (int64_t)sm_count() * dense)
            return launch_backward_shape<T, kLanes, kVPL, kRef, kVB, true>(pb, td, grad_out, gv32,
                                                                           grad_loc, grad_attn, st,
                                                                           grad_ref);
    }
    const int resident = resident_ctas<backward_kernel<T, kLanes, kVPL, kRef, kVB>>(kThreads);
    const TileGrid tg = tile_grid(pb, 32 / kLanes, resident, kWarps, waves);
    return launch_backward_shape<T, kLanes, kVPL, kRef, kVB, false>(pb, tg, grad_out, gv32,
                                                                    grad_loc, grad_attn, st,
                                                                    grad_ref);
}

#ifndef MSDA_FWD_VEC32
#define MSDA_FWD_VEC32 1
#endif

template <typename T, int kVB>
cudaError_t dispatch_forward_vec(const Problem& pb, void* out, cudaStream_t st) {
    const int nvec = pb.D * (int)sizeof(T) / kVB;
    Layout ly{1, 1};
    if (nvec <= 32) {
        while (ly.lanes < nvec) ly.lanes <<= 1;
    } else {
        ly.lanes = 32;
        ly.vpl = nvec <= 64 ? 2 : 4;
    }
    if (kVB == 16 && ly.lanes < 4) ly.lanes = 4;
    if (ly.vpl == 1) {
        switch (ly.lanes) {
            case 1: return launch_forward_t<T, 1, 1, kVB>(pb, out, st);
            case 2: return launch_forward_t<T, 2, 1, kVB>(pb, out, st);
            case 4: return launch_forward_t<T, 4, 1, kVB>(pb, out, st);
            case 8: return launch_forward_t<T, 8, 1, kVB>(pb, out, st);
            case 16: return launch_forward_t<T, 16, 1, kVB>(pb, out, st);
            default: return launch_forward_t<T, 32, 1, kVB>(pb, out, st);
        }
    }
    if (ly.vpl == 2) return launch_forward_t<T, 32, 2, kVB>(pb, out, st);
    return launch_forward_t<T, 32, 4, kVB>(pb, out, st);
}

// Rows of 1 KB or more (two or more 16-byte vectors per lane) use 256-bit
// loads: half the load instructions, measured faster on head_dim 256 fp32.
// Shorter rows keep 128-bit loads, which measured as fast or faster.
// Lane groups of the fused kernels: enough for the row's vectors, at least
// `min_lanes`, and enough that one round (2 * lanes samples per group) holds
// a whole (b, q, m) row of L*P <= 64 samples.
Layout fused_layout(const Problem& pb, int nvec, int min_lanes) {
    Layout ly = choose_layout(nvec);
    int need = min_lanes;
    while (2 * need < pb.L * pb.P) need <<= 1;
    if (ly.lanes < need) ly.lanes = need;
    return ly;
}

template <typename T, int kRef>
cudaError_t dispatch_forward_fused_ref(const Problem& pb, void* out, cudaStream_t st) {
    const Layout ly = fused_layout(pb, pb.D / IO<T>::kVec, 4);
    if constexpr (sizeof(T) == 2) {
        // The group is widened so one round holds the whole row of L*P samples;
        // where 16-byte vectors of a 16-bit row would leave lanes of it idle and
        // 8-byte vectors (four channels a lane) fit the same group, lanes read
        // those instead (more lanes busy at the same queries per warp).
        if (ly.vpl == 1 && ly.lanes > pb.D / IO<T>::kVec && pb.D / 4 <= 32 &&
            fused_layout(pb, pb.D / 4, 4).lanes == ly.lanes) {
            switch (ly.lanes) {
                case 4: return launch_forward_t<T, 4, 1, 8, kRef>(pb, out, st);
                case 8: return launch_forward_t<T, 8, 1, 8, kRef>(pb, out, st);
                case 16: return launch_forward_t<T, 16, 1, 8, kRef>(pb, out, st);
                default: return launch_forward_t<T, 32, 1, 8, kRef>(pb, out, st);
            }
        }
    }
    if (ly.vpl == 1) {
        switch (ly.lanes) {
            case 4: return launch_forward_t<T, 4, 1, 16, kRef>(pb, out, st);
            case 8: return launch_forward_t<T, 8, 1, 16, kRef>(pb, out, st);
            case 16: return launch_forward_t<T, 16, 1, 16, kRef>(pb, out, st);
            default: return launch_forward_t<T, 32, 1, 16, kRef>(pb, out, st);
        }
    }
    if (ly.vpl == 2) return launch_forward_t<T, 32, 2, 16, kRef>(pb, out, st);
    return launch_forward_t<T, 32, 4, 16, kRef>(pb, out, st);
}

template <typename T>
cudaError_t dispatch_forward_fused(const Problem& pb, void* out, cudaStream_t st) {
    return pb.ref_dim == 4 ? dispatch_forward_fused_ref<T, 4>(pb, out, st)
                           : dispatch_forward_fused_ref<T, 2>(pb, out, st);
}

template <typename T>
cudaError_t dispatch_forward(const Problem& pb, void* out, cudaStream_t st) {
    if (pb.ref_dim != 0) return dispatch_forward_fused<T>(pb, out, st);
    const int row = pb.D * (int)sizeof(T);
    if (row % 32 == 0 && row <= 2048 &&
        (MSDA_FWD_VEC32 == 2 || (MSDA_FWD_VEC32 == 1 && row >= 1024)))
        return dispatch_forward_vec<T, 32>(pb, out, st);
    return dispatch_forward_vec<T, 16>(pb, out, st);
}

template <typename T, int kLanes, int kVPL>
cudaError_t launch_backward_merge_t(const Problem& pb, int log2_points, const void* grad_out,
                                    float* gv32, void* grad_loc, void* grad_attn,
                                    cudaStream_t st) {
    auto kernel = backward_merge_kernel<T, kLanes, kVPL>;
    constexpr int kThreads = MSDA_MERGE_WARPS * 32;
    const int resident = resident_ctas<backward_merge_kernel<T, kLanes, kVPL>>(kThreads);
    const TileGrid tg = tile_grid(pb, 32 / kLanes, resident, MSDA_MERGE_WARPS,
                                  persistent_waves(pb, (int)sizeof(T), true));
    kernel<<<tg.grid, kThreads, 0, st>>>(
        static_cast<const T*>(pb.value), pb.shapes, pb.lsi, pb.idx32, static_cast<const T*>(pb.loc),
        static_cast<const T*>(pb.attn), static_cast<const T*>(grad_out), gv32,
        static_cast<T*>(grad_loc), static_cast<T*>(grad_attn), pb.K, pb.M, pb.D, pb.L, pb.P,
        log2_points, pb.Q, tg.num_qtiles, tg.num_tiles, tg.tiles_per_cta);
    return cudaGetLastError();
}

// backward_kernel reads four channels per lane vector: 16 bytes of fp32, 8 bytes
// of a 16-bit type, so that a lane's share of a corner's fp32 grad_value row is
// one 16-byte red and the lane group's reds cover whole 32-byte sectors.
template <typename T>
constexpr int backward_vec_bytes() { return sizeof(T) == 2 ? 8 : 16; }

template <typename T>
int backward_nvec(const Problem& pb) { return pb.D * (int)sizeof(T) / backward_vec_bytes<T>(); }

template <typename T, int kRef, int kMinLanes>
cudaError_t launch_backward_layout(const Problem& pb, Layout ly, const void* g, float* gv32,
                                   void* gl, void* ga, cudaStream_t st, float* gref) {
    constexpr int kVB = backward_vec_bytes<T>();
    if (ly.vpl == 1) {
        switch (ly.lanes) {
            case 4:
                if constexpr (kMinLanes <= 4)
                    return launch_backward_t<T, 4, 1, kRef, kVB>(pb, g, gv32, gl, ga, st, gref);
                [[fallthrough]];
            case 8: return launch_backward_t<T, 8, 1, kRef, kVB>(pb, g, gv32, gl, ga, st, gref);
            case 16: return launch_backward_t<T, 16, 1, kRef, kVB>(pb, g, gv32, gl, ga, st, gref);
            default: return launch_backward_t<T, 32, 1, kRef, kVB>(pb, g, gv32, gl, ga, st, gref);
        }
    }
    if (ly.vpl == 2) return launch_backward_t<T, 32, 2, kRef, kVB>(pb, g, gv32, gl, ga, st, gref);
    return launch_backward_t<T, 32, 4, kRef, kVB>(pb, g, gv32, gl, ga, st, gref);
}

template <typename T, int kRef>
cudaError_t dispatch_backward_fused_ref(const Problem& pb, const void* g, float* gv32, void* gl,
                                        void* ga, cudaStream_t st, float* gref) {
    return launch_backward_layout<T, kRef, 8>(pb, fused_layout(pb, backward_nvec<T>(pb), 8), g,
                                              gv32, gl, ga, st, gref);
}

template <typename T>
cudaError_t dispatch_backward_fused(const Problem& pb, const void* g, float* gv32, void* gl,
                                    void* ga, cudaStream_t st, float* gref) {
    return pb.ref_dim == 4 ? dispatch_backward_fused_ref<T, 4>(pb, g, gv32, gl, ga, st, gref)
                           : dispatch_backward_fused_ref<T, 2>(pb, g, gv32, gl, ga, st, gref);
}

template <typename T>
cudaError_t dispatch_backward(const Problem& pb, const void* g, float* gv32, void* gl, void* ga,
                              cudaStream_t st, float* gref) {
    if (pb.ref_dim != 0) return dispatch_backward_fused<T>(pb, g, gv32, gl, ga, st, gref);
    const Layout ly = choose_layout(pb.D / IO<T>::kVec);
#ifndef MSDA_NO_MERGE_PATH
    // Merged scatter for rows of at least 512 bytes (one lane group per warp,
    // one query per tile): duplicate corner rows among the query's samples of a
    // 32-sample round are sent to L2 once.  For shorter rows the per-sample
    // reds of backward_kernel measured faster (the merge costs more issue
    // slots than the L2 write traffic it saves).
    int log2p = 0;
    while ((1 << log2p) < pb.P) ++log2p;
    if (ly.lanes == 32 && (1 << log2p) == pb.P && pb.P <= 32) {
        if (ly.vpl == 1) return launch_backward_merge_t<T, 32, 1>(pb, log2p, g, gv32, gl, ga, st);
        // fp32 1 KB rows: two queries per warp tile (16 lanes x 4 vectors), so the
        // duplicate rows of neighbouring queries merge too (D = 256 envelope
        // backward 2551 -> 2485 us against one query per tile)
        if (ly.vpl == 2 && sizeof(T) == 4)
            return launch_backward_merge_t<T, 16, 4>(pb, log2p, g, gv32, gl, ga, st);
        if (ly.vpl == 2) return launch_backward_merge_t<T, 32, 2>(pb, log2p, g, gv32, gl, ga, st);
        return launch_backward_merge_t<T, 32, 4>(pb, log2p, g, gv32, gl, ga, st);
    }
#endif
    return launch_backward_layout<T, 0, 4>(pb, choose_layout(backward_nvec<T>(pb)), g, gv32, gl,
                                           ga, st, gref);
}

int grid_for(size_t n, int threads) {
    const int sms = sm_count();
    const size_t want = (n + threads - 1) / threads;
    return (int)std::max<size_t>(1, std::min<size_t>(want, (size_t)sms * 8));
}

}  // namespace

cudaError_t launch_forward(const Problem& pb, void* out, int dtype, cudaStream_t st) {
    if (dtype == kF32) return dispatch_forward<float>(pb, out, st);
    if (dtype == kF16) return dispatch_forward<__half>(pb, out, st);
    return dispatch_forward<__nv_bfloat16>(pb, out, st);
}

cudaError_t launch_backward(const Problem& pb, const void* grad_out, float* gv32, void* grad_loc,
                            void* grad_attn, int dtype, cudaStream_t st, float* grad_ref) {
    if (dtype == kF32)
        return dispatch_backward<float>(pb, grad_out, gv32, grad_loc, grad_attn, st, grad_ref);
    if (dtype == kF16)
        return dispatch_backward<__half>(pb, grad_out, gv32, grad_loc, grad_attn, st, grad_ref);
    return dispatch_backward<__nv_bfloat16>(pb, grad_out, gv32, grad_loc, grad_attn, st,
                                            grad_ref);
}

cudaError_t launch_zero_fill(void* p, size_t bytes, cudaStream_t st) {
    if (bytes == 0) return cudaSuccess;
    const size_t n16 = bytes / 16;
    zero_fill_kernel<<<grid_for(n16 + 1, 256), 256, 0, st>>>(static_cast<uint4*>(p), n16,
                                                              (int)(bytes % 16));
    return cudaGetLastError();
}

cudaError_t launch_finalize_half(const float* ws, void* grad_value, size_t elems, bool accumulate,
                                 int dtype, cudaStream_t st) {
    const size_t n8 = elems / 8;
    if (n8 == 0) return cudaSuccess;
    if (dtype == kF16)
        finalize_half_kernel<__half><<<grid_for(n8, 256), 256, 0, st>>>(
            reinterpret_cast<const float4*>(ws), static_cast<__half*>(grad_value), n8,
            accumulate ? 1 : 0);
    else
        finalize_half_kernel<__nv_bfloat16><<<grid_for(n8, 256), 256, 0, st>>>(
            reinterpret_cast<const float4*>(ws), static_cast<__nv_bfloat16*>(grad_value), n8,
            accumulate ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t check_shapes_blocking(const int64_t* shapes, const int64_t* lsi, int num_levels,
                                  int num_keys, cudaStream_t st, bool* ok) {
    check_shapes_kernel<<<1, 32, 0, st>>>(shapes, lsi, num_levels, num_keys);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int h = 0;
    e = cudaMemcpyFromSymbolAsync(&h, g_shape_check, sizeof(int), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    *ok = (h != 0);
    return e;
}

cudaError_t read_and_clear_error(cudaStream_t st, unsigned* word) {
    unsigned h = 0;
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_error_word, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                                st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    *word = h;
    return e;
}

}  // namespace msda

// The tensor-core linear projection (msda_linear), in this translation unit
// because it shares the device error word.
#include "msda_linear.cuh"
