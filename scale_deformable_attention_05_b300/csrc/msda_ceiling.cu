// On-chip ceilings of the operator's data movement, measured on the GPU it
// runs on (libmsda_ceiling.so; `python bench.py --ceiling` prints them).
//
// The operator's kernels gather and scatter rows of one head's channels at
// data-dependent keys: for head_dim 32 in fp32 a row is one 128-byte line.
// These probes replay those access patterns in isolation, with random rows,
// and report rows (or warp instructions) per SM clock:
//   kGatherLdg16  128-bit loads, 8 lanes per row, 4 rows per warp instruction
//   kGatherLdg32  256-bit loads, 4 lanes per row, 8 rows per warp instruction
//   kGatherLds16  the same 128-bit pattern from shared memory
//   kRedShared    scalar fp32 reductions into shared memory, 4 rows per warp
//                 instruction, one float per lane (the pattern of a row
//                 scatter into a shared-memory window)
//   kRedGlobalV4  red.global.add.v4.f32, 8 lanes per row (the global scatter)
//   kRmwShared    plain load + add + store in shared memory (no atomicity),
//                 for comparison with kRedShared
//   kGatherTma4   TMA tile::gather4 (four random rows per copy, one row-high
//                 box) into shared-memory rings, each slot then read once
//                 with 128-bit shared loads: 8 producer / consumer warp pairs
//                 per CTA, 8 slots of 512 bytes each (the copy engine as a
//                 gather path that bypasses the L1 tags)
// `param` selects the region: for the global probes its size in bytes (a
// region that fits L1 measures L1 hits, one of tens of MB measures L2 hits);
// for kRedShared / kRmwShared the bank pattern of the four rows an
// instruction touches (0: four distinct bank residues, conflict-free; 1: one
// residue, a 4-way conflict; 2: rows of 33 floats at random, the pattern of a
// padded window).
//
// Not part of the operator's ABI: a measurement tool, allocating its own
// buffers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace {

enum Probe {
    kGatherLdg16 = 0,
    kGatherLdg32 = 1,
    kGatherLds16 = 2,
    kRedShared = 3,
    kRedGlobalV4 = 4,
    kRmwShared = 5,
    kGatherTma4 = 6,
};

constexpr int kThreads = 512;            // 16 warps per CTA
constexpr int kSharedRows = 512;         // 64 KB of 128-byte rows
constexpr int kSubRows = 128;            // rows per bank class of the shared window

__device__ __forceinline__ uint32_t lcg(uint32_t x) { return x * 1664525u + 1013904223u; }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

struct Stamp {
    long long clk0, clk1;
    unsigned long long ns0, ns1;
};

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Random 128-byte rows of a region of row_mask + 1 rows (a power of two), each
// read by 128 / kBytesPerLane lanes; every lane folds what it reads into one
// register.
template <int kBytesPerLane>
__global__ void __launch_bounds__(kThreads) gather_ldg(const float* __restrict__ base,
                                                       uint32_t row_mask, int iters,
                                                       float* __restrict__ sink,
                                                       Stamp* __restrict__ stamps) {
    constexpr int kLanes = 128 / kBytesPerLane;   // lanes per row
    const int lane = threadIdx.x & 31, g = lane / kLanes, li = lane % kLanes;
    const int warp_id = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    uint32_t x = lcg(0x9e3779b9u * (warp_id * 8 + g + 1));
    float acc = 0.f;
    const char* b = reinterpret_cast<const char*>(base) + li * kBytesPerLane;
    __syncthreads();
    long long c0 = clock64();
    unsigned long long t0 = global_ns();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
        float v[4][kBytesPerLane / 4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            x = lcg(x);
            const char* p = b + (size_t)((x >> 7) & row_mask) * 128;
            if constexpr (kBytesPerLane == 16) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(p));
                v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
            } else {
                asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=f"(v[u][0]), "=f"(v[u][1]), "=f"(v[u][2]), "=f"(v[u][3]),
                               "=f"(v[u][4]), "=f"(v[u][5]), "=f"(v[u][6]), "=f"(v[u][7])
                             : "l"(p));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int e = 0; e < kBytesPerLane / 4; ++e) acc += v[u][e];
    }
    __syncthreads();
    if (threadIdx.x == 0) stamps[blockIdx.x] = Stamp{c0, clock64(), t0, global_ns()};
    sink[blockIdx.x * kThreads + threadIdx.x] = acc;
}

__global__ void __launch_bounds__(kThreads) gather_lds(int iters, float* __restrict__ sink,
                                                       Stamp* __restrict__ stamps) {
    extern __shared__ float4 s_rows[];    // kSharedRows rows of 8 float4
    for (int i = threadIdx.x; i < kSharedRows * 8; i += kThreads)
        s_rows[i] = make_float4(i * 1e-9f, 0.f, 1e-9f, 0.f);
    const int lane = threadIdx.x & 31, g = lane >> 3, li = lane & 7;
    const int warp_id = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    uint32_t x = lcg(0x9e3779b9u * (warp_id * 8 + g + 1));
    float acc = 0.f;
    __syncthreads();
    long long c0 = clock64();
    unsigned long long t0 = global_ns();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            x = lcg(x);
            v[u] = s_rows[((x >> 7) & (kSharedRows - 1)) * 8 + li];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) acc += v[u].x + v[u].y + v[u].z + v[u].w;
    }
    __syncthreads();
    if (threadIdx.x == 0) stamps[blockIdx.x] = Stamp{c0, clock64(), t0, global_ns()};
    sink[blockIdx.x * kThreads + threadIdx.x] = acc;
}

// Shared-memory row scatter: per iteration each lane adds its 4 channels of
// one row (4 scalar instructions), the 4 lane groups of a warp into 4 rows.
// pattern 0: group g's rows live in bank class g (window base = g mod 4).
template <bool kAtomic>
__global__ void __launch_bounds__(kThreads) scatter_lds(int iters, int pattern,
                                                        float* __restrict__ sink,
                                                        Stamp* __restrict__ stamps) {
    extern __shared__ float s_win[];      // 4 classes x (kSubRows x 32 + 4) floats
    constexpr int kClass = kSubRows * 32 + 4;
    for (int i = threadIdx.x; i < 4 * kClass; i += kThreads) s_win[i] = 0.f;
    const int lane = threadIdx.x & 31, g = lane >> 3, li = lane & 7;
    const int warp_id = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    uint32_t x = lcg(0x9e3779b9u * (warp_id * 8 + g + 1));
    const float val = 1e-7f;
    __syncthreads();
    long long c0 = clock64();
    unsigned long long t0 = global_ns();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            x = lcg(x);
            const uint32_t r = (x >> 7) & (kSubRows - 1);
            int off;
            if (pattern == 0) off = g * kClass + g + r * 32 + li * 4;        // residue g
            else if (pattern == 1) off = g * kClass + r * 32 + li * 4;       // one residue
            else off = (int)((x >> 7) & (4 * kSubRows - 1)) * 33 % (4 * kClass - 32) + li * 4;
            float* p = s_win + off;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (kAtomic)
                    asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(smem_addr(p + e)), "f"(val)
                                 : "memory");
                else
                    p[e] += val;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) stamps[blockIdx.x] = Stamp{c0, clock64(), t0, global_ns()};
    sink[blockIdx.x * kThreads + threadIdx.x] = s_win[threadIdx.x];
}

__global__ void __launch_bounds__(kThreads) scatter_red_global(float* __restrict__ base,
                                                               uint32_t row_mask, int iters,
                                                               Stamp* __restrict__ stamps) {
    const int lane = threadIdx.x & 31, g = lane >> 3, li = lane & 7;
    const int warp_id = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    uint32_t x = lcg(0x9e3779b9u * (warp_id * 8 + g + 1));
    char* b = reinterpret_cast<char*>(base) + li * 16;
    const float val = 1e-7f;
    __syncthreads();
    long long c0 = clock64();
    unsigned long long t0 = global_ns();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            x = lcg(x);
            float* p = reinterpret_cast<float*>(b + (size_t)((x >> 7) & row_mask) * 128);
            asm volatile("red.global.add.v4.f32 [%0], {%1, %1, %1, %1};" ::"l"(p), "f"(val)
                         : "memory");
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) stamps[blockIdx.x] = Stamp{c0, clock64(), t0, global_ns()};
}

// kGatherTma4: warps 0..7 produce (lane 0 issues the copies of its ring), warps
// 8..15 consume.  Every wait is bounded; a wait that runs out sets `err`.
constexpr int kTmaPairs = 8, kTmaSlots = 8;
__device__ unsigned g_tma_err;

__device__ __forceinline__ bool tma_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < (1 << 22); ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    atomicOr(&g_tma_err, 1u);
    return false;
}

__global__ void __launch_bounds__(kThreads) gather_tma4(const __grid_constant__ CUtensorMap map,
                                                        uint32_t row_mask, int iters,
                                                        float* __restrict__ sink,
                                                        Stamp* __restrict__ stamps) {
    __shared__ __align__(1024) float ring[kTmaPairs][kTmaSlots][128];
    __shared__ __align__(8) unsigned long long full[kTmaPairs][kTmaSlots];
    __shared__ __align__(8) unsigned long long empty[kTmaPairs][kTmaSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = warp % kTmaPairs;
    if (threadIdx.x == 0) {
        for (int p = 0; p < kTmaPairs; ++p)
            for (int s = 0; s < kTmaSlots; ++s) {
                asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[p][s])));
                asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&empty[p][s])));
            }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    long long c0 = clock64();
    unsigned long long t0 = global_ns();
    float acc = 0.f;
    if (warp < kTmaPairs) {
        if (lane == 0) {
            uint32_t x = lcg(blockIdx.x * 977u + (uint32_t)pair * 131u + 1u);
            int it = 0;
            for (; it < iters; ++it) {
                const int s = it % kTmaSlots;
                if (!tma_wait(smem_addr(&empty[pair][s]), ((it / kTmaSlots) & 1) ^ 1)) break;
                const uint32_t fb = smem_addr(&full[pair][s]);
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                             "r"(512)
                             : "memory");
                int r[4];
                for (int k = 0; k < 4; ++k) {
                    x = lcg(x);
                    r[k] = (int)((x >> 7) & row_mask);
                }
                asm volatile(
                    "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::"
                    "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(
                        smem_addr(ring[pair][s])),
                    "l"(reinterpret_cast<uint64_t>(&map)), "r"(0), "r"(r[0]), "r"(r[1]), "r"(r[2]),
                    "r"(r[3]), "r"(fb)
                    : "memory");
            }
            // wait for the copies still in flight before the CTA may leave
            for (int j = it > kTmaSlots ? it - kTmaSlots : 0; j < it; ++j)
                tma_wait(smem_addr(&full[pair][j % kTmaSlots]), (j / kTmaSlots) & 1);
        }
    } else {
        for (int it = 0; it < iters; ++it) {
            const int s = it % kTmaSlots;
            if (!tma_wait(smem_addr(&full[pair][s]), (it / kTmaSlots) & 1)) break;
            const float4 v = reinterpret_cast<const float4*>(ring[pair][s])[lane];
            acc += v.x + v.y + v.z + v.w;
            __syncwarp();
            if (lane == 0)
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                                 smem_addr(&empty[pair][s]))
                             : "memory");
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        stamps[0].clk0 = c0;
        stamps[0].clk1 = clock64();
        stamps[0].ns0 = t0;
        stamps[0].ns1 = global_ns();
    }
    sink[blockIdx.x * kThreads + threadIdx.x] = acc;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A [rows, 32] fp32 map with a one-row box (the gather4 form).
bool row_map(CUtensorMap* map, float* region, size_t rows) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    const cuuint64_t dims[2] = {32, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {32, 1};
    const cuuint32_t estr[2] = {1, 1};
    return reinterpret_cast<EncodeTiled>(fn)(
               map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, region, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__global__ void fill_kernel(float* p, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = (float)(i & 1023) * 1e-6f;
}

}  // namespace

// Runs probe `probe` with `param` (see above) on `ctas_per_sm` CTAs of 16
// warps per SM, `iters` iterations of 4 rows per lane group.  out[0]: rows per
// SM clock (for the shared scatters: rows of 32 floats, i.e. 4 scalar
// instructions per lane per row); out[1]: kernel time in ms (CUDA events);
// out[2]: SM clock in MHz (clock64 over %globaltimer in CTA 0); out[3]: rows
// moved.  Returns 0, or the CUDA error code.
extern "C" __attribute__((visibility("default"))) int msda_ceiling_run(int probe, long long param,
                                                                       int ctas_per_sm, int iters,
                                                                       double* out) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = sms * ctas_per_sm;
    float* sink = nullptr;
    Stamp* stamps = nullptr;
    float* region = nullptr;
    const bool global_probe = probe == kGatherLdg16 || probe == kGatherLdg32 ||
                              probe == kRedGlobalV4 || probe == kGatherTma4;
    size_t region_bytes = global_probe ? (size_t)param : 0;
    if (region_bytes < 128 || (region_bytes & (region_bytes - 1)) != 0) region_bytes = 0;
    if (probe < kGatherLdg16 || probe > kGatherTma4 || iters < 1 || ctas_per_sm < 1 ||
        (global_probe && region_bytes == 0))
        return (int)cudaErrorInvalidValue;
    if ((e = cudaMalloc(&sink, (size_t)grid * kThreads * sizeof(float))) != cudaSuccess) return e;
    if ((e = cudaMalloc(&stamps, (size_t)grid * sizeof(Stamp))) != cudaSuccess) return e;
    if (region_bytes) {
        if ((e = cudaMalloc(&region, region_bytes)) != cudaSuccess) return e;
        fill_kernel<<<sms * 4, 256>>>(region, region_bytes / 4);
    }
    const uint32_t row_mask = region_bytes ? (uint32_t)(region_bytes / 128 - 1) : 0;
    CUtensorMap map;
    if (probe == kGatherTma4) {
        if (!row_map(&map, region, region_bytes / 128)) return (int)cudaErrorInvalidValue;
        const unsigned zero = 0;
        if ((e = cudaMemcpyToSymbol(g_tma_err, &zero, sizeof(zero))) != cudaSuccess) return e;
    }
    const size_t lds_bytes = (size_t)kSharedRows * 128;
    const size_t win_bytes = (size_t)4 * (kSubRows * 32 + 4) * sizeof(float);
    auto launch = [&]() {
        switch (probe) {
            case kGatherLdg16:
                gather_ldg<16><<<grid, kThreads>>>(region, row_mask, iters, sink, stamps);
                break;
            case kGatherLdg32:
                gather_ldg<32><<<grid, kThreads>>>(region, row_mask, iters, sink, stamps);
                break;
            case kGatherLds16:
                gather_lds<<<grid, kThreads, lds_bytes>>>(iters, sink, stamps);
                break;
            case kRedShared:
                scatter_lds<true><<<grid, kThreads, win_bytes>>>(iters, (int)param, sink, stamps);
                break;
            case kRmwShared:
                scatter_lds<false><<<grid, kThreads, win_bytes>>>(iters, (int)param, sink, stamps);
                break;
            case kRedGlobalV4:
                scatter_red_global<<<grid, kThreads>>>(region, row_mask, iters, stamps);
                break;
            case kGatherTma4:
                gather_tma4<<<grid, kThreads>>>(map, row_mask, iters, sink, stamps);
                break;
            default: break;
        }
    };
    if (probe == kGatherLds16)
        cudaFuncSetAttribute(gather_lds, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)lds_bytes);
    if (probe == kRedShared || probe == kRmwShared) {
        cudaFuncSetAttribute(scatter_lds<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)win_bytes);
        cudaFuncSetAttribute(scatter_lds<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)win_bytes);
    }
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    launch();                               // warm-up (fills L1 / L2)
    cudaEventRecord(a);
    launch();
    cudaEventRecord(b);
    e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaGetLastError();
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    Stamp s0{};
    if (e == cudaSuccess) e = cudaMemcpy(&s0, stamps, sizeof(Stamp), cudaMemcpyDeviceToHost);
    const int lanes_per_row = probe == kGatherLdg32 ? 4 : 8;
    const double rows = probe == kGatherTma4
                            ? (double)grid * kTmaPairs * 4.0 * iters
                            : (double)grid * kThreads / lanes_per_row * 4.0 * iters;
    if (e == cudaSuccess && probe == kGatherTma4) {
        unsigned err = 0;
        e = cudaMemcpyFromSymbol(&err, g_tma_err, sizeof(err));
        if (e == cudaSuccess && err != 0) e = cudaErrorLaunchTimeout;   // a bounded wait ran out
    }
    const double mhz = s0.ns1 > s0.ns0 ? (double)(s0.clk1 - s0.clk0) / (double)(s0.ns1 - s0.ns0) * 1e3
                                       : 0.0;
    out[0] = (ms > 0 && mhz > 0) ? rows / ((double)ms * 1e-3 * mhz * 1e6 * sms) : 0.0;
    out[1] = ms;
    out[2] = mhz;
    out[3] = rows;
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaFree(sink);
    cudaFree(stamps);
    if (region) cudaFree(region);
    return (int)e;
}
