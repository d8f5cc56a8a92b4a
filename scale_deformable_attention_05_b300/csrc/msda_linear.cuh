// Linear projection y = x * w^T + bias on the fifth-generation tensor cores
// (tcgen05), bf16 operands with fp32 accumulation, for the projections around
// the operator in MSDeformAttn.forward (Deformable DETR walk-through, "2.2.4
// 源码分析": value_proj, sampling_offsets, attention_weights and output_proj
// are nn.Linear layers of input width d_model).
//
//   x    [rows, K]  bf16, row-major (K contiguous)
//   w    [N, K]     bf16, the nn.Linear weight layout (K contiguous)
//   bias [N]        fp32 or NULL
//   y    [rows, N]  bf16, y[r, n] = sum_k x[r, k] w[n, k] + bias[n], rounded once
//
// Design (one persistent CTA of 6 warps per SM over 128-row tiles):
//   * w stays in shared memory for the whole launch (N x K bf16 <= 128 KB),
//     loaded once with TMA in 128-byte-swizzled 64-column blocks;
//   * warp 0 streams the 128 x 64 blocks of x through a ring of kStages
//     shared-memory stages with TMA (same swizzled layout);
//   * warp 1 issues, per block, four tcgen05.mma (M = 128, N, K = 16, both
//     operands K-major) into one of two fp32 accumulators of 256 columns in
//     tensor memory, frees the block's stage with tcgen05.commit, and hands a
//     finished accumulator to the epilogue with another commit;
//   * warps 2..9 (two per tensor-memory lane quarter, each taking every other
//     32-column piece) read the accumulator with tcgen05.ld, add the bias (kept
//     in shared memory), round to bf16, stage 32 x 32 pieces in shared memory
//     and write them with TMA stores (which clip the ragged last tile), then
//     free the accumulator for the tile after next.
// So loads, MMAs and the epilogue of consecutive tiles overlap.  Every wait on
// an mbarrier has an iteration limit; when it runs out the thread records
// kErrTimeout in the device error word and stops, and the CTA frees its
// tensor memory and returns.  Compiled as part of msda_kernels.cu (it shares
// the error word).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "../../include/msda.h"
#include "msda_device.cuh"

namespace msda {
namespace linear {

constexpr int kBM = 128;                 // rows per tile (the MMA's M)
constexpr int kBK = 64;                  // bf16 columns per 128-byte swizzle atom
constexpr int kStages = 4;               // x blocks in flight
constexpr int kEpiWarps = 8;             // warps 2..9, two per tensor-memory lane quarter
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kAccCols = 256;            // tensor-memory columns per accumulator
constexpr int kChunk = 32;               // output columns per staged piece
constexpr unsigned kErrTimeout = 4u;     // bit of the device error word (an mbarrier wait ran out)
constexpr int kSpinLimit = 1 << 22;      // try_wait rounds before giving up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for the phase with parity `parity` of the mbarrier to complete
// (a fresh barrier counts its phase of parity 1 as complete).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    atomicOr(&msda::g_error_word, kErrTimeout);
    return false;
}

// Before a CTA leaves, its producer waits (bounded) for the TMA loads it issued
// into the last `depth` stages of a ring (issues it - depth .. it - 1; stage s's
// full barrier at full0 + 8 s), so that no copy lands in shared memory after the
// CTA has gone, also when another role gave up on a wait.  After a normal run
// every such phase has completed and each wait returns at once.
__device__ __forceinline__ void drain_loads(uint32_t full0, uint32_t it, int depth) {
    for (uint32_t j = it > (uint32_t)depth ? it - (uint32_t)depth : 0u; j < it; ++j)
        mbar_wait(full0 + 8u * (j % (uint32_t)depth), (j / (uint32_t)depth) & 1u);
}

// The MMA issuer's last step: a commit tracking every tcgen05.mma it issued,
// waited on (bounded), so that tensor memory is freed only after they finish.
__device__ __forceinline__ void drain_mmas(uint32_t bar);

// 2-d TMA tile load into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 2-d TMA tile store from shared memory (elements past the tensor are not written).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1,
                                             uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(src)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand stored as 128-byte rows
// with the 128-byte swizzle (what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B):
// start address, stride of 1024 bytes between 8-row groups, version 1, layout
// SWIZZLE_128B.  The leading-dimension offset is unused for this layout (the
// MMA's 16 columns never leave one 128-byte atom).
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);          // start address (16-byte units)
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused): 16 B
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: 1024 B
    d |= (uint64_t)1 << 46;                          // descriptor version
    d |= (uint64_t)2 << 61;                          // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with bf16 (or, with f16, fp16) A and B,
// fp32 D, both K-major, M = 128 and N = n.
__host__ __device__ constexpr uint32_t bf16_idesc(int n, bool f16 = false) {
    return (1u << 4)                         // D format: f32
           | ((f16 ? 0u : 1u) << 7)          // A format: bf16 (1) or f16 (0)
           | ((f16 ? 0u : 1u) << 10)         // B format: the same type as A
           | ((uint32_t)(n >> 3) << 17)      // N / 8
           | ((uint32_t)(kBM >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void drain_mmas(uint32_t bar) {
    umma_commit(bar);
    mbar_wait(bar, 0);
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory layout of one CTA (byte offsets from a 1024-aligned base).
struct Smem {
    uint32_t w, x, stage_out, bias, bars, tmem_slot, total;
};
__host__ __device__ inline Smem smem_layout(int n, int k) {
    Smem s;
    s.w = 0;                                                 // K/64 blocks of n rows x 128 B
    s.x = s.w + (uint32_t)n * (uint32_t)k * 2;               // kStages blocks of 128 x 128 B
    s.stage_out = s.x + (uint32_t)kStages * kBM * 128;       // 2 x 32 x 32 bf16 per epilogue warp
    s.bias = s.stage_out + (uint32_t)kEpiWarps * 2 * kChunk * kChunk * 2;   // 256 fp32
    s.bars = s.bias + MSDA_LINEAR_MAX_FEATURES * 4;
    s.tmem_slot = s.bars + (1 + 2 * kStages + 4 + 1) * 8;
    s.total = s.tmem_slot + 8;
    return s;
}

// Two fp32 values rounded to nearest even in T and packed low, high.
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// The 16-bit kernels' body; T is __nv_bfloat16 or __half (both operands, the
// output, and the bias when bias_half).
template <typename T>
__device__ __forceinline__ void linear16_body(const CUtensorMap& x_map, const CUtensorMap& w_map,
                                              const CUtensorMap& y_map,
                                              const void* __restrict__ bias, int bias_half,
                                              int rows, int n, int k) {
    constexpr bool kF16 = std::is_same<T, __half>::value;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // TMA destinations with the 128-byte swizzle must sit on 1024-byte boundaries
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Smem L = smem_layout(n, k);
    const uint32_t s_w = smem_u32(base + L.w), s_x = smem_u32(base + L.x);
    const uint32_t bars = smem_u32(base + L.bars);
    const uint32_t w_full = bars;
    auto x_full = [&](int s) { return bars + 8u * (1 + s); };
    auto x_empty = [&](int s) { return bars + 8u * (1 + kStages + s); };
    auto acc_full = [&](int a) { return bars + 8u * (1 + 2 * kStages + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (3 + 2 * kStages + a); };
    const uint32_t mma_done = bars + 8u * (5 + 2 * kStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.tmem_slot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kblocks = k / kBK;
    const int tiles = (rows + kBM - 1) / kBM;

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(2 * kAccCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        mbar_init(w_full, 1);
        mbar_init(mma_done, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(x_full(s), 1);
            mbar_init(x_empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), kEpiWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---- producer: w once, then the x blocks of every tile through the ring
        if (lane == 0) {
            mbar_expect_tx(w_full, (uint32_t)n * (uint32_t)k * 2);
            for (int kb = 0; kb < kblocks; ++kb)
                tma_load_2d(s_w + (uint32_t)kb * (uint32_t)n * 128, &w_map, kb * kBK, 0, w_full);
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x)
                for (int kb = 0; kb < kblocks && ok; ++kb, ++it) {
                    const int s = (int)(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    ok = mbar_wait(x_empty(s), ph ^ 1u);
                    if (!ok) break;
                    mbar_expect_tx(x_full(s), (uint32_t)kBM * 128);
                    tma_load_2d(s_x + (uint32_t)s * kBM * 128, &x_map, kb * kBK, t * kBM,
                                x_full(s));
                }
            mbar_wait(w_full, 0);
            drain_loads(x_full(0), it, kStages);
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = bf16_idesc(n, kF16);
            bool ok = mbar_wait(w_full, 0);
            uint32_t it = 0, acc_it = 0;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++acc_it) {
                const int a = (int)(acc_it & 1u);
                const uint32_t aph = (acc_it >> 1) & 1u;
                ok = mbar_wait(acc_empty(a), aph ^ 1u);
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(a * kAccCols);
                for (int kb = 0; kb < kblocks && ok; ++kb, ++it) {
                    const int s = (int)(it % kStages);
                    const uint32_t ph = (it / kStages) & 1u;
                    ok = mbar_wait(x_full(s), ph);
                    if (!ok) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks) {
                        const uint32_t koff = (uint32_t)ks * 32;   // 16 bf16 columns
                        umma_bf16(d, kmajor_sw128_desc(s_x + (uint32_t)s * kBM * 128 + koff),
                                  kmajor_sw128_desc(s_w + (uint32_t)kb * (uint32_t)n * 128 + koff),
                                  idesc, kb > 0 || ks > 0);
                    }
                    umma_commit(x_empty(s));     // the stage is free once these MMAs finish
                }
                if (ok) umma_commit(acc_full(a));
            }
            drain_mmas(mma_done);
        }
    } else {
        // ---- epilogue: warp w (2..9) reads lanes 32 * (w % 4) .. + 31 of the
        //      accumulator, the 32-column pieces c0 = 32 * half, 32 * half + 64, ...
        const int quarter = warp & 3;
        const int ew = warp - 2;
        const int half = ew >> 2;
        float* s_bias = reinterpret_cast<float*>(base + L.bias);
        // the bias, zero past n, in shared memory (the epilogue warps' own copy)
        for (int c = ew * 32 + lane; c < MSDA_LINEAR_MAX_FEATURES; c += kEpiWarps * 32) {
            float bv = 0.f;
            if (bias != nullptr && c < n)
                bv = bias_half ? (float)static_cast<const T*>(bias)[c]
                               : static_cast<const float*>(bias)[c];
            s_bias[c] = bv;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        const uint32_t stage_base =
            smem_u32(base + L.stage_out) + (uint32_t)ew * 2 * kChunk * kChunk * 2;
        unsigned char* stage_ptr = base + L.stage_out + (size_t)ew * 2 * kChunk * kChunk * 2;
        uint32_t acc_it = 0, piece = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++acc_it) {
            const int a = (int)(acc_it & 1u);
            ok = mbar_wait(acc_full(a), (acc_it >> 1) & 1u);
            if (!ok) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t taddr =
                tmem + (uint32_t)(a * kAccCols) + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = half * kChunk; c0 < n; c0 += 2 * kChunk, ++piece) {
                float v[32];
                tmem_ld32(taddr + (uint32_t)c0, v);
                const float4* bq = reinterpret_cast<const float4*>(s_bias + c0);
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 bb = bq[i];
                    o[2 * i] = pack2<T>(v[4 * i] + bb.x, v[4 * i + 1] + bb.y);
                    o[2 * i + 1] = pack2<T>(v[4 * i + 2] + bb.z, v[4 * i + 3] + bb.w);
                }
                // the staging buffer of this piece must have been read by its previous store
                const int buf = (int)(piece & 1u);
                if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                __syncwarp();
                uint4* dst = reinterpret_cast<uint4*>(stage_ptr + (size_t)buf * kChunk * kChunk * 2 +
                                                      (size_t)lane * kChunk * 2);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    tma_store_2d(&y_map, c0, t * kBM + quarter * 32,
                                 stage_base + (uint32_t)buf * kChunk * kChunk * 2);
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(a));   // accumulator free for tile + 2
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(2 * kAccCols)
                     : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    linear_bf16_kernel(const __grid_constant__ CUtensorMap x_map,
                       const __grid_constant__ CUtensorMap w_map,
                       const __grid_constant__ CUtensorMap y_map, const void* __restrict__ bias,
                       int bias_half, int rows, int n, int k) {
    linear16_body<__nv_bfloat16>(x_map, w_map, y_map, bias, bias_half, rows, n, k);
}

__global__ void __launch_bounds__(kThreads, 1)
    linear_f16_kernel(const __grid_constant__ CUtensorMap x_map,
                      const __grid_constant__ CUtensorMap w_map,
                      const __grid_constant__ CUtensorMap y_map, const void* __restrict__ bias,
                      int bias_half, int rows, int n, int k) {
    linear16_body<__half>(x_map, w_map, y_map, bias, bias_half, rows, n, k);
}

// ---------------------------------------------------------- fp32 (3 x TF32)
// fp32 projections keep fp32 accuracy on the tensor cores by splitting each
// operand into its TF32 rounding and the fp32 remainder, a = a_hi + a_lo with
// a_hi = a rounded to nearest TF32 (10 explicit mantissa bits) and a_lo = a -
// a_hi exact, and summing three TF32 products, x_hi w_hi + x_hi w_lo + x_lo
// w_hi, in the fp32 accumulator (the dropped x_lo w_lo and the TF32 reading of
// the remainders are below 2^-19 of |x||w|).
//   * w is split once per call by a small kernel into the caller's workspace;
//   * the work is cut into units of 128 rows x up to 256 output columns (a
//     row tile and one column part);
//   * warp 0 loads, per stage, one raw 128 x 16 fp32 block of x and the split
//     16-column blocks of the unit's w rows (w_hi, w_lo) with TMA (64-byte
//     swizzle; small stages keep four of them in flight, which the loads'
//     latency needs); the parts of a row tile run on neighbouring CTAs at the
//     same time, so later reads of the x block come from L2;
//   * warps 10..13 split the x block in shared memory: x_hi over the raw
//     block in place and x_lo into the stage's second buffer, at the same
//     offsets (the split is elementwise, so the swizzled layout carries over);
//   * warp 1 issues, per K step of 8, the three kind::tf32 MMAs into one of
//     two fp32 accumulators in tensor memory;
//   * warps 2..9 drain a finished accumulator as in the bf16 kernel, adding
//     the bias and writing fp32 32 x 32 pieces with TMA stores.
constexpr int kBKF = 16;                 // fp32 columns per stage: 64-byte rows, 64-byte swizzle
constexpr int kStagesF = 4;
constexpr int kPartF = 256;              // output columns per unit (the MMA's N, at most)
constexpr uint32_t kRowF = kBKF * 4;     // bytes per operand row in a stage
constexpr int kConvWarps = 4;            // warps 10..13: one 32-row quarter of the x block each
constexpr int kThreadsF = 32 * (2 + kEpiWarps + kConvWarps);

__global__ void split_tf32_kernel(const float4* __restrict__ a, float4* __restrict__ hi,
                                  float4* __restrict__ lo, size_t n4) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = a[i];
        float h[4];
        const float in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t t;
            asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(in[j]));
            h[j] = __uint_as_float(t);
        }
        hi[i] = make_float4(h[0], h[1], h[2], h[3]);
        lo[i] = make_float4(in[0] - h[0], in[1] - h[1], in[2] - h[2], in[3] - h[3]);
    }
}

// Shared-memory matrix descriptor of a K-major operand stored as 64-byte rows
// with the 64-byte swizzle (CU_TENSOR_MAP_SWIZZLE_64B): 8-row groups 512 bytes
// apart, version 1, layout SWIZZLE_64B; the MMA's 8 TF32 columns (32 bytes)
// never leave one 64-byte row.
__device__ __forceinline__ uint64_t kmajor_sw64_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);          // start address (16-byte units)
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused): 16 B
    d |= (uint64_t)(512 >> 4) << 32;                 // stride byte offset: 512 B
    d |= (uint64_t)1 << 46;                          // descriptor version
    d |= (uint64_t)4 << 61;                          // layout: 64-byte swizzle
    return d;
}

// Instruction descriptor of kind::tf32 (TF32 A and B, fp32 D, both K-major), M = 128, N = n.
__host__ __device__ constexpr uint32_t tf32_idesc(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

struct SmemF {
    uint32_t stage_bytes, stages, stage_out, bias, bars, tmem_slot, total;
};
__host__ __device__ inline SmemF smem_layout_f() {
    SmemF s;
    s.stage_bytes = 2u * kBM * kRowF + 2u * kPartF * kRowF;    // x (-> x_hi), x_lo, w_hi, w_lo
    s.stages = 0;
    s.stage_out = s.stages + kStagesF * s.stage_bytes;         // 32 x 32 fp32 per epilogue warp
    s.bias = s.stage_out + (uint32_t)kEpiWarps * kChunk * kChunk * 4;
    s.bars = s.bias + MSDA_LINEAR_MAX_FEATURES * 4;
    s.tmem_slot = s.bars + (3 * kStagesF + 4 + 1) * 8;
    s.total = s.tmem_slot + 8;
    return s;
}

__global__ void __launch_bounds__(kThreadsF, 1)
    linear_f32x3_kernel(const __grid_constant__ CUtensorMap x_map,
                        const __grid_constant__ CUtensorMap whi_map,
                        const __grid_constant__ CUtensorMap wlo_map,
                        const __grid_constant__ CUtensorMap y_map, const float* __restrict__ bias,
                        int rows, int n, int k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemF L = smem_layout_f();
    const uint32_t s_stage = smem_u32(base + L.stages);
    auto xhi = [&](int s) { return s_stage + (uint32_t)s * L.stage_bytes; };
    auto xlo = [&](int s) { return xhi(s) + (uint32_t)kBM * kRowF; };
    auto whi = [&](int s) { return xhi(s) + 2u * kBM * kRowF; };
    auto wlo = [&](int s) { return whi(s) + (uint32_t)kPartF * kRowF; };
    const uint32_t bars = smem_u32(base + L.bars);
    auto x_full = [&](int s) { return bars + 8u * s; };                   // TMA landed
    auto x_split = [&](int s) { return bars + 8u * (kStagesF + s); };     // x split in place
    auto x_empty = [&](int s) { return bars + 8u * (2 * kStagesF + s); }; // MMAs done with it
    auto acc_full = [&](int a) { return bars + 8u * (3 * kStagesF + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (3 * kStagesF + 2 + a); };
    const uint32_t mma_done = bars + 8u * (3 * kStagesF + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.tmem_slot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kblocks = k / kBKF;
    const int parts = (n + kPartF - 1) / kPartF;
    const int units = (rows + kBM - 1) / kBM * parts;   // unit u: row tile u / parts, part u % parts

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(2 * kPartF)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        mbar_init(mma_done, 1);
        for (int s = 0; s < kStagesF; ++s) {
            mbar_init(x_full(s), 1);
            mbar_init(x_split(s), kConvWarps);
            mbar_init(x_empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), kEpiWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---- producer: the raw x block and both parts of the unit's w block per stage
        //      (the w box is min(n, kPartF) rows; rows past n read as zero and count in full)
        if (lane == 0) {
            const uint32_t wrows = (uint32_t)min(n, kPartF);     // the w box's rows
            const uint32_t bytes = (uint32_t)kBM * kRowF + 2u * wrows * kRowF;
            uint32_t it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const int t = u / parts, part = u - t * parts;
                for (int kb = 0; kb < kblocks && ok; ++kb, ++it) {
                    const int s = (int)(it % kStagesF);
                    ok = mbar_wait(x_empty(s), ((it / kStagesF) & 1u) ^ 1u);
                    if (!ok) break;
                    mbar_expect_tx(x_full(s), bytes);
                    tma_load_2d(xhi(s), &x_map, kb * kBKF, t * kBM, x_full(s));
                    tma_load_2d(whi(s), &whi_map, kb * kBKF, part * kPartF, x_full(s));
                    tma_load_2d(wlo(s), &wlo_map, kb * kBKF, part * kPartF, x_full(s));
                }
            }
            drain_loads(x_full(0), it, kStagesF);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: three TF32 products per K step of 8
        if (lane == 0) {
            bool ok = true;
            uint32_t it = 0, acc_it = 0;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++acc_it) {
                const int part = u % parts;
                const int cols = min(kPartF, n - part * kPartF);
                const uint32_t idesc = tf32_idesc(cols);
                const int a = (int)(acc_it & 1u);
                ok = mbar_wait(acc_empty(a), ((acc_it >> 1) & 1u) ^ 1u);
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(a * kPartF);
                for (int kb = 0; kb < kblocks && ok; ++kb, ++it) {
                    const int s = (int)(it % kStagesF);
                    const uint32_t ph = (it / kStagesF) & 1u;
                    ok = mbar_wait(x_full(s), ph) && mbar_wait(x_split(s), ph);
                    if (!ok) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                    for (int ks = 0; ks < kBKF / 8; ++ks) {
                        const uint32_t koff = (uint32_t)ks * 32;   // 8 fp32 columns
                        const uint64_t ah = kmajor_sw64_desc(xhi(s) + koff);
                        const uint64_t al = kmajor_sw64_desc(xlo(s) + koff);
                        const uint64_t bh = kmajor_sw64_desc(whi(s) + koff);
                        const uint64_t bl = kmajor_sw64_desc(wlo(s) + koff);
                        umma_tf32(d, ah, bh, idesc, kb > 0 || ks > 0);
                        umma_tf32(d, ah, bl, idesc, true);
                        umma_tf32(d, al, bh, idesc, true);
                    }
                    umma_commit(x_empty(s));
                }
                if (ok) umma_commit(acc_full(a));
            }
            drain_mmas(mma_done);
        }
    } else if (warp >= 2 + kEpiWarps) {
        // ---- x split: converter warp c takes rows 32c .. 32c+31 of the block (2 KB),
        //      four 16-byte chunks per lane, consecutive lanes on consecutive chunks
        const int c = warp - 2 - kEpiWarps;
        unsigned char* stage0 = base + L.stages;
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x)
            for (int kb = 0; kb < kblocks && ok; ++kb, ++it) {
                const int s = (int)(it % kStagesF);
                ok = mbar_wait(x_full(s), (it / kStagesF) & 1u);
                if (!ok) break;
                float4* hi = reinterpret_cast<float4*>(stage0 + (size_t)s * L.stage_bytes +
                                                       (size_t)c * 32 * kRowF);
                float4* lo = reinterpret_cast<float4*>(reinterpret_cast<unsigned char*>(hi) +
                                                       kBM * kRowF);
#pragma unroll
                for (int i = 0; i < (int)(32 * kRowF / 16 / 32); ++i) {
                    const int j = i * 32 + lane;
                    const float4 v = hi[j];
                    const float in[4] = {v.x, v.y, v.z, v.w};
                    float h[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t r;
                        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(in[e]));
                        h[e] = __uint_as_float(r);
                    }
                    hi[j] = make_float4(h[0], h[1], h[2], h[3]);
                    lo[j] = make_float4(in[0] - h[0], in[1] - h[1], in[2] - h[2], in[3] - h[3]);
                }
                // the tensor cores read these buffers through the async proxy
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(x_split(s));
            }
    } else {
        // ---- epilogue: warps 2..9 as in the bf16 kernel; fp32 pieces staged with the
        //      128-byte swizzle (chunk j of row r at j ^ (r % 8)) that the store map reads
        const int quarter = warp & 3;
        const int ew = warp - 2;
        const int half = ew >> 2;
        float* s_bias = reinterpret_cast<float*>(base + L.bias);
        for (int c = ew * 32 + lane; c < MSDA_LINEAR_MAX_FEATURES; c += kEpiWarps * 32)
            s_bias[c] = bias != nullptr && c < n ? bias[c] : 0.f;
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        const uint32_t stage_addr =
            smem_u32(base + L.stage_out) + (uint32_t)ew * kChunk * kChunk * 4;
        unsigned char* row = base + L.stage_out + (size_t)ew * kChunk * kChunk * 4 +
                             (size_t)lane * 128;
        uint32_t acc_it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++acc_it) {
            const int t = u / parts, part = u - t * parts;
            const int col0 = part * kPartF, cols = min(kPartF, n - col0);
            const int a = (int)(acc_it & 1u);
            ok = mbar_wait(acc_full(a), (acc_it >> 1) & 1u);
            if (!ok) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t taddr =
                tmem + (uint32_t)(a * kPartF) + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = half * kChunk; c0 < cols; c0 += 2 * kChunk) {
                float v[32];
                tmem_ld32(taddr + (uint32_t)c0, v);
                const float4* bq = reinterpret_cast<const float4*>(s_bias + col0 + c0);
                // the staging buffer must have been read by this warp's previous store
                if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 bb = bq[j];
                    *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
                        make_float4(v[4 * j] + bb.x, v[4 * j + 1] + bb.y, v[4 * j + 2] + bb.z,
                                    v[4 * j + 3] + bb.w);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    tma_store_2d(&y_map, col0 + c0, t * kBM + quarter * 32, stage_addr);
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(a));
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(2 * kPartF)
                     : "memory");
}

// ------------------------------------------------ fp32 weight gradient (3 x TF32)
// The projections' parameter gradients, gw = gy^T x ([n, k], a sum over all
// rows) and gb = sum over rows of gy ([n]), in fp32 on the tensor cores with the
// same three-TF32-product split.  As an MMA, D[m, j] = sum_r A[m, r] B[j, r]
// with A = gy^T and B = x^T, whose rows are strided in memory; the kernel
// loads row-major blocks of gy and x and transposes them while it splits them:
//   * each CTA owns one 128-column tile of gy (m0 = 128 * tile) and one
//     contiguous range of rows, so its whole contribution accumulates in one
//     [128, k] fp32 accumulator in tensor memory;
//   * warp 0 loads 16-row blocks of gy (128 columns) and x (k columns) with
//     TMA into a ring of raw stages;
//   * warps 2..9 (thread t owns column t of x, and column m0 + t % 128 of gy
//     for rows 8 * (t / 128) .. + 7 of each block) read 4 rows at a time, add
//     gy's values to a running bias sum, split them into TF32 head and
//     remainder, and write both as K-major rows of 16 elements with the
//     64-byte swizzle (16-byte chunk c of row i at c ^ ((i >> 1) & 3) within
//     its 512-byte group) into a ring of split stages;
//   * warp 1 issues the three kind::tf32 MMAs per 8 rows;
//   * at the end warps 2..9 read the accumulator (two warps per lane quarter,
//     alternate 32-column pieces) and add it to gw with red.global.add.v4.f32,
//     and their bias sums to gb with atomicAdd.
// Rows past the matrices read as zero (TMA fill), so ragged ranges need no
// special case.  gw and gb must hold zeros (or the sums to add to) on entry.
constexpr int kWgRows = 16;              // rows (the MMA's K) per stage
constexpr int kWgRaw = 5, kWgSplit = 2;  // raw ring deep enough to cover HBM latency
constexpr int kWgConvWarps = 8;
constexpr int kWgThreads = 32 * (2 + kWgConvWarps);

struct SmemWg {
    uint32_t raw_bytes, split_bytes, raw, split, bars, tmem_slot, total;
};
__host__ __device__ inline SmemWg smem_layout_wg() {
    SmemWg s;
    s.raw_bytes = kWgRows * (kBM + MSDA_LINEAR_MAX_FEATURES) * 4;          // gy block, x block
    s.split_bytes = 2u * kBM * kWgRows * 4 + 2u * MSDA_LINEAR_MAX_FEATURES * kWgRows * 4;
    s.split = 0;                                                         // A_hi, A_lo, B_hi, B_lo
    s.raw = s.split + kWgSplit * s.split_bytes;
    s.bars = s.raw + kWgRaw * s.raw_bytes;
    s.tmem_slot = s.bars + (2 * kWgRaw + 2 * kWgSplit + 2) * 8;
    s.total = s.tmem_slot + 8;
    return s;
}

// Byte offset of element (row i, column r) of a K-major operand with 16-element
// rows and the 64-byte swizzle, r a multiple of 4 (one 16-byte chunk).
__device__ __forceinline__ uint32_t sw64_offset(int i, int r) {
    return (uint32_t)(i >> 3) * 512u + (uint32_t)(i & 7) * 64u +
           ((uint32_t)((r >> 2) ^ ((i >> 1) & 3)) << 4);
}

__device__ __forceinline__ void split4(const float (&v)[4], float4& hi, float4& lo) {
    float h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        uint32_t r;
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v[e]));
        h[e] = __uint_as_float(r);
    }
    hi = make_float4(h[0], h[1], h[2], h[3]);
    lo = make_float4(v[0] - h[0], v[1] - h[1], v[2] - h[2], v[3] - h[3]);
}

__global__ void __launch_bounds__(kWgThreads, 1)
    linear_wgrad_f32_kernel(const __grid_constant__ CUtensorMap gy_map,
                            const __grid_constant__ CUtensorMap x_map, float* __restrict__ gw,
                            float* __restrict__ gb, int rows, int n, int k, int tiles_m,
                            int rows_per_cta) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemWg L = smem_layout_wg();
    const uint32_t bars = smem_u32(base + L.bars);
    auto raw_full = [&](int s) { return bars + 8u * s; };
    auto raw_empty = [&](int s) { return bars + 8u * (kWgRaw + s); };
    auto split_full = [&](int s) { return bars + 8u * (2 * kWgRaw + s); };
    auto split_empty = [&](int s) { return bars + 8u * (2 * kWgRaw + kWgSplit + s); };
    const uint32_t acc_full = bars + 8u * (2 * kWgRaw + 2 * kWgSplit);
    const uint32_t mma_done = acc_full + 8u;
    auto raw_gy = [&](int s) { return base + L.raw + (size_t)s * L.raw_bytes; };
    auto raw_x = [&](int s) { return raw_gy(s) + (size_t)kWgRows * kBM * 4; };
    auto a_hi = [&](int s) { return base + L.split + (size_t)s * L.split_bytes; };
    auto a_lo = [&](int s) { return a_hi(s) + (size_t)kBM * kWgRows * 4; };
    auto b_hi = [&](int s) { return a_hi(s) + (size_t)2 * kBM * kWgRows * 4; };
    auto b_lo = [&](int s) {
        return b_hi(s) + (size_t)MSDA_LINEAR_MAX_FEATURES * kWgRows * 4;
    };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.tmem_slot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x % tiles_m;
    const int m0 = tile * kBM;
    const int r_begin = (blockIdx.x / tiles_m) * rows_per_cta;
    const int r_end = min(rows, r_begin + rows_per_cta);
    const int stages = r_end > r_begin ? (r_end - r_begin + kWgRows - 1) / kWgRows : 0;

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(MSDA_LINEAR_MAX_FEATURES)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kWgRaw; ++s) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), kWgConvWarps);
        }
        for (int s = 0; s < kWgSplit; ++s) {
            mbar_init(split_full(s), kWgConvWarps);
            mbar_init(split_empty(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(mma_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---- producer: 16-row blocks of gy (columns m0 .. m0+127) and of x
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)kWgRows * (kBM + k) * 4;
            uint32_t issued = 0;
            bool ok = true;
            for (int it = 0; it < stages && ok; ++it) {
                const int s = it % kWgRaw;
                ok = mbar_wait(raw_empty(s), ((it / kWgRaw) & 1) ^ 1);
                if (!ok) break;
                mbar_expect_tx(raw_full(s), bytes);
                const int r0 = r_begin + it * kWgRows;
                tma_load_2d(smem_u32(raw_gy(s)), &gy_map, m0, r0, raw_full(s));
                tma_load_2d(smem_u32(raw_x(s)), &x_map, 0, r0, raw_full(s));
                issued = (uint32_t)it + 1;
            }
            drain_loads(raw_full(0), issued, kWgRaw);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: D[m, j] += three TF32 products over 8 rows at a time
        if (lane == 0 && stages > 0) {
            const uint32_t idesc = tf32_idesc(k);
            bool ok = true;
            for (int it = 0; it < stages && ok; ++it) {
                const int s = it % kWgSplit;
                ok = mbar_wait(split_full(s), (it / kWgSplit) & 1);
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                for (int ks = 0; ks < kWgRows / 8; ++ks) {
                    const uint32_t koff = (uint32_t)ks * 32;   // 8 rows (fp32) per MMA
                    const uint64_t ah = kmajor_sw64_desc(smem_u32(a_hi(s)) + koff);
                    const uint64_t al = kmajor_sw64_desc(smem_u32(a_lo(s)) + koff);
                    const uint64_t bh = kmajor_sw64_desc(smem_u32(b_hi(s)) + koff);
                    const uint64_t bl = kmajor_sw64_desc(smem_u32(b_lo(s)) + koff);
                    umma_tf32(tmem, ah, bh, idesc, it > 0 || ks > 0);
                    umma_tf32(tmem, ah, bl, idesc, true);
                    umma_tf32(tmem, al, bh, idesc, true);
                }
                umma_commit(split_empty(s));
            }
            if (ok) umma_commit(acc_full);
            drain_mmas(mma_done);
        }
    } else {
        // ---- converters (warps 2..9), then the epilogue
        const int t = (warp - 2) * 32 + lane;          // x column t; gy column m0 + (t & 127)
        const int tg = t & (kBM - 1), q0 = (t >> 7) * 2;   // gy rows 4*q0 .. 4*q0 + 7
        float bias_sum = 0.f;
        bool ok = true;
        for (int it = 0; it < stages && ok; ++it) {
            const int sr = it % kWgRaw, ss = it % kWgSplit;
            ok = mbar_wait(raw_full(sr), (it / kWgRaw) & 1) &&
                 mbar_wait(split_empty(ss), ((it / kWgSplit) & 1) ^ 1);
            if (!ok) break;
            const float* gys = reinterpret_cast<const float*>(raw_gy(sr));
            const float* xs = reinterpret_cast<const float*>(raw_x(sr));
            float v[4];
            float4 hi, lo;
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int q = q0 + qq;
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = gys[(4 * q + e) * kBM + tg];
                bias_sum += (v[0] + v[1]) + (v[2] + v[3]);
                split4(v, hi, lo);
                const uint32_t off = sw64_offset(tg, 4 * q);
                *reinterpret_cast<float4*>(a_hi(ss) + off) = hi;
                *reinterpret_cast<float4*>(a_lo(ss) + off) = lo;
            }
            if (t < k) {
#pragma unroll
                for (int q = 0; q < kWgRows / 4; ++q) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = xs[(4 * q + e) * k + t];
                    split4(v, hi, lo);
                    const uint32_t off = sw64_offset(t, 4 * q);
                    *reinterpret_cast<float4*>(b_hi(ss) + off) = hi;
                    *reinterpret_cast<float4*>(b_lo(ss) + off) = lo;
                }
            }
            // the tensor cores read the split stage through the async proxy
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(split_full(ss));
                mbar_arrive(raw_empty(sr));
            }
        }
        if (ok && stages > 0) {
            if (gb != nullptr && m0 + tg < n) atomicAdd(gb + m0 + tg, bias_sum);
            ok = mbar_wait(acc_full, 0);
            if (ok) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const int quarter = warp & 3;   // the tensor-memory lanes this warp may read
                const int half = (warp - 2) >> 2;
                const int m = m0 + quarter * 32 + lane;
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
                for (int c0 = half * 32; c0 < k; c0 += 64) {
                    float v32[32];
                    tmem_ld32(taddr + (uint32_t)c0, v32);
                    if (m < n) {
                        float* dst = gw + (size_t)m * k + c0;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (c0 + 4 * j < k)
                                msda::red_add_v4(dst + 4 * j, v32[4 * j], v32[4 * j + 1],
                                                 v32[4 * j + 2], v32[4 * j + 3]);
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(MSDA_LINEAR_MAX_FEATURES)
                     : "memory");
}

// ------------------------------------------------------------ bias gradient
// Column sums of a projection's output gradient, grad_b[c] = sum_r grad_y[r, c],
// for the bf16 and fp16 layers (whose weight gradients run on the library GEMM):
// a streaming read of grad_y at HBM speed, fp32 sums.  Each CTA takes a
// contiguous range of rows; its threads hold one 16-byte vector of columns each
// for a set of rows, the CTA adds its rows up in shared memory and adds its
// column sums to grad_b with atomicAdd.
constexpr int kColThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kColThreads)
    column_sum_kernel(const T* __restrict__ gy, float* __restrict__ out, int rows, int n,
                      int rows_per_cta) {
    constexpr int V = IO<T>::kVec;
    __shared__ float s_part[kColThreads * V];
    const int vpr = n / V;                          // vectors per row (<= kColThreads)
    const int rpp = kColThreads / vpr;              // rows in parallel
    const int cv = threadIdx.x % vpr, rsub = threadIdx.x / vpr;
    const int r0 = blockIdx.x * rows_per_cta;
    const int r1 = min(rows, r0 + rows_per_cta);
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
    if (rsub < rpp) {
        const T* base = gy + (size_t)cv * V;
        int r = r0 + rsub;
        for (; r + 3 * rpp < r1; r += 4 * rpp) {   // four independent rows in flight
            float v[4][V];
#pragma unroll
            for (int u = 0; u < 4; ++u) IO<T>::load_vec_stream(base + (size_t)(r + u * rpp) * n, v[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < V; ++j) acc[j] += v[u][j];
        }
        for (; r < r1; r += rpp) {
            float v[V];
            IO<T>::load_vec_stream(base + (size_t)r * n, v);
#pragma unroll
            for (int j = 0; j < V; ++j) acc[j] += v[j];
        }
#pragma unroll
        for (int j = 0; j < V; ++j) s_part[rsub * n + cv * V + j] = acc[j];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < n; c += kColThreads) {
        float t = 0.f;
        for (int i = 0; i < rpp; ++i) t += s_part[i * n + c];
        atomicAdd(out + c, t);
    }
}

// ------------------------------------------------------------------- host
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
    static const EncodeTiled fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult found = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &found) != cudaSuccess ||
            found != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

// Row-major bf16 (or fp32, or fp16) matrix [outer, inner] moved in boxes of [box_rows, box_cols]
// (with the 128- or 64-byte swizzle, or none); elements past the matrix read as
// zero and are not written.
bool make_map(CUtensorMap* map, const void* ptr, int inner, int outer, int box_cols, int box_rows,
              int swizzle_bytes, bool fp32 = false, bool f16 = false) {
    const EncodeTiled enc = encode_tiled();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * (fp32 ? 4 : 2)};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType type = fp32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return enc(map, type, 2,
               const_cast<void*>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
               : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                     : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// A host action taken once per device (kernel attributes belong to the device's
// context): run() calls f the first time it is called with a given device current.
struct PerDevice {
    std::mutex m;
    bool done[64] = {};
    template <typename F>
    void run(F&& f) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
            f();
            return;
        }
        std::lock_guard<std::mutex> lock(m);
        if (!done[dev]) {
            f();
            done[dev] = true;
        }
    }
};

int sm_count() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace linear
}  // namespace msda

extern "C" int msda_linear(const void* x, const void* w, const void* bias, void* y,
                                    int rows, int in_features, int out_features, int dtype,
                                    void* stream) {
    const int type = dtype & ~MSDA_LINEAR_BIAS_HALF;
    if (type != MSDA_BF16 && type != MSDA_F16) return MSDA_ERR_UNSUPPORTED;
    const bool f16 = type == MSDA_F16;
    const int bias_half = (dtype & MSDA_LINEAR_BIAS_HALF) ? 1 : 0;
    if (rows < 0 || in_features < 0 || out_features < 0) return MSDA_ERR_DIM;
    using namespace msda::linear;
    if (in_features % kBK != 0 || in_features < kBK || in_features > MSDA_LINEAR_MAX_FEATURES ||
        out_features % 16 != 0 || out_features < 16 || out_features > MSDA_LINEAR_MAX_FEATURES)
        return MSDA_ERR_UNSUPPORTED;
    if (rows == 0) return MSDA_OK;
    if (x == nullptr || w == nullptr || y == nullptr) return MSDA_ERR_NULL;
    const auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(x) || misaligned(w) || misaligned(y) || (bias && misaligned(bias)))
        return MSDA_ERR_ALIGN;
    if ((int64_t)rows * in_features > 2147483647LL * 64) return MSDA_ERR_DIM;
    CUtensorMap xm, wm, ym;
    if (!make_map(&xm, x, in_features, rows, kBK, kBM, 128, false, f16) ||
        !make_map(&wm, w, in_features, out_features, kBK, out_features, 128, false, f16) ||
        !make_map(&ym, y, out_features, rows, kChunk, kChunk, 0, false, f16))
        return MSDA_ERR_CUDA;
    const Smem L = smem_layout(out_features, in_features);
    const size_t smem = (size_t)L.total + 1024;
    static PerDevice attr_once;
    attr_once.run([] {
        const int most =
            (int)(smem_layout(MSDA_LINEAR_MAX_FEATURES, MSDA_LINEAR_MAX_FEATURES).total + 1024);
        cudaFuncSetAttribute(linear_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        cudaFuncSetAttribute(linear_f16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    });
    const int tiles = (rows + kBM - 1) / kBM;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    if (f16)
        linear_f16_kernel<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
            xm, wm, ym, bias, bias_half, rows, out_features, in_features);
    else
        linear_bf16_kernel<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
            xm, wm, ym, bias, bias_half, rows, out_features, in_features);
    return cudaGetLastError() == cudaSuccess ? MSDA_OK : MSDA_ERR_CUDA;
}

extern "C" size_t msda_linear_workspace_bytes(int rows, int in_features, int out_features,
                                              int dtype) {
    (void)rows;
    if (dtype != MSDA_F32 || in_features < 0 || out_features < 0) return 0;
    return (size_t)out_features * (size_t)in_features * 2 * sizeof(float);   // w_hi, w_lo
}

extern "C" int msda_linear_f32(const float* x, const float* w, const float* bias, float* y,
                               void* workspace, size_t workspace_bytes, int rows, int in_features,
                               int out_features, void* stream) {
    using namespace msda::linear;
    if (rows < 0 || in_features < 0 || out_features < 0) return MSDA_ERR_DIM;
    if (in_features % kBKF != 0 || in_features < kBKF ||
        in_features > MSDA_LINEAR_MAX_FEATURES || out_features % 16 != 0 || out_features < 16 ||
        out_features > MSDA_LINEAR_MAX_FEATURES)
        return MSDA_ERR_UNSUPPORTED;
    if (rows == 0) return MSDA_OK;
    if (x == nullptr || w == nullptr || y == nullptr) return MSDA_ERR_NULL;
    const auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(x) || misaligned(w) || misaligned(y) || (bias && misaligned(bias)))
        return MSDA_ERR_ALIGN;
    const size_t need = msda_linear_workspace_bytes(rows, in_features, out_features, MSDA_F32);
    if (workspace == nullptr || workspace_bytes < need) return MSDA_ERR_WORKSPACE;
    if (misaligned(workspace)) return MSDA_ERR_ALIGN;
    float* w_hi = static_cast<float*>(workspace);
    float* w_lo = w_hi + (size_t)out_features * in_features;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t nw4 = (size_t)out_features * in_features / 4;
    split_tf32_kernel<<<(int)((nw4 + 255) / 256), 256, 0, st>>>(
        reinterpret_cast<const float4*>(w), reinterpret_cast<float4*>(w_hi),
        reinterpret_cast<float4*>(w_lo), nw4);
    if (cudaGetLastError() != cudaSuccess) return MSDA_ERR_CUDA;
    CUtensorMap xm, wh, wl, ym;
    if (!make_map(&xm, x, in_features, rows, kBKF, kBM, 64, true) ||
        !make_map(&wh, w_hi, in_features, out_features, kBKF, std::min(out_features, kPartF), 64,
                  true) ||
        !make_map(&wl, w_lo, in_features, out_features, kBKF, std::min(out_features, kPartF), 64,
                  true) ||
        !make_map(&ym, y, out_features, rows, kChunk, kChunk, 128, true))
        return MSDA_ERR_CUDA;
    const SmemF L = smem_layout_f();
    static PerDevice attr_once;
    attr_once.run([] {
        cudaFuncSetAttribute(linear_f32x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(smem_layout_f().total + 1024));
    });
    const int units = (rows + kBM - 1) / kBM * ((out_features + kPartF - 1) / kPartF);
    const int sms = sm_count();
    const int grid = units < sms ? units : sms;
    linear_f32x3_kernel<<<grid, kThreadsF, (size_t)L.total + 1024, st>>>(xm, wh, wl, ym, bias,
                                                                          rows, out_features,
                                                                          in_features);
    return cudaGetLastError() == cudaSuccess ? MSDA_OK : MSDA_ERR_CUDA;
}

extern "C" int msda_linear_wgrad_f32(const float* grad_y, const float* x, float* grad_w,
                                     float* grad_b, int rows, int in_features, int out_features,
                                     unsigned flags, void* stream) {
    using namespace msda::linear;
    if (rows < 0 || in_features < 0 || out_features < 0) return MSDA_ERR_DIM;
    if (flags & ~MSDA_GRAD_VALUE_ACCUMULATE) return MSDA_ERR_UNSUPPORTED;
    if (in_features % 16 != 0 || in_features < 16 || in_features > MSDA_LINEAR_MAX_FEATURES ||
        out_features % 16 != 0 || out_features < 16 ||
        out_features > MSDA_LINEAR_MAX_FEATURES)
        return MSDA_ERR_UNSUPPORTED;
    if (grad_w == nullptr) return MSDA_ERR_NULL;
    const auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(grad_w) || (grad_b && misaligned(grad_b))) return MSDA_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!(flags & MSDA_GRAD_VALUE_ACCUMULATE)) {
        if (msda::launch_zero_fill(grad_w, (size_t)out_features * in_features * 4, st) !=
                cudaSuccess ||
            (grad_b && msda::launch_zero_fill(grad_b, (size_t)out_features * 4, st) != cudaSuccess))
            return MSDA_ERR_CUDA;
    }
    if (rows == 0) return MSDA_OK;
    if (grad_y == nullptr || x == nullptr) return MSDA_ERR_NULL;
    if (misaligned(grad_y) || misaligned(x)) return MSDA_ERR_ALIGN;
    CUtensorMap gym, xm;
    if (!make_map(&gym, grad_y, out_features, rows, kBM, kWgRows, 0, true) ||
        !make_map(&xm, x, in_features, rows, in_features, kWgRows, 0, true))
        return MSDA_ERR_CUDA;
    static PerDevice attr_once;
    attr_once.run([] {
        cudaFuncSetAttribute(linear_wgrad_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(smem_layout_wg().total + 1024));
    });
    // one CTA per SM: tiles_m column tiles of gy, each with sms / tiles_m row ranges
    const int tiles_m = (out_features + kBM - 1) / kBM;
    const int sms = sm_count();
    const int blocks16 = (rows + kWgRows - 1) / kWgRows;
    int ranges = sms / tiles_m;
    if (ranges < 1) ranges = 1;
    if (ranges > blocks16) ranges = blocks16;
    const int rows_per_cta = (blocks16 + ranges - 1) / ranges * kWgRows;
    ranges = (rows + rows_per_cta - 1) / rows_per_cta;
    linear_wgrad_f32_kernel<<<ranges * tiles_m, kWgThreads, (size_t)smem_layout_wg().total + 1024,
                              st>>>(gym, xm, grad_w, grad_b, rows, out_features, in_features,
                                    tiles_m, rows_per_cta);
    return cudaGetLastError() == cudaSuccess ? MSDA_OK : MSDA_ERR_CUDA;
}

extern "C" int msda_linear_bias_grad(const void* grad_y, float* grad_b, int rows, int features,
                                     int dtype, unsigned flags, void* stream) {
    using namespace msda;
    if (rows < 0 || features < 0) return MSDA_ERR_DIM;
    if (flags & ~MSDA_GRAD_VALUE_ACCUMULATE) return MSDA_ERR_UNSUPPORTED;
    if (dtype != MSDA_F32 && dtype != MSDA_BF16 && dtype != MSDA_F16) return MSDA_ERR_UNSUPPORTED;
    const int vec = dtype == MSDA_F32 ? 4 : 8;
    if (features == 0 || features % vec != 0 || features / vec > linear::kColThreads)
        return MSDA_ERR_UNSUPPORTED;
    if (grad_b == nullptr) return MSDA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(grad_b) & 15u) != 0) return MSDA_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!(flags & MSDA_GRAD_VALUE_ACCUMULATE) &&
        launch_zero_fill(grad_b, (size_t)features * 4, st) != cudaSuccess)
        return MSDA_ERR_CUDA;
    if (rows == 0) return MSDA_OK;
    if (grad_y == nullptr) return MSDA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(grad_y) & 15u) != 0) return MSDA_ERR_ALIGN;
    // a few CTAs per SM, each over a contiguous range of at least 32 rows
    int grid = linear::sm_count() * 4;
    const int max_grid = (rows + 31) / 32;
    if (grid > max_grid) grid = max_grid;
    const int rows_per_cta = (rows + grid - 1) / grid;
    grid = (rows + rows_per_cta - 1) / rows_per_cta;
    if (dtype == MSDA_F32)
        linear::column_sum_kernel<float><<<grid, linear::kColThreads, 0, st>>>(
            static_cast<const float*>(grad_y), grad_b, rows, features, rows_per_cta);
    else if (dtype == MSDA_BF16)
        linear::column_sum_kernel<__nv_bfloat16><<<grid, linear::kColThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(grad_y), grad_b, rows, features, rows_per_cta);
    else
        linear::column_sum_kernel<__half><<<grid, linear::kColThreads, 0, st>>>(
            static_cast<const __half*>(grad_y), grad_b, rows, features, rows_per_cta);
    return cudaGetLastError() == cudaSuccess ? MSDA_OK : MSDA_ERR_CUDA;
}
