// Host-side launchers between the C ABI (msda_api.cpp) and the device code
// (msda_kernels.cu).  Arguments are already validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace msda {

struct Problem {
    const void* value;
    const void* shapes;   // int64 or int32 (idx32) [L, 2]
    const void* lsi;      // int64 or int32 (idx32) [L]
    const void* loc;
    const void* attn;
    int bs, K, M, D, L, P, Q;
    int idx32;            // index arrays are int32
    // Fused entry points: loc holds sampling offsets, attn the attention
    // logits, ref the reference points [bs, Q, L, ref_dim]; ref_dim 0 otherwise.
    const void* ref = nullptr;
    int ref_dim = 0;
    // Fused entry points: optional key padding mask [bs, K], nonzero = padded.
    const unsigned char* mask = nullptr;
};

// Element type codes (the low byte of the ABI's dtype argument).
constexpr int kF32 = 0, kBF16 = 1, kF16 = 2;

cudaError_t launch_forward(const Problem& pb, void* out, int dtype, cudaStream_t st);
// gv32: fp32 grad_value accumulator (the caller's fp32 grad_value, or the
// 16-bit paths' workspace), already zeroed or holding the sum to add to.
// grad_ref: fused mode's fp32 reference-point gradient (already zeroed), or null.
cudaError_t launch_backward(const Problem& pb, const void* grad_out, float* gv32, void* grad_loc,
                            void* grad_attn, int dtype, cudaStream_t st,
                            float* grad_ref = nullptr);
// Zeroes `bytes` bytes at p (16-byte aligned; any byte count).
cudaError_t launch_zero_fill(void* p, size_t bytes, cudaStream_t st);
// fp32 workspace -> bf16 (dtype kBF16) or fp16 (kF16) grad_value.
cudaError_t launch_finalize_half(const float* ws, void* grad_value, size_t elems, bool accumulate,
                                 int dtype, cudaStream_t st);
cudaError_t check_shapes_blocking(const int64_t* shapes, const int64_t* lsi, int num_levels,
                                  int num_keys, cudaStream_t st, bool* ok);
cudaError_t read_and_clear_error(cudaStream_t st, unsigned* word);

}  // namespace msda
