// C ABI of the library (declared in include/msda.h): host-side argument
// validation, then the launchers of msda_kernels.cu.  Every check runs before
// anything is enqueued, so a rejected call leaves the stream untouched.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/msda.h"
#include "msda_launch.h"

namespace {

constexpr int64_t kIntMax = 2147483647;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The element type is the low byte of `dtype`; MSDA_INDEX_INT32 may be OR-ed in.
int value_type(int dtype) { return dtype & 0xff; }
int index32(int dtype) { return (dtype & MSDA_INDEX_INT32) ? 1 : 0; }
bool known_dtype(int dtype) {
    const int v = value_type(dtype);
    return (dtype & ~(0xff | MSDA_INDEX_INT32)) == 0 &&
           (v == MSDA_F32 || v == MSDA_BF16 || v == MSDA_F16);
}
int elem_bytes(int dtype) { return value_type(dtype) == MSDA_F32 ? 4 : 2; }

struct Dims {
    int64_t bs, K, M, D, L, P, Q;
    int64_t value_elems() const { return bs * K * M * D; }
    int64_t out_elems() const { return bs * Q * M * D; }
    int64_t points() const { return bs * Q * M * L * P; }
    int64_t rows() const { return bs * Q * M; }
};

// Shared checks of forward and backward (everything but the pointers).
int check_dims(const Dims& d, int dtype) {
    if (!known_dtype(dtype)) return MSDA_ERR_UNSUPPORTED;
    if (d.bs < 0 || d.K < 0 || d.M < 0 || d.D < 0 || d.L < 0 || d.P < 0 || d.Q < 0)
        return MSDA_ERR_DIM;
    if (d.L > MSDA_MAX_LEVELS || d.L * d.P > MSDA_MAX_LEVEL_POINTS) return MSDA_ERR_UNSUPPORTED;
    if (d.D % 8 != 0 || d.D > MSDA_MAX_HEAD_DIM) return MSDA_ERR_UNSUPPORTED;
    // 32-bit indices inside the kernels: keys, rows and per-row offsets.
    if (d.M * d.D > kIntMax) return MSDA_ERR_DIM;
    if (d.rows() > kIntMax / 2) return MSDA_ERR_DIM;
    if (d.bs * d.K > kIntMax || d.value_elems() > (int64_t(1) << 46)) return MSDA_ERR_DIM;
    if (d.points() > (int64_t(1) << 46)) return MSDA_ERR_DIM;
    return MSDA_OK;
}

// The fused entry points keep each (b, q, m) row's L*P samples in one round of
// a warp: at most MSDA_MAX_FUSED_LEVEL_POINTS of them.
int check_fused(const Dims& d, int ref_dim) {
    if (ref_dim != 2 && ref_dim != 4) return MSDA_ERR_UNSUPPORTED;
    if (d.L * d.P > MSDA_MAX_FUSED_LEVEL_POINTS) return MSDA_ERR_UNSUPPORTED;
    return MSDA_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MSDA_OK : MSDA_ERR_CUDA; }

// Device pointer argument: must be non-null and 16-byte aligned when the
// tensor it points to holds at least one element.
int check_ptr(const void* p, int64_t elems) {
    if (elems == 0) return MSDA_OK;
    if (p == nullptr) return MSDA_ERR_NULL;
    if (!aligned16(p)) return MSDA_ERR_ALIGN;
    return MSDA_OK;
}

#define MSDA_TRY(expr)                 \
    do {                               \
        const int _rc = (expr);        \
        if (_rc != MSDA_OK) return _rc; \
    } while (0)

}  // namespace

extern "C" {

int msda_version(void) { return MSDA_VERSION; }

const char* msda_status_string(int status) {
    switch (status) {
        case MSDA_OK: return "ok";
        case MSDA_ERR_NULL: return "a required pointer is NULL";
        case MSDA_ERR_DIM: return "invalid dimension (negative, or index range exceeded)";
        case MSDA_ERR_UNSUPPORTED:
            return "unsupported configuration (dtype, index type, flags, head_dim % 8, "
                   "head_dim > 512, num_levels > 16 or num_levels*num_points > 256)";
        case MSDA_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
        case MSDA_ERR_WORKSPACE: return "workspace missing or too small";
        case MSDA_ERR_CUDA: return "CUDA runtime error";
        case MSDA_ERR_SHAPES:
            return "spatial_shapes / level_start_index inconsistent with num_keys";
        case MSDA_ERR_DEVICE_BOUNDS:
            return "a kernel skipped a level whose pixels fall outside [0, num_keys), or a row "
                   "index outside its tensor (bounds-checked build)";
        default: return "unknown status";
    }
}

}  // extern "C"

namespace {

// Shared body of msda_forward (ref_dim 0: sampling_loc / attn_weight are
// locations and weights) and msda_forward_fused (ref_dim 2 or 4:
// sampling_loc / attn_weight are offsets and logits, ref the reference points).
int forward_impl(const void* value, const void* spatial_shapes, const void* level_start_index,
                 const void* sampling_loc, const void* attn_weight, const void* ref,
                 int ref_dim, const void* mask, void* output, const Dims& d, int dtype,
                 void* stream) {
    MSDA_TRY(check_dims(d, dtype));
    if (ref_dim != 0) MSDA_TRY(check_fused(d, ref_dim));
    MSDA_TRY(check_ptr(output, d.out_elems()));
    const bool work = d.points() > 0 && d.out_elems() > 0;
    if (work) {
        MSDA_TRY(check_ptr(value, d.value_elems()));
        MSDA_TRY(check_ptr(sampling_loc, d.points()));
        MSDA_TRY(check_ptr(attn_weight, d.points()));
        if (ref_dim != 0) MSDA_TRY(check_ptr(ref, d.bs * d.Q * d.L * ref_dim));
        if (spatial_shapes == nullptr || level_start_index == nullptr) return MSDA_ERR_NULL;
    }
    if (d.out_elems() == 0) return MSDA_OK;
    cudaStream_t st = as_stream(stream);
    if (!work)  // no samples: the output is all zeros
        return cuda_status(msda::launch_zero_fill(output, d.out_elems() * elem_bytes(dtype), st));
    msda::Problem pb{value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                     (int)d.bs, (int)d.K, (int)d.M, (int)d.D, (int)d.L, (int)d.P, (int)d.Q,
                     index32(dtype)};
    pb.ref = ref;
    pb.ref_dim = ref_dim;
    pb.mask = static_cast<const unsigned char*>(mask);
    return cuda_status(msda::launch_forward(pb, output, value_type(dtype), st));
}

// Shared body of msda_backward and msda_backward_fused (see forward_impl);
// grad_ref (fused only, fp32, may be null) is zero-filled and accumulated.
int backward_impl(const void* value, const void* spatial_shapes, const void* level_start_index,
                  const void* sampling_loc, const void* attn_weight, const void* ref, int ref_dim,
                  const void* mask, const void* grad_output, void* grad_value,
                  void* grad_sampling_loc,
                  void* grad_attn_weight, float* grad_ref, void* workspace,
                  size_t workspace_bytes, const Dims& d, int dtype, unsigned flags,
                  void* stream) {
    MSDA_TRY(check_dims(d, dtype));
    if (ref_dim != 0) MSDA_TRY(check_fused(d, ref_dim));
    if (flags & ~MSDA_GRAD_VALUE_ACCUMULATE) return MSDA_ERR_UNSUPPORTED;
    const bool accumulate = (flags & MSDA_GRAD_VALUE_ACCUMULATE) != 0;
    MSDA_TRY(check_ptr(grad_value, d.value_elems()));
    MSDA_TRY(check_ptr(grad_sampling_loc, 2 * d.points()));
    MSDA_TRY(check_ptr(grad_attn_weight, d.points()));
    const int64_t ref_elems = ref_dim != 0 ? d.bs * d.Q * d.L * ref_dim : 0;
    if (grad_ref != nullptr && !aligned16(grad_ref)) return MSDA_ERR_ALIGN;
    const bool work = d.points() > 0 && d.value_elems() > 0;
    if (work) {
        MSDA_TRY(check_ptr(value, d.value_elems()));
        MSDA_TRY(check_ptr(sampling_loc, d.points()));
        MSDA_TRY(check_ptr(attn_weight, d.points()));
        MSDA_TRY(check_ptr(grad_output, d.out_elems()));
        if (ref_dim != 0) MSDA_TRY(check_ptr(ref, ref_elems));
        if (spatial_shapes == nullptr || level_start_index == nullptr) return MSDA_ERR_NULL;
    }
    const size_t ws_need =
        msda_backward_workspace_bytes((int)d.bs, (int)d.K, (int)d.M, (int)d.D, dtype);
    if (ws_need > 0) {
        if (workspace == nullptr || workspace_bytes < ws_need) return MSDA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return MSDA_ERR_ALIGN;
    }
    cudaStream_t st = as_stream(stream);
    const int e = elem_bytes(dtype);
    const size_t value_bytes = (size_t)d.value_elems() * e;
    if (grad_ref != nullptr && ref_elems > 0)
        MSDA_TRY(cuda_status(msda::launch_zero_fill(grad_ref, ref_elems * sizeof(float), st)));
    if (!work) {
        // No sample reads value: zero location / weight grads, and grad_value
        // stays as it is (accumulate) or becomes zero.
        if (!accumulate) MSDA_TRY(cuda_status(msda::launch_zero_fill(grad_value, value_bytes, st)));
        MSDA_TRY(cuda_status(msda::launch_zero_fill(grad_sampling_loc, 2 * d.points() * e, st)));
        return cuda_status(msda::launch_zero_fill(grad_attn_weight, d.points() * e, st));
    }
    msda::Problem pb{value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                     (int)d.bs, (int)d.K, (int)d.M, (int)d.D, (int)d.L, (int)d.P, (int)d.Q,
                     index32(dtype)};
    pb.ref = ref;
    pb.ref_dim = ref_dim;
    pb.mask = static_cast<const unsigned char*>(mask);
    const int vt = value_type(dtype);
    float* gv32;
    if (vt == MSDA_F32) {
        gv32 = static_cast<float*>(grad_value);
        if (!accumulate) MSDA_TRY(cuda_status(msda::launch_zero_fill(gv32, value_bytes, st)));
    } else {
        gv32 = static_cast<float*>(workspace);
        MSDA_TRY(cuda_status(msda::launch_zero_fill(gv32, ws_need, st)));
    }
    MSDA_TRY(cuda_status(msda::launch_backward(pb, grad_output, gv32, grad_sampling_loc,
                                               grad_attn_weight, vt, st, grad_ref)));
    if (vt != MSDA_F32)
        return cuda_status(msda::launch_finalize_half(gv32, grad_value, (size_t)d.value_elems(),
                                                      accumulate, vt, st));
    return MSDA_OK;
}

}  // namespace

extern "C" {

int msda_forward(const void* value, const void* spatial_shapes,
                 const void* level_start_index, const void* sampling_loc,
                 const void* attn_weight, void* output, int bs, int num_keys, int num_heads,
                 int head_dim, int num_levels, int num_points, int num_queries, int dtype,
                 void* stream) {
    const Dims d{bs, num_keys, num_heads, head_dim, num_levels, num_points, num_queries};
    return forward_impl(value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                        nullptr, 0, nullptr, output, d, dtype, stream);
}

int msda_forward_fused(const void* value, const void* spatial_shapes,
                       const void* level_start_index, const void* reference_points,
                       const void* sampling_offsets, const void* attn_logits,
                       const void* key_padding_mask, void* output, int bs, int num_keys,
                       int num_heads, int head_dim, int num_levels, int num_points,
                       int num_queries, int ref_dim, int dtype, void* stream) {
    const Dims d{bs, num_keys, num_heads, head_dim, num_levels, num_points, num_queries};
    if (ref_dim != 2 && ref_dim != 4) return MSDA_ERR_UNSUPPORTED;
    return forward_impl(value, spatial_shapes, level_start_index, sampling_offsets, attn_logits,
                        reference_points, ref_dim, key_padding_mask, output, d, dtype, stream);
}

size_t msda_backward_workspace_bytes(int bs, int num_keys, int num_heads, int head_dim,
                                     int dtype) {
    if (!known_dtype(dtype) || value_type(dtype) == MSDA_F32) return 0;
    if (bs < 0 || num_keys < 0 || num_heads < 0 || head_dim < 0) return 0;
    return (size_t)bs * (size_t)num_keys * (size_t)num_heads * (size_t)head_dim * sizeof(float);
}

int msda_backward(const void* value, const void* spatial_shapes,
                  const void* level_start_index, const void* sampling_loc,
                  const void* attn_weight, const void* grad_output, void* grad_value,
                  void* grad_sampling_loc, void* grad_attn_weight, void* workspace,
                  size_t workspace_bytes, int bs, int num_keys, int num_heads, int head_dim,
                  int num_levels, int num_points, int num_queries, int dtype, unsigned flags,
                  void* stream) {
    const Dims d{bs, num_keys, num_heads, head_dim, num_levels, num_points, num_queries};
    return backward_impl(value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                         nullptr, 0, nullptr, grad_output, grad_value, grad_sampling_loc,
                         grad_attn_weight, nullptr, workspace, workspace_bytes, d, dtype, flags,
                         stream);
}

int msda_backward_fused(const void* value, const void* spatial_shapes,
                        const void* level_start_index, const void* reference_points,
                        const void* sampling_offsets, const void* attn_logits,
                        const void* key_padding_mask, const void* grad_output, void* grad_value,
                        void* grad_sampling_offsets,
                        void* grad_attn_logits, float* grad_reference_points, void* workspace,
                        size_t workspace_bytes, int bs, int num_keys, int num_heads,
                        int head_dim, int num_levels, int num_points, int num_queries,
                        int ref_dim, int dtype, unsigned flags, void* stream) {
    const Dims d{bs, num_keys, num_heads, head_dim, num_levels, num_points, num_queries};
    if (ref_dim != 2 && ref_dim != 4) return MSDA_ERR_UNSUPPORTED;
    return backward_impl(value, spatial_shapes, level_start_index, sampling_offsets,
                         attn_logits, reference_points, ref_dim, key_padding_mask, grad_output,
                         grad_value,
                         grad_sampling_offsets, grad_attn_logits, grad_reference_points,
                         workspace, workspace_bytes, d, dtype, flags, stream);
}

int msda_zero_fill(void* ptr, size_t bytes, void* stream) {
    if (bytes == 0) return MSDA_OK;
    if (ptr == nullptr) return MSDA_ERR_NULL;
    if (!aligned16(ptr) || bytes % 16 != 0) return MSDA_ERR_ALIGN;
    return cuda_status(msda::launch_zero_fill(ptr, bytes, as_stream(stream)));
}

int msda_check_shapes(const int64_t* spatial_shapes, const int64_t* level_start_index,
                      int num_levels, int num_keys, void* stream) {
    if (num_levels < 0 || num_keys < 0) return MSDA_ERR_DIM;
    if (num_levels > MSDA_MAX_LEVELS) return MSDA_ERR_UNSUPPORTED;
    if (num_levels == 0) return num_keys == 0 ? MSDA_OK : MSDA_ERR_SHAPES;
    if (spatial_shapes == nullptr || level_start_index == nullptr) return MSDA_ERR_NULL;
    bool ok = false;
    MSDA_TRY(cuda_status(msda::check_shapes_blocking(spatial_shapes, level_start_index,
                                                     num_levels, num_keys, as_stream(stream),
                                                     &ok)));
    return ok ? MSDA_OK : MSDA_ERR_SHAPES;
}

int msda_last_device_error(void* stream) {
    unsigned word = 0;
    MSDA_TRY(cuda_status(msda::read_and_clear_error(as_stream(stream), &word)));
    return word ? MSDA_ERR_DEVICE_BOUNDS : MSDA_OK;
}

}  // extern "C"
