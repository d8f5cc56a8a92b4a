/*
 * msda.h -- C ABI of the B300 (sm_103a) multi-scale deformable attention library.
 *
 * The operator (Deformable DETR walk-through, zhangshiyu.com/post/59697.html,
 * section "2.2.4 源码分析", ms_deform_attn_core_pytorch and
 * MSDeformAttn.forward; argument shapes and dtypes from the Ascend
 * DrivingSDK page "multi_scale_deformable_attn", section "参数说明"):
 *
 *   output[b, q, m*D + d] = sum_{l<L} sum_{p<P} attention_weights[b,q,m,l,p] *
 *                           bilinear_zero(value[b, lsi[l] + y*W_l + x, m, d], x_im, y_im)
 *   x_im = sampling_locations[b,q,m,l,p,0] * W_l - 0.5
 *   y_im = sampling_locations[b,q,m,l,p,1] * H_l - 0.5
 *
 * i.e. torch grid_sample(mode=bilinear, padding_mode=zeros,
 * align_corners=False) at grid = 2*loc - 1, per level and head, weighted and
 * summed over levels and points.  The backward returns the gradients with
 * respect to value, sampling_locations and attention_weights (the three
 * gradients of MSDeformAttnFunction.backward on the DQ-DETR ops page,
 * blog.csdn.net/qq_43298381/article/details/145882935, section "关键代码").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layouts  All tensors are dense, C-contiguous, innermost index last:
 *             value               [bs, num_keys, num_heads, head_dim]      (dtype)
 *             spatial_shapes      [num_levels, 2] int64 (or int32), rows (H, W)
 *             level_start_index   [num_levels]    int64 (or int32)
 *             sampling_loc        [bs, num_queries, num_heads, num_levels, num_points, 2] (dtype), (x, y)
 *             attn_weight         [bs, num_queries, num_heads, num_levels, num_points]    (dtype)
 *             output, grad_output [bs, num_queries, num_heads * head_dim]  (dtype)
 *           Gradients have the shape and dtype of their input.
 *  Memory   Every tensor pointer is a DEVICE pointer (cudaMalloc or equivalent)
 *           on the current device, 16-byte aligned.  The caller owns and
 *           allocates every buffer, including the backward workspace; the
 *           library allocates nothing and keeps no per-call state.
 *  Streams  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *           default stream).  Every call only enqueues work on it and returns
 *           without synchronising, except the two calls marked BLOCKING.
 *  Numerics fp32, bf16 and fp16 inputs all accumulate in fp32.  Pixel
 *           coordinates are one fp32 fused multiply-add, loc*W - 0.5 rounded
 *           once.  A sample contributes only when -1 < x_im < W and
 *           -1 < y_im < H; pixels outside the map count as zero.  bf16 and
 *           fp16 results are rounded to nearest even.
 *  Errors   Arguments are validated on the host before anything is enqueued;
 *           a failed check returns a non-zero msda_status and enqueues
 *           nothing.  MSDA_ERR_CUDA reports a launch error from the CUDA
 *           runtime.  Device-side contents (shapes and start indices
 *           consistent with num_keys) are preconditions: kernels never read
 *           outside value for inconsistent levels -- such a level contributes
 *           nothing and raises the device error word that
 *           msda_last_device_error() returns.
 *  Empty    bs, num_queries, num_levels or num_points may be 0; the call then
 *           writes zeros to its outputs.  num_keys may be 0 only with no
 *           level holding pixels.
 *  Threads  Calls are re-entrant; concurrent calls on different streams with
 *           disjoint outputs are safe.
 */
#ifndef MSDA_H_
#define MSDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSDA_VERSION 1

#if defined(__GNUC__)
#define MSDA_API __attribute__((visibility("default")))
#else
#define MSDA_API
#endif

/* Element type of value, sampling_loc, attn_weight, output and all gradients
 * (the low byte of the `dtype` argument).  The Ascend page ("参数说明") lists
 * float32 and float16; bf16 is the other half-width type.  All of them
 * accumulate in fp32. */
typedef enum { MSDA_F32 = 0, MSDA_BF16 = 1, MSDA_F16 = 2 } msda_dtype;

/* OR-ed into `dtype`: spatial_shapes and level_start_index are int32 arrays
 * instead of int64 (the Ascend page lists both index types). */
#define MSDA_INDEX_INT32 0x100

typedef enum {
    MSDA_OK = 0,
    MSDA_ERR_NULL = 1,          /* a required pointer is NULL */
    MSDA_ERR_DIM = 2,           /* a dimension is negative, or a size overflows the index range */
    MSDA_ERR_UNSUPPORTED = 3,   /* head_dim % 8 != 0 or > MSDA_MAX_HEAD_DIM, num_levels >
                                   MSDA_MAX_LEVELS, num_levels*num_points > MSDA_MAX_LEVEL_POINTS,
                                   unknown dtype, index type or flag */
    MSDA_ERR_ALIGN = 4,         /* a tensor pointer is not 16-byte aligned */
    MSDA_ERR_WORKSPACE = 5,     /* workspace NULL or smaller than msda_backward_workspace_bytes() */
    MSDA_ERR_CUDA = 6,          /* the CUDA runtime reported an error */
    MSDA_ERR_SHAPES = 7,        /* spatial_shapes / level_start_index inconsistent with num_keys */
    MSDA_ERR_DEVICE_BOUNDS = 8  /* a kernel met an inconsistent level (or, in a library built
                                   with MSDA_BOUNDS_CHECK, a row index outside its tensor)
                                   and skipped it */
} msda_status;

/* Limits of this implementation.  The Ascend page's envelope ("约束说明":
 * num_levels*num_points <= 64, num_heads <= 8, embed_dims <= 256,
 * embed_dims % 8 == 0) lies inside them; num_heads is not limited. */
#define MSDA_MAX_LEVELS 16
#define MSDA_MAX_LEVEL_POINTS 256
#define MSDA_MAX_HEAD_DIM 512
/* num_levels*num_points limit of the fused entry points (the Ascend envelope). */
#define MSDA_MAX_FUSED_LEVEL_POINTS 64

/* Flags of msda_backward. */
#define MSDA_GRAD_VALUE_ACCUMULATE 1u /* add into grad_value instead of overwriting it */

/*
 * Forward: writes output [bs, num_queries, num_heads*head_dim].
 * Defined by ms_deform_attn_core_pytorch (walk-through, "2.2.4 源码分析")
 * with the interface of mx_driving.multi_scale_deformable_attn (Ascend page,
 * "接口原型").  output is fully overwritten.  One kernel launch.
 */
MSDA_API int msda_forward(const void* value, const void* spatial_shapes,
                 const void* level_start_index, const void* sampling_loc,
                 const void* attn_weight, void* output, int bs, int num_keys, int num_heads,
                 int head_dim, int num_levels, int num_points, int num_queries, int dtype,
                 void* stream);

/*
 * Bytes of device workspace msda_backward needs: 0 for MSDA_F32; for
 * MSDA_BF16 and MSDA_F16 an fp32 accumulator of bs*num_keys*num_heads*head_dim
 * floats.  Returns 0 for invalid arguments as well.
 */
MSDA_API size_t msda_backward_workspace_bytes(int bs, int num_keys, int num_heads, int head_dim,
                                     int dtype);

/*
 * Backward: gradients of sum(output * grad_output) with respect to value,
 * sampling_loc and attn_weight (the three tensors MSDeformAttnFunction.backward
 * returns, DQ-DETR ops page "关键代码").
 *   grad_sampling_loc and grad_attn_weight are fully overwritten.
 *   grad_value is overwritten (zero-filled, then accumulated), or added to
 *   when flags has MSDA_GRAD_VALUE_ACCUMULATE.
 *   workspace: device buffer of at least msda_backward_workspace_bytes()
 *   (may be NULL when that is 0); its contents on entry do not matter.
 * Samples outside the map get zero location and weight gradients.  The
 * gradient at an integer pixel coordinate is the one of the cell to its
 * right.  grad_value is summed with fp32 atomics: its last bits may differ
 * between runs.  Launches: zero-fill (unless accumulating), the gather /
 * scatter kernel, and for bf16 / fp16 one fp32 -> half finalize kernel.
 */
MSDA_API int msda_backward(const void* value, const void* spatial_shapes,
                  const void* level_start_index, const void* sampling_loc,
                  const void* attn_weight, const void* grad_output, void* grad_value,
                  void* grad_sampling_loc, void* grad_attn_weight, void* workspace,
                  size_t workspace_bytes, int bs, int num_keys, int num_heads, int head_dim,
                  int num_levels, int num_points, int num_queries, int dtype, unsigned flags,
                  void* stream);

/*
 * Fused preparation + forward: the step before the operator in
 * MSDeformAttn.forward (walk-through, "2.2.4 源码分析"; 4-d references from
 * section "2.4") is done inside the kernel.  Instead of locations and weights
 * it takes
 *   reference_points  [bs, num_queries, num_levels, ref_dim] (dtype), ref_dim
 *                     2: (x, y), or 4: (x, y, w, h) boxes
 *   sampling_offsets  [bs, num_queries, num_heads, num_levels, num_points, 2]
 *   attn_logits       [bs, num_queries, num_heads, num_levels*num_points]
 * and computes, per sample, a = softmax of its (b, q, m) row of logits and
 *   ref_dim 2: loc = ref + off / (W_l, H_l)
 *   ref_dim 4: loc = ref_xy + off / num_points * ref_wh * 0.5
 * in binary32, one correctly rounded operation at a time, left to right, with
 * IEEE division: fl(ref + fl(off / W)) and fl(ref_xy + fl(fl(fl(off /
 * num_points) * w) * 0.5)), then the same sum as msda_forward.
 *   key_padding_mask  [bs, num_keys] bytes (a torch.bool tensor), nonzero =
 *                     padded key, or NULL.  The module's masked_fill of value
 *                     (walk-through, "2.2.4", MSDeformAttn.forward) fused into
 *                     the value load: every head's row of a padded key reads
 *                     as zero.  Any byte alignment.
 * num_levels*num_points must not exceed MSDA_MAX_FUSED_LEVEL_POINTS (else
 * MSDA_ERR_UNSUPPORTED), ref_dim must be 2 or 4.  Saves the caller's softmax,
 * location and masking kernels and their round trips through memory.  One
 * kernel launch.
 */
MSDA_API int msda_forward_fused(const void* value, const void* spatial_shapes,
                                const void* level_start_index, const void* reference_points,
                                const void* sampling_offsets, const void* attn_logits,
                                const void* key_padding_mask, void* output, int bs,
                                int num_keys, int num_heads, int head_dim, int num_levels,
                                int num_points, int num_queries, int ref_dim, int dtype,
                                void* stream);

/*
 * Backward of msda_forward_fused: grad_value (as msda_backward, same
 * workspace rule and flags), grad_sampling_offsets (shape and dtype of the
 * offsets), grad_attn_logits (through the softmax: a * (g_a - sum_j a_j g_a_j)
 * per row), and, when grad_reference_points is not NULL, the gradient of the
 * reference points summed over heads and points into that fp32
 * [bs, num_queries, num_levels, ref_dim] buffer (16-byte aligned, overwritten).
 * With key_padding_mask, grad_value is the gradient with respect to the value
 * before masking: padded rows receive none (zero, or unchanged when
 * accumulating).  Launches: zero-fills, one gather / scatter kernel, and for
 * half types the finalize kernel.
 */
MSDA_API int msda_backward_fused(const void* value, const void* spatial_shapes,
                                 const void* level_start_index, const void* reference_points,
                                 const void* sampling_offsets, const void* attn_logits,
                                 const void* key_padding_mask, const void* grad_output,
                                 void* grad_value,
                                 void* grad_sampling_offsets, void* grad_attn_logits,
                                 float* grad_reference_points, void* workspace,
                                 size_t workspace_bytes, int bs, int num_keys, int num_heads,
                                 int head_dim, int num_levels, int num_points, int num_queries,
                                 int ref_dim, int dtype, unsigned flags, void* stream);

/*
 * Zero `bytes` bytes of device memory at `ptr` on `stream` with the
 * library's vectorised fill kernel (ptr 16-byte aligned, bytes a multiple
 * of 16).  For callers that accumulate gradients across calls with
 * MSDA_GRAD_VALUE_ACCUMULATE.
 */
MSDA_API int msda_zero_fill(void* ptr, size_t bytes, void* stream);

/*
 * BLOCKING.  For int64 index arrays: checks on the device that level_start_index is the exclusive
 * prefix sum of H*W (Ascend page call example; walk-through "2.3.1") and
 * that the levels add up to num_keys (the assertion at the top of
 * MSDeformAttn.forward).  Returns MSDA_OK or MSDA_ERR_SHAPES.  Synchronises
 * `stream`.  A debugging aid: the hot path does not call it.
 */
MSDA_API int msda_check_shapes(const int64_t* spatial_shapes, const int64_t* level_start_index,
                      int num_levels, int num_keys, void* stream);

/*
 * BLOCKING.  Synchronises `stream`, then returns MSDA_ERR_DEVICE_BOUNDS if
 * any kernel of this library on the current device met a level whose pixels
 * fall outside [0, num_keys) since the previous call -- or, in a library built
 * with -DMSDA_BOUNDS_CHECK, a value / grad_value row index outside the tensor
 * (the access is skipped) -- else MSDA_OK; clears the word.
 */
MSDA_API int msda_last_device_error(void* stream);

/* Static, human-readable text of a status code. */
MSDA_API const char* msda_status_string(int status);

/*
 * Allocation-free bf16 backward.  Not part of the method: an addition for
 * callers that cannot allocate device memory (a host framework that owns every
 * allocation, a plug-in without access to the allocator, code that must not
 * call cudaMalloc while work is captured or timed).  Same arguments, results
 * and launches as msda_backward with dtype MSDA_BF16, except that there is no
 * workspace argument: the fp32 accumulator is a fixed array of
 * MSDA_NOALLOC_MAX_WORKSPACE_BYTES in the library's own device memory, which
 * every GPU that loads the library holds until the process exits.
 *   - Returns MSDA_ERR_WORKSPACE when bs*num_keys*num_heads*head_dim*4 exceeds
 *     MSDA_NOALLOC_MAX_WORKSPACE_BYTES, and MSDA_ERR_UNSUPPORTED for any dtype
 *     but MSDA_BF16 (optionally with MSDA_INDEX_INT32; the fp32 backward needs
 *     no workspace: use msda_backward).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it with the device's CUDA context; make
 *     that first call before any stream capture.  A call in a new context of
 *     the device (after cudaDeviceReset) looks the address up again.
 *   - Each loaded copy of the library holds its own array (64 MiB per copy
 *     and device).
 *   - Every call on a device shares the one array and zero-fills the part it
 *     uses before accumulating; calls whose work overlaps on the GPU (other
 *     streams, other host threads) race on it and must be serialised.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define MSDA_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)64 << 20)
MSDA_API int msda_backward_noalloc(const void* value, const void* spatial_shapes,
                                   const void* level_start_index, const void* sampling_loc,
                                   const void* attn_weight, const void* grad_output,
                                   void* grad_value, void* grad_sampling_loc,
                                   void* grad_attn_weight, int bs, int num_keys, int num_heads,
                                   int head_dim, int num_levels, int num_points, int num_queries,
                                   int dtype, unsigned flags, void* stream);

/*
 * Linear projection on the tensor cores: y = x * w^T + bias, the nn.Linear
 * layers around the operator in MSDeformAttn.forward (walk-through, "2.2.4
 * 源码分析": value_proj, sampling_offsets, attention_weights, output_proj).
 *   x    [rows, in_features]          bf16 (fp16 when dtype is MSDA_F16),
 *                                      row-major, device pointer
 *   w    [out_features, in_features]  the same type (nn.Linear weight layout)
 *   bias [out_features]               fp32, or the operands' type when dtype
 *                                      has MSDA_LINEAR_BIAS_HALF, or NULL
 *   y    [rows, out_features]         the operands' type, overwritten; fp32
 *                                      accumulation, one rounding after the bias
 * dtype must be MSDA_BF16 or MSDA_F16 (optionally | MSDA_LINEAR_BIAS_HALF;
 * MSDA_LINEAR_BIAS_BF16 is the same flag).  in_features
 * must be a multiple of 64 and
 * out_features a multiple of 16, both at most MSDA_LINEAR_MAX_FEATURES (else
 * MSDA_ERR_UNSUPPORTED); every pointer 16-byte aligned (MSDA_ERR_ALIGN).
 * One kernel launch (one persistent CTA per SM: TMA loads, tcgen05.mma into
 * two alternating accumulators in tensor memory, TMA stores).  A device-side
 * wait that runs out of its iteration limit stops the kernel and raises the
 * error word msda_last_device_error() reads.  The first call of each
 * projection entry point on a device raises its kernel's shared-memory limit
 * (cudaFuncSetAttribute): make it before capturing a CUDA graph of later calls.
 * The entry points allocate nothing and never synchronise, so later calls can
 * be captured.
 */
#define MSDA_LINEAR_MAX_FEATURES 256
#define MSDA_LINEAR_BIAS_HALF 0x200
#define MSDA_LINEAR_BIAS_BF16 MSDA_LINEAR_BIAS_HALF
MSDA_API int msda_linear(const void* x, const void* w, const void* bias, void* y, int rows,
                         int in_features, int out_features, int dtype, void* stream);

/*
 * The same projection in fp32 on the tensor cores, to fp32 accuracy: each
 * operand is split into its TF32 rounding and the exact remainder,
 * a = a_hi + a_lo, and the product is accumulated in fp32 as
 * x_hi w_hi + x_hi w_lo + x_lo w_hi (three tcgen05.mma of kind::tf32 per K
 * step).  The dropped x_lo w_lo term and the TF32 reading of the remainders
 * contribute below 2^-19 of sum_k |x[r,k]| |w[n,k]|, under fp32 accumulation's
 * own rounding.
 *   x    [rows, in_features]          fp32, row-major, device pointer
 *   w    [out_features, in_features]  fp32 (nn.Linear weight layout)
 *   bias [out_features]               fp32 or NULL
 *   y    [rows, out_features]         fp32, overwritten
 *   workspace  device scratch of at least msda_linear_workspace_bytes(rows,
 *              in_features, out_features, MSDA_F32) bytes (the two parts of
 *              w, 8 * out_features * in_features), 16-byte aligned, owned by
 *              the caller; overwritten
 * in_features and out_features must be multiples of 16, both at most
 * MSDA_LINEAR_MAX_FEATURES (else MSDA_ERR_UNSUPPORTED); every
 * pointer 16-byte aligned (MSDA_ERR_ALIGN); a short or NULL workspace gives
 * MSDA_ERR_WORKSPACE.  Two launches on `stream`: the split of w, then the
 * GEMM (persistent CTAs, TMA loads and stores, x split in shared memory, two
 * accumulators in tensor memory).  A device-side wait that runs out of its iteration limit
 * stops the kernel and raises the error word msda_last_device_error() reads.
 */
MSDA_API size_t msda_linear_workspace_bytes(int rows, int in_features, int out_features,
                                            int dtype);
MSDA_API int msda_linear_f32(const float* x, const float* w, const float* bias, float* y,
                             void* workspace, size_t workspace_bytes, int rows, int in_features,
                             int out_features, void* stream);

/*
 * Parameter gradients of that fp32 projection on the tensor cores, with the
 * same three-TF32-product split:
 *   grad_w[n, k] (+)= sum_r grad_y[r, n] x[r, k]      (grad_y^T x)
 *   grad_b[n]    (+)= sum_r grad_y[r, n]              (skipped when grad_b is NULL)
 *   grad_y [rows, out_features], x [rows, in_features]: fp32, row-major,
 *          device pointers (the layer's output gradient and input)
 *   grad_w [out_features, in_features], grad_b [out_features]: fp32, device
 * flags: 0 overwrites grad_w and grad_b, MSDA_GRAD_VALUE_ACCUMULATE adds to
 * them.  in_features and out_features must be multiples of 16, both at most
 * MSDA_LINEAR_MAX_FEATURES (else MSDA_ERR_UNSUPPORTED); every pointer 16-byte
 * aligned (MSDA_ERR_ALIGN).  Launches on `stream`: zero-fills unless
 * accumulating, then one kernel of one CTA per SM, each summing a contiguous
 * range of rows for 128 columns of grad_y in tensor memory and adding its
 * partial sums with fp32 reductions (so the order of the additions, and the
 * last bits of the result, vary between runs).  A device-side wait that runs
 * out of its iteration limit stops the kernel and raises the error word
 * msda_last_device_error() reads.
 */
MSDA_API int msda_linear_wgrad_f32(const float* grad_y, const float* x, float* grad_w,
                                   float* grad_b, int rows, int in_features, int out_features,
                                   unsigned flags, void* stream);

/*
 * Bias gradient of a projection: grad_b[c] (+)= sum_r grad_y[r, c], summed in
 * fp32 (the bf16 and fp16 layers' bias gradients; the fp32 layers get theirs
 * from msda_linear_wgrad_f32).
 *   grad_y [rows, features]  dtype MSDA_F32, MSDA_BF16 or MSDA_F16, row-major,
 *                            device pointer
 *   grad_b [features]        fp32, device pointer; overwritten unless flags
 *                            has MSDA_GRAD_VALUE_ACCUMULATE
 * features must be a multiple of the 16-byte vector (4 fp32 or 8 half
 * elements) and at most 256 vectors (else MSDA_ERR_UNSUPPORTED); pointers
 * 16-byte aligned (MSDA_ERR_ALIGN).  Launches on `stream` (a zero-fill unless
 * accumulating, then one kernel whose CTAs add their partial sums with
 * atomicAdd, so the last bits vary between runs).
 */
MSDA_API int msda_linear_bias_grad(const void* grad_y, float* grad_b, int rows, int features,
                                   int dtype, unsigned flags, void* stream);

/* MSDA_VERSION of the built library. */
MSDA_API int msda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSDA_H_ */
