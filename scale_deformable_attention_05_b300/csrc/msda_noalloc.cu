// Allocation-free variant of the bf16 backward (msda_backward_noalloc).
//
// The bf16 backward accumulates grad_value in an fp32 scratch buffer before
// rounding it to bf16.  msda_backward takes that buffer from the caller.  Some
// callers cannot allocate device memory at all: code running inside a
// framework's memory pool that forbids extra allocations, plug-ins whose host
// application owns every allocation, or processes that must not call
// cudaMalloc while other work is being captured or timed.  This entry point
// serves them: its scratch is a fixed-size array in the library's own device
// memory, so the caller only passes inputs and outputs.
//
// The array is file-scope device memory.  On the host its name is only a
// stand-in symbol, never a device address: the address is looked up with
// cudaGetSymbolAddress on the first call on each device (made with that device
// current) and cached with the device's context; a later call in a new context
// (after a device reset) looks it up again.  The first call on a device should
// therefore come before any stream capture.  Every call on a device shares the
// one array and zero-fills it before use; calls whose work overlaps on the GPU
// race on it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/msda.h"
#include "msda_launch.h"

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[MSDA_NOALLOC_MAX_WORKSPACE_BYTES /
                                                        sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;

// The array's device address on one device, and the CUDA context it belongs to.
// A device reset (cudaDeviceReset) destroys the context and loads the module
// again in a new one, where the array may sit elsewhere: the address is looked
// up again whenever the calling thread's context differs from the cached one.
struct ScratchAddress {
    void* context;
    float* ptr;
};
ScratchAddress g_scratch[kMaxDevices] = {};

// The calling thread's current context (the driver's cuCtxGetCurrent, reached
// through the runtime's entry-point query, so the library needs no link to the
// driver library), or null when it cannot be queried.
void* current_context() {
    using GetCurrent = int (*)(void**);
    static const GetCurrent get = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult found = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &found) != cudaSuccess ||
            found != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<GetCurrent>(fn);
    }();
    void* ctx = nullptr;
    if (get == nullptr || get(&ctx) != 0) return nullptr;
    return ctx;
}

// Device address of g_noalloc_scratch on the current device, looked up with that
// device current on the first call and again after its context changed.
int scratch_for_current_device(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MSDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MSDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddress& entry = g_scratch[dev];
    void* ctx = current_context();
    if (entry.ptr == nullptr || ctx == nullptr || entry.context != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MSDA_ERR_CUDA;
        entry.ptr = static_cast<float*>(p);
        entry.context = current_context();   // the lookup makes the context current if needed
    }
    *out = entry.ptr;
    return MSDA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_tensor(const void* p, int64_t elems) {
    if (elems == 0) return MSDA_OK;
    if (p == nullptr) return MSDA_ERR_NULL;
    return aligned16(p) ? MSDA_OK : MSDA_ERR_ALIGN;
}

}  // namespace

extern "C" MSDA_API int msda_backward_noalloc(
    const void* value, const void* spatial_shapes, const void* level_start_index,
    const void* sampling_loc, const void* attn_weight, const void* grad_output, void* grad_value,
    void* grad_sampling_loc, void* grad_attn_weight, int bs, int num_keys, int num_heads,
    int head_dim, int num_levels, int num_points, int num_queries, int dtype, unsigned flags,
    void* stream) {
    // only the bf16 backward (optionally with int32 index arrays) runs here
    if ((dtype & ~MSDA_INDEX_INT32) != MSDA_BF16) return MSDA_ERR_UNSUPPORTED;
    const int idx32 = (dtype & MSDA_INDEX_INT32) ? 1 : 0;
    if (flags & ~MSDA_GRAD_VALUE_ACCUMULATE) return MSDA_ERR_UNSUPPORTED;
    if (bs < 0 || num_keys < 0 || num_heads < 0 || head_dim < 0 || num_levels < 0 ||
        num_points < 0 || num_queries < 0)
        return MSDA_ERR_DIM;
    if (num_levels > MSDA_MAX_LEVELS || (int64_t)num_levels * num_points > MSDA_MAX_LEVEL_POINTS ||
        head_dim % 8 != 0 || head_dim > MSDA_MAX_HEAD_DIM)
        return MSDA_ERR_UNSUPPORTED;
    const int64_t value_elems = (int64_t)bs * num_keys * num_heads * head_dim;
    const int64_t points = (int64_t)bs * num_queries * num_heads * num_levels * num_points;
    const int64_t out_elems = (int64_t)bs * num_queries * num_heads * head_dim;
    if ((int64_t)num_heads * head_dim > 2147483647 || (int64_t)bs * num_queries * num_heads >
        1073741823 || (int64_t)bs * num_keys > 2147483647)
        return MSDA_ERR_DIM;
    // The fp32 accumulator must fit the library's fixed scratch array.
    if ((size_t)value_elems * sizeof(float) > (size_t)MSDA_NOALLOC_MAX_WORKSPACE_BYTES)
        return MSDA_ERR_WORKSPACE;
    int rc;
    if ((rc = check_tensor(grad_value, value_elems)) != MSDA_OK) return rc;
    if ((rc = check_tensor(grad_sampling_loc, 2 * points)) != MSDA_OK) return rc;
    if ((rc = check_tensor(grad_attn_weight, points)) != MSDA_OK) return rc;
    const bool work = points > 0 && value_elems > 0;
    if (work) {
        if ((rc = check_tensor(value, value_elems)) != MSDA_OK) return rc;
        if ((rc = check_tensor(sampling_loc, points)) != MSDA_OK) return rc;
        if ((rc = check_tensor(attn_weight, points)) != MSDA_OK) return rc;
        if ((rc = check_tensor(grad_output, out_elems)) != MSDA_OK) return rc;
        if (spatial_shapes == nullptr || level_start_index == nullptr) return MSDA_ERR_NULL;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool accumulate = (flags & MSDA_GRAD_VALUE_ACCUMULATE) != 0;
    if (!work) {
        if (!accumulate && msda::launch_zero_fill(grad_value, value_elems * 2, st) != cudaSuccess)
            return MSDA_ERR_CUDA;
        if (msda::launch_zero_fill(grad_sampling_loc, 2 * points * 2, st) != cudaSuccess)
            return MSDA_ERR_CUDA;
        return msda::launch_zero_fill(grad_attn_weight, points * 2, st) == cudaSuccess
                   ? MSDA_OK : MSDA_ERR_CUDA;
    }
    float* scratch = nullptr;
    if ((rc = scratch_for_current_device(&scratch)) != MSDA_OK) return rc;
    // The array keeps the previous call's sums: clear the part this call uses.
    if (msda::launch_zero_fill(scratch, (size_t)value_elems * sizeof(float), st) != cudaSuccess)
        return MSDA_ERR_CUDA;
    const msda::Problem pb{value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                           bs, num_keys, num_heads, head_dim, num_levels, num_points,
                           num_queries, idx32};
    if (msda::launch_backward(pb, grad_output, scratch, grad_sampling_loc, grad_attn_weight,
                              msda::kBF16, st) != cudaSuccess)
        return MSDA_ERR_CUDA;
    return msda::launch_finalize_half(scratch, grad_value, (size_t)value_elems, accumulate,
                                      msda::kBF16, st) == cudaSuccess
               ? MSDA_OK
               : MSDA_ERR_CUDA;
}
