// moe_finalize_unfused_noalloc: the unfused finalize for callers that cannot
// allocate device memory.
//
// moe_finalize_unfused needs a [T, H] bf16 workspace between its combine
// kernel and its shared-add kernel, and expects the caller to provide it.
// Some callers have no way to do that: serving engines that plan every
// device byte before they start and forbid allocation on the request path,
// and plugins whose host framework owns all device memory and offers them
// no allocator.  This entry point serves them from a fixed scratch array
// compiled into the library instead.
//
// The array is a file-scope __device__ variable, so every GPU on which the
// library's device code is loaded holds its kNoallocScratchBytes until the
// process exits.  Host code cannot use the array's name as a device address
// (on the host it names a stand-in object): the device address is looked up
// with cudaGetSymbolAddress once per device, with that device current, on
// the first call made on that device, and then passed to the kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "moe_finalize.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[MOEF_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kNoallocScratchBytes = MOEF_NOALLOC_SCRATCH_BYTES;   // 8 MiB
constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (looked up once
// per device; the lookup allocates nothing).  The cached address belongs to
// the device's primary context at the time of the lookup; a context that is
// destroyed and recreated (cudaDeviceReset) leaves it stale.
cudaError_t scratch_address(void **out) {
    static std::atomic<void *> cached[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *ptr = cached[dev].load(std::memory_order_relaxed);
    if (!ptr) {
        err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        cached[dev].store(ptr, std::memory_order_relaxed);
    }
    *out = ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" {

moef_status moe_finalize_unfused_noalloc(const void *permuted_out, int64_t P,
                                         const int32_t *idx_map, const void *weights,
                                         moef_weight_kind wkind, float routed_scale,
                                         const void *shared_out, const void *residual,
                                         const void *gamma, float eps, void *out,
                                         void *residual_out, void *norm_out, int T, int K, int H,
                                         cudaStream_t stream) {
    if (T > 0 && H > 0 &&
        moe_finalize_unfused_workspace_bytes(T, H) > kNoallocScratchBytes)
        return MOEF_ERR_SHAPE;   // T * H * 2 bytes do not fit the fixed scratch
    if (T <= 0 || H <= 0)        // nothing to enqueue, or an argument error
        return moe_finalize_unfused(permuted_out, P, idx_map, weights, wkind, routed_scale,
                                    shared_out, residual, gamma, eps, out, residual_out,
                                    norm_out, T, K, H, nullptr, 0, stream);
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) {
        (void)cudaGetLastError();   // reported by the status, not left for the next launch
        return MOEF_ERR_CUDA;
    }
    return moe_finalize_unfused(permuted_out, P, idx_map, weights, wkind, routed_scale,
                                shared_out, residual, gamma, eps, out, residual_out, norm_out,
                                T, K, H, scratch, kNoallocScratchBytes, stream);
}

}  // extern "C"
