// Routing-word kernels: unpacking (expert_id << 16) | bf16(weight) words and
// counting out-of-range entries of the [token, top_k] row map.
//
// Packed format: "[Deepseek V4] Keep fp32 routing weights in the mxfp4
// trtllm MoE", description.  Row-map bounds: "[Kimi K2.5] Fuse deferred MoE
// finalize into next-layer AR + residual + RMSNorm", Key modifications (a
// flat index map read with the wrong top_k went out of bounds).
//
// Both are small elementwise passes over T*K words (grid-stride loops,
// grids capped at a few CTAs per SM); they are bound by launch latency,
// not by bandwidth.
#include "internal.cuh"

namespace moef {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
unpack_kernel(const int32_t *__restrict__ packed, int64_t n,
              int32_t *__restrict__ expert_ids, float *__restrict__ weights) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const uint32_t u = static_cast<uint32_t>(__ldg(packed + i));
        if (expert_ids) expert_ids[i] = static_cast<int32_t>(u >> 16);
        if (weights) weights[i] = __uint_as_float(u << 16);
    }
}

__global__ void __launch_bounds__(kThreads)
check_kernel(const int32_t *__restrict__ idx, int64_t n, int64_t P, int32_t *bad_count) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    unsigned local = 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const int32_t r = __ldg(idx + i);
        local += (r < 0 || static_cast<int64_t>(r) >= P) ? 1u : 0u;
    }
    // every lane of the (full) warp reaches this point
    local = __reduce_add_sync(0xFFFFFFFFu, local);
    if ((threadIdx.x & 31) == 0 && local) atomicAdd(bad_count, static_cast<int32_t>(local));
}

unsigned grid_for(int64_t n, int num_sms) {
    int64_t blocks = (n + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_unpack(const int32_t *packed, int64_t n, int32_t *expert_ids,
                          float *weights, int num_sms, cudaStream_t stream) {
    void *args[] = {&packed, &n, &expert_ids, &weights};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&unpack_kernel),
                            dim3(grid_for(n, num_sms)), dim3(kThreads), args, 0, stream);
}

cudaError_t launch_check_indices(const int32_t *idx, int64_t n, int64_t P,
                                 int32_t *d_bad_count, int num_sms, cudaStream_t stream) {
    cudaError_t err = cudaMemsetAsync(d_bad_count, 0, sizeof(int32_t), stream);
    if (err != cudaSuccess) return err;
    if (n == 0) return cudaSuccess;
    void *args[] = {&idx, &n, &P, &d_bad_count};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&check_kernel),
                            dim3(grid_for(n, num_sms)), dim3(kThreads), args, 0, stream);
}

}  // namespace moef
