// Unfused finalize: the same result computed the way the pages' baselines
// ran it, as separate kernels with bf16 intermediates in global memory:
//
//   1. combine:  tmp = bf16( sum_k (w[t,k] * routed_scale) * permuted_out[idx[t,k], :] )
//   2. add:      out = bf16( tmp + shared_out )
//   3. (with a residual) residual + RMSNorm:
//                residual_out = bf16( out + residual ),
//                norm_out = bf16( residual_out * rsqrt(mean(residual_out^2) + eps) * gamma )
//
// "Support deferred MoE finalize for MXFP4 and FP8 block-scale", Speed: the
// baseline launched an in-kernel combine and an elementwise add for the
// shared expert, which the deferred finalize merges into one kernel.
// "[Kimi K2.5] Fuse deferred MoE finalize into next-layer AR + residual +
// RMSNorm", Numerics & speed: the fallback runs the finalize and then a
// separate residual + RMSNorm kernel (there fused with the all-reduce).
//
// It exists to measure the fusion on this GPU against the same inputs: one
// or two extra launches, the [T, H] intermediate written and read back, and
// up to three more bf16 roundings than the fused kernel.
#include "internal.cuh"
#include "vec.cuh"

namespace moef {
namespace {

constexpr int kCombineThreadsMax = 256;
constexpr int kAddThreads = 256;
constexpr int kNormThreads = 256;

// One CTA per (token, slice) as in the fused kernel's plan; each thread walks
// its vectors of the slice.
template <int VEC>
__global__ void __launch_bounds__(kCombineThreadsMax)
combine_kernel(const __grid_constant__ FinalizeParams p, uint16_t *tmp) {
    using Ops = VecOps<VEC>;
    using V = typename Ops::V;
    __shared__ const uint16_t *s_row[MOEF_MAX_K];
    __shared__ float s_w[MOEF_MAX_K];

    const int S = p.splits;
    const int t = blockIdx.x / S;
    const int split = blockIdx.x - t * S;
    const int K = p.K;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x < K) {
        const int64_t i = static_cast<int64_t>(t) * K + threadIdx.x;
        const int r = __ldg(p.idx + i);
        s_row[threadIdx.x] = p.x + static_cast<int64_t>(r) * p.H;
        s_w[threadIdx.x] = decode_weight(p.weights, p.wkind, i) * p.routed_scale;
    }
    __syncthreads();
    const int64_t tok = static_cast<int64_t>(t) * p.H;
    const int v_begin = split * p.slice;
    const int v_end = min(v_begin + p.slice, p.nvec);
    for (int v = v_begin + threadIdx.x; v < v_end; v += blockDim.x) {
        const int64_t e = static_cast<int64_t>(v) * VEC;
        float acc[VEC];
#pragma unroll
        for (int q = 0; q < VEC; ++q) acc[q] = 0.f;
        for (int k0 = 0; k0 < K; k0 += 8) {
            V xv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (k0 + u < K) xv[u] = Ops::load_row(s_row[k0 + u] + e);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k0 + u < K) {
                    float xf[VEC];
                    Ops::to_f32(xv[u], xf);
                    const float w = s_w[k0 + u];
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc[q] = fmaf(w, xf[q], acc[q]);
                }
            }
        }
        Ops::store(tmp + tok + e, Ops::from_f32(acc));
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// out = bf16(a + b) over n vectors (grid-stride).
template <int VEC>
__global__ void __launch_bounds__(kAddThreads)
add_kernel(const uint16_t *a, const uint16_t *b, uint16_t *out, int64_t n) {
    using Ops = VecOps<VEC>;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < n;
         v += stride) {
        float fa[VEC], fb[VEC];
        Ops::to_f32(Ops::load(a + v * VEC), fa);
        Ops::to_f32(Ops::load(b + v * VEC), fb);
#pragma unroll
        for (int q = 0; q < VEC; ++q) fa[q] += fb[q];
        Ops::store(out + v * VEC, Ops::from_f32(fa));
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One CTA per row: residual_out = bf16(x + residual), then RMSNorm of
// residual_out (re-read from global memory: each thread reads back only the
// vectors it wrote).
template <int VEC>
__global__ void __launch_bounds__(kNormThreads)
residual_rmsnorm_kernel(const uint16_t *x, const uint16_t *residual, const uint16_t *gamma,
                        uint16_t *residual_out, uint16_t *norm_out, int nvec, int H,
                        float eps) {
    using Ops = VecOps<VEC>;
    __shared__ float s_warp[kNormThreads / 32];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t row = static_cast<int64_t>(blockIdx.x) * H;
    float ss = 0.f;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        const int64_t e = row + static_cast<int64_t>(v) * VEC;
        float fx[VEC], fr[VEC];
        Ops::to_f32(Ops::load(x + e), fx);
        Ops::to_f32(Ops::load(residual + e), fr);
#pragma unroll
        for (int q = 0; q < VEC; ++q) fx[q] += fr[q];
        const typename Ops::V s = Ops::from_f32(fx);
        Ops::store(residual_out + e, s);
        Ops::to_f32(s, fx);
#pragma unroll
        for (int q = 0; q < VEC; ++q) ss = fmaf(fx[q], fx[q], ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
    __syncthreads();
    float total = 0.f;
    for (int w = 0; w < static_cast<int>((blockDim.x + 31) >> 5); ++w) total += s_warp[w];
    const float inv = rsqrtf(total / static_cast<float>(H) + eps);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        const int64_t e = row + static_cast<int64_t>(v) * VEC;
        float fs[VEC], fg[VEC];
        Ops::to_f32(Ops::load(residual_out + e), fs);
        Ops::to_f32(Ops::load_reused(gamma + static_cast<int64_t>(v) * VEC), fg);
#pragma unroll
        for (int q = 0; q < VEC; ++q) fs[q] = fs[q] * inv * fg[q];
        Ops::store(norm_out + e, Ops::from_f32(fs));
    }
}

cudaError_t launch_pdl(const void *kernel, dim3 grid, dim3 block, void **args,
                       cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

template <int VEC>
cudaError_t launch_all(const FinalizeParams &p, const moef_plan &plan, uint16_t *tmp,
                       int num_sms, cudaStream_t stream) {
    FinalizeParams pc = p;
    void *cargs[] = {&pc, &tmp};
    cudaError_t err = launch_pdl(reinterpret_cast<const void *>(&combine_kernel<VEC>),
                                 dim3(static_cast<unsigned>(plan.grid)), dim3(plan.threads),
                                 cargs, stream);
    if (err != cudaSuccess) return err;

    const int64_t n = static_cast<int64_t>(p.T) * p.nvec;
    int64_t blocks = (n + kAddThreads - 1) / kAddThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    const uint16_t *a = tmp;
    const uint16_t *b = p.shared;
    uint16_t *out = p.out;
    int64_t nn = n;
    void *aargs[] = {&a, &b, &out, &nn};
    err = launch_pdl(reinterpret_cast<const void *>(&add_kernel<VEC>),
                     dim3(static_cast<unsigned>(blocks)), dim3(kAddThreads), aargs, stream);
    if (err != cudaSuccess || !p.residual) return err;

    const uint16_t *x = p.out;
    const uint16_t *res = p.residual;
    const uint16_t *g = p.gamma;
    uint16_t *ro = p.residual_out;
    uint16_t *no = p.norm_out;
    int nvec = p.nvec;
    int H = p.H;
    float eps = p.eps;
    void *nargs[] = {&x, &res, &g, &ro, &no, &nvec, &H, &eps};
    return launch_pdl(reinterpret_cast<const void *>(&residual_rmsnorm_kernel<VEC>),
                      dim3(static_cast<unsigned>(p.T)), dim3(kNormThreads), nargs, stream);
}

}  // namespace

cudaError_t launch_unfused(const FinalizeParams &p, const moef_plan &plan, uint16_t *tmp,
                           int num_sms, cudaStream_t stream) {
    if (plan.vec == 8) return launch_all<8>(p, plan, tmp, num_sms, stream);
    if (plan.vec == 1) return launch_all<1>(p, plan, tmp, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace moef
