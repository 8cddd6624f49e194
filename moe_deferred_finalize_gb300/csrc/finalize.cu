// Deferred MoE finalize kernel for sm_103a.
//
// One CTA finalizes one slice of one token row:
//
//   m = sum_k (w[t,k] * routed_scale) * permuted_out[idx[t,k], slice]
//       + shared_out[t, slice]
//   out = bf16(m);  with a residual: residual_out = bf16(m + residual),
//   norm_out = bf16(residual_out * rsqrt(mean(residual_out^2) + eps) * gamma)
//
// ("Support deferred MoE finalize for MXFP4 and FP8 block-scale",
// Motivation and Modifications item 2; "[Kimi K2.5] Fuse deferred MoE
// finalize into next-layer AR + residual + RMSNorm", Summary.)
//
// Memory plan: the path is an HBM-bound gather-reduce (about 0.4 flop per
// byte), so there is no tensor-core work.  Each thread owns whole 16-byte
// vectors (8 bf16 values) of the row; for every vector it issues the K
// gathered-row loads back to back (read-only path, no L1 allocation: each
// gathered byte is read exactly once), plus the shared and residual loads,
// and accumulates in fp32 registers.  Outputs are written with streaming
// stores.  The token's row indices and scaled weights are staged once in
// shared memory.  With RMSNorm the bf16-rounded residual_out vectors are kept
// in shared memory between the two passes (each thread its own column, so
// no barrier is needed; in registers they cost 32 registers per thread and
// halved the resident CTAs, and with them the loads in flight).  The sum of
// squares is reduced with warp shuffles and shared memory, and across the
// CTAs of a split row through distributed shared memory of a thread-block
// cluster (every CTA adds the partials in the same order, so all slices use
// the same inverse RMS).
//
// Two builds of every launch shape: one for the common top-8 routing, with
// K fixed at compile time, and one for any K.  With K fixed the compiler
// needs 40-56 registers instead of 64, so more CTAs fit an SM, which pays
// on larger grids: with RMSNorm from one CTA per SM (T = 48: 3.98 vs 4.04
// us; T = 96: 5.17 vs 5.53 us), without it from four (T = 96: 3.81 vs 3.87
// us; T = 128: 4.26 vs 4.43 us).  On smaller grids the time is a chain of
// memory latencies, and there the any-K build, which issues all of a
// vector's K row loads before its first FMA, is faster (T = 1: 2.37 vs 2.68
// us; without RMSNorm T = 32: 2.79 vs 3.10 us).  Both sum the K terms in
// the same order, so their results are bit-identical.
//
// Launch order: the kernel is a programmatic dependent of the previous
// kernel on the stream.  It touches global memory only after
// griddepcontrol.wait (the row map and weights may come first when the
// caller vouches that no earlier kernel still writes them), and it lets the
// next kernel start launching once its gathered loads are done.  No thread
// ever spins: the only waits are barriers.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <atomic>

#include "internal.cuh"
#include "vec.cuh"

namespace cg = cooperative_groups;

namespace moef {
namespace {

constexpr int kMaxThreads = 256;
constexpr int kMaxClusterCtas = 16;

// fp32 vector store: 8 values as two 16-byte stores, or one value.
template <int VEC>
__device__ __forceinline__ void store_f32(float *q, const float (&f)[VEC]) {
    if constexpr (VEC == 8) {
        reinterpret_cast<float4 *>(q)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4 *>(q)[1] = make_float4(f[4], f[5], f[6], f[7]);
    } else {
        q[0] = f[0];
    }
}

// KC: the slot count K when fixed at compile time, else 0 (K from p.K).
// F32: m is stored unrounded to p.out_f32 (fp32) instead of out (one
// tensor-parallel rank's partial, without residual or RMSNorm).
template <int VPT, int VEC, bool NORM, bool CLUSTER, int KC, bool F32>
__global__ void __launch_bounds__(kMaxThreads)
finalize_kernel(const __grid_constant__ FinalizeParams p) {
    using Ops = VecOps<VEC>;
    using V = typename Ops::V;

    __shared__ const uint16_t *s_row[MOEF_MAX_K];
    __shared__ float s_w[MOEF_MAX_K];
    __shared__ float s_warp[kMaxThreads / 32];
    __shared__ float s_part[kMaxClusterCtas];   // partial sums of the cluster's CTAs
    // With RMSNorm: the bf16 residual_out vectors of this CTA's slice, kept
    // for the second pass ([VPT][blockDim.x], each thread its own column).
    extern __shared__ __align__(16) unsigned char s_dyn[];
    V *s_keep = reinterpret_cast<V *>(s_dyn);

    // Cluster CTAs write into each other's shared memory below, which is
    // only allowed once every CTA of the cluster has started: announce it now
    // (non-blocking) and wait for the others just before the first remote write.
    if constexpr (CLUSTER) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    const int S = p.splits;
    const int t = blockIdx.x / S;
    const int split = blockIdx.x - t * S;
    const int K = KC ? KC : p.K;
    const int nt = blockDim.x;

    const int64_t tok = static_cast<int64_t>(t) * p.H;
    const int v_begin = split * p.slice;
    const int v_end = min(v_begin + p.slice, p.nvec);

    // Stage the token's row pointers and scaled weights (the routed scale
    // folded into the weight once, "Support deferred MoE finalize ...",
    // Modifications item 2).
    const bool stage = threadIdx.x < K;
    int r = 0;
    float w = 0.f;
    const int64_t slot = static_cast<int64_t>(t) * K + threadIdx.x;
    // The routing inputs may be read before the grid dependency wait when the
    // caller says no earlier kernel still writes them.
    if (p.routing_ready && stage) {
        r = __ldg(p.idx + slot);
        w = decode_weight(p.weights, p.wkind, slot);
    }

    // Launched as a programmatic dependent of the previous kernel on the
    // stream: nothing else before this point touches global memory, so the
    // launch and CTA set-up overlap the previous kernel's tail, and every read
    // and write below sees it complete.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (!p.routing_ready && stage) {
        r = __ldg(p.idx + slot);
        w = decode_weight(p.weights, p.wkind, slot);
    }
    // This thread's first dense operands do not depend on the row map: their
    // loads go out before the staging barrier, beside the row-map loads.
    const int v_first = v_begin + threadIdx.x;
    V sh_first, rs_first;
    if (v_first < v_end) {
        sh_first = Ops::load(p.shared + tok + static_cast<int64_t>(v_first) * VEC);
        if (NORM) rs_first = Ops::load(p.residual + tok + static_cast<int64_t>(v_first) * VEC);
    }
    if (stage) {
        s_row[threadIdx.x] = p.x + static_cast<int64_t>(r) * p.H;
        s_w[threadIdx.x] = w * p.routed_scale;
    }
    __syncthreads();

    float ss = 0.f;

    for (int base = v_begin; base < v_end; base += nt * VPT) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = base + threadIdx.x + j * nt;
            if (v < v_end) {
                const int64_t e = static_cast<int64_t>(v) * VEC;
                const bool first = (j == 0) && (base == v_begin);
                const V sh = first ? sh_first : Ops::load(p.shared + tok + e);
                V rs;
                if (NORM) rs = first ? rs_first : Ops::load(p.residual + tok + e);

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
                float f[VEC];
                Ops::to_f32(sh, f);
#pragma unroll
                for (int q = 0; q < VEC; ++q) acc[q] += f[q];
                if constexpr (F32) {
                    store_f32<VEC>(p.out_f32 + tok + e, acc);
                } else if (p.out) {
                    Ops::store(p.out + tok + e, Ops::from_f32(acc));
                }
                if (NORM) {
                    Ops::to_f32(rs, f);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) acc[q] += f[q];
                    const V sv = Ops::from_f32(acc);
                    Ops::store(p.residual_out + tok + e, sv);
                    s_keep[j * nt + threadIdx.x] = sv;
                    Ops::to_f32(sv, f);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) ss = fmaf(f[q], f[q], ss);
                }
            }
        }
        if (NORM) break;   // the plan gives a norm row slice one pass
    }
    // All gathered loads of this CTA are done: the next kernel on the stream
    // may begin launching (it waits for this grid before touching memory).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if constexpr (NORM) {
        // gamma loads go out before the reductions so their latency overlaps
        V g[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = v_begin + threadIdx.x + j * nt;
            if (v < v_end) g[j] = Ops::load_reused(p.gamma + static_cast<int64_t>(v) * VEC);
        }

        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
        __syncthreads();
        float total = 0.f;
        const int nw = (nt + 31) >> 5;
        for (int w = 0; w < nw; ++w) total += s_warp[w];

        if constexpr (CLUSTER) {
            // Push this CTA's partial into slot [own rank] of every CTA of the
            // cluster (thread r writes to CTA r), then one cluster barrier
            // (release/acquire) makes all S partials visible locally.  No CTA
            // touches another's shared memory after the barrier, so each may
            // leave when done.
            cg::cluster_group cluster = cg::this_cluster();
            const unsigned own = cluster.block_rank();
            asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // all CTAs started
            if (threadIdx.x < static_cast<unsigned>(S))
                *cluster.map_shared_rank(&s_part[own], static_cast<int>(threadIdx.x)) = total;
            cluster.sync();
            total = 0.f;
            for (int r = 0; r < S; ++r) total += s_part[r];    // same order in every CTA
        }

        const float inv = rsqrtf(total / static_cast<float>(p.H) + p.eps);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = v_begin + threadIdx.x + j * nt;
            if (v < v_end) {
                float sf[VEC], gf[VEC];
                Ops::to_f32(s_keep[j * nt + threadIdx.x], sf);
                Ops::to_f32(g[j], gf);
#pragma unroll
                for (int q = 0; q < VEC; ++q) sf[q] = sf[q] * inv * gf[q];
                Ops::store(p.norm_out + tok + static_cast<int64_t>(v) * VEC, Ops::from_f32(sf));
            }
        }
    }
}

constexpr int kFixedK = 8;

template <int VPT, int VEC, bool NORM, bool CLUSTER, bool F32 = false>
cudaError_t launch_t(const FinalizeParams &p, const moef_plan &plan, int num_sms,
                     cudaStream_t stream) {
    const int64_t fixed_k_grid = static_cast<int64_t>(num_sms) * (NORM ? 1 : 4);
    const int fixed_k = (p.K == kFixedK && plan.grid > fixed_k_grid) ? 1 : 0;
    auto kern = fixed_k ? finalize_kernel<VPT, VEC, NORM, CLUSTER, kFixedK, F32>
                        : finalize_kernel<VPT, VEC, NORM, CLUSTER, 0, F32>;
    cudaLaunchAttribute attr[2];
    unsigned num_attrs = 0;
    if (p.pdl) {
        attr[num_attrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[num_attrs].val.programmaticStreamSerializationAllowed = 1;
        ++num_attrs;
    }
    if (CLUSTER) {
        if (plan.cluster > 8) {
            // Clusters of 9..16 CTAs are opt-in per kernel and device (setting
            // the attribute twice from racing host threads is harmless).
            static std::atomic<int> enabled[2][64];
            int dev = 0;
            cudaError_t err = cudaGetDevice(&dev);
            if (err != cudaSuccess) return err;
            if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
            std::atomic<int> &done = enabled[fixed_k][dev];
            if (!done.load(std::memory_order_relaxed)) {
                err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (err != cudaSuccess) return err;
                done.store(1, std::memory_order_relaxed);
            }
        }
        attr[num_attrs].id = cudaLaunchAttributeClusterDimension;
        attr[num_attrs].val.clusterDim.x = static_cast<unsigned>(plan.cluster);
        attr[num_attrs].val.clusterDim.y = 1;
        attr[num_attrs].val.clusterDim.z = 1;
        ++num_attrs;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(plan.threads));
    cfg.dynamicSmemBytes =
        NORM ? static_cast<size_t>(plan.threads) * VPT * sizeof(typename VecOps<VEC>::V) : 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = num_attrs;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int VPT, int VEC>
cudaError_t launch_v(const FinalizeParams &p, const moef_plan &plan, int num_sms,
                     cudaStream_t stream) {
    if (p.out_f32) {
        if (p.residual) return cudaErrorInvalidValue;
        return launch_t<VPT, VEC, false, false, true>(p, plan, num_sms, stream);
    }
    if (!p.residual) return launch_t<VPT, VEC, false, false>(p, plan, num_sms, stream);
    if (plan.cluster > 1) return launch_t<VPT, VEC, true, true>(p, plan, num_sms, stream);
    return launch_t<VPT, VEC, true, false>(p, plan, num_sms, stream);
}

template <int VEC>
cudaError_t launch_vec(const FinalizeParams &p, const moef_plan &plan, int num_sms,
                       cudaStream_t stream) {
    switch (plan.vpt) {
        case 1: return launch_v<1, VEC>(p, plan, num_sms, stream);
        case 2: return launch_v<2, VEC>(p, plan, num_sms, stream);
        case 4: return launch_v<4, VEC>(p, plan, num_sms, stream);
        case 8: return launch_v<8, VEC>(p, plan, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_finalize(const FinalizeParams &p, const moef_plan &plan, int num_sms,
                            cudaStream_t stream) {
    // The RMSNorm form makes one pass over its slice (the sum of squares of
    // the whole row must be complete before the second pass), so its plan
    // must give every vector of the slice a thread in that pass.
    if (p.residual && static_cast<int64_t>(plan.threads) * plan.vpt < plan.slice)
        return cudaErrorInvalidValue;
    if (plan.vec == 8) return launch_vec<8>(p, plan, num_sms, stream);
    if (plan.vec == 1) return launch_vec<1>(p, plan, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace moef
