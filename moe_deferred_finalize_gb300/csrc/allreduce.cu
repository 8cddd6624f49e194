// The deferred finalize of R tensor-parallel ranks, summed over the ranks,
// then the residual add and RMSNorm ("[Kimi K2.5] Fuse deferred MoE finalize
// into next-layer AR + residual + RMSNorm", Summary: weighted expert combine
// + shared-expert add + all-reduce + residual + RMSNorm in one kernel, with
// residual_out kept; Numerics & speed: the same result from a standalone
// finalize followed by an all-reduce fused with residual + RMSNorm):
//
//   p_r = sum_k (w_r[t,k] * routed_scale) * x_r[idx_r[t,k], :] + shared_r[t, :]
//   m   = p_0 + p_1 + ... + p_{R-1}          (in rank order, fp32)
//   out = bf16(m);  residual_out = bf16(m + residual);
//   norm_out = bf16(residual_out * rsqrt(mean(residual_out^2) + eps) * gamma)
//
// The kernel templates here serve two entry points:
//   * one-shot (moe_finalize_allreduce): every rank's rows are gathered in
//     one launch, from local or peer-mapped memory;
//   * phase 2 (moe_finalize_allreduce_reduce): the fp32 partials of all
//     ranks summed, then the epilogue.
// Phase 1 (moe_finalize_partial, one rank's p_r stored in fp32) is the plain
// finalize kernel's fp32-output build: the same fp32 operations on each
// element in the same order as a rank's partial here.  The one-shot and the
// two-phase forms therefore run the same arithmetic in the same order, and
// phase 2 keeps the one-shot's launch plan, so their results are
// bit-identical.
//
// Thread layout of the one-shot kernels: a CTA's
// threads form `lanes` groups of `nvc` threads, and group g works for the
// R / lanes consecutive ranks from g * R / lanes on.  In one pass thread
// (g, j) obtains its ranks' partials of vector j of the CTA's slice one
// after another (per rank K gathered-row loads, 16 bytes each, plus the
// shared-output load), so a pass keeps `lanes` times as many loads in flight
// as one thread summing all ranks would.  Group 0 adds its own ranks'
// partials in registers and the other groups' from shared memory, in rank
// order, and finishes the vector.
// Decode sizes use lanes = R (or R / 2 from 8 tokens on when R > 4, and 2
// from 44 tokens on when R >= 6); with many tokens, enough vectors to fill
// the GPU, lanes = 1: each thread sums all ranks itself, with no exchange or
// barrier per pass.  Phase 2 of a
// one-rank-per-group plan runs in the same groups over the fp32 partials;
// phase 2 of the other plans runs a kernel of its own over the same
// vector-to-thread map, each finishing thread loading the R partials of its
// vector itself (all at once, or four at a time for grids too large to be
// resident at once).  With RMSNorm the bf16 residual_out vectors stay in shared
// memory for the second pass, and a split row combines its partial sums of
// squares across the CTAs of a thread-block cluster through distributed
// shared memory, as in the plain finalize.  The finishing threads, their
// vectors, passes and warps are the same in every form of one plan, and so
// is the order of the sum of squares: the forms' results are bit-identical.
//
// Launch order: a programmatic dependent of the previous kernel on the
// stream (griddepcontrol.wait before any global memory access); it lets the
// next kernel begin launching once its loads are done.  No thread spins.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <atomic>

#include "internal.cuh"
#include "vec.cuh"

namespace cg = cooperative_groups;

namespace moef {
namespace {

constexpr int kArMaxThreads = 512;
constexpr int kArMaxCluster = 16;
constexpr int kMaxSlots = MOEF_MAX_RANKS * MOEF_MAX_K;

// fp32 vectors of the partials: 8 values as two 16-byte loads, or one.
template <int VEC>
struct F32Ops;

template <>
struct F32Ops<8> {
    static __device__ __forceinline__ void load(const float *p, float f[8]) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

template <>
struct F32Ops<1> {
    static __device__ __forceinline__ void load(const float *p, float f[1]) { f[0] = __ldcs(p); }
};

// Rank r's entry of a per-rank pointer array of the kernel parameters.  Each
// entry is read with a compile-time index (a constant-bank operand) and the
// rank's one selected, instead of indexing the parameter array with a
// run-time rank, which would turn every such read into a dependent load.
template <typename T>
__device__ __forceinline__ T rank_entry(const T (&a)[MOEF_MAX_RANKS], int r) {
    T v = a[0];
#pragma unroll
    for (int i = 1; i < MOEF_MAX_RANKS; ++i)
        if (r == i) v = a[i];
    return v;
}

// Rank partial of one vector at element offset e: sum_k (w_k * row_k) as fp32
// FMAs in slot order, then the rank's shared output added.
template <int VEC>
__device__ __forceinline__ void rank_partial(const uint16_t *const *rows, const float *ws, int K,
                                             int64_t e, const typename VecOps<VEC>::V &sh,
                                             float (&acc)[VEC]) {
    using Ops = VecOps<VEC>;
    using V = typename Ops::V;
#pragma unroll
    for (int u = 0; u < VEC; ++u) acc[u] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 8) {
        V xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (k0 + u < K) xv[u] = Ops::load_row(rows[k0 + u] + e);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (k0 + u < K) {
                float xf[VEC];
                Ops::to_f32(xv[u], xf);
                const float w = ws[k0 + u];
#pragma unroll
                for (int c = 0; c < VEC; ++c) acc[c] = fmaf(w, xf[c], acc[c]);
            }
        }
    }
    float f[VEC];
    Ops::to_f32(sh, f);
#pragma unroll
    for (int c = 0; c < VEC; ++c) acc[c] += f[c];
}

// The finishing thread's epilogue of one rank-summed vector `acc` at element
// offset `at`: out, then with RMSNorm the residual add, residual_out, the
// kept bf16 vector and its sum of squares.
template <int VEC, bool NORM>
__device__ __forceinline__ void finish_vector(const ArParams &p, int64_t at, float (&acc)[VEC],
                                              const typename VecOps<VEC>::V &rs,
                                              typename VecOps<VEC>::V *keep, float &ss) {
    using Ops = VecOps<VEC>;
    if (p.out) Ops::store(p.out + at, Ops::from_f32(acc));
    if constexpr (NORM) {
        float f[VEC];
        Ops::to_f32(rs, f);
#pragma unroll
        for (int c = 0; c < VEC; ++c) acc[c] += f[c];
        const typename Ops::V sv = Ops::from_f32(acc);
        Ops::store(p.residual_out + at, sv);
        *keep = sv;
        Ops::to_f32(sv, f);
#pragma unroll
        for (int c = 0; c < VEC; ++c) ss = fmaf(f[c], f[c], ss);
    }
}

// RMSNorm of a CTA's kept residual_out vectors.  The row's sum of squares:
// each thread's own (its passes in order), warp shuffles, the CTA's warps in
// order, then with CLUSTER every CTA pushes its partial into slot [own rank]
// of every CTA of the cluster and one release/acquire cluster barrier; then
// norm_out.  Every thread of the CTA takes part; `finisher` marks those that
// hold vectors (thread j of a pass holds vector v_begin + q * nvc + j).
template <int VEC, bool CLUSTER, int PASSES>
__device__ __forceinline__ void norm_tail(const ArParams &p, bool finisher, int j, int v_begin,
                                          int v_end, int64_t tok,
                                          const typename VecOps<VEC>::V *s_keep, float ss,
                                          float *s_warp, float *s_part) {
    using Ops = VecOps<VEC>;
    using V = typename Ops::V;
    const int nvc = p.nvc;
    V g[PASSES];
#pragma unroll
    for (int qq = 0; qq < PASSES; ++qq) {
        const int v = v_begin + qq * nvc + j;
        if (finisher && v < v_end)
            g[qq] = Ops::load_reused(p.gamma + static_cast<int64_t>(v) * VEC);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
    __syncthreads();
    float total = 0.f;
    const int nw = (blockDim.x + 31) >> 5;
    for (int w = 0; w < nw; ++w) total += s_warp[w];

    if constexpr (CLUSTER) {
        cg::cluster_group cluster = cg::this_cluster();
        const unsigned own = cluster.block_rank();
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        if (threadIdx.x < static_cast<unsigned>(p.splits))
            *cluster.map_shared_rank(&s_part[own], static_cast<int>(threadIdx.x)) = total;
        cluster.sync();
        total = 0.f;
        for (int c = 0; c < p.splits; ++c) total += s_part[c];
    }

    const float inv = rsqrtf(total / static_cast<float>(p.H) + p.eps);
    if (finisher) {
#pragma unroll
        for (int qq = 0; qq < PASSES; ++qq) {
            const int v = v_begin + qq * nvc + j;
            if (v < v_end) {
                float sf[VEC], gf[VEC];
                Ops::to_f32(s_keep[qq * nvc + j], sf);
                Ops::to_f32(g[qq], gf);
#pragma unroll
                for (int c = 0; c < VEC; ++c) sf[c] = sf[c] * inv * gf[c];
                Ops::store(p.norm_out + tok + static_cast<int64_t>(v) * VEC, Ops::from_f32(sf));
            }
        }
    }
}

// One rank per group (lanes = R): the one-shot call (every rank's rows),
// and, with p.reduce, phase 2 of the same plans over the ranks' fp32 partials, a thread per rank and vector
// keeping the partials' loads spread over the CTA.  Every group's partial of
// a pass meets group 0 in shared memory.
// PASSES: with RMSNorm, the number of passes over the slice (1, 2, 4 or 8),
// fixed so that the gamma vectors can be held in registers; 0 without
// RMSNorm (any number of passes).
// MINB: CTAs of 512 threads that must fit one SM.  2 (64 registers) for
// grids above one CTA per SM, where resident warps hide latency; 1 (up to
// 128 registers) for smaller grids, whose time is a chain of memory
// latencies: there the registers let every gathered load of a vector go out
// before the first FMA, while 64 registers with RMSNorm spill and split them.
// (Measured on GB300: building the one-shot-only form of this kernel,
// without the phase-2 branch, made the decode calls 0.1-0.35 us slower.)
// KC: K when fixed at compile time (top-8), else 0.
template <int VEC, bool NORM, bool CLUSTER, int PASSES, int MINB, int KC>
__global__ void __launch_bounds__(kArMaxThreads, MINB)
finalize_ar_kernel(const __grid_constant__ ArParams p) {
    using Ops = VecOps<VEC>;
    using FOps = F32Ops<VEC>;
    using V = typename Ops::V;

    __shared__ const uint16_t *s_row[kMaxSlots];   // [rank][slot]
    __shared__ float s_w[kMaxSlots];
    __shared__ float s_warp[kArMaxThreads / 32];
    __shared__ float s_part[kArMaxCluster];
    // dynamic: the ranks' partials of one pass, float [lanes][nvc][VEC]
    // (lanes > 1), then with RMSNorm the kept residual_out vectors, V [PASSES][nvc]
    extern __shared__ __align__(16) unsigned char s_dyn[];
    const int lanes = p.lanes;
    const int nvc = p.nvc;
    float *s_p = reinterpret_cast<float *>(s_dyn);
    V *s_keep = reinterpret_cast<V *>(s_dyn + (lanes > 1 ? sizeof(float) * VEC * lanes * nvc : 0));

    if constexpr (CLUSTER) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    const int r = threadIdx.x / nvc;        // the rank this thread works for
    const int j = threadIdx.x - r * nvc;    // its vector within a pass
    const int S = p.splits;
    const int t = blockIdx.x / S;
    const int split = blockIdx.x - t * S;
    const int K = KC ? KC : p.K;
    const int64_t tok = static_cast<int64_t>(t) * p.H;
    const int v_begin = split * p.slice;
    const int v_end = min(v_begin + p.slice, p.nvec);
    const bool gather = p.reduce == 0;
    // this thread's rank's dense operand: its shared output (gather) or its
    // fp32 partial (phase 2)
    const void *dense_r = gather ? static_cast<const void *>(rank_entry(p.shared, r))
                                 : static_cast<const void *>(rank_entry(p.partial, r));

    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (gather) {
        // every rank's row pointers and scaled weights for this token
        const int nslots = lanes * K;
        for (int i = threadIdx.x; i < nslots; i += blockDim.x) {
            const int rr = i / K;
            const int64_t slot = static_cast<int64_t>(t) * K + (i - rr * K);
            const int row = __ldg(rank_entry(p.idx, rr) + slot);
            s_row[i] = rank_entry(p.x, rr) + static_cast<int64_t>(row) * p.H;
            s_w[i] = decode_weight(rank_entry(p.weights, rr), p.wkind, slot) * p.routed_scale;
        }
    }
    // The first pass's dense operands do not depend on the staged pointers:
    // their loads go out before the staging barrier, beside the row-map
    // loads (the finishing threads' residual; in the small-grid build, whose
    // time is a chain of latencies and which has the registers for it, also
    // this thread's rank's shared output or fp32 partial).
    constexpr bool kHoist = MINB == 1;
    V sh_first, rs_first;
    float part_first[VEC];
    if (v_begin + j < v_end) {
        const int64_t e = static_cast<int64_t>(v_begin + j) * VEC;
        if (kHoist && gather)
            sh_first = Ops::load(static_cast<const uint16_t *>(dense_r) + tok + e);
        else if (kHoist)
            FOps::load(static_cast<const float *>(dense_r) + tok + e, part_first);
        if (NORM && r == 0) rs_first = Ops::load(p.residual + tok + e);
    }
    __syncthreads();

    float ss = 0.f;
    int q = 0;
    for (int base = v_begin; base < v_end; base += nvc, ++q) {
        const int v = base + j;
        const bool active = v < v_end;
        const int64_t e = static_cast<int64_t>(v) * VEC;
        float acc[VEC];
        if (active) {
            if (gather) {
                const V sh = (kHoist && q == 0)
                                 ? sh_first
                                 : Ops::load(static_cast<const uint16_t *>(dense_r) + tok + e);
                rank_partial<VEC>(s_row + r * K, s_w + r * K, K, e, sh, acc);
            } else if (kHoist && q == 0) {
#pragma unroll
                for (int c = 0; c < VEC; ++c) acc[c] = part_first[c];
            } else {
                FOps::load(static_cast<const float *>(dense_r) + tok + e, acc);
            }
        }
        if (lanes > 1) {
            float *mine = s_p + (static_cast<int64_t>(r) * nvc + j) * VEC;
            if (active) {
#pragma unroll
                for (int c = 0; c < VEC; ++c) mine[c] = acc[c];
            }
            __syncthreads();
            if (r == 0 && active) {
                for (int rr = 1; rr < lanes; ++rr) {
                    const float *other = s_p + (static_cast<int64_t>(rr) * nvc + j) * VEC;
#pragma unroll
                    for (int c = 0; c < VEC; ++c) acc[c] += other[c];
                }
            }
            if (base + nvc < v_end) __syncthreads();   // s_p is refilled by the next pass
        }
        if (r == 0 && active) {
            V rs{};
            if constexpr (NORM) rs = (q == 0) ? rs_first : Ops::load(p.residual + tok + e);
            finish_vector<VEC, NORM>(p, tok + e, acc, rs, s_keep + q * nvc + j, ss);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if constexpr (NORM)
        norm_tail<VEC, CLUSTER, PASSES>(p, r == 0, j, v_begin, v_end, tok, s_keep, ss, s_warp,
                                        s_part);
}

// Groups of several ranks, gathering only (one-shot), 16-byte vectors:
// MODE kRankGroups (1 < lanes < R: group g sums its c = R / lanes ranks
// g*c .. g*c + c - 1 one after the other; groups other than 0 store each
// rank's partial, and group 0 adds ranks c .. R-1 from shared memory in rank
// order) or kAllRanks (lanes = 1: each thread sums every rank's partial in
// rank order itself, no exchange).
enum { kRankGroups = 1, kAllRanks = 2 };

// KC: K when fixed at compile time (top-8: no predicated slots, and the
// rank-group build then fits 64 registers without spilling), else 0.
template <int VEC, bool NORM, bool CLUSTER, int PASSES, int MODE, int KC>
__global__ void __launch_bounds__(kArMaxThreads, 2)
finalize_ar_multi_kernel(const __grid_constant__ ArParams p) {
    using Ops = VecOps<VEC>;
    using V = typename Ops::V;

    __shared__ const uint16_t *s_row[kMaxSlots];       // [rank][slot]
    __shared__ float s_w[kMaxSlots];
    __shared__ const uint16_t *s_sh[MOEF_MAX_RANKS];   // each rank's shared-output row
    __shared__ float s_warp[kArMaxThreads / 32];
    __shared__ float s_part[kArMaxCluster];
    const int nvc = p.nvc;
    const int R = p.ranks;
    // ranks per group: R / lanes (2 or R / 2), a run-time count (measured
    // faster in this kernel than a constant 2 for pairs), or all R
    const int c = MODE == kRankGroups ? R / p.lanes : R;
    // dynamic: the partials of ranks c .. R-1 for one pass, float
    // [R - c][nvc][VEC]; then with RMSNorm the kept residual_out vectors, V [PASSES][nvc]
    extern __shared__ __align__(16) unsigned char s_dyn[];
    float *s_p = reinterpret_cast<float *>(s_dyn);
    V *s_keep = reinterpret_cast<V *>(s_dyn + sizeof(float) * VEC * (R - c) * nvc);

    if constexpr (CLUSTER) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    const int g = MODE == kRankGroups ? threadIdx.x / nvc : 0;   // this thread's group
    const int j = threadIdx.x - g * nvc;                        // its vector within a pass
    const int r0 = g * c;                                       // the group's first rank
    const int S = p.splits;
    const int t = blockIdx.x / S;
    const int split = blockIdx.x - t * S;
    const int K = KC ? KC : p.K;
    const int64_t tok = static_cast<int64_t>(t) * p.H;
    const int v_begin = split * p.slice;
    const int v_end = min(v_begin + p.slice, p.nvec);

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // every rank's row pointers and scaled weights for this token, and its
    // shared-output row
    const int nslots = R * K;
    for (int i = threadIdx.x; i < nslots; i += blockDim.x) {
        const int rr = i / K;
        const int64_t slot = static_cast<int64_t>(t) * K + (i - rr * K);
        const int row = __ldg(rank_entry(p.idx, rr) + slot);
        s_row[i] = rank_entry(p.x, rr) + static_cast<int64_t>(row) * p.H;
        s_w[i] = decode_weight(rank_entry(p.weights, rr), p.wkind, slot) * p.routed_scale;
    }
    if (static_cast<int>(threadIdx.x) < R)
        s_sh[threadIdx.x] = rank_entry(p.shared, static_cast<int>(threadIdx.x)) + tok;
    V rs_first;
    if (NORM && g == 0 && v_begin + j < v_end)
        rs_first = Ops::load(p.residual + tok + static_cast<int64_t>(v_begin + j) * VEC);
    __syncthreads();

    float ss = 0.f;
    int q = 0;
    for (int base = v_begin; base < v_end; base += nvc, ++q) {
        const int v = base + j;
        const bool active = v < v_end;
        const int64_t e = static_cast<int64_t>(v) * VEC;
        float acc[VEC];
        if (active) {
            // the group's ranks one after the other: a loop that is not
            // unrolled, so a rank's loads wait for the previous rank's FMAs
            // (two ranks' loads in flight need more than 64 registers)
#pragma unroll 1
            for (int i = 0; i < c; ++i) {
                const int rr = r0 + i;
                float pr[VEC];
                rank_partial<VEC>(s_row + rr * K, s_w + rr * K, K, e, Ops::load(s_sh[rr] + e), pr);
                if (g == 0) {
#pragma unroll
                    for (int u = 0; u < VEC; ++u) acc[u] = i == 0 ? pr[u] : acc[u] + pr[u];
                } else {
                    float *mine = s_p + (static_cast<int64_t>(rr - c) * nvc + j) * VEC;
#pragma unroll
                    for (int u = 0; u < VEC; ++u) mine[u] = pr[u];
                }
            }
        }
        if constexpr (MODE == kRankGroups) {
            __syncthreads();
            if (g == 0 && active) {
                for (int rr = c; rr < R; ++rr) {
                    const float *other = s_p + (static_cast<int64_t>(rr - c) * nvc + j) * VEC;
#pragma unroll
                    for (int u = 0; u < VEC; ++u) acc[u] += other[u];
                }
            }
            if (base + nvc < v_end) __syncthreads();   // s_p is refilled by the next pass
        }
        if (g == 0 && active) {
            V rs{};
            if constexpr (NORM) rs = (q == 0) ? rs_first : Ops::load(p.residual + tok + e);
            finish_vector<VEC, NORM>(p, tok + e, acc, rs, s_keep + q * nvc + j, ss);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if constexpr (NORM)
        norm_tail<VEC, CLUSTER, PASSES>(p, g == 0, j, v_begin, v_end, tok, s_keep, ss, s_warp,
                                        s_part);
}

// Phase 2 of plans with groups of several ranks: the plan's finishing
// threads alone (nvc rounded up to whole warps), each loading the R fp32
// partials of its vector at once and adding them in rank order, then the
// epilogue.  No shared-memory exchange.
// MINB: 1 (up to 128 registers: every partial's load in flight at once) for
// grids that are resident all at once with that many registers; 2 (64
// registers, the partials loaded 4 at a time) for larger grids, which then
// fit twice as many CTAs per SM (R = 8, T = 256: 512 CTAs of 224 threads in
// one wave instead of two).
template <int VEC, bool NORM, bool CLUSTER, int PASSES, int MINB>
__global__ void __launch_bounds__(kArMaxThreads, MINB)
finalize_ar_reduce_kernel(const __grid_constant__ ArParams p) {
    using Ops = VecOps<VEC>;
    using FOps = F32Ops<VEC>;
    using V = typename Ops::V;

    __shared__ float s_warp[kArMaxThreads / 32];
    __shared__ float s_part[kArMaxCluster];
    // dynamic: with RMSNorm the kept residual_out vectors, V [PASSES][nvc]
    extern __shared__ __align__(16) unsigned char s_dyn[];
    V *s_keep = reinterpret_cast<V *>(s_dyn);

    if constexpr (CLUSTER) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    const int nvc = p.nvc;
    const int j = threadIdx.x;
    const bool finisher = j < nvc;
    const int S = p.splits;
    const int t = blockIdx.x / S;
    const int split = blockIdx.x - t * S;
    const int R = p.ranks;
    const int64_t tok = static_cast<int64_t>(t) * p.H;
    const int v_begin = split * p.slice;
    const int v_end = min(v_begin + p.slice, p.nvec);

    asm volatile("griddepcontrol.wait;" ::: "memory");

    float ss = 0.f;
    int q = 0;
    for (int base = v_begin; base < v_end; base += nvc, ++q) {
        const int v = base + j;
        if (finisher && v < v_end) {
            const int64_t at = tok + static_cast<int64_t>(v) * VEC;
            V rs{};
            if constexpr (NORM) rs = Ops::load(p.residual + at);
            float acc[VEC];
            FOps::load(p.partial[0] + at, acc);
            // the other ranks' partials in batches of kBatch loads in flight
            // (all at once with the registers of the small-grid build)
            constexpr int kBatch = MINB == 1 ? MOEF_MAX_RANKS - 1 : 4;
#pragma unroll
            for (int b0 = 1; b0 < MOEF_MAX_RANKS; b0 += kBatch) {
                float f[kBatch][VEC];
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    const int rr = b0 + i;
                    if (rr < MOEF_MAX_RANKS && rr < R) FOps::load(p.partial[rr] + at, f[i]);
                }
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    const int rr = b0 + i;
                    if (rr < MOEF_MAX_RANKS && rr < R) {
#pragma unroll
                        for (int c = 0; c < VEC; ++c) acc[c] += f[i][c];
                    }
                }
            }
            finish_vector<VEC, NORM>(p, at, acc, rs, s_keep + q * nvc + j, ss);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if constexpr (NORM)
        norm_tail<VEC, CLUSTER, PASSES>(p, finisher, j, v_begin, v_end, tok, s_keep, ss, s_warp,
                                        s_part);
}

// Launches `kern` over `grid` CTAs of `threads` threads as a programmatic
// dependent of the previous kernel on the stream, in clusters of `cluster`
// CTAs when cluster > 1.  `big` records, per device, that the kernel was
// allowed clusters above the portable 8 CTAs.
template <typename Kern>
cudaError_t launch_ar_kernel(Kern kern, std::atomic<int> (&big)[64], const ArParams &p,
                             int64_t grid, int threads, int smem, int cluster,
                             cudaStream_t stream) {
    cudaLaunchAttribute attr[2];
    unsigned num_attrs = 0;
    attr[num_attrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[num_attrs].val.programmaticStreamSerializationAllowed = 1;
    ++num_attrs;
    if (cluster > 1) {
        if (cluster > 8) {
            // clusters of 9..16 CTAs are opt-in per kernel and device
            int dev = 0;
            cudaError_t err = cudaGetDevice(&dev);
            if (err != cudaSuccess) return err;
            if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
            if (!big[dev].load(std::memory_order_relaxed)) {
                err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (err != cudaSuccess) return err;
                big[dev].store(1, std::memory_order_relaxed);
            }
        }
        attr[num_attrs].id = cudaLaunchAttributeClusterDimension;
        attr[num_attrs].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[num_attrs].val.clusterDim.y = 1;
        attr[num_attrs].val.clusterDim.z = 1;
        ++num_attrs;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = num_attrs;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// The multi-rank kernel (16-byte vectors): one thread summing all ranks
// (lanes = 1) or groups of several ranks.
template <bool NORM, bool CLUSTER, int PASSES, int KC>
cudaError_t launch_multi(const ArParams &p, const moef_ar_plan &plan, int cluster,
                         cudaStream_t stream) {
    static std::atomic<int> big[2][64];
    if (plan.lanes == 1)
        return launch_ar_kernel(finalize_ar_multi_kernel<8, NORM, CLUSTER, PASSES, kAllRanks, KC>,
                                big[1], p, plan.grid, plan.threads, plan.smem_bytes, cluster,
                                stream);
    return launch_ar_kernel(finalize_ar_multi_kernel<8, NORM, CLUSTER, PASSES, kRankGroups, KC>,
                            big[0], p, plan.grid, plan.threads, plan.smem_bytes, cluster, stream);
}

template <int VEC, bool NORM, bool CLUSTER, int PASSES>
cudaError_t launch_ar_t(const ArParams &p, const moef_ar_plan &plan, int num_sms,
                        cudaStream_t stream) {
    const int cluster = CLUSTER ? plan.cluster : 1;
    // the 128-register builds (one CTA of 512 threads per SM) for grids of
    // at most one CTA per SM whose clusters also fit: about 7 clusters of up
    // to 16 such CTAs are resident at once
    const int64_t rows = plan.grid / plan.splits;
    const bool small = plan.grid <= num_sms && (plan.threads <= 256 || rows <= 7);
    // phase 2 of a one-rank-per-group plan: in the finishing threads alone,
    // which load every rank's partial at once (R = 8, T = 1: 2.55 against
    // 2.69 us; T = 8: 2.91 against 3.23 us; R = 3, T = 32: 3.20 against 4.28
    // us; R = 2, T = 48: 3.32 against 4.44 us), except over small grids with
    // up to 3 ranks, where the rank groups measured 0.05 us faster
    if (plan.lanes == p.ranks && !(p.reduce && (!small || p.ranks >= 4))) {
        // one rank per group: gathering, or phase 2 in rank groups.  Top-8
        // gathers over large grids take the build with K fixed (R = 8, T = 8:
        // 6.09 -> 5.74 us; R = 4, T = 32: 7.03 -> 6.41 us); the small-grid
        // build, a chain of latencies, measured 0.2 us slower with it.
        static std::atomic<int> big[3][64];
        if (small)
            return launch_ar_kernel(finalize_ar_kernel<VEC, NORM, CLUSTER, PASSES, 1, 0>, big[1],
                                    p, plan.grid, plan.threads, plan.smem_bytes, cluster, stream);
        if (VEC == 8 && p.K == 8 && !p.reduce)
            return launch_ar_kernel(finalize_ar_kernel<VEC, NORM, CLUSTER, PASSES, 2, 8>, big[2],
                                    p, plan.grid, plan.threads, plan.smem_bytes, cluster, stream);
        return launch_ar_kernel(finalize_ar_kernel<VEC, NORM, CLUSTER, PASSES, 2, 0>, big[0], p,
                                plan.grid, plan.threads, plan.smem_bytes, cluster, stream);
    }
    if (p.reduce) {
        static std::atomic<int> big[2][64];
        const int threads = (plan.nvc + 31) / 32 * 32;
        const int smem =
            NORM ? PASSES * plan.nvc * static_cast<int>(sizeof(typename VecOps<VEC>::V)) : 0;
        const int64_t resident = static_cast<int64_t>(num_sms) * (65536 / (threads * 128));
        if (plan.grid <= resident)
            return launch_ar_kernel(finalize_ar_reduce_kernel<VEC, NORM, CLUSTER, PASSES, 1>,
                                    big[1], p, plan.grid, threads, smem, cluster, stream);
        return launch_ar_kernel(finalize_ar_reduce_kernel<VEC, NORM, CLUSTER, PASSES, 2>, big[0],
                                p, plan.grid, threads, smem, cluster, stream);
    }
    // groups of several ranks: planned for 16-byte vectors only
    if constexpr (VEC == 8) {
        if (plan.lanes == 1 || p.ranks % plan.lanes == 0) {
            if (p.K == 8)
                return launch_multi<NORM, CLUSTER, PASSES, 8>(p, plan, cluster, stream);
            return launch_multi<NORM, CLUSTER, PASSES, 0>(p, plan, cluster, stream);
        }
    }
    return cudaErrorInvalidValue;
}

template <int VEC, bool CLUSTER>
cudaError_t launch_ar_norm(const ArParams &p, const moef_ar_plan &plan, int num_sms,
                           cudaStream_t stream) {
    switch (plan.passes) {
        case 1: return launch_ar_t<VEC, true, CLUSTER, 1>(p, plan, num_sms, stream);
        case 2: return launch_ar_t<VEC, true, CLUSTER, 2>(p, plan, num_sms, stream);
        case 4: return launch_ar_t<VEC, true, CLUSTER, 4>(p, plan, num_sms, stream);
        case 8: return launch_ar_t<VEC, true, CLUSTER, 8>(p, plan, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int VEC>
cudaError_t launch_ar_vec(const ArParams &p, const moef_ar_plan &plan, int num_sms,
                          cudaStream_t stream) {
    if (!p.residual) return launch_ar_t<VEC, false, false, 0>(p, plan, num_sms, stream);
    if (plan.cluster > 1) return launch_ar_norm<VEC, true>(p, plan, num_sms, stream);
    return launch_ar_norm<VEC, false>(p, plan, num_sms, stream);
}

}  // namespace

cudaError_t launch_finalize_ar(const ArParams &p, const moef_ar_plan &plan, int num_sms,
                               cudaStream_t stream) {
    // the plan must match the parameters it is launched with: `lanes`
    // groups of nvc threads (lanes divides R), whole warps where the
    // RMSNorm epilogue shuffles, and with RMSNorm every vector of the slice
    // covered within the kernel's fixed number of passes
    if (p.ranks < 1 || p.ranks > MOEF_MAX_RANKS) return cudaErrorInvalidValue;
    if (plan.lanes != p.lanes || plan.lanes < 1 || p.ranks % plan.lanes != 0 ||
        plan.nvc != p.nvc || plan.threads != p.lanes * p.nvc || plan.threads > kArMaxThreads ||
        plan.splits != p.splits || plan.slice != p.slice)
        return cudaErrorInvalidValue;
    if (p.residual && (static_cast<int64_t>(plan.passes) * plan.nvc < plan.slice ||
                       plan.threads % 32 != 0))
        return cudaErrorInvalidValue;
    if (p.reduce == 0 && p.ranks * p.K > kMaxSlots) return cudaErrorInvalidValue;
    if (plan.vec == 8) return launch_ar_vec<8>(p, plan, num_sms, stream);
    if (plan.vec == 1) return launch_ar_vec<1>(p, plan, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace moef
