// C ABI of libmoe_finalize.so: argument checks, launch planning and the
// entry points declared in moe_finalize.h.  Host code only; every step of
// the computation runs in the kernels of finalize.cu and routing.cu.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "internal.cuh"

namespace {

constexpr int kMaxThreads = 256;   // matches the kernels' launch bounds
constexpr int kMaxVpt = 8;
constexpr int kMaxCluster = 16;    // non-portable cluster size limit
constexpr int kMaxDevices = 64;

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Smallest supported vectors-per-thread count >= need (1, 2, 4 or 8), or
// need itself when it is larger than 8.
int vpt_bucket(int need) {
    if (need <= 1) return 1;
    if (need <= 2) return 2;
    if (need <= 4) return 4;
    if (need <= 8) return 8;
    return need;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Multiprocessor count of the current device, cached per device (host
// threads may race to fill an entry; they all store the same value).
cudaError_t current_sms(int *sms) {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = cache[dev].load(std::memory_order_relaxed);
        if (cached > 0) {
            *sms = cached;
            return cudaSuccess;
        }
    }
    int n = 0;
    err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    *sms = n;
    return cudaSuccess;
}

// Status of a runtime call.  A refused call also leaves its error in the
// thread's last-error slot, where the caller's next unrelated launch check
// would find it; the error is reported here, so it is taken out of the slot.
moef_status cuda_status(cudaError_t err) {
    if (err == cudaSuccess) return MOEF_OK;
    (void)cudaGetLastError();
    return MOEF_ERR_CUDA;
}

}  // namespace

extern "C" {

int moef_abi_version(void) { return MOEF_ABI_VERSION; }

const char *moef_status_string(moef_status s) {
    switch (s) {
        case MOEF_OK: return "ok";
        case MOEF_ERR_NULL: return "a required pointer is NULL";
        case MOEF_ERR_SHAPE: return "a size is out of range";
        case MOEF_ERR_ALIGN: return "a pointer is not aligned to its element size";
        case MOEF_ERR_ARG: return "invalid argument (enum, scalar or optional-argument pairing)";
        case MOEF_ERR_CUDA: return "the CUDA runtime returned an error";
        case MOEF_ERR_INDEX: return "an index lies outside [0, P)";
    }
    return "unknown status";
}

// Plan choice, from sweeps of T = 1..4096 at H = 7168 on GB300 (graph
// replay, inputs larger than L2):
//  * without RMSNorm a row is cut into 128-vector slices, one CTA of 128
//    threads each, one vector per thread, at every T: at decode sizes every
//    gathered load of the call is then in flight at once (the time is a few
//    memory latencies), and at large T the many small CTAs avoid the wave
//    quantisation that whole-row CTAs hit (T = 1536: 32.1 vs 36.6 us).  When
//    that grid would need between one and two waves, 64-thread CTAs taking
//    two vectors each fit it in one (T = 256: 7.2 vs 7.7 us).
//  * with RMSNorm a row must be finished by one CTA or one cluster.  Rows
//    start as slices of at most 256 vectors (one per thread of a 256-thread
//    CTA, 4-CTA clusters at H = 7168).  The aim is a grid of one wave,
//    which held up to about 4.75 CTAs of 224 threads per SM, 4.25 of 256
//    threads and 7.5 of 128 threads (a step past that cost a wave more:
//    7.74 per SM fitted in 4-CTA clusters, not in 3-CTA ones).  So past
//    that size the same slices go to 128-thread CTAs with two vectors a
//    thread while those fit (H = 7168, T = 192 / 256: 8.52 / 9.68 -> 8.29 /
//    9.24 us; H = 5120, T = 300: 9.03 -> 8.80 us), unless a whole row fits
//    one CTA at two vectors a thread, which then wins without a cluster
//    (H = 4096, T = 400: 8.18 against 9.11 us); otherwise the split is
//    halved while the grid exceeds 4.25 CTAs per SM (H = 7168, T = 320:
//    12.36 -> 10.75 us against the former 3.5 per SM, which also halved
//    T = 144-176 too early: 7.56-8.30 -> 6.24-6.82 us); with no split one
//    CTA takes a whole row (256 threads below 4 rows per SM or for rows of
//    at most 512 vectors, then 128).
//    7-CTA clusters at T = 512 were 1.5x slower than this.  At H = 2048 and
//    4096, T = 2048, 256 threads beat 128 by 5.8 % and 2.9 %; at H = 5120
//    and 7168, 128 threads win.
// A row with RMSNorm must fit one pass of one CTA (256 x 8 vectors) or one
// cluster of at most 16 such CTAs.
moef_status moe_finalize_plan(int T, int K, int H, int with_norm, int vec_ok, int num_sms,
                              int splits_hint, int threads_hint, moef_plan *plan) {
    if (!plan) return MOEF_ERR_NULL;
    if (T < 0 || K < 1 || K > MOEF_MAX_K || H < 1) return MOEF_ERR_SHAPE;
    if (num_sms < 1 || splits_hint < 0 || threads_hint < 0) return MOEF_ERR_ARG;
    if (threads_hint && (threads_hint > kMaxThreads || threads_hint % 32)) return MOEF_ERR_ARG;

    const int vec = (vec_ok && H % 8 == 0) ? 8 : 1;
    const int nvec = H / vec;
    const int64_t rows = T > 0 ? T : 1;

    int splits;
    int threads_auto = 0;
    if (splits_hint) {
        splits = splits_hint < nvec ? splits_hint : nvec;
    } else if (with_norm) {
        const int row_fit = ceil_div(nvec, kMaxThreads * kMaxVpt);
        splits = ceil_div(nvec, kMaxThreads);
        // CTAs resident at once for a CTA size, in quarter CTAs per SM
        const auto fits_one_wave = [&](int64_t ctas, int threads) {
            const int64_t quarters = threads <= 128 ? 30 : threads <= 224 ? 19 : 17;
            return 4 * ctas <= quarters * static_cast<int64_t>(num_sms);
        };
        const int sl0 = ceil_div(nvec, splits);
        const int t0 = round_up(sl0 < kMaxThreads ? sl0 : kMaxThreads, 32);
        if (splits > 1 && splits <= kMaxCluster && !fits_one_wave(rows * splits, t0)) {
            if (t0 > 128 && nvec > 2 * kMaxThreads && fits_one_wave(rows * splits, 128)) {
                threads_auto = 128;    // the same slices, two vectors a thread
            } else {
                while (splits > row_fit && splits > 1 &&
                       !fits_one_wave(rows * splits, kMaxThreads))
                    splits = ceil_div(splits, 2);
            }
        }
        if (splits < row_fit) splits = row_fit;
        if (splits > kMaxCluster) splits = kMaxCluster;
        // one CTA per row: 256 threads below 4 rows per SM, and for rows of at
        // most 512 vectors (one or two per thread, all row loads in flight at
        // once); otherwise 128 threads with up to 8 vectors each
        if (splits == 1)
            threads_auto = (rows < 4 * static_cast<int64_t>(num_sms) || nvec <= 2 * kMaxThreads)
                               ? kMaxThreads
                               : 128;
    } else {
        // 128-vector slices; if that grid would need between one and two
        // waves of 128-thread CTAs (8 per SM at 64 registers), 64-thread CTAs
        // with two vectors each fit it in one wave instead.
        splits = ceil_div(nvec, 128);
        if (rows * splits > 0x7FFFFFFFLL) splits = static_cast<int>(0x7FFFFFFFLL / rows);
        if (splits < 1) splits = 1;
        const int64_t slots128 = static_cast<int64_t>(num_sms) * 8;
        const int64_t grid = rows * splits;
        if (!threads_hint && grid > slots128 && grid < 2 * slots128 && nvec >= 128)
            threads_auto = 64;
    }
    if (with_norm && splits > kMaxCluster) return MOEF_ERR_ARG;

    const int slice = ceil_div(nvec, splits);
    splits = ceil_div(nvec, slice);   // no empty CTAs

    int threads;
    if (threads_hint) {
        threads = threads_hint;
    } else if (threads_auto) {
        threads = threads_auto;
        if (ceil_div(slice, threads) > kMaxVpt) threads = kMaxThreads;
    } else {
        const int cap = splits > 1 ? kMaxThreads : 128;
        threads = round_up(slice < cap ? slice : cap, 32);
        if (ceil_div(slice, threads) > kMaxVpt) threads = kMaxThreads;
    }
    int vpt = vpt_bucket(ceil_div(slice, threads));
    if (vpt > kMaxVpt) {
        if (with_norm) return MOEF_ERR_SHAPE;
        vpt = kMaxVpt;     // several passes over the slice
    }

    const int64_t grid = static_cast<int64_t>(T) * splits;
    if (grid > 0x7FFFFFFFLL) return MOEF_ERR_SHAPE;

    plan->vec = vec;
    plan->splits = splits;
    plan->slice = slice;
    plan->threads = threads;
    plan->vpt = vpt;
    plan->cluster = (with_norm && splits > 1) ? splits : 1;
    plan->grid = grid;
    return MOEF_OK;
}

namespace {

// Checks shared by every finalize entry point; fills `p` (all but the plan
// fields) and reports whether the 16-byte path applies.
moef_status check_finalize_args(const void *permuted_out, int64_t P, const int32_t *idx_map,
                                const void *weights, moef_weight_kind wkind, float routed_scale,
                                const void *shared_out, const void *residual, const void *gamma,
                                float eps, void *out, void *residual_out, void *norm_out,
                                int T, int K, int H, moef::FinalizeParams *p, bool *vec_ok) {
    if (T < 0 || K < 1 || K > MOEF_MAX_K || H < 1) return MOEF_ERR_SHAPE;
    if (wkind != MOEF_W_FP32 && wkind != MOEF_W_BF16 && wkind != MOEF_W_PACKED_TOPK)
        return MOEF_ERR_ARG;
    if (T == 0) return MOEF_OK;
    if (P < 1) return MOEF_ERR_SHAPE;
    if (!permuted_out || !idx_map || !weights || !shared_out) return MOEF_ERR_NULL;

    const bool norm = residual != nullptr;
    if ((residual == nullptr) != (gamma == nullptr)) return MOEF_ERR_ARG;
    if (norm) {
        if (!residual_out || !norm_out) return MOEF_ERR_NULL;
        if (!(eps >= 0.f) || isinf(eps)) return MOEF_ERR_ARG;
    } else {
        if (residual_out || norm_out) return MOEF_ERR_ARG;
        if (!out) return MOEF_ERR_NULL;
    }

    const void *bf16_ptrs[] = {permuted_out, shared_out, residual, gamma, out, residual_out,
                               norm_out};
    for (const void *q : bf16_ptrs)
        if (q && !aligned(q, 2)) return MOEF_ERR_ALIGN;
    if (!aligned(idx_map, 4)) return MOEF_ERR_ALIGN;
    if (!aligned(weights, wkind == MOEF_W_BF16 ? 2 : 4)) return MOEF_ERR_ALIGN;

    bool v = (H % 8) == 0;
    for (const void *q : bf16_ptrs)
        if (q && !aligned(q, 16)) v = false;
    *vec_ok = v;

    p->x = static_cast<const uint16_t *>(permuted_out);
    p->idx = idx_map;
    p->weights = weights;
    p->shared = static_cast<const uint16_t *>(shared_out);
    p->residual = static_cast<const uint16_t *>(residual);
    p->gamma = static_cast<const uint16_t *>(gamma);
    p->out = static_cast<uint16_t *>(out);
    p->residual_out = static_cast<uint16_t *>(residual_out);
    p->norm_out = static_cast<uint16_t *>(norm_out);
    p->out_f32 = nullptr;
    p->routed_scale = routed_scale;
    p->eps = eps;
    p->wkind = static_cast<int>(wkind);
    p->T = T;
    p->K = K;
    p->H = H;
    p->routing_ready = 0;
    p->pdl = 1;
    return MOEF_OK;
}

void apply_plan(const moef_plan &plan, moef::FinalizeParams *p) {
    p->nvec = p->H / plan.vec;
    p->splits = plan.splits;
    p->slice = plan.slice;
}

}  // namespace

moef_status moe_finalize_ex(const void *permuted_out, int64_t P, const int32_t *idx_map,
                            const void *weights, moef_weight_kind wkind, float routed_scale,
                            const void *shared_out, const void *residual, const void *gamma,
                            float eps, void *out, void *residual_out, void *norm_out,
                            int T, int K, int H, int splits_hint, int threads_hint,
                            unsigned flags, cudaStream_t stream) {
    if (splits_hint < 0 || threads_hint < 0) return MOEF_ERR_ARG;
    if (flags & ~(MOEF_FLAG_ROUTING_READY | MOEF_FLAG_NO_PDL)) return MOEF_ERR_ARG;
    moef::FinalizeParams p;
    bool vec_ok = false;
    moef_status st = check_finalize_args(permuted_out, P, idx_map, weights, wkind, routed_scale,
                                         shared_out, residual, gamma, eps, out, residual_out,
                                         norm_out, T, K, H, &p, &vec_ok);
    if (st != MOEF_OK || T == 0) return st;

    int sms = 0;
    st = cuda_status(current_sms(&sms));
    if (st != MOEF_OK) return st;
    moef_plan plan;
    st = moe_finalize_plan(T, K, H, residual ? 1 : 0, vec_ok ? 1 : 0, sms, splits_hint,
                           threads_hint, &plan);
    if (st != MOEF_OK) return st;
    apply_plan(plan, &p);
    p.routing_ready = (flags & MOEF_FLAG_ROUTING_READY) ? 1 : 0;
    p.pdl = (flags & MOEF_FLAG_NO_PDL) ? 0 : 1;
    return cuda_status(moef::launch_finalize(p, plan, sms, stream));
}

size_t moe_finalize_unfused_workspace_bytes(int T, int H) {
    if (T <= 0 || H <= 0) return 0;
    return static_cast<size_t>(T) * static_cast<size_t>(H) * 2u;
}

moef_status moe_finalize_unfused(const void *permuted_out, int64_t P, const int32_t *idx_map,
                                 const void *weights, moef_weight_kind wkind,
                                 float routed_scale, const void *shared_out,
                                 const void *residual, const void *gamma, float eps, void *out,
                                 void *residual_out, void *norm_out, int T, int K, int H,
                                 void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    moef::FinalizeParams p;
    bool vec_ok = false;
    moef_status st = check_finalize_args(permuted_out, P, idx_map, weights, wkind, routed_scale,
                                         shared_out, residual, gamma, eps, out, residual_out,
                                         norm_out, T, K, H, &p, &vec_ok);
    if (st != MOEF_OK || T == 0) return st;
    if (!out) return MOEF_ERR_NULL;              // the unfused path always writes out
    if (!workspace) return MOEF_ERR_NULL;
    if (workspace_bytes < moe_finalize_unfused_workspace_bytes(T, H)) return MOEF_ERR_SHAPE;
    if (!aligned(workspace, 2)) return MOEF_ERR_ALIGN;
    if (!aligned(workspace, 16)) vec_ok = false;

    int sms = 0;
    st = cuda_status(current_sms(&sms));
    if (st != MOEF_OK) return st;
    moef_plan plan;
    st = moe_finalize_plan(T, K, H, 0, vec_ok ? 1 : 0, sms, 0, 0, &plan);
    if (st != MOEF_OK) return st;
    apply_plan(plan, &p);
    return cuda_status(
        moef::launch_unfused(p, plan, static_cast<uint16_t *>(workspace), sms, stream));
}

moef_status moe_finalize(const void *permuted_out, int64_t P, const int32_t *idx_map,
                         const void *weights, moef_weight_kind wkind, float routed_scale,
                         const void *shared_out, const void *residual, const void *gamma,
                         float eps, void *out, void *residual_out, void *norm_out,
                         int T, int K, int H, cudaStream_t stream) {
    return moe_finalize_ex(permuted_out, P, idx_map, weights, wkind, routed_scale, shared_out,
                           residual, gamma, eps, out, residual_out, norm_out, T, K, H, 0, 0, 0u,
                           stream);
}

moef_status moe_topk_route(const float *logits, int T, int E, int K, moef_gate_kind kind,
                           int32_t *expert_ids, float *weights, int32_t *packed,
                           cudaStream_t stream) {
    if (T < 0 || E < 1 || E > MOEF_MAX_EXPERTS || K < 1 || K > MOEF_MAX_K || K > E)
        return MOEF_ERR_SHAPE;
    if (kind != MOEF_GATE_SOFTMAX && kind != MOEF_GATE_SIGMOID) return MOEF_ERR_ARG;
    if (T == 0) return MOEF_OK;
    if (!logits || (!expert_ids && !weights && !packed)) return MOEF_ERR_NULL;
    if (!aligned(logits, 4) || (expert_ids && !aligned(expert_ids, 4)) ||
        (weights && !aligned(weights, 4)) || (packed && !aligned(packed, 4)))
        return MOEF_ERR_ALIGN;
    return cuda_status(moef::launch_topk_route(logits, T, E, K, static_cast<int>(kind), expert_ids,
                                               weights, packed, stream));
}

moef_status pack_topk_ids(const int32_t *expert_ids, const float *weights, int64_t n,
                          int32_t *packed, cudaStream_t stream) {
    if (n < 0) return MOEF_ERR_SHAPE;
    if (n == 0) return MOEF_OK;
    if (!expert_ids || !weights || !packed) return MOEF_ERR_NULL;
    if (!aligned(expert_ids, 4) || !aligned(weights, 4) || !aligned(packed, 4))
        return MOEF_ERR_ALIGN;
    int sms = 0;
    moef_status st = cuda_status(current_sms(&sms));
    if (st != MOEF_OK) return st;
    return cuda_status(moef::launch_pack(expert_ids, weights, n, packed, sms, stream));
}

moef_status unpack_topk_ids(const int32_t *packed, int64_t n, int32_t *expert_ids,
                            float *weights_f32, cudaStream_t stream) {
    if (n < 0) return MOEF_ERR_SHAPE;
    if (n == 0) return MOEF_OK;
    if (!packed || (!expert_ids && !weights_f32)) return MOEF_ERR_NULL;
    if (!aligned(packed, 4) || (expert_ids && !aligned(expert_ids, 4)) ||
        (weights_f32 && !aligned(weights_f32, 4)))
        return MOEF_ERR_ALIGN;
    int sms = 0;
    moef_status st = cuda_status(current_sms(&sms));
    if (st != MOEF_OK) return st;
    return cuda_status(moef::launch_unpack(packed, n, expert_ids, weights_f32, sms, stream));
}

moef_status moe_finalize_check_indices(const int32_t *idx_map, int T, int K, int64_t P,
                                       int32_t *d_bad_count, cudaStream_t stream) {
    if (T < 0 || K < 1 || K > MOEF_MAX_K || P < 0) return MOEF_ERR_SHAPE;
    if (!d_bad_count) return MOEF_ERR_NULL;
    const int64_t n = static_cast<int64_t>(T) * K;
    if (n > 0 && !idx_map) return MOEF_ERR_NULL;
    if (!aligned(d_bad_count, 4) || (idx_map && !aligned(idx_map, 4))) return MOEF_ERR_ALIGN;
    int sms = 0;
    moef_status st = cuda_status(current_sms(&sms));
    if (st != MOEF_OK) return st;
    return cuda_status(moef::launch_check_indices(idx_map, n, P, d_bad_count, sms, stream));
}

// ---------------------------------------------------------------------------
// All-reduce-fused finalize (kernels in allreduce.cu)

namespace {

constexpr int kArMaxThreads = 512;    // the all-reduce kernels' launch bounds
constexpr int kArMaxPasses = 8;

// Tokens from which the ranks of a vector are summed in sequence by one
// thread (lanes = 1), and the vectors of such a plan's slice.
#ifndef MOEF_AR_SEQ_MIN_TOKENS
#define MOEF_AR_SEQ_MIN_TOKENS 64
#endif
#ifndef MOEF_AR_SEQ_SLICE
#define MOEF_AR_SEQ_SLICE 128
#endif
// Largest rank group count past the decode sizes (R > this: groups of 2 ranks).
#ifndef MOEF_AR_MID_LANES
#define MOEF_AR_MID_LANES 4
#endif
constexpr int kArSeqMinTokens = MOEF_AR_SEQ_MIN_TOKENS;
constexpr int kArSeqSlice = MOEF_AR_SEQ_SLICE;
// Largest CTA of a sequential-ranks plan with RMSNorm.
#ifndef MOEF_AR_SEQ_MAX_THREADS
#define MOEF_AR_SEQ_MAX_THREADS 256
#endif
// Tokens up to which a row takes the decode plan (CTAs of up to 512 threads,
// one cluster of up to 16 CTAs a row, one CTA per SM in the 128-register
// build): about 7 such clusters are resident at once
// (launch__cluster_max_active).  R = 8: T = 5 / 7 take 4.80 / 5.20 us
// against 7.17 / 7.35 us with the rank pairs of larger T; R = 6, T = 5: 4.53
// against 7.02 us; R = 2 and 4: 0.05-0.17 us faster.
// With more than kArMidLanes ranks, where the alternative is rank pairs, up
// to 14 tokens: past 7 the kernels take their 64-register build, two CTAs
// per SM, and twice the clusters fit (R = 8, T = 8 / 14: 6.12 / 6.83 us
// against 7.53 / 8.18 us with rank pairs, the two-phase form unchanged).
constexpr int kArDecodeTokensBase = 7;
constexpr int kArDecodeTokensWide = 14;
constexpr int kArMidLanes = MOEF_AR_MID_LANES;
constexpr int kArSeqMaxThreads = MOEF_AR_SEQ_MAX_THREADS;

int pow2_bucket(int need) {
    int b = 1;
    while (b < need) b *= 2;
    return b;
}

}  // namespace

// Plan of the all-reduce-fused kernels.  At decode sizes a CTA holds R
// groups of threads, one per rank, each thread obtaining one rank's partial
// of one vector per pass, so that every rank's row loads are in flight at
// once (lanes = R); past the decode sizes, with more than kArMidLanes ranks
// and 16-byte vectors, R / 2 groups of two ranks each:
//  * without RMSNorm, 128 threads per CTA (`lanes` groups of 128 / lanes, at
//    least 16 threads), one vector per thread: slices of 128 / lanes vectors;
//  * with RMSNorm, one CTA or one cluster of up to 16 CTAs finishes a row.
//    Each extra pass over a slice costs a full chain of loads, barrier and
//    epilogue (about 2.8 us at R = 8, T = 1), so the decode sizes (up to
//    kArDecodeTokensBase tokens, kArDecodeTokensWide with R > kArMidLanes)
//    take CTAs of up to 512 threads (`lanes` groups of 512 / lanes, at most
//    256), enough for one pass, and with R > 1 a split row over a full
//    cluster of 16 (slices of at least 32 vectors), so that more SMs share
//    the ranks' rows: with R = 8 at H = 7168, 16 CTAs of 8 x 64 threads
//    (T = 1: 4.28 -> 4.24 us against 14 CTAs; R = 2: 4.19 -> 3.91 us against
//    4 CTAs of 2 x 224 threads; R = 4: 4.31 -> 4.04 us; H = 4096: 0.05-0.24
//    us faster).  Past the decode sizes CTAs of 256 threads win even with a
//    second pass (R = 4, T = 16: 14 x 256 threads 5.6 us vs 7 x 512 threads
//    9.3 us; R = 8: 16 x 224 threads 9.2 us vs 14 x 512 threads 11.9 us).
//    The split is halved while the grid exceeds 4 CTAs per SM, each thread
//    then taking up to 8 passes.
// Past the decode sizes up to the sequential-ranks plans, R >= 4 ranks (even) go in
// two groups of R / 2 (CTAs of 2 x 128 threads) once the plan above would
// not have all its rows' clusters resident at once, or would need a second
// pass.  14-CTA clusters of 256-thread CTAs fit about 35 at a time: R = 8,
// T = 36: 13.3 us against 17.6 us one-shot; R = 4, T = 36: 8.7 / 7.0
// against 11.2 / 10.0 us (one-shot / two-phase per rank).  192-thread CTAs
// (R = 6 pairs) fit about 43, so R = 6 keeps its pairs up to T = 43 (T = 40:
// 10.9 against 11.9 us one-shot).  Past 4 CTAs per SM pairs would take a
// second pass: R = 8, T = 48: 15.3 / 8.2 us against 16.7 / 9.4 us; R = 6:
// 12.8 / 7.8 against 14.4 / 8.8.  Up to T = 80 the one-shot keeps gaining
// (R = 8, T = 64: 17.1 against 18.6 us), but the two-phase form, the faster
// one there, loses (9.2 against 8.8 us), so the sequential plans take over
// at kArSeqMinTokens.
// With many tokens (R > 1, T >= kArSeqMinTokens, 16-byte vectors) the
// tokens alone fill the GPU, and each thread sums the ranks of its vector in
// sequence (lanes = 1).  Slices start at kArSeqSlice vectors, one pass each;
// with RMSNorm a row is one cluster of up to 16 CTAs of up to 256 threads,
// the split halved (up to 8 passes) until every CTA of the grid is resident
// at once (CTAs per SM at 64 registers a thread for that CTA size, whole
// clusters per GPC: R = 8, T = 168 took 42.5 us on 7 CTAs a row, 1176 CTAs
// that fit the SMs but not as 7-CTA clusters, against 38.0 us halved).  Even a
// small second wave costs more than the passes: R = 8, T = 160: 7 CTAs of
// 128 threads per row, 29.6 us, against 37.2 us halved at 4 CTAs per SM;
// T = 176 (just past one wave): 38.5 us for 2 CTAs x 2 passes of 224
// threads against 43.0 us for 7 CTAs; T = 256: 46.3 against 47.9 us.
// Splits stepped down one at a time (3 CTAs x 2 passes of 160 threads at
// T = 176-288) measured 2-4 % slower than halving.  Measured
// on GB300 at H = 7168 (one-shot / two-phase per rank, us): R = 8, T = 16:
// rank pairs 8.9 / 6.5, one rank per group 9.2 / 8.5; T = 32: rank pairs
// 11.1 / 7.7, one rank per group 15.3 / 8.8, sequential 17.2 / 8.0; T = 64:
// sequential 18.9 / 9.2, one rank per group 19.1 / 12.8.
moef_status moe_finalize_allreduce_plan(int R, int T, int H, int with_norm, int vec_ok,
                                        int num_sms, moef_ar_plan *plan) {
    if (!plan) return MOEF_ERR_NULL;
    if (R < 1 || R > MOEF_MAX_RANKS || T < 0 || H < 1) return MOEF_ERR_SHAPE;
    if (num_sms < 1) return MOEF_ERR_ARG;
    const int vec = (vec_ok && H % 8 == 0) ? 8 : 1;
    const int nvec = H / vec;
    const int64_t rows = T > 0 ? T : 1;
    const int decode_tokens = R > kArMidLanes ? kArDecodeTokensWide : kArDecodeTokensBase;
    int lanes = R, nvc = 0, splits = 0, slice = 0, passes = 0;
    if (R > 1 && vec == 8 && T >= kArSeqMinTokens) {
        lanes = 1;
        if (!with_norm) {
            nvc = kArSeqSlice < nvec ? kArSeqSlice : nvec;
            slice = nvc;
            splits = ceil_div(nvec, slice);
            if (rows * splits > 0x7FFFFFFFLL) {
                splits = static_cast<int>(0x7FFFFFFFLL / rows);
                if (splits < 1) splits = 1;
                slice = ceil_div(nvec, splits);
            }
            passes = ceil_div(slice, nvc);
        } else {
            splits = ceil_div(nvec, kArSeqSlice);
            if (splits > kMaxCluster) splits = kMaxCluster;
            // the most slices per row whose CTAs are all resident at once
            // (64 registers a thread), halving the split otherwise
            for (;;) {
                if (splits <= 1) break;
                const int sl = ceil_div(nvec, splits);
                const int pa = pow2_bucket(ceil_div(sl, kArSeqMaxThreads));
                const int nv = round_up(ceil_div(sl, pa), 32);
                // a row's CTAs are one cluster, placed within one of the GPU's
                // 8 GPCs (num_sms / 8 SMs each): whole clusters per GPC, less
                // one cluster's room for clusters of 4 CTAs or more (measured:
                // 7-CTA clusters of 128 threads run in one wave at 160 rows but
                // not at 168; 2-CTA clusters of 224 threads at 304 rows)
                const int64_t per_gpc = static_cast<int64_t>(num_sms / 8) * (1024 / nv) -
                                        (splits >= 4 ? splits : 0);
                if (rows <= 8 * (per_gpc / splits)) break;
                const int half = ceil_div(splits, 2);
                if (ceil_div(ceil_div(nvec, half), kArSeqMaxThreads) > kArMaxPasses) break;
                splits = half;
            }

            slice = ceil_div(nvec, splits);
            passes = pow2_bucket(ceil_div(slice, kArSeqMaxThreads));
            if (passes > kArMaxPasses) {
                lanes = R;                   // too long a row: the rank-group plan decides
            } else {
                nvc = round_up(ceil_div(slice, passes), 32);
                if (nvc > kArSeqMaxThreads) nvc = kArSeqMaxThreads;
            }
        }
    }
    // the plan of `ln` groups of threads (ln > 1, or R = 1)
    auto group_plan = [&](int ln, int *nvc_o, int *splits_o, int *slice_o,
                          int *passes_o) -> moef_status {
        int nv, sp, sl, pa;
        if (!with_norm) {
            nv = 128 / ln / 16 * 16;
            if (nv < 16) nv = 16;
            if (nv > nvec) nv = nvec;
            sl = nv;
            sp = ceil_div(nvec, sl);
            // two vectors a thread when one a thread would take more than one
            // wave (R = 1, T = 256: 8.20 -> 8.04 us; T = 1024: 28.8 -> 28.1 us)
            if (rows * sp > static_cast<int64_t>(num_sms) * (1024 / round_up(ln * nv, 32))) {
                sl = 2 * nv;
                sp = ceil_div(nvec, sl);
            }
            if (rows * sp > 0x7FFFFFFFLL) {
                sp = static_cast<int>(0x7FFFFFFFLL / rows);
                if (sp < 1) sp = 1;
                sl = ceil_div(nvec, sp);
            }
            pa = ceil_div(sl, nv);
        } else {
            int nvc_max = (T <= decode_tokens ? kArMaxThreads : kArMaxThreads / 2) / ln;
            if (nvc_max > 256) nvc_max = 256;
            nvc_max = nvc_max / 32 * 32;
            sp = ceil_div(nvec, nvc_max);
            // a few tokens over several ranks, a row already split: the row
            // over a full cluster (slices of at least 32 vectors), so that
            // more SMs share the ranks' rows.  A row that fits one CTA stays
            // there: a cluster's barrier costs more than it gains (R = 2,
            // H = 2048: 3.23 us in one CTA, 3.63 us over 8)
            if (T <= decode_tokens && R > 1 && sp > 1 && sp < kMaxCluster) {
                const int wide = nvec / 32 < kMaxCluster ? nvec / 32 : kMaxCluster;
                if (wide > sp) sp = wide;
            }
            if (sp > kMaxCluster) sp = kMaxCluster;
            if (ceil_div(ceil_div(nvec, sp), nvc_max) > kArMaxPasses) return MOEF_ERR_SHAPE;
            while (sp > 1 && rows * sp > 4 * static_cast<int64_t>(num_sms)) {
                const int half = ceil_div(sp, 2);
                if (ceil_div(ceil_div(nvec, half), nvc_max) > kArMaxPasses) break;
                sp = half;
            }
            sl = ceil_div(nvec, sp);
            pa = pow2_bucket(ceil_div(sl, nvc_max));
            nv = ceil_div(sl, pa);
            if (nv > 32) nv = round_up(nv, 32);
            if (nv > nvc_max) nv = nvc_max;
        }
        *nvc_o = nv;
        *splits_o = sp;
        *slice_o = sl;
        *passes_o = pa;
        return MOEF_OK;
    };
    if (lanes > 1 || R == 1) {
        if (T > decode_tokens && R > kArMidLanes && R % 2 == 0 && vec == 8) lanes = R / 2;
        moef_status st = group_plan(lanes, &nvc, &splits, &slice, &passes);
        if (st != MOEF_OK) return st;
        // Two groups of R / 2 ranks instead, when the rows' clusters would
        // not all be resident at once (CTAs of 64 registers a thread, about
        // 4/5 of the SMs' room usable by clusters, as measured with
        // launch__cluster_max_active) or would need a second pass
        if (with_norm && R >= 4 && R % 2 == 0 && vec == 8 && T > decode_tokens && lanes > 2 &&
            splits > 1) {
            const int64_t per_sm = 1024 / (static_cast<int64_t>(lanes) * nvc);
            const int64_t fit = static_cast<int64_t>(num_sms) * per_sm * 4 / 5 / splits;
            if (T > fit || passes > 1) {
                int nv2, sp2, sl2, pa2;
                if (group_plan(2, &nv2, &sp2, &sl2, &pa2) == MOEF_OK && pa2 <= passes) {
                    lanes = 2;
                    nvc = nv2;
                    splits = sp2;
                    slice = sl2;
                    passes = pa2;
                }
            }
        }
    }
    // whole warps (the RMSNorm epilogue reduces with full-warp shuffles):
    // lanes * nvc a multiple of 32
    int unit = 32;
    while (unit > 1 && lanes % 2 == 0 && (unit / 2) * lanes % 32 == 0) unit /= 2;
    nvc = round_up(nvc, unit);
    splits = ceil_div(nvec, slice);   // no empty CTAs
    const int64_t grid = static_cast<int64_t>(T) * splits;
    if (grid > 0x7FFFFFFFLL) return MOEF_ERR_SHAPE;
    const int vbytes = vec == 8 ? 16 : 2;
    // the exchanged partials of a pass: every group's with one rank per group,
    // ranks c .. R-1 with groups of c = R / lanes ranks, none when one thread
    // sums all ranks
    const int exchanged = lanes == R ? (lanes > 1 ? R : 0) : lanes > 1 ? R - R / lanes : 0;
    int64_t smem = static_cast<int64_t>(sizeof(float)) * vec * exchanged * nvc +
                   (with_norm ? static_cast<int64_t>(passes) * nvc * vbytes : 0);
    plan->vec = vec;
    plan->lanes = lanes;
    plan->nvc = nvc;
    plan->threads = lanes * nvc;
    plan->splits = splits;
    plan->slice = slice;
    plan->passes = passes;
    plan->cluster = (with_norm && splits > 1) ? splits : 1;
    plan->smem_bytes = static_cast<int>(smem);
    plan->grid = grid;
    return MOEF_OK;
}

namespace {

// Argument checks of the residual / RMSNorm epilogue shared by the one-shot
// and phase-2 calls (the rules of moe_finalize).
moef_status check_epilogue(const void *residual, const void *gamma, float eps, void *out,
                           void *residual_out, void *norm_out) {
    if ((residual == nullptr) != (gamma == nullptr)) return MOEF_ERR_ARG;
    if (residual) {
        if (!residual_out || !norm_out) return MOEF_ERR_NULL;
        if (!(eps >= 0.f) || isinf(eps)) return MOEF_ERR_ARG;
    } else {
        if (residual_out || norm_out) return MOEF_ERR_ARG;
        if (!out) return MOEF_ERR_NULL;
    }
    const void *ptrs[] = {residual, gamma, out, residual_out, norm_out};
    for (const void *q : ptrs)
        if (q && !aligned(q, 2)) return MOEF_ERR_ALIGN;
    return MOEF_OK;
}

bool epilogue_vec_ok(const void *residual, const void *gamma, const void *out,
                     const void *residual_out, const void *norm_out) {
    const void *ptrs[] = {residual, gamma, out, residual_out, norm_out};
    for (const void *q : ptrs)
        if (q && !aligned(q, 16)) return false;
    return true;
}

void fill_epilogue(moef::ArParams *p, const void *residual, const void *gamma, float eps,
                   void *out, void *residual_out, void *norm_out) {
    p->residual = static_cast<const uint16_t *>(residual);
    p->gamma = static_cast<const uint16_t *>(gamma);
    p->out = static_cast<uint16_t *>(out);
    p->residual_out = static_cast<uint16_t *>(residual_out);
    p->norm_out = static_cast<uint16_t *>(norm_out);
    p->eps = eps;
}

// Checks one rank's gather operands; clears *vec_ok when one of them rules
// out the 16-byte path.
moef_status check_rank(const moef_rank_inputs &rk, moef_weight_kind wkind, bool *vec_ok) {
    if (rk.P < 1) return MOEF_ERR_SHAPE;
    if (!rk.permuted_out || !rk.idx_map || !rk.weights || !rk.shared_out) return MOEF_ERR_NULL;
    if (!aligned(rk.permuted_out, 2) || !aligned(rk.shared_out, 2) || !aligned(rk.idx_map, 4) ||
        !aligned(rk.weights, wkind == MOEF_W_BF16 ? 2 : 4))
        return MOEF_ERR_ALIGN;
    if (!aligned(rk.permuted_out, 16) || !aligned(rk.shared_out, 16)) *vec_ok = false;
    return MOEF_OK;
}

moef_status launch_ar(moef::ArParams &p, int R, int T, int H, bool norm, bool vec_ok,
                      cudaStream_t stream) {
    int sms = 0;
    moef_status st = cuda_status(current_sms(&sms));
    if (st != MOEF_OK) return st;
    moef_ar_plan plan;
    st = moe_finalize_allreduce_plan(R, T, H, norm ? 1 : 0, vec_ok ? 1 : 0, sms, &plan);
    if (st != MOEF_OK) return st;
    p.H = H;
    p.nvec = H / plan.vec;
    p.ranks = R;
    p.lanes = plan.lanes;
    p.nvc = plan.nvc;
    p.splits = plan.splits;
    p.slice = plan.slice;
    return cuda_status(moef::launch_finalize_ar(p, plan, sms, stream));
}

}  // namespace

moef_status moe_finalize_allreduce(const moef_rank_inputs *ranks, int R, moef_weight_kind wkind,
                                   float routed_scale, const void *residual, const void *gamma,
                                   float eps, void *out, void *residual_out, void *norm_out,
                                   int T, int K, int H, cudaStream_t stream) {
    if (R < 1 || R > MOEF_MAX_RANKS || T < 0 || K < 1 || K > MOEF_MAX_K || H < 1)
        return MOEF_ERR_SHAPE;
    if (wkind != MOEF_W_FP32 && wkind != MOEF_W_BF16 && wkind != MOEF_W_PACKED_TOPK)
        return MOEF_ERR_ARG;
    if (T == 0) return MOEF_OK;
    if (!ranks) return MOEF_ERR_NULL;
    moef::ArParams p = {};
    bool vec_ok = (H % 8) == 0;
    for (int r = 0; r < R; ++r) {
        moef_status st = check_rank(ranks[r], wkind, &vec_ok);
        if (st != MOEF_OK) return st;
        p.x[r] = static_cast<const uint16_t *>(ranks[r].permuted_out);
        p.idx[r] = ranks[r].idx_map;
        p.weights[r] = ranks[r].weights;
        p.shared[r] = static_cast<const uint16_t *>(ranks[r].shared_out);
    }
    moef_status st = check_epilogue(residual, gamma, eps, out, residual_out, norm_out);
    if (st != MOEF_OK) return st;
    if (!epilogue_vec_ok(residual, gamma, out, residual_out, norm_out)) vec_ok = false;
    fill_epilogue(&p, residual, gamma, eps, out, residual_out, norm_out);
    p.routed_scale = routed_scale;
    p.wkind = static_cast<int>(wkind);
    p.K = K;
    p.reduce = 0;
    return launch_ar(p, R, T, H, residual != nullptr, vec_ok, stream);
}

moef_status moe_finalize_partial(const void *permuted_out, int64_t P, const int32_t *idx_map,
                                 const void *weights, moef_weight_kind wkind, float routed_scale,
                                 const void *shared_out, float *partial, int T, int K, int H,
                                 cudaStream_t stream) {
    if (T < 0 || K < 1 || K > MOEF_MAX_K || H < 1) return MOEF_ERR_SHAPE;
    if (wkind != MOEF_W_FP32 && wkind != MOEF_W_BF16 && wkind != MOEF_W_PACKED_TOPK)
        return MOEF_ERR_ARG;
    if (T == 0) return MOEF_OK;
    const moef_rank_inputs rk = {permuted_out, P, idx_map, weights, shared_out};
    bool vec_ok = (H % 8) == 0;
    moef_status st = check_rank(rk, wkind, &vec_ok);
    if (st != MOEF_OK) return st;
    if (!partial) return MOEF_ERR_NULL;
    if (!aligned(partial, 4)) return MOEF_ERR_ALIGN;
    if (!aligned(partial, 16)) vec_ok = false;
    // the plain finalize kernel, storing m unrounded: per element the same
    // fp32 operations in the same order as a rank's partial in the one-shot
    // kernel (and 0.15-0.6 us faster than that kernel's phase-1 form at
    // T <= 64, the same at T = 256)
    moef::FinalizeParams f = {};
    f.x = static_cast<const uint16_t *>(permuted_out);
    f.idx = idx_map;
    f.weights = weights;
    f.shared = static_cast<const uint16_t *>(shared_out);
    f.out_f32 = partial;
    f.routed_scale = routed_scale;
    f.wkind = static_cast<int>(wkind);
    f.T = T;
    f.K = K;
    f.H = H;
    f.pdl = 1;
    int sms = 0;
    st = cuda_status(current_sms(&sms));
    if (st != MOEF_OK) return st;
    moef_plan plan;
    st = moe_finalize_plan(T, K, H, 0, vec_ok ? 1 : 0, sms, 0, 0, &plan);
    if (st != MOEF_OK) return st;
    apply_plan(plan, &f);
    return cuda_status(moef::launch_finalize(f, plan, sms, stream));
}

moef_status moe_finalize_allreduce_reduce(const float *const *partials, int R,
                                          const void *residual, const void *gamma, float eps,
                                          void *out, void *residual_out, void *norm_out,
                                          int T, int H, cudaStream_t stream) {
    if (R < 1 || R > MOEF_MAX_RANKS || T < 0 || H < 1) return MOEF_ERR_SHAPE;
    if (T == 0) return MOEF_OK;
    if (!partials) return MOEF_ERR_NULL;
    moef::ArParams p = {};
    bool vec_ok = (H % 8) == 0;
    for (int r = 0; r < R; ++r) {
        if (!partials[r]) return MOEF_ERR_NULL;
        if (!aligned(partials[r], 4)) return MOEF_ERR_ALIGN;
        if (!aligned(partials[r], 16)) vec_ok = false;
        p.partial[r] = partials[r];
    }
    moef_status st = check_epilogue(residual, gamma, eps, out, residual_out, norm_out);
    if (st != MOEF_OK) return st;
    if (!epilogue_vec_ok(residual, gamma, out, residual_out, norm_out)) vec_ok = false;
    fill_epilogue(&p, residual, gamma, eps, out, residual_out, norm_out);
    p.K = 1;
    p.reduce = 1;
    return launch_ar(p, R, T, H, residual != nullptr, vec_ok, stream);
}

}  // extern "C"
