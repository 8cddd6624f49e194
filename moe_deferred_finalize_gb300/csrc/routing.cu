// Routing kernels: the top-K gate that produces routing weights, packing and
// unpacking of (expert_id << 16) | bf16(weight) words, and counting
// out-of-range entries of the [token, top_k] row map.
//
// Packed format: "[Deepseek V4] Keep fp32 routing weights in the mxfp4
// trtllm MoE", description.  Row-map bounds: "[Kimi K2.5] Fuse deferred MoE
// finalize into next-layer AR + residual + RMSNorm", Key modifications (a
// flat index map read with the wrong top_k went out of bounds).
//
// Pack, unpack and check are small elementwise passes over T*K words
// (grid-stride loops, grids capped at a few CTAs per SM); the gate reads
// T*E logits once, one warp per token.  All are bound by launch latency at
// decode sizes.
#include <math.h>

#include <cuda_bf16.h>

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

// fp32 -> bf16 bits, round to nearest even (hardware conversion); a NaN
// keeps its payload's upper bits with the quiet bit set.
__device__ __forceinline__ uint32_t bf16_bits_rne(float w) {
    const uint32_t u = __float_as_uint(w);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (u >> 16) | 0x0040u;
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(w)));
}

__global__ void __launch_bounds__(kThreads)
pack_kernel(const int32_t *__restrict__ expert_ids, const float *__restrict__ weights,
            int64_t n, int32_t *__restrict__ packed) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const uint32_t e = static_cast<uint32_t>(__ldg(expert_ids + i));
        packed[i] = static_cast<int32_t>((e << 16) | bf16_bits_rne(__ldg(weights + i)));
    }
}

// Top-K gate, one warp per token.  Lane l holds logits l, l+32, l+64, ...
// (EPL of them), each turned once into an order-preserving 32-bit key.
//
// Usual case: a threshold, then a parallel ranking.  K rounds of a warp
// maximum over the 32 lane maxima give theta, the K-th largest of them (the
// lane number rides in the low 5 bits, so each maximum names its lane; theta
// keeps only the bits above them); the K lanes above it hold K logits >=
// theta, so the token's top K all lie at or above theta.  Those candidates
// (about K + 1 at E = 256, K = 8) are compacted into shared memory as one
// (key, inverted id) word each, and lane i ranks candidate i against all of
// them with one 64-bit comparison each (larger logit first, equal logits
// lowest expert id first).
//
// When more than 32 logits reach theta (many equal logits), K rounds of
// selection instead: each lane keeps its two best unselected keys, and each
// round finds the warp's largest unselected logit with two single-
// instruction warp reductions, the maximum key and then the minimum expert
// id among the lanes holding it.  The winning lane promotes its second-best
// key; only a lane that wins a second time before it has rescanned goes over
// its keys again.
//
// For E = 256 and K = 8 a faster selection runs first: one packed 32-bit
// word per logit (the upper 24 bits of its key above its inverted id), a
// sort of each lane's 8 words, and nine single-instruction warp maxima.  It
// hands the token to the paths above when two of the nine largest words
// could be out of order (equal upper key bits, different logits).
//
// All leave the k-th selected logit on lane k; the weights are a softmax or
// a normalised sigmoid over the K kept logits (recovered exactly from their
// keys), reduced across lanes 0..K-1.  All select the same logits in the
// same order, so the outputs do not depend on which ran.
constexpr int kRouteWarps = 4;

// Order-preserving map from fp32 to uint32 (non-NaN inputs): a larger
// float gives a larger key, equal floats (-0 and +0 too) equal keys; every
// key is above 0, which marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.f);   // -0 + 0 = +0 (round to nearest)
    // sign set: all bits flipped; sign clear: the sign bit set
    return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The two best untaken keys of the lane and their slots (key 0: none).  On
// equal keys the lower slot ranks first.
template <int EPL>
__device__ __forceinline__ void lane_best2(const uint32_t (&key)[EPL], uint32_t taken,
                                           uint32_t *b1, int *j1, uint32_t *b2, int *j2) {
    *b1 = 0u;
    *b2 = 0u;
    *j1 = 0;
    *j2 = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const uint32_t kj = ((taken >> j) & 1u) ? 0u : key[j];
        if (kj > *b1) {
            *b2 = *b1; *j2 = *j1;
            *b1 = kj; *j1 = j;
        } else if (kj > *b2) {
            *b2 = kj; *j2 = j;
        }
    }
}

// Sorts 8 words into descending order in place (a 19-comparator network,
// depth 6).
__device__ __forceinline__ void sort8_desc(uint32_t (&w)[8]) {
    constexpr int kPairs[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6},
                                   {3, 7}, {0, 1}, {2, 3}, {4, 5}, {6, 7}, {2, 4}, {3, 5},
                                   {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int c = 0; c < 19; ++c) {
        const uint32_t a = w[kPairs[c][0]], b = w[kPairs[c][1]];
        w[kPairs[c][0]] = max(a, b);
        w[kPairs[c][1]] = min(a, b);
    }
}

// Slot j of lane l holds expert id(l, j): with CONTIG (E = 32 * EPL, every
// lane full) the lane's block l * EPL + j, read with 16-byte loads when VEC4;
// otherwise the strided l + 32 * j, so that E >= K logits always sit on at
// least K lanes (the threshold below relies on it).
template <int EPL, bool CONTIG>
__device__ __forceinline__ int slot_id(int lane, int j) {
    return CONTIG ? lane * EPL + j : lane + 32 * j;
}

template <int EPL, bool CONTIG>
__device__ __forceinline__ int slot_lane(uint32_t id) {
    return CONTIG ? static_cast<int>(id / EPL) : static_cast<int>(id & 31u);
}

// KT: K when fixed at compile time (the common top-8), else 0 (K from Kp).
template <int EPL, bool CONTIG, bool VEC4, int KT>
__global__ void __launch_bounds__(kRouteWarps * 32)
topk_route_kernel(const float *__restrict__ logits, int T, int E, int Kp, int kind,
                  int32_t *__restrict__ expert_ids, float *__restrict__ weights,
                  int32_t *__restrict__ packed) {
    __shared__ uint64_t s_cand[kRouteWarps][32];   // candidates, then the kept ones by rank
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int K = KT ? KT : Kp;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t >= T) return;                 // whole warps leave together
    const float *z = logits + static_cast<int64_t>(t) * E;
    uint32_t key[EPL];
    if constexpr (VEC4) {
        const float4 *z4 = reinterpret_cast<const float4 *>(z + lane * EPL);
#pragma unroll
        for (int q = 0; q < EPL / 4; ++q) {
            const float4 f = __ldg(z4 + q);
            key[4 * q + 0] = order_key(f.x);
            key[4 * q + 1] = order_key(f.y);
            key[4 * q + 2] = order_key(f.z);
            key[4 * q + 3] = order_key(f.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = slot_id<EPL, CONTIG>(lane, j);
            key[j] = e < E ? order_key(__ldg(z + e)) : 0u;
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    uint32_t kept_key = 0u, top_key = 0u;
    int kept_id = 0;
    bool selected = false;              // taken by the packed-word path
    if constexpr (EPL == 8 && CONTIG && KT == 8) {
        // E = 256, K = 8: each logit becomes one 32-bit word, the upper 24
        // bits of its key above its inverted expert id, so that every word
        // is unique and a larger word is a larger logit, or an equal one
        // with a lower id.  Each lane sorts its 8 words; nine rounds of one
        // warp maximum take the nine largest, the winning lane shifting its
        // list.  The words order the logits exactly unless two share their
        // upper 24 key bits with different values.  The winners' logits,
        // read again, rule that out: adjacent winners with equal truncated
        // keys must hold equal logits, and the 8th and 9th must differ in
        // their truncated keys; otherwise the exact selection below runs.
        uint32_t wd[8];
        const uint32_t inv = 255u - static_cast<uint32_t>(lane * 8);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            wd[j] = (key[j] & 0xFFFFFF00u) | (inv - static_cast<uint32_t>(j));
        sort8_desc(wd);
        uint32_t mine = 0u;             // lane r: the r-th largest word, r < 9
#pragma unroll
        for (int r = 0; r < 9; ++r) {
            const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, wd[0]);
            if (lane == r) mine = m;
            if (wd[0] == m) {
#pragma unroll
                for (int j = 0; j < 7; ++j) wd[j] = wd[j + 1];
                wd[7] = 0u;
            }
        }
        const int id = 255 - static_cast<int>(mine & 255u);
        float v = 0.f;
        if (lane < 9) v = __ldg(z + id) + 0.f;
        const uint32_t tr = mine >> 8;
        const uint32_t tr_next = __shfl_down_sync(0xFFFFFFFFu, tr, 1);
        const float v_next = __shfl_down_sync(0xFFFFFFFFu, v, 1);
        const bool unsure = (lane < 7 && tr == tr_next && v != v_next) ||
                            (lane == 7 && tr == tr_next);
        if (!__any_sync(0xFFFFFFFFu, unsure)) {
            selected = true;
            kept_key = order_key(v);
            kept_id = id;
            top_key = __shfl_sync(0xFFFFFFFFu, kept_key, 0);
        }
    }
    if (!selected) {

        // Threshold: the K-th largest of the 32 lane maxima.  The K lanes holding
        // the largest maxima hold K logits at or above it, so every one of the
        // token's top K is at or above it too.
        uint32_t lane_max = 0u;
#pragma unroll
        for (int j = 0; j < EPL; ++j) lane_max = max(lane_max, key[j]);
        uint32_t theta = 0u;
        {
            // the lane number in the low 5 bits makes every lane's value unique,
            // so one warp maximum names the winning lane
            uint32_t mm = (lane_max & ~31u) | static_cast<uint32_t>(31 - lane);
            for (int k = 0; k < K; ++k) {
                theta = __reduce_max_sync(0xFFFFFFFFu, mm);
                if (static_cast<int>(theta & 31u) == 31 - lane) mm = 0u;
            }
            theta &= ~31u;   // K lanes have maxima >= theta: still a lower bound
        }
        // theta > 0 (E >= K logits sit on at least K lanes), so empty slots
        // (key 0) never count as candidates.
        uint32_t cmask = 0u;
#pragma unroll
        for (int j = 0; j < EPL; ++j) cmask |= (key[j] >= theta ? 1u : 0u) << j;
        const unsigned cnt = __popc(cmask);
        const unsigned C = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (C <= 32u) {
            const int w = threadIdx.x >> 5;
            unsigned incl = cnt;            // inclusive prefix of the counts
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            unsigned pos = incl - cnt;
            // (key, inverted id) in one word: a larger word is a larger logit,
            // or an equal logit with a lower id
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                if ((cmask >> j) & 1u) {
                    s_cand[w][pos] = (static_cast<uint64_t>(key[j]) << 32) |
                                     (0xFFFFFFFFu - static_cast<uint32_t>(slot_id<EPL, CONTIG>(lane, j)));
                    ++pos;
                }
            }
            __syncwarp();
            // lane i ranks candidate i against all of them
            uint64_t mine = 0u;
            unsigned rank = 32u;
            if (lane < static_cast<int>(C)) {
                mine = s_cand[w][lane];
                rank = 0u;
#pragma unroll 4
                for (unsigned j = 0; j < C; ++j) rank += s_cand[w][j] > mine ? 1u : 0u;
            }
            __syncwarp();
            if (rank < static_cast<unsigned>(K)) s_cand[w][rank] = mine;
            __syncwarp();
            if (lane < K) {
                const uint64_t kept = s_cand[w][lane];
                kept_key = static_cast<uint32_t>(kept >> 32);
                kept_id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kept));
            }
            top_key = static_cast<uint32_t>(s_cand[w][0] >> 32);
        } else {                            // more than 32 candidates
            uint32_t taken = 0u;            // slots this lane has given up
            uint32_t b1, b2;
            int j1, j2;
            lane_best2(key, taken, &b1, &j1, &b2, &j2);
            bool second_known = true;       // b2 is the lane's true second best
            for (int k = 0; k < K; ++k) {
                const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, b1);
                const uint32_t wi = __reduce_min_sync(
                    0xFFFFFFFFu,
                    b1 == wk ? static_cast<uint32_t>(slot_id<EPL, CONTIG>(lane, j1)) : 0xFFFFFFFFu);
                if (lane == k) { kept_key = wk; kept_id = static_cast<int>(wi); }
                if (k == 0) top_key = wk;
                if (slot_lane<EPL, CONTIG>(wi) == lane) {   // this lane's best was taken
                    taken |= 1u << j1;
                    if (second_known) {
                        b1 = b2;
                        j1 = j2;
                        second_known = false;
                    } else {
                        lane_best2(key, taken, &b1, &j1, &b2, &j2);
                        second_known = true;
                    }
                }
            }
        }
    }
    const float kept_v = key_value(kept_key);
    const float top = key_value(top_key);
    float s = 0.f;
    if (lane < K)
        s = (kind == MOEF_GATE_SOFTMAX) ? expf(kept_v - top) : 1.f / (1.f + expf(-kept_v));
    float total = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
    if (lane < K) {
        const float w = s / total;
        const int64_t i = static_cast<int64_t>(t) * K + lane;
        if (expert_ids) expert_ids[i] = kept_id;
        if (weights) weights[i] = w;
        if (packed)
            packed[i] = static_cast<int32_t>((static_cast<uint32_t>(kept_id) << 16) |
                                             bf16_bits_rne(w));
    }
}

unsigned grid_for(int64_t n, int num_sms) {
    int64_t blocks = (n + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<unsigned>(blocks);
}

template <int EPL, bool CONTIG, bool VEC4, int KT>
cudaError_t launch_route_k(const float *logits, int T, int E, int K, int kind, int32_t *ids,
                           float *w, int32_t *packed, cudaStream_t stream) {
    void *args[] = {&logits, &T, &E, &K, &kind, &ids, &w, &packed};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((T + kRouteWarps - 1) / kRouteWarps));
    cfg.blockDim = dim3(kRouteWarps * 32);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(
        &cfg, reinterpret_cast<const void *>(&topk_route_kernel<EPL, CONTIG, VEC4, KT>), args);
}

// Full rows (E = 32 * EPL) take the contiguous layout, with 16-byte loads
// when every row starts 16-byte aligned; top-8 routing takes the build with
// K fixed.
template <int EPL>
cudaError_t launch_route_t(const float *logits, int T, int E, int K, int kind, int32_t *ids,
                           float *w, int32_t *packed, cudaStream_t stream) {
    const bool full = E == 32 * EPL;
    const bool vec4 = full && EPL % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) % 16) == 0;
    if (vec4 && K == 8)
        return launch_route_k<EPL, true, (EPL % 4 == 0), 8>(logits, T, E, K, kind, ids, w,
                                                            packed, stream);
    if (vec4) return launch_route_k<EPL, true, (EPL % 4 == 0), 0>(logits, T, E, K, kind, ids, w,
                                                                  packed, stream);
    if (full) return launch_route_k<EPL, true, false, 0>(logits, T, E, K, kind, ids, w, packed,
                                                        stream);
    return launch_route_k<EPL, false, false, 0>(logits, T, E, K, kind, ids, w, packed, stream);
}

}  // namespace

cudaError_t launch_pack(const int32_t *expert_ids, const float *weights, int64_t n,
                        int32_t *packed, int num_sms, cudaStream_t stream) {
    void *args[] = {&expert_ids, &weights, &n, &packed};
    return cudaLaunchKernel(reinterpret_cast<const void *>(&pack_kernel),
                            dim3(grid_for(n, num_sms)), dim3(kThreads), args, 0, stream);
}

cudaError_t launch_topk_route(const float *logits, int T, int E, int K, int kind,
                              int32_t *expert_ids, float *weights, int32_t *packed,
                              cudaStream_t stream) {
    if (E <= 32) return launch_route_t<1>(logits, T, E, K, kind, expert_ids, weights, packed, stream);
    if (E <= 64) return launch_route_t<2>(logits, T, E, K, kind, expert_ids, weights, packed, stream);
    if (E <= 128) return launch_route_t<4>(logits, T, E, K, kind, expert_ids, weights, packed, stream);
    if (E <= 256) return launch_route_t<8>(logits, T, E, K, kind, expert_ids, weights, packed, stream);
    if (E <= 512) return launch_route_t<16>(logits, T, E, K, kind, expert_ids, weights, packed, stream);
    return launch_route_t<32>(logits, T, E, K, kind, expert_ids, weights, packed, stream);
}

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
