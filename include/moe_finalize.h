/*
 * moe_finalize.h -- C ABI of the deferred MoE finalize library
 * (libmoe_finalize.so), hand-written CUDA for sm_103a.
 *
 * The operation.  A mixture-of-experts layer whose expert kernel skips its
 * own top-k combine leaves behind unweighted expert outputs, one row per
 * (token, slot), grouped by expert and padded per expert ("Support deferred
 * MoE finalize for MXFP4 and FP8 block-scale", Motivation; "[Kimi K2.5] Fuse
 * deferred MoE finalize into next-layer AR + residual + RMSNorm", Numerics &
 * speed: the padded permuted gemm2_out that the index map gathers from).
 * The finalize then does, per token t and hidden column h, in one pass:
 *
 *   m[t,h]            = sum_k (w[t,k] * routed_scale) * permuted_out[idx[t,k], h]
 *                       + shared_out[t,h]
 *   out[t,h]          = bf16(m)
 *   with a residual:
 *   s[t,h]            = m + residual[t,h]
 *   residual_out[t,h] = bf16(s)
 *   norm_out[t,h]     = bf16(r * inv * gamma[h]),  r = residual_out[t,h],
 *                       inv = 1 / sqrt(mean_h(r^2) + eps)
 *
 * Sources: the weighted combine merged with the shared-expert add
 * ("Support deferred MoE finalize ...", Motivation); the routed scaling
 * factor multiplied into the weight held in a register, 1.0 for callers
 * without one (same page, Modifications item 2); residual add + RMSNorm
 * with residual_out kept, and the [token, top_k] shape of the index map and
 * weights ("[Kimi K2.5] Fuse deferred MoE finalize ...", Summary and Key
 * modifications); fp32 or bf16 routing weights and the packed
 * (expert_id << 16) | bf16(weight) words ("[Deepseek V4] Keep fp32 routing
 * weights in the mxfp4 trtllm MoE", description).
 *
 * Arithmetic: all sums in fp32 registers, one round-to-nearest-even to bf16
 * per output.  The norm is computed from the bf16-rounded residual_out, so a
 * consumer holding only residual_out can reproduce norm_out.
 *
 * Conventions for every entry point:
 *   - all array pointers are DEVICE pointers unless stated otherwise:
 *     addresses the current device can load from and store to.  Page-locked
 *     host memory (cudaHostAlloc / cudaHostRegister) qualifies under unified
 *     addressing: the kernels then read and write host memory in place over
 *     the host link, with no separate copies (slower than HBM, but input
 *     reads, compute and output writes overlap);
 *     bf16 arrays are raw IEEE bfloat16 bit patterns (uint16_t storage);
 *   - all arrays are dense, row-major, with no padding between rows;
 *   - the caller owns every buffer; the library allocates no memory, never
 *     synchronises the device or the stream, and keeps no per-call state;
 *     work is enqueued on `stream` and the call returns at once;
 *   - kernels run on the calling thread's current CUDA device (the device
 *     of the context current on the thread); `stream` must belong to it
 *     (0 = its legacy default stream);
 *   - argument errors are detected on the host before anything is enqueued
 *     and returned as a status; nothing is launched then;
 *   - kernels never trap: an index outside [0, P) is a contract violation
 *     (undefined results), detectable beforehand with
 *     moe_finalize_check_indices;
 *   - MOEF_ERR_CUDA means the CUDA runtime refused a launch or a query; that
 *     error is then taken out of the runtime's per-thread last-error slot
 *     (cudaGetLastError), so the status is its only report.
 */
#ifndef MOE_FINALIZE_H_
#define MOE_FINALIZE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Encoding of the routing-weight operand [T, K].  Exactly one encoding is
 * accepted per call; it is never inferred from the bytes (reading fp32
 * weights as bf16 is the failure reported in "[Deepseek V4] Keep fp32
 * routing weights in the mxfp4 trtllm MoE", revert note). */
typedef enum {
    MOEF_W_FP32 = 0,        /* float32 weights                                  */
    MOEF_W_BF16 = 1,        /* bfloat16 bit patterns, widened exactly to fp32    */
    MOEF_W_PACKED_TOPK = 2  /* int32 (expert_id << 16) | bf16(weight); the       */
                            /* weight is the low half, the expert id is unused   */
} moef_weight_kind;

typedef enum {
    MOEF_OK = 0,
    MOEF_ERR_NULL = 1,   /* a required pointer is NULL                          */
    MOEF_ERR_SHAPE = 2,  /* a size is out of range                              */
    MOEF_ERR_ALIGN = 3,  /* a pointer is not aligned to its element size        */
    MOEF_ERR_ARG = 4,    /* an enum, a scalar or an optional-argument pairing   */
    MOEF_ERR_CUDA = 5,   /* the CUDA runtime returned an error                  */
    MOEF_ERR_INDEX = 6   /* reserved for index errors reported by callers       */
} moef_status;

/* Largest top_k accepted. */
#define MOEF_MAX_K 32

/*
 * moe_finalize -- the deferred finalize (see the file comment).
 *
 *   permuted_out  bf16 [P, H]  unweighted expert rows, padded per expert;
 *                              padding rows are never read
 *   P             rows of permuted_out (>= 1); used for argument checks and
 *                              by moe_finalize_check_indices
 *   idx_map       int32 [T, K] row of permuted_out for slot (t, k)
 *                              (expanded_idx_to_permuted_idx); every entry
 *                              must lie in [0, P)
 *   weights       [T, K]       routing weights, encoding given by wkind
 *   routed_scale  multiplies every routing weight (1.0 when unused)
 *   shared_out    bf16 [T, H]  shared-expert output, required
 *   residual      bf16 [T, H]  optional; residual and gamma go together
 *   gamma         bf16 [H]     RMSNorm weight, optional
 *   eps           RMSNorm epsilon (>= 0); ignored without a residual
 *   out           bf16 [T, H]  finalized MoE output; may be NULL only when a
 *                              residual is given (then only residual_out and
 *                              norm_out are written)
 *   residual_out  bf16 [T, H]  required iff residual is given
 *   norm_out      bf16 [T, H]  required iff residual is given
 *   T             tokens (>= 0; T = 0 returns MOEF_OK and enqueues nothing)
 *   K             top_k, 1 <= K <= MOEF_MAX_K
 *   H             hidden size (>= 1)
 *   stream        CUDA stream to enqueue on (0 = legacy default stream)
 *
 * In place: out may equal shared_out and residual_out may equal residual
 * (each element is read before it is written, by the same thread).  No
 * other overlap between outputs and inputs is allowed.
 *
 * Alignment: bf16 pointers must be 2-byte aligned, idx_map and fp32/packed
 * weights 4-byte aligned (else MOEF_ERR_ALIGN).  The 16-byte vector path
 * is used when H % 8 == 0 and every bf16 pointer is 16-byte aligned; any
 * other case takes a scalar path with the same results.
 *
 * Ordering: the kernel is launched as a programmatic dependent of the
 * previous kernel on `stream` (programmatic stream serialization).  It
 * touches no global memory before the previous kernel has completed and
 * flushed, so ordinary stream order holds; only the launch and CTA set-up
 * overlap the previous kernel's tail.  After its loads it allows the next
 * kernel, if that one is launched the same way, to begin launching.
 *
 * The call allocates nothing and does not synchronise, so it may be
 * captured in a CUDA graph ("[Kimi K2.5] Fuse deferred MoE finalize ...",
 * Key modifications: workspace sized before capture, never grown inside
 * captured graphs).  The first call on a device that splits an RMSNorm row
 * over more than 8 CTAs sets a kernel attribute (once per kernel build: K
 * fixed at 8 on grids above one CTA per SM, or any K); make such calls, with
 * the shapes that will be captured, before any capture.
 */
moef_status moe_finalize(const void *permuted_out, int64_t P,
                         const int32_t *idx_map,
                         const void *weights, moef_weight_kind wkind,
                         float routed_scale,
                         const void *shared_out,
                         const void *residual, const void *gamma, float eps,
                         void *out, void *residual_out, void *norm_out,
                         int T, int K, int H, cudaStream_t stream);

/*
 * Launch plan of moe_finalize: how a call is split over CTAs.  Each token
 * row is cut into `splits` slices of `slice` vectors of `vec` bf16 values;
 * one CTA of `threads` threads finalizes one slice, each thread handling up
 * to `vpt` vectors.  With a residual and splits > 1 the CTAs of one token
 * form a thread-block cluster of size `splits` and combine their partial
 * sums of squares through distributed shared memory.
 */
typedef struct {
    int vec;        /* bf16 values per vector: 8 (16-byte path) or 1 (scalar)  */
    int splits;     /* CTAs per token                                         */
    int slice;      /* vectors per CTA (the last CTA of a token may have fewer) */
    int threads;    /* threads per CTA                                        */
    int vpt;        /* vectors per thread per pass (1, 2, 4 or 8)              */
    int cluster;    /* cluster size along x (1 = no cluster)                   */
    int64_t grid;   /* CTAs launched = T * splits                              */
} moef_plan;

/*
 * moe_finalize_plan -- the plan moe_finalize uses (pure host computation,
 * no CUDA call).  with_norm: a residual is given; vec_ok: the 16-byte path
 * applies (H % 8 == 0 and 16-byte aligned pointers); num_sms: multiprocessor
 * count of the device.  splits_hint / threads_hint: 0 for the automatic
 * choice, else the requested value (validated).  Returns MOEF_ERR_SHAPE if
 * the sizes cannot be served (e.g. an RMSNorm row too long for one cluster),
 * MOEF_ERR_ARG for a bad hint.
 */
moef_status moe_finalize_plan(int T, int K, int H, int with_norm, int vec_ok,
                              int num_sms, int splits_hint, int threads_hint,
                              moef_plan *plan);

/*
 * Flags of moe_finalize_ex.
 *
 * MOEF_FLAG_ROUTING_READY: idx_map and weights were complete before the
 * previous kernel on `stream` started (in an MoE layer they come from the
 * routing step, while the kernel just before the finalize is the expert
 * GEMM that writes permuted_out).  The kernel then reads them before it
 * waits for the previous kernel, which takes one dependent memory round
 * trip off its critical path when launches overlap.  Everything else
 * (permuted_out, shared_out, residual, gamma, the outputs) is still touched
 * only after the previous kernel has completed.  Do not set it when the
 * previous kernel may write idx_map or weights.
 */
#define MOEF_FLAG_ROUTING_READY 1u

/*
 * MOEF_FLAG_NO_PDL: launch the kernel as a plain stream-ordered kernel, not
 * as a programmatic dependent of the previous kernel: its launch and CTA
 * set-up then wait for the previous kernel to complete instead of
 * overlapping its tail.  Results are the same.  For callers whose previous
 * kernel must not share the GPU with the finalize's CTAs, and to measure
 * what the dependent launch saves.
 */
#define MOEF_FLAG_NO_PDL 2u

/*
 * moe_finalize_ex -- moe_finalize with launch hints (0 = automatic), for
 * callers that pin a launch shape (e.g. one captured graph for several
 * batch sizes) and for tuning, and with `flags` (MOEF_FLAG_*, 0 = none;
 * unknown bits give MOEF_ERR_ARG).  Same arguments and rules otherwise.
 */
moef_status moe_finalize_ex(const void *permuted_out, int64_t P,
                            const int32_t *idx_map,
                            const void *weights, moef_weight_kind wkind,
                            float routed_scale,
                            const void *shared_out,
                            const void *residual, const void *gamma, float eps,
                            void *out, void *residual_out, void *norm_out,
                            int T, int K, int H,
                            int splits_hint, int threads_hint, unsigned flags,
                            cudaStream_t stream);

/*
 * moe_finalize_unfused -- the same operation as moe_finalize, computed as
 * separate kernels the way the pages' baselines ran it, for A/B measurement
 * of the fusion ("Support deferred MoE finalize for MXFP4 and FP8
 * block-scale", Speed: in-kernel combine + elementwise add for the shared
 * expert; "[Kimi K2.5] Fuse deferred MoE finalize ...", Numerics & speed:
 * finalize followed by a separate residual + RMSNorm kernel):
 *
 *   tmp = bf16(sum_k (w * routed_scale) * row)   (kernel 1, into workspace)
 *   out = bf16(tmp + shared_out)                 (kernel 2)
 *   residual_out = bf16(out + residual), norm_out from residual_out
 *                                                (kernel 3, with a residual)
 *
 * Arguments and rules as for moe_finalize, except: out is always required
 * (it is kernel 3's input), and `workspace` is a caller-owned device buffer
 * of at least moe_finalize_unfused_workspace_bytes(T, H) bytes (else
 * MOEF_ERR_NULL / MOEF_ERR_SHAPE), 2-byte aligned, not overlapping any
 * other argument; its contents on entry do not matter and are overwritten.
 * Results differ from moe_finalize by the intermediate bf16 roundings.
 */
size_t moe_finalize_unfused_workspace_bytes(int T, int H);

moef_status moe_finalize_unfused(const void *permuted_out, int64_t P,
                                 const int32_t *idx_map,
                                 const void *weights, moef_weight_kind wkind,
                                 float routed_scale,
                                 const void *shared_out,
                                 const void *residual, const void *gamma, float eps,
                                 void *out, void *residual_out, void *norm_out,
                                 int T, int K, int H,
                                 void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * moe_finalize_unfused_noalloc -- moe_finalize_unfused without a workspace
 * argument, for callers that cannot allocate device memory: serving engines
 * that fix every device allocation before they start and forbid allocation
 * on the request path, and plugins whose host framework owns all device
 * memory and gives them no allocator.  The pages have no counterpart to this
 * entry point.
 *
 * The workspace is a fixed array of MOEF_NOALLOC_SCRATCH_BYTES (8 MiB)
 * compiled into the library; every GPU on which the library's device code
 * is loaded holds it until the process exits.  Requests needing more,
 * T * H * 2 > MOEF_NOALLOC_SCRATCH_BYTES (T > 585 at H = 7168), return
 * MOEF_ERR_SHAPE without enqueuing anything.  The call allocates nothing
 * (no cudaMalloc, no library allocator).
 *
 * Set-up: the first call made on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  The address is kept for the life of the
 * device's primary context: after cudaDeviceReset (or anything else that
 * destroys that context) it is stale, and calls are not supported.
 *
 * Sharing: all calls on a device use the same array, and it keeps whatever
 * the last call left in it.  Nothing in it needs to start at zero (the first
 * kernel writes every byte the second reads), but two calls whose kernels
 * overlap on the GPU (e.g. on two streams without ordering) race on it:
 * order them.  Arguments, rules and results are otherwise those of
 * moe_finalize_unfused.
 */
#define MOEF_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

moef_status moe_finalize_unfused_noalloc(const void *permuted_out, int64_t P,
                                         const int32_t *idx_map,
                                         const void *weights, moef_weight_kind wkind,
                                         float routed_scale,
                                         const void *shared_out,
                                         const void *residual, const void *gamma, float eps,
                                         void *out, void *residual_out, void *norm_out,
                                         int T, int K, int H, cudaStream_t stream);

/*
 * ---------------------------------------------------------------------------
 * The finalize fused with the tensor-parallel all-reduce, residual add and
 * RMSNorm ("[Kimi K2.5] Fuse deferred MoE finalize into next-layer AR +
 * residual + RMSNorm", Summary: weighted expert combine + shared-expert add
 * + all-reduce + residual + RMSNorm in one kernel, keeping residual_out;
 * Numerics & speed: the all-reduce is over the finalized token rows, and the
 * separate-finalize fallback reaches the same result as a finalize followed
 * by an all-reduce fused with residual + RMSNorm).
 *
 * R ranks of one tensor-parallel group each hold their own expert rows, row
 * map, routing weights and shared-expert output, each a partial sum over the
 * rank's slice of the weights.  Every rank computes, per token t:
 *
 *   p_r          = sum_k (w_r[t,k] * routed_scale) * permuted_out_r[idx_r[t,k], :]
 *                  + shared_out_r[t, :]                       (fp32)
 *   m            = p_0 + p_1 + ... + p_{R-1}                  (fp32, rank order)
 *   out          = bf16(m)
 *   residual_out = bf16(m + residual),  norm_out as for moe_finalize
 *
 * The partials are summed in fp32, in the order of the rank array, so every
 * rank that passes the ranks in the same order obtains bit-identical
 * outputs, and the two forms below give bit-identical results.  (norm_out
 * also depends on the order in which the sum of squares is added, which
 * the launch plan fixes: it is bit-identical between calls whose buffers
 * allow the same vector width, i.e. all 16-byte aligned with H % 8 == 0, or
 * not; out and residual_out are bit-identical in every case.)
 *
 * Two forms, for two ways of ordering the ranks' work:
 *   one-shot  moe_finalize_allreduce: one launch reads every rank's rows
 *             directly (local or peer-mapped memory) and writes this rank's
 *             outputs;
 *   two-phase moe_finalize_partial on every rank (p_r in fp32, into a
 *             buffer the other ranks can read), then, once all partials are
 *             complete, moe_finalize_allreduce_reduce on every rank.
 *
 * Cross-device ordering is the caller's: the library never waits on another
 * device.  Every pointer given for a rank must be addressable from the
 * current device (its own memory, or a peer's mapped through peer access or
 * IPC); everything a call reads must be complete before its launch on
 * `stream` (e.g. cudaStreamWaitEvent on an event each rank records after its
 * producer), and no rank may overwrite a buffer until every rank's call that
 * reads it has finished.  No multicast memory is used.
 * ---------------------------------------------------------------------------
 */

/* Largest tensor-parallel group the all-reduce-fused finalize serves. */
#define MOEF_MAX_RANKS 8

/* One rank's operands of the all-reduce-fused finalize, as for moe_finalize:
 * permuted_out bf16 [P, H] (P >= 1 rows; padding rows are never read),
 * idx_map int32 [T, K] with every entry in [0, P), weights [T, K] in the
 * call's encoding, shared_out bf16 [T, H]. */
typedef struct {
    const void *permuted_out;
    int64_t P;
    const int32_t *idx_map;
    const void *weights;
    const void *shared_out;
} moef_rank_inputs;

/*
 * moe_finalize_allreduce -- the one-shot form.  ranks: a HOST array of R
 * moef_rank_inputs (1 <= R <= MOEF_MAX_RANKS; read during the call only).
 * wkind, routed_scale: for every rank.  residual, gamma, eps, out,
 * residual_out, norm_out, T, K, H: as for moe_finalize (one residual, the
 * same on every rank; out may be NULL only with a residual).  In place:
 * residual_out may equal residual; no other overlap.  Alignment rules as for
 * moe_finalize, per rank.  The launch reads R * K gathered rows per token.
 * Errors: MOEF_ERR_SHAPE for R outside [1, MOEF_MAX_RANKS] or a size out of
 * range; otherwise as for moe_finalize.
 */
moef_status moe_finalize_allreduce(const moef_rank_inputs *ranks, int R,
                                   moef_weight_kind wkind, float routed_scale,
                                   const void *residual, const void *gamma, float eps,
                                   void *out, void *residual_out, void *norm_out,
                                   int T, int K, int H, cudaStream_t stream);

/*
 * moe_finalize_partial -- phase 1 of the two-phase form: this rank's p_r
 * (see above), written unrounded as fp32 [T, H] into `partial` (4-byte
 * aligned; 16-byte aligned with H % 8 == 0 for the vector path; not
 * overlapping an input).  Other arguments as for moe_finalize without a
 * residual, and launched as moe_finalize is, under moe_finalize_plan(T, K,
 * H, 0, ...); each element gets the same fp32 operations in the same order
 * as the rank's partial inside moe_finalize_allreduce, so the two forms stay
 * bit-identical.  The partial is read by every rank's phase 2.
 */
moef_status moe_finalize_partial(const void *permuted_out, int64_t P,
                                 const int32_t *idx_map,
                                 const void *weights, moef_weight_kind wkind,
                                 float routed_scale, const void *shared_out,
                                 float *partial, int T, int K, int H, cudaStream_t stream);

/*
 * moe_finalize_allreduce_reduce -- phase 2: m = sum of the R fp32 partials
 * [T, H] in array order, then out / residual_out / norm_out exactly as
 * moe_finalize_allreduce writes them.  partials: a HOST array of R device
 * pointers (1 <= R <= MOEF_MAX_RANKS), each 4-byte aligned.  Other arguments
 * as for moe_finalize_allreduce.
 */
moef_status moe_finalize_allreduce_reduce(const float *const *partials, int R,
                                          const void *residual, const void *gamma, float eps,
                                          void *out, void *residual_out, void *norm_out,
                                          int T, int H, cudaStream_t stream);

/*
 * Launch plan of the all-reduce-fused kernels.  A one-shot CTA holds `lanes`
 * groups of `nvc` threads (threads = lanes * nvc; lanes divides R); in one
 * pass thread j of group g obtains the partials of vector j of the CTA's
 * slice for the R / lanes consecutive ranks from g * R / lanes on, and
 * thread j of group 0 sums all ranks in rank order and finishes the vector.
 * Each token row is cut into `splits` slices of `slice` vectors of `vec`
 * values, taken in `passes` passes; with a residual and splits > 1 the CTAs
 * of a token form a cluster of `cluster` CTAs.  Phase 2 runs the nvc
 * finishing threads alone (rounded up to whole warps), over the same
 * vectors.  smem_bytes: dynamic shared memory per one-shot CTA.
 */
typedef struct {
    int vec;
    int lanes;
    int nvc;
    int threads;
    int splits;
    int slice;
    int passes;
    int cluster;
    int smem_bytes;
    int64_t grid;
} moef_ar_plan;

/*
 * moe_finalize_allreduce_plan -- the plan of the one-shot and phase-2 calls
 * (the two share it, which keeps their results bit-identical: lanes = R at
 * decode sizes; for even R >= 4 from 8 tokens on, groups of ranks, R / 2 or
 * 2 of them; 1 from 64 tokens on).  with_norm = 0 plans the calls without
 * a residual.  Pure host computation: the plan depends on its arguments
 * only, num_sms included, so every call with the same arguments gets the
 * same plan.
 * Returns MOEF_ERR_SHAPE when an RMSNorm row is too long for one cluster
 * (more than 16 CTAs x 8 passes), else as moe_finalize_plan.
 */
moef_status moe_finalize_allreduce_plan(int R, int T, int H, int with_norm, int vec_ok,
                                        int num_sms, moef_ar_plan *plan);

/*
 * Routing gate: the producer of the routing weights the finalize consumes
 * ("[Deepseek V4] Keep fp32 routing weights in the mxfp4 trtllm MoE",
 * description: a fused gate kernel yields fp32 routing weights, and a
 * separate packing launch turns them into (expert_id << 16) | bf16(weight)
 * words).  The pages do not define the gate; this one takes, per token,
 * the K largest of E logits in descending order (equal logits: lowest
 * expert id first) and weights them over the K selected logits z_k by
 *   MOEF_GATE_SOFTMAX: w_k = exp(z_k - max z) / sum_j exp(z_j - max z)
 *   MOEF_GATE_SIGMOID: w_k = s(z_k) / sum_j s(z_j),  s(z) = 1 / (1 + exp(-z))
 * in fp32.  The expert ids are exact; the weights carry fp32 rounding.
 */
typedef enum { MOEF_GATE_SOFTMAX = 0, MOEF_GATE_SIGMOID = 1 } moef_gate_kind;

/* Largest expert count the gate accepts. */
#define MOEF_MAX_EXPERTS 1024

/*
 * moe_topk_route -- the gate above.  logits: fp32 [T, E], finite.
 * Outputs, each [T, K] and each nullable (at least one non-NULL):
 * expert_ids int32; weights fp32; packed int32 (expert_id << 16) |
 * bf16(weight), the bf16 rounded to nearest even from the fp32 weight
 * written to `weights`.  1 <= K <= min(E, MOEF_MAX_K), 1 <= E <=
 * MOEF_MAX_EXPERTS, T >= 0 (T = 0 enqueues nothing).  One warp per token.
 */
moef_status moe_topk_route(const float *logits, int T, int E, int K, moef_gate_kind kind,
                           int32_t *expert_ids, float *weights, int32_t *packed,
                           cudaStream_t stream);

/*
 * pack_topk_ids -- n words (expert_id << 16) | bf16(weight) from expert ids
 * (int32, used modulo 65536) and fp32 weights; bf16 rounds to nearest even,
 * a NaN keeps its upper payload bits with the quiet bit set.  Bit-exact.
 * The three arrays must not overlap.  n = 0 enqueues nothing.
 */
moef_status pack_topk_ids(const int32_t *expert_ids, const float *weights, int64_t n,
                          int32_t *packed, cudaStream_t stream);

/*
 * unpack_topk_ids -- split n packed routing words (expert_id << 16) |
 * bf16(weight) ("[Deepseek V4] Keep fp32 routing weights in the mxfp4
 * trtllm MoE", description) into expert ids (the high 16 bits as an
 * unsigned field, 0..65535) and fp32 weights (the low 16 bits widened
 * exactly).  Bit-exact.  packed: int32 [n]; expert_ids: int32 [n] or NULL;
 * weights_f32: float [n] or NULL (at least one non-NULL).  n = 0 returns
 * MOEF_OK and enqueues nothing.  The three arrays must not overlap.
 */
moef_status unpack_topk_ids(const int32_t *packed, int64_t n,
                            int32_t *expert_ids, float *weights_f32,
                            cudaStream_t stream);

/*
 * moe_finalize_check_indices -- count the entries of idx_map [T, K] that
 * lie outside [0, P) (the out-of-bounds class named in "[Kimi K2.5] Fuse
 * deferred MoE finalize ...", Key modifications: a flat index map read
 * with the wrong top_k).  d_bad_count: one caller-owned device int32; it is
 * zeroed on `stream` and then receives the count.  Enqueued work only: read
 * the count after synchronising the stream.
 */
moef_status moe_finalize_check_indices(const int32_t *idx_map, int T, int K,
                                       int64_t P, int32_t *d_bad_count,
                                       cudaStream_t stream);

/* Static English text for a status value (never NULL). */
const char *moef_status_string(moef_status s);

/* Version of this interface: raised whenever an entry point's arguments,
 * their meaning or a struct layout changes.  moef_abi_version() returns the
 * value the library was built with; a caller compiled against this header
 * should refuse a library that reports another. */
#define MOEF_ABI_VERSION 1
int moef_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FINALIZE_H_ */
