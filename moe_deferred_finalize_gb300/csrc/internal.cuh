// Internal declarations shared by the kernel and host translation units of
// libmoe_finalize.so.  Not part of the public ABI (that is moe_finalize.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_finalize.h"

namespace moef {

// Everything one finalize launch needs, passed by value as the kernel's
// single parameter (fits the 4 KB parameter space many times over).
struct FinalizeParams {
    const uint16_t *x;          // permuted_out, bf16 [P, H]
    const int32_t *idx;         // [T, K]
    const void *weights;        // [T, K], encoding in wkind
    const uint16_t *shared;     // bf16 [T, H]
    const uint16_t *residual;   // bf16 [T, H] or null
    const uint16_t *gamma;      // bf16 [H] or null
    uint16_t *out;              // bf16 [T, H] or null
    uint16_t *residual_out;     // bf16 [T, H] or null
    uint16_t *norm_out;         // bf16 [T, H] or null
    float *out_f32;             // fp32 [T, H] or null: m unrounded, in place of out
    float routed_scale;
    float eps;
    int wkind;
    int T, K, H;
    int nvec;                   // vectors per row = H / vec
    int splits;                 // CTAs per token
    int slice;                  // vectors per CTA
    int routing_ready;          // idx/weights may be read before the grid dependency wait
    int pdl;                    // launched as a programmatic dependent of the previous kernel
};

// Launches one finalize according to `plan` (validated by the caller) on a
// device with `num_sms` multiprocessors.
cudaError_t launch_finalize(const FinalizeParams &p, const moef_plan &plan, int num_sms,
                            cudaStream_t stream);

// Everything one launch of the all-reduce-fused finalize kernel needs
// (one-shot or phase 2; allreduce.cu).
struct ArParams {
    const uint16_t *x[MOEF_MAX_RANKS];          // each rank's permuted_out, bf16 [P_r, H]
    const int32_t *idx[MOEF_MAX_RANKS];         // each rank's [T, K] row map
    const void *weights[MOEF_MAX_RANKS];        // each rank's [T, K] weights (wkind)
    const uint16_t *shared[MOEF_MAX_RANKS];     // each rank's shared_out, bf16 [T, H]
    const float *partial[MOEF_MAX_RANKS];       // phase 2: each rank's fp32 [T, H] partial
    const uint16_t *residual;                   // bf16 [T, H] or null
    const uint16_t *gamma;                      // bf16 [H] or null
    uint16_t *out;                              // bf16 [T, H] or null
    uint16_t *residual_out;                     // bf16 [T, H] or null
    uint16_t *norm_out;                         // bf16 [T, H] or null
    float routed_scale;
    float eps;
    int wkind;
    int K, H;
    int nvec;                                   // vectors per row
    int ranks;                                  // R: ranks summed
    int lanes;                                  // thread groups per CTA: R, or 1
    int nvc;                                    // threads per group = vectors per pass
    int splits;                                 // CTAs per token
    int slice;                                  // vectors per CTA
    int reduce;                                 // 1: sum fp32 partials (phase 2)
};

// Launches the all-reduce-fused finalize kernel according to `plan` on a
// device with `num_sms` multiprocessors.
cudaError_t launch_finalize_ar(const ArParams &p, const moef_ar_plan &plan, int num_sms,
                               cudaStream_t stream);

// Launches the unfused three-kernel finalize (combine into tmp, add the
// shared output, residual + RMSNorm); `plan` is a plan without RMSNorm.
cudaError_t launch_unfused(const FinalizeParams &p, const moef_plan &plan, uint16_t *tmp,
                           int num_sms, cudaStream_t stream);

cudaError_t launch_pack(const int32_t *expert_ids, const float *weights, int64_t n,
                        int32_t *packed, int num_sms, cudaStream_t stream);

cudaError_t launch_topk_route(const float *logits, int T, int E, int K, int kind,
                              int32_t *expert_ids, float *weights, int32_t *packed,
                              cudaStream_t stream);

cudaError_t launch_unpack(const int32_t *packed, int64_t n, int32_t *expert_ids,
                          float *weights, int num_sms, cudaStream_t stream);

cudaError_t launch_check_indices(const int32_t *idx, int64_t n, int64_t P,
                                 int32_t *d_bad_count, int num_sms, cudaStream_t stream);

}  // namespace moef
