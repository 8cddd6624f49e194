/*
 * Deferred MoE finalize: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  It shares no
 * code, header, table or helper with the CUDA path, and the CUDA path never
 * calls it.  It is deliberately slow and obvious: single-threaded loops in
 * the order the operation is defined, every product and sum in double
 * precision from the exact input values, no blocking, no fusion.
 *
 * What it computes (sources are the sglang pull-request pages):
 *
 *   "Support deferred MoE finalize for MXFP4 and FP8 block-scale",
 *   Motivation: the expert kernel returns unweighted expert outputs; a
 *   separate kernel performs the top-k weighted combine merged with the
 *   shared-expert addition.
 *   Same page, Modifications item 2: the routed scaling factor is multiplied
 *   into the expert weight (callers without one pass 1.0).
 *
 *   "[Kimi K2.5] Fuse deferred MoE finalize into next-layer AR + residual +
 *   RMSNorm", Summary and Key modifications: the combined output is then
 *   added to the residual and RMS-normalised, residual_out is kept, and the
 *   permuted-row map and the routing weights are shaped [token, top_k].
 *
 *   "[Deepseek V4] Keep fp32 routing weights in the mxfp4 trtllm MoE",
 *   description: packed topk_ids are (expert_id << 16) | bf16(weight); the
 *   finalize exists with fp32 and with bf16 routing weights.
 *
 * For token t, hidden column h, with x = permuted_out, r_k = idx[t,k]:
 *
 *   w_k    = decode(weights[t,k])                      (exact)
 *   m[t,h] = sum_k (routed_scale * w_k) * x[r_k, h] + shared[t,h]
 *   out    = m
 *   if a residual is given:
 *     s            = m + residual[t,h]
 *     residual_out = s
 *     norm_out     = s / sqrt(mean_h(s^2) + eps) * gamma[h]
 *
 * All outputs are returned in double and never rounded to bf16.
 *
 * Readings where the pages are silent:
 *   - packed weights: the low 16 bits are the bf16 bit pattern, the high 16
 *     bits the expert id read as an unsigned field;
 *   - fp32 -> bf16 packing rounds to nearest, ties to even; NaN stays a
 *     quiet NaN;
 *   - RMSNorm is x * (mean(x^2) + eps)^(-1/2) * gamma with the mean over
 *     exactly H columns and no (1 + gamma) offset;
 *   - every idx is a valid row by contract; this oracle reports a bad one
 *     instead of reading it.
 *
 * Parity pins (outside this file): special cases K=1 / zero weights /
 * zero scale, slot-permutation invariance, linearity, NaN-filled padding,
 * RMSNorm closed forms and a library RMSNorm, hand-worked golden values,
 * exhaustive pack/unpack round trips against a library bf16 conversion.
 * For the all-reduce-fused form (oref_moe_finalize_ar, at the end): a
 * hand-worked two-rank golden case, one rank = the plain finalize, R ranks =
 * one rank over all the ranks' slots with the shared outputs summed, rank
 * order, an exact tensor-parallel split, per-rank index bounds.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Weight encodings of the routing-weight operand, numbered for this file
 * only (the Python wrapper maps names to them). */
enum { OREF_W_FP32 = 0, OREF_W_BF16 = 1, OREF_W_PACKED = 2 };

/* A bf16 value is the upper 16 bits of an IEEE binary32 value; widening
 * appends sixteen zero bits, which is exact.  (All bf16 operands of the
 * finalize: the permuted rows, shared output, residual and gamma of the
 * pages above.) */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bits_to_float(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest with ties to even, from the IEEE
 * definition: keep the upper half, look at the sixteen discarded bits.
 * More than half an upper-half ulp rounds up, less rounds down, exactly
 * half rounds to the even neighbour.  A carry out of the mantissa moves
 * into the exponent, which is the correct next representable value (and
 * gives infinity past the largest finite bf16).  NaN stays NaN, with the
 * quiet bit set so that truncating its payload cannot make it infinity. */
uint16_t oref_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t exponent = (u >> 23) & 0xFFu;
    uint32_t mantissa = u & 0x7FFFFFu;
    if (exponent == 0xFFu && mantissa != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* Packed routing word: expert id in the high half, the bf16 weight in the
 * low half ("[Deepseek V4] Keep fp32 routing weights in the mxfp4 trtllm
 * MoE", description). */
int32_t oref_pack_topk_id(int32_t expert_id, float weight) {
    uint32_t word = ((uint32_t)expert_id << 16) | (uint32_t)oref_f32_to_bf16(weight);
    int32_t out;
    memcpy(&out, &word, sizeof out);
    return out;
}

/* The inverse of the packing above, for n words: expert id = the high
 * sixteen bits as an unsigned field, weight = the low sixteen bits read as
 * a bf16 value and widened to fp32 (exact).  Either output may be NULL. */
void oref_unpack_topk_ids(const int32_t *packed, int64_t n,
                          int32_t *expert_ids, float *weights) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t word;
        memcpy(&word, &packed[i], sizeof word);
        if (expert_ids) expert_ids[i] = (int32_t)(word >> 16);
        if (weights) weights[i] = bits_to_float((word & 0xFFFFu) << 16);
    }
}

/* Routing weight of one (t, k) slot, decoded exactly to double: fp32, bf16,
 * or the low half of a packed word ("[Deepseek V4] Keep fp32 routing
 * weights in the mxfp4 trtllm MoE", description: the finalize exists with
 * bf16 and with fp32 weights; packed words carry a bf16 weight). */
static double decode_weight(const void *weights, int wkind, int64_t i) {
    if (wkind == OREF_W_FP32)
        return (double)((const float *)weights)[i];
    if (wkind == OREF_W_BF16)
        return bf16_to_double(((const uint16_t *)weights)[i]);
    {
        float w;
        oref_unpack_topk_ids(&((const int32_t *)weights)[i], 1, NULL, &w);
        return (double)w;
    }
}

/* RMSNorm of T rows of H values given in double:
 * y = x / sqrt(mean(x^2) + eps) * gamma  ("[Kimi K2.5] Fuse deferred MoE
 * finalize into next-layer AR + residual + RMSNorm", Summary: RMSNorm of the
 * residual sum; the standard form is the reading taken). */
static void rmsnorm_rows_double(const double *x, const uint16_t *gamma, double eps,
                                int64_t T, int64_t H, double *y) {
    for (int64_t t = 0; t < T; ++t) {
        const double *row = x + t * H;
        double sum_sq = 0.0;
        for (int64_t h = 0; h < H; ++h) sum_sq += row[h] * row[h];
        double inv_rms = 1.0 / sqrt(sum_sq / (double)H + eps);
        for (int64_t h = 0; h < H; ++h)
            y[t * H + h] = row[h] * inv_rms * bf16_to_double(gamma[h]);
    }
}

/* RMSNorm of T rows of bf16 values (same definition and source as above);
 * used to check a norm against the residual a device actually emitted. */
void oref_rmsnorm_bf16(const uint16_t *x, const uint16_t *gamma, double eps,
                       int64_t T, int64_t H, double *y) {
    for (int64_t t = 0; t < T; ++t) {
        double sum_sq = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double v = bf16_to_double(x[t * H + h]);
            sum_sq += v * v;
        }
        double inv_rms = 1.0 / sqrt(sum_sq / (double)H + eps);
        for (int64_t h = 0; h < H; ++h)
            y[t * H + h] = bf16_to_double(x[t * H + h]) * inv_rms * bf16_to_double(gamma[h]);
    }
}

/* The deferred finalize ("Support deferred MoE finalize for MXFP4 and FP8
 * block-scale", Motivation and Modifications item 2; "[Kimi K2.5] Fuse
 * deferred MoE finalize ...", Summary and Key modifications); see the file
 * comment for the definition.
 *
 * permuted_out  bf16 bits [P, H]   unweighted expert rows, padded per expert
 * idx           int32 [T, K]       row of permuted_out for slot (t, k)
 * weights       [T, K]             fp32, bf16 bits or packed int32 (wkind)
 * shared        bf16 bits [T, H]
 * residual      bf16 bits [T, H]   may be NULL (then gamma, residual_out and
 * gamma         bf16 bits [H]        norm_out are ignored)
 * out, residual_out, norm_out      double [T, H]; out may be NULL
 *
 * Returns 0, or -1 (and writes nothing further) when an idx lies outside
 * [0, P), or -2 for an unknown wkind. */
int oref_moe_finalize(const uint16_t *permuted_out, int64_t P, int64_t H,
                      const int32_t *idx, const void *weights, int wkind,
                      double routed_scale, const uint16_t *shared,
                      const uint16_t *residual, const uint16_t *gamma, double eps,
                      int64_t T, int64_t K,
                      double *out, double *residual_out, double *norm_out) {
    if (wkind != OREF_W_FP32 && wkind != OREF_W_BF16 && wkind != OREF_W_PACKED)
        return -2;
    for (int64_t i = 0; i < T * K; ++i)
        if (idx[i] < 0 || (int64_t)idx[i] >= P) return -1;

    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            double m = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = routed_scale * decode_weight(weights, wkind, t * K + k);
                const uint16_t *row = permuted_out + (int64_t)idx[t * K + k] * H;
                m += w * bf16_to_double(row[h]);
            }
            m += bf16_to_double(shared[t * H + h]);
            if (out) out[t * H + h] = m;
            if (residual) residual_out[t * H + h] = m + bf16_to_double(residual[t * H + h]);
        }
    }
    if (residual) rmsnorm_rows_double(residual_out, gamma, eps, T, H, norm_out);
    return 0;
}

/* The deferred finalize fused with the tensor-parallel all-reduce, residual
 * add and RMSNorm ("[Kimi K2.5] Fuse deferred MoE finalize into next-layer
 * AR + residual + RMSNorm", Summary: weighted expert combine + shared-expert
 * add + all-reduce + residual + RMSNorm in one kernel, residual_out kept;
 * Numerics & speed: the all-reduce runs over the finalized token rows, and
 * the separate-finalize fallback computes the same thing as a finalize
 * followed by an all-reduce fused with residual + RMSNorm).
 *
 * R ranks of one tensor-parallel group each hold their own expert output
 * rows, row map, routing weights and shared-expert output (each a partial
 * sum over that rank's slice of the expert and shared-expert weights).  For
 * token t and column h:
 *
 *   p_r[t,h] = sum_k (routed_scale * w_r[t,k]) * x_r[idx_r[t,k], h]
 *              + shared_r[t,h]                   (rank r's own finalize)
 *   m[t,h]   = sum_r p_r[t,h]                    (the all-reduce)
 *   out      = m
 *   if a residual is given:
 *     s            = m + residual[t,h]
 *     residual_out = s
 *     norm_out     = s / sqrt(mean_h(s^2) + eps) * gamma[h]
 *
 * The residual and gamma are the same on every rank, so they appear once;
 * every rank obtains the same outputs.  All arithmetic in double from the
 * exact input values, ranks summed r = 0..R-1.
 *
 * permuted_out[r], P[r], idx[r], weights[r], shared[r]: rank r's operands,
 * shaped as for oref_moe_finalize (weights in one encoding, wkind, for all
 * ranks).  Returns 0; -1 when an index of some rank lies outside [0, P[r]);
 * -2 for an unknown wkind; -3 for R < 1. */
int oref_moe_finalize_ar(int64_t R, const uint16_t *const *permuted_out, const int64_t *P,
                         int64_t H, const int32_t *const *idx, const void *const *weights,
                         int wkind, double routed_scale, const uint16_t *const *shared,
                         const uint16_t *residual, const uint16_t *gamma, double eps,
                         int64_t T, int64_t K,
                         double *out, double *residual_out, double *norm_out) {
    if (R < 1) return -3;
    if (wkind != OREF_W_FP32 && wkind != OREF_W_BF16 && wkind != OREF_W_PACKED)
        return -2;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t i = 0; i < T * K; ++i)
            if (idx[r][i] < 0 || (int64_t)idx[r][i] >= P[r]) return -1;

    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            double m = 0.0;
            for (int64_t r = 0; r < R; ++r) {
                double partial = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double w = routed_scale * decode_weight(weights[r], wkind, t * K + k);
                    const uint16_t *row = permuted_out[r] + (int64_t)idx[r][t * K + k] * H;
                    partial += w * bf16_to_double(row[h]);
                }
                partial += bf16_to_double(shared[r][t * H + h]);
                m += partial;
            }
            if (out) out[t * H + h] = m;
            if (residual) residual_out[t * H + h] = m + bf16_to_double(residual[t * H + h]);
        }
    }
    if (residual) rmsnorm_rows_double(residual_out, gamma, eps, T, H, norm_out);
    return 0;
}
