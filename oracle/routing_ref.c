/*
 * Routing gate and routing-word packing: plain CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY (see finalize_ref.c): loaded by the test suite
 * only, shares nothing with the CUDA path.
 *
 * The finalize consumes routing weights that a gate produced; the pages
 * name the producer (a fused gate kernel that yields fp32 weights) and the
 * packing launch that turns (expert id, weight) pairs into
 * (expert_id << 16) | bf16(weight) words ("[Deepseek V4] Keep fp32 routing
 * weights in the mxfp4 trtllm MoE", description).  They do not define the
 * gate, so the plainest reading is taken:
 *
 *   - selection: the K largest logits of the token, in descending order;
 *     equal logits are taken lowest expert id first;
 *   - weights over the K selected logits z_1..z_K:
 *       softmax:            w_k = exp(z_k - max z) / sum_j exp(z_j - max z)
 *       normalised sigmoid: w_k = s(z_k) / sum_j s(z_j), s(z) = 1/(1+exp(-z))
 *   - packing: round each weight to bf16 (nearest, ties to even) and put the
 *     expert id in the high 16 bits.
 *
 * Weights are returned in double, computed from the exact fp32 logits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

int32_t oref_pack_topk_id(int32_t expert_id, float weight);   /* finalize_ref.c */

enum { OREF_GATE_SOFTMAX = 0, OREF_GATE_SIGMOID = 1 };

/* n packed words from n (expert id, fp32 weight) pairs: the packing launch
 * of "[Deepseek V4] Keep fp32 routing weights in the mxfp4 trtllm MoE"
 * (description), one word per pair. */
void oref_pack_topk_ids(const int32_t *expert_ids, const float *weights, int64_t n,
                        int32_t *packed) {
    for (int64_t i = 0; i < n; ++i) packed[i] = oref_pack_topk_id(expert_ids[i], weights[i]);
}

/* Top-K routing of T tokens over E experts, the gate named (not defined) in
 * "[Deepseek V4] Keep fp32 routing weights ..." (description); selection
 * and weighting follow the readings in the file comment.  logits: fp32 [T, E];
 * expert_ids: int32 [T, K] (descending logit, ties lowest id first);
 * weights: double [T, K].  Returns 0, or -1 for bad sizes or kind. */
int oref_topk_route(const float *logits, int64_t T, int E, int K, int kind,
                    int32_t *expert_ids, double *weights) {
    if (E < 1 || K < 1 || K > E || (kind != OREF_GATE_SOFTMAX && kind != OREF_GATE_SIGMOID))
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        const float *z = logits + t * E;
        int32_t *ids = expert_ids + t * K;
        double *w = weights + t * K;
        /* selection by repeated scans: the best unselected logit each time */
        for (int k = 0; k < K; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int j = 0; j < k; ++j)
                    if (ids[j] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || z[e] > z[best]) best = e;   /* strict: ties keep the lower id */
            }
            ids[k] = best;
        }
        double total = 0.0;
        if (kind == OREF_GATE_SOFTMAX) {
            double zmax = (double)z[ids[0]];
            for (int k = 0; k < K; ++k) {
                w[k] = exp((double)z[ids[k]] - zmax);
                total += w[k];
            }
        } else {
            for (int k = 0; k < K; ++k) {
                w[k] = 1.0 / (1.0 + exp(-(double)z[ids[k]]));
                total += w[k];
            }
        }
        for (int k = 0; k < K; ++k) w[k] /= total;
    }
    return 0;
}
