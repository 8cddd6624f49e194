"""Plants plausible mistakes in copies of the oracle's C source and checks
that the pins catch every one of them.  CPU only; the real oracle source is
never modified."""
import os

import pytest

import oracle
from oracle.build import SOURCES, compile_source

import pins

# (name, text in finalize_ref.c, replacement)
MUTANTS = [
    ("drop_shared", "m += bf16_to_double(shared[t * H + h]);", ""),
    ("shared_sign", "m += bf16_to_double(shared[t * H + h]);",
     "m -= bf16_to_double(shared[t * H + h]);"),
    ("drop_routed_scale", "double w = routed_scale * decode_weight(",
     "double w = decode_weight("),
    ("scale_added", "double w = routed_scale * decode_weight(weights, wkind, t * K + k);",
     "double w = routed_scale + decode_weight(weights, wkind, t * K + k);"),
    ("idx_transposed", "permuted_out + (int64_t)idx[t * K + k] * H",
     "permuted_out + (int64_t)idx[k * T + t] * H"),
    ("weight_slot_shift", "decode_weight(weights, wkind, t * K + k)",
     "decode_weight(weights, wkind, t * K + (k + 1) % K)"),
    ("drop_last_slot", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k < K - 1; ++k) {"),
    ("drop_residual", "m + bf16_to_double(residual[t * H + h])", "m"),
    ("eps_outside_root", "1.0 / sqrt(sum_sq / (double)H + eps)",
     "1.0 / (sqrt(sum_sq / (double)H) + eps)"),
    ("mean_over_h_minus_1", "double inv_rms = 1.0 / sqrt(sum_sq / (double)H + eps);\n"
     "        for (int64_t h = 0; h < H; ++h)\n            y[t * H + h] = row[h]",
     "double inv_rms = 1.0 / sqrt(sum_sq / (double)(H - 1) + eps);\n"
     "        for (int64_t h = 0; h < H; ++h)\n            y[t * H + h] = row[h]"),
    ("drop_gamma", "y[t * H + h] = row[h] * inv_rms * bf16_to_double(gamma[h]);",
     "y[t * H + h] = row[h] * inv_rms;"),
    ("gamma_offset", "y[t * H + h] = row[h] * inv_rms * bf16_to_double(gamma[h]);",
     "y[t * H + h] = row[h] * inv_rms * (1.0 + bf16_to_double(gamma[h]));"),
    ("norm_of_out_not_residual", "rmsnorm_rows_double(residual_out, gamma",
     "rmsnorm_rows_double(out, gamma"),
    ("expert_id_signed_shift", "expert_ids[i] = (int32_t)(word >> 16);",
     "expert_ids[i] = packed[i] >> 16;"),
    ("weight_sign_dropped", "bits_to_float((word & 0xFFFFu) << 16)",
     "bits_to_float((word & 0x7FFFu) << 16)"),
    ("weight_from_high_half", "bits_to_float((word & 0xFFFFu) << 16)",
     "bits_to_float(word & 0xFFFF0000u)"),
    ("pack_truncates", "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))",
     "if (0)"),
    ("pack_ties_away", "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))",
     "if (dropped >= 0x8000u)"),
    ("bf16_weight_read_as_packed", "if (wkind == OREF_W_BF16)", "if (0)"),
    ("bad_index_accepted", "if (idx[i] < 0 || (int64_t)idx[i] >= P) return -1;",
     "if (idx[i] < 0) return -1;"),
]


# the all-reduce-fused finalize (oref_moe_finalize_ar)
AR_MUTANTS = [
    ("ar_drop_last_rank", "for (int64_t r = 0; r < R; ++r) {\n                double partial",
     "for (int64_t r = 0; r < R - 1; ++r) {\n                double partial"),
    ("ar_rank0_rows_everywhere", "const uint16_t *row = permuted_out[r] +",
     "const uint16_t *row = permuted_out[0] +"),
    ("ar_rank0_map_everywhere", "(int64_t)idx[r][t * K + k] * H", "(int64_t)idx[0][t * K + k] * H"),
    ("ar_rank0_weights_everywhere", "decode_weight(weights[r], wkind", "decode_weight(weights[0], wkind"),
    ("ar_shared_of_rank0_only", "partial += bf16_to_double(shared[r][t * H + h]);",
     "if (r == 0) partial += bf16_to_double(shared[0][t * H + h]);"),
    ("ar_mean_not_sum", "m += partial;", "m += partial / (double)R;"),
    ("ar_residual_per_rank", "m += partial;",
     "m += partial + (residual && r > 0 ? bf16_to_double(residual[t * H + h]) : 0.0);"),
    ("ar_scale_on_shared_too", "partial += bf16_to_double(shared[r][t * H + h]);",
     "partial += routed_scale * bf16_to_double(shared[r][t * H + h]);"),
    ("ar_bound_of_rank0", "(int64_t)idx[r][i] >= P[r]", "(int64_t)idx[r][i] >= P[0]"),
]


ROUTING_MUTANTS = [
    ("route_ties_keep_higher_id", "if (best < 0 || z[e] > z[best])",
     "if (best < 0 || z[e] >= z[best])"),
    ("route_selects_smallest", "if (best < 0 || z[e] > z[best])",
     "if (best < 0 || z[e] < z[best])"),
    ("route_sigmoid_sign", "w[k] = 1.0 / (1.0 + exp(-(double)z[ids[k]]));",
     "w[k] = 1.0 / (1.0 + exp((double)z[ids[k]]));"),
    ("route_not_normalised", "for (int k = 0; k < K; ++k) w[k] /= total;", ""),
    ("pack_array_swaps_operands", "packed[i] = oref_pack_topk_id(expert_ids[i], weights[i]);",
     "packed[i] = oref_pack_topk_id((int32_t)weights[i], (float)expert_ids[i]);"),
]
ALL = ([(n, o, r, 0) for n, o, r in MUTANTS + AR_MUTANTS] +
       [(n, o, r, 1) for n, o, r in ROUTING_MUTANTS])


@pytest.mark.parametrize("name,old,new,which", ALL, ids=[m[0] for m in ALL])
def test_pins_catch_mutant(tmp_path, name, old, new, which):
    src = open(SOURCES[which]).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    srcs = list(SOURCES)
    srcs[which] = path
    lib = compile_source(srcs, os.path.join(tmp_path, f"lib{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the mutant {name}"
