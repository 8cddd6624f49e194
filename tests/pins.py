"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` takes an oracle object (the real one, or a copy built from a
deliberately broken source by the mutation test) and raises AssertionError
when the oracle disagrees with:

  * values worked out by hand (``tests/golden``);
  * special cases with an exact answer (one slot of weight 1, zero weights,
    zero routed scale, a constant row under RMSNorm);
  * invariants (slot order, linearity, padding never read, equal tokens);
  * library routines (torch's bf16 conversion and RMSNorm).

The operation is the deferred finalize of "Support deferred MoE finalize for
MXFP4 and FP8 block-scale" (Motivation; Modifications item 2), with the
residual and RMSNorm of "[Kimi K2.5] Fuse deferred MoE finalize into
next-layer AR + residual + RMSNorm" (Summary) and the packed routing words of
"[Deepseek V4] Keep fp32 routing weights in the mxfp4 trtllm MoE".
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

from moe_deferred_finalize_gb300.workloads import bf16_bits_to_f32, synth, to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(x):
    return to_bf16_bits(np.asarray(x, np.float64))


def _rand_problem(seed, T=5, K=3, H=40, P=None, with_norm=False):
    rng = np.random.default_rng(seed)
    P = P or (T * K + 7)
    x = _bits(rng.standard_normal((P, H)))
    idx = np.stack([rng.choice(P, K, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    shared = _bits(rng.standard_normal((T, H)))
    res = _bits(2 * rng.standard_normal((T, H))) if with_norm else None
    gamma = _bits(rng.uniform(0.5, 1.5, H)) if with_norm else None
    return x, idx, w, shared, res, gamma


# ------------------------------------------------------------ finalize pins


def pin_golden_hand_worked(orc):
    g = _load("hand_worked_t2_k2_h3.json")
    x = _bits(g["permuted_out"])
    idx = np.array(g["idx"], np.int32)
    shared = _bits(g["shared"])
    res = _bits(g["residual"])
    gamma = _bits(g["gamma"])
    weights = {
        "fp32": np.array(g["weights_fp32"], np.float32),
        "bf16": np.array(g["weights_bf16_bits"], np.uint16),
        "packed": np.array(g["weights_packed"], np.int64).astype(np.int32).reshape(2, 2),
    }
    want_norm = np.array([[float(Fraction(v)) for v in row] for row in g["norm_out"]])
    for kind, w in weights.items():
        r = orc.moe_finalize(x, idx, w, kind, g["routed_scale"], shared, res, gamma, g["eps"])
        assert np.array_equal(r["out"], np.array(g["out"], np.float64)), (kind, r["out"])
        assert np.array_equal(r["residual_out"], np.array(g["residual_out"], np.float64)), kind
        assert np.allclose(r["norm_out"], want_norm, rtol=1e-15, atol=0), (kind, r["norm_out"])
        r2 = orc.moe_finalize(x, idx, w, kind, g["routed_scale"], shared)
        assert np.array_equal(r2["out"], np.array(g["out"], np.float64)), kind


def _exact_weight(wkind, word):
    """A routing weight as an exact rational, decoded here independently of
    the oracle: fp32 value, bf16 bits, or the low half of a packed word."""
    if wkind == "fp32":
        return Fraction(float(np.float32(word)))
    bits = int(word) & 0xFFFF
    return Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))


def pin_exact_rational_brute_force(orc):
    """Brute force in exact rational arithmetic on tiny problems.  Every
    input is a binary fraction, so out and residual_out have exact values;
    the oracle's double results must lie within a few ulps of them.
    norm_out uses a 50-digit square root."""
    import decimal
    decimal.getcontext().prec = 50
    problems = []
    wl = synth("exact_tiny", T=4, K=2, H=64, E=8, tile=4, P=32, weight_rule="softmax",
               routed_scale=1.0, seed=0)
    problems.append((wl.permuted_out, wl.idx, wl.weights, wl.wkind, 1.0, wl.shared, None, None))
    for seed, wkind in ((1, "fp32"), (2, "bf16"), (3, "packed")):
        x, idx, w, shared, res, gamma = _rand_problem(40 + seed, T=3, K=4, H=24, with_norm=True)
        w[:, 1] = -w[:, 1]            # a negative weight in every token
        if wkind == "bf16":
            w = _bits(w)
        elif wkind == "packed":    # words built here, with torch's bf16 rounding
            experts = (7 * np.arange(4)[None, :] + np.arange(3)[:, None]).astype(np.uint32)
            w = ((experts << 16) | _bits(w).astype(np.uint32)).view(np.int32)
        problems.append((x, idx, w, wkind, 2.5, shared, res, gamma))
    eps = 1e-6
    for x, idx, w, wkind, scale, shared, res, gamma in problems:
        got = orc.moe_finalize(x, idx, w, wkind, scale, shared, res, gamma, eps)
        xf = bf16_bits_to_f32(x).astype(np.float64)
        T, K = idx.shape
        H = x.shape[1]
        for t in range(T):
            wk = [_exact_weight(wkind, w[t, k]) * Fraction(scale) for k in range(K)]
            m = [sum(wk[k] * Fraction(float(xf[idx[t, k], h])) for k in range(K)) +
                 Fraction(float(bf16_bits_to_f32(shared[t, h]))) for h in range(H)]
            for h in range(H):
                assert abs(Fraction(got["out"][t, h]) - m[h]) <= \
                    Fraction(2.0 ** -50) * (abs(m[h]) + 1), ("out", t, h)
            if res is None:
                continue
            s = [m[h] + Fraction(float(bf16_bits_to_f32(res[t, h]))) for h in range(H)]
            for h in range(H):
                assert abs(Fraction(got["residual_out"][t, h]) - s[h]) <= \
                    Fraction(2.0 ** -50) * (abs(s[h]) + 1), ("residual_out", t, h)
            ms = sum(v * v for v in s) / H + Fraction(eps)
            inv = 1 / (decimal.Decimal(ms.numerator) / decimal.Decimal(ms.denominator)).sqrt()
            for h in range(H):
                want = float(decimal.Decimal(s[h].numerator) / decimal.Decimal(s[h].denominator)
                             * inv * decimal.Decimal(float(bf16_bits_to_f32(gamma[h]))))
                assert math.isclose(got["norm_out"][t, h], want, rel_tol=1e-12, abs_tol=1e-14), \
                    ("norm_out", t, h)


def pin_k1_identity(orc):
    """K=1, weight 1, scale 1, zero shared: out is the gathered row, exactly."""
    x, idx, _, shared, _, _ = _rand_problem(1, T=7, K=1, H=33)
    w = np.ones((7, 1), np.float32)
    zero = np.zeros_like(shared)
    r = orc.moe_finalize(x, idx, w, "fp32", 1.0, zero)
    assert np.array_equal(r["out"], bf16_bits_to_f32(x[idx[:, 0]]).astype(np.float64))


def pin_zero_weights(orc):
    """All routing weights 0: out is the shared-expert output, exactly."""
    x, idx, _, shared, _, _ = _rand_problem(2)
    w = np.zeros(idx.shape, np.float32)
    r = orc.moe_finalize(x, idx, w, "fp32", 2.5, shared)
    assert np.array_equal(r["out"], bf16_bits_to_f32(shared).astype(np.float64))


def pin_zero_scale(orc):
    """Routed scale 0 with nonzero weights: out is the shared output, exactly."""
    x, idx, w, shared, _, _ = _rand_problem(3)
    r = orc.moe_finalize(x, idx, w, "fp32", 0.0, shared)
    assert np.array_equal(r["out"], bf16_bits_to_f32(shared).astype(np.float64))


def pin_slot_permutation(orc):
    """Reordering the k slots (row and weight together) changes nothing."""
    x, idx, w, shared, res, gamma = _rand_problem(4, K=6, with_norm=True)
    a = orc.moe_finalize(x, idx, w, "fp32", 2.5, shared, res, gamma, 1e-6)
    perm = np.random.default_rng(5).permutation(6)
    b = orc.moe_finalize(x, idx[:, perm], w[:, perm], "fp32", 2.5, shared, res, gamma, 1e-6)
    for key in a:
        assert np.allclose(a[key], b[key], rtol=1e-13, atol=1e-13), key


def pin_linearity(orc):
    """out - shared scales with the routed scale; out moves one-for-one with shared."""
    x, idx, w, shared, _, _ = _rand_problem(6)
    sh = bf16_bits_to_f32(shared).astype(np.float64)
    r1 = orc.moe_finalize(x, idx, w, "fp32", 1.0, shared)["out"] - sh
    r3 = orc.moe_finalize(x, idx, w, "fp32", 3.0, shared)["out"] - sh
    assert np.allclose(r3, 3.0 * r1, rtol=1e-13, atol=1e-12)
    assert np.abs(r1).max() > 0.1
    zero = np.zeros_like(shared)
    r0 = orc.moe_finalize(x, idx, w, "fp32", 1.0, zero)["out"]
    assert np.allclose(r0 + sh, r1 + sh, rtol=1e-13, atol=1e-12)
    assert np.allclose(orc.moe_finalize(x, idx, w, "fp32", 1.0, shared)["out"], r0 + sh,
                       rtol=1e-13, atol=1e-12)


def pin_padding_never_read(orc):
    """NaN in every padding row leaves every output finite."""
    wl = synth("pad", T=24, K=4, H=48, E=64, tile=16, P=128, weight_rule="sigmoid",
               routed_scale=2.5, with_norm=True, seed=7)
    x = wl.permuted_out.copy()
    x[~wl.valid_rows] = 0x7FC0          # bf16 quiet NaN
    r = orc.moe_finalize(x, wl.idx, wl.weights, "fp32", wl.routed_scale, wl.shared,
                         wl.residual, wl.gamma, wl.eps)
    for key, v in r.items():
        assert np.isfinite(v).all(), key


def pin_duplicate_tokens(orc):
    """Two tokens with identical inputs give identical rows."""
    x, idx, w, shared, res, gamma = _rand_problem(8, T=4, with_norm=True)
    idx[2], w[2], shared[2], res[2] = idx[0], w[0], shared[0], res[0]
    r = orc.moe_finalize(x, idx, w, "fp32", 1.5, shared, res, gamma, 1e-6)
    for key, v in r.items():
        assert np.array_equal(v[0], v[2]), key
        assert not np.array_equal(v[0], v[1]), key


def pin_residual_add(orc):
    """residual_out - out is the residual, to fp64 rounding."""
    x, idx, w, shared, res, gamma = _rand_problem(9, with_norm=True)
    r = orc.moe_finalize(x, idx, w, "fp32", 2.5, shared, res, gamma, 1e-6)
    assert np.allclose(r["residual_out"] - r["out"], bf16_bits_to_f32(res), rtol=0, atol=1e-12)


def pin_bad_index(orc):
    x, idx, w, shared, _, _ = _rand_problem(10)
    for bad in (-1, x.shape[0]):
        j = idx.copy()
        j[1, 1] = bad
        try:
            orc.moe_finalize(x, j, w, "fp32", 1.0, shared)
        except ValueError:
            continue
        raise AssertionError(f"index {bad} accepted")


# ------------------------------------------------------------- RMSNorm pins


def _norm_only(orc, s_bits, gamma_bits, eps):
    """RMSNorm through the finalize: K=1 slot of weight 0, shared 0, residual s."""
    T, H = s_bits.shape
    x = np.zeros((1, H), np.uint16)
    idx = np.zeros((T, 1), np.int32)
    w = np.zeros((T, 1), np.float32)
    zero = np.zeros((T, H), np.uint16)
    return orc.moe_finalize(x, idx, w, "fp32", 1.0, zero, s_bits, gamma_bits, eps)["norm_out"]


def pin_rmsnorm_constant_row(orc):
    """A constant row c gives c / sqrt(c^2 + eps) * gamma."""
    H = 37
    gamma = _bits(np.linspace(0.5, 1.5, H))
    g = bf16_bits_to_f32(gamma).astype(np.float64)
    for c, eps in ((3.0, 1e-6), (-0.125, 1e-2), (1.0, 0.0)):
        s = _bits(np.full((2, H), c))
        y = _norm_only(orc, s, gamma, eps)
        want = c / math.sqrt(c * c + eps) * g
        assert np.allclose(y, want[None, :], rtol=1e-14, atol=0), (c, eps)


def pin_rmsnorm_unit_mean_square(orc):
    """mean((norm_out / gamma)^2) = ms / (ms + eps) for any row."""
    rng = np.random.default_rng(11)
    T, H, eps = 3, 96, 0.5
    s = _bits(2 * rng.standard_normal((T, H)))
    gamma = _bits(rng.uniform(0.5, 1.5, H))
    y = _norm_only(orc, s, gamma, eps)
    sf = bf16_bits_to_f32(s).astype(np.float64)
    ms = (sf * sf).mean(axis=1)
    got = ((y / bf16_bits_to_f32(gamma)) ** 2).mean(axis=1)
    assert np.allclose(got, ms / (ms + eps), rtol=1e-13)


def pin_rmsnorm_library(orc):
    """Agrees with torch's RMSNorm in float64 (mean over H, eps inside the root)."""
    rng = np.random.default_rng(12)
    T, H, eps = 4, 130, 1e-6
    s = _bits(2 * rng.standard_normal((T, H)))
    gamma = _bits(rng.uniform(0.5, 1.5, H))
    y = _norm_only(orc, s, gamma, eps)
    ref = torch.nn.functional.rms_norm(
        torch.from_numpy(bf16_bits_to_f32(s).astype(np.float64)), (H,),
        weight=torch.from_numpy(bf16_bits_to_f32(gamma).astype(np.float64)), eps=eps).numpy()
    assert np.allclose(y, ref, rtol=1e-13, atol=0)
    y2 = orc.rmsnorm_bf16(s, gamma, eps)
    assert np.allclose(y2, ref, rtol=1e-13, atol=0)


# -------------------------------------------------------- pack/unpack pins


def _u32(h):
    return np.array([int(h, 16)], np.uint64).astype(np.uint32).view(np.int32)[0]


def pin_unpack_golden(orc):
    g = _load("packed_topk_ids.json")
    words = np.array([_u32(e["word_hex"]) for e in g["unpack"]], np.int32)
    ex, w = orc.unpack_topk_ids(words)
    for i, e in enumerate(g["unpack"]):
        assert ex[i] == e["expert"], e
        want = {"inf": math.inf, "-0": -0.0, "2^-133": 2.0 ** -133}.get(e["weight"], e["weight"])
        assert w[i] == want and math.copysign(1, w[i]) == math.copysign(1, want), (e, w[i])


def pin_pack_golden(orc):
    g = _load("packed_topk_ids.json")
    for e in g["pack"]:
        f = np.array([_u32(e["weight_f32_hex"])], np.int32).view(np.float32)[0]
        assert orc.pack_topk_id(e["expert"], f) == _u32(e["word_hex"]), e


def pin_unpack_exhaustive(orc):
    """Every low half, against torch's bf16 -> fp32 widening; expert ids as
    unsigned high halves; pack(unpack(x)) == x except for signalling NaNs."""
    low = np.arange(65536, dtype=np.uint32)
    hi = np.array([0, 1, 255, 383, 32767, 32768, 65535], np.uint32)
    words = ((hi[:, None] << 16) | low[None, :]).ravel().view(np.int32)
    ex, w = orc.unpack_topk_ids(words)
    ref = torch.from_numpy(low.astype(np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()
    ref = np.tile(ref, hi.size)
    assert np.array_equal(ex, np.repeat(hi, 65536).astype(np.int32))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(w), nan)
    assert np.array_equal(w[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # round trip on one high half (the C packer is called per value)
    sel = np.arange(0, 65536, 7)
    for i in sel:
        if nan[i]:
            continue
        assert orc.pack_topk_id(int(ex[i]), float(w[i])) == words[i], hex(int(words[i]))


def pin_bf16_rounding_library(orc):
    """fp32 -> bf16 agrees with torch's conversion (round to nearest even)."""
    rng = np.random.default_rng(13)
    u = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2**16, 3000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    special = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF,
                        0x00008000, 0x00018000, 0x3F808000, 0x3F818000, 0x7F7F8000],
                       np.uint32)
    f = np.concatenate([u, ties, special]).view(np.float32)
    f = f[~np.isnan(f)]
    mine = orc.f32_to_bf16(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    qnan = orc.f32_to_bf16(np.array([0x7F800001, 0xFFC00000], np.uint32).view(np.float32))
    assert np.isnan(bf16_bits_to_f32(qnan)).all() and ((qnan & 0x0040) != 0).all()




# ------------------------------------------------------------ routing pins


def pin_route_golden(orc):
    g = _load("routing_gate_hand.json")
    z = np.array([g["logits"]], np.float32)
    ids, w = orc.topk_route(z, 3, "softmax")
    assert ids[0].tolist() == g["ids_k3"], ids
    e3 = math.exp(-3.0)
    want = np.array([1.0, e3, e3]) / (1.0 + 2.0 * e3)
    assert np.allclose(w[0], want, rtol=1e-15, atol=0), w
    ids, w = orc.topk_route(z, 3, "sigmoid")
    s = lambda v: 1.0 / (1.0 + math.exp(-v))
    want = np.array([s(5), s(2), s(2)]) / (s(5) + 2 * s(2))
    assert ids[0].tolist() == g["ids_k3"] and np.allclose(w[0], want, rtol=1e-15, atol=0)
    ids, _ = orc.topk_route(z, 5, "softmax")
    assert ids[0].tolist() == g["ids_k5"], ids


def pin_route_equal_logits(orc):
    """All logits equal: experts 0..K-1, every weight 1/K, for both rules."""
    z = np.full((3, 16), 0.75, np.float32)
    for kind in ("softmax", "sigmoid"):
        ids, w = orc.topk_route(z, 5, kind)
        assert (ids == np.arange(5)).all()
        assert np.allclose(w, 0.2, rtol=1e-15, atol=0)


def pin_route_library_order(orc):
    """Selection equals numpy's stable descending sort, also with many ties."""
    rng = np.random.default_rng(14)
    for z in (rng.standard_normal((40, 256)).astype(np.float32),
              (np.round(rng.standard_normal((40, 256)) * 2) / 2).astype(np.float32)):
        ids, _ = orc.topk_route(z, 8, "sigmoid")
        ref = np.argsort(-z, axis=1, kind="stable")[:, :8]
        assert np.array_equal(ids, ref)


def pin_route_library_weights(orc):
    """Weights equal scipy's softmax / expit over the selected logits."""
    from scipy.special import expit, softmax
    rng = np.random.default_rng(15)
    z = (3 * rng.standard_normal((30, 384))).astype(np.float32)
    ids, w = orc.topk_route(z, 8, "softmax")
    sel = np.take_along_axis(z, ids, axis=1).astype(np.float64)
    assert np.allclose(w, softmax(sel, axis=1), rtol=1e-13, atol=0)
    ids, w = orc.topk_route(z, 8, "sigmoid")
    sel = np.take_along_axis(z, ids, axis=1).astype(np.float64)
    e = expit(sel)
    assert np.allclose(w, e / e.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)


def pin_pack_array_library(orc):
    """Array packing: high half the expert id, low half torch's bf16 of the weight."""
    rng = np.random.default_rng(16)
    ids = rng.integers(0, 65536, 5000).astype(np.int32)
    ties = ((rng.integers(0, 2**16, 1000) << 16) | 0x8000).astype(np.uint32).view(np.float32)
    w = np.concatenate([rng.random(4000).astype(np.float32), ties])
    w[~np.isfinite(w)] = np.float32(0.5)
    got = orc.pack_topk_ids(ids, w).view(np.uint32)
    ref_lo = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got >> 16, ids.astype(np.uint32))
    assert np.array_equal((got & 0xFFFF).astype(np.uint16), ref_lo)




def _every_bf16_weight():
    """All finite bf16 bit patterns of magnitude <= 2^100 (products stay finite)."""
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = bf16_bits_to_f32(b)
    keep = np.isfinite(f) & (np.abs(f) <= 2.0 ** 100)
    return b[keep], f[keep]


def pin_weight_decode_exhaustive(orc):
    """With one slot, a row of ones, zero shared and scale 1, out is the
    decoded weight itself: every finite bf16 weight, the same words packed
    beside a range of expert ids, and their fp32 widenings."""
    bits, vals = _every_bf16_weight()
    T = bits.size
    x = _bits(np.ones((1, 8)))
    idx = np.zeros((T, 1), np.int32)
    zero = np.zeros((T, 8), np.uint16)
    want = np.repeat(vals.astype(np.float64)[:, None], 8, axis=1)
    r = orc.moe_finalize(x, idx, bits.reshape(T, 1), "bf16", 1.0, zero)
    assert np.array_equal(r["out"], want)
    experts = (np.arange(T) % 65536).astype(np.uint32)
    words = ((experts << 16) | bits.astype(np.uint32)).view(np.int32).reshape(T, 1)
    r = orc.moe_finalize(x, idx, words, "packed", 1.0, zero)
    assert np.array_equal(r["out"], want)
    r = orc.moe_finalize(x, idx, vals.reshape(T, 1), "fp32", 1.0, zero)
    assert np.array_equal(r["out"], want)


# ------------------------------------------- all-reduce-fused finalize pins
#
# The finalize of R tensor-parallel ranks summed over the ranks, then the
# residual add and RMSNorm ("[Kimi K2.5] Fuse deferred MoE finalize into
# next-layer AR + residual + RMSNorm", Summary; Numerics & speed).


def _rand_ranks(seed, R, T=4, K=3, H=24, wkind="fp32", P=None):
    """R ranks with their own rows (different row counts), maps, weights and
    shared outputs."""
    ranks = []
    for r in range(R):
        x, idx, w, shared, _, _ = _rand_problem(seed * 100 + r, T=T, K=K, H=H,
                                                P=(P or T * K + 5) + 3 * r)
        w[:, 0] = -w[:, 0]                 # a negative weight on every rank
        if wkind == "bf16":
            w = _bits(w)
        elif wkind == "packed":
            experts = (5 * np.arange(K)[None, :] + np.arange(T)[:, None] + r).astype(np.uint32)
            w = ((experts << 16) | _bits(w).astype(np.uint32)).view(np.int32)
        ranks.append({"permuted_out": x, "idx": idx, "weights": w, "shared": shared})
    return ranks


def _torch_rms_norm(s, gamma_bits, eps):
    """RMSNorm of float64 rows by torch's own routine."""
    g = torch.from_numpy(bf16_bits_to_f32(gamma_bits).astype(np.float64))
    return torch.nn.functional.rms_norm(torch.from_numpy(s), (s.shape[1],), weight=g,
                                        eps=eps).numpy()


def pin_ar_golden_hand_worked(orc):
    g = _load("hand_worked_ar_r2_t2_k2_h3.json")
    ranks = [{"permuted_out": _bits(r["permuted_out"]), "idx": np.array(r["idx"], np.int32),
              "weights": np.array(r["weights_fp32"], np.float32), "shared": _bits(r["shared"])}
             for r in g["ranks"]]
    res, gamma = _bits(g["residual"]), _bits(g["gamma"])
    got = orc.moe_finalize_ar(ranks, "fp32", g["routed_scale"], res, gamma, g["eps"])
    assert np.array_equal(got["out"], np.array(g["out"], np.float64)), got["out"]
    assert np.array_equal(got["residual_out"], np.array(g["residual_out"], np.float64))
    want_norm = np.array([[float(Fraction(v)) for v in row] for row in g["norm_out"]])
    assert np.allclose(got["norm_out"], want_norm, rtol=1e-15, atol=0), got["norm_out"]
    # each rank's own partial is the single-rank finalize of its operands
    for rk, r in zip(ranks, g["ranks"]):
        one = orc.moe_finalize(rk["permuted_out"], rk["idx"], rk["weights"], "fp32",
                               g["routed_scale"], rk["shared"])
        assert np.array_equal(one["out"], np.array(r["partial"], np.float64))


def pin_ar_single_rank_is_the_finalize(orc):
    """With one rank the all-reduce is the identity: exactly the finalize."""
    for seed, wkind in ((1, "fp32"), (2, "bf16"), (3, "packed")):
        rk = _rand_ranks(seed, 1, wkind=wkind)[0]
        _, _, _, _, res, gamma = _rand_problem(seed, T=4, K=3, H=24, with_norm=True)
        a = orc.moe_finalize_ar([rk], wkind, 2.5, res, gamma, 1e-6)
        b = orc.moe_finalize(rk["permuted_out"], rk["idx"], rk["weights"], wkind, 2.5,
                             rk["shared"], res, gamma, 1e-6)
        for key in b:
            assert np.array_equal(a[key], b[key]), (wkind, key)


def pin_ar_equals_one_rank_over_all_slots(orc):
    """R ranks equal one rank whose buffer stacks the ranks' rows and whose
    K*R slots are the ranks' slots side by side (rows offset into the stack),
    plus every rank's shared output, summed here in double; the RMSNorm of
    that sum by torch's routine."""
    for seed, R, wkind in ((11, 2, "fp32"), (12, 3, "bf16"), (13, 4, "packed"),
                           (14, 8, "fp32")):
        ranks = _rand_ranks(seed, R, wkind=wkind)
        _, _, _, _, res, gamma = _rand_problem(seed, T=4, K=3, H=24, with_norm=True)
        eps = 1e-6
        got = orc.moe_finalize_ar(ranks, wkind, 2.5, res, gamma, eps)
        offsets = np.cumsum([0] + [rk["permuted_out"].shape[0] for rk in ranks])[:-1]
        x = np.concatenate([rk["permuted_out"] for rk in ranks])
        idx = np.concatenate([rk["idx"] + off for rk, off in zip(ranks, offsets)], axis=1)
        w = np.concatenate([rk["weights"] for rk in ranks], axis=1)
        zero = np.zeros_like(ranks[0]["shared"])
        routed = orc.moe_finalize(x, idx.astype(np.int32), w, wkind, 2.5, zero)["out"]
        shared = sum(bf16_bits_to_f32(rk["shared"]).astype(np.float64) for rk in ranks)
        m = routed + shared
        s = m + bf16_bits_to_f32(res)
        assert np.allclose(got["out"], m, rtol=1e-13, atol=1e-13), (R, wkind)
        assert np.allclose(got["residual_out"], s, rtol=1e-13, atol=1e-13), (R, wkind)
        assert np.allclose(got["norm_out"], _torch_rms_norm(s, gamma, eps), rtol=1e-12,
                           atol=1e-13), (R, wkind)


def pin_ar_rank_order(orc):
    """The sum over ranks does not depend on which rank is which."""
    ranks = _rand_ranks(21, 4)
    _, _, _, _, res, gamma = _rand_problem(21, T=4, K=3, H=24, with_norm=True)
    a = orc.moe_finalize_ar(ranks, "fp32", 1.5, res, gamma, 1e-6)
    b = orc.moe_finalize_ar([ranks[i] for i in (2, 0, 3, 1)], "fp32", 1.5, res, gamma, 1e-6)
    for key in a:
        assert np.allclose(a[key], b[key], rtol=1e-13, atol=1e-13), key


def pin_ar_tensor_parallel_split(orc):
    """Splitting one rank's expert rows and shared output into R equal
    shares (exact: R is a power of two) over R ranks with the same routing
    gives the one-rank result: the all-reduce sums, it does not average."""
    x, idx, w, shared, res, gamma = _rand_problem(31, T=5, K=4, H=40, with_norm=True)
    one = orc.moe_finalize(x, idx, w, "fp32", 2.5, shared, res, gamma, 1e-6)
    for R in (2, 4, 8):
        share = lambda b: _bits(bf16_bits_to_f32(b).astype(np.float64) / R)
        assert np.array_equal(bf16_bits_to_f32(share(x)) * R, bf16_bits_to_f32(x))
        ranks = [{"permuted_out": share(x), "idx": idx, "weights": w, "shared": share(shared)}
                 for _ in range(R)]
        got = orc.moe_finalize_ar(ranks, "fp32", 2.5, res, gamma, 1e-6)
        for key in one:
            assert np.allclose(got[key], one[key], rtol=1e-13, atol=1e-13), (R, key)


def pin_ar_bad_index(orc):
    """Each rank's indices are checked against that rank's own row count."""
    ranks = _rand_ranks(41, 2, P=12)       # rank 0 has 12 rows, rank 1 has 15
    ranks[1]["idx"] = ranks[1]["idx"].copy()
    ranks[1]["idx"][0, 0] = 14             # valid on rank 1 only
    orc.moe_finalize_ar(ranks, "fp32", 1.0)      # the valid maps are accepted
    for r, bad in ((0, 12), (1, 15), (1, -1), (0, -1)):
        rr = [dict(rk) for rk in ranks]
        j = rr[r]["idx"].copy()
        j[1, 2] = bad
        rr[r]["idx"] = j
        try:
            orc.moe_finalize_ar(rr, "fp32", 1.0)
        except ValueError:
            continue
        raise AssertionError(f"rank {r} index {bad} accepted")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
