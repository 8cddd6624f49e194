"""Accuracy of the fused finalize against the unfused kernels, both against
the fp64 oracle: the comparison "[Kimi K2.5] Fuse deferred MoE finalize into
next-layer AR + residual + RMSNorm" makes (Numerics & speed: mean relative
error of residual and norm against a high-precision truth, fused vs the
separate-kernel fallback).  Here fusing removes bf16 roundings (the combined
rows, then out), so the fused kernel must be at least as accurate."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import f64_of, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _mean_rel(gpu, ref):
    return float(np.abs(gpu - ref).mean() / np.abs(ref).mean())


@pytest.mark.parametrize("name", ["fused_norm_bs16", "decode_bs256"])
def test_fused_at_least_as_accurate_as_unfused(cuda_lib, orc, name, capsys):
    wl = W.make(name)
    dev = to_device(wl)
    ref = run_oracle(orc, wl)
    fused = run_gpu(cuda_lib, wl, dev)
    unf = cuda_lib.moe_finalize_unfused(dev["x"], dev["idx"], dev["w"], wl.wkind, dev["shared"],
                                        routed_scale=wl.routed_scale,
                                        residual=dev.get("residual"), gamma=dev.get("gamma"),
                                        eps=wl.eps)
    torch.cuda.synchronize()
    report = {}
    for key in ref:
        f = _mean_rel(f64_of(fused[key]), ref[key])
        u = _mean_rel(f64_of(unf[key]), ref[key])
        report[key] = (f, u)
        assert f <= u * 1.0001, (key, f, u)
        assert f < 2.0 ** -8                      # a single bf16 rounding: at most 2^-9 relative
    with capsys.disabled():
        print(f"\n{name}: mean relative error vs fp64, fused / unfused: " +
              ", ".join(f"{k} {f:.3e} / {u:.3e}" for k, (f, u) in report.items()))


def test_allreduce_fused_keeps_single_rounding_accuracy(cuda_lib, orc, capsys):
    """The all-reduce-fused finalize over 8 ranks (the Kimi K2.5 page's
    shape: bs = 16, H = 7168, top-8) sums the ranks' partials in fp32 and
    rounds once, so its mean relative error stays that of one bf16
    rounding.  For comparison, an exchange of bf16-rounded rank outputs (each
    rank's finalize rounded to bf16, then summed; computed here on the host
    from the GPU's own per-rank outputs) carries the extra rounding the
    page's fused kernel had."""
    from test_allreduce import one_shot, oracle_ar, ranks_dev
    g = W.tp_decode(8, 16)
    ref = oracle_ar(orc, g)
    rd = ranks_dev(g)
    fused = one_shot(cuda_lib, g, rd)
    # bf16 exchange: per-rank finalize outputs rounded to bf16, summed in fp64
    m = sum(f64_of(cuda_lib.moe_finalize(r["permuted_out"], r["idx_map"], r["weights"], g.wkind,
                                         r["shared_out"], routed_scale=g.routed_scale)["out"])
            for r in rd)
    torch.cuda.synchronize()
    s = m + W.bf16_bits_to_f32(g.residual).astype(np.float64)
    s_bits = W.to_bf16_bits(s)        # residual_out as a bf16 consumer holds it
    norm = W.to_bf16_bits(orc.rmsnorm_bf16(s_bits, g.gamma, g.eps))    # stored as bf16 too
    exch = {"residual_out": W.bf16_bits_to_f32(s_bits).astype(np.float64),
            "norm_out": W.bf16_bits_to_f32(norm).astype(np.float64)}
    report = {}
    for key in ("residual_out", "norm_out"):
        f = _mean_rel(f64_of(fused[key]), ref[key])
        e = _mean_rel(exch[key], ref[key])
        report[key] = (f, e)
        assert f < 2.0 ** -8
        assert f <= e * 1.0001, (key, f, e)
    with capsys.disabled():
        print("\nR=8 T=16: mean relative error vs fp64, fp32 partials / bf16 exchange: " +
              ", ".join(f"{k} {f:.3e} / {e:.3e}" for k, (f, e) in report.items()))
