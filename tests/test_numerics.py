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
