"""The T=16384, K=8, H=7168 residual + RMSNorm workload at full size, in the
launch configuration the benchmark times (automatic plan, out not written):
sampled token rows against the fp64 oracle, properties on every row."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import compare, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prefill():
    return W.make("prefill_t16384")


def test_prefill_sampled_rows_and_properties(cuda_lib, orc, prefill):
    wl = prefill
    dev = to_device(wl)
    res = run_gpu(cuda_lib, wl, dev, write_out=False)
    assert res["out"] is None

    rng = np.random.default_rng(0)
    toks = np.unique(np.r_[0, 1, wl.T - 1, rng.choice(wl.T, 61, replace=False)])
    ref = orc.moe_finalize(wl.permuted_out, wl.idx[toks], wl.weights[toks], wl.wkind,
                           wl.routed_scale, wl.shared[toks], wl.residual[toks], wl.gamma,
                           wl.eps, want_out=False)
    sel = torch.from_numpy(toks).cuda()
    got = {k: res[k].index_select(0, sel) for k in ("residual_out", "norm_out")}
    compare(got, {k: ref[k] for k in ("residual_out", "norm_out")}, "prefill sample: ")

    r = res["residual_out"].float()
    n = res["norm_out"].float()
    g = dev["gamma"].float()
    assert torch.isfinite(r).all() and torch.isfinite(n).all()
    # a leaked 1e4 padding row would put |values| in the hundreds
    assert r.abs().max().item() < 100.0
    # every norm row has unit mean square once gamma is divided out
    ms = r.double().pow(2).mean(dim=1)
    unit = (n.double() / g.double()).pow(2).mean(dim=1)
    want = ms / (ms + wl.eps)
    assert torch.allclose(unit, want, rtol=1e-2, atol=0)
