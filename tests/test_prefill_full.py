"""The T=16384, K=8, H=7168 residual + RMSNorm workload at full size, in the
launch configuration the benchmark times (automatic plan, out not written):
every element against the fp64 oracle, plus properties on every row."""
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import assert_close, f64_of, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prefill():
    return W.make("prefill_t16384")


def test_prefill_every_element_and_properties(cuda_lib, orc, prefill):
    wl = prefill
    dev = to_device(wl)
    res = run_gpu(cuda_lib, wl, dev, write_out=False)
    assert res["out"] is None

    # every token, every column: the C oracle does the whole workload in seconds
    ref = orc.moe_finalize(wl.permuted_out, wl.idx, wl.weights, wl.wkind, wl.routed_scale,
                           wl.shared, wl.residual, wl.gamma, wl.eps, want_out=False)
    for key in ("residual_out", "norm_out"):
        assert_close(f64_of(res[key]), ref[key], "prefill " + key)
    del ref

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
