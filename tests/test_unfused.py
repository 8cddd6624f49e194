"""The unfused A/B baseline (combine -> bf16 workspace, shared add, residual
+ RMSNorm as separate kernels) against the fp64 oracle.

Its tolerance is derived from its arithmetic: besides the final rounding it
rounds the combined rows (c = out - shared) to bf16, then out, then
residual_out, each a relative error of at most 2^-9 of the value rounded.
So |out - ref| <= 2^-7 |ref| + 2^-8 |c| + 2e-3, residual_out adds the
rounding of out (2^-8 |out|), and norm_out scales the residual_out error by
inv_rms * gamma."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import assert_close, bits_of, f64_of, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _check(res, ref, wl, what):
    sh = W.bf16_bits_to_f32(wl.shared).astype(np.float64)
    c = np.abs(ref["out"] - sh)
    out = f64_of(res["out"])
    bound_out = 2.0 ** -7 * np.abs(ref["out"]) + 2.0 ** -8 * c + 2e-3
    assert (np.abs(out - ref["out"]) <= bound_out).all(), what + "out"
    if wl.with_norm:
        ro_ref = ref["residual_out"]
        bound_ro = 2.0 ** -7 * np.abs(ro_ref) + 2.0 ** -8 * (c + np.abs(ref["out"])) + 2e-3
        assert (np.abs(f64_of(res["residual_out"]) - ro_ref) <= bound_ro).all(), what + "r_out"
        inv = 1.0 / np.sqrt((ro_ref ** 2).mean(axis=1, keepdims=True) + wl.eps)
        g = W.bf16_bits_to_f32(wl.gamma).astype(np.float64)[None, :]
        bound_n = 2.0 ** -7 * np.abs(ref["norm_out"]) + 2.0 * bound_ro * inv * g
        assert (np.abs(f64_of(res["norm_out"]) - ref["norm_out"]) <= bound_n).all(), what + "norm"


def _run(mf, wl, dev, **kw):
    res = mf.moe_finalize_unfused(dev["x"], dev["idx"], dev["w"], wl.wkind, dev["shared"],
                                  routed_scale=wl.routed_scale, residual=dev.get("residual"),
                                  gamma=dev.get("gamma"), eps=wl.eps, **kw)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("name", ["tiny", "decode_bs1_packed", "decode_bs256", "fused_norm_bs16"])
def test_unfused_named(cuda_lib, orc, name):
    wl = W.make(name)
    dev = to_device(wl)
    _check(_run(cuda_lib, wl, dev), run_oracle(orc, wl), wl, f"{name}: ")


@pytest.mark.parametrize("T,K,H,norm", [(5, 3, 100, True), (300, 8, 7168, False),
                                        (3, 9, 7176, True), (1, 1, 8, False)])
def test_unfused_shapes(cuda_lib, orc, T, K, H, norm):
    nb = max(K + 1, (T * K + 7) // 8)
    wl = W.synth("u", T=T, K=K, H=H, E=2 * nb + 64, tile=32, P=nb * 32, weight_rule="sigmoid",
                 routed_scale=2.5, with_norm=norm, seed=T + K + H, require_all=False)
    _check(_run(cuda_lib, wl, to_device(wl)), run_oracle(orc, wl), wl, f"T={T} H={H}: ")


def test_unfused_matches_fused_where_no_extra_rounding(cuda_lib):
    """With zero shared output and no residual the only extra rounding is
    bf16(bf16(c) + 0) = bf16(c): out is bit-identical to the fused kernel."""
    wl = W.make("decode_bs256")
    dev = to_device(wl)
    dev["shared"] = torch.zeros_like(dev["shared"])
    a = cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                              routed_scale=wl.routed_scale)["out"]
    b = _run(cuda_lib, wl, dev)["out"]
    assert np.array_equal(bits_of(a), bits_of(b))


def test_unfused_workspace_rules(cuda_lib):
    wl = W.make("tiny")
    dev = to_device(wl)
    need = cuda_lib.unfused_workspace_bytes(wl.T, wl.H)
    assert need == wl.T * wl.H * 2
    small = torch.empty(need - 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.MoefError) as e:
        _run(cuda_lib, wl, dev, workspace=small)
    assert e.value.status == 2
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")   # stale contents
    res = _run(cuda_lib, wl, dev, workspace=ws)
    assert torch.isfinite(res["out"].float()).all()
