"""moe_finalize_unfused_noalloc, the entry point for callers that cannot
allocate device memory (engines with a fixed memory plan, plugins without an
allocator): it must give the same result as
moe_finalize_unfused with a caller-owned workspace, call after call, even
though every call reuses one fixed scratch array inside the library.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test; it also passes on its own."""
import ctypes

import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import assert_close, bits_of, f64_of, to_device

pytestmark = pytest.mark.gpu


def _raw_noalloc(mf, wl, dev, outs):
    """The new entry point, called through the C ABI with raw pointers."""
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return mf.lib().moe_finalize_unfused_noalloc(
        p(dev["x"]), wl.P, p(dev["idx"]), p(dev["w"]), mf.WKIND[wl.wkind], wl.routed_scale,
        p(dev["shared"]), p(dev.get("residual")), p(dev.get("gamma")), wl.eps,
        p(outs["out"]), p(outs.get("residual_out")), p(outs.get("norm_out")),
        wl.T, wl.K, wl.H, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _with_workspace(mf, wl, dev):
    ws = torch.empty(mf.unfused_workspace_bytes(wl.T, wl.H), dtype=torch.uint8, device="cuda")
    res = mf.moe_finalize_unfused(dev["x"], dev["idx"], dev["w"], wl.wkind, dev["shared"],
                                  routed_scale=wl.routed_scale, residual=dev.get("residual"),
                                  gamma=dev.get("gamma"), eps=wl.eps, workspace=ws)
    torch.cuda.synchronize()
    return res


def test_noalloc_matches_workspace_path_two_calls_in_a_row(cuda_lib):
    # two different problems back to back: the second finds the first one's
    # data in the shared scratch and must not be affected by it
    for name in ("decode_bs256", "fused_norm_bs16"):
        wl = W.make(name)
        dev = to_device(wl)
        ref = _with_workspace(cuda_lib, wl, dev)
        outs = {k: torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
                for k in ref if ref[k] is not None}
        assert _raw_noalloc(cuda_lib, wl, dev, outs) == 0
        torch.cuda.synchronize()
        for key in outs:
            assert_close(f64_of(outs[key]), f64_of(ref[key]), f"{name} {key}")
            assert np.array_equal(bits_of(outs[key]), bits_of(ref[key])), key


def test_noalloc_repeated_calls_same_problem(cuda_lib):
    wl = W.make("decode_bs1_packed")
    dev = to_device(wl)
    ref = _with_workspace(cuda_lib, wl, dev)["out"]
    for _ in range(2):
        out = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
        assert _raw_noalloc(cuda_lib, wl, dev, {"out": out}) == 0
        torch.cuda.synchronize()
        assert_close(f64_of(out), f64_of(ref), "packed decode")


def test_noalloc_rejects_requests_beyond_its_scratch(cuda_lib):
    wl = W.make("tiny")
    dev = to_device(wl)
    H = wl.H
    T_max = (8 << 20) // (2 * H)
    # a request one token past the limit is refused before anything runs
    big = {"x": dev["x"], "idx": torch.zeros((T_max + 1, wl.K), dtype=torch.int32, device="cuda"),
           "w": torch.zeros((T_max + 1, wl.K), dtype=torch.float32, device="cuda"),
           "shared": torch.zeros((T_max + 1, H), dtype=torch.bfloat16, device="cuda")}
    wl_big = W.Workload(**{**wl.__dict__, "T": T_max + 1})
    out = torch.zeros((T_max + 1, H), dtype=torch.bfloat16, device="cuda")
    assert _raw_noalloc(cuda_lib, wl_big, big, {"out": out}) == 2      # MOEF_ERR_SHAPE
    with pytest.raises(ValueError):
        cuda_lib.moe_finalize_unfused_noalloc(big["x"], big["idx"], big["w"], "fp32",
                                              big["shared"], out=out)


def test_noalloc_at_the_largest_accepted_size(cuda_lib, orc):
    """T * H * 2 equal to the scratch size exactly (T = 4096 at H = 1024) is
    accepted and matches both the workspace path, bit for bit, and the
    oracle within the unfused path's derived tolerance (its intermediate is
    rounded to bf16)."""
    from gpu_util import run_oracle
    from test_unfused import _check
    H = 1024
    T = (8 << 20) // (2 * H)
    wl = W.synth("noalloc_max", T=T, K=4, H=H, E=2048, tile=32, P=32 * 2048,
                 weight_rule="sigmoid", routed_scale=2.5, seed=5, require_all=False)
    assert T * H * 2 == 8 << 20
    dev = to_device(wl)
    ref = _with_workspace(cuda_lib, wl, dev)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _raw_noalloc(cuda_lib, wl, dev, {"out": out}) == 0
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(out), bits_of(ref["out"]))
    _check({"out": out}, run_oracle(orc, wl), wl, "noalloc at 8 MiB: ")
