"""Stream-order guarantees of the finalize, which launches as a programmatic
dependent of the previous kernel: a kernel that rewrites the inputs right
before it on the same stream must be fully visible to it, and a kernel
right after it must see its outputs.  Fresh data every iteration, so a read
that slipped ahead of the dependency wait would show as a mismatch."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import bits_of, compare, run_oracle, to_device

pytestmark = pytest.mark.gpu


def test_producer_kernel_then_finalize_same_stream(cuda_lib, orc):
    wl = W.make("fused_norm_bs16")
    dev = to_device(wl)
    rng = np.random.default_rng(0)
    staging = {k: torch.empty_like(dev[k]) for k in ("x", "shared", "residual")}
    outs = {k: torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
            for k in ("out", "residual_out", "norm_out")}
    for it in range(6):
        # new inputs on the host, staged to the device, then written into the
        # finalize's input buffers by kernels on the same stream just before it
        x = W.to_bf16_bits(rng.standard_normal(wl.permuted_out.shape))
        sh = W.to_bf16_bits(rng.standard_normal(wl.shared.shape))
        rs = W.to_bf16_bits(2 * rng.standard_normal(wl.residual.shape))
        for k, a in (("x", x), ("shared", sh), ("residual", rs)):
            staging[k].copy_(torch.from_numpy(a.view(np.int16)).view(torch.bfloat16))
        torch.cuda.synchronize()
        for k in ("x", "shared", "residual"):
            torch.mul(staging[k], 1.0, out=dev[k])          # producer kernels
        cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                              routed_scale=wl.routed_scale, residual=dev["residual"],
                              gamma=dev["gamma"], eps=wl.eps, **outs)
        consumed = outs["norm_out"].float() * 1.0             # consumer kernel
        torch.cuda.synchronize()
        wl_it = W.Workload(**{**wl.__dict__, "permuted_out": x, "shared": sh, "residual": rs})
        ref = run_oracle(orc, wl_it)
        compare(outs, ref, f"iteration {it}: ")
        assert torch.equal(consumed, outs["norm_out"].float())


def test_two_streams_concurrently(cuda_lib, orc):
    wa, wb = W.make("decode_bs256"), W.make("fused_norm_bs16")
    da, db = to_device(wa), to_device(wb)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    res = {}
    for _ in range(3):
        with torch.cuda.stream(sa):
            res["a"] = cuda_lib.moe_finalize(da["x"], da["idx"], da["w"], "fp32", da["shared"],
                                             routed_scale=wa.routed_scale)
        with torch.cuda.stream(sb):
            res["b"] = cuda_lib.moe_finalize(db["x"], db["idx"], db["w"], "fp32", db["shared"],
                                             routed_scale=wb.routed_scale,
                                             residual=db["residual"], gamma=db["gamma"],
                                             eps=wb.eps)
    torch.cuda.synchronize()
    compare(res["a"], run_oracle(orc, wa), "stream a: ")
    compare(res["b"], run_oracle(orc, wb), "stream b: ")


def test_routing_ready_with_producer_of_rows(cuda_lib):
    """With MOEF_FLAG_ROUTING_READY the row map may be read early, but rows
    written by the kernel just before must still be seen."""
    wl = W.make("decode_bs256")
    dev = to_device(wl)
    base = cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                                 routed_scale=wl.routed_scale)["out"].clone()
    src = dev["x"].clone()
    dev["x"].zero_()
    torch.cuda.synchronize()
    for pdl in (True, False):
        dev["x"].zero_()
        torch.cuda.synchronize()
        torch.mul(src, 1.0, out=dev["x"])                       # producer of the rows
        out = cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                                    routed_scale=wl.routed_scale, routing_ready=True,
                                    pdl=pdl)["out"]
        torch.cuda.synchronize()
        assert np.array_equal(bits_of(out), bits_of(base)), pdl
