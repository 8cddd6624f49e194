"""moe_finalize_host: the finalize on pinned host buffers, read and written
in place by the kernel.  Same results as the device-buffer call, and the
oracle's within tolerance."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import bits_of, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _pinned(a):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
        else torch.from_numpy(a)
    return t.pin_memory()


@pytest.mark.parametrize("name", ["fused_norm_bs16", "decode_bs1_packed", "tiny"])
def test_host_buffers_match_device_and_oracle(cuda_lib, orc, name):
    wl = W.make(name)
    h = {"x": _pinned(wl.permuted_out), "idx": _pinned(wl.idx), "w": _pinned(wl.weights),
         "shared": _pinned(wl.shared)}
    if wl.with_norm:
        h["residual"], h["gamma"] = _pinned(wl.residual), _pinned(wl.gamma)
    res = cuda_lib.moe_finalize_host(h["x"], h["idx"], h["w"], wl.wkind, h["shared"],
                                     routed_scale=wl.routed_scale, residual=h.get("residual"),
                                     gamma=h.get("gamma"), eps=wl.eps)
    torch.cuda.synchronize()
    for t in res.values():
        assert t.device.type == "cpu" and t.is_pinned()
    compare(res, run_oracle(orc, wl), f"{name} host: ")
    dev = run_gpu(cuda_lib, wl)
    for key in res:
        assert np.array_equal(bits_of(res[key]), bits_of(dev[key])), key


def test_host_buffers_must_be_pinned(cuda_lib):
    wl = W.make("tiny")
    x = torch.from_numpy(wl.permuted_out.view(np.int16)).view(torch.bfloat16)   # pageable
    with pytest.raises(ValueError):
        cuda_lib.moe_finalize_host(x, torch.from_numpy(wl.idx), torch.from_numpy(wl.weights),
                                   "fp32", torch.from_numpy(wl.shared.view(np.int16)).view(
                                       torch.bfloat16))
