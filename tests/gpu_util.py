"""Helpers for the GPU tests: move a workload to the device, run the CUDA
path, compare with the oracle under the stated tolerance."""
import numpy as np
import torch

# |gpu - oracle| <= 2^-7 * |oracle| + 2e-3, elementwise, on every bf16 output.
REL_TOL = 2.0 ** -7
ABS_TOL = 2e-3


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of(t: torch.Tensor) -> np.ndarray:
    return (bits_of(t).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def weights_dev(wl) -> torch.Tensor:
    if wl.wkind == "fp32":
        return torch.from_numpy(np.ascontiguousarray(wl.weights)).cuda()
    if wl.wkind == "bf16":
        return bf16_dev(wl.weights)
    return torch.from_numpy(np.ascontiguousarray(wl.weights)).cuda()


def to_device(wl) -> dict:
    d = {"x": bf16_dev(wl.permuted_out),
         "idx": torch.from_numpy(np.ascontiguousarray(wl.idx)).cuda(),
         "w": weights_dev(wl),
         "shared": bf16_dev(wl.shared)}
    if wl.with_norm:
        d["residual"] = bf16_dev(wl.residual)
        d["gamma"] = bf16_dev(wl.gamma)
    return d


def run_gpu(mf, wl, dev=None, **kw) -> dict:
    dev = dev or to_device(wl)
    res = mf.moe_finalize(dev["x"], dev["idx"], dev["w"], wl.wkind, dev["shared"],
                          routed_scale=wl.routed_scale, residual=dev.get("residual"),
                          gamma=dev.get("gamma"), eps=wl.eps, **kw)
    torch.cuda.synchronize()
    return res


def run_oracle(orc, wl):
    return orc.moe_finalize(wl.permuted_out, wl.idx, wl.weights, wl.wkind, wl.routed_scale,
                            wl.shared, wl.residual, wl.gamma, wl.eps)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str, rel=REL_TOL, abs_=ABS_TOL):
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    bound = rel * np.abs(ref) + abs_
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; first at "
            f"{tuple(i)}: gpu={gpu[tuple(i)]!r} oracle={ref[tuple(i)]!r}")


def compare(res_gpu: dict, res_ref: dict, what: str = ""):
    for key, ref in res_ref.items():
        if ref is None or res_gpu.get(key) is None:
            continue
        assert_close(f64_of(res_gpu[key]), ref, f"{what}{key}")
