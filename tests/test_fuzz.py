"""Seeded random sweep of the finalize's argument space against the oracle:
sizes (including H % 8 != 0), weight encodings, RMSNorm or not, launch
hints, 2-byte-offset (unaligned) operands and in-place outputs."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import bf16_dev, compare, run_oracle, to_device

pytestmark = pytest.mark.gpu

N_CASES = 80


def _case(i):
    rng = np.random.default_rng(1000 + i)
    K = int(rng.choice([1, 2, 3, 4, 6, 8, 9, 16, 32]))
    T = int(rng.integers(1, max(2, 2000 // K)))
    T = min(T, 600)
    H = int(rng.choice([8, 64, 136, 1024, 2048, int(rng.integers(1, 2049))]))
    return dict(T=T, K=K, H=H, wkind=str(rng.choice(["fp32", "bf16", "packed"])),
                norm=bool(rng.integers(2)), unaligned=bool(rng.random() < 0.25),
                in_place=bool(rng.random() < 0.25), scale=float(rng.choice([1.0, 2.5, 0.5])),
                splits=int(rng.choice([0, 0, 0, 1, 2, 3, 5, 16])),
                threads=int(rng.choice([0, 0, 32, 64, 128, 256])), seed=i)


def _unaligned(t):
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = flat[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_case(cuda_lib, orc, i):
    c = _case(i)
    T, K, H = c["T"], c["K"], c["H"]
    nb = max(K + 1, (T * K + 7) // 8)
    wl = W.synth("fuzz", T=T, K=K, H=H, E=2 * nb + 64, tile=32, P=nb * 32,
                 weight_rule="sigmoid", wkind=c["wkind"], routed_scale=c["scale"],
                 with_norm=c["norm"], seed=c["seed"], require_all=False)
    dev = to_device(wl)
    if c["unaligned"]:
        for k in ("x", "shared", "residual", "gamma"):
            if k in dev:
                dev[k] = _unaligned(dev[k])
    try:
        plan = cuda_lib.plan(T, K, H, c["norm"], not c["unaligned"] and H % 8 == 0,
                             splits=c["splits"], threads=c["threads"])
    except cuda_lib.MoefError:
        c["splits"] = c["threads"] = 0          # the hint does not fit this shape
    kw = {}
    if c["in_place"]:
        kw["out"] = dev["shared"] = dev["shared"].clone()
        if c["norm"]:
            kw["residual_out"] = dev["residual"] = dev["residual"].clone()
    res = cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], wl.wkind, dev["shared"],
                                routed_scale=wl.routed_scale, residual=dev.get("residual"),
                                gamma=dev.get("gamma"), eps=wl.eps, splits=c["splits"],
                                threads=c["threads"], **kw)
    torch.cuda.synchronize()
    compare(res, run_oracle(orc, wl), f"case {i} {c}: ")


N_AR_CASES = 40


def _ar_case(i):
    rng = np.random.default_rng(5000 + i)
    R = int(rng.integers(1, 9))
    K = int(rng.choice([1, 2, 3, 4, 8, 9, 16, 32]))
    T = int(rng.integers(1, max(2, 600 // (R * K) + 2)))
    H = int(rng.choice([8, 64, 136, 1024, 7168, int(rng.integers(1, 2049))]))
    return dict(R=R, T=T, K=K, H=H, wkind=str(rng.choice(["fp32", "bf16", "packed"])),
                norm=bool(rng.integers(2)), unaligned=bool(rng.random() < 0.25),
                in_place=bool(rng.random() < 0.25), scale=float(rng.choice([1.0, 2.5, 0.5])),
                seed=i)


@pytest.mark.parametrize("i", range(N_AR_CASES))
def test_fuzz_allreduce_case(cuda_lib, orc, i):
    """The all-reduce-fused finalize over random rank counts, sizes,
    encodings, epilogues, unaligned operands and in-place residuals: the
    one-shot against the oracle, the two-phase form bit-identical to it."""
    from test_allreduce import oracle_ar
    c = _ar_case(i)
    R, T, K, H = c["R"], c["T"], c["K"], c["H"]
    nb = max(K + 1, (T * K + 7) // 8)
    g = W.tp_group("fuzz_ar", R, T=T, K=K, H=H, E=2 * nb + 64, tile=32, P=nb * 32,
                   wkind=c["wkind"], routed_scale=c["scale"], with_norm=c["norm"],
                   seed=c["seed"])
    move = _unaligned if c["unaligned"] else (lambda t: t)
    ranks = []
    for wl in g.ranks:
        d = to_device(wl)
        ranks.append({"permuted_out": move(d["x"]), "idx_map": d["idx"], "weights": d["w"],
                      "shared_out": move(d["shared"])})
    ep = {}
    if g.with_norm:
        ep = {"residual": move(bf16_dev(g.residual)), "gamma": move(bf16_dev(g.gamma)),
              "eps": g.eps}
        if c["in_place"]:
            ep["residual_out"] = ep["residual"]
    ref = oracle_ar(orc, g)
    a = cuda_lib.moe_finalize_allreduce(ranks, g.wkind, routed_scale=g.routed_scale, **ep)
    torch.cuda.synchronize()
    compare(a, ref, f"case {i} {c}: ")
    if c["in_place"] and g.with_norm:
        return                      # the residual has been overwritten
    parts = [cuda_lib.moe_finalize_partial(r["permuted_out"], r["idx_map"], r["weights"],
                                           g.wkind, r["shared_out"], routed_scale=g.routed_scale)
             for r in ranks]
    b = cuda_lib.moe_finalize_allreduce_reduce(parts, **ep)
    torch.cuda.synchronize()
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key].view(torch.int16), b[key].view(torch.int16)), (i, key)
