"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Tolerance (every bf16 output): |gpu - oracle| <= 2^-7 |oracle| + 2e-3.
Bit-exact where the arithmetic leaves no choice (one slot of weight 1,
zero weights, identical tokens, launch shape changes for out/residual_out).
"""
import ctypes
import dataclasses
import types

import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import (assert_close, bf16_dev, bits_of, compare, f64_of, run_gpu, run_oracle,
                      to_device)
from test_unfused import _check as check_unfused

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "decode_bs1_packed", "decode_bs256", "fused_norm_bs16"])
def test_named_workloads(cuda_lib, orc, name):
    wl = W.make(name)
    ref = run_oracle(orc, wl)
    compare(run_gpu(cuda_lib, wl), ref, f"{name}: ")
    if wl.with_norm:
        res = run_gpu(cuda_lib, wl, write_out=False)
        assert res["out"] is None
        compare(res, ref, f"{name} (no out): ")


def test_norm_reproducible_from_residual_out(cuda_lib, orc):
    """norm_out is the RMSNorm of the bf16 residual_out the kernel emitted."""
    wl = W.make("fused_norm_bs16")
    res = run_gpu(cuda_lib, wl)
    ref = orc.rmsnorm_bf16(bits_of(res["residual_out"]), wl.gamma, wl.eps)
    assert_close(f64_of(res["norm_out"]), ref, "norm_out vs own residual_out",
                 rel=2.0 ** -8, abs_=1e-3)


CASES = [
    # (T, K, H, wkind, norm)
    (1, 1, 8, "fp32", False),
    (3, 2, 64, "bf16", True),
    (5, 3, 100, "fp32", True),         # H % 8 != 0: scalar path
    (7, 9, 136, "packed", False),      # K > 8: two slot groups
    (2, 32, 264, "fp32", True),        # K at its maximum
    (16, 8, 7168, "bf16", True),
    (3, 8, 7176, "fp32", True),        # ragged: 897 vectors
    (300, 8, 7168, "packed", False),
    (300, 6, 1000, "fp32", True),
    (700, 8, 7168, "fp32", True),      # just past the latency regime
    (2, 4, 16384, "fp32", True),       # cluster of 8 CTAs
    (2, 4, 32768, "bf16", True),       # cluster of 16 CTAs (non-portable size)
    (40, 2, 24576, "fp32", True),      # norm rows over 12-CTA clusters
    (33, 5, 40000, "bf16", False),     # several passes per slice without norm
    (9, 4, 4098, "fp32", True),        # H % 8 == 2: scalar path with cluster
    (2048, 8, 4096, "fp32", True),     # bandwidth regime, other hidden sizes
    (1500, 6, 5120, "bf16", True),
    (1200, 9, 8192, "packed", False),
    # each RMSNorm plan of the mid-size batches at H = 7168 (one wave: 4-CTA
    # clusters of 224 threads, then of 128 threads with two vectors each,
    # then 2-CTA clusters), and 3-CTA clusters of 128 threads at H = 6144
    (176, 8, 7168, "packed", True),
    (256, 8, 7168, "fp32", True),
    (300, 8, 7168, "bf16", True),
    (360, 8, 6144, "fp32", True),
]


@pytest.mark.parametrize("T,K,H,wkind,norm", CASES)
def test_random_shapes(cuda_lib, orc, T, K, H, wkind, norm):
    # about 8 rows per 32-row expert block: no block overflows in practice
    tile = 32
    n_blocks = max(K + 1, (T * K + 7) // 8)
    wl = W.synth("case", T=T, K=K, H=H, E=2 * n_blocks + 64, tile=tile,
                 P=n_blocks * tile, weight_rule="sigmoid", wkind=wkind,
                 routed_scale=2.5, with_norm=norm, seed=T * 1000 + K * 10 + H, require_all=False)
    compare(run_gpu(cuda_lib, wl), run_oracle(orc, wl), f"T={T} K={K} H={H} {wkind}: ")


def test_longest_rmsnorm_row(cuda_lib, orc):
    """H = 262144 with RMSNorm: the longest row one cluster of 16 CTAs x 256
    threads x 8 vectors can normalise; one more vector is refused."""
    H = 16 * 256 * 8 * 8
    wl = W.synth("long", T=2, K=4, H=H, E=64, tile=8, P=64, weight_rule="sigmoid",
                 routed_scale=2.5, with_norm=True, seed=31, require_all=False)
    p = cuda_lib.plan(wl.T, wl.K, H, True)
    assert p["cluster"] == 16 and p["threads"] == 256 and p["vpt"] == 8
    compare(run_gpu(cuda_lib, wl), run_oracle(orc, wl), "H=262144: ")
    with pytest.raises(cuda_lib.MoefError) as e:
        cuda_lib.plan(2, 4, H + 8, True)
    assert e.value.status == 2


@pytest.mark.parametrize("splits,threads", [(1, 0), (1, 256), (2, 0), (3, 64), (7, 128),
                                            (8, 0), (13, 96), (16, 0)])
def test_launch_shapes_agree(cuda_lib, orc, splits, threads):
    """Every legal launch shape gives the oracle's result; out and
    residual_out are bit-identical across shapes (same per-element
    arithmetic), norm_out agrees within tolerance."""
    wl = W.make("fused_norm_bs16")
    dev = to_device(wl)
    base = run_gpu(cuda_lib, wl, dev)
    res = run_gpu(cuda_lib, wl, dev, splits=splits, threads=threads)
    compare(res, run_oracle(orc, wl), f"splits={splits} threads={threads}: ")
    assert np.array_equal(bits_of(res["out"]), bits_of(base["out"]))
    assert np.array_equal(bits_of(res["residual_out"]), bits_of(base["residual_out"]))


@pytest.mark.parametrize("splits,threads", [(1, 0), (1, 32), (4, 64), (28, 32), (56, 0),
                                            (112, 32), (896, 32)])
def test_launch_shapes_agree_without_norm(cuda_lib, orc, splits, threads):
    """Without RMSNorm a row may be cut into any number of slices."""
    wl = W.make("decode_bs256")
    dev = to_device(wl)
    base = run_gpu(cuda_lib, wl, dev)
    res = run_gpu(cuda_lib, wl, dev, splits=splits, threads=threads)
    compare(res, run_oracle(orc, wl), f"splits={splits} threads={threads}: ")
    assert np.array_equal(bits_of(res["out"]), bits_of(base["out"]))


@pytest.mark.parametrize("norm,splits,threads", [
    (False, 1, 128), (False, 2, 128), (False, 4, 128), (False, 7, 128), (False, 1, 32),
    (True, 1, 128), (True, 1, 256), (True, 2, 256), (True, 4, 224), (True, 4, 128),
    (True, 16, 64)])
def test_fixed_k_and_any_k_builds_agree(cuda_lib, orc, norm, splits, threads):
    """With K = 8 a grid of more than one CTA per SM (with RMSNorm; four
    without) runs the build with K fixed at compile time, a smaller grid the
    any-K build.  The first tokens of a large batch, finalized alone in the
    same launch shape, go through the other build: every output must be
    bit-identical (same per-element arithmetic and order), and the large
    batch must match the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    limit = sms * (1 if norm else 4)
    t_small = max(1, limit // splits)
    t_large = limit // splits + 8
    assert t_small * splits <= limit < t_large * splits
    wl = W.synth("builds", T=t_large, K=8, H=7168, E=256, tile=64, P=64 * 96,
                 weight_rule="sigmoid", routed_scale=2.5, with_norm=norm, seed=splits * 7 + norm,
                 require_all=False)
    small = dataclasses.replace(
        wl, T=t_small, idx=wl.idx[:t_small], expert_ids=wl.expert_ids[:t_small],
        weights_f32=wl.weights_f32[:t_small], weights=wl.weights[:t_small],
        shared=wl.shared[:t_small], residual=None if wl.residual is None else wl.residual[:t_small])
    plan_large = cuda_lib.plan(t_large, 8, 7168, norm, splits=splits, threads=threads)
    plan_small = cuda_lib.plan(t_small, 8, 7168, norm, splits=splits, threads=threads)
    assert {k: v for k, v in plan_large.items() if k != "grid"} == \
           {k: v for k, v in plan_small.items() if k != "grid"}
    big = run_gpu(cuda_lib, wl, splits=splits, threads=threads)
    compare(big, run_oracle(orc, wl), f"T={t_large} splits={splits} threads={threads}: ")
    sub = run_gpu(cuda_lib, small, splits=splits, threads=threads)
    for key in ("out", "residual_out", "norm_out"):
        if sub.get(key) is not None:
            assert np.array_equal(bits_of(sub[key]), bits_of(big[key][:t_small])), key


def test_norm_split_beyond_cluster_limit_is_rejected(cuda_lib):
    wl = W.make("fused_norm_bs16")
    dev = to_device(wl)
    with pytest.raises(cuda_lib.MoefError) as e:
        run_gpu(cuda_lib, wl, dev, splits=17)
    assert e.value.status == 4


@pytest.mark.parametrize("name", ["decode_bs1_packed", "fused_norm_bs16", "decode_bs256"])
def test_routing_ready_flag_same_result(cuda_lib, name):
    """Reading the row map and weights before the grid dependency wait
    changes no bit of the result."""
    wl = W.make(name)
    dev = to_device(wl)
    a = run_gpu(cuda_lib, wl, dev)
    b = run_gpu(cuda_lib, wl, dev, routing_ready=True)
    c = run_gpu(cuda_lib, wl, dev, pdl=False)             # MOEF_FLAG_NO_PDL
    d = run_gpu(cuda_lib, wl, dev, routing_ready=True, pdl=False)
    for key in a:
        if a[key] is not None:
            for other in (b, c, d):
                assert np.array_equal(bits_of(a[key]), bits_of(other[key])), key


def test_one_slot_weight_one_is_the_row(cuda_lib):
    wl = W.synth("k1", T=9, K=1, H=7168, E=64, tile=16, P=256, seed=21, require_all=False)
    dev = to_device(wl)
    dev["w"] = torch.ones((9, 1), dtype=torch.float32, device="cuda")
    dev["shared"] = torch.zeros((9, 7168), dtype=torch.bfloat16, device="cuda")
    res = cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                                routed_scale=1.0)
    assert np.array_equal(bits_of(res["out"]), wl.permuted_out[wl.idx[:, 0]])


def test_zero_weights_and_zero_scale_give_shared(cuda_lib):
    wl = W.make("decode_bs256")
    dev = to_device(wl)
    res = cuda_lib.moe_finalize(dev["x"], dev["idx"], torch.zeros_like(dev["w"]), "fp32",
                                dev["shared"], routed_scale=2.5)
    assert np.array_equal(bits_of(res["out"]), wl.shared)
    res = cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                                routed_scale=0.0)
    assert np.array_equal(bits_of(res["out"]), wl.shared)


def test_slot_order_and_duplicates(cuda_lib, orc):
    wl = W.make("fused_norm_bs16")
    perm = np.random.default_rng(3).permutation(wl.K)
    wl2 = W.Workload(**{**wl.__dict__, "idx": np.ascontiguousarray(wl.idx[:, perm]),
                        "weights": np.ascontiguousarray(wl.weights[:, perm])})
    compare(run_gpu(cuda_lib, wl2), run_oracle(orc, wl), "permuted slots: ")
    # token 5 made identical to token 2: identical output rows, bit for bit
    wl3 = W.Workload(**{**wl.__dict__})
    for f in ("idx", "weights", "shared", "residual"):
        a = getattr(wl, f).copy()
        a[5] = a[2]
        setattr(wl3, f, a)
    res = run_gpu(cuda_lib, wl3)
    for key in ("out", "residual_out", "norm_out"):
        b = bits_of(res[key])
        assert np.array_equal(b[5], b[2]), key


def test_row_offsets_beyond_2_to_the_31_elements(cuda_lib, orc):
    """permuted_out of 300,000 rows x 7168 (4.3 GB, 2.15e9 elements): the
    referenced rows lie past element 2^31, so row offsets must be computed in
    64 bits.  The oracle sees a compact copy of just those rows."""
    H, P, T, K = 7168, 300_000, 6, 8
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(np.arange(P - 400, P), T * K, replace=False))
    assert rows.min() * H > 2 ** 31
    x = torch.empty((P, H), dtype=torch.bfloat16, device="cuda")
    vals = W.to_bf16_bits(rng.standard_normal((T * K, H)))
    x[torch.from_numpy(rows).cuda()] = bf16_dev(vals)
    perm = rng.permutation(T * K)
    idx = rows[perm].reshape(T, K).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    shared = W.to_bf16_bits(rng.standard_normal((T, H)))
    for norm in (False, True):
        kw = {}
        residual = gamma = None
        if norm:
            residual = W.to_bf16_bits(2 * rng.standard_normal((T, H)))
            gamma = W.to_bf16_bits(rng.uniform(0.5, 1.5, H))
            kw = dict(residual=bf16_dev(residual), gamma=bf16_dev(gamma))
        res = cuda_lib.moe_finalize(x, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                                    "fp32", bf16_dev(shared), routed_scale=2.5, eps=1e-6, **kw)
        torch.cuda.synchronize()
        ref = orc.moe_finalize(vals, perm.reshape(T, K).astype(np.int32), w, "fp32", 2.5,
                               shared, residual, gamma, 1e-6)
        compare(res, ref, f"rows past 2^31 elements, norm={norm}: ")
    del x
    torch.cuda.empty_cache()


def test_token_offsets_beyond_2_to_the_31_elements(cuda_lib, orc):
    """300,000 tokens x 7168 (each dense operand 4.3 GB): token offsets into
    shared_out, residual and the outputs pass element 2^31.  The dense inputs
    are zero except on sampled tokens, which are checked against the oracle;
    every other row must equal the weighted sum of its gathered rows."""
    H, P, T, K = 7168, 64, 300_000, 2
    rng = np.random.default_rng(12)
    x_host = W.to_bf16_bits(rng.standard_normal((P, H)))
    idx = rng.integers(0, P, (T, K)).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    samp = np.array([0, 1, 149_999, 299_592, 299_593, T - 2, T - 1])
    assert samp[-1] * H > 2 ** 31
    sh_s = W.to_bf16_bits(rng.standard_normal((len(samp), H)))
    rs_s = W.to_bf16_bits(2 * rng.standard_normal((len(samp), H)))
    gamma = W.to_bf16_bits(rng.uniform(0.5, 1.5, H))
    sel = torch.from_numpy(samp).cuda()
    x = bf16_dev(x_host)
    idx_d, w_d = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    for norm in (False, True):
        shared = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
        shared[sel] = bf16_dev(sh_s)
        kw = {}
        if norm:
            residual = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
            residual[sel] = bf16_dev(rs_s)
            kw = dict(residual=residual, gamma=bf16_dev(gamma))
        res = cuda_lib.moe_finalize(x, idx_d, w_d, "fp32", shared, routed_scale=2.5, eps=1e-6,
                                    **kw)
        torch.cuda.synchronize()
        ref = orc.moe_finalize(x_host, idx[samp], w[samp], "fp32", 2.5, sh_s,
                               rs_s if norm else None, gamma if norm else None, 1e-6)
        compare({k: v.index_select(0, sel) for k, v in res.items() if v is not None}, ref,
                f"tokens past 2^31 elements, norm={norm}: ")
        # the unfused A/B kernels index the same tensors (their own tolerance:
        # they also round the combined rows to bf16)
        unf = cuda_lib.moe_finalize_unfused(x, idx_d, w_d, "fp32", shared, routed_scale=2.5,
                                            eps=1e-6, **kw)
        torch.cuda.synchronize()
        sampled = types.SimpleNamespace(shared=sh_s, with_norm=norm, eps=1e-6, gamma=gamma)
        check_unfused({k: v.index_select(0, sel) for k, v in unf.items() if v is not None},
                      ref, sampled, f"unfused, tokens past 2^31 elements, norm={norm}: ")
        del unf
        # the other rows: routed sum only (zero shared / residual), in bf16
        routed = (w_d[:, :1] * 2.5 * x.float()[idx_d[:, 0]] +
                  w_d[:, 1:] * 2.5 * x.float()[idx_d[:, 1]])
        out = res["residual_out"] if norm else res["out"]
        keep = torch.ones(T, dtype=torch.bool, device="cuda")
        keep[sel] = False
        diff = (out.float() - routed)[keep].abs()
        assert (diff <= 2.0 ** -7 * routed[keep].abs() + 2e-3).all()
        del shared, res, routed, out, diff, kw
        torch.cuda.empty_cache()


def test_padding_never_read(cuda_lib):
    wl = W.make("decode_bs256")
    x = wl.permuted_out.copy()
    x[~wl.valid_rows] = 0x7FC0      # NaN everywhere a row is not referenced
    wl2 = W.Workload(**{**wl.__dict__, "permuted_out": x})
    res = run_gpu(cuda_lib, wl2)
    assert torch.isfinite(res["out"].float()).all()
    wl = W.make("fused_norm_bs16")
    x = wl.permuted_out.copy()
    x[~wl.valid_rows] = 0x7FC0
    res = run_gpu(cuda_lib, W.Workload(**{**wl.__dict__, "permuted_out": x}))
    for key in ("out", "residual_out", "norm_out"):
        assert torch.isfinite(res[key].float()).all(), key


def test_in_place(cuda_lib):
    wl = W.make("fused_norm_bs16")
    dev = to_device(wl)
    ref = run_gpu(cuda_lib, wl, dev)
    sh, rs = dev["shared"].clone(), dev["residual"].clone()
    cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", sh, routed_scale=1.0,
                          residual=rs, gamma=dev["gamma"], eps=wl.eps, out=sh, residual_out=rs)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(sh), bits_of(ref["out"]))
    assert np.array_equal(bits_of(rs), bits_of(ref["residual_out"]))


def test_unaligned_pointers_take_scalar_path(cuda_lib, orc):
    """Operands at a 2-byte offset (not 16-byte aligned) give the same result."""
    wl = W.make("fused_norm_bs16")
    ref = run_oracle(orc, wl)
    T, H = wl.T, wl.H

    def shifted(bits):
        flat = np.zeros(bits.size + 1, np.uint16)
        flat[1:] = bits.ravel()
        return bf16_dev(flat)[1:].view(bits.shape)

    dev = to_device(wl)
    x = shifted(wl.permuted_out)
    sh, rs, g = shifted(wl.shared), shifted(wl.residual), shifted(wl.gamma)
    outs = [torch.empty(T * H + 1, dtype=torch.bfloat16, device="cuda")[1:].view(T, H)
            for _ in range(3)]
    assert x.data_ptr() % 16 == 2
    res = cuda_lib.moe_finalize(x, dev["idx"], dev["w"], "fp32", sh, routed_scale=1.0,
                                residual=rs, gamma=g, eps=wl.eps, out=outs[0],
                                residual_out=outs[1], norm_out=outs[2])
    torch.cuda.synchronize()
    compare(res, ref, "unaligned: ")
    base = run_gpu(cuda_lib, wl, dev)
    assert np.array_equal(bits_of(res["out"]), bits_of(base["out"]))


def test_empty_batch(cuda_lib):
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    w = torch.zeros((0, 2), dtype=torch.float32, device="cuda")
    sh = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    res = cuda_lib.moe_finalize(x, idx, w, "fp32", sh)
    assert res["out"].shape == (0, 64)


def test_fp32_weights_read_as_bf16_fail_parity(cuda_lib, orc):
    """The failure of "[Deepseek V4] Keep fp32 routing weights in the mxfp4
    trtllm MoE" (revert note): fp32 weight buffers reinterpreted as bf16.
    The parity check must see it."""
    wl = W.make("decode_bs256")
    dev = to_device(wl)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    lib = cuda_lib.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.moe_finalize(p(dev["x"]), wl.P, p(dev["idx"]), p(dev["w"]), 1, 2.5,
                          p(dev["shared"]), None, None, 0.0, p(out), None, None,
                          wl.T, wl.K, wl.H, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    with pytest.raises(AssertionError):
        assert_close(f64_of(out), run_oracle(orc, wl)["out"], "misread weights")


def _wide_cluster_workload():
    """T=2, H=32768 with RMSNorm: rows split over a 16-CTA cluster."""
    return W.synth("wide", T=2, K=4, H=32768, E=64, tile=8, P=64, weight_rule="sigmoid",
                   routed_scale=1.0, with_norm=True, seed=21, require_all=False)


@pytest.mark.parametrize("which", ["fused_norm_bs16", "cluster16"])
def test_graph_capture_replay(cuda_lib, orc, which):
    wl = W.make(which) if which != "cluster16" else _wide_cluster_workload()
    if which == "cluster16":
        assert cuda_lib.plan(wl.T, wl.K, wl.H, True)["cluster"] == 16
    dev = to_device(wl)
    outs = {k: torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
            for k in ("out", "residual_out", "norm_out")}

    def step():
        cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                              routed_scale=1.0, residual=dev["residual"], gamma=dev["gamma"],
                              eps=wl.eps, **outs)

    step()                      # first call outside capture (sets any cluster attribute)
    torch.cuda.synchronize()
    for t in outs.values():
        t.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    compare(outs, run_oracle(orc, wl), "graph replay: ")


def test_error_statuses_on_device(cuda_lib):
    wl = W.make("tiny")
    dev = to_device(wl)
    with pytest.raises(cuda_lib.MoefError) as e:
        cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"], "fp32", dev["shared"],
                              splits=40, threads=48)
    assert e.value.status == 4
    with pytest.raises(ValueError):
        cuda_lib.moe_finalize(dev["x"], dev["idx"], dev["w"].double(), "fp32", dev["shared"])


@pytest.mark.parametrize("wkind", ["bf16", "packed", "fp32"])
def test_every_bf16_weight_through_the_kernel(cuda_lib, orc, wkind):
    """One slot, a row of ones, zero shared, scale 1: out is exactly the
    decoded weight, for every finite bf16 pattern (bit-exact vs the oracle)."""
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = W.bf16_bits_to_f32(b)
    keep = np.isfinite(f) & (np.abs(f) <= 2.0 ** 100)
    bits, vals = b[keep], f[keep]
    T = bits.size
    if wkind == "bf16":
        w = bf16_dev(bits.reshape(T, 1))
        w_host = bits.reshape(T, 1)
    elif wkind == "packed":
        words = (((np.arange(T) % 65536).astype(np.uint32) << 16) | bits).view(np.int32)
        w_host = words.reshape(T, 1)
        w = torch.from_numpy(w_host).cuda()
    else:
        w_host = vals.reshape(T, 1)
        w = torch.from_numpy(w_host).cuda()
    x = W.to_bf16_bits(np.ones((1, 8)))
    idx = np.zeros((T, 1), np.int32)
    zero = np.zeros((T, 8), np.uint16)
    out = cuda_lib.moe_finalize(bf16_dev(x), torch.from_numpy(idx).cuda(), w, wkind,
                                bf16_dev(zero), routed_scale=1.0)["out"]
    torch.cuda.synchronize()
    got = bits_of(out)
    want = np.where(bits == 0x8000, 0, bits).astype(np.uint16)   # -0 * 1 + 0 = +0
    assert np.array_equal(got, np.repeat(want[:, None], 8, axis=1))
    ref = orc.moe_finalize(x, idx, w_host, wkind, 1.0, zero)["out"]
    assert np.array_equal(W.bf16_bits_to_f32(got).astype(np.float64), ref)


@pytest.mark.parametrize("name", ["decode_bs1_packed", "fused_norm_bs16"])
def test_bound_call_matches_direct_call(cuda_lib, name):
    """bind() (packed C-struct replay when built) gives the direct call's bits,
    on the bound stream and on another stream, with and without routing_ready."""
    wl = W.make(name)
    dev = to_device(wl)
    ref = run_gpu(cuda_lib, wl, dev)
    for ready in (False, True):
        f = cuda_lib.bind(dev["x"], dev["idx"], dev["w"], wl.wkind, dev["shared"],
                          routed_scale=wl.routed_scale, residual=dev.get("residual"),
                          gamma=dev.get("gamma"), eps=wl.eps, routing_ready=ready)
        for t in f.outputs.values():
            if t is not None:
                t.zero_()
        f()
        torch.cuda.synchronize()
        for key in ref:
            if ref[key] is not None:
                assert np.array_equal(bits_of(f.outputs[key]), bits_of(ref[key])), key
        s = torch.cuda.Stream()
        for t in f.outputs.values():
            if t is not None:
                t.zero_()
        torch.cuda.synchronize()
        f(stream=s)
        s.synchronize()
        for key in ref:
            if ref[key] is not None:
                assert np.array_equal(bits_of(f.outputs[key]), bits_of(ref[key])), key
