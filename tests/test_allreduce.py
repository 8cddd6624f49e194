"""The all-reduce-fused finalize against the fp64 oracle of R tensor-parallel
ranks ("[Kimi K2.5] Fuse deferred MoE finalize into next-layer AR + residual
+ RMSNorm", Summary; Numerics & speed), through the C ABI.

On one GPU the R ranks are R buffer sets on the same device: the one-shot
call reads all of them in one launch, and the two-phase form runs phase 1
once per rank (stream-ordered) and phase 2 once, so no kernel ever waits on
another.

Tolerance (every bf16 output): |gpu - oracle| <= 2^-7 |oracle| + 2e-3.  The
fp32 partial of phase 1 is checked against a bound derived from its
arithmetic (K + 2 fp32 roundings of terms no larger than their magnitudes).
Bit-exact where the arithmetic leaves no choice: one-shot vs two-phase (same
operations in the same order), one rank vs the plain finalize (out,
residual_out), two identical ranks vs one rank with doubled scale and shared.
"""
import ctypes

import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import assert_close, bf16_dev, bits_of, compare, f64_of, weights_dev

pytestmark = pytest.mark.gpu


def ranks_dev(g):
    return [{"permuted_out": bf16_dev(wl.permuted_out),
             "idx_map": torch.from_numpy(np.ascontiguousarray(wl.idx)).cuda(),
             "weights": weights_dev(wl), "shared_out": bf16_dev(wl.shared)} for wl in g.ranks]


def epilogue_dev(g):
    if not g.with_norm:
        return {}
    return {"residual": bf16_dev(g.residual), "gamma": bf16_dev(g.gamma), "eps": g.eps}


def oracle_ar(orc, g, want_out=True):
    ranks = [{"permuted_out": wl.permuted_out, "idx": wl.idx, "weights": wl.weights,
              "shared": wl.shared} for wl in g.ranks]
    return orc.moe_finalize_ar(ranks, g.wkind, g.routed_scale, g.residual, g.gamma, g.eps,
                               want_out=want_out)


def one_shot(mf, g, rd=None, **kw):
    rd = rd or ranks_dev(g)
    res = mf.moe_finalize_allreduce(rd, g.wkind, routed_scale=g.routed_scale,
                                    **epilogue_dev(g), **kw)
    torch.cuda.synchronize()
    return res


def two_phase(mf, g, rd=None, **kw):
    rd = rd or ranks_dev(g)
    partials = [mf.moe_finalize_partial(r["permuted_out"], r["idx_map"], r["weights"], g.wkind,
                                        r["shared_out"], routed_scale=g.routed_scale)
                for r in rd]
    res = mf.moe_finalize_allreduce_reduce(partials, **epilogue_dev(g), **kw)
    torch.cuda.synchronize()
    return res, partials


def assert_same_bits(a, b, what):
    for key in a:
        if a[key] is None:
            assert b.get(key) is None, key
            continue
        assert np.array_equal(bits_of(a[key]), bits_of(b[key])), f"{what}: {key}"


@pytest.mark.parametrize("T", [1, 16, 256])
@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_decode_shapes_against_oracle(cuda_lib, orc, R, T):
    """The pages' decode shapes (H = 7168, top-8), RMSNorm, every output."""
    g = W.tp_decode(R, T)
    ref = oracle_ar(orc, g)
    rd = ranks_dev(g)
    a = one_shot(cuda_lib, g, rd)
    compare(a, ref, f"one-shot R={R} T={T}: ")
    b, _ = two_phase(cuda_lib, g, rd)
    compare(b, ref, f"two-phase R={R} T={T}: ")
    assert_same_bits(a, b, f"R={R} T={T} one-shot vs two-phase")


CASES = [
    # (R, T, K, H, wkind, norm)
    (3, 5, 4, 1000, "bf16", True),       # R not a power of two
    (2, 7, 8, 7168, "packed", False),    # no residual: out only
    (8, 3, 32, 512, "fp32", True),       # R * K = 256 slots, the most staged
    (5, 4, 1, 64, "fp32", False),        # K = 1
    (3, 6, 3, 100, "fp32", True),        # H % 8 != 0: scalar path
    (2, 9, 6, 4104, "bf16", True),       # ragged: 513 vectors
    (8, 2, 8, 16384, "fp32", True),      # long norm row over a 16-CTA cluster
    (4, 400, 8, 7168, "fp32", True),     # large T: split halved, several passes
    (8, 300, 8, 2048, "packed", True),
    (7, 33, 5, 5120, "fp32", False),
    (3, 5, 2, 64, "fp32", True),         # a row shorter than a warp per rank: padded to whole warps
    (5, 2, 3, 40, "bf16", True),         # scalar path, 5 ranks, 40 values a row
    (6, 16, 8, 7168, "fp32", True),      # 3 groups of rank pairs
    (6, 20, 8, 7168, "bf16", False),     # rank pairs, no residual
    (8, 20, 4, 4104, "fp32", True),      # rank pairs over a ragged row
    (6, 64, 8, 7168, "packed", True),    # one thread sums 6 ranks
    (3, 70, 4, 4104, "fp32", True),      # one thread sums 3 ranks, ragged row
    (2, 100, 8, 2048, "bf16", False),    # one thread sums 2 ranks, no residual
    (7, 16, 8, 7168, "fp32", True),      # odd R: one rank per group from 5 tokens on
    (8, 7, 8, 7168, "fp32", True),       # decode plan: 16 CTAs of 512 threads a row
    (8, 12, 8, 7168, "fp32", True),      # decode plan past 7 tokens (64-register build)
    (8, 48, 8, 7168, "fp32", True),      # two groups of 4 ranks
    (6, 50, 4, 7176, "bf16", True),      # two groups of 3 ranks, ragged row
    # both sides of every switch of the plan at H = 7168 (the plan does not
    # depend on K; K = 2 keeps the large-T operands small)
    (8, 14, 8, 7168, "fp32", True),      # last decode-plan size
    (8, 15, 8, 7168, "packed", True),    # first rank-pair size
    (8, 34, 8, 7168, "fp32", True),      # last rank-pair size
    (8, 35, 8, 7168, "bf16", True),      # first two-group size
    (6, 43, 8, 7168, "fp32", True),      # R = 6: last rank-pair size
    (6, 44, 8, 7168, "fp32", True),      # R = 6: first two-group size
    (8, 63, 8, 7168, "fp32", True),      # last two-group size
    (8, 64, 8, 7168, "fp32", True),      # first all-ranks size
    (8, 160, 2, 7168, "fp32", True),     # 7 CTAs a row, one wave
    (8, 161, 2, 7168, "bf16", True),     # 2 CTAs a row, 2 passes
    (8, 304, 2, 7168, "fp32", True),     # last 2-CTA size
    (8, 305, 2, 7168, "packed", True),   # a row per CTA, 4 passes
]


@pytest.mark.parametrize("R,T,K,H,wkind,norm", CASES)
def test_shapes_against_oracle(cuda_lib, orc, R, T, K, H, wkind, norm):
    tile = 16
    n_blocks = max(K + 1, (T * K + 3) // 4)
    g = W.tp_group("case", R, T=T, K=K, H=H, E=2 * n_blocks + 8, tile=tile, P=n_blocks * tile,
                   wkind=wkind, routed_scale=1.5, with_norm=norm, seed=R * 100 + T)
    ref = oracle_ar(orc, g)
    rd = ranks_dev(g)
    a = one_shot(cuda_lib, g, rd)
    compare(a, ref, f"one-shot R={R} T={T} K={K} H={H}: ")
    b, _ = two_phase(cuda_lib, g, rd)
    assert_same_bits(a, b, f"R={R} T={T} H={H}")
    if norm:
        c = one_shot(cuda_lib, g, rd, write_out=False)
        assert c["out"] is None
        assert_same_bits({k: c[k] for k in ("residual_out", "norm_out")},
                         {k: a[k] for k in ("residual_out", "norm_out")}, "without out")


def test_phase1_partial_within_its_fp32_bound(cuda_lib, orc):
    """The fp32 partial of each rank is that rank's own finalize, within
    (K + 2) fp32 roundings of the magnitudes summed."""
    g = W.tp_decode(4, 16)
    _, partials = two_phase(cuda_lib, g)
    for wl, part in zip(g.ranks, partials):
        ref = orc.moe_finalize(wl.permuted_out, wl.idx, wl.weights, wl.wkind, wl.routed_scale,
                               wl.shared)["out"]
        x = W.bf16_bits_to_f32(wl.permuted_out).astype(np.float64)
        w = np.abs(wl.weights.astype(np.float64) * wl.routed_scale)
        mag = np.einsum("tk,tkh->th", w, np.abs(x[wl.idx])) + \
            np.abs(W.bf16_bits_to_f32(wl.shared))
        bound = (wl.K + 2) * 2.0 ** -24 * mag + 1e-30
        err = np.abs(part.cpu().numpy().astype(np.float64) - ref)
        assert (err <= bound).all(), float((err / bound).max())


def test_partials_at_16_byte_aligned_addresses(cuda_lib):
    """Partials at addresses that are 16-byte but not 32-byte aligned (the
    16-byte path's minimum): phase 1 writes the same bits there, and phase 2
    reading them gives the same outputs."""
    g = W.tp_decode(2, 16)
    rd = ranks_dev(g)
    T, H = g.T, g.H
    ref, aligned = two_phase(cuda_lib, g, rd)
    shifted = []
    for r in rd:
        buf = torch.empty(T * H + 4, dtype=torch.float32, device="cuda")
        part = buf[4:].view(T, H)
        assert part.data_ptr() % 32 == 16
        cuda_lib.moe_finalize_partial(r["permuted_out"], r["idx_map"], r["weights"], g.wkind,
                                      r["shared_out"], routed_scale=g.routed_scale,
                                      partial=part)
        shifted.append(part)
    res = cuda_lib.moe_finalize_allreduce_reduce(shifted, **epilogue_dev(g))
    torch.cuda.synchronize()
    for a, b in zip(aligned, shifted):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert_same_bits(res, ref, "16-byte-aligned partials")


def test_scalar_one_shot_against_vector_two_phase(cuda_lib, orc):
    """A one-shot call whose outputs sit 2 bytes off a 16-byte boundary takes
    the scalar path (its own plan); the two-phase form on aligned buffers
    takes the 16-byte path.  out and residual_out are per-element the same
    fp32 arithmetic and stay bit-identical; norm_out (whose sum of squares
    each plan orders its own way) stays within tolerance of the oracle."""
    g = W.tp_decode(2, 16)
    rd = ranks_dev(g)
    T, H = g.T, g.H
    ref = oracle_ar(orc, g)
    b, _ = two_phase(cuda_lib, g, rd, write_out=True)
    bufs = {k: torch.empty(T * H + 1, dtype=torch.bfloat16, device="cuda")
            for k in ("out", "residual_out", "norm_out")}
    offs = {k: v[1:].view(T, H) for k, v in bufs.items()}
    assert all(v.data_ptr() % 16 == 2 for v in offs.values())
    a = one_shot(cuda_lib, g, rd, **offs)
    for key in ("out", "residual_out"):
        assert np.array_equal(bits_of(a[key]), bits_of(b[key])), key
    compare(a, ref, "scalar one-shot: ")
    compare(b, ref, "vector two-phase: ")


def test_one_rank_is_the_plain_finalize(cuda_lib, orc):
    """R = 1: out and residual_out equal moe_finalize's bit for bit (same fp32
    operations in the same order); norm_out within tolerance of the oracle."""
    g = W.tp_decode(1, 16)
    wl = g.ranks[0]
    rd = ranks_dev(g)[0]
    plain = cuda_lib.moe_finalize(rd["permuted_out"], rd["idx_map"], rd["weights"], wl.wkind,
                                  rd["shared_out"], routed_scale=wl.routed_scale,
                                  **epilogue_dev(g))
    a = one_shot(cuda_lib, g)
    for key in ("out", "residual_out"):
        assert np.array_equal(bits_of(a[key]), bits_of(plain[key])), key
    compare(a, oracle_ar(orc, g), "R=1: ")


def test_two_identical_ranks_are_one_rank_doubled(cuda_lib):
    """Two ranks with the same operands sum to exactly twice one rank, which
    is the plain finalize with the routed scale and shared output doubled
    (every scaling by 2 is exact)."""
    g = W.tp_decode(1, 16)
    wl = g.ranks[0]
    rd = ranks_dev(g)
    a = one_shot(cuda_lib, W.TPGroup("twice", [wl, wl], g.residual, g.gamma, g.eps),
                 rd + rd)
    shared2 = (rd[0]["shared_out"].float() * 2).to(torch.bfloat16)
    plain = cuda_lib.moe_finalize(rd[0]["permuted_out"], rd[0]["idx_map"], rd[0]["weights"],
                                  wl.wkind, shared2, routed_scale=2 * wl.routed_scale,
                                  **epilogue_dev(g))
    torch.cuda.synchronize()
    for key in ("out", "residual_out"):
        assert np.array_equal(bits_of(a[key]), bits_of(plain[key])), key


def test_rank_order_changes_only_rounding(cuda_lib, orc):
    g = W.tp_decode(4, 1)
    rd = ranks_dev(g)
    a = one_shot(cuda_lib, g, rd)
    perm = [2, 0, 3, 1]
    gp = W.TPGroup("perm", [g.ranks[i] for i in perm], g.residual, g.gamma, g.eps)
    b = one_shot(cuda_lib, gp, [rd[i] for i in perm])
    ref = oracle_ar(orc, g)
    compare(a, ref, "order 0123: ")
    compare(b, ref, "order 2031: ")


def test_in_place_residual(cuda_lib, orc):
    """residual_out may be the residual buffer itself."""
    g = W.tp_decode(2, 16)
    ref = oracle_ar(orc, g)
    ep = epilogue_dev(g)
    res = cuda_lib.moe_finalize_allreduce(ranks_dev(g), g.wkind, routed_scale=g.routed_scale,
                                          residual_out=ep["residual"], **ep)
    torch.cuda.synchronize()
    assert res["residual_out"].data_ptr() == ep["residual"].data_ptr()
    compare(res, ref, "in place: ")


def test_padding_rows_never_read(cuda_lib, orc):
    """NaN in every padding row of every rank leaves the outputs finite."""
    g = W.tp_decode(4, 16)
    for wl in g.ranks:
        wl.permuted_out[~wl.valid_rows] = 0x7FC0
    res = one_shot(cuda_lib, g)
    for key, t in res.items():
        assert np.isfinite(f64_of(t)).all(), key
    compare(res, oracle_ar(orc, g), "NaN padding: ")


def test_zero_tokens_and_argument_errors(cuda_lib):
    g = W.tp_decode(2, 1)
    rd = ranks_dev(g)
    lib = cuda_lib.lib()
    arr = (cuda_lib._abi.RankInputs * 2)(*[cuda_lib._abi.RankInputs(
        r["permuted_out"].data_ptr(), 256, r["idx_map"].data_ptr(), r["weights"].data_ptr(),
        r["shared_out"].data_ptr()) for r in rd])
    out = torch.empty((1, 7168), dtype=torch.bfloat16, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    call = lambda R, T, **kw: lib.moe_finalize_allreduce(
        kw.get("arr", arr), R, 0, 2.5, None, None, 1e-6, kw.get("out", out.data_ptr()), None,
        None, T, 8, 7168, s)
    assert call(2, 0) == 0                   # T = 0: nothing enqueued
    assert call(0, 1) == 2 and call(9, 1) == 2
    assert call(2, 1, arr=None) == 1
    assert call(2, 1, out=None) == 1
    assert call(2, 1, out=out.data_ptr() + 1) == 3
    assert call(2, 1) == 0
    torch.cuda.synchronize()


def test_graph_capture_replay(cuda_lib, orc):
    """Both forms captured in one CUDA graph (the one-shot with a 14-CTA
    cluster at R = 8; the first eager call sets the cluster attribute) and
    replayed on new contents of the same buffers."""
    g = W.tp_decode(8, 1)
    rd = ranks_dev(g)
    ep = epilogue_dev(g)
    outs = {k: torch.empty((1, 7168), dtype=torch.bfloat16, device="cuda")
            for k in ("out", "residual_out", "norm_out")}
    outs2 = {k: torch.empty_like(v) for k, v in outs.items()}
    partials = [torch.empty((1, 7168), dtype=torch.float32, device="cuda") for _ in rd]

    def step():
        cuda_lib.moe_finalize_allreduce(rd, g.wkind, routed_scale=g.routed_scale, **ep, **outs)
        for r, p in zip(rd, partials):
            cuda_lib.moe_finalize_partial(r["permuted_out"], r["idx_map"], r["weights"],
                                          g.wkind, r["shared_out"], routed_scale=g.routed_scale,
                                          partial=p)
        cuda_lib.moe_finalize_allreduce_reduce(partials, **ep, **outs2)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    g2 = W.tp_decode(8, 1, seed=77)
    for r, wl in zip(rd, g2.ranks):
        r["permuted_out"].copy_(bf16_dev(wl.permuted_out))
        r["idx_map"].copy_(torch.from_numpy(wl.idx))
        r["weights"].copy_(weights_dev(wl))
        r["shared_out"].copy_(bf16_dev(wl.shared))
    ep["residual"].copy_(bf16_dev(g2.residual))
    ep["gamma"].copy_(bf16_dev(g2.gamma))
    graph.replay()
    torch.cuda.synchronize()
    ref = oracle_ar(orc, g2)
    compare(outs, ref, "graph one-shot: ")
    compare(outs2, ref, "graph two-phase: ")
    assert_same_bits(outs, outs2, "graph one-shot vs two-phase")


@pytest.mark.slow
@pytest.mark.parametrize("R,T,H,E,tile,P,plan", [
    # each thread sums the 8 ranks in sequence: one CTA per row, 2 passes
    (8, 1024, 4096, 512, 64, 16384, dict(lanes=1, splits=1, passes=2, cluster=1)),
    # 2 groups of four ranks, 2 passes per thread, 8-CTA clusters
    (8, 40, 16384, 64, 32, 1024, dict(lanes=2, splits=8, passes=2, cluster=8)),
    # 2 groups of two ranks, 4 passes per thread, 8-CTA clusters
    (4, 48, 32768, 64, 32, 1024, dict(lanes=2, splits=8, passes=4, cluster=8)),
    # one group per rank (odd R), 8 passes per thread, 8-CTA clusters
    (5, 48, 16384, 64, 32, 1024, dict(lanes=5, splits=8, passes=8, cluster=8)),
])
def test_large_sampled_rows(cuda_lib, orc, R, T, H, E, tile, P, plan):
    """Sizes with long rows or many tokens: sampled token rows against the
    oracle, every row against the two-phase form."""
    g = W.tp_group("large", R, T=T, K=8, H=H, E=E, tile=tile, P=P, routed_scale=2.5, seed=9)
    p = cuda_lib.allreduce_plan(R, T, H, True)
    assert {k: p[k] for k in plan} == plan
    rd = ranks_dev(g)
    a = one_shot(cuda_lib, g, rd)
    b, _ = two_phase(cuda_lib, g, rd)
    assert_same_bits(a, b, f"T={T} H={H} R={R}")
    rows = np.sort(np.random.default_rng(0).choice(g.T, min(48, g.T), replace=False))
    sub = W.TPGroup("rows", [W.Workload(**{**wl.__dict__, "T": len(rows), "idx": wl.idx[rows],
                                           "weights": wl.weights[rows],
                                           "shared": wl.shared[rows]}) for wl in g.ranks],
                    g.residual[rows], g.gamma, g.eps)
    ref = oracle_ar(orc, sub)
    for key in ref:
        assert_close(f64_of(a[key])[rows], ref[key], f"T={T} H={H} sampled {key}")


def test_tp_orchestration_one_rank(cuda_lib, orc):
    """The tensor-parallel orchestration with its CUDA transport (IPC
    handles, interprocess events) and library backend, as one rank of a
    one-rank gloo group: two steps of different token counts, through both
    partial buffers, against the oracle."""
    import socket
    import torch.distributed as dist
    from moe_deferred_finalize_gb300 import tp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                           world_size=1)
    try:
        group = tp.TPFinalize(dist.group.WORLD, 16, 7168)
        for T in (16, 5):
            g = W.tp_decode(1, 16, seed=T)
            if T != 16:
                wl = g.ranks[0]
                g = W.TPGroup("sub", [W.Workload(**{**wl.__dict__, "T": T, "idx": wl.idx[:T],
                                                    "weights": wl.weights[:T],
                                                    "shared": wl.shared[:T]})],
                              g.residual[:T], g.gamma, g.eps)
            rd = ranks_dev(g)[0]
            ep = epilogue_dev(g)
            outs = {k: torch.empty((T, 7168), dtype=torch.bfloat16, device="cuda")
                    for k in ("out", "residual_out", "norm_out")}
            res = group.step(rd, g.wkind, g.routed_scale, T, residual=ep["residual"],
                             gamma=ep["gamma"], eps=ep["eps"], outs=outs)
            torch.cuda.synchronize()
            compare(res, oracle_ar(orc, g), f"orchestrated T={T}: ")
        assert group.step_index == 2
        group.close()
    finally:
        dist.destroy_process_group()


def _tp_worker(rank, port, steps, q):
    """One rank of a two-process group on GPU 0: real CUDA IPC buffers and
    interprocess events, gloo for set-up and the per-step host barrier."""
    import os
    import sys
    import traceback
    try:
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        sys.path.insert(0, os.path.join(root, "tests"))
        import torch
        import torch.distributed as dist
        from moe_deferred_finalize_gb300 import tp
        from moe_deferred_finalize_gb300 import workloads as W2
        from gpu_util import bf16_dev, bits_of, weights_dev
        torch.cuda.set_device(0)
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                world_size=2)
        try:
            group = tp.TPFinalize(dist.group.WORLD, 16, 7168)
            got = []
            for T, seed in steps:
                g = W2.tp_decode(2, T, seed=seed)
                wl = g.ranks[rank]
                x = {"permuted_out": bf16_dev(wl.permuted_out),
                     "idx_map": torch.from_numpy(wl.idx).cuda(), "weights": weights_dev(wl),
                     "shared_out": bf16_dev(wl.shared)}
                outs = {k: torch.empty((T, 7168), dtype=torch.bfloat16, device="cuda")
                        for k in ("out", "residual_out", "norm_out")}
                group.step(x, g.wkind, g.routed_scale, T, residual=bf16_dev(g.residual),
                           gamma=bf16_dev(g.gamma), eps=g.eps, outs=outs)
                torch.cuda.synchronize()
                got.append({k: bits_of(v) for k, v in outs.items()})
            group.close()
            # the one-shot form over shared input sets (room for the largest buffer)
            one = tp.TPFinalize(dist.group.WORLD, 16, 7168, one_shot=(2048, 8, "fp32"))
            shots = []
            for T, seed in steps:
                g = W2.tp_decode(2, T, seed=seed)
                wl = g.ranks[rank]
                x = one.inputs()
                x["permuted_out"][:wl.P].copy_(bf16_dev(wl.permuted_out))
                x["idx_map"][:T].copy_(torch.from_numpy(wl.idx))
                x["weights"][:T].copy_(weights_dev(wl))
                x["shared_out"][:T].copy_(bf16_dev(wl.shared))
                outs = {k: torch.empty((T, 7168), dtype=torch.bfloat16, device="cuda")
                        for k in ("out", "residual_out", "norm_out")}
                one.step_one_shot(T, routed_scale=g.routed_scale, residual=bf16_dev(g.residual),
                                  gamma=bf16_dev(g.gamma), eps=g.eps, outs=outs)
                torch.cuda.synchronize()
                shots.append({k: bits_of(v) for k, v in outs.items()})
            one.close()
            q.put((rank, "ok", (got, shots)))
        finally:
            dist.destroy_process_group()
    except Exception:
        q.put((rank, "error", traceback.format_exc()))


def test_tp_orchestration_two_processes_one_gpu(cuda_lib, orc):
    """The orchestration with two processes sharing one GPU: each opens the
    other's buffers and events through CUDA IPC, and its stream waits on the
    other's events (no kernel waits on another).  Three two-phase steps of
    different token counts, then the same three as one-shot steps over the
    shared input sets: every output of both ranks in both forms equal bit for
    bit, and matching the oracle of the whole group."""
    import socket
    import torch.multiprocessing as tmp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    steps = [(16, 41), (1, 42), (16, 43)]
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_tp_worker, args=(r, port, steps, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(2):
        rank, status, payload = q.get(timeout=300)
        got[rank] = (status, payload)
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for rank in (0, 1):
        assert got[rank][0] == "ok", got[rank][1]
    for i, (T, seed) in enumerate(steps):
        a, b = got[0][1][0][i], got[1][1][0][i]
        for key in a:
            assert np.array_equal(a[key], b[key]), (T, key)
            # the one-shot form on both ranks: bit-identical to the two-phase
            for rank in (0, 1):
                assert np.array_equal(got[rank][1][1][i][key], a[key]), (T, key, rank)
        ref = oracle_ar(orc, W.tp_decode(2, T, seed=seed))
        for key in ref:
            f = (a[key].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            assert_close(f, ref[key], f"two processes, step {i} (T={T}) {key}")
