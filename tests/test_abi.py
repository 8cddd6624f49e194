"""The C-ABI library without a GPU: it loads, exports every symbol the
header declares, rejects bad arguments before touching CUDA, and plans
launches as documented.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

from moe_deferred_finalize_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def mf():
    build.build_library()
    import moe_deferred_finalize_gb300 as m
    return m


def declared_functions():
    names = []
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^(?:const\s+)?\w+\s+\**\s*(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"moe_finalize", "moe_finalize_ex", "moe_finalize_plan", "unpack_topk_ids",
            "moe_finalize_check_indices", "moef_status_string"} <= names


def test_library_exports_every_declared_symbol(mf):
    lib = ctypes.CDLL(build.LIB)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_matches_header_and_binding(mf):
    text = open(os.path.join(HEADER_DIR, "moe_finalize.h")).read()
    version = int(re.search(r"#define MOEF_ABI_VERSION (\d+)", text).group(1))
    from moe_deferred_finalize_gb300 import _abi
    assert mf.lib().moef_abi_version() == version == _abi.ABI_VERSION


def test_library_of_another_interface_version_is_refused(mf, monkeypatch):
    from moe_deferred_finalize_gb300 import _abi
    monkeypatch.setattr(_abi, "_LIB", None)
    monkeypatch.setattr(_abi, "ABI_VERSION", _abi.ABI_VERSION + 1)
    with pytest.raises(RuntimeError, match="interface version"):
        _abi._lib()


def test_unknown_flags_rejected(mf):
    f = mf.lib().moe_finalize_ex
    assert f(A, 16, A, A, 0, 1.0, A, None, None, 1e-6, A, None, None, 0, 2, 8, 0, 0, 4, None) == 4
    for flags in (1, 2, 3):     # MOEF_FLAG_ROUTING_READY, MOEF_FLAG_NO_PDL
        assert f(A, 16, A, A, 0, 1.0, A, None, None, 1e-6, A, None, None, 0, 2, 8, 0, 0, flags,
                 None) == 0


def test_status_strings(mf):
    s = mf.lib().moef_status_string
    for code in range(7):
        assert s(code) and s(code) != b"unknown status"
    assert s(99) == b"unknown status"


# Argument errors are returned before any CUDA call, so they are checked here
# with made-up (never dereferenced) addresses.
A = 0x10000   # 64 KiB aligned fake addresses
NULL = None


def call(mf, **kw):
    args = dict(x=A, P=16, idx=A, w=A, wkind=0, scale=1.0, shared=A, residual=NULL,
                gamma=NULL, eps=1e-6, out=A, residual_out=NULL, norm_out=NULL, T=2, K=2, H=8,
                stream=NULL)
    args.update(kw)
    return mf.lib().moe_finalize(args["x"], args["P"], args["idx"], args["w"], args["wkind"],
                                 args["scale"], args["shared"], args["residual"], args["gamma"],
                                 args["eps"], args["out"], args["residual_out"],
                                 args["norm_out"], args["T"], args["K"], args["H"],
                                 args["stream"])


def test_argument_errors(mf):
    OK, NUL, SHAPE, ALIGN, ARG = 0, 1, 2, 3, 4
    assert call(mf, T=0) == OK                      # empty batch: nothing enqueued
    assert call(mf, T=0, x=NULL) == OK
    assert call(mf, T=-1) == SHAPE
    assert call(mf, K=0) == SHAPE
    assert call(mf, K=33) == SHAPE
    assert call(mf, H=0) == SHAPE
    assert call(mf, P=0) == SHAPE
    assert call(mf, wkind=3) == ARG
    assert call(mf, x=NULL) == NUL
    assert call(mf, idx=NULL) == NUL
    assert call(mf, w=NULL) == NUL
    assert call(mf, shared=NULL) == NUL
    assert call(mf, out=NULL) == NUL                # no residual: out is required
    assert call(mf, residual=A) == ARG              # residual without gamma
    assert call(mf, gamma=A) == ARG
    assert call(mf, residual=A, gamma=A) == NUL     # residual_out / norm_out missing
    assert call(mf, residual=A, gamma=A, residual_out=A) == NUL
    assert call(mf, residual_out=A) == ARG          # output without its input
    assert call(mf, residual=A, gamma=A, residual_out=A, norm_out=A, eps=-1.0) == ARG
    assert call(mf, residual=A, gamma=A, residual_out=A, norm_out=A, eps=float("nan")) == ARG
    assert call(mf, residual=A, gamma=A, residual_out=A, norm_out=A, eps=float("inf")) == ARG
    assert call(mf, x=A + 1) == ALIGN
    assert call(mf, out=A + 1) == ALIGN
    assert call(mf, idx=A + 2) == ALIGN
    assert call(mf, w=A + 2) == ALIGN               # fp32 weights need 4 bytes
    u = mf.lib().unpack_topk_ids
    assert u(A, 0, A, A, NULL) == OK
    assert u(A, -1, A, A, NULL) == SHAPE
    assert u(NULL, 4, A, A, NULL) == NUL
    assert u(A, 4, NULL, NULL, NULL) == NUL
    assert u(A + 2, 4, A, NULL, NULL) == ALIGN
    g = mf.lib().moe_topk_route
    assert g(A, 0, 256, 8, 0, A, NULL, NULL, NULL) == OK
    assert g(A, 4, 256, 0, 0, A, NULL, NULL, NULL) == SHAPE
    assert g(A, 4, 4, 8, 0, A, NULL, NULL, NULL) == SHAPE        # K > E
    assert g(A, 4, 2048, 8, 0, A, NULL, NULL, NULL) == SHAPE     # E > 1024
    assert g(A, 4, 256, 33, 0, A, NULL, NULL, NULL) == SHAPE
    assert g(A, 4, 256, 8, 2, A, NULL, NULL, NULL) == ARG
    assert g(NULL, 4, 256, 8, 0, A, NULL, NULL, NULL) == NUL
    assert g(A, 4, 256, 8, 0, NULL, NULL, NULL, NULL) == NUL
    assert g(A + 2, 4, 256, 8, 0, A, NULL, NULL, NULL) == ALIGN
    pk = mf.lib().pack_topk_ids
    assert pk(A, A, 0, A, NULL) == OK
    assert pk(A, A, -1, A, NULL) == SHAPE
    assert pk(NULL, A, 4, A, NULL) == NUL
    assert pk(A, A, 4, A + 2, NULL) == ALIGN
    c = mf.lib().moe_finalize_check_indices
    assert c(A, 2, 2, 16, NULL, NULL) == NUL
    assert c(A, -1, 2, 16, A, NULL) == SHAPE
    assert c(A, 2, 0, 16, A, NULL) == SHAPE
    assert c(NULL, 2, 2, 16, A, NULL) == NUL
    assert c(A, 2, 2, 16, A + 2, NULL) == ALIGN


def test_plan_regimes(mf):
    # decode sizes: one 16-byte vector per thread, 128-vector slices
    p = mf.plan(1, 8, 7168, False)
    assert (p["vec"], p["splits"], p["slice"], p["threads"], p["vpt"], p["cluster"]) == \
        (8, 7, 128, 128, 1, 1)
    p = mf.plan(16, 8, 7168, True)          # RMSNorm: 4-CTA clusters, one vector per thread
    assert (p["splits"], p["threads"], p["vpt"], p["cluster"], p["grid"]) == (4, 224, 1, 4, 64)
    # one wave: up to 4.75 CTAs of 224 threads per SM (T <= 180 at 152 SMs),
    # then the same slices on 128-thread CTAs, two vectors a thread, up to
    # 7.5 per SM (T <= 285), then the split halved while above 4.25 per SM
    # (T <= 323), then one CTA per row
    for T, want in ((128, (4, 224, 1, 4)), (180, (4, 224, 1, 4)), (181, (4, 128, 2, 4)),
                    (256, (4, 128, 2, 4)), (285, (4, 128, 2, 4)), (286, (2, 256, 2, 2)),
                    (323, (2, 256, 2, 2)), (324, (1, 256, 4, 1)), (384, (1, 256, 4, 1)),
                    (512, (1, 256, 4, 1))):
        p = mf.plan(T, 8, 7168, True)
        assert (p["splits"], p["threads"], p["vpt"], p["cluster"]) == want, (T, p)
    # 256-thread slices (H = 4096) keep their size up to 4.25 CTAs per SM;
    # past that a whole row goes to one CTA, two vectors a thread
    assert mf.plan(323, 8, 4096, True)["threads"] == 256
    p = mf.plan(324, 8, 4096, True)
    assert (p["splits"], p["threads"], p["vpt"]) == (1, 256, 2)
    p = mf.plan(380, 8, 5120, True)     # 3-CTA clusters of 128 threads up to 7.5 per SM
    assert (p["splits"], p["threads"], p["vpt"]) == (3, 128, 2)
    assert mf.plan(381, 8, 5120, True)["splits"] == 1
    p = mf.plan(128, 8, 7168, False)
    assert (p["splits"], p["threads"], p["vpt"], p["grid"]) == (7, 128, 1, 896)
    p = mf.plan(256, 8, 7168, False)        # 1792 CTAs: 64-thread CTAs fit one wave
    assert (p["splits"], p["threads"], p["vpt"], p["grid"]) == (7, 64, 2, 1792)
    p = mf.plan(4096, 8, 7168, False)       # large T without RMSNorm: still 128-vector slices
    assert (p["splits"], p["threads"], p["vpt"]) == (7, 128, 1)
    # bandwidth sizes: one CTA of 128 threads per token row
    p = mf.plan(16384, 8, 7168, True)
    assert (p["splits"], p["threads"], p["vpt"], p["cluster"], p["grid"]) == (1, 128, 8, 1, 16384)
    # scalar path when H is not a multiple of 8 or pointers are unaligned
    assert mf.plan(4, 2, 100, False)["vec"] == 1
    assert mf.plan(4, 2, 64, False, vec_ok=False)["vec"] == 1
    # long RMSNorm rows use a cluster, up to 16 CTAs
    p = mf.plan(4096, 8, 32768, True)
    assert p["cluster"] == 2 and p["threads"] == 256 and p["vpt"] == 8
    p = mf.plan(8, 8, 16384, True)
    assert p["cluster"] == 8 and p["threads"] == 256 and p["vpt"] == 1
    p = mf.plan(2, 8, 32768, True)
    assert p["cluster"] == 16 and p["vpt"] == 1


def test_plan_invariants(mf):
    for T in (1, 3, 16, 256, 700, 5000, 16384):
        for H in (8, 64, 100, 1000, 7168, 7176, 16384, 40000):
            for norm in (False, True):
                for vec_ok in (True, False):
                    try:
                        p = mf.plan(T, 8, H, norm, vec_ok)
                    except mf.MoefError as e:
                        assert e.status == 2 and norm     # only over-long norm rows fail
                        continue
                    nvec = H // p["vec"]
                    assert p["vec"] in (1, 8) and (p["vec"] == 1 or H % 8 == 0)
                    assert p["splits"] * p["slice"] >= nvec > (p["splits"] - 1) * p["slice"]
                    assert p["threads"] % 32 == 0 and 32 <= p["threads"] <= 256
                    assert p["vpt"] in (1, 2, 4, 8)
                    assert p["grid"] == T * p["splits"]
                    if norm:
                        assert p["threads"] * p["vpt"] >= p["slice"]   # one pass per slice
                        assert p["cluster"] == p["splits"] <= 16
                    else:
                        assert p["cluster"] == 1


def test_plans_every_token_count(mf):
    """The plain finalize's plan at every token count from 1 to 640 and at
    the powers of two up to 2^16 (the decode split, the cluster and
    threads-per-CTA switches), for top-1/2/6/8/9 routing at common hidden
    sizes: every plan is one the launcher accepts."""
    Ts = list(range(1, 641)) + [2 ** i for i in range(10, 17)]
    for H in (2048, 4096, 5120, 7168, 8192):
        for K in (1, 2, 6, 8, 9):
            for norm in (False, True):
                for T in Ts:
                    p = mf.plan(T, K, H, norm)
                    where = (T, K, H, norm, p)
                    nvec = H // p["vec"]
                    assert p["vec"] == 8, where
                    assert p["splits"] * p["slice"] >= nvec > (p["splits"] - 1) * p["slice"], where
                    assert p["threads"] % 32 == 0 and 32 <= p["threads"] <= 256, where
                    assert p["vpt"] in (1, 2, 4, 8) and p["grid"] == T * p["splits"], where
                    if norm:
                        assert p["threads"] * p["vpt"] >= p["slice"], where
                        assert p["cluster"] == p["splits"] <= 16, where
                    else:
                        assert p["cluster"] == 1, where


def test_allreduce_argument_errors(mf):
    """The all-reduce-fused entry points check every rank's operands and the
    epilogue before any CUDA call."""
    from moe_deferred_finalize_gb300 import _abi
    OK, NUL, SHAPE, ALIGN, ARG = 0, 1, 2, 3, 4
    lib = mf.lib()

    def ranks(n, **bad):
        arr = (_abi.RankInputs * max(n, 1))()
        for r in range(n):
            f = dict(permuted_out=A, P=16, idx_map=A, weights=A, shared_out=A)
            if r == n - 1:
                f.update(bad)
            arr[r] = _abi.RankInputs(f["permuted_out"], f["P"], f["idx_map"], f["weights"],
                                     f["shared_out"])
        return arr

    def ar(R=2, T=2, K=2, H=8, wkind=0, arr=None, residual=NULL, gamma=NULL, eps=1e-6,
           out=A, residual_out=NULL, norm_out=NULL, **bad):
        arr = ranks(R, **bad) if arr is None else arr
        return lib.moe_finalize_allreduce(arr, R, wkind, 1.0, residual, gamma, eps, out,
                                          residual_out, norm_out, T, K, H, NULL)

    assert ar(T=0) == OK
    for R in (0, -1, 9):
        assert ar(R=R, arr=ranks(1)) == SHAPE
    assert ar(K=0) == SHAPE and ar(K=33) == SHAPE and ar(H=0) == SHAPE and ar(T=-1) == SHAPE
    assert ar(wkind=3) == ARG
    assert lib.moe_finalize_allreduce(None, 2, 0, 1.0, NULL, NULL, 1e-6, A, NULL, NULL,
                                      2, 2, 8, NULL) == NUL
    assert ar(P=0) == SHAPE                      # the last rank's buffer is empty
    for field in ("permuted_out", "idx_map", "weights", "shared_out"):
        assert ar(**{field: NULL}) == NUL, field
    assert ar(permuted_out=A + 1) == ALIGN
    assert ar(shared_out=A + 1) == ALIGN
    assert ar(idx_map=A + 2) == ALIGN
    assert ar(weights=A + 2) == ALIGN            # fp32 weights need 4 bytes
    assert ar(wkind=1, weights=A + 2) != ALIGN   # bf16 weights need 2
    assert ar(out=NULL) == NUL
    assert ar(residual=A) == ARG and ar(gamma=A) == ARG
    assert ar(residual=A, gamma=A) == NUL
    assert ar(residual_out=A) == ARG
    assert ar(residual=A, gamma=A, residual_out=A, norm_out=A, eps=-1.0) == ARG
    assert ar(out=A + 1) == ALIGN

    part = lib.moe_finalize_partial
    assert part(A, 16, A, A, 0, 1.0, A, A, 0, 2, 8, NULL) == OK
    assert part(A, 16, A, A, 0, 1.0, A, NULL, 2, 2, 8, NULL) == NUL
    assert part(A, 16, A, A, 0, 1.0, A, A + 2, 2, 2, 8, NULL) == ALIGN
    assert part(A, 0, A, A, 0, 1.0, A, A, 2, 2, 8, NULL) == SHAPE
    assert part(A, 16, A, A, 5, 1.0, A, A, 2, 2, 8, NULL) == ARG
    assert part(NULL, 16, A, A, 0, 1.0, A, A, 2, 2, 8, NULL) == NUL

    red = lib.moe_finalize_allreduce_reduce
    parts = (ctypes.c_void_p * 3)(A, A, A)
    assert red(parts, 3, NULL, NULL, 1e-6, A, NULL, NULL, 0, 8, NULL) == OK
    assert red(parts, 0, NULL, NULL, 1e-6, A, NULL, NULL, 2, 8, NULL) == SHAPE
    assert red(parts, 9, NULL, NULL, 1e-6, A, NULL, NULL, 2, 8, NULL) == SHAPE
    assert red(None, 3, NULL, NULL, 1e-6, A, NULL, NULL, 2, 8, NULL) == NUL
    assert red((ctypes.c_void_p * 3)(A, NULL, A), 3, NULL, NULL, 1e-6, A, NULL, NULL,
               2, 8, NULL) == NUL
    assert red((ctypes.c_void_p * 3)(A, A + 2, A), 3, NULL, NULL, 1e-6, A, NULL, NULL,
               2, 8, NULL) == ALIGN
    assert red(parts, 3, A, NULL, 1e-6, A, NULL, NULL, 2, 8, NULL) == ARG
    assert red(parts, 3, NULL, NULL, 1e-6, NULL, NULL, NULL, 2, 8, NULL) == NUL


def test_allreduce_plans(mf):
    """Plan invariants over ranks, sizes and both epilogues: R groups of
    threads per CTA at decode sizes (R / 2 groups of two ranks from 8 tokens
    on when R > 4; one thread summing all ranks from 64 tokens on), every
    vector of a row covered, and with RMSNorm one cluster of at most 16 CTAs
    and at most 8 passes per thread."""
    for R in range(1, 9):
        for H in (8, 64, 100, 1000, 2048, 4104, 7168, 16384, 65536):
            for T in (1, 16, 48, 64, 256, 4096):
                for norm in (False, True):
                    for vec_ok in (True, False):
                        try:
                            p = mf.allreduce_plan(R, T, H, norm, vec_ok)
                        except mf.MoefError as e:
                            assert e.status == 2 and norm
                            continue
                        nvec = H // p["vec"]
                        # rank groups at decode sizes; each thread summing the
                        # ranks in sequence once the tokens fill the GPU
                        seq = R > 1 and p["vec"] == 8 and T >= 64
                        groups = {R}                      # the layouts this size may take
                        if p["vec"] == 8 and T > 7 and R % 2 == 0:
                            if R > 4:
                                groups.add(R // 2)
                            if R >= 4 and norm:
                                groups.add(2)
                        if seq and p["lanes"] != 1:
                            assert norm and -(-nvec // 16) > 8 * 512   # row too long for one
                            assert p["lanes"] in groups
                        else:
                            assert p["lanes"] in ({1} if seq else groups)
                        assert p["threads"] == p["lanes"] * p["nvc"] <= 512
                        assert p["threads"] % 32 == 0          # whole warps: full-mask shuffles
                        assert p["splits"] * p["slice"] >= nvec > (p["splits"] - 1) * p["slice"]
                        assert p["passes"] * p["nvc"] >= p["slice"]
                        assert p["grid"] == T * p["splits"]
                        if norm:
                            assert p["passes"] in (1, 2, 4, 8)
                            assert p["cluster"] == p["splits"] <= 16
                        else:
                            assert p["cluster"] == 1
                        assert p["smem_bytes"] <= 48 * 1024
    # the decode shapes: every rank's loads of a vector in flight in one pass
    p = mf.allreduce_plan(8, 1, 7168, True)
    assert (p["nvc"], p["splits"], p["passes"], p["cluster"]) == (64, 16, 1, 16)
    p = mf.allreduce_plan(2, 1, 7168, True)           # a split row widened to 16 CTAs
    assert (p["nvc"], p["splits"], p["cluster"]) == (64, 16, 16)
    p = mf.allreduce_plan(2, 1, 2048, True)           # a row that fits one CTA stays there
    assert (p["splits"], p["cluster"]) == (1, 1)
    # rank groups switch to two halves where the rows' 14-CTA clusters would
    # not all be resident at once (T > ~35 for 256-thread CTAs, ~43 for 192)
    for R, T, lanes in ((8, 34, 4), (8, 35, 2), (4, 34, 4), (4, 35, 2), (6, 43, 3), (6, 44, 2)):
        assert mf.allreduce_plan(R, T, 7168, True)["lanes"] == lanes, (R, T)
    # the decode plan (16 CTAs a row, one rank per thread group) up to T = 7,
    # or up to 14 with more than 4 ranks (whose alternative is rank pairs)
    for R, T, lanes in ((4, 7, 4), (4, 8, 4), (8, 14, 8), (8, 15, 4), (6, 14, 6), (6, 15, 3)):
        p = mf.allreduce_plan(R, T, 7168, True)
        decode = T <= (14 if R > 4 else 7)
        assert p["lanes"] == lanes and p["splits"] == (16 if decode else 14), (R, T, p)
    # one thread summing all ranks: 7 CTAs a row while the rows' 7-CTA
    # clusters are resident at once (160 rows), then 2 x 2 passes (up to 304
    # rows of 2-CTA clusters), then 1 x 4 passes
    for T, splits, passes in ((64, 7, 1), (160, 7, 1), (161, 2, 2), (304, 2, 2), (305, 1, 4)):
        p = mf.allreduce_plan(8, T, 7168, True)
        assert (p["lanes"], p["splits"], p["passes"]) == (1, splits, passes), (T, p)
    # many tokens: one thread per vector summing the 8 ranks, rows in 2
    # slices of 2 passes over 224 vectors
    p = mf.allreduce_plan(8, 256, 7168, True)
    assert (p["lanes"], p["nvc"], p["splits"], p["passes"], p["cluster"], p["grid"]) == \
        (1, 224, 2, 2, 2, 512)
    with pytest.raises(mf.MoefError):
        mf.allreduce_plan(8, 1, 8 * 8 * 16 * 64 + 8, True)    # longer than 16 CTAs x 8 passes
    with pytest.raises(mf.MoefError):
        mf.allreduce_plan(9, 1, 7168, True)


def test_allreduce_plans_every_token_count(mf):
    """Every token count from 1 to 640 (all the plan's switch points: the
    decode limits, the two-group and all-ranks layouts, the cluster and
    pass changes) at the hidden sizes of common models: each plan is one the
    launcher accepts and the kernels were built for (lanes dividing R, whole
    warps with RMSNorm, 1/2/4/8 passes covering the slice, at most 16 CTAs
    a cluster, groups of several ranks only with 16-byte vectors), and the
    size a plan picks never needs more shared memory than a CTA gets
    without opting in."""
    for R in range(1, 9):
        for H in (2048, 4096, 5120, 6144, 7168, 8192):
            for norm in (False, True):
                for T in range(1, 641):
                    p = mf.allreduce_plan(R, T, H, norm)
                    lanes, nvc, vec = p["lanes"], p["nvc"], p["vec"]
                    where = (R, T, H, norm, p)
                    assert R % lanes == 0 and (lanes in (1, R) or vec == 8), where
                    assert p["threads"] == lanes * nvc <= 512, where
                    assert p["splits"] * p["slice"] >= H // vec, where
                    assert p["grid"] == T * p["splits"], where
                    assert p["smem_bytes"] <= 48 * 1024, where
                    if norm:
                        assert p["threads"] % 32 == 0, where
                        assert p["passes"] in (1, 2, 4, 8), where
                        assert p["passes"] * nvc >= p["slice"], where
                        assert p["cluster"] == p["splits"] <= 16, where
                        # phase 2's kept vectors fit its shared memory too
                        assert p["passes"] * nvc * 16 <= 48 * 1024, where
                    else:
                        assert p["cluster"] == 1, where


def test_allreduce_parity_shapes_cover_every_layout(mf):
    """The all-reduce parity cases run every kernel layout the planner can
    pick: one rank per thread group, rank pairs and one thread summing all
    ranks, each with and without RMSNorm, and the scalar (unaligned-H) path."""
    from test_allreduce import CASES
    seen = set()
    for R, T, K, H, wkind, norm in CASES:
        p = mf.allreduce_plan(R, T, H, norm)
        layout = ("scalar" if p["vec"] == 1 else
                  "one rank per group" if p["lanes"] == R else
                  "all ranks" if p["lanes"] == 1 else
                  "rank pairs" if 2 * p["lanes"] == R else "two rank groups")
        seen.add((layout, norm))
    want = {(lay, norm) for lay in ("one rank per group", "rank pairs", "all ranks")
            for norm in (False, True)} | {("scalar", True), ("two rank groups", True)}
    assert want <= seen, want - seen


def test_allreduce_kernel_indices_stay_in_their_buffers(mf):
    """The all-reduce kernel's index arithmetic, replayed on the host for
    every plan of the decode, test and benchmark shapes: each thread's rank
    and vector, the shared-memory words it writes (the ranks' partials of a
    pass, the kept residual_out vectors), the slot staging and the cluster
    pushes all stay inside what the plan allocates."""
    for R in range(1, 9):
        for T in (1, 4, 5, 16, 48, 64, 256, 1024):
            for H in (64, 100, 512, 1000, 2048, 4096, 4104, 5120, 7168, 16384):
                for norm in (False, True):
                    try:
                        p = mf.allreduce_plan(R, T, H, norm)
                    except mf.MoefError:
                        continue
                    vec, nvc, lanes, threads = p["vec"], p["nvc"], p["lanes"], p["threads"]
                    nvec = H // vec
                    vbytes = 16 if vec == 8 else 2
                    c = R // lanes                      # ranks per group
                    assert c * lanes == R and (c == 1 or vec == 8)
                    # exchanged partials of a pass: every group's (one rank per
                    # group), ranks c .. R-1 (groups of c ranks), none (one
                    # thread summing all ranks)
                    sp_bytes = 4 * vec * (R if 1 < lanes == R else R - c if lanes > 1 else 0) * nvc
                    keep_bytes = p["passes"] * nvc * vbytes if norm else 0
                    assert sp_bytes + keep_bytes == p["smem_bytes"]
                    assert threads <= 512 and threads // 32 <= 16 and R * 32 <= 256
                    assert lanes in (1, 2, R, R // 2)
                    for split in range(p["splits"]):
                        v_begin = split * p["slice"]
                        v_end = min(v_begin + p["slice"], nvec)
                        for tid in range(threads):
                            g, j = divmod(tid, nvc)
                            assert g < lanes
                            for rr in range(g * c, g * c + c):
                                assert rr < R
                                if lanes == R > 1:    # partial word (rr, j, .) of a pass
                                    assert (rr * nvc + j + 1) * vec * 4 <= sp_bytes
                                elif g > 0:           # groups of c: word (rr - c, j, .)
                                    assert 0 <= (rr - c) * nvc + j and \
                                        ((rr - c) * nvc + j + 1) * vec * 4 <= sp_bytes
                            q = 0
                            for base in range(v_begin, v_end, nvc):
                                v = base + j
                                if v < v_end:
                                    assert v * vec + vec <= H
                                    if norm:
                                        assert sp_bytes + (q * nvc + j + 1) * vbytes <= \
                                            p["smem_bytes"]
                                q += 1
                            if norm:
                                assert q <= p["passes"]
                    if norm and p["cluster"] > 1:
                        assert p["cluster"] == p["splits"] <= min(16, threads)
                    # phase 2 of plans with groups of several ranks: the nvc
                    # finishing threads alone, in whole warps, with the kept
                    # vectors at the start of shared memory
                    threads2 = -(-nvc // 32) * 32
                    assert threads2 <= 512 and (not norm or threads % 32 == 0)
                    for split in range(p["splits"]):
                        v_begin = split * p["slice"]
                        v_end = min(v_begin + p["slice"], nvec)
                        for j in range(nvc):
                            q = 0
                            for base in range(v_begin, v_end, nvc):
                                if base + j < v_end:
                                    assert (base + j) * vec + vec <= H
                                    if norm:
                                        assert (q * nvc + j + 1) * vbytes <= keep_bytes
                                q += 1
                    if norm and p["cluster"] > 1:
                        assert p["cluster"] <= threads2


def test_every_accepted_norm_plan_covers_its_slice_in_one_pass(mf):
    """The RMSNorm kernel makes one pass over its slice, and its launcher
    refuses a plan that leaves vectors without a thread; so every plan the
    planner accepts with RMSNorm, automatic or hinted, must cover its slice."""
    accepted = 0
    for H in (8, 40, 64, 1000, 2048, 4096, 4104, 5120, 7168, 8192, 16384, 32768, 65536,
              262144):
        for T in (1, 16, 192, 640, 4096):
            for splits in (0, 1, 2, 3, 4, 7, 8, 12, 16):
                for threads in (0, 32, 64, 128, 256):
                    for vec_ok in (True, False):
                        try:
                            p = mf.plan(T, 8, H, True, vec_ok, splits=splits, threads=threads)
                        except mf.MoefError as e:
                            assert e.status in (2, 4)
                            continue
                        accepted += 1
                        assert p["threads"] * p["vpt"] >= p["slice"], (H, T, splits, threads, p)
                        assert p["splits"] * p["slice"] >= H // p["vec"]
    assert accepted > 1000


def test_plan_size_limits(mf):
    # the grid is T * splits CTAs and must fit a signed 32-bit count
    p = mf.plan(2**31 // 8, 8, 7168, False)
    assert p["grid"] == (2**31 // 8) * p["splits"] <= 2**31 - 1
    with pytest.raises(mf.MoefError) as e:
        mf.plan(2**31 - 1, 8, 7168, True, splits=2)
    assert e.value.status == 2
    # RMSNorm rows: at most 16 CTAs x 256 threads x 8 vectors of 8 values
    assert mf.plan(1, 8, 262144, True)["cluster"] == 16
    with pytest.raises(mf.MoefError):
        mf.plan(1, 8, 262152, True)
    # without RMSNorm any row length works
    p = mf.plan(1, 8, 8 * 2**20, False)
    assert p["splits"] * p["slice"] * 8 >= 8 * 2**20
    p = mf.plan(2**30, 8, 7168, False)      # grid capped: fewer, longer slices
    assert p["grid"] <= 2**31 - 1 and p["vpt"] == 8


def test_plan_hints(mf):
    p = mf.plan(1, 8, 7168, False, splits=28, threads=32)
    assert (p["splits"], p["slice"], p["threads"], p["vpt"]) == (28, 32, 32, 1)
    with pytest.raises(mf.MoefError):
        mf.plan(1, 8, 7168, False, threads=48)
    with pytest.raises(mf.MoefError):
        mf.plan(1, 8, 7168, True, splits=17)
    with pytest.raises(mf.MoefError):
        mf.plan(1, 8, 7168, True, splits=1, threads=32)   # norm row needs 28 vectors/thread


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libmoe_finalize.so there is no other path: every call raises."""
    from moe_deferred_finalize_gb300 import _abi
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_abi, "_LIB", None)
    with pytest.raises(RuntimeError, match="not built"):
        _abi.lib()
    with pytest.raises(RuntimeError, match="not built"):
        _abi.plan(1, 8, 7168, False)


def test_fastcall_packs_arguments_in_abi_order(mf):
    """The extension's packed replay (bind()) and direct call (moe_finalize)
    pass each argument to the same position as ctypes does: every error
    below is triggered by one argument alone."""
    from moe_deferred_finalize_gb300 import _abi
    fast = _abi._fastcall()
    if fast is None:
        pytest.skip("_fastcall not built (no Python headers)")
    lib = mf.lib()
    fn = ctypes.cast(lib.moe_finalize_ex, ctypes.c_void_p).value
    base = dict(x=A, P=16, idx=A, w=A, wkind=0, scale=1.0, shared=A, residual=None,
                gamma=None, eps=1e-6, out=A, residual_out=None, norm_out=None, T=2, K=2, H=8,
                splits=0, threads=0, flags=0)
    order = list(base)
    cases = [dict(T=0), dict(x=None), dict(idx=None), dict(w=None), dict(shared=None),
             dict(out=None), dict(residual=A), dict(gamma=A), dict(residual_out=A),
             dict(norm_out=A), dict(wkind=3), dict(K=33), dict(H=0), dict(P=0), dict(x=A + 1),
             dict(out=A + 1), dict(idx=A + 2), dict(w=A + 2), dict(splits=-1),
             dict(flags=4), dict(residual=A, gamma=A, residual_out=A, norm_out=A, eps=-1.0)]
    seen = set()
    for c in cases:
        a = {**base, **c}
        vals = [a[k] for k in order]
        st_ctypes = lib.moe_finalize_ex(*vals, None)
        st_fast = fast.call(fast.pack(fn, *vals), 0)
        assert st_fast == st_ctypes, (c, st_fast, st_ctypes)
        st_now = fast.call_now(fn, *vals, 0)
        assert st_now == st_ctypes, (c, st_now, st_ctypes)
        seen.add(st_ctypes)
    assert seen == {0, 1, 2, 3, 4}
    with pytest.raises(ValueError):
        fast.pack(0, *[base[k] for k in order])
    with pytest.raises(TypeError):
        fast.call_now(fn, *[base[k] for k in order])     # the stream is missing


def test_calls_switch_to_the_tensors_device(monkeypatch):
    """The library enqueues on the calling thread's current CUDA device, so
    the binding makes the tensors' device current around each call."""
    import contextlib
    import torch
    from moe_deferred_finalize_gb300 import _abi
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    assert isinstance(_abi._on(torch.device("cuda", 0)), contextlib.nullcontext)
    assert isinstance(_abi._on(torch.device("cuda")), contextlib.nullcontext)
    guard = _abi._on(torch.device("cuda", 1))
    assert isinstance(guard, torch.cuda.device) and guard.idx == 1


def test_fastcall_checked_call_refuses_what_the_binding_refuses(mf):
    """checked_call does the binding's checks on DLPack descriptions: one
    hand-made description per tensor (made-up addresses, never read), each
    single violation refused with -1; a valid set passes the checks and
    reaches the library, which returns its CUDA status here (no GPU)."""
    from moe_deferred_finalize_gb300 import _abi
    fast = _abi._fastcall()
    if fast is None:
        pytest.skip("_fastcall not built (no Python headers)")

    class DLTensor(ctypes.Structure):
        _fields_ = [("data", ctypes.c_void_p), ("device_type", ctypes.c_int32),
                    ("device_id", ctypes.c_int32), ("ndim", ctypes.c_int32),
                    ("code", ctypes.c_uint8), ("bits", ctypes.c_uint8),
                    ("lanes", ctypes.c_uint16), ("shape", ctypes.POINTER(ctypes.c_int64)),
                    ("strides", ctypes.POINTER(ctypes.c_int64)),
                    ("byte_offset", ctypes.c_uint64)]

    class DLManaged(ctypes.Structure):
        _fields_ = [("t", DLTensor), ("ctx", ctypes.c_void_p), ("deleter", ctypes.c_void_p)]

    new_capsule = ctypes.pythonapi.PyCapsule_New
    new_capsule.restype = ctypes.py_object
    new_capsule.argtypes = [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_void_p]
    keep = []

    def cap(shape, code=4, bits=16, dev=0, dev_type=2, strides=None, addr=A):
        shp = (ctypes.c_int64 * len(shape))(*shape)
        st = None
        if strides is not None:
            st = (ctypes.c_int64 * len(strides))(*strides)
        m = DLManaged(DLTensor(addr, dev_type, dev, len(shape), code, bits, 1,
                               ctypes.cast(shp, ctypes.POINTER(ctypes.c_int64)),
                               ctypes.cast(st, ctypes.POINTER(ctypes.c_int64)) if st else None,
                               0), None, None)
        keep.extend([shp, st, m])
        return new_capsule(ctypes.addressof(m), b"dltensor", None)

    T, K, H, P = 3, 2, 16, 8
    fn = ctypes.cast(mf.lib().moe_finalize_ex, ctypes.c_void_p).value

    def base():
        return dict(x=cap((P, H)), idx=cap((T, K), 0, 32), w=cap((T, K), 2, 32),
                    sh=cap((T, H)), res=None, gam=None, out=cap((T, H)), rout=None, nout=None)

    def run(**kw):
        a = {**base(), **kw}
        return fast.checked_call(fn, 0, 2, 32, 1.0, 1e-6, 0, 0, 0, 0, 0,
                                 a["x"], a["idx"], a["w"], a["sh"], a["res"], a["gam"],
                                 a["out"], a["rout"], a["nout"])

    passes = run()
    assert passes in (0, 5)       # the library ran: launched, or no CUDA device here
    norm = dict(res=cap((T, H)), gam=cap((H,)), rout=cap((T, H)), nout=cap((T, H)))
    assert run(**norm) == passes and run(**{**norm, "out": None}) == passes
    bad = [dict(x=cap((P, H), dev=1)), dict(x=cap((P, H), dev_type=1)),
           dict(x=cap((P, H), code=2, bits=32)), dict(x=cap((P, H, 1))),
           dict(x=cap((P, H), strides=(1, P))), dict(idx=cap((T, K), 2, 32)),
           dict(idx=cap((T + 1, K), 0, 32)), dict(w=cap((T, K), 4, 16)),
           dict(w=cap((T, K + 1), 2, 32)), dict(sh=cap((T, H + 8))), dict(sh=cap((T + 1, H))),
           dict(out=None), dict(out=cap((T, H), code=0)), dict(out=cap((T, H), strides=(H + 8, 1))),
           dict(res=cap((T, H))), dict(rout=cap((T, H))), dict(**{**norm, "nout": None}),
           dict(**{**norm, "gam": cap((H + 8,))}), dict(**{**norm, "rout": cap((T, H - 8))})]
    for kw in bad:
        assert run(**kw) == -1, kw
    # a strided size-1 dimension is still dense (torch reports such strides)
    assert run(out=cap((1, H), strides=(999, 1)), sh=cap((1, H)), idx=cap((1, K), 0, 32),
               w=cap((1, K), 2, 32)) == passes
