"""Deferred MoE finalize: fp64 CPU oracle (Python face of ``finalize_ref.c``).

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  Nothing here is shared
with the CUDA path and nothing here touches a GPU.

All bf16 operands are passed as their uint16 bit patterns (numpy arrays);
outputs are float64 arrays, never rounded.  The definition, the sources and
the readings are in the header comment of ``finalize_ref.c``.
"""
import ctypes

import numpy as np

from .build import build_oracle

_WKIND = {"fp32": 0, "bf16": 1, "packed": 2}
_WDTYPE = {"fp32": np.float32, "bf16": np.uint16, "packed": np.int32}


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """The oracle library at ``libpath`` (a mutated copy can be loaded too)."""

    def __init__(self, libpath):
        lib = ctypes.CDLL(libpath)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oref_moe_finalize.restype = ctypes.c_int
        lib.oref_moe_finalize.argtypes = [p, i64, i64, p, p, ctypes.c_int, ctypes.c_double,
                                          p, p, p, ctypes.c_double, i64, i64, p, p, p]
        lib.oref_unpack_topk_ids.restype = None
        lib.oref_unpack_topk_ids.argtypes = [p, i64, p, p]
        lib.oref_pack_topk_id.restype = ctypes.c_int32
        lib.oref_pack_topk_id.argtypes = [ctypes.c_int32, ctypes.c_float]
        lib.oref_f32_to_bf16.restype = ctypes.c_uint16
        lib.oref_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oref_rmsnorm_bf16.restype = None
        lib.oref_rmsnorm_bf16.argtypes = [p, p, ctypes.c_double, i64, i64, p]
        lib.oref_pack_topk_ids.restype = None
        lib.oref_pack_topk_ids.argtypes = [p, p, i64, p]
        lib.oref_moe_finalize_ar.restype = ctypes.c_int
        lib.oref_moe_finalize_ar.argtypes = [i64, p, p, i64, p, p, ctypes.c_int,
                                             ctypes.c_double, p, p, p, ctypes.c_double,
                                             i64, i64, p, p, p]
        lib.oref_topk_route.restype = ctypes.c_int
        lib.oref_topk_route.argtypes = [p, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p]
        self.lib = lib

    def moe_finalize(self, permuted_out, idx, weights, wkind, routed_scale, shared,
                     residual=None, gamma=None, eps=1e-6, want_out=True):
        """fp64 deferred finalize.

        permuted_out: uint16 [P, H] bf16 bits; idx: int32 [T, K];
        weights: float32 [T, K] (wkind "fp32"), uint16 [T, K] ("bf16") or
        int32 [T, K] packed topk_ids ("packed"); shared: uint16 [T, H];
        residual: uint16 [T, H] or None; gamma: uint16 [H] (with residual).
        Returns a dict with float64 "out", and "residual_out"/"norm_out" when
        a residual is given.  Raises ValueError on an index outside [0, P).
        """
        permuted_out = _c(permuted_out, np.uint16)
        idx = _c(idx, np.int32)
        weights = _c(weights, _WDTYPE[wkind])
        shared = _c(shared, np.uint16)
        P, H = permuted_out.shape
        T, K = idx.shape
        if weights.shape != (T, K) or shared.shape != (T, H):
            raise ValueError("shape mismatch")
        if (residual is None) != (gamma is None):
            raise ValueError("residual and gamma go together")
        residual = _c(residual, np.uint16)
        gamma = _c(gamma, np.uint16)
        out = np.empty((T, H), np.float64) if want_out else None
        res_out = norm_out = None
        if residual is not None:
            if residual.shape != (T, H) or gamma.shape != (H,):
                raise ValueError("shape mismatch")
            res_out = np.empty((T, H), np.float64)
            norm_out = np.empty((T, H), np.float64)
        rc = self.lib.oref_moe_finalize(
            _ptr(permuted_out), P, H, _ptr(idx), _ptr(weights), _WKIND[wkind],
            float(routed_scale), _ptr(shared), _ptr(residual), _ptr(gamma), float(eps),
            T, K, _ptr(out), _ptr(res_out), _ptr(norm_out))
        if rc == -1:
            raise ValueError("index outside [0, P)")
        if rc != 0:
            raise ValueError(f"oracle returned {rc}")
        res = {"out": out}
        if residual is not None:
            res["residual_out"] = res_out
            res["norm_out"] = norm_out
        return res

    def moe_finalize_ar(self, ranks, wkind, routed_scale, residual=None, gamma=None,
                        eps=1e-6, want_out=True):
        """fp64 deferred finalize of R tensor-parallel ranks, all-reduced,
        then residual + RMSNorm.

        ranks: a list of R dicts with "permuted_out" uint16 [P_r, H],
        "idx" int32 [T, K], "weights" [T, K] (encoding ``wkind``, the same
        for every rank) and "shared" uint16 [T, H].  residual uint16 [T, H]
        and gamma uint16 [H] are common to all ranks.  Returns a dict like
        ``moe_finalize``.  Raises ValueError on an index outside a rank's
        [0, P_r).
        """
        if not ranks:
            raise ValueError("at least one rank")
        R = len(ranks)
        xs = [_c(r["permuted_out"], np.uint16) for r in ranks]
        idxs = [_c(r["idx"], np.int32) for r in ranks]
        ws = [_c(r["weights"], _WDTYPE[wkind]) for r in ranks]
        shs = [_c(r["shared"], np.uint16) for r in ranks]
        H = xs[0].shape[1]
        T, K = idxs[0].shape
        for x, i, w, sh in zip(xs, idxs, ws, shs):
            if x.ndim != 2 or x.shape[1] != H or i.shape != (T, K) or w.shape != (T, K) \
                    or sh.shape != (T, H):
                raise ValueError("shape mismatch between ranks")
        if (residual is None) != (gamma is None):
            raise ValueError("residual and gamma go together")
        residual = _c(residual, np.uint16)
        gamma = _c(gamma, np.uint16)
        out = np.empty((T, H), np.float64) if want_out else None
        res_out = norm_out = None
        if residual is not None:
            if residual.shape != (T, H) or gamma.shape != (H,):
                raise ValueError("shape mismatch")
            res_out = np.empty((T, H), np.float64)
            norm_out = np.empty((T, H), np.float64)
        ptrs = lambda arrs: (ctypes.c_void_p * R)(*[a.ctypes.data for a in arrs])
        P = (ctypes.c_int64 * R)(*[x.shape[0] for x in xs])
        rc = self.lib.oref_moe_finalize_ar(
            R, ptrs(xs), P, H, ptrs(idxs), ptrs(ws), _WKIND[wkind], float(routed_scale),
            ptrs(shs), _ptr(residual), _ptr(gamma), float(eps), T, K,
            _ptr(out), _ptr(res_out), _ptr(norm_out))
        if rc == -1:
            raise ValueError("index outside [0, P) on some rank")
        if rc != 0:
            raise ValueError(f"oracle returned {rc}")
        res = {"out": out}
        if residual is not None:
            res["residual_out"] = res_out
            res["norm_out"] = norm_out
        return res

    def rmsnorm_bf16(self, x_bits, gamma_bits, eps):
        """fp64 RMSNorm of bf16 rows: x / sqrt(mean(x^2) + eps) * gamma."""
        x = _c(x_bits, np.uint16)
        g = _c(gamma_bits, np.uint16)
        T, H = x.shape
        y = np.empty((T, H), np.float64)
        self.lib.oref_rmsnorm_bf16(_ptr(x), _ptr(g), float(eps), T, H, _ptr(y))
        return y

    def unpack_topk_ids(self, packed):
        """Packed int32 words -> (expert ids int32, weights float32)."""
        packed = _c(packed, np.int32)
        e = np.empty(packed.shape, np.int32)
        w = np.empty(packed.shape, np.float32)
        self.lib.oref_unpack_topk_ids(_ptr(packed), packed.size, _ptr(e), _ptr(w))
        return e, w

    def pack_topk_id(self, expert_id, weight):
        """One packed word (expert_id << 16) | bf16_rne(weight), as int32."""
        return int(self.lib.oref_pack_topk_id(int(expert_id), float(weight)))

    def pack_topk_ids(self, expert_ids, weights):
        """Packed words for arrays of expert ids (int32) and fp32 weights."""
        e = _c(expert_ids, np.int32)
        w = _c(weights, np.float32)
        out = np.empty(e.shape, np.int32)
        self.lib.oref_pack_topk_ids(_ptr(e), _ptr(w), e.size, _ptr(out))
        return out

    def topk_route(self, logits, K, kind):
        """Top-K gate over fp32 logits [T, E]: (ids int32 [T, K] in
        descending logit order, ties lowest id first; weights float64 [T, K],
        kind "softmax" or "sigmoid" over the selected logits)."""
        z = _c(logits, np.float32)
        T, E = z.shape
        ids = np.empty((T, K), np.int32)
        w = np.empty((T, K), np.float64)
        rc = self.lib.oref_topk_route(_ptr(z), T, E, K, {"softmax": 0, "sigmoid": 1}[kind],
                                      _ptr(ids), _ptr(w))
        if rc != 0:
            raise ValueError("bad sizes or kind")
        return ids, w

    def f32_to_bf16(self, x):
        """fp32 -> bf16 bits, round to nearest even, one value at a time."""
        flat = np.asarray(x, np.float32).ravel()
        f = self.lib.oref_f32_to_bf16
        out = np.fromiter((f(float(v)) for v in flat), np.uint16, flat.size)
        return out.reshape(np.shape(x))


_default = None


def default() -> Oracle:
    """The oracle built from ``finalize_ref.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build_oracle())
    return _default


def moe_finalize(*args, **kwargs):
    return default().moe_finalize(*args, **kwargs)


def moe_finalize_ar(*args, **kwargs):
    return default().moe_finalize_ar(*args, **kwargs)


def rmsnorm_bf16(*args, **kwargs):
    return default().rmsnorm_bf16(*args, **kwargs)


def unpack_topk_ids(packed):
    return default().unpack_topk_ids(packed)


def pack_topk_id(expert_id, weight):
    return default().pack_topk_id(expert_id, weight)


def f32_to_bf16(x):
    return default().f32_to_bf16(x)


def pack_topk_ids(expert_ids, weights):
    return default().pack_topk_ids(expert_ids, weights)


def topk_route(logits, K, kind):
    return default().topk_route(logits, K, kind)
