"""ctypes binding of libmoe_finalize.so (declared in include/moe_finalize.h).

Argument marshalling only: shape/dtype checks, output allocation through
torch, the current CUDA stream, and status -> exception.  Every step of the
finalize runs in the library's CUDA kernels; there is no other code path,
and calls fail loudly when the library has not been built.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch
import torch.utils.dlpack

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_finalize.so")
ABI_VERSION = 1     # MOEF_ABI_VERSION of include/moe_finalize.h

WKIND = {"fp32": 0, "bf16": 1, "packed": 2}
_WDTYPE = {"fp32": (torch.float32,), "bf16": (torch.bfloat16, torch.int16),
           "packed": (torch.int32,)}

STATUS = {0: "MOEF_OK", 1: "MOEF_ERR_NULL", 2: "MOEF_ERR_SHAPE", 3: "MOEF_ERR_ALIGN",
          4: "MOEF_ERR_ARG", 5: "MOEF_ERR_CUDA", 6: "MOEF_ERR_INDEX"}


class MoefError(RuntimeError):
    """A non-OK status from the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        text = _lib().moef_status_string(status).decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({text})")


class Plan(ctypes.Structure):
    _fields_ = [("vec", ctypes.c_int), ("splits", ctypes.c_int), ("slice", ctypes.c_int),
                ("threads", ctypes.c_int), ("vpt", ctypes.c_int), ("cluster", ctypes.c_int),
                ("grid", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class RankInputs(ctypes.Structure):
    """moef_rank_inputs: one rank's operands of the all-reduce-fused finalize."""
    _fields_ = [("permuted_out", ctypes.c_void_p), ("P", ctypes.c_int64),
                ("idx_map", ctypes.c_void_p), ("weights", ctypes.c_void_p),
                ("shared_out", ctypes.c_void_p)]


class ArPlan(ctypes.Structure):
    _fields_ = [("vec", ctypes.c_int), ("lanes", ctypes.c_int), ("nvc", ctypes.c_int),
                ("threads", ctypes.c_int), ("splits", ctypes.c_int), ("slice", ctypes.c_int),
                ("passes", ctypes.c_int), ("cluster", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("grid", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


MAX_RANKS = 8       # MOEF_MAX_RANKS


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libmoe_finalize.so is not built (there is no fallback path); build it with "
                "`python -m moe_deferred_finalize_gb300.build` or __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        common = [vp, i64, vp, vp, i32, f32, vp, vp, vp, f32, vp, vp, vp, i32, i32, i32]
        lib.moe_finalize.argtypes = common + [vp]
        lib.moe_finalize.restype = i32
        lib.moe_finalize_ex.argtypes = common + [i32, i32, ctypes.c_uint, vp]
        lib.moe_finalize_ex.restype = i32
        lib.moe_finalize_unfused.argtypes = common + [vp, ctypes.c_size_t, vp]
        lib.moe_finalize_unfused.restype = i32
        lib.moe_finalize_unfused_noalloc.argtypes = common + [vp]
        lib.moe_finalize_unfused_noalloc.restype = i32
        lib.moe_finalize_unfused_workspace_bytes.argtypes = [i32, i32]
        lib.moe_finalize_unfused_workspace_bytes.restype = ctypes.c_size_t
        lib.moe_finalize_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32,
                                          ctypes.POINTER(Plan)]
        lib.moe_finalize_plan.restype = i32
        lib.moe_finalize_allreduce.argtypes = [ctypes.POINTER(RankInputs), i32, i32, f32, vp, vp,
                                               f32, vp, vp, vp, i32, i32, i32, vp]
        lib.moe_finalize_allreduce.restype = i32
        lib.moe_finalize_partial.argtypes = [vp, i64, vp, vp, i32, f32, vp, vp, i32, i32, i32,
                                             vp]
        lib.moe_finalize_partial.restype = i32
        lib.moe_finalize_allreduce_reduce.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32, vp,
                                                      vp, f32, vp, vp, vp, i32, i32, vp]
        lib.moe_finalize_allreduce_reduce.restype = i32
        lib.moe_finalize_allreduce_plan.argtypes = [i32, i32, i32, i32, i32, i32,
                                                    ctypes.POINTER(ArPlan)]
        lib.moe_finalize_allreduce_plan.restype = i32
        lib.moe_topk_route.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp]
        lib.moe_topk_route.restype = i32
        lib.pack_topk_ids.argtypes = [vp, vp, i64, vp, vp]
        lib.pack_topk_ids.restype = i32
        lib.unpack_topk_ids.argtypes = [vp, i64, vp, vp, vp]
        lib.unpack_topk_ids.restype = i32
        lib.moe_finalize_check_indices.argtypes = [vp, i32, i32, i64, vp, vp]
        lib.moe_finalize_check_indices.restype = i32
        lib.moef_status_string.argtypes = [i32]
        lib.moef_status_string.restype = ctypes.c_char_p
        lib.moef_abi_version.argtypes = []
        lib.moef_abi_version.restype = i32
        if lib.moef_abi_version() != ABI_VERSION:
            raise RuntimeError(
                f"libmoe_finalize.so reports interface version {lib.moef_abi_version()}, "
                f"this binding expects {ABI_VERSION}: rebuild the library")
        _LIB = lib
    return _LIB


def lib():
    """The loaded ctypes library (raw C ABI)."""
    return _lib()


_FAST = False


def _fastcall():
    """The _fastcall extension (bound-call replay) if it was built, else None."""
    global _FAST
    if _FAST is False:
        try:
            from . import _fastcall as fast
        except ImportError:
            fast = None
        _FAST = fast
    return _FAST


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


# The current stream's raw handle for a device index, without building a
# torch.cuda.Stream object (a tenth of the host time of current_stream()).
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device) -> int:
    """cudaStream_t handle (an int) for a call on ``device``: ``stream`` if
    given (torch.cuda.Stream, ctypes.c_void_p or int), else the device's
    current stream."""
    if stream is None:
        if _RAW_STREAM is not None and device is not None and device.index is not None:
            return _RAW_STREAM(device.index)
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, ctypes.c_void_p):
        return stream.value or 0
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


_EX_ADDRESS = None


def _call_ex(args, stream: int) -> int:
    """One moe_finalize_ex call: through the _fastcall extension when it was
    built (direct argument conversion), else through ctypes."""
    global _EX_ADDRESS
    fast = _fastcall()
    if fast is not None:
        if _EX_ADDRESS is None:
            _EX_ADDRESS = ctypes.cast(_lib().moe_finalize_ex, ctypes.c_void_p).value
        return fast.call_now(_EX_ADDRESS, *args, stream)
    return _lib().moe_finalize_ex(*args, stream)


def _on(device):
    """Make ``device`` the current CUDA device for the duration of a call:
    the library enqueues on the calling thread's current device."""
    if device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _check(t, name, dtypes, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device is _PINNED:
        if t.is_cuda or not t.is_pinned():
            raise ValueError(f"{name} must be a pinned (page-locked) CPU tensor")
    elif not t.is_cuda or t.get_device() != device.index:
        raise ValueError(f"{name} is on {t.device}, expected a CUDA tensor on {device}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_BF16 = (torch.bfloat16,)
_PINNED = object()      # "device" of host tensors read and written in place by the kernel


def _empty_like(t, device):
    """An uninitialised bf16 tensor shaped like the checked [T, H] tensor t."""
    if device is _PINNED:
        return torch.empty(t.shape, dtype=torch.bfloat16, pin_memory=True)
    return torch.empty_like(t)


FLAG_ROUTING_READY = 1
FLAG_NO_PDL = 2


def _marshal(permuted_out, idx_map, weights, wkind, shared_out, routed_scale, residual, gamma,
             eps, out, residual_out, norm_out, write_out, splits, threads, host=False,
             routing_ready=False, pdl=True):
    """Validate, allocate missing outputs; returns (C arguments, outputs).
    host=True: every tensor is a pinned CPU tensor, used in place."""
    if wkind not in WKIND:
        raise ValueError(f"wkind must be one of {sorted(WKIND)}")
    if host:
        device = _PINNED
    else:
        device = permuted_out.device
        if device.type != "cuda":
            raise ValueError("permuted_out must be a CUDA tensor")
    if permuted_out.dim() != 2 or idx_map.dim() != 2:
        raise ValueError("permuted_out is [P, H] and idx_map is [T, K]")
    P, H = permuted_out.shape
    T, K = idx_map.shape
    _check(permuted_out, "permuted_out", _BF16, (P, H), device)
    _check(idx_map, "idx_map", (torch.int32,), (T, K), device)
    _check(weights, "weights", _WDTYPE[wkind], (T, K), device)
    _check(shared_out, "shared_out", _BF16, (T, H), device)
    norm = residual is not None
    if norm != (gamma is not None):
        raise ValueError("residual and gamma go together")
    if norm:
        _check(residual, "residual", _BF16, (T, H), device)
        _check(gamma, "gamma", _BF16, (H,), device)
        if residual_out is None:
            residual_out = _empty_like(shared_out, device)
        if norm_out is None:
            norm_out = _empty_like(shared_out, device)
        _check(residual_out, "residual_out", _BF16, (T, H), device)
        _check(norm_out, "norm_out", _BF16, (T, H), device)
    elif residual_out is not None or norm_out is not None:
        raise ValueError("residual_out / norm_out need a residual")
    if not norm or write_out:
        if out is None:
            out = _empty_like(shared_out, device)
        _check(out, "out", _BF16, (T, H), device)
    else:
        out = None
    args = (_ptr(permuted_out), P, _ptr(idx_map), _ptr(weights), WKIND[wkind],
            float(routed_scale), _ptr(shared_out), _ptr(residual), _ptr(gamma), float(eps),
            _ptr(out), _ptr(residual_out), _ptr(norm_out), T, K, H, int(splits), int(threads),
            (FLAG_ROUTING_READY if routing_ready else 0) | (0 if pdl else FLAG_NO_PDL))
    res = {"out": out}
    if norm:
        res["residual_out"] = residual_out
        res["norm_out"] = norm_out
    return args, res


def moe_finalize(permuted_out: torch.Tensor, idx_map: torch.Tensor, weights: torch.Tensor,
                 wkind: str, shared_out: torch.Tensor, *, routed_scale: float = 1.0,
                 residual: Optional[torch.Tensor] = None, gamma: Optional[torch.Tensor] = None,
                 eps: float = 1e-6, out: Optional[torch.Tensor] = None,
                 residual_out: Optional[torch.Tensor] = None,
                 norm_out: Optional[torch.Tensor] = None, write_out: bool = True,
                 splits: int = 0, threads: int = 0, routing_ready: bool = False,
                 pdl: bool = True, stream=None) -> dict:
    """Deferred MoE finalize on the GPU (see include/moe_finalize.h).

    permuted_out bf16 [P, H]; idx_map int32 [T, K]; weights [T, K] encoded
    as ``wkind`` ("fp32": float32, "bf16": bfloat16, "packed": int32 words
    (expert_id << 16) | bf16(weight)); shared_out bf16 [T, H]; optional
    residual bf16 [T, H] with gamma bf16 [H].  Outputs are allocated when not
    given; with a residual, ``write_out=False`` skips ``out``.  Returns a dict
    with "out" and, with a residual, "residual_out" and "norm_out".
    Enqueued on the current stream (or ``stream``); nothing is synchronised.
    ``routing_ready``: idx_map and weights were complete before the previous
    kernel on the stream started (MOEF_FLAG_ROUTING_READY).  ``pdl=False``:
    launch as a plain stream-ordered kernel (MOEF_FLAG_NO_PDL).
    """
    res = _checked_fast(permuted_out, idx_map, weights, wkind, shared_out, routed_scale,
                        residual, gamma, eps, out, residual_out, norm_out, write_out, splits,
                        threads, (FLAG_ROUTING_READY if routing_ready else 0) |
                        (0 if pdl else FLAG_NO_PDL), stream)
    if res is not None:
        return res
    args, res = _marshal(permuted_out, idx_map, weights, wkind, shared_out, routed_scale,
                         residual, gamma, eps, out, residual_out, norm_out, write_out, splits,
                         threads, routing_ready=routing_ready, pdl=pdl)
    device = permuted_out.device
    with _on(device):
        st = _call_ex(args, _stream(stream, device))
    if st != 0:
        raise MoefError(st, "moe_finalize")
    return res


# DLPack element types of the weight encodings (code, bits): fp32, bf16 bits,
# packed int32 words
_WCODE = {"fp32": (2, 32), "bf16": (4, 16), "packed": (0, 32)}
_TO_DLPACK = torch.utils.dlpack.to_dlpack


def _checked_fast(permuted_out, idx_map, weights, wkind, shared_out, routed_scale, residual,
                  gamma, eps, out, residual_out, norm_out, write_out, splits, threads, flags,
                  stream):
    """The checked call in one pass through the _fastcall extension: each
    tensor is described by one DLPack export, and the extension checks
    device, dtype, rank, shapes and layout before calling moe_finalize_ex.
    Returns the result dict, or None when the extension is missing or any
    check fails (the caller then runs the Python checks, which name the
    problem); a failed library status raises as usual."""
    fast = _fastcall()
    if fast is None or wkind not in _WCODE or not isinstance(shared_out, torch.Tensor):
        return None
    try:
        dev = permuted_out.get_device()
        if dev < 0 or dev != torch.cuda.current_device():
            return None
        if residual is not None:
            if residual_out is None:
                residual_out = torch.empty_like(shared_out)
            if norm_out is None:
                norm_out = torch.empty_like(shared_out)
            if not write_out:
                out = None
            elif out is None:
                out = torch.empty_like(shared_out)
        elif out is None:
            out = torch.empty_like(shared_out)
        d = _TO_DLPACK
        caps = [None if t is None else d(t)
                for t in (permuted_out, idx_map, weights, shared_out, residual, gamma, out,
                          residual_out, norm_out)]
    except (AttributeError, TypeError, RuntimeError):
        return None
    global _EX_ADDRESS
    if _EX_ADDRESS is None:
        _EX_ADDRESS = ctypes.cast(_lib().moe_finalize_ex, ctypes.c_void_p).value
    code, bits = _WCODE[wkind]
    st = fast.checked_call(_EX_ADDRESS, WKIND[wkind], code, bits, float(routed_scale),
                           float(eps), dev, int(splits), int(threads), flags,
                           _RAW_STREAM(dev) if stream is None and _RAW_STREAM is not None
                           else _stream(stream, torch.device("cuda", dev)), *caps)
    if st < 0:
        return None
    if st != 0:
        raise MoefError(st, "moe_finalize")
    res = {"out": out}
    if residual is not None:
        res["residual_out"] = residual_out
        res["norm_out"] = norm_out
    return res


def unfused_workspace_bytes(T: int, H: int) -> int:
    """Bytes of workspace moe_finalize_unfused needs for T tokens of H values."""
    return int(_lib().moe_finalize_unfused_workspace_bytes(int(T), int(H)))


def moe_finalize_unfused(permuted_out: torch.Tensor, idx_map: torch.Tensor,
                         weights: torch.Tensor, wkind: str, shared_out: torch.Tensor, *,
                         routed_scale: float = 1.0, residual: Optional[torch.Tensor] = None,
                         gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
                         out: Optional[torch.Tensor] = None,
                         residual_out: Optional[torch.Tensor] = None,
                         norm_out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, stream=None) -> dict:
    """The finalize as separate kernels (combine, shared add, residual +
    RMSNorm) with a bf16 intermediate in ``workspace`` (allocated when not
    given): the A/B baseline of the fused ``moe_finalize``.  Same arguments;
    ``out`` is always produced."""
    args, res = _marshal(permuted_out, idx_map, weights, wkind, shared_out, routed_scale,
                         residual, gamma, eps, out, residual_out, norm_out, True, 0, 0)
    T, H = idx_map.shape[0], permuted_out.shape[1]
    need = unfused_workspace_bytes(T, H)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=permuted_out.device)
    if workspace.device != permuted_out.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the same device")
    nbytes = workspace.numel() * workspace.element_size()
    with _on(permuted_out.device):
        st = _lib().moe_finalize_unfused(*args[:16], _ptr(workspace), nbytes,
                                         _stream(stream, permuted_out.device))
    if st != 0:
        raise MoefError(st, "moe_finalize_unfused")
    return res


NOALLOC_SCRATCH_BYTES = 8 << 20


def moe_finalize_unfused_noalloc(permuted_out: torch.Tensor, idx_map: torch.Tensor,
                                 weights: torch.Tensor, wkind: str, shared_out: torch.Tensor,
                                 *, routed_scale: float = 1.0,
                                 residual: Optional[torch.Tensor] = None,
                                 gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
                                 out: torch.Tensor, residual_out: Optional[torch.Tensor] = None,
                                 norm_out: Optional[torch.Tensor] = None, stream=None) -> dict:
    """``moe_finalize_unfused`` for callers that cannot allocate device
    memory (fixed-memory serving engines, plugins with no allocator): the
    workspace is the library's fixed 8 MiB scratch array,
    so T * H * 2 must not exceed ``NOALLOC_SCRATCH_BYTES``.  All outputs must
    be given (this wrapper allocates nothing either).  Calls on one device
    share the scratch: order them (one stream, or events)."""
    T, H = idx_map.shape[0], permuted_out.shape[1]
    if T * H * 2 > NOALLOC_SCRATCH_BYTES:
        raise ValueError(f"T*H*2 = {T * H * 2} bytes exceed the fixed scratch of "
                         f"{NOALLOC_SCRATCH_BYTES} bytes")
    if residual is not None and (residual_out is None or norm_out is None):
        raise ValueError("with a residual, residual_out and norm_out must be given")
    args, res = _marshal(permuted_out, idx_map, weights, wkind, shared_out, routed_scale,
                         residual, gamma, eps, out, residual_out, norm_out, True, 0, 0)
    with _on(permuted_out.device):
        st = _lib().moe_finalize_unfused_noalloc(*args[:16],
                                                 _stream(stream, permuted_out.device))
    if st != 0:
        raise MoefError(st, "moe_finalize_unfused_noalloc")
    return res


def moe_finalize_host(permuted_out: torch.Tensor, idx_map: torch.Tensor, weights: torch.Tensor,
                      wkind: str, shared_out: torch.Tensor, *, device=None,
                      routed_scale: float = 1.0, residual: Optional[torch.Tensor] = None,
                      gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
                      out: Optional[torch.Tensor] = None,
                      residual_out: Optional[torch.Tensor] = None,
                      norm_out: Optional[torch.Tensor] = None, write_out: bool = True,
                      stream=None) -> dict:
    """The finalize on host buffers, without copies: every tensor is a
    pinned (page-locked) CPU tensor, and the kernel on ``device`` (default:
    the current CUDA device) reads the inputs and writes the outputs in host
    memory directly over the host link, so input reads, compute and output
    writes overlap.  Outputs are allocated pinned when not given.  Arguments
    as for ``moe_finalize``; results are bit-identical to it for the same
    launch plan.  Enqueued on the device's current stream (or ``stream``):
    synchronise before reading the outputs."""
    args, res = _marshal(permuted_out, idx_map, weights, wkind, shared_out, routed_scale,
                         residual, gamma, eps, out, residual_out, norm_out, write_out, 0, 0,
                         host=True)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    with _on(dev):
        st = _call_ex(args, _stream(stream, dev))
    if st != 0:
        raise MoefError(st, "moe_finalize_host")
    return res


class BoundFinalize:
    """A finalize whose arguments were checked and marshalled once.

    Calling it enqueues the same finalize again (same buffers, new contents
    allowed) with no per-call Python checks: the decode-loop form of
    ``moe_finalize``.  The tensors passed to ``bind`` must stay alive and
    keep their storage while the object is used, and their device must be
    the current CUDA device when the object is called (no per-call switch).
    """

    def __init__(self, args, res, stream, device):
        self._fn = _lib().moe_finalize_ex
        self._args = args
        self._stream = _stream(stream, device)
        self.outputs = res
        self._packed = None
        fast = _fastcall()
        if fast is not None:
            # the same arguments packed once into a C struct: each call then
            # passes only the stream to moe_finalize_ex
            fn = ctypes.cast(self._fn, ctypes.c_void_p).value
            self._packed = fast.pack(fn, *args)
            self._call = fast.call

    def __call__(self, stream=None):
        s = self._stream if stream is None else _stream(stream, None)
        if self._packed is not None:
            st = self._call(self._packed, s)
        else:
            st = self._fn(*self._args, s)
        if st != 0:
            raise MoefError(st, "moe_finalize")
        return self.outputs


def bind(permuted_out: torch.Tensor, idx_map: torch.Tensor, weights: torch.Tensor, wkind: str,
         shared_out: torch.Tensor, *, routed_scale: float = 1.0,
         residual: Optional[torch.Tensor] = None, gamma: Optional[torch.Tensor] = None,
         eps: float = 1e-6, out: Optional[torch.Tensor] = None,
         residual_out: Optional[torch.Tensor] = None, norm_out: Optional[torch.Tensor] = None,
         write_out: bool = True, splits: int = 0, threads: int = 0,
         routing_ready: bool = False, pdl: bool = True, stream=None) -> BoundFinalize:
    """Check and marshal a finalize once (arguments as for ``moe_finalize``);
    the returned object enqueues it on ``stream`` (default: the current
    stream at bind time) each time it is called."""
    args, res = _marshal(permuted_out, idx_map, weights, wkind, shared_out, routed_scale,
                         residual, gamma, eps, out, residual_out, norm_out, write_out, splits,
                         threads, routing_ready=routing_ready, pdl=pdl)
    return BoundFinalize(args, res, stream, permuted_out.device)


def plan(T: int, K: int, H: int, with_norm: bool, vec_ok: bool = True, num_sms: int = 152,
         splits: int = 0, threads: int = 0) -> dict:
    """The launch plan moe_finalize uses for these sizes (host computation only)."""
    p = Plan()
    st = _lib().moe_finalize_plan(T, K, H, int(with_norm), int(vec_ok), num_sms, splits,
                                  threads, ctypes.byref(p))
    if st != 0:
        raise MoefError(st, "moe_finalize_plan")
    return p.as_dict()


# ------------------------------------------ all-reduce-fused finalize


def _check_peer(t, name, dtypes, shape):
    """A rank's operand: a contiguous CUDA tensor on any device (a peer's
    buffer must be reachable from the calling device; that is the caller's
    set-up)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _epilogue(T, H, device, residual, gamma, out, residual_out, norm_out, write_out, like):
    """Checks (and allocates) the residual / RMSNorm operands and outputs."""
    norm = residual is not None
    if norm != (gamma is not None):
        raise ValueError("residual and gamma go together")
    if norm:
        _check(residual, "residual", _BF16, (T, H), device)
        _check(gamma, "gamma", _BF16, (H,), device)
        if residual_out is None:
            residual_out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        if norm_out is None:
            norm_out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        _check(residual_out, "residual_out", _BF16, (T, H), device)
        _check(norm_out, "norm_out", _BF16, (T, H), device)
    elif residual_out is not None or norm_out is not None:
        raise ValueError("residual_out / norm_out need a residual")
    if not norm or write_out:
        if out is None:
            out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        _check(out, "out", _BF16, (T, H), device)
    else:
        out = None
    res = {"out": out}
    if norm:
        res["residual_out"] = residual_out
        res["norm_out"] = norm_out
    return res


def _call_device(device, *candidates):
    if device is not None:
        return torch.device(device)
    for t in candidates:
        if isinstance(t, torch.Tensor) and t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def moe_finalize_allreduce(ranks, wkind: str, *, routed_scale: float = 1.0,
                           residual: Optional[torch.Tensor] = None,
                           gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
                           out: Optional[torch.Tensor] = None,
                           residual_out: Optional[torch.Tensor] = None,
                           norm_out: Optional[torch.Tensor] = None, write_out: bool = True,
                           device=None, stream=None) -> dict:
    """One-shot all-reduce-fused finalize (include/moe_finalize.h).

    ranks: a list of R dicts, in rank order, with "permuted_out" bf16
    [P_r, H], "idx_map" int32 [T, K], "weights" [T, K] (encoding ``wkind``)
    and "shared_out" bf16 [T, H]; CUDA tensors reachable from the calling
    device.  The residual, gamma and outputs are on the calling device
    (``device``, else the residual's or out's device, else the current one).
    Returns a dict like ``moe_finalize``.  Every rank's operands must be
    complete before the launch on the stream (the caller orders devices)."""
    if wkind not in WKIND:
        raise ValueError(f"wkind must be one of {sorted(WKIND)}")
    R = len(ranks)
    if not 1 <= R <= MAX_RANKS:
        raise ValueError(f"1 <= R <= {MAX_RANKS} ranks")
    dev = _call_device(device, residual, out, residual_out)
    x0, i0 = ranks[0]["permuted_out"], ranks[0]["idx_map"]
    if x0.dim() != 2 or i0.dim() != 2:
        raise ValueError("permuted_out is [P, H] and idx_map is [T, K]")
    H = x0.shape[1]
    T, K = i0.shape
    arr = (RankInputs * R)()
    for r, rk in enumerate(ranks):
        x = rk["permuted_out"]
        _check_peer(x, f"ranks[{r}].permuted_out", _BF16, None)
        if x.dim() != 2 or x.shape[1] != H:
            raise ValueError(f"ranks[{r}].permuted_out must be [P, {H}]")
        _check_peer(rk["idx_map"], f"ranks[{r}].idx_map", (torch.int32,), (T, K))
        _check_peer(rk["weights"], f"ranks[{r}].weights", _WDTYPE[wkind], (T, K))
        _check_peer(rk["shared_out"], f"ranks[{r}].shared_out", _BF16, (T, H))
        arr[r] = RankInputs(x.data_ptr(), x.shape[0], rk["idx_map"].data_ptr(),
                            rk["weights"].data_ptr(), rk["shared_out"].data_ptr())
    res = _epilogue(T, H, dev, residual, gamma, out, residual_out, norm_out, write_out, x0)
    with _on(dev):
        st = _lib().moe_finalize_allreduce(
            arr, R, WKIND[wkind], float(routed_scale), _ptr(residual), _ptr(gamma), float(eps),
            _ptr(res["out"]), _ptr(res.get("residual_out")), _ptr(res.get("norm_out")),
            T, K, H, _stream(stream, dev))
    if st != 0:
        raise MoefError(st, "moe_finalize_allreduce")
    return res


def moe_finalize_partial(permuted_out: torch.Tensor, idx_map: torch.Tensor,
                         weights: torch.Tensor, wkind: str, shared_out: torch.Tensor, *,
                         routed_scale: float = 1.0, partial: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """Phase 1 of the two-phase all-reduce-fused finalize: this rank's
    unrounded partial (weighted rows + shared output) as fp32 [T, H]
    (allocated when not given).  Arguments as for ``moe_finalize``."""
    if wkind not in WKIND:
        raise ValueError(f"wkind must be one of {sorted(WKIND)}")
    device = permuted_out.device
    if device.type != "cuda" or permuted_out.dim() != 2 or idx_map.dim() != 2:
        raise ValueError("permuted_out is a CUDA [P, H] tensor and idx_map is [T, K]")
    P, H = permuted_out.shape
    T, K = idx_map.shape
    _check(permuted_out, "permuted_out", _BF16, (P, H), device)
    _check(idx_map, "idx_map", (torch.int32,), (T, K), device)
    _check(weights, "weights", _WDTYPE[wkind], (T, K), device)
    _check(shared_out, "shared_out", _BF16, (T, H), device)
    if partial is None:
        partial = torch.empty((T, H), dtype=torch.float32, device=device)
    _check(partial, "partial", (torch.float32,), (T, H), device)
    with _on(device):
        st = _lib().moe_finalize_partial(_ptr(permuted_out), P, _ptr(idx_map), _ptr(weights),
                                         WKIND[wkind], float(routed_scale), _ptr(shared_out),
                                         _ptr(partial), T, K, H, _stream(stream, device))
    if st != 0:
        raise MoefError(st, "moe_finalize_partial")
    return partial


def moe_finalize_allreduce_reduce(partials, *, residual: Optional[torch.Tensor] = None,
                                  gamma: Optional[torch.Tensor] = None, eps: float = 1e-6,
                                  out: Optional[torch.Tensor] = None,
                                  residual_out: Optional[torch.Tensor] = None,
                                  norm_out: Optional[torch.Tensor] = None,
                                  write_out: bool = True, device=None, stream=None) -> dict:
    """Phase 2: sum the ranks' fp32 partials [T, H] (a list in rank order,
    CUDA tensors reachable from the calling device), then the residual add
    and RMSNorm; outputs as for ``moe_finalize_allreduce`` and bit-identical
    to it."""
    R = len(partials)
    if not 1 <= R <= MAX_RANKS:
        raise ValueError(f"1 <= R <= {MAX_RANKS} partials")
    if partials[0].dim() != 2:
        raise ValueError("partials are [T, H]")
    T, H = partials[0].shape
    for r, t in enumerate(partials):
        _check_peer(t, f"partials[{r}]", (torch.float32,), (T, H))
    dev = _call_device(device, residual, out, residual_out)
    res = _epilogue(T, H, dev, residual, gamma, out, residual_out, norm_out, write_out, None)
    arr = (ctypes.c_void_p * R)(*[t.data_ptr() for t in partials])
    with _on(dev):
        st = _lib().moe_finalize_allreduce_reduce(
            arr, R, _ptr(residual), _ptr(gamma), float(eps), _ptr(res["out"]),
            _ptr(res.get("residual_out")), _ptr(res.get("norm_out")), T, H, _stream(stream, dev))
    if st != 0:
        raise MoefError(st, "moe_finalize_allreduce_reduce")
    return res


def allreduce_plan(R: int, T: int, H: int, with_norm: bool, vec_ok: bool = True,
                   num_sms: int = 152) -> dict:
    """The launch plan of the one-shot and phase-2 calls (phase 1: R = 1,
    with_norm = False); host computation only."""
    p = ArPlan()
    st = _lib().moe_finalize_allreduce_plan(R, T, H, int(with_norm), int(vec_ok), num_sms,
                                            ctypes.byref(p))
    if st != 0:
        raise MoefError(st, "moe_finalize_allreduce_plan")
    return p.as_dict()


GATE = {"softmax": 0, "sigmoid": 1}


def topk_route(logits: torch.Tensor, K: int, kind: str = "sigmoid", *,
               want_ids: bool = True, want_weights: bool = True, want_packed: bool = False,
               stream=None) -> dict:
    """Top-K gate over fp32 logits [T, E] (see include/moe_finalize.h):
    returns the requested of "expert_ids" int32 [T, K], "weights" fp32
    [T, K] and "packed" int32 [T, K] words."""
    if kind not in GATE:
        raise ValueError(f"kind must be one of {sorted(GATE)}")
    if logits.device.type != "cuda" or logits.dtype != torch.float32 or logits.dim() != 2 \
            or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous float32 [T, E] CUDA tensor")
    T, E = logits.shape
    dev = logits.device
    res = {}
    if want_ids:
        res["expert_ids"] = torch.empty((T, K), dtype=torch.int32, device=dev)
    if want_weights:
        res["weights"] = torch.empty((T, K), dtype=torch.float32, device=dev)
    if want_packed:
        res["packed"] = torch.empty((T, K), dtype=torch.int32, device=dev)
    with _on(dev):
        st = _lib().moe_topk_route(_ptr(logits), T, E, int(K), GATE[kind],
                                   _ptr(res.get("expert_ids")), _ptr(res.get("weights")),
                                   _ptr(res.get("packed")), _stream(stream, dev))
    if st != 0:
        raise MoefError(st, "moe_topk_route")
    return res


def pack_topk_ids(expert_ids: torch.Tensor, weights: torch.Tensor,
                  packed: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """(expert_id << 16) | bf16_rne(weight) words, same shape as the inputs."""
    if not isinstance(expert_ids, torch.Tensor) or not expert_ids.is_cuda:
        raise ValueError("expert_ids must be a CUDA tensor")
    dev = expert_ids.device
    _check(expert_ids, "expert_ids", (torch.int32,), expert_ids.shape, dev)
    _check(weights, "weights", (torch.float32,), expert_ids.shape, dev)
    if packed is None:
        packed = torch.empty_like(expert_ids)
    _check(packed, "packed", (torch.int32,), expert_ids.shape, dev)
    with _on(dev):
        st = _lib().pack_topk_ids(_ptr(expert_ids), _ptr(weights), expert_ids.numel(),
                                  _ptr(packed), _stream(stream, dev))
    if st != 0:
        raise MoefError(st, "pack_topk_ids")
    return packed


def unpack_topk_ids(packed: torch.Tensor, expert_ids: Optional[torch.Tensor] = None,
                    weights: Optional[torch.Tensor] = None, stream=None):
    """Packed int32 words -> (expert ids int32, weights float32), same shape."""
    if packed.device.type != "cuda" or packed.dtype != torch.int32 or not packed.is_contiguous():
        raise ValueError("packed must be a contiguous int32 CUDA tensor")
    device = packed.device
    if expert_ids is None:
        expert_ids = torch.empty_like(packed)
    if weights is None:
        weights = torch.empty(packed.shape, dtype=torch.float32, device=device)
    _check(expert_ids, "expert_ids", (torch.int32,), packed.shape, device)
    _check(weights, "weights", (torch.float32,), packed.shape, device)
    with _on(device):
        st = _lib().unpack_topk_ids(_ptr(packed), packed.numel(), _ptr(expert_ids),
                                    _ptr(weights), _stream(stream, device))
    if st != 0:
        raise MoefError(st, "unpack_topk_ids")
    return expert_ids, weights


def check_indices(idx_map: torch.Tensor, P: int, counter: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """Enqueue a count of idx_map entries outside [0, P); returns the device
    int32 [1] counter (read it after the stream has run)."""
    if idx_map.dim() != 2 or idx_map.dtype != torch.int32 or not idx_map.is_contiguous():
        raise ValueError("idx_map must be a contiguous int32 [T, K] tensor")
    device = idx_map.device
    if counter is None:
        counter = torch.empty(1, dtype=torch.int32, device=device)
    T, K = idx_map.shape
    with _on(device):
        st = _lib().moe_finalize_check_indices(_ptr(idx_map), T, K, int(P), _ptr(counter),
                                               _stream(stream, device))
    if st != 0:
        raise MoefError(st, "moe_finalize_check_indices")
    return counter
