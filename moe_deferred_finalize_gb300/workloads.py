"""Seeded synthetic inputs for the deferred MoE finalize.

This module only *makes inputs*: the padded, expert-grouped permuted row
buffer that an expert GEMM run without its finalize would leave behind, the
[token, top_k] row map into it, the routing weights and the dense operands.
It holds none of the finalize's arithmetic.  Both the CUDA path's tests and
benchmark and the CPU oracle's tests consume what it returns.

Layout of the permuted buffer (the expert kernel's "unweighted expert
outputs", padded per expert, "[Kimi K2.5] Fuse deferred MoE finalize into
next-layer AR + residual + RMSNorm", Numerics & speed):

  * experts own tile-aligned blocks in ascending expert-id order;
  * an expert's valid rows fill the front of its block in token order;
  * the rest of a block is padding, filled with the sentinel 1e4
    (bf16 bits 0x461C) that must never reach an output.

Routing comes in two forms.  A *pool* routing draws each token's K distinct
experts uniformly from a seeded pool of ``P / tile`` experts (each owning one
block), redrawing until no block overflows (and, if asked, every pool expert
has a token); this keeps the stated row count P and tile exactly.  An
*exact-count* routing fixes how many tokens each expert receives, shuffles
that multiset of expert ids into [T, K] slots and repairs repeated experts
within a token by seeded swaps.

Values: valid rows, the shared-expert output ~ N(0, 1); the residual
~ N(0, 4) (variance 4, standard deviation 2); gamma ~ U(0.5, 1.5); routing
weights are a softmax or a normalised sigmoid of K standard-normal logits.
Every float operand is rounded to bf16 by torch's CPU conversion.  Packed
routing words are (expert_id << 16) | bf16(weight), the format named in
"[Deepseek V4] Keep fp32 routing weights in the mxfp4 trtllm MoE".

Every draw comes from ``numpy.random.PCG64`` streams spawned from one
``SeedSequence(seed)``, one stream per operand and one per chunk of rows,
so results do not depend on the number of threads used to make them.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Optional

import numpy as np
import torch

PAD_BITS = 0x461C          # bf16 bit pattern of 1e4 (exactly 9984.0)
ROWS_PER_CHUNK = 256

Alloc = Callable[[tuple, np.dtype], np.ndarray]


def _np_alloc(shape, dtype):
    return np.empty(shape, dtype)


@dataclasses.dataclass
class Workload:
    """One finalize problem, all host numpy arrays (bf16 as uint16 bits)."""
    name: str
    T: int
    K: int
    H: int
    E: int
    P: int
    tile: int
    wkind: str                       # "fp32" | "bf16" | "packed"
    routed_scale: float
    eps: float
    permuted_out: np.ndarray         # uint16 [P, H]
    idx: np.ndarray                  # int32 [T, K]
    expert_ids: np.ndarray           # int32 [T, K]
    weights_f32: np.ndarray          # float32 [T, K], the routing weights as drawn
    weights: np.ndarray              # what the finalize receives, per wkind
    shared: np.ndarray               # uint16 [T, H]
    residual: Optional[np.ndarray]   # uint16 [T, H] or None
    gamma: Optional[np.ndarray]      # uint16 [H] or None
    valid_rows: np.ndarray           # bool [P]: rows some (t, k) maps to

    @property
    def with_norm(self) -> bool:
        return self.residual is not None


# ---------------------------------------------------------------- helpers


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float array -> uint16 bf16 bit patterns (torch's CPU conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact widening)."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _fill_rows(out: np.ndarray, seed_seq: np.random.SeedSequence, kind: str,
               a: float, b: float, threads: int) -> None:
    """Fill out[R, H] (uint16 bf16 bits) chunk by chunk, one PCG64 stream per
    chunk of ROWS_PER_CHUNK rows.  kind "normal": N(a, b^2); "uniform": U(a, b)."""
    R = out.shape[0]
    n_chunks = (R + ROWS_PER_CHUNK - 1) // ROWS_PER_CHUNK
    kids = seed_seq.spawn(n_chunks)

    def work(i):
        r0, r1 = i * ROWS_PER_CHUNK, min(R, (i + 1) * ROWS_PER_CHUNK)
        rng = np.random.Generator(np.random.PCG64(kids[i]))
        shape = (r1 - r0,) + out.shape[1:]
        if kind == "normal":
            f = rng.standard_normal(shape, dtype=np.float32)
            if b != 1.0:
                f *= np.float32(b)
            if a != 0.0:
                f += np.float32(a)
        else:
            f = rng.uniform(a, b, shape).astype(np.float32)
        out[r0:r1] = to_bf16_bits(f)

    if n_chunks == 1 or threads <= 1:
        for i in range(n_chunks):
            work(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(n_chunks)))


def _routing_weights(rng: np.random.Generator, T: int, K: int, rule: str) -> np.ndarray:
    z = rng.standard_normal((T, K))
    if rule == "softmax":
        e = np.exp(z - z.max(axis=1, keepdims=True))
        w = e / e.sum(axis=1, keepdims=True)
    elif rule == "sigmoid":
        s = 1.0 / (1.0 + np.exp(-z))
        w = s / s.sum(axis=1, keepdims=True)
    else:
        raise ValueError(rule)
    return w.astype(np.float32)


def _pool_routing(rng, T, K, E, n_blocks, tile, require_all, max_tries=1000):
    """K distinct experts per token from a pool of n_blocks experts."""
    if K > n_blocks:
        raise ValueError("top_k larger than the expert pool")
    pool = np.sort(rng.choice(E, size=n_blocks, replace=False)) if n_blocks < E \
        else np.arange(E)
    for _ in range(max_tries):
        # K distinct pool positions per token: the first K of a random order
        pos = np.argsort(rng.random((T, n_blocks)), axis=1)[:, :K] if T else \
            np.zeros((0, K), np.int64)
        counts = np.bincount(pos.ravel(), minlength=n_blocks)
        if counts.max(initial=0) <= tile and (not require_all or counts.min() > 0):
            block_rows = np.full(n_blocks, tile, np.int64)
            return pool[pos].astype(np.int32), pos, block_rows
    raise RuntimeError("could not draw a routing that fits the blocks")


def _exact_count_routing(rng, T, K, counts_per_expert, tile):
    """Each expert e receives exactly counts_per_expert[e] (t, k) slots."""
    E = counts_per_expert.size
    ids = np.repeat(np.arange(E, dtype=np.int32), counts_per_expert)
    assert ids.size == T * K
    rng.shuffle(ids)
    g = ids.reshape(T, K)
    # repair repeated experts inside a token by swaps with random other slots
    for _ in range(100):
        srt = np.sort(g, axis=1)
        bad = np.nonzero((srt[:, 1:] == srt[:, :-1]).any(axis=1))[0]
        if bad.size == 0:
            break
        for t in bad:
            while True:
                row = g[t]
                vals, first = np.unique(row, return_index=True)
                dup_pos = np.setdiff1d(np.arange(K), first)
                if dup_pos.size == 0:
                    break
                j = dup_pos[0]
                u = int(rng.integers(T))
                l = int(rng.integers(K))
                if u == t:
                    continue
                a, b = row[j], g[u, l]
                if b in row or a in g[u]:
                    continue
                g[t, j], g[u, l] = b, a
    else:
        raise RuntimeError("could not repair repeated experts")
    block_rows = ((counts_per_expert + tile - 1) // tile) * tile
    return g, g.astype(np.int64), block_rows


# ---------------------------------------------------------------- builder


def synth(name: str, T: int, K: int, H: int, E: int, tile: int, *,
          P: Optional[int] = None, counts_per_expert: Optional[np.ndarray] = None,
          weight_rule: str = "softmax", wkind: str = "fp32",
          routed_scale: float = 1.0, with_norm: bool = False, eps: float = 1e-6,
          require_all: bool = True, seed: int = 0, alloc: Alloc = _np_alloc,
          threads: Optional[int] = None) -> Workload:
    """Build one seeded workload.

    Either ``P`` (pool routing over P / tile experts) or
    ``counts_per_expert`` (exact-count routing over all E experts) is given.
    ``alloc(shape, dtype)`` supplies the big arrays (e.g. pinned memory).
    """
    threads = threads or min(32, os.cpu_count() or 1)
    ss = np.random.SeedSequence(seed)
    s_route, s_w, s_x, s_shared, s_res, s_gamma = ss.spawn(6)
    rng_route = np.random.Generator(np.random.PCG64(s_route))
    rng_w = np.random.Generator(np.random.PCG64(s_w))

    if counts_per_expert is not None:
        counts_per_expert = np.asarray(counts_per_expert, np.int64)
        expert_ids, block_of_slot, block_rows = _exact_count_routing(
            rng_route, T, K, counts_per_expert, tile)
        n_blocks = E
    else:
        assert P is not None and P % tile == 0
        n_blocks = P // tile
        expert_ids, block_of_slot, block_rows = _pool_routing(
            rng_route, T, K, E, n_blocks, tile, require_all)
    block_start = np.concatenate([[0], np.cumsum(block_rows)[:-1]])
    P_total = int(block_rows.sum())
    if P is not None:
        assert P_total == P, (P_total, P)

    # rows fill each block from the front in (t, k) order
    flat = block_of_slot.ravel()
    order = np.argsort(flat, kind="stable")
    first_of_block = np.searchsorted(flat[order], np.arange(n_blocks))
    rank = np.empty(flat.size, np.int64)
    rank[order] = np.arange(flat.size) - first_of_block[flat[order]]
    idx = (block_start[flat] + rank).reshape(T, K).astype(np.int32)
    valid_rows = np.zeros(P_total, bool)
    valid_rows[idx.ravel()] = True

    weights_f32 = _routing_weights(rng_w, T, K, weight_rule)
    if wkind == "fp32":
        weights = weights_f32
    elif wkind == "bf16":
        weights = to_bf16_bits(weights_f32)
    elif wkind == "packed":
        low = to_bf16_bits(weights_f32).astype(np.uint32)
        weights = ((expert_ids.astype(np.uint32) << 16) | low).view(np.int32)
    else:
        raise ValueError(wkind)

    permuted_out = alloc((P_total, H), np.uint16)
    _fill_rows(permuted_out, s_x, "normal", 0.0, 1.0, threads)
    pad = np.nonzero(~valid_rows)[0]
    if pad.size:
        permuted_out[pad] = PAD_BITS

    shared = alloc((T, H), np.uint16)
    _fill_rows(shared, s_shared, "normal", 0.0, 1.0, threads)
    residual = gamma = None
    if with_norm:
        residual = alloc((T, H), np.uint16)
        _fill_rows(residual, s_res, "normal", 0.0, 2.0, threads)
        gamma = alloc((H,), np.uint16)
        rng_g = np.random.Generator(np.random.PCG64(s_gamma))
        gamma[:] = to_bf16_bits(rng_g.uniform(0.5, 1.5, H))

    return Workload(name=name, T=T, K=K, H=H, E=E, P=P_total, tile=tile, wkind=wkind,
                    routed_scale=float(np.float32(routed_scale)), eps=eps,
                    permuted_out=permuted_out, idx=idx, expert_ids=expert_ids,
                    weights_f32=weights_f32, weights=weights, shared=shared,
                    residual=residual, gamma=gamma, valid_rows=valid_rows)


# ------------------------------------------------------ the five workloads


def balanced_counts(T: int, K: int, E: int, seed_seq: np.random.SeedSequence) -> np.ndarray:
    """Load-balanced exact counts for T tokens x top-K over E experts: with
    base = T*K/E, 16 experts take base + base/16 slots, 16 take base - base/16
    and the rest take base (T*K must be a multiple of 16*E).  For 16384
    tokens x top-8 over 256 experts that is 16 x 544, 16 x 480, 224 x 512
    slots: 131072 slots in 1040 tiles of 128 rows = 133120 permuted rows."""
    if (T * K) % (16 * E):
        raise ValueError("T*K must be a multiple of 16*E")
    base = T * K // E
    delta = base // 16
    rng = np.random.Generator(np.random.PCG64(seed_seq))
    counts = np.full(E, base, np.int64)
    who = rng.permutation(E)
    counts[who[:16]] = base + delta
    counts[who[16:32]] = base - delta
    return counts


def prefill(T: int, alloc: Alloc = _np_alloc, threads: Optional[int] = None,
            name: Optional[str] = None) -> Workload:
    """Prefill-shaped workload with T tokens: K=8 of E=256 experts with
    balanced exact counts, blocks padded to 128 rows, H=7168, fp32
    normalised-sigmoid routing, routed scale 2.5, residual + RMSNorm."""
    counts = balanced_counts(T, 8, 256, np.random.SeedSequence([4, 1]))
    return synth(name or f"prefill_t{T}", T=T, K=8, H=7168, E=256, tile=128,
                 counts_per_expert=counts, weight_rule="sigmoid", routed_scale=2.5,
                 with_norm=True, eps=1e-6, seed=4, alloc=alloc, threads=threads)


CONFIG_NAMES = ("tiny", "decode_bs1_packed", "decode_bs256",
                "fused_norm_bs16", "prefill_t16384")


def make(name: str, alloc: Alloc = _np_alloc, threads: Optional[int] = None) -> Workload:
    """The five named workloads (seed 0 for the tiny one, 1..4 for the rest)."""
    if name == "tiny":
        return synth(name, T=4, K=2, H=64, E=8, tile=4, P=32, weight_rule="softmax",
                     routed_scale=1.0, require_all=False, seed=0, alloc=alloc,
                     threads=threads)
    if name == "decode_bs1_packed":
        return synth(name, T=1, K=8, H=7168, E=256, tile=32, P=256, weight_rule="sigmoid",
                     wkind="packed", routed_scale=2.5, seed=1, alloc=alloc, threads=threads)
    if name == "decode_bs256":
        return synth(name, T=256, K=8, H=7168, E=256, tile=128, P=6272,
                     weight_rule="sigmoid", routed_scale=2.5, seed=2, alloc=alloc,
                     threads=threads)
    if name == "fused_norm_bs16":
        return synth(name, T=16, K=8, H=7168, E=384, tile=64, P=2048, weight_rule="softmax",
                     routed_scale=1.0, with_norm=True, eps=1e-6, seed=3, alloc=alloc,
                     threads=threads)
    if name == "prefill_t16384":
        return prefill(16384, alloc=alloc, threads=threads, name=name)
    raise KeyError(name)


# ------------------------------------------------- tensor-parallel groups


@dataclasses.dataclass
class TPGroup:
    """One all-reduce-fused finalize problem: R ranks' own operands (each a
    Workload without residual) and the residual, gamma and eps they share."""
    name: str
    ranks: list
    residual: Optional[np.ndarray]   # uint16 [T, H] or None
    gamma: Optional[np.ndarray]      # uint16 [H] or None
    eps: float

    @property
    def R(self) -> int:
        return len(self.ranks)

    @property
    def with_norm(self) -> bool:
        return self.residual is not None

    def __getattr__(self, item):      # T, K, H, wkind, routed_scale: as on every rank
        if item in ("T", "K", "H", "E", "wkind", "routed_scale"):
            return getattr(self.ranks[0], item)
        raise AttributeError(item)


def tp_group(name: str, R: int, T: int, K: int, H: int, E: int, tile: int, P: int, *,
             weight_rule: str = "sigmoid", wkind: str = "fp32", routed_scale: float = 1.0,
             with_norm: bool = True, eps: float = 1e-6, seed: int = 0,
             require_all: bool = False, alloc: Alloc = _np_alloc,
             threads: Optional[int] = None) -> TPGroup:
    """R ranks of one tensor-parallel group, each with its own expert rows
    (the rank's partial of every expert output), routing and shared-expert
    partial, from seeds spawned off ``seed``; the residual ~ N(0, 4) and
    gamma ~ U(0.5, 1.5) are common to all ranks.  Pool routing as for
    ``synth`` (P rows in blocks of ``tile``)."""
    ss = np.random.SeedSequence([seed, R])
    rank_seeds = ss.spawn(R + 1)
    ranks = [synth(f"{name}_rank{r}", T=T, K=K, H=H, E=E, tile=tile, P=P,
                   weight_rule=weight_rule, wkind=wkind, routed_scale=routed_scale,
                   require_all=require_all,
                   seed=int(rank_seeds[r].generate_state(1)[0]), alloc=alloc, threads=threads)
             for r in range(R)]
    residual = gamma = None
    if with_norm:
        s_res, s_gamma = rank_seeds[R].spawn(2)
        residual = alloc((T, H), np.uint16)
        _fill_rows(residual, s_res, "normal", 0.0, 2.0, threads or 1)
        gamma = alloc((H,), np.uint16)
        rng_g = np.random.Generator(np.random.PCG64(s_gamma))
        gamma[:] = to_bf16_bits(rng_g.uniform(0.5, 1.5, H))
    return TPGroup(name=name, ranks=ranks, residual=residual, gamma=gamma, eps=eps)


# The decode shapes of the all-reduce-fused finalize: Kimi K2.5-like
# (H = 7168, top-8 of 384 experts) at batch 1 and 16, as in the
# "[Kimi K2.5] Fuse deferred MoE finalize ..." page's timings, and batch 256
# with the 6272-row permuted buffer named there.
TP_SHAPES = {1: dict(E=384, tile=32, P=256), 16: dict(E=384, tile=64, P=2048),
             256: dict(E=256, tile=128, P=6272)}


def tp_decode(R: int, T: int, with_norm: bool = True, seed: int = 5,
              alloc: Alloc = _np_alloc) -> TPGroup:
    """R ranks at decode batch T (1, 16 or 256), H = 7168, K = 8, fp32
    normalised-sigmoid routing, routed scale 2.5, residual + RMSNorm."""
    shape = TP_SHAPES[T]
    return tp_group(f"tp{R}_t{T}", R, T=T, K=8, H=7168, weight_rule="sigmoid",
                    routed_scale=2.5, with_norm=with_norm, seed=seed, alloc=alloc, **shape)
