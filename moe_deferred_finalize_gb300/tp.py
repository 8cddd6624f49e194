"""Host orchestration of the all-reduce-fused finalize across the processes
of one tensor-parallel group, one GPU per process ("[Kimi K2.5] Fuse
deferred MoE finalize into next-layer AR + residual + RMSNorm", Summary and
Numerics & speed: the finalize of every rank summed over the group, then
residual + RMSNorm, within one NVLink domain).

Every step of the arithmetic runs in the library's kernels
(moe_finalize_partial and moe_finalize_allreduce_reduce for the two-phase
form, moe_finalize_allreduce for the one-shot).  Each rank owns two fp32
partial buffers
[max_tokens, H] (double-buffered by step parity) and one interprocess event
per buffer; at set-up the ranks exchange handles to them over a
torch.distributed process group and open their peers'.  One step on rank r:

  1. phase 1 into its partial buffer b = step % 2, on its stream;
  2. record its event b on that stream;
  3. a host barrier over the group: every rank has recorded event b of this
     step, so the waits below cannot see an older record;
  4. its stream waits on every peer's event b (ordering on the GPUs; no
     thread of any kernel waits on another device);
  5. phase 2 over the R partial buffers b in rank order.

Double buffering makes the reuse of a buffer safe: a rank writes buffer b
again only in step s + 2, after its own phase 2 of step s + 1, which waited
on every peer's event of step s + 1, recorded after the peer's phase 2 of
step s finished reading buffer b.

The one-shot form is orchestrated the same way when the group is set up
with ``one_shot=(P, K, wkind)``: each rank then also owns two sets of input
buffers (permuted_out [P, H], idx_map and weights [max_tokens, K],
shared_out [max_tokens, H]), shared with the peers.  A step fills this
rank's set b (``inputs()``) on its stream, records event b, meets the host
barrier, waits on every peer's event b and launches one
moe_finalize_allreduce over the R sets b.  A set is rewritten two steps
later only, after the peers' launches that read it (same argument).

Cross-device plumbing goes through a transport (buffers, events, IPC
handles); ``CudaTransport`` uses torch's CUDA IPC (shared tensors and
interprocess events).  The kernels go through a backend; ``LibraryBackend``
calls the library.  Both are parameters so that the protocol can be run
with stand-ins where no GPU is present.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import _abi


class CudaTransport:
    """Buffers and events shared between processes through CUDA IPC: torch's
    tensor sharing (the allocation's IPC handle plus the offset) and
    interprocess CUDA events."""

    def __init__(self, device):
        self.device = torch.device(device)

    def alloc(self, shape, dtype):
        return torch.empty(shape, dtype=dtype, device=self.device)

    def export(self, t):
        from torch.multiprocessing.reductions import reduce_tensor
        return reduce_tensor(t)

    def open(self, handle):
        rebuild, args = handle
        return rebuild(*args)

    def new_event(self):
        return torch.cuda.Event(interprocess=True)

    def export_event(self, ev):
        return ev.ipc_handle()

    def open_event(self, handle):
        return torch.cuda.Event.from_ipc_handle(self.device, handle)

    def stream(self, stream=None):
        return stream if stream is not None else torch.cuda.current_stream(self.device)

    def record(self, ev, stream):
        ev.record(stream)

    def wait(self, ev, stream):
        stream.wait_event(ev)

    def synchronize(self, stream):
        stream.synchronize()


class LibraryBackend:
    """The two phases as the library's kernels."""

    def partial(self, rank_inputs, wkind, routed_scale, partial, stream):
        x = rank_inputs
        _abi.moe_finalize_partial(x["permuted_out"], x["idx_map"], x["weights"], wkind,
                                  x["shared_out"], routed_scale=routed_scale, partial=partial,
                                  stream=stream)

    def reduce(self, partials, residual, gamma, eps, outs, stream):
        _abi.moe_finalize_allreduce_reduce(partials, residual=residual, gamma=gamma, eps=eps,
                                           stream=stream, **outs)

    def one_shot(self, ranks, wkind, routed_scale, residual, gamma, eps, outs, stream):
        _abi.moe_finalize_allreduce(ranks, wkind, routed_scale=routed_scale, residual=residual,
                                    gamma=gamma, eps=eps, stream=stream, **outs)


class TPFinalize:
    """The all-reduce-fused finalize of one rank of a tensor-parallel group,
    two-phase (``step``) or, when set up with ``one_shot``, one-shot
    (``step_one_shot``); see the module docstring for the protocol.

    group: the torch.distributed process group of the R ranks (any backend;
    it carries only set-up objects and the per-step host barrier).
    max_tokens, H: the largest T of any step and the hidden size; one_shot:
    (P, K, wkind) of the shared input sets, or None.  Every rank must pass
    the same values (checked at set-up, on every rank)."""

    def __init__(self, group, max_tokens: int, H: int, transport=None, backend=None,
                 device=None, one_shot=None):
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        if not 1 <= self.world <= _abi.MAX_RANKS:
            raise ValueError(f"a group of 1 to {_abi.MAX_RANKS} ranks, not {self.world}")
        self.max_tokens, self.H = int(max_tokens), int(H)
        self.transport = transport or CudaTransport(device if device is not None
                                                    else torch.cuda.current_device())
        self.backend = backend or LibraryBackend()
        self.step_index = 0

        self.one_shot = None if one_shot is None else (int(one_shot[0]), int(one_shot[1]),
                                                         str(one_shot[2]))
        mine = {"rank": self.rank, "max_tokens": self.max_tokens, "H": self.H,
                "one_shot": self.one_shot}
        configs = [None] * self.world
        dist.all_gather_object(configs, mine, group=group)
        for r, c in enumerate(configs):
            if c["rank"] != r or (c["max_tokens"], c["H"], c["one_shot"]) != \
                    (self.max_tokens, self.H, self.one_shot):
                raise ValueError(f"rank {r} set up with max_tokens={c['max_tokens']}, "
                                 f"H={c['H']}, one_shot={c['one_shot']}; rank {self.rank} with "
                                 f"{self.max_tokens}, {self.H}, {self.one_shot}: every rank "
                                 f"must agree")

        self.local = [self.transport.alloc((self.max_tokens, self.H), torch.float32)
                      for _ in range(2)]
        self.events = [self.transport.new_event() for _ in range(2)]
        self.local_inputs = None
        if self.one_shot is not None:
            P, K, wkind = self.one_shot
            wdtype = {"fp32": torch.float32, "bf16": torch.bfloat16,
                      "packed": torch.int32}[wkind]
            self.local_inputs = [
                {"permuted_out": self.transport.alloc((P, self.H), torch.bfloat16),
                 "idx_map": self.transport.alloc((self.max_tokens, K), torch.int32),
                 "weights": self.transport.alloc((self.max_tokens, K), wdtype),
                 "shared_out": self.transport.alloc((self.max_tokens, self.H), torch.bfloat16)}
                for _ in range(2)]
        # a one-rank group shares nothing (an exported buffer that no peer
        # opens would stay registered for sharing until the process exits)
        handles = None
        if self.world > 1:
            handles = {"buffers": [self.transport.export(b) for b in self.local],
                       "events": [self.transport.export_event(e) for e in self.events],
                       "inputs": None if self.local_inputs is None else
                       [{k: self.transport.export(t) for k, t in d.items()}
                        for d in self.local_inputs]}
        everyone = [None] * self.world
        dist.all_gather_object(everyone, handles, group=group)
        # rank-ordered tables: the local objects for this rank, opened peers' otherwise
        self.buffers = [[self.local[b] if r == self.rank else self.transport.open(h["buffers"][b])
                         for r, h in enumerate(everyone)] for b in range(2)]
        self.peer_events = [[None if r == self.rank else self.transport.open_event(h["events"][b])
                             for r, h in enumerate(everyone)] for b in range(2)]
        self.inputs_table = None
        if self.one_shot is not None:
            self.inputs_table = [
                [self.local_inputs[b] if r == self.rank else
                 {k: self.transport.open(v) for k, v in h["inputs"][b].items()}
                 for r, h in enumerate(everyone)] for b in range(2)]

    def step(self, rank_inputs: dict, wkind: str, routed_scale: float, T: int, *,
             residual=None, gamma=None, eps: float = 1e-6, outs: Optional[dict] = None,
             stream=None) -> dict:
        """One all-reduce-fused finalize over the group for T tokens (T at
        most max_tokens).  rank_inputs: this rank's "permuted_out",
        "idx_map", "weights", "shared_out".  outs: "out", "residual_out",
        "norm_out" as moe_finalize_allreduce_reduce takes them.  Every rank
        must call step() in the same order; it blocks on the host only for
        the barrier of item 3."""
        if not 0 < T <= self.max_tokens:
            raise ValueError(f"T={T} outside 1..{self.max_tokens}")
        b = self.step_index % 2
        s = self.transport.stream(stream)
        self.backend.partial(rank_inputs, wkind, routed_scale, self.local[b][:T], s)
        self.transport.record(self.events[b], s)
        dist.barrier(group=self.group)
        for r in range(self.world):
            if r != self.rank:
                self.transport.wait(self.peer_events[b][r], s)
        views = [buf[:T] for buf in self.buffers[b]]
        outs = dict(outs or {})
        self.backend.reduce(views, residual, gamma, eps, outs, s)
        self.step_index += 1
        return outs

    def inputs(self) -> dict:
        """This rank's input buffers for the next one-shot step: fill
        "permuted_out" [P, H] and the first T rows of "idx_map",
        "weights" and "shared_out" (on the stream the step will run on)."""
        if self.local_inputs is None:
            raise RuntimeError("set up with one_shot=(P, K, wkind) for the one-shot form")
        return self.local_inputs[self.step_index % 2]

    def step_one_shot(self, T: int, *, routed_scale: float = 1.0, residual=None, gamma=None,
                      eps: float = 1e-6, outs: Optional[dict] = None, stream=None) -> dict:
        """One all-reduce-fused finalize over the group for T tokens in one
        launch per rank, reading every rank's input set of this step (filled
        through ``inputs()``).  Every rank must call it in the same order as
        its other steps."""
        if self.inputs_table is None:
            raise RuntimeError("set up with one_shot=(P, K, wkind) for the one-shot form")
        if not 0 < T <= self.max_tokens:
            raise ValueError(f"T={T} outside 1..{self.max_tokens}")
        b = self.step_index % 2
        s = self.transport.stream(stream)
        self.transport.record(self.events[b], s)
        dist.barrier(group=self.group)
        for r in range(self.world):
            if r != self.rank:
                self.transport.wait(self.peer_events[b][r], s)
        ranks = [{"permuted_out": d["permuted_out"], "idx_map": d["idx_map"][:T],
                  "weights": d["weights"][:T], "shared_out": d["shared_out"][:T]}
                 for d in self.inputs_table[b]]
        outs = dict(outs or {})
        self.backend.one_shot(ranks, self.one_shot[2], routed_scale, residual, gamma, eps, outs, s)
        self.step_index += 1
        return outs

    def close(self, stream=None):
        """Release the peers' buffers and events this rank opened, once its
        work on them is done, then wait at a barrier until every rank has:
        no rank frees a buffer while a peer still maps it.  Call on every
        rank before the process exits; the object is unusable afterwards."""
        self.transport.synchronize(self.transport.stream(stream))
        self.buffers = self.peer_events = self.inputs_table = None
        dist.barrier(group=self.group)
