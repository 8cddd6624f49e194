"""Host orchestration of the all-reduce-fused finalize across the processes
of one tensor-parallel group, one GPU per process ("[Kimi K2.5] Fuse
deferred MoE finalize into next-layer AR + residual + RMSNorm", Summary and
Numerics & speed: the finalize of every rank summed over the group, then
residual + RMSNorm, within one NVLink domain).

Only the two-phase form needs orchestration across processes; every step of
the arithmetic runs in the library's kernels (moe_finalize_partial and
moe_finalize_allreduce_reduce).  Each rank owns two fp32 partial buffers
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


class TPFinalize:
    """The two-phase all-reduce-fused finalize of one rank of a
    tensor-parallel group (see the module docstring for the protocol).

    group: the torch.distributed process group of the R ranks (any backend;
    it carries only set-up objects and the per-step host barrier).
    max_tokens, H: the largest T of any step and the hidden size; every rank
    must pass the same values (checked at set-up, on every rank)."""

    def __init__(self, group, max_tokens: int, H: int, transport=None, backend=None,
                 device=None):
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

        mine = {"rank": self.rank, "max_tokens": self.max_tokens, "H": self.H}
        configs = [None] * self.world
        dist.all_gather_object(configs, mine, group=group)
        for r, c in enumerate(configs):
            if c["rank"] != r or (c["max_tokens"], c["H"]) != (self.max_tokens, self.H):
                raise ValueError(f"rank {r} set up with max_tokens={c['max_tokens']}, "
                                 f"H={c['H']}; rank {self.rank} with {self.max_tokens}, "
                                 f"{self.H}: every rank must agree")

        self.local = [self.transport.alloc((self.max_tokens, self.H), torch.float32)
                      for _ in range(2)]
        self.events = [self.transport.new_event() for _ in range(2)]
        # a one-rank group shares nothing (an exported buffer that no peer
        # opens would stay registered for sharing until the process exits)
        handles = None
        if self.world > 1:
            handles = {"buffers": [self.transport.export(b) for b in self.local],
                       "events": [self.transport.export_event(e) for e in self.events]}
        everyone = [None] * self.world
        dist.all_gather_object(everyone, handles, group=group)
        # rank-ordered tables: the local objects for this rank, opened peers' otherwise
        self.buffers = [[self.local[b] if r == self.rank else self.transport.open(h["buffers"][b])
                         for r, h in enumerate(everyone)] for b in range(2)]
        self.peer_events = [[None if r == self.rank else self.transport.open_event(h["events"][b])
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

    def close(self, stream=None):
        """Release the peers' buffers and events this rank opened, once its
        work on them is done, then wait at a barrier until every rank has:
        no rank frees a buffer while a peer still maps it.  Call on every
        rank before the process exits; the object is unusable afterwards."""
        self.transport.synchronize(self.transport.stream(stream))
        self.buffers = self.peer_events = None
        dist.barrier(group=self.group)
