"""The tensor-parallel orchestration of the all-reduce-fused finalize
(moe_deferred_finalize_gb300.tp) with two gloo ranks on CPU.

No GPU is involved: the transport shares numpy buffers between the two
processes through POSIX shared memory and logs event records and waits,
and the backend stands in for the two kernels (phase 1 through the fp64
oracle's finalize of the rank's own operands, rounded to fp32 as the kernel
stores its partial; phase 2 as the plain fp64 sum of the partials in rank
order, then residual + RMSNorm).  What is checked is the orchestration: the
rank-ordered tables built from the exchanged handles, the double-buffered
partials, the record / barrier / wait / reduce order of every step, the
set-up check that all ranks agree, and the outputs of three steps with
different token counts against the oracle of the whole group."""
import os
import socket
import sys
import traceback

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STEPS = (5, 2, 7)           # token counts of the three steps
MAX_T, H, K = 8, 48, 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class ShmTransport:
    """Buffers in POSIX shared memory (the handle is the segment name);
    events are log entries, since the stand-in kernels run synchronously."""

    def __init__(self, rank, log):
        self.rank, self.log, self.segments, self.n = rank, log, [], 0

    def alloc(self, shape, dtype):
        from multiprocessing import shared_memory
        assert dtype == torch.float32
        seg = shared_memory.SharedMemory(create=True, size=int(np.prod(shape)) * 4)
        self.segments.append(seg)
        arr = np.ndarray(shape, np.float32, buffer=seg.buf)
        arr[:] = np.nan
        return torch.from_numpy(arr)

    def export(self, t):
        seg = next(s for s in self.segments
                   if np.shares_memory(np.ndarray(t.shape, np.float32, buffer=s.buf), t.numpy()))
        return (seg.name, tuple(t.shape))

    def open(self, handle):
        from multiprocessing import shared_memory
        name, shape = handle
        seg = shared_memory.SharedMemory(name=name)
        self.segments.append(seg)
        return torch.from_numpy(np.ndarray(shape, np.float32, buffer=seg.buf))

    def new_event(self):
        self.n += 1
        return ("event", self.rank, self.n - 1)

    def export_event(self, ev):
        return ev

    def open_event(self, handle):
        return handle

    def stream(self, stream=None):
        return "stream"

    def record(self, ev, stream):
        self.log.append(("record", ev[1], ev[2]))

    def wait(self, ev, stream):
        self.log.append(("wait", ev[1], ev[2]))

    def synchronize(self, stream):
        self.log.append(("synchronize",))

    def close(self):
        for s in self.segments:
            s.close()


class OracleBackend:
    def __init__(self, orc, log):
        self.orc, self.log = orc, log

    def partial(self, x, wkind, scale, partial, stream):
        r = self.orc.moe_finalize(x["permuted_out"], x["idx_map"], x["weights"], wkind, scale,
                                  x["shared_out"])["out"]
        partial.numpy()[:] = r.astype(np.float32)
        self.log.append(("partial", partial.shape[0]))

    def reduce(self, partials, residual, gamma, eps, outs, stream):
        m = sum(p.numpy().astype(np.float64) for p in partials)
        s = m + residual
        g = torch.from_numpy(gamma)
        outs["out"] = m
        outs["residual_out"] = s
        outs["norm_out"] = torch.nn.functional.rms_norm(torch.from_numpy(s), (s.shape[1],),
                                                        weight=g, eps=eps).numpy()
        self.log.append(("reduce", len(partials)))


def _group():
    from moe_deferred_finalize_gb300 import workloads as W
    return [W.tp_group(f"gloo{T}", 2, T=T, K=K, H=H, E=64, tile=8, P=64, routed_scale=2.5,
                       seed=100 + T) for T in STEPS]


def _worker(rank, port, q, bad_h):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        import torch.distributed as dist
        import oracle
        from moe_deferred_finalize_gb300 import tp
        from moe_deferred_finalize_gb300.workloads import bf16_bits_to_f32
        dist.init_process_group("gloo", rank=rank, world_size=2)
        log = []
        transport = ShmTransport(rank, log)
        try:
            h = H + 8 if (bad_h and rank == 1) else H
            try:
                group = tp.TPFinalize(dist.group.WORLD, MAX_T, h, transport=transport,
                                      backend=OracleBackend(oracle.default(), log))
            except ValueError as e:
                q.put((rank, "refused", str(e)))
                return
            results = []
            for g in _group():
                wl = g.ranks[rank]
                x = {"permuted_out": wl.permuted_out, "idx_map": wl.idx, "weights": wl.weights,
                     "shared_out": wl.shared}
                outs = group.step(x, g.wkind, g.routed_scale, g.T,
                                  residual=bf16_bits_to_f32(g.residual).astype(np.float64),
                                  gamma=bf16_bits_to_f32(g.gamma).astype(np.float64),
                                  eps=g.eps)
                results.append({k: np.asarray(v) for k, v in outs.items()})
            group.close()
            assert log[-1] == ("synchronize",) and group.buffers is None
            q.put((rank, "ok", (results, log)))
        finally:
            transport.close()
            dist.destroy_process_group()
    except Exception:
        q.put((rank, "error", traceback.format_exc()))


def _run(bad_h=False):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q, bad_h)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict()
    for _ in range(2):
        rank, status, payload = q.get(timeout=300)
        got[rank] = (status, payload)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    return got


def test_two_phase_protocol_and_results_gloo(orc):
    got = _run()
    for rank in (0, 1):
        assert got[rank][0] == "ok", got[rank][1]
    groups = _group()
    for rank in (0, 1):
        results, log = got[rank][1]
        # per step: phase 1 into buffer (step % 2), record that buffer's event,
        # wait on the peer's event of the same buffer, reduce over both ranks
        peer = 1 - rank
        for s, T in enumerate(STEPS):
            b = s % 2
            assert log[4 * s:4 * s + 4] == [("partial", T), ("record", rank, b),
                                            ("wait", peer, b), ("reduce", 2)], log
        for g, res in zip(groups, results):
            ranks = [{"permuted_out": wl.permuted_out, "idx": wl.idx, "weights": wl.weights,
                      "shared": wl.shared} for wl in g.ranks]
            ref = orc.moe_finalize_ar(ranks, g.wkind, g.routed_scale, g.residual, g.gamma,
                                      g.eps)
            for key in ref:
                # the only rounding is the fp32 store of each rank's partial
                assert np.allclose(res[key], ref[key], rtol=1e-6, atol=1e-6), (g.name, key)
    # both ranks hold the same outputs: the partials were summed in rank order
    for a, b in zip(got[0][1][0], got[1][1][0]):
        for key in a:
            assert np.array_equal(a[key], b[key]), key


def test_ranks_that_disagree_are_refused_on_every_rank():
    got = _run(bad_h=True)
    for rank in (0, 1):
        status, msg = got[rank]
        assert status == "refused", msg
        assert "every rank must agree" in msg
