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
        self.rank, self.log, self.segments, self.created, self.n = rank, log, [], [], 0

    # bf16 buffers hold raw bit patterns here
    NP = {torch.float32: np.float32, torch.int32: np.int32, torch.bfloat16: np.uint16}

    def alloc(self, shape, dtype):
        from multiprocessing import shared_memory
        nd = np.dtype(self.NP[dtype])
        seg = shared_memory.SharedMemory(create=True, size=int(np.prod(shape)) * nd.itemsize)
        self.segments.append(seg)
        self.created.append(seg)
        arr = np.ndarray(shape, nd, buffer=seg.buf)
        arr[:] = 0
        return torch.from_numpy(arr)

    def export(self, t):
        a = t.numpy()
        seg = next(s for s in self.segments
                   if np.shares_memory(np.ndarray(s.size, np.uint8, buffer=s.buf), a))
        return (seg.name, tuple(t.shape), a.dtype.str)

    def open(self, handle):
        from multiprocessing import shared_memory
        name, shape, dt = handle
        seg = shared_memory.SharedMemory(name=name)
        self.segments.append(seg)
        return torch.from_numpy(np.ndarray(shape, np.dtype(dt), buffer=seg.buf))

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
        """Called after the group's closing barrier: no peer maps a segment
        any more, so the creator may remove it."""
        for s in self.segments:
            s.close()
        for s in self.created:
            s.unlink()


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

    def one_shot(self, ranks, wkind, scale, residual, gamma, eps, outs, stream):
        rk = [{"permuted_out": r["permuted_out"].numpy(), "idx": r["idx_map"].numpy(),
               "weights": r["weights"].numpy(), "shared": r["shared_out"].numpy()}
              for r in ranks]
        outs.update(self.orc.moe_finalize_ar(rk, wkind, scale, residual, gamma, eps))
        self.log.append(("one_shot", len(ranks)))


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
            log_two_phase = list(log)
            # the one-shot form: every rank fills its shared input set, then one
            # launch per rank reads all of them
            del log[:]
            g0 = _group()[0]
            one = tp.TPFinalize(dist.group.WORLD, MAX_T, H, transport=transport,
                                backend=OracleBackend(oracle.default(), log),
                                one_shot=(g0.ranks[0].P, K, "fp32"))
            shots = []
            for g in _group():
                wl = g.ranks[rank]
                x = one.inputs()
                x["permuted_out"].numpy()[:] = wl.permuted_out
                x["idx_map"].numpy()[:g.T] = wl.idx
                x["weights"].numpy()[:g.T] = wl.weights
                x["shared_out"].numpy()[:g.T] = wl.shared
                shots.append(one.step_one_shot(g.T, routed_scale=g.routed_scale,
                                               residual=g.residual, gamma=g.gamma, eps=g.eps))
            one.close()
            q.put((rank, "ok", (results, log_two_phase, shots, list(log))))
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
        results, log, shots, log_one = got[rank][1]
        # one-shot steps: record this step's event, wait on the peer's, one launch
        # (the one-shot group's events are the transport's third and fourth)
        for s, T in enumerate(STEPS):
            b = 2 + s % 2
            assert log_one[3 * s:3 * s + 3] == [("record", rank, b), ("wait", 1 - rank, b),
                                                ("one_shot", 2)], log_one
        for g, res in zip(_group(), shots):
            ranks = [{"permuted_out": wl.permuted_out, "idx": wl.idx, "weights": wl.weights,
                      "shared": wl.shared} for wl in g.ranks]
            ref = orc.moe_finalize_ar(ranks, g.wkind, g.routed_scale, g.residual, g.gamma,
                                      g.eps)
            for key in ref:
                # the stand-in launch is the oracle over the shared input sets
                assert np.array_equal(res[key], ref[key]), (g.name, key)
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
