"""Benchmark of the deferred MoE finalize (one JSON line on stdout).

Headline: HBM GB/s of one finalize step at T=16384, K=8, H=7168 with
residual add + RMSNorm (residual_out and norm_out emitted, out not written),
inputs resident in HBM.  Algorithmic bytes per step = gathered rows
(T*K*H*2) + shared and residual read + residual_out and norm_out written
(4*T*H*2) + gamma (H*2) + idx and fp32 weights (T*K*8).

Also reported on the same line:
  * decode latency, microseconds per call at T=1 (packed routing) and
    T=256 (fp32 routing), each call on inputs no earlier call touched
    (rotating copies larger than L2), timed as CUDA-graph replays and as
    back-to-back eager calls;
  * roofline of the finalize kernel against the measured HBM copy peak;
  * e2e: the same GB/s with inputs and outputs in pinned host memory,
    through the host-buffer call (the kernel reads and writes host memory in
    place over the host link); e2e_copy: the same with H2D copies of the
    inputs and D2H copies of the results around a device-buffer call;
  * cpu_baseline: the fp64 CPU oracle on the host cores (test
    infrastructure, timed only here);
  * SM clocks and throttle reasons sampled during the timed region.

``--impl reference`` times the fp64 CPU oracle on the same workload
(bounded token samples per step) and prints the same line shape.

Multi-GPU: every rank runs its own full-size problem (the finalize is
token-local, no data exchange); the job value is the bytes of all ranks
over the slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_deferred_finalize_gb300 import workloads as W  # noqa: E402

WORKLOAD = "prefill_t16384"
METRIC = "finalize µs/call at T=1,256; HBM GB/s (% of peak) at T=16384, H=7168"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRCS = [os.path.join(ROOT, "moe_deferred_finalize_gb300", "csrc", f)
               for f in ("finalize.cu", "vec.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


# ------------------------------------------------------------------ helpers


def algorithmic_bytes(T, K, H, wbytes, norm, write_out):
    """Bytes the finalize must move: every gathered valid row once, every
    dense [T, H] operand once, gamma once, the row map and weights once."""
    dense = 1 + (1 if write_out else 0) + (3 if norm else 0)   # shared, out, residual, r_out, n_out
    return T * K * H * 2 + dense * T * H * 2 + (H * 2 if norm else 0) + T * K * (4 + wbytes)


def workload_bytes(wl, write_out):
    wbytes = {"fp32": 4, "bf16": 2, "packed": 4}[wl.wkind]
    return algorithmic_bytes(wl.T, wl.K, wl.H, wbytes, wl.with_norm, write_out)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_code_digest():
    """SHA-256 of the kernel sources with comments and whitespace removed:
    it changes with the code, not with its comments."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SRCS:
        text = open(f).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()


def recorded_traffic():
    """ncu DRAM bytes per launch recorded for the current kernel code, else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("kernel_code_sha256") != kernel_code_digest() or d.get("workload") != WORKLOAD:
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 10 ms with
    timestamps; only the samples inside the timed window are summarised
    (the nearest one after the window opened when the window is shorter
    than the sampling period)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def mark(self, t0, t1):
        """The timed window, in host wall-clock seconds."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        import datetime
        samples = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        t0, t1 = self.window or (samples[0][0], samples[-1][0])
        inside = [x for x in samples if t0 <= x[0] <= t1]
        in_window = len(inside)
        if not inside:
            after = [x for x in samples if x[0] >= t0]
            inside = after[:1] or samples[-1:]
        reasons = sorted({n for x in inside for n, v in zip(self.REASONS, x[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside), "samples": len(inside),
                "samples_in_window": in_window, "window_ms": round(1e3 * (t1 - t0), 1),
                "reasons": reasons}


def pinned_alloc(shape, dtype):
    tdt = {np.dtype(np.uint16): torch.int16, np.dtype(np.int32): torch.int32,
           np.dtype(np.float32): torch.float32}[np.dtype(dtype)]
    t = torch.empty(shape, dtype=tdt, pin_memory=True)
    a = t.numpy()
    return a.view(np.uint16) if np.dtype(dtype) == np.uint16 else a


def host_tensor(a):
    """torch view (no copy) of a numpy array; bf16 bits become bfloat16."""
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return t


# --------------------------------------------------------- GPU measurement


def device_inputs(wl, device):
    d = {"x": host_tensor(wl.permuted_out).to(device),
         "idx": host_tensor(wl.idx).to(device),
         "w": host_tensor(np.ascontiguousarray(wl.weights)).to(device),
         "shared": host_tensor(wl.shared).to(device)}
    if wl.with_norm:
        d["residual"] = host_tensor(wl.residual).to(device)
        d["gamma"] = host_tensor(wl.gamma).to(device)
    return d


def call(mf, wl, d, outs, stream=None, routing_ready=False, pdl=True):
    mf.moe_finalize(d["x"], d["idx"], d["w"], wl.wkind, d["shared"],
                    routed_scale=wl.routed_scale, residual=d.get("residual"),
                    gamma=d.get("gamma"), eps=wl.eps, out=outs.get("out"),
                    residual_out=outs.get("residual_out"), norm_out=outs.get("norm_out"),
                    write_out="out" in outs, routing_ready=routing_ready, pdl=pdl,
                    stream=stream)


def graph_us(fn, device, calls, n_pass, reps=5):
    """µs per call of ``fn`` (which enqueues ``calls`` calls) captured once in
    a CUDA graph and replayed ``n_pass`` times per repetition; median of
    ``reps`` repetitions timed with CUDA events on the replaying stream."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    cur = torch.cuda.current_stream(device)
    cur.wait_stream(s)
    g.replay()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    samples = []
    for _ in range(reps):
        a.record(cur)
        for _ in range(n_pass):
            g.replay()
        b.record(cur)
        torch.cuda.synchronize(device)
        samples.append(a.elapsed_time(b) * 1e3 / (n_pass * calls))
    del g
    return statistics.median(samples)


def time_headline(mf, wl, d, outs, steps, warmup, ws, device):
    """The timed steps: ``warmup`` untimed calls, then ``steps`` back-to-back
    calls between a barrier and a synchronize on each side.  Returns (total
    ms from the first step's start event to the last step's end event,
    per-step ms, host wall-clock window)."""
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        call(mf, wl, d, outs)
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(ws)
    torch.cuda.synchronize(device)
    t0 = time.time()
    for a, b in ev:
        a.record(stream)
        call(mf, wl, d, outs)
        b.record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    barrier(ws)
    per = [a.elapsed_time(b) for a, b in ev]
    total_ms = ev[0][0].elapsed_time(ev[-1][1])
    return total_ms, per, (t0, t1)


def time_roofline(mf, wl, d, outs, device, min_seconds):
    """Per-launch CUDA-event durations of back-to-back headline launches on
    the launching stream, for at least ``min_seconds`` of GPU time (so that
    the clock sampler sees many samples whatever --steps is).  Returns
    (durations in ms, host wall-clock window)."""
    stream = torch.cuda.current_stream(device)
    probe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(10)]
    for a, b in probe:
        a.record(stream)
        call(mf, wl, d, outs)
        b.record(stream)
    torch.cuda.synchronize(device)
    est_ms = statistics.median(a.elapsed_time(b) for a, b in probe)
    n = int(max(200, np.ceil(min_seconds * 1e3 / max(est_ms, 1e-3))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    torch.cuda.synchronize(device)
    t0 = time.time()
    for a, b in ev:
        a.record(stream)
        call(mf, wl, d, outs)
        b.record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    return [a.elapsed_time(b) for a, b in ev], (t0, t1)


def decode_latency(mf, name, device, reps, peak, producer=False, sequential=False):
    """µs per call on inputs rotated through copies whose total exceeds L2.

    With ``producer``: also the µs the finalize adds behind a kernel that
    writes its row buffer, as in an MoE layer where the expert GEMM has just
    written permuted_out: (producer + finalize) - (producer alone) per call,
    both as CUDA-graph replays, with the finalize launched as a programmatic
    dependent (the default), as a plain stream-ordered kernel, and with
    MOEF_FLAG_ROUTING_READY.

    With ``sequential``: also the same calls with a row map that reads
    consecutive rows (t * K + k) instead of each token's expert rows, which
    isolates what the gather itself costs."""
    wl = W.make(name)
    d = device_inputs(wl, device)
    norm = wl.with_norm
    touched = workload_bytes(wl, True)
    R = max(2, int(np.ceil(2 * L2_BYTES / touched)))
    R = min(R, 2048)

    def rep(t):   # R copies at distinct addresses
        return t.unsqueeze(0).expand(R, *t.shape).contiguous()

    xs, shs = rep(d["x"]), rep(d["shared"])
    rss = rep(d["residual"]) if norm else None
    outs = {k: torch.empty((R, wl.T, wl.H), dtype=torch.bfloat16, device=device)
            for k in (("out", "residual_out", "norm_out") if norm else ("out",))}
    sets = []
    for r in range(R):
        dd = {"x": xs[r], "idx": d["idx"], "w": d["w"], "shared": shs[r]}
        if norm:
            dd["residual"], dd["gamma"] = rss[r], d["gamma"]
        sets.append((dd, {k: v[r] for k, v in outs.items()}))
    bound = [mf.bind(dd["x"], dd["idx"], dd["w"], wl.wkind, dd["shared"],
                     routed_scale=wl.routed_scale, residual=dd.get("residual"),
                     gamma=dd.get("gamma"), eps=wl.eps, **oo) for dd, oo in sets]
    ws = torch.empty(mf.unfused_workspace_bytes(wl.T, wl.H), dtype=torch.uint8, device=device)

    def one_pass():
        for dd, oo in sets:
            call(mf, wl, dd, oo)

    def one_pass_bound():
        for f in bound:
            f()

    def one_pass_ready():     # idx/weights are not written inside the loop
        for dd, oo in sets:
            call(mf, wl, dd, oo, routing_ready=True)

    def one_pass_warm():      # the same inputs every call: rows stay in L2, as right
        dd, oo = sets[0]      # after the expert GEMM that wrote them
        for _ in range(R):
            call(mf, wl, dd, oo)

    def one_pass_unfused():
        for dd, oo in sets:
            mf.moe_finalize_unfused(dd["x"], dd["idx"], dd["w"], wl.wkind, dd["shared"],
                                    routed_scale=wl.routed_scale, residual=dd.get("residual"),
                                    gamma=dd.get("gamma"), eps=wl.eps, workspace=ws, **oo)

    one_pass()
    one_pass_bound()
    one_pass_unfused()
    torch.cuda.synchronize(device)
    n_pass = max(1, reps // R)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def eager(fn):
        samples = []
        for _ in range(5):
            a.record()
            for _ in range(n_pass):
                fn()
            b.record()
            torch.cuda.synchronize(device)
            samples.append(a.elapsed_time(b) * 1e3 / (n_pass * R))
        return statistics.median(samples)

    def graph(fn):
        return graph_us(fn, device, R, n_pass)

    eager_checked_us = eager(one_pass)      # argument checks on every call
    eager_us = eager(one_pass_bound)        # checked once, then raw C-ABI calls
    graph_us_ = graph(one_pass)
    ready_us = graph(one_pass_ready)
    unfused_us = graph(one_pass_unfused)
    warm_us = graph(one_pass_warm)
    res = {"T": wl.T, "K": wl.K, "H": wl.H, "routing": wl.wkind, "rmsnorm": norm,
           "us_per_call_graph": round(graph_us_, 3), "us_per_call_eager": round(eager_us, 3),
           "us_per_call_eager_checked": round(eager_checked_us, 3),
           "us_per_call_graph_routing_ready": round(ready_us, 3),
           "unfused_us_per_call_graph": round(unfused_us, 3),
           "us_per_call_graph_rows_in_l2": round(warm_us, 3),
           "bytes_per_call": touched,
           "GBps_graph": round(touched / (graph_us_ * 1e-6) / 1e9, 1),
           "frac": round(touched / (graph_us_ * 1e-6) / 1e9 / peak, 4),
           "us_bytes_at_peak": round(touched / (peak * 1e9) * 1e6, 3),
           "copies": R, "calls": n_pass * R,
           "plan": mf.plan(wl.T, wl.K, wl.H, norm, True,
                           torch.cuda.get_device_properties(device).multi_processor_count)}

    if sequential:
        seq = torch.arange(wl.T * wl.K, dtype=torch.int32, device=device).view(wl.T, wl.K)
        assert wl.T * wl.K <= wl.P

        def one_pass_seq():
            for dd, oo in sets:
                call(mf, wl, {**dd, "idx": seq}, oo)

        res["us_per_call_graph_sequential_rows"] = round(graph(one_pass_seq), 3)
        del seq

    if producer:
        # Two producers rewrite each copy's row buffer [P, H] just before its
        # call, reading a source buffer of the same size:
        #  * a plain elementwise kernel, which never signals its dependents
        #    early (griddepcontrol.launch_dependents), like most library
        #    kernels (not a copy: a copy would be captured as a memcpy node);
        #  * a kernel that does signal them after its loads, as a producer
        #    written for programmatic dependent launch would: this library's
        #    finalize with K = 1 and zero weights, so that out = the source.
        src = d["x"].clone()
        zero_idx = torch.zeros((wl.P, 1), dtype=torch.int32, device=device)
        zero_w = torch.zeros((wl.P, 1), dtype=torch.float32, device=device)

        def plain(dd):
            torch.mul(src, 1.0, out=dd["x"])

        def pdl_aware(dd):
            mf.moe_finalize(src[:1], zero_idx, zero_w, "fp32", src, out=dd["x"])

        def prod(kind):
            def f():
                for dd, _ in sets:
                    kind(dd)
            return f

        def prod_then(kind, **kw):
            def f():
                for dd, oo in sets:
                    kind(dd)
                    call(mf, wl, dd, oo, **kw)
            return f

        res["us_added_after_producer"] = {}
        res["producer_us_per_call_graph"] = {}
        for name, kind in (("plain_kernel", plain), ("pdl_aware_kernel", pdl_aware)):
            alone = graph(prod(kind))
            added = {"pdl": graph(prod_then(kind)) - alone,
                     "no_pdl": graph(prod_then(kind, pdl=False)) - alone,
                     "routing_ready": graph(prod_then(kind, routing_ready=True)) - alone}
            res["producer_us_per_call_graph"][name] = round(alone, 3)
            res["us_added_after_producer"][name] = {k: round(v, 3) for k, v in added.items()}
        res["producer"] = (f"a kernel writing the whole [{wl.P}, {wl.H}] bf16 row buffer "
                           f"({wl.P * wl.H * 2} bytes) from a source of the same size just "
                           f"before each call; plain_kernel: torch elementwise multiply by 1; "
                           f"pdl_aware_kernel: moe_finalize with K=1 and zero weights "
                           f"(out = shared = the source), which signals its dependents after "
                           f"its loads")
        del src, zero_idx, zero_w
    del xs, shs, rss, outs, bound, ws
    return res


def gate_latency(mf, device, T, E=256, K=8, calls=2000):
    """µs per top-K gate call (logits -> ids, fp32 weights, packed words),
    CUDA-graph replay over rotating logits copies larger than L2 when they fit."""
    per = T * E * 4
    R = int(min(max(2, np.ceil(2 * L2_BYTES / per)), 4096))
    g_ = torch.Generator(device=device).manual_seed(T)
    z = torch.randn((R, T, E), generator=g_, device=device, dtype=torch.float32)
    outs = [(torch.empty((T, K), dtype=torch.int32, device=device),
             torch.empty((T, K), dtype=torch.float32, device=device),
             torch.empty((T, K), dtype=torch.int32, device=device)) for _ in range(R)]
    lib = mf.lib()
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    args = [(P(z[r]), P(outs[r][0]), P(outs[r][1]), P(outs[r][2])) for r in range(R)]

    def one_pass(stream):
        sv = ctypes.c_void_p(stream.cuda_stream)
        for a_ in args:
            st = lib.moe_topk_route(a_[0], T, E, K, 1, a_[1], a_[2], a_[3], sv)
            if st != 0:
                raise RuntimeError(f"moe_topk_route status {st}")

    cur = torch.cuda.current_stream(device)
    one_pass(cur)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(cur)
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            one_pass(s)
    cur.wait_stream(s)
    g.replay()
    torch.cuda.synchronize(device)
    n_pass = max(1, calls // R)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    samples = []
    for _ in range(3):
        a.record()
        for _ in range(n_pass):
            g.replay()
        b.record()
        torch.cuda.synchronize(device)
        samples.append(a.elapsed_time(b) * 1e3 / (n_pass * R))
    del g, z, outs
    return round(statistics.median(samples), 3)


def allreduce_bytes(R, T, K, H, wbytes=4):
    """Algorithmic bytes of one one-shot all-reduce-fused call that writes
    residual_out and norm_out: every rank's gathered rows, shared output and
    routing once, the residual once, the two outputs, gamma."""
    return R * (T * K * H * 2 + T * H * 2 + T * K * (4 + wbytes)) + 3 * T * H * 2 + H * 2


def allreduce_copies(R, T, K, H):
    """Buffer copies the all-reduce entry rotates over: (C, Cr, bytes).  C
    copies of every rank's operands for the one-shot; Cr copies of one
    rank's operands, the R partials, residual and outputs for phase 1,
    phase 2 and the plain finalize, as many as the smaller of phase 1's and
    phase 2's working sets needs to exceed twice the L2 (capped at 4096).
    bytes: the one-shot's, phase 1's and phase 2's algorithmic bytes."""
    nbytes = allreduce_bytes(R, T, K, H)
    p1_bytes = T * K * H * 2 + T * H * 2 + T * K * 8 + T * H * 4
    p2_bytes = R * T * H * 4 + 3 * T * H * 2 + H * 2

    def n_copies(b):
        return int(min(max(2, np.ceil(2 * L2_BYTES / b)), 4096))

    return n_copies(nbytes), n_copies(min(p1_bytes, p2_bytes)), (nbytes, p1_bytes, p2_bytes)


def allreduce_latency(mf, device, R, T, peak, calls=1000):
    """µs per call of the all-reduce-fused finalize at decode size T over R
    ranks' buffer sets on this one GPU (CUDA-graph replay; every call on
    buffer copies no other call in the pass touched, the copies a timed
    call rotates over together at least twice the L2):

      * one-shot: one launch reading every rank's rows (what each rank
        would run, with the peers' rows read over NVLink instead of HBM);
      * two-phase, one rank: phase 1 for its own partial, then phase 2 over
        all R partials (the other R - 1 already in place);
      * phase 1 and phase 2 alone;
      * the plain finalize of one rank's operands with residual + RMSNorm,
        for comparison with R of them.

    The one-shot rotates over copies of every rank's operands; the other
    calls touch far fewer bytes and rotate over copies of their own (rank
    0's operands, the R partials, residual and outputs), as many as the
    smallest of their working sets needs."""
    g = W.tp_decode(R, T)
    K, H = g.K, g.H
    C, Cr, (nbytes, _, p2_bytes) = allreduce_copies(R, T, K, H)

    def rep(a, n):   # n copies at distinct addresses
        t = host_tensor(np.ascontiguousarray(a)).to(device)
        return t.unsqueeze(0).expand(n, *t.shape).contiguous()

    keys = ("permuted_out", "idx_map", "weights", "shared_out")

    def operands(wl, n):
        return dict(zip(keys, (rep(a, n) for a in (wl.permuted_out, wl.idx, wl.weights,
                                                      wl.shared))))

    def epilogue_sets(n):
        res_in, r_out = rep(g.residual, n), torch.empty((n, T, H), dtype=torch.bfloat16,
                                                         device=device)
        n_out = torch.empty_like(r_out)
        return [dict(residual=res_in[c], gamma=gamma, eps=g.eps, residual_out=r_out[c],
                     norm_out=n_out[c], write_out=False) for c in range(n)]

    gamma = host_tensor(g.gamma).to(device)
    ranks = [operands(wl, C) for wl in g.ranks]
    one_sets = list(zip([[{k: v[c] for k, v in rk.items()} for rk in ranks] for c in range(C)],
                        epilogue_sets(C)))
    own = operands(g.ranks[0], Cr)
    partials = torch.empty((Cr, R, T, H), dtype=torch.float32, device=device)
    rank_sets = list(zip([{k: v[c] for k, v in own.items()} for c in range(Cr)],
                         epilogue_sets(Cr), partials))
    scale = g.routed_scale

    def oneshot():
        for rks, ep in one_sets:
            mf.moe_finalize_allreduce(rks, g.wkind, routed_scale=scale, **ep)

    def phase1(r0, part):
        mf.moe_finalize_partial(r0["permuted_out"], r0["idx_map"], r0["weights"], g.wkind,
                                r0["shared_out"], routed_scale=scale, partial=part[0])

    def two_phase_rank():
        for r0, ep, part in rank_sets:
            phase1(r0, part)
            mf.moe_finalize_allreduce_reduce(list(part), **ep)

    def phase1_only():
        for r0, _, part in rank_sets:
            phase1(r0, part)

    def phase2_only():
        for _, ep, part in rank_sets:
            mf.moe_finalize_allreduce_reduce(list(part), **ep)

    def standalone():
        for r0, ep, _ in rank_sets:
            mf.moe_finalize(r0["permuted_out"], r0["idx_map"], r0["weights"], g.wkind,
                            r0["shared_out"], routed_scale=scale, **ep)

    # every partial in place once: rank r's from its operands (copy 0 of the
    # one-shot's), the same values in every copy
    for r in range(R):
        rk = {k: v[0] for k, v in ranks[r].items()}
        mf.moe_finalize_partial(rk["permuted_out"], rk["idx_map"], rk["weights"], g.wkind,
                                rk["shared_out"], routed_scale=scale, partial=partials[0, r])
    partials[1:].copy_(partials[0].unsqueeze(0).expand(Cr - 1, R, T, H))
    oneshot()
    torch.cuda.synchronize(device)
    t = {name: graph_us(fn, device, n, max(1, calls // n))
         for name, fn, n in (("one_shot", oneshot, C), ("two_phase_rank", two_phase_rank, Cr),
                             ("phase1", phase1_only, Cr), ("phase2", phase2_only, Cr),
                             ("standalone_finalize", standalone, Cr))}
    out = {f"us_{k}": round(v, 3) for k, v in t.items()}
    out.update({"R": R, "T": T, "K": K, "H": H, "bytes_one_shot": nbytes,
                "GBps_one_shot": round(nbytes / (t["one_shot"] * 1e-6) / 1e9, 1),
                "frac_one_shot": round(nbytes / (t["one_shot"] * 1e-6) / 1e9 / peak, 4),
                "bytes_phase2": p2_bytes,
                "frac_phase2": round(p2_bytes / (t["phase2"] * 1e-6) / 1e9 / peak, 4),
                "us_R_x_standalone_finalize": round(R * t["standalone_finalize"], 3),
                "copies": C, "copies_one_rank": Cr,
                "calls": max(1, calls // C) * C,
                "plan": mf.allreduce_plan(R, T, H, True)})
    del ranks, one_sets, own, partials, rank_sets
    torch.cuda.empty_cache()
    return out


def link_gbs(device, h2d_bytes, d2h_bytes, reps=5):
    """Plain pinned-memory copy rates of the host link for the given byte
    counts: one H2D copy and one D2H copy each, median of ``reps``."""
    res = {}
    for name, nb in (("h2d", h2d_bytes), ("d2h", d2h_bytes)):
        host = torch.empty(nb, dtype=torch.uint8, pin_memory=True)
        dev = torch.empty(nb, dtype=torch.uint8, device=device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        samples = []
        for _ in range(reps + 1):
            a.record()
            if name == "h2d":
                dev.copy_(host, non_blocking=True)
            else:
                host.copy_(dev, non_blocking=True)
            b.record()
            torch.cuda.synchronize(device)
            samples.append(nb / (a.elapsed_time(b) * 1e-3) / 1e9)
        res[name] = round(statistics.median(samples[1:]), 1)
        del host, dev
    return res


def e2e_zero_copy(mf, wl, host, device, steps):
    """GB/s with the inputs and outputs in pinned host memory, through the
    public host-buffer call: the kernel reads the inputs and writes the
    outputs over the host link in place (no separate copies)."""
    outs = {k: torch.empty((wl.T, wl.H), dtype=torch.bfloat16, pin_memory=True)
            for k in ("residual_out", "norm_out")}

    def step():
        mf.moe_finalize_host(host["x"], host["idx"], host["w"], wl.wkind, host["shared"],
                             device=device, routed_scale=wl.routed_scale,
                             residual=host["residual"], gamma=host["gamma"], eps=wl.eps,
                             write_out=False, **outs)

    step()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / steps
    nb = workload_bytes(wl, write_out=False)
    d2h = sum(t.numel() * t.element_size() for t in outs.values())
    return ms, nb - d2h, d2h


def e2e_copy(mf, wl, host, device, steps):
    """GB/s with host inputs: per step, H2D copies of every input, the call on
    device buffers, D2H copies of the results, all inside the timed region."""
    d = {k: v.to(device) for k, v in host.items()}
    outs = {"residual_out": torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device),
            "norm_out": torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device)}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    def step():
        for k, t in host.items():
            d[k].copy_(t, non_blocking=True)
        call(mf, wl, d, outs)
        for k, t in outs.items():
            host_out[k].copy_(t, non_blocking=True)

    step()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / steps
    del d, outs
    return ms, h2d, d2h


# ---------------------------------------------------------- CPU baseline


def oracle_gbps(wl, tokens, repeat_until_s=0.0):
    """fp64 oracle over the given token rows; returns (GB/s, seconds, passes)."""
    import oracle   # test infrastructure: timed here, never used by the GPU path
    orc = oracle.default()
    sub = dict(idx=wl.idx[tokens], weights=np.ascontiguousarray(wl.weights[tokens]),
               shared=wl.shared[tokens],
               residual=None if wl.residual is None else wl.residual[tokens])
    passes, t0 = 0, time.perf_counter()
    while True:
        orc.moe_finalize(wl.permuted_out, sub["idx"], sub["weights"], wl.wkind,
                         wl.routed_scale, sub["shared"], sub["residual"], wl.gamma, wl.eps,
                         want_out=False)
        passes += 1
        el = time.perf_counter() - t0
        if el >= repeat_until_s or passes >= 3:
            break
    nbytes = algorithmic_bytes(len(tokens), wl.K, wl.H, 4, wl.with_norm, False)
    return nbytes * passes / el / 1e9, el / passes, passes


def oracle_times(wl, want_out, reps=3, min_seconds=0.0):
    """Median seconds of one oracle pass over every token of ``wl``: on one
    thread (at least ``reps`` passes, more until ``min_seconds`` have run),
    and as token blocks from one thread per host core (``reps`` passes).

    The oracle is unchanged: each thread calls it on a contiguous block of
    tokens (ctypes releases the GIL for the duration of the C call).  Returns
    (seconds on one thread, seconds on all cores, threads)."""
    import oracle   # test infrastructure: timed here, never used by the GPU path
    from concurrent.futures import ThreadPoolExecutor
    orc = oracle.default()
    w = np.ascontiguousarray(wl.weights)

    def run(a, b):
        orc.moe_finalize(wl.permuted_out, wl.idx[a:b], w[a:b], wl.wkind, wl.routed_scale,
                         wl.shared[a:b], None if wl.residual is None else wl.residual[a:b],
                         wl.gamma, wl.eps, want_out=want_out)

    single = []
    while len(single) < reps or sum(single) < min_seconds:
        t0 = time.perf_counter()
        run(0, wl.T)
        single.append(time.perf_counter() - t0)
    threads = max(1, len(os.sched_getaffinity(0)))
    bounds = np.linspace(0, wl.T, 4 * threads + 1).astype(int)
    chunks = [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    parallel = []
    with ThreadPoolExecutor(threads) as pool:
        for _ in range(reps):
            t0 = time.perf_counter()
            list(pool.map(lambda ab: run(*ab), chunks))
            parallel.append(time.perf_counter() - t0)
    return statistics.median(single), statistics.median(parallel), threads


def oracle_allreduce_seconds(R, T):
    """Seconds of one single-threaded fp64 oracle pass over the R-rank
    decode problem at batch T (the all-reduce-fused finalize)."""
    import oracle   # test infrastructure: timed here, never used by the GPU path
    g = W.tp_decode(R, T)
    ranks = [{"permuted_out": wl.permuted_out, "idx": wl.idx, "weights": wl.weights,
              "shared": wl.shared} for wl in g.ranks]
    t0 = time.perf_counter()
    oracle.default().moe_finalize_ar(ranks, g.wkind, g.routed_scale, g.residual, g.gamma,
                                     g.eps, want_out=False)
    return time.perf_counter() - t0


CONFIG_KEYS = {"tiny": "T4_tiny", "decode_bs1_packed": "T1", "decode_bs256": "T256",
               "fused_norm_bs16": "T16_rmsnorm"}


def per_config_summary(decode, kernel_ms, achieved, peak, nbytes, cpu):
    """µs per call, GB/s, fraction of the HBM peak and the oracle's times for
    each of the five workloads, side by side."""
    out = {}
    wms = (cpu or {}).get("workloads_ms", {})
    for name, key in CONFIG_KEYS.items():
        dd = decode.get(key)
        if not dd:
            continue
        out[name] = {"us_per_call": dd["us_per_call_graph"], "GBps": dd["GBps_graph"],
                     "frac": dd["frac"], "us_bytes_at_peak": dd["us_bytes_at_peak"],
                     "floor_us_dependent_launch": dd["floor_us_dependent_launch"],
                     "timing": "CUDA-graph replay, inputs rotated over copies larger than L2"}
    out[WORKLOAD] = {"us_per_call": round(kernel_ms * 1e3, 2), "GBps": round(achieved, 1),
                     "frac": round(achieved / peak, 4),
                     "us_bytes_at_peak": round(nbytes / (peak * 1e9) * 1e6, 2),
                     "timing": "mean CUDA-event duration of back-to-back launches"}
    for name, v in out.items():
        if name in wms:
            v["oracle_ms_one_thread"] = wms[name]["one_thread"]
            v["oracle_ms_all_cores"] = wms[name]["all_cores"]
    return out


# Which outputs each workload writes in the benchmark (the prefill emits
# residual_out and norm_out only; every other workload writes out as well).
def writes_out(name, wl):
    return name != WORKLOAD or not wl.with_norm


# ------------------------------------------------------------------- main


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    wl = W.make(WORKLOAD)
    # per step a token sample sized so that all steps take about ref_budget_s
    per_token_s = 4e-4
    n_tok = int(np.clip(args.ref_budget_s / max(1, args.steps + args.warmup) / per_token_s,
                        8, wl.T))
    starts = [(i * n_tok) % (wl.T - n_tok + 1) for i in range(args.steps + args.warmup)]
    times = []
    for i, s0 in enumerate(starts):
        toks = np.arange(s0, s0 + n_tok)
        _, sec, _ = oracle_gbps(wl, toks)
        if i >= args.warmup:
            times.append(sec)
    nbytes = algorithmic_bytes(n_tok, wl.K, wl.H, 4, True, False)
    ms = 1e3 * sum(times) / len(times)
    value = nbytes / (ms * 1e-3) / 1e9
    sample = f"{n_tok} consecutive tokens of {WORKLOAD} per step, full rows"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "T": wl.T, "K": wl.K, "H": wl.H, "E": wl.E,
                       "P": wl.P, "tokens_per_step": n_tok},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, ws, rank, local):
    from moe_deferred_finalize_gb300 import build
    build.build_library()          # no-op when already built; there is no fallback
    import moe_deferred_finalize_gb300 as mf

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl = W.make(WORKLOAD, alloc=pinned_alloc)
    d = device_inputs(wl, device)
    outs = {"residual_out": torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device),
            "norm_out": torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device)}
    nbytes = workload_bytes(wl, write_out=False)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    plan = mf.plan(wl.T, wl.K, wl.H, True, True, sms)

    sampler = ClockSampler(device.index if device.index is not None else 0)
    if rank == 0:
        sampler.start()
    total_ms, per, (win0, _) = time_headline(mf, wl, d, outs, args.steps, args.warmup, ws,
                                             device)
    roof_ms, (_, win1) = time_roofline(mf, wl, d, outs, device, args.roofline_seconds)
    if rank == 0:
        sampler.mark(win0, win1)     # the timed steps and the roofline launches
    clocks = sampler.stop() if rank == 0 else None

    ms_step = max_over_ranks(total_ms / args.steps, ws)
    kernel_ms = statistics.mean(roof_ms)
    value = sum_over_ranks(nbytes, ws) / (ms_step * 1e-3) / 1e9

    peak, peak_src = measured_peaks()
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    traffic = recorded_traffic()

    del d, outs
    torch.cuda.empty_cache()
    host = {"x": host_tensor(wl.permuted_out), "idx": host_tensor(wl.idx).pin_memory(),
            "w": host_tensor(np.ascontiguousarray(wl.weights)).pin_memory(),
            "shared": host_tensor(wl.shared), "residual": host_tensor(wl.residual),
            "gamma": host_tensor(wl.gamma)}
    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, h2d, d2h = e2e_zero_copy(mf, wl, host, device, e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, ws)
    e2e_value = sum_over_ranks(nbytes, ws) / (e2e_ms * 1e-3) / 1e9
    c_ms, c_h2d, c_d2h = e2e_copy(mf, wl, host, device, e2e_steps)
    c_ms = max_over_ranks(c_ms, ws)
    link = link_gbs(device, h2d, d2h)
    torch.cuda.empty_cache()
    decode = {}
    if not args.skip_decode:
        decode = {"T1": decode_latency(mf, "decode_bs1_packed", device, 4000, peak,
                                       producer=True),
                  "T256": decode_latency(mf, "decode_bs256", device, 2000, peak, producer=True,
                                         sequential=True),
                  "T16_rmsnorm": decode_latency(mf, "fused_norm_bs16", device, 2000, peak,
                                                producer=True),
                  "T4_tiny": decode_latency(mf, "tiny", device, 2000, peak)}
        floor = decode["T4_tiny"]["us_per_call_graph"]
        for v in decode.values():
            v["floor_us_dependent_launch"] = floor

    gate = {}
    if not args.skip_decode:
        gate = {"E": 256, "K": 8, "kind": "sigmoid", "outputs": "ids, fp32 weights, packed",
                "us_per_call_graph": {f"T{T}": gate_latency(mf, device, T)
                                      for T in (1, 256, 16384)}}

    allreduce = {}
    if not args.skip_decode:
        for R in (1, 2, 4, 8):
            for T in (1, 16, 256):
                allreduce[f"R{R}_T{T}"] = allreduce_latency(mf, device, R, T, peak)

    cpu = None
    if rank == 0 and not args.skip_cpu:
        sec, psec, nthr = oracle_times(wl, want_out=False, min_seconds=10.0)
        cpu = {"value": round(nbytes / sec / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"all {wl.T} tokens of {WORKLOAD}, repeated for at least 10 s, "
                         f"median {sec:.2f} s per pass, single-threaded fp64"}
        cpu["all_cores"] = {"value": round(nbytes / psec / 1e9, 4), "unit": "GB/s",
                            "cores": nthr,
                            "sample": f"all {wl.T} tokens, median of 3 passes, {psec:.3f} s "
                                      f"per pass, token blocks on {nthr} threads"}
        # every other workload, whole, for the per-workload table
        cpu["workloads_ms"] = {WORKLOAD: {"one_thread": round(1e3 * sec, 3),
                                          "all_cores": round(1e3 * psec, 3)}}
        for name in W.CONFIG_NAMES:
            if name == WORKLOAD:
                continue
            cw = W.make(name)
            s1, sn, _ = oracle_times(cw, want_out=writes_out(name, cw))
            cpu["workloads_ms"][name] = {"one_thread": round(1e3 * s1, 3),
                                         "all_cores": round(1e3 * sn, 3)}
        if allreduce:
            cpu["allreduce_ms_one_thread"] = {
                key: round(1e3 * oracle_allreduce_seconds(v["R"], v["T"]), 3)
                for key, v in allreduce.items()}

    configs = per_config_summary(decode, kernel_ms, achieved, peak, nbytes, cpu)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": wl.T, "K": wl.K, "H": wl.H, "E": wl.E,
                   "P": wl.P, "routing": "fp32 normalised sigmoid", "routed_scale": 2.5,
                   "rmsnorm": True, "emits": ["residual_out", "norm_out"], "io": "bf16",
                   "bytes_per_step": nbytes, "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (%.2f GB read per step)" % (
                       (nbytes - 2 * wl.T * wl.H * 2) / 1e9),
                   "plan": plan},
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "per_call_us": ({"T1": decode["T1"]["us_per_call_graph"],
                         "T256": decode["T256"]["us_per_call_graph"],
                         "timing": "CUDA-graph replay of back-to-back calls, inputs rotated "
                                   "over copies larger than L2"} if decode else None),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": peak_src, "kernel_ms": round(kernel_ms, 5),
                     "launches": len(roof_ms),
                     "window_s": round(sum(roof_ms) * 1e-3, 3),
                     "sm_mhz_median": clocks.get("sm_mhz") if clocks else None},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": round(e2e_ms, 3),
                "mode": "moe_finalize_host: pinned host inputs read and pinned host outputs "
                        "written by the kernel over the host link, no separate copies",
                "link_gbs": link,
                "link_ms_per_step": round(h2d / (link["h2d"] * 1e9) * 1e3, 3),
                "frac_of_link": round(h2d / (link["h2d"] * 1e9) * 1e3 / e2e_ms, 4)},
        "e2e_copy": {"value": round(sum_over_ranks(nbytes, ws) / (c_ms * 1e-3) / 1e9, 1),
                     "unit": "GB/s", "h2d_bytes_per_step": c_h2d, "d2h_bytes_per_step": c_d2h,
                     "steps": e2e_steps, "ms_per_step": round(c_ms, 3),
                     "mode": "H2D copies of all inputs, call on device buffers, D2H copies"},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "configs": configs,
        "decode": decode,
        "gate": gate,
        "allreduce": allreduce,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-decode", action="store_true", help="omit the decode latency lines")
    ap.add_argument("--skip-cpu", action="store_true", help="omit the CPU oracle baseline")
    ap.add_argument("--roofline-seconds", type=float, default=2.0,
                    help="GPU seconds of back-to-back launches behind roofline.kernel_ms")
    ap.add_argument("--ref-budget-s", type=float, default=60.0,
                    help="--impl reference: seconds of oracle work over all steps")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            return run_reference(args, ws, rank)
        return run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
