"""Run the finalize on one synthetic configuration a few times (no checks).

For profilers: one process, a handful of launches, a known input size.

  python -m moe_deferred_finalize_gb300.run_case --workload decode_bs256 --iters 3
  python -m moe_deferred_finalize_gb300.run_case --prefill-tokens 4096 --iters 3
  python -m moe_deferred_finalize_gb300.run_case --workload decode_bs1_packed --unfused
  python -m moe_deferred_finalize_gb300.run_case --gate-tokens 16384 --iters 3
  python -m moe_deferred_finalize_gb300.run_case --tp 8 16 --form one_shot --iters 3
  python -m moe_deferred_finalize_gb300.run_case --tp-procs 16 --iters 300

--tp-procs times the orchestration of the all-reduce-fused finalize across
processes (moe_deferred_finalize_gb300.tp, two-phase form): two processes on
GPU 0, a gloo group for set-up and the per-step host barrier; it prints the
wall time per step and of the barrier alone.
"""
import argparse
import time

import numpy as np
import torch

import moe_deferred_finalize_gb300 as mf
from moe_deferred_finalize_gb300 import workloads as W


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def _tp_procs_worker(rank, port, T, steps, q):
    import torch.distributed as dist
    from moe_deferred_finalize_gb300 import tp
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=2)
    try:
        g = W.tp_decode(2, T, seed=7)
        wl = g.ranks[rank]
        x = {"permuted_out": _dev(wl.permuted_out), "idx_map": _dev(wl.idx),
             "weights": _dev(wl.weights), "shared_out": _dev(wl.shared)}
        outs = {k: torch.empty((T, g.H), dtype=torch.bfloat16, device="cuda")
                for k in ("out", "residual_out", "norm_out")}
        ep = dict(residual=_dev(g.residual), gamma=_dev(g.gamma), eps=g.eps)
        group = tp.TPFinalize(dist.group.WORLD, T, g.H)
        res = {}
        for n, key in ((20, None), (steps, "us_per_step")):
            torch.cuda.synchronize()
            dist.barrier()
            t0 = time.perf_counter()
            for _ in range(n):
                group.step(x, g.wkind, g.routed_scale, T, outs=outs, **ep)
            torch.cuda.synchronize()
            if key:
                res[key] = (time.perf_counter() - t0) / n * 1e6
        t0 = time.perf_counter()
        for _ in range(steps):
            dist.barrier()
        res["us_per_barrier"] = (time.perf_counter() - t0) / steps * 1e6
        group.close()
        q.put((rank, res))
    finally:
        dist.destroy_process_group()


def _tp_procs(T, steps):
    import multiprocessing as mp
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_tp_procs_worker, args=(r, port, T, steps, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    got = dict(q.get(timeout=600) for _ in procs)
    for pr in procs:
        pr.join(120)
        if pr.exitcode != 0:
            raise RuntimeError(f"rank process exited with {pr.exitcode}")
    for rank in sorted(got):
        r = got[rank]
        print(f"tp-procs: rank {rank} T={T} steps={steps}: {r['us_per_step']:.1f} us per "
              f"two-phase step, {r['us_per_barrier']:.1f} us per host barrier")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    g = ap.add_mutually_exclusive_group(required=True)
    g.add_argument("--workload", choices=W.CONFIG_NAMES)
    g.add_argument("--prefill-tokens", type=int)
    g.add_argument("--gate-tokens", type=int,
                   help="run the top-K gate (E=256, K=8, sigmoid, packed) on this many tokens")
    g.add_argument("--tp", type=int, nargs=2, metavar=("R", "T"),
                   help="the all-reduce-fused finalize over R ranks at decode batch T "
                        "(1, 16 or 256), H=7168, residual + RMSNorm")
    g.add_argument("--tp-procs", type=int, metavar="T",
                   help="time the two-process orchestration (two-phase form, R=2) at batch T "
                        "(1, 16 or 256) on GPU 0 for --iters steps")
    ap.add_argument("--form", choices=["one_shot", "two_phase", "plain"], default="one_shot",
                    help="with --tp: one-shot, two-phase (phase 1 per rank, then phase 2), "
                         "or the plain finalize of rank 0's operands")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--write-out", action="store_true",
                    help="with a residual, also write out (default: residual_out + norm_out only)")
    ap.add_argument("--unfused", action="store_true", help="run the unfused A/B path")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--threads", type=int, default=0)
    args = ap.parse_args(argv)
    if args.tp_procs:
        _tp_procs(args.tp_procs, args.iters)
        return
    if args.gate_tokens:
        g_ = torch.Generator(device="cuda").manual_seed(0)
        z = torch.randn((args.gate_tokens, 256), generator=g_, device="cuda")
        for _ in range(args.iters):
            mf.topk_route(z, 8, "sigmoid", want_packed=True)
        torch.cuda.synchronize()
        print(f"gate: T={args.gate_tokens} E=256 K=8 iters={args.iters} ok")
        return
    if args.tp:
        R, T = args.tp
        g = W.tp_decode(R, T)
        ranks = [{"permuted_out": _dev(wl.permuted_out), "idx_map": _dev(wl.idx),
                  "weights": _dev(wl.weights), "shared_out": _dev(wl.shared)} for wl in g.ranks]
        ep = dict(residual=_dev(g.residual), gamma=_dev(g.gamma), eps=g.eps, write_out=False)
        for _ in range(args.iters):
            if args.form == "one_shot":
                mf.moe_finalize_allreduce(ranks, g.wkind, routed_scale=g.routed_scale, **ep)
            elif args.form == "two_phase":
                parts = [mf.moe_finalize_partial(r["permuted_out"], r["idx_map"], r["weights"],
                                                 g.wkind, r["shared_out"],
                                                 routed_scale=g.routed_scale) for r in ranks]
                mf.moe_finalize_allreduce_reduce(parts, **ep)
            else:
                r0 = ranks[0]
                mf.moe_finalize(r0["permuted_out"], r0["idx_map"], r0["weights"], g.wkind,
                                r0["shared_out"], routed_scale=g.routed_scale, **ep)
        torch.cuda.synchronize()
        print(f"tp: R={R} T={T} form={args.form} iters={args.iters} ok")
        return
    wl = W.make(args.workload) if args.workload else W.prefill(args.prefill_tokens)
    x, idx, w, sh = _dev(wl.permuted_out), _dev(wl.idx), _dev(wl.weights), _dev(wl.shared)
    res = _dev(wl.residual) if wl.with_norm else None
    gam = _dev(wl.gamma) if wl.with_norm else None
    for _ in range(args.iters):
        if args.unfused:
            mf.moe_finalize_unfused(x, idx, w, wl.wkind, sh, routed_scale=wl.routed_scale,
                                    residual=res, gamma=gam, eps=wl.eps)
        else:
            mf.moe_finalize(x, idx, w, wl.wkind, sh, routed_scale=wl.routed_scale, residual=res,
                            gamma=gam, eps=wl.eps, write_out=args.write_out or not wl.with_norm,
                            splits=args.splits, threads=args.threads)
    torch.cuda.synchronize()
    print(f"{wl.name}: T={wl.T} K={wl.K} H={wl.H} P={wl.P} iters={args.iters} ok")


if __name__ == "__main__":
    main()
