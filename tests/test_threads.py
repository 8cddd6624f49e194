"""Concurrent calls: host threads enqueue finalizes on their own streams at
the same time (ctypes releases the GIL for each library call), racing on the
library's lazily filled per-device caches (multiprocessor count, the opt-in
for 16-CTA clusters).  Every thread's outputs must be bit-identical to the
same call made alone."""
import threading

import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import bits_of, to_device

pytestmark = pytest.mark.gpu

OUT_KEYS = ("out", "residual_out", "norm_out")


def _workloads():
    return [
        W.make("decode_bs1_packed"),                       # any-K build, 7 CTAs
        W.make("decode_bs256"),                            # K=8 build, 1792 CTAs
        W.make("fused_norm_bs16"),                         # 4-CTA clusters
        W.synth("c16", T=2, K=4, H=32768, E=64, tile=8, P=64, weight_rule="sigmoid",
                routed_scale=2.5, with_norm=True, seed=5, require_all=False),  # 16-CTA clusters
    ]


def _call(mf, wl, dev, stream):
    return mf.moe_finalize(dev["x"], dev["idx"], dev["w"], wl.wkind, dev["shared"],
                           routed_scale=wl.routed_scale, residual=dev.get("residual"),
                           gamma=dev.get("gamma"), eps=wl.eps, stream=stream)


def test_threads_on_own_streams_match_serial_calls(cuda_lib):
    wls = _workloads()
    devs = [to_device(wl) for wl in wls]
    want = []
    for wl, dev in zip(wls, devs):
        res = _call(cuda_lib, wl, dev, None)
        torch.cuda.synchronize()
        want.append({k: bits_of(v) for k, v in res.items() if v is not None and k in OUT_KEYS})

    n_threads, iters = 8, 24
    start = threading.Barrier(n_threads)
    errors = []

    def worker(tid):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream()
            start.wait()
            for it in range(iters):
                i = (tid + it) % len(wls)
                res = _call(cuda_lib, wls[i], devs[i], stream)
                stream.synchronize()
                for k, bits in want[i].items():
                    if not np.array_equal(bits_of(res[k]), bits):
                        errors.append((tid, it, wls[i].name, k))
        except Exception as e:          # reported below, in the main thread
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors[:5]
