"""bench.py host logic without a GPU: algorithmic byte counts, the CPU
baselines, the clock sampler's window filtering and throttle-reason
parsing, and the traffic record's comment-insensitive key."""
import os
import shutil

import pytest

import bench


def test_algorithmic_bytes_match_the_stated_figures():
    # T=16384, K=8, H=7168, fp32 weights, residual + RMSNorm, out not written
    assert bench.algorithmic_bytes(16384, 8, 7168, 4, True, False) == 2_819_635_200
    # ... with out written too
    assert bench.algorithmic_bytes(16384, 8, 7168, 4, True, True) == 2_819_635_200 + 16384 * 7168 * 2
    # T=256 decode, fp32 weights, out written
    assert bench.algorithmic_bytes(256, 8, 7168, 4, False, True) == 36_716_544
    # T=1, packed (4-byte) weights: 8 rows + shared + out + idx/words
    assert bench.algorithmic_bytes(1, 8, 7168, 4, False, True) == 8 * 14336 + 2 * 14336 + 64


class _FakeProc:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def _line(ts, sm, reasons=("Not Active",) * 4):
    return f"{ts}, {sm}, 2070, 900.0, 0x0, " + ", ".join(reasons)


def test_clock_sampler_keeps_only_the_timed_window():
    import datetime
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    stamp = lambda s: (base + datetime.timedelta(seconds=s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    lines = [_line(stamp(0.00), 1200), _line(stamp(0.10), 2070), _line(stamp(0.20), 2070),
             _line(stamp(0.30), 2070, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(stamp(0.40), 900)]
    s = bench.ClockSampler(0)
    s.proc = _FakeProc("\n".join(lines) + "\n")
    s.mark(base.timestamp() + 0.05, base.timestamp() + 0.35)
    r = s.stop()
    assert r["samples_in_window"] == 3 and r["sm_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_sampler_short_window_takes_the_next_sample():
    import datetime
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    stamp = lambda s: (base + datetime.timedelta(seconds=s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    s = bench.ClockSampler(0)
    s.proc = _FakeProc(_line(stamp(0.0), 1000) + "\n" + _line(stamp(0.012), 2070) + "\n")
    s.mark(base.timestamp() + 0.004, base.timestamp() + 0.006)
    r = s.stop()
    assert r["samples_in_window"] == 0 and r["samples"] == 1 and r["sm_mhz"] == 2070.0


def test_traffic_key_ignores_comments_not_code(tmp_path, monkeypatch):
    srcs = []
    for f in bench.KERNEL_SRCS:
        dst = tmp_path / os.path.basename(f)
        shutil.copy(f, dst)
        srcs.append(str(dst))
    monkeypatch.setattr(bench, "KERNEL_SRCS", srcs)
    d0 = bench.kernel_code_digest()
    with open(srcs[0], "a") as fh:
        fh.write("\n// a new comment\n/* and a block\n   comment */\n")
    assert bench.kernel_code_digest() == d0
    with open(srcs[0], "a") as fh:
        fh.write("\nstatic int changed_code = 1;\n")
    assert bench.kernel_code_digest() != d0


def test_cpu_baselines_time_the_oracle_on_every_token():
    from moe_deferred_finalize_gb300 import workloads as W
    import numpy as np
    wl = W.make("fused_norm_bs16")
    gbps, sec, passes = bench.oracle_gbps(wl, np.arange(wl.T))
    assert gbps > 0 and sec > 0 and passes >= 1
    s1, sn, threads = bench.oracle_times(wl, want_out=True)
    assert s1 > 0 and sn > 0
    assert threads == len(os.sched_getaffinity(0))
    assert bench.writes_out("fused_norm_bs16", wl)
    assert not bench.writes_out(bench.WORKLOAD, W.Workload(**{**wl.__dict__, "name": bench.WORKLOAD}))


def test_allreduce_bytes():
    # R ranks' rows, shared output and fp32 routing, then residual in and
    # residual_out + norm_out written, gamma once
    T, K, H = 16, 8, 7168
    for R in (1, 2, 8):
        want = R * (T * K * H * 2 + T * H * 2 + T * K * 8) + 3 * T * H * 2 + H * 2
        assert bench.allreduce_bytes(R, T, K, H) == want
    # one rank with residual + RMSNorm and no out is the plain finalize's count
    assert bench.allreduce_bytes(1, T, K, H) == bench.algorithmic_bytes(T, K, H, 4, True, False)


def test_allreduce_rotation_exceeds_l2_for_every_timed_call():
    """Each call the all-reduce entry times (one-shot; phase 1, phase 2 and
    the plain finalize of one rank) rotates over copies that together hold
    at least twice the L2, so none of them is timed from L2, unless the
    copy count is at its cap."""
    for R in (1, 2, 4, 8):
        for T in (1, 16, 256, 1024):
            C, Cr, (one, p1, p2) = bench.allreduce_copies(R, T, 8, 7168)
            assert C == 4096 or C * one >= 2 * bench.L2_BYTES, (R, T)
            for b in (p1, p2):
                assert Cr == 4096 or Cr * b >= 2 * bench.L2_BYTES, (R, T, b)
            # the one-rank calls touch fewer bytes, so they need at least as
            # many copies as the one-shot
            assert Cr >= C


def test_per_config_summary_puts_the_oracle_beside_each_workload():
    decode = {k: {"us_per_call_graph": 2.0, "GBps_graph": 100.0, "frac": 0.01,
                  "us_bytes_at_peak": 0.1, "floor_us_dependent_launch": 1.7}
              for k in bench.CONFIG_KEYS.values()}
    cpu = {"workloads_ms": {n: {"one_thread": 1.0, "all_cores": 0.5}
                            for n in list(bench.CONFIG_KEYS) + [bench.WORKLOAD]}}
    out = bench.per_config_summary(decode, 0.4, 7000.0, 7000.0, 2_819_635_200, cpu)
    assert set(out) == set(bench.CONFIG_KEYS) | {bench.WORKLOAD}
    for v in out.values():
        assert {"us_per_call", "GBps", "frac", "oracle_ms_one_thread",
                "oracle_ms_all_cores"} <= set(v)
    assert out[bench.WORKLOAD]["frac"] == 1.0 and out[bench.WORKLOAD]["us_per_call"] == 400.0
    # without a CPU leg the GPU figures stand alone
    assert "oracle_ms_one_thread" not in bench.per_config_summary(decode, 0.4, 1, 1, 1, None)["tiny"]
