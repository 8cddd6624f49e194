"""The seeded input generator: stated row counts, padded expert-grouped
layout, distinct experts per token, determinism.  CPU only."""
import numpy as np
import pytest

from moe_deferred_finalize_gb300 import workloads as W


def _check_layout(wl):
    T, K = wl.idx.shape
    assert wl.permuted_out.shape == (wl.P, wl.H)
    assert wl.idx.min() >= 0 and wl.idx.max() < wl.P
    # every permuted row is used by at most one (t, k) slot
    assert np.bincount(wl.idx.ravel(), minlength=wl.P).max() <= 1
    # distinct experts per token
    for row in wl.expert_ids:
        assert len(set(row.tolist())) == K
    # padding rows hold the 1e4 sentinel, valid rows do not
    pad = ~wl.valid_rows
    assert (wl.permuted_out[pad] == W.PAD_BITS).all()
    assert (wl.permuted_out[wl.valid_rows] != W.PAD_BITS).any(axis=1).all()
    # rows of one expert are contiguous, in token order, at the front of a tile-aligned block
    order = np.argsort(wl.idx.ravel())
    ex = wl.expert_ids.ravel()[order]
    rows = wl.idx.ravel()[order]
    starts = np.r_[0, np.nonzero(np.diff(ex))[0] + 1]
    assert len(np.unique(ex)) == len(starts)          # each expert one block
    assert (np.diff(ex) >= 0).all()                    # ascending expert ids
    for s, e in zip(starts, np.r_[starts[1:], len(ex)]):
        assert rows[s] % wl.tile == 0
        assert (np.diff(rows[s:e]) == 1).all()
        tok = order[s:e] // K
        assert (np.diff(tok) > 0).all()
    assert np.allclose(wl.weights_f32.sum(axis=1), 1.0, atol=1e-6)


@pytest.mark.parametrize("name", ["tiny", "decode_bs1_packed", "decode_bs256", "fused_norm_bs16"])
def test_named_workload_layout(name):
    wl = W.make(name)
    want = {"tiny": (4, 2, 64, 32), "decode_bs1_packed": (1, 8, 7168, 256),
            "decode_bs256": (256, 8, 7168, 6272), "fused_norm_bs16": (16, 8, 7168, 2048)}[name]
    assert (wl.T, wl.K, wl.H, wl.P) == want
    _check_layout(wl)


def test_packed_words_carry_expert_and_bf16_weight():
    wl = W.make("decode_bs1_packed")
    u = wl.weights.view(np.uint32)
    assert np.array_equal((u >> 16).astype(np.int32), wl.expert_ids)
    assert np.array_equal((u & 0xFFFF).astype(np.uint16), W.to_bf16_bits(wl.weights_f32))


def test_deterministic():
    a, b = W.make("decode_bs256", threads=1), W.make("decode_bs256", threads=8)
    for f in ("permuted_out", "idx", "weights", "shared"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f


def test_prefill_exact_counts_routing():
    counts = W.balanced_counts(16384, 8, 256, np.random.SeedSequence([4, 1]))
    assert counts.sum() == 16384 * 8
    assert int((((counts + 127) // 128) * 128).sum()) == 133120
    rng = np.random.Generator(np.random.PCG64(0))
    g, _, block_rows = W._exact_count_routing(rng, 16384, 8, counts, 128)
    assert np.array_equal(np.bincount(g.ravel(), minlength=256), counts)
    srt = np.sort(g, axis=1)
    assert not (srt[:, 1:] == srt[:, :-1]).any()
    assert block_rows.sum() == 133120


def test_small_random_layout():
    wl = W.synth("x", T=37, K=5, H=24, E=100, tile=16, P=320, weight_rule="sigmoid",
                 wkind="bf16", seed=9, with_norm=True)
    _check_layout(wl)
    assert wl.weights.dtype == np.uint16 and wl.gamma.shape == (24,)


def test_prefill_scaled_counts():
    counts = W.balanced_counts(4096, 8, 256, np.random.SeedSequence([4, 1]))
    assert sorted(set(counts.tolist())) == [120, 128, 136]
    assert int((((counts + 127) // 128) * 128).sum()) == 34816
