"""moe_topk_route (top-K gate) and pack_topk_ids on the GPU against the
oracle: expert ids bit-exact (the selection compares the same fp32 logits on
both sides), weights within fp32 rounding, packed words bit-exact against
the oracle's packing of the GPU's own fp32 weights (the bf16 rounding
decision is taken from the same fp32 value on both sides)."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

from gpu_util import bf16_dev, compare

pytestmark = pytest.mark.gpu


def _logits(T, E, seed, ties=False):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, E))
    if ties:
        z = np.round(z * 2) / 2      # many equal logits
    return z.astype(np.float32)


@pytest.mark.parametrize("T,E,K", [(1, 256, 8), (3, 8, 8), (256, 256, 8), (4100, 384, 8),
                                   (5, 256, 8), (1023, 256, 8), (17, 256, 7), (9, 256, 16),
                                   (5, 1000, 32), (7, 33, 1), (64, 64, 6), (2, 1024, 16)])
@pytest.mark.parametrize("kind", ["softmax", "sigmoid"])
def test_gate_matches_oracle(cuda_lib, orc, T, E, K, kind):
    for ties in (False, True):
        z = _logits(T, E, T * 7 + E + K, ties)
        res = cuda_lib.topk_route(torch.from_numpy(z).cuda(), K, kind, want_packed=True)
        torch.cuda.synchronize()
        ids = res["expert_ids"].cpu().numpy()
        w = res["weights"].cpu().numpy()
        packed = res["packed"].cpu().numpy()
        rid, rw = orc.topk_route(z, K, kind)
        assert np.array_equal(ids, rid), (kind, ties)
        assert np.allclose(w, rw, rtol=2e-6, atol=1e-9), np.abs(w - rw).max()
        assert np.array_equal(packed, orc.pack_topk_ids(ids, w))


def test_gate_outputs_optional_and_consistent(cuda_lib, orc):
    z = torch.from_numpy(_logits(300, 256, 1)).cuda()
    full = cuda_lib.topk_route(z, 8, "sigmoid", want_packed=True)
    only_packed = cuda_lib.topk_route(z, 8, "sigmoid", want_ids=False, want_weights=False,
                                      want_packed=True)
    assert torch.equal(full["packed"], only_packed["packed"])
    e, w = cuda_lib.unpack_topk_ids(full["packed"])
    assert torch.equal(e, full["expert_ids"])
    assert torch.equal(w, full["weights"].to(torch.bfloat16).float())


def test_gate_negative_infinity_logits(cuda_lib, orc):
    z = _logits(4, 64, 3)
    z[:, 10:] = -np.inf             # only 10 finite logits per token
    res = cuda_lib.topk_route(torch.from_numpy(z).cuda(), 12, "sigmoid")
    rid, rw = orc.topk_route(z, 12, "sigmoid")
    assert np.array_equal(res["expert_ids"].cpu().numpy(), rid)
    assert np.allclose(res["weights"].cpu().numpy(), rw, rtol=2e-6, atol=1e-9)


def test_gate_signed_zero_ties(cuda_lib, orc):
    """-0 and +0 are equal logits: the lower expert id comes first."""
    z = np.zeros((6, 96), np.float32)
    z[:, ::2] = -0.0
    z[1, 50] = 1.0
    z[2, 7] = -1.0
    for kind in ("softmax", "sigmoid"):
        res = cuda_lib.topk_route(torch.from_numpy(z).cuda(), 8, kind)
        rid, rw = orc.topk_route(z, 8, kind)
        assert np.array_equal(res["expert_ids"].cpu().numpy(), rid)
        assert np.allclose(res["weights"].cpu().numpy(), rw, rtol=2e-6, atol=1e-9)


def test_pack_bit_exact(cuda_lib, orc):
    rng = np.random.default_rng(5)
    n = 200003
    ids = rng.integers(0, 65536, n).astype(np.int32)
    bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    bits[::7] = (bits[::7] & 0xFFFF0000) | 0x8000          # exact ties
    bits[1::11] = 0x7F800001 | (bits[1::11] & 0x807F0000)  # NaNs with payloads
    bits[2::13] = 0x7F7FFFFF                                 # rounds up to infinity
    w = bits.view(np.float32)
    got = cuda_lib.pack_topk_ids(torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    assert np.array_equal(got.cpu().numpy(), orc.pack_topk_ids(ids, w))


def _permute(ids, E, tile):
    """Expert-grouped, tile-padded row map for given routing (test helper)."""
    T, K = ids.shape
    counts = np.bincount(ids.ravel(), minlength=E)
    blocks = ((counts + tile - 1) // tile) * tile
    start = np.concatenate([[0], np.cumsum(blocks)[:-1]])
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")
    first = np.searchsorted(flat[order], np.arange(E))
    rank = np.empty(flat.size, np.int64)
    rank[order] = np.arange(flat.size) - first[flat[order]]
    return (start[flat] + rank).reshape(T, K).astype(np.int32), int(blocks.sum())


def test_gate_then_finalize_with_packed_weights(cuda_lib, orc):
    """The decode chain through this library's kernels: gate -> packed words
    -> finalize, against the oracle fed the same words."""
    T, E, K, H = 16, 256, 8, 7168
    z = _logits(T, E, 11)
    res = cuda_lib.topk_route(torch.from_numpy(z).cuda(), K, "sigmoid", want_packed=True)
    ids = res["expert_ids"].cpu().numpy()
    packed = res["packed"].cpu().numpy()
    idx, P = _permute(ids, E, 32)
    rng = np.random.default_rng(12)
    x = W.to_bf16_bits(rng.standard_normal((P, H)))
    shared = W.to_bf16_bits(rng.standard_normal((T, H)))
    out = cuda_lib.moe_finalize(bf16_dev(x), torch.from_numpy(idx).cuda(), res["packed"],
                                "packed", bf16_dev(shared), routed_scale=2.5)
    torch.cuda.synchronize()
    ref = orc.moe_finalize(x, idx, packed, "packed", 2.5, shared)
    compare(out, ref, "gate->finalize: ")


def test_gate_packed_word_edge_cases(cuda_lib, orc):
    """Top-8 of 256 first orders one 32-bit word per logit: the upper 24 bits
    of its order key above its inverted id.  Tokens built to defeat that
    ordering must still match the oracle bit for bit: the 12 largest logits
    equal in their upper 24 key bits and different below, the 8th and 9th
    differing only there, all 8 largest on one lane (its whole list taken),
    and an exact tie inside the top 8 (which the words order by id)."""
    rng = np.random.default_rng(2024)
    T = 6
    z = rng.standard_normal((T, 256)).astype(np.float32)
    base = np.float32(3.0).view(np.uint32)
    top = rng.choice(256, 12, replace=False)
    low = rng.choice(256, 12, replace=False).astype(np.uint32)   # distinct low bits
    z[0, top] = ((base & np.uint32(0xFFFFFF00)) | low).view(np.float32)
    order = np.argsort(-z[1])
    z[1, order[8]] = np.nextafter(z[1, order[7]], np.float32(np.inf))   # 9th above 8th by 1 ulp
    z[2, 40:48] = 10.0 + np.arange(8, dtype=np.float32)           # lane 5 holds the top 8
    z[3, [3, 200]] = 7.0                                          # an exact tie, ranks 1-2
    z[4, [9, 17, 250]] = -0.0                                     # signed zeros among the rest
    z[4, 100:108] = 2.0 + np.arange(8, dtype=np.float32)
    z[5, :] = np.round(z[5, :] * 4) / 4                          # many ties
    for kind in ("softmax", "sigmoid"):
        res = cuda_lib.topk_route(torch.from_numpy(z).cuda(), 8, kind, want_packed=True)
        torch.cuda.synchronize()
        rid, rw = orc.topk_route(z, 8, kind)
        ids = res["expert_ids"].cpu().numpy()
        w = res["weights"].cpu().numpy()
        assert np.array_equal(ids, rid), kind
        assert np.allclose(w, rw, rtol=2e-6, atol=1e-9)
        assert np.array_equal(res["packed"].cpu().numpy(), orc.pack_topk_ids(ids, w))
    assert list(rid[2]) == list(range(47, 39, -1))
    assert list(rid[3][:2]) == [3, 200]


@pytest.mark.parametrize("n_top", [31, 32, 33, 40])
def test_gate_candidate_count_boundary(cuda_lib, orc, n_top):
    """n_top equal largest logits spread over the lanes: with 32 or fewer the
    gate ranks the candidates at or above its threshold, with more it falls
    back to round-by-round selection.  Either way the lowest ids win."""
    rng = np.random.default_rng(n_top)
    z = -np.abs(rng.standard_normal((9, 256))).astype(np.float32) - 1.0
    z[:, :n_top] = 5.0
    z[3, n_top + 7] = 6.0              # one token with a unique largest logit
    for kind in ("softmax", "sigmoid"):
        res = cuda_lib.topk_route(torch.from_numpy(z).cuda(), 8, kind, want_packed=True)
        rid, rw = orc.topk_route(z, 8, kind)
        ids = res["expert_ids"].cpu().numpy()
        assert np.array_equal(ids, rid), (n_top, kind)
        assert np.allclose(res["weights"].cpu().numpy(), rw, rtol=2e-6, atol=1e-9)
        assert np.array_equal(ids[0], np.arange(8))


def test_gate_warp_with_mixed_tokens(cuda_lib, orc):
    """Top-8 of 256 takes four tokens per warp; tokens with many equal
    largest logits (more candidates than one segment can rank) sit in the
    same warps as ordinary ones, and the last warp holds fewer than four
    tokens.  Every token must still match the oracle."""
    rng = np.random.default_rng(77)
    T = 13
    z = rng.standard_normal((T, 256)).astype(np.float32)
    for t in range(T):
        if t % 5 == 2:
            z[t, rng.choice(256, 40, replace=False)] = 4.0    # 40 equal maxima
    z[7, :] = 1.5                                             # every logit equal
    for kind in ("softmax", "sigmoid"):
        res = cuda_lib.topk_route(torch.from_numpy(z).cuda(), 8, kind, want_packed=True)
        torch.cuda.synchronize()
        rid, rw = orc.topk_route(z, 8, kind)
        ids = res["expert_ids"].cpu().numpy()
        assert np.array_equal(ids, rid), kind
        assert np.array_equal(ids[7], np.arange(8))
        assert np.allclose(res["weights"].cpu().numpy(), rw, rtol=2e-6, atol=1e-9)
        assert np.array_equal(res["packed"].cpu().numpy(),
                              orc.pack_topk_ids(ids, res["weights"].cpu().numpy()))
