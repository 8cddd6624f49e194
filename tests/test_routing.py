"""unpack_topk_ids and moe_finalize_check_indices on the GPU: bit-exact
against the oracle and against planted bad indices."""
import numpy as np
import pytest
import torch

from moe_deferred_finalize_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_unpack_every_low_half(cuda_lib, orc):
    low = np.arange(65536, dtype=np.uint32)
    hi = np.array([0, 1, 7, 255, 383, 32767, 32768, 65535], np.uint32)
    words = ((hi[:, None] << 16) | low[None, :]).ravel().view(np.int32)
    e, w = cuda_lib.unpack_topk_ids(torch.from_numpy(words).cuda())
    torch.cuda.synchronize()
    re, rw = orc.unpack_topk_ids(words)
    assert np.array_equal(e.cpu().numpy(), re)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), rw.view(np.uint32))


@pytest.mark.parametrize("n", [1, 3, 8, 1000, 131072, 131075])
def test_unpack_sizes(cuda_lib, orc, n):
    rng = np.random.default_rng(n)
    words = rng.integers(-2**31, 2**31, n, dtype=np.int64).astype(np.int32)
    e, w = cuda_lib.unpack_topk_ids(torch.from_numpy(words).cuda())
    re, rw = orc.unpack_topk_ids(words)
    assert np.array_equal(e.cpu().numpy(), re)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), rw.view(np.uint32))


def test_unpack_one_output_only(cuda_lib, orc):
    wl = W.make("decode_bs1_packed")
    packed = torch.from_numpy(wl.weights).cuda()
    lib = cuda_lib.lib()
    import ctypes
    w = torch.full(packed.shape, -1.0, device="cuda")
    st = lib.unpack_topk_ids(ctypes.c_void_p(packed.data_ptr()), packed.numel(), None,
                             ctypes.c_void_p(w.data_ptr()),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy(), orc.unpack_topk_ids(wl.weights)[1])
    assert np.array_equal(w.cpu().numpy().view(np.uint32) >> 16, W.to_bf16_bits(wl.weights_f32))


def test_check_indices(cuda_lib):
    wl = W.make("decode_bs256")
    idx = torch.from_numpy(wl.idx).cuda()
    assert cuda_lib.check_indices(idx, wl.P).item() == 0
    bad = wl.idx.copy()
    bad[0, 0], bad[17, 3], bad[255, 7], bad[100, 1] = -1, wl.P, 2**31 - 1, wl.P - 1
    cnt = cuda_lib.check_indices(torch.from_numpy(bad).cuda(), wl.P)
    assert cnt.item() == 3
    # the counter is reset by every call
    assert cuda_lib.check_indices(idx, wl.P, counter=cnt).item() == 0
    empty = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    assert cuda_lib.check_indices(empty, 5).item() == 0


def test_check_indices_flat_map_misread(cuda_lib):
    """A [T*K] flat map read as [T*K, 1] passes, read with the wrong top_k does not
    stay in range when P is the true row count."""
    rng = np.random.default_rng(0)
    T, K, P = 1000, 8, 1000 * 8
    idx = rng.permutation(P).astype(np.int32).reshape(T, K)
    assert cuda_lib.check_indices(torch.from_numpy(idx).cuda(), P).item() == 0
    assert cuda_lib.check_indices(torch.from_numpy(idx).cuda(), P // 2).item() == \
        int((idx >= P // 2).sum())
