"""tp_csr_build_noalloc: the CSR builder for callers that cannot allocate
device memory themselves (a plugin's enqueue callback that is handed only the
tensors it reads and writes, or a program whose device memory belongs to
another allocator).

It is called here through the C ABI with caller-owned outputs only, twice in a
row, and must give exactly what tp_csr_build (which takes a caller workspace)
gives, and exactly the oracle's stable counting sort - the sort is integer
work, so "within the tests' tolerance" means bit-exact. The file is named to be
collected last; it passes on its own in a fresh process as well as after the
other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import tp

pytestmark = pytest.mark.gpu


def _call_noalloc(tpc, keys, N):
    E = keys.shape[0]
    perm = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    row_ptr = torch.full((N + 1,), -1, dtype=torch.int32, device="cuda")
    ks = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    vp = lambda t: ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)
    st = tpc._lib.tp_csr_build_noalloc(vp(keys), E, N, vp(perm), vp(row_ptr), vp(ks), stream)
    assert st == 0, tpc.tp_status_string(st)
    torch.cuda.synchronize()
    return perm, row_ptr, ks


@pytest.mark.parametrize("E,N", [(131064, 4096), (5000, 37), (262144, 70000), (1, 1)])
def test_noalloc_matches_workspace_entry_point(tpc, E, N):
    rng = np.random.default_rng(E + 7 * N)
    keys = torch.as_tensor(rng.integers(0, N, E).astype(np.int32)).cuda()
    ref = tpc.tp_csr_build(keys, N)
    torch.cuda.synchronize()
    oracle = tp.csr_build(keys.cpu().numpy(), N)
    for _ in range(2):   # the scratch array keeps the previous call's contents
        got = _call_noalloc(tpc, keys, N)
        for a, b, c in zip(got, ref, oracle):
            assert torch.equal(a, b)
            assert np.array_equal(a.cpu().numpy(), c)
    assert tpc.tp_device_status(reset=True) == 0


def test_noalloc_rejects_too_many_edges(tpc):
    cap = tpc.tp_csr_build_noalloc_max_edges()
    assert cap == 1 << 18
    vp = ctypes.c_void_p
    # rejected before any launch: the pointers are never used
    st = tpc._lib.tp_csr_build_noalloc(vp(0x10000), cap + 1, 10, vp(0x10000), vp(0x10000), vp(0), vp(0))
    assert tpc.STATUS_NAMES[st] == "TP_ERR_CAPACITY"
