"""The allocation-free indexer + top-k entry point (sgqa_index_topk_noalloc).

It serves callers that cannot allocate device memory at the point of the call (an
engine that has reserved nearly all of HBM for its KV cache, a plugin interface that
passes tensors but no scratch buffer): its scratch is a fixed array inside the library.
Its selections must equal those of sgqa_index_topk with a caller workspace, bit for bit
(the tolerance the other selection tests use), on two calls in a row that share the
array.  This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

from block_sparse_long_18_b300 import inputs as gen


@pytest.fixture(scope="module")
def sg():
    from block_sparse_long_18_b300 import build

    build.build()
    from block_sparse_long_18_b300 import sgqa

    return sgqa


def _both_paths(sg, wl, seed):
    inp = gen.make_inputs(wl, seed=seed, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, B=wl.B, k=wl.k)
    nb = (wl.C + wl.B - 1) // wl.B
    k_blk = torch.zeros((wl.G, nb, wl.P), dtype=torch.bfloat16, device="cuda")
    sg.sgqa_build_block_index(prm, inp.k_proxy, 0, wl.C, k_blk)
    # existing entry point, caller workspace
    ws = torch.empty(sg.sgqa_workspace_bytes(prm, sg.SGQA_OP_INDEX_TOPK, wl.T, wl.C), dtype=torch.uint8, device="cuda")
    ref_idx = torch.empty((wl.G, wl.T, wl.k), dtype=torch.int32, device="cuda")
    ref_cnt = torch.empty((wl.G, wl.T), dtype=torch.int32, device="cuda")
    sg.sgqa_index_topk(prm, inp.q_proxy, 0, k_blk, ref_idx, ref_cnt, ws)
    # the allocation-free entry point, called through the C ABI
    idx = torch.full_like(ref_idx, -7)
    cnt = torch.full_like(ref_cnt, -7)
    stream = torch.cuda.current_stream().cuda_stream
    rc = sg._lib.sgqa_index_topk_noalloc(ctypes.byref(prm), ctypes.c_void_p(inp.q_proxy.data_ptr()), wl.T, 0,
                                         ctypes.c_void_p(k_blk.data_ptr()), nb, ctypes.c_void_p(idx.data_ptr()),
                                         ctypes.c_void_p(cnt.data_ptr()), ctypes.c_void_p(stream))
    assert rc == 0, sg.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    return ref_idx, ref_cnt, idx, cnt


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_two_calls_in_a_row(sg):
    # first call: one pass through the scratch array
    wl1 = gen.small_workload(T=700, G=2, Hg=16, B=8, k=12, planted=True)
    r_idx, r_cnt, idx, cnt = _both_paths(sg, wl1, seed=21)
    assert torch.equal(cnt, r_cnt) and torch.equal(idx, r_idx)
    # second call, other shape: 20,000 rows x 4 groups x 2,500 candidates do not fit in one
    # pass (32 MiB), so the array is reused pass after pass, starting from call 1's contents
    wl2 = gen.small_workload(T=20000, G=4, Hg=16, B=8, k=64, planted=True)
    r_idx, r_cnt, idx, cnt = _both_paths(sg, wl2, seed=22)
    assert torch.equal(cnt, r_cnt) and torch.equal(idx, r_idx)


def test_noalloc_rejects_requests_beyond_its_scratch(sg):
    """Host-side check, no kernel launched: one pass of 128 rows x 4 groups x 131,071
    candidates (256 MiB) exceeds the 32 MiB array."""
    prm = sg.params()
    a = ctypes.c_void_p(1 << 12)
    rc = sg._lib.sgqa_index_topk_noalloc(ctypes.byref(prm), a, 8192, (1 << 20) - 8192, a, 1 << 17, a, a, None)
    assert rc == 3  # SGQA_ERR_WORKSPACE_TOO_SMALL
    assert sg.NOALLOC_SCRATCH_BYTES == 32 * 1024 * 1024
