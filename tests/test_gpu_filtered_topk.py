"""The bound-filtered indexer + top-k, which serves rows past 16,384 candidates when the
workspace holds its buffers: the selections equal the oracle's and the plain path's bit for
bit, including rows where every candidate ties (all of them reach the bound, more than one
CTA holds: the rows are redone from their scores) and both group sizes of the bound (16
candidates for k - 1 <= 1,024, else 8)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    from block_sparse_long_18_b300 import build

    build.build()
    from block_sparse_long_18_b300 import sgqa

    assert torch.cuda.is_available()
    return sgqa


def _select(sg, prm, q_proxy, k_blk, q_start, ws_bytes=None):
    G, T, _ = q_proxy.shape
    if ws_bytes is None:
        ws_bytes = sg.sgqa_workspace_bytes(prm, sg.SGQA_OP_INDEX_TOPK, T, q_start + T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    idx = torch.empty((G, T, prm.top_k_blocks), dtype=torch.int32, device="cuda")
    cnt = torch.empty((G, T), dtype=torch.int32, device="cuda")
    sg.sgqa_index_topk(prm, q_proxy, q_start, k_blk, idx, cnt, ws)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    return idx.cpu().numpy(), cnt.cpu().numpy()


def _plain_ws_bytes(G, T, max_cand, k):
    """A workspace for the plain path's layout for all T rows (scores, segment pairs and
    counts) that cannot also hold the bound-filtered buffers."""
    ld = (max_cand + 3) // 4 * 4
    nseg = -(-max_cand // 16384)
    a = lambda n: -(-n // 256) * 256
    r = G * T
    return a(r * ld * 4) + 2 * a(r * nseg * (k - 1) * 4) + a(r * nseg * 4)


def test_all_equal_scores_redone_from_the_scores(sg):
    """Zero proxies: every score is 0, so every one of the ~40,000 candidates reaches the
    bound; the tie rule keeps the k-1 largest indices (blocks b_t - (k-1) .. b_t)."""
    G, T, P, B, k, q_start = 2, 16, 64, 1, 33, 40000
    prm = sg.params(G=G, Hg=1, P=P, B=B, k=k)
    q_proxy = torch.zeros((G, T, P), dtype=torch.bfloat16, device="cuda")
    k_blk = torch.zeros((G, q_start + T, P), dtype=torch.bfloat16, device="cuda")
    idx, cnt = _select(sg, prm, q_proxy, k_blk, q_start)
    for i in range(T):
        bt = q_start + i
        want = np.arange(bt - (k - 1), bt + 1, dtype=np.int32)
        for g in range(G):
            assert cnt[g, i] == k
            assert np.array_equal(idx[g, i], want), (g, i)


@pytest.mark.parametrize("k", [33, 1500], ids=["groups_of_16", "groups_of_8"])
def test_filtered_equals_oracle_and_plain_path(sg, k):
    """Integer proxies in [-4, 4] over P = 64 (many equal scores) at 30,000-30,063 tokens
    (B = 1): the default workspace takes the bound-filtered path, a workspace holding only
    the plain layout the plain one; both equal the oracle."""
    G, T, P, B, q_start = 2, 64, 64, 1, 30000
    prm = sg.params(G=G, Hg=1, P=P, B=B, k=k)
    gen = torch.Generator().manual_seed(k)
    qp = torch.randint(-4, 5, (G, T, P), generator=gen).to(torch.bfloat16)
    kb = torch.randint(-4, 5, (G, q_start + T, P), generator=gen).to(torch.bfloat16)
    q_proxy, k_blk = qp.cuda(), kb.cuda()
    idx_f, cnt_f = _select(sg, prm, q_proxy, k_blk, q_start)
    max_cand = (q_start + T - 1) // B
    idx_p, cnt_p = _select(sg, prm, q_proxy, k_blk, q_start, _plain_ws_bytes(G, T, max_cand, k))
    assert np.array_equal(idx_f, idx_p) and np.array_equal(cnt_f, cnt_p)
    d = oracle.dims(G, 1, 192, P, B, k)
    kb_u = u16(kb)
    for g in range(G):
        pos = np.arange(q_start, q_start + T, dtype=np.int64)
        sel, cnt = oracle.select(d, pos, np.full(T, g, np.int32), u16(qp[g]), kb_u)
        assert np.array_equal(idx_f[g], sel) and np.array_equal(cnt_f[g], cnt), g
