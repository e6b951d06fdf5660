"""A partly filled block's mean is rounded once, as the exact quotient sum / n would be
(ai4snews item, Interpretation para 2, read as the element-wise mean of the tokens
present).  Token proxies are chosen so that each fp32 sum is exact and sits on n times a
rounding midpoint of the storage format, or a few fp32 steps beside it; the block index
(bf16, and the FP8 E4M3 decode cache) must equal the oracle's fp64 mean bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from midpoint_sums import midpoint_sums, split_bf16
from parity_util import u16

pytestmark = pytest.mark.gpu

G, P, B, NBLK = 2, 256, 8, 96


@pytest.fixture(scope="module")
def sg():
    from block_sparse_long_18_b300 import build

    build.build()
    from block_sparse_long_18_b300 import sgqa

    assert torch.cuda.is_available()
    return sgqa


def _inputs(fmt, seed):
    """Proxies [G, NBLK * B, P]: block i holds t0, t1, t2 in its first three tokens (zeros
    after), summing to a midpoint case for n_i = 3 .. 7 tokens."""
    rng = np.random.default_rng(seed)
    n = np.array([(3, 5, 6, 7, 3, 7)[i % 6] for i in range(NBLK)])
    s = midpoint_sums(rng, np.broadcast_to(n[None, :, None], (G, NBLK, P)).astype(np.float64), fmt)
    t0, t1, t2 = split_bf16(s)
    kp = np.zeros((G, NBLK, B, P), np.float32)
    kp[:, :, 0], kp[:, :, 1], kp[:, :, 2] = t0, t1, t2
    kp = torch.from_numpy(kp.reshape(G, NBLK * B, P)).to(torch.bfloat16)
    assert np.array_equal(kp.float().numpy().reshape(G, NBLK, B, P)[:, :, 0], t0)
    return kp, n


@pytest.mark.parametrize("fmt", ["bf16", "e4m3"])
def test_partial_block_means_at_rounding_midpoints(sg, fmt):
    kp, n = _inputs(fmt, seed=5 if fmt == "bf16" else 6)
    prm = sg.params(G=G, Hg=16, P=P, B=B, k=8)
    e4m3 = fmt == "e4m3"
    kb = torch.zeros((G, NBLK, P), dtype=torch.uint8 if e4m3 else torch.bfloat16, device="cuda")
    kp_d = kp.cuda()
    want = np.zeros((G, NBLK, P), np.uint8 if e4m3 else np.uint16)
    kp_u = u16(kp)
    for i in range(NBLK):  # one call per block: block i alone, its first n_i tokens present
        lo, hi = i * B, i * B + int(n[i])
        if e4m3:
            sg.sgqa_build_block_index_fp8(prm, kp_d, lo, hi, kb)
            want = oracle.block_index_e4m3(kp_u, B, lo, hi, k_blk=want, nb_cap=NBLK)
        else:
            sg.sgqa_build_block_index(prm, kp_d, lo, hi, kb)
            want = oracle.block_index(kp_u, B, lo, hi, k_blk=want, nb_cap=NBLK)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    got = kb.cpu().numpy() if e4m3 else u16(kb)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} block means differ, first at {bad[0].tolist()}"
