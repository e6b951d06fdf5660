"""GPU parity of the FP8 (E4M3) block-proxy cache: the cache itself bit for bit against the
oracle's E4M3 block index, and decode steps over it (selections bit for bit, outputs within
the attention tolerance) against the oracle scoring that same E4M3 cache."""
import gc

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_18_b300 import inputs as gen
from parity_util import LSE_ABS, check_outputs, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    from block_sparse_long_18_b300 import build

    build.build()
    from block_sparse_long_18_b300 import sgqa

    return sgqa


@pytest.mark.parametrize("B", [8, 16, 4, 1])
def test_build_block_index_fp8_matches_oracle(sg, B):
    """Integer proxies (the benchmark's recipe), a ragged context (partial last block) and a
    build in two calls (a prefix, then the rest)."""
    wl = gen.small_workload(T=1003, G=2, Hg=4, B=B, k=8, planted=True)
    inp = gen.make_inputs(wl, seed=31, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, P=wl.P, B=B, k=wl.k)
    nb = (wl.C + B - 1) // B
    kb = torch.zeros((wl.G, nb, wl.P), dtype=torch.uint8, device="cuda")
    cut = 517 - 517 % B
    sg.sgqa_build_block_index_fp8(prm, inp.k_proxy, 0, cut, kb)
    sg.sgqa_build_block_index_fp8(prm, inp.k_proxy, cut, wl.C, kb)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    want = oracle.block_index_e4m3(u16(inp.k_proxy), B, 0, wl.C)
    assert np.array_equal(kb.cpu().numpy(), want)


def _run_decode_fp8(sg, inp, wl, prm):
    G, H, D, P, B, k = wl.G, wl.H, wl.D, wl.P, wl.B, wl.k
    total = inp.k.shape[1]
    batch = len(inp.ctx_len)
    k_blk = torch.zeros((G, total // B, P), dtype=torch.uint8, device="cuda")
    for L, off in zip(inp.ctx_len, inp.kv_off):  # the cache before the step: all but the newest token
        sg.sgqa_build_block_index_fp8(prm, inp.k_proxy, off, off + L - 1, k_blk)
    sel = torch.empty((G, batch, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((G, batch), dtype=torch.int32, device="cuda")
    out = torch.empty((batch, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((batch, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(sg.sgqa_workspace_bytes(prm, sg.SGQA_OP_DECODE, 1, max(inp.ctx_len), batch), dtype=torch.uint8,
                     device="cuda")
    sg.sgqa_decode_fp8(prm, inp.ctx_len, inp.kv_off, inp.q, inp.q_proxy, inp.gate, inp.k, inp.v, inp.k_proxy, k_blk,
                       sel, cnt, out, lse, ws)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    return k_blk, sel, cnt, out, lse


def _check_sequences_fp8(inp, wl, res, seqs):
    k_blk, sel, cnt, out, lse = res
    d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k)
    for s in seqs:
        L, off = inp.ctx_len[s], inp.kv_off[s]
        nb = (L + wl.B - 1) // wl.B
        codes = oracle.block_index_e4m3(u16(inp.k_proxy[:, off:off + L]), wl.B, 0, L)
        assert np.array_equal(k_blk[:, off // wl.B:off // wl.B + nb].cpu().numpy(), codes), \
            f"seq {s}: E4M3 block proxies differ"
        kb = oracle.e4m3_as_bf16(codes)
        K = u16(inp.k[:, off:off + L])
        V = u16(inp.v[:, off:off + L])
        for g in range(wl.G):
            pos = np.array([L - 1])
            grp = np.array([g], np.int32)
            osel, ocnt = oracle.select(d, pos, grp, u16(inp.q_proxy[g, s:s + 1]), kb)
            assert int(cnt[g, s]) == int(ocnt[0]), f"seq {s} group {g}: count"
            assert np.array_equal(sel[g, s].cpu().numpy(), osel[0]), f"seq {s} group {g}: selection differs"
            hs = slice(g * wl.Hg, (g + 1) * wl.Hg)
            ref, ref_lse = oracle.attention(d, pos, grp, u16(inp.q[s:s + 1, hs]), u16(inp.gate[s:s + 1, hs]), K, V,
                                            osel, ocnt)
            check_outputs(u16(out[s:s + 1, hs]), ref, f"seq {s} group {g}")
            assert np.max(np.abs(lse[s, hs].cpu().numpy() - ref_lse[0])) <= LSE_ABS


@pytest.mark.parametrize("P", [256, 192, 128, 64])
def test_decode_fp8_ragged(sg, P):
    """Ragged contexts (1 .. 3,000 tokens, partial newest blocks) for every proxy width the
    E4M3 indexer lays out differently (16, 8 or 4 lanes per cache row; P = 192 takes 16
    lanes of which 12 hold codes)."""
    wl = gen.Workload(f"dec8_P{P}", T=1, C=0, G=2, Hg=16, P=P, k=16, batch=5, ctx_lo=1, ctx_hi=3000)
    inp = gen.make_decode_inputs(wl, seed=32, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, P=P, k=wl.k)
    res = _run_decode_fp8(sg, inp, wl, prm)
    _check_sequences_fp8(inp, wl, res, range(wl.batch))


@pytest.mark.parametrize("scale", [2.0 ** 17, 2.0 ** -30], ids=["q_above_f16_range", "q_below_f16_range"])
def test_decode_fp8_query_not_f16_exact(sg, scale):
    """Query proxies scaled by a power of two out of f16's exact range (past 65,504, or below
    its smallest subnormal): the indexer's products then come from fp32 operands rather than
    f16 ones; selections and outputs still equal the oracle's."""
    wl = gen.Workload("dec8_qscale", T=1, C=0, G=2, Hg=16, k=16, batch=4, ctx_lo=1, ctx_hi=3000)
    inp = gen.make_decode_inputs(wl, seed=33, device="cuda")
    inp.q_proxy = (inp.q_proxy.float() * scale).to(torch.bfloat16)
    assert not torch.equal(inp.q_proxy.float(), inp.q_proxy.half().float())
    prm = sg.params(G=wl.G, Hg=wl.Hg, k=wl.k)
    res = _run_decode_fp8(sg, inp, wl, prm)
    _check_sequences_fp8(inp, wl, res, range(wl.batch))


def test_decode_fp8_full_config_sampled_sequences(sg):
    """The 8-sequence decode workload (contexts uniform in [256K, 1M]) over an E4M3 cache;
    the shortest and the longest sequence are checked in full."""
    wl = gen.WORKLOADS["decode"]
    inp = gen.make_decode_inputs(wl, seed=0, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, k=wl.k)
    res = _run_decode_fp8(sg, inp, wl, prm)
    order = np.argsort(inp.ctx_len)
    _check_sequences_fp8(inp, wl, res, [int(order[0]), int(order[-1])])
    del inp, res
    gc.collect()
    torch.cuda.empty_cache()
