"""GPU parity of the decode step (one new query per sequence, packed caches) against the
CPU oracle, sequence by sequence."""
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


def _run_decode(sg, inp, wl, prm):
    G, H, D, P, B, k = wl.G, wl.H, wl.D, wl.P, wl.B, wl.k
    total = inp.k.shape[1]
    batch = len(inp.ctx_len)
    k_blk = torch.zeros((G, total // B, P), dtype=torch.bfloat16, device="cuda")
    # the block-proxy cache as it stands before the step: every token but the newest
    for L, off in zip(inp.ctx_len, inp.kv_off):
        sg.sgqa_build_block_index(prm, inp.k_proxy, off, off + L - 1, k_blk)
    sel = torch.empty((G, batch, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((G, batch), dtype=torch.int32, device="cuda")
    out = torch.empty((batch, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((batch, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(sg.sgqa_workspace_bytes(prm, sg.SGQA_OP_DECODE, 1, max(inp.ctx_len), batch), dtype=torch.uint8,
                     device="cuda")
    sg.sgqa_decode(prm, inp.ctx_len, inp.kv_off, inp.q, inp.q_proxy, inp.gate, inp.k, inp.v, inp.k_proxy, k_blk, sel,
                   cnt, out, lse, ws)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    return k_blk, sel, cnt, out, lse


def _check_sequences(inp, wl, res, seqs, gate_per_dim=1):
    k_blk, sel, cnt, out, lse = res
    d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k, gate_per_dim=gate_per_dim)
    for s in seqs:
        L, off = inp.ctx_len[s], inp.kv_off[s]
        nb = (L + wl.B - 1) // wl.B
        kp = u16(inp.k_proxy[:, off:off + L])
        kb = oracle.block_index(kp, wl.B, 0, L)
        assert np.array_equal(u16(k_blk[:, off // wl.B:off // wl.B + nb]), kb), f"seq {s}: block proxies differ"
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


@pytest.mark.parametrize("P", [256, 192])
def test_decode_ragged_small(sg, P):
    """Ragged contexts (1 .. 3,000 tokens); P = 192 leaves 8 lanes of the indexer's row load idle."""
    wl = gen.Workload(f"dec_small_P{P}", T=1, C=0, G=2, Hg=16, P=P, k=16, batch=5, ctx_lo=1, ctx_hi=3000)
    inp = gen.make_decode_inputs(wl, seed=4, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, P=P, k=wl.k)
    res = _run_decode(sg, inp, wl, prm)
    _check_sequences(inp, wl, res, range(wl.batch))


@pytest.mark.parametrize("B,k,gate_per_dim", [(16, 8, 1), (4, 12, 1), (2, 24, 1), (1, 48, 1), (8, 10, 0)],
                         ids=["B16", "B4_bulk_copy", "B2_bulk_copy", "B1_token_level", "per_head_gate"])
def test_decode_ragged_block_sizes_and_gates(sg, B, k, gate_per_dim):
    """Ragged contexts with blocks of 16 (one block per stage), blocks of 4, 2 and 1 (the
    bulk-copy loader with split-K; B = 1 is token-level selection), and a per-head gate."""
    wl = gen.Workload(f"dec_B{B}", T=1, C=0, G=2, Hg=16, B=B, k=k, batch=4, ctx_lo=1, ctx_hi=2500)
    inp = gen.make_decode_inputs(wl, seed=6, device="cuda")
    if not gate_per_dim:
        inp.gate = inp.gate[:, :, 0].contiguous()  # [batch, H]
    prm = sg.params(G=wl.G, Hg=wl.Hg, B=B, k=wl.k, gate_per_dim=gate_per_dim)
    res = _run_decode(sg, inp, wl, prm)
    _check_sequences(inp, wl, res, range(wl.batch), gate_per_dim=gate_per_dim)


def test_decode_matches_prefill_last_row(sg):
    """A decode step for a sequence equals the prefill output of that sequence's last row."""
    wl = gen.small_workload(T=1500, G=2, Hg=16, B=8, k=20, planted=True)
    inp = gen.make_inputs(wl, seed=11, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, k=wl.k)
    plan = sg.PrefillPlan(prm, wl.T, wl.C)
    pre = plan.run(inp.q, inp.k, inp.v, inp.gate, inp.q_proxy, inp.k_proxy)
    # decode caches hold a whole number of blocks: pad 1500 -> 1504 rows (never attended)
    pad = lambda x: torch.nn.functional.pad(x, (0, 0, 0, 4)).contiguous()
    dec_in = gen.Inputs(wl, inp.q[-1:].contiguous(), pad(inp.k), pad(inp.v), inp.gate[-1:].contiguous(),
                        inp.q_proxy[:, -1:].contiguous(), pad(inp.k_proxy), inp.carry[-1:], None, ctx_len=[wl.T],
                        kv_off=[0])
    k_blk, sel, cnt, out, lse = _run_decode(sg, dec_in, wl, prm)
    assert torch.equal(sel[:, 0], pre.sel_idx[:, -1]) and torch.equal(cnt[:, 0], pre.sel_cnt[:, -1])
    d = (out[0].float() - pre.out[-1].float()).abs().max().item()
    assert d <= 1e-2, d
    assert (lse[0] - pre.lse[-1]).abs().max().item() <= LSE_ABS


def test_decode_full_config_sampled_sequences(sg):
    """8 sequences, contexts uniform in [256K, 1M]; the shortest and the longest sequence
    are checked against the oracle in full (block proxies, selections, outputs)."""
    wl = gen.WORKLOADS["decode"]
    inp = gen.make_decode_inputs(wl, seed=0, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, k=wl.k)
    res = _run_decode(sg, inp, wl, prm)
    order = np.argsort(inp.ctx_len)
    _check_sequences(inp, wl, res, [int(order[0]), int(order[-1])])
    del inp, res
    gc.collect()
    torch.cuda.empty_cache()
