"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded
inputs.  Selections (and the block index) must match bit for bit; attention outputs
within the tolerance stated in parity_util.  Large workloads are checked on sampled rows
(plus the edge rows of the method) in the launch configuration the benchmark times."""
import gc

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_18_b300 import inputs as gen
from parity_util import LSE_ABS, check_outputs, sample_rows, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    from block_sparse_long_18_b300 import build

    build.build()
    from block_sparse_long_18_b300 import sgqa

    assert torch.cuda.is_available()
    return sgqa


def _prm(sg, wl, gate_per_dim=1):
    return sg.params(G=wl.G, Hg=wl.Hg, D=wl.D, P=wl.P, B=wl.B, k=wl.k, gate_per_dim=gate_per_dim)


def _to_cuda(inp):
    for name in ("q", "k", "v", "gate", "q_proxy", "k_proxy"):
        setattr(inp, name, getattr(inp, name).cuda())
    return inp


def _gpu_prefill(sg, inp, wl, prm, gate=None):
    plan = sg.PrefillPlan(prm, wl.T, wl.C, wl.q_start)
    if wl.q_start > 0:  # blocks of the cached prefix, built once before the chunk
        sg.sgqa_build_block_index(prm, inp.k_proxy, 0, wl.q_start, plan.k_blk)
    res = plan.run(inp.q, inp.k, inp.v, inp.gate if gate is None else gate, inp.q_proxy, inp.k_proxy)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    return res


def _check_prefill(inp, wl, res, rows, groups=None, gate_per_dim=1, gate_rows_all=None, check_blocks=True,
                   kb_oracle=None, attn_rows=None):
    d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k, gate_per_dim=gate_per_dim)
    nb = (wl.C + wl.B - 1) // wl.B
    if kb_oracle is None:
        kb_oracle = oracle.block_index(u16(inp.k_proxy), wl.B, 0, wl.C)
    if check_blocks:
        assert np.array_equal(u16(res.k_blk)[:, :nb], kb_oracle), "block index differs"
    K, V = u16(inp.k), u16(inp.v)
    rows = np.asarray(rows, dtype=np.int64)
    attn_rows = rows if attn_rows is None else np.asarray(attn_rows, dtype=np.int64)
    stats = []
    for g in (range(wl.G) if groups is None else groups):
        pos = wl.q_start + rows
        grp = np.full(len(rows), g, np.int32)
        sel, cnt = oracle.select(d, pos, grp, u16(inp.q_proxy[g][torch.as_tensor(rows, device=inp.q_proxy.device)]),
                                 kb_oracle)
        gsel = res.sel_idx[g].cpu().numpy()[rows]
        gcnt = res.sel_cnt[g].cpu().numpy()[rows]
        assert np.array_equal(gcnt, cnt), f"group {g}: sel_cnt differs"
        bad = np.argwhere(np.any(gsel != sel, axis=1))
        assert bad.size == 0, f"group {g}: selection differs at rows {rows[bad[:5, 0]].tolist()}"
        if attn_rows.size == 0:
            continue
        ai = np.searchsorted(rows, attn_rows)
        hs = slice(g * wl.Hg, (g + 1) * wl.Hg)
        ar = torch.as_tensor(attn_rows, device=inp.q.device)
        q_rows = u16(inp.q[ar][:, hs])
        gsrc = inp.gate if gate_rows_all is None else gate_rows_all
        gate_rows = u16(gsrc[ar][:, hs])
        out, lse = oracle.attention(d, pos[ai], grp[ai], q_rows, gate_rows, K, V, sel[ai], cnt[ai])
        stats.append(check_outputs(u16(res.out[ar][:, hs]), out, f"group {g} out"))
        glse = res.lse[ar][:, hs].cpu().numpy()
        assert np.max(np.abs(glse - lse)) <= LSE_ABS, f"group {g}: lse max err {np.max(np.abs(glse - lse))}"
    return stats


# ---------------------------------------------------------------------------------------
# small and ragged cases: every row checked
# ---------------------------------------------------------------------------------------

SMALL = [
    dict(T=300, G=2, Hg=16, B=8, k=8),                    # ragged T, several tiles, G>1
    dict(T=129, G=1, Hg=16, B=8, k=5, q_start=200),       # chunk with a cached prefix
    dict(T=64, G=1, Hg=4, B=8, k=1),                      # k = 1: own block only
    dict(T=7, G=1, Hg=4, B=8, k=4),                       # T < B
    dict(T=1, G=1, Hg=4, B=8, k=4),                       # single token
    dict(T=520, G=1, Hg=2, B=1, k=64),                    # token-level (B = 1) reference form
    dict(T=300, G=1, Hg=16, B=16, k=6),                   # B = 16
    dict(T=200, G=1, Hg=8, B=4, k=9),                     # B = 4 (cp.async loader)
    dict(T=150, G=1, Hg=4, B=2, k=20),                    # B = 2
    dict(T=260, G=1, Hg=1, B=8, k=7, P=64),               # P = 64, single head
    dict(T=333, G=2, Hg=16, B=8, k=40, P=128, planted=True),
    dict(T=300, G=2, Hg=8, B=8, k=12, P=192),             # P = 192: three 64-wide indexer chunks
]


# Rows with more candidates than one top-k CTA holds in registers (16,384): the two-level
# selection (per-slice lists, then a merge), and the streaming instance where the merged
# lists would not fit either.  Integer proxies in [-4, 4] over P = 64 give many equal
# scores, so the tie rule is exercised across slice boundaries.
LONG_ROWS = [
    dict(T=96, G=2, Hg=1, B=1, k=33, P=64, q_start=40000),    # 3 slices, merge in 128 threads
    dict(T=40, G=1, Hg=2, B=1, k=3000, P=64, q_start=36000),  # 3 slices, merge in 512 threads
    dict(T=24, G=1, Hg=1, B=1, k=6000, P=64, q_start=40000),  # merged lists too long: streaming
    dict(T=70, G=1, Hg=4, B=1, k=12, P=64, q_start=16350),    # rows on both sides of 16,384
]


@pytest.mark.parametrize("case", LONG_ROWS, ids=[f"q{c['q_start']}_k{c['k']}" for c in LONG_ROWS])
def test_prefill_long_rows_all_rows(sg, case):
    wl = gen.small_workload(**case)
    inp = _to_cuda(gen.make_inputs(wl, seed=4))
    prm = _prm(sg, wl)
    res = _gpu_prefill(sg, inp, wl, prm)
    _check_prefill(inp, wl, res, np.arange(wl.T))


@pytest.mark.parametrize("case", SMALL, ids=[f"T{c['T']}_B{c['B']}_k{c['k']}_G{c['G']}" for c in SMALL])
def test_prefill_small_all_rows(sg, case):
    wl = gen.small_workload(**case)
    inp = _to_cuda(gen.make_inputs(wl, seed=3))
    prm = _prm(sg, wl)
    res = _gpu_prefill(sg, inp, wl, prm)
    _check_prefill(inp, wl, res, np.arange(wl.T))


def test_prefill_tiny_config_all_rows(sg):
    """The tiny workload: T = 2,048, 1 group x 4 heads, k = 32 blocks, every row."""
    wl = gen.WORKLOADS["tiny"]
    inp = _to_cuda(gen.make_inputs(wl, seed=0))
    res = _gpu_prefill(sg, inp, wl, _prm(sg, wl))
    stats = _check_prefill(inp, wl, res, np.arange(wl.T))
    assert stats[0]["n"] == wl.T * wl.Hg * wl.D


@pytest.mark.parametrize("seed", [1, 2])
def test_prefill_tiny_other_seeds(sg, seed):
    wl = gen.WORKLOADS["tiny"]
    inp = _to_cuda(gen.make_inputs(wl, seed=seed))
    res = _gpu_prefill(sg, inp, wl, _prm(sg, wl))
    _check_prefill(inp, wl, res, np.arange(wl.T))


def test_per_head_gate(sg):
    wl = gen.small_workload(T=200, G=2, Hg=16, B=8, k=6)
    inp = _to_cuda(gen.make_inputs(wl, seed=5))
    gate_h = inp.gate[:, :, 0].contiguous()                      # [T, H]
    prm = _prm(sg, wl, gate_per_dim=0)
    res = _gpu_prefill(sg, inp, wl, prm, gate=gate_h)
    d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k, gate_per_dim=0)
    kb = oracle.block_index(u16(inp.k_proxy), wl.B, 0, wl.C)
    rows = np.arange(wl.T)
    for g in range(wl.G):
        sel, cnt = oracle.select(d, rows, np.full(wl.T, g, np.int32), u16(inp.q_proxy[g]), kb)
        hs = slice(g * wl.Hg, (g + 1) * wl.Hg)
        out, _ = oracle.attention(d, rows, np.full(wl.T, g, np.int32), u16(inp.q[:, hs]), u16(gate_h[:, hs]),
                                  u16(inp.k), u16(inp.v), sel, cnt)
        check_outputs(u16(res.out[:, hs]), out, "per-head gate")


def test_dense_mode_equals_dense_attention(sg):
    wl = gen.small_workload(T=400, G=2, Hg=16, B=8, k=4)
    inp = _to_cuda(gen.make_inputs(wl, seed=6))
    prm = _prm(sg, wl)
    out = torch.empty_like(inp.q)
    lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
    dummy_idx = torch.zeros((wl.G, wl.T, wl.k), dtype=torch.int32, device="cuda")
    dummy_cnt = torch.zeros((wl.G, wl.T), dtype=torch.int32, device="cuda")
    sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, dummy_idx, dummy_cnt, 0, out, lse, dense_mode=True)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k)
    rows = np.arange(wl.T)
    for g in range(wl.G):
        hs = slice(g * wl.Hg, (g + 1) * wl.Hg)
        ref, ref_lse = oracle.attention(d, rows, np.full(wl.T, g, np.int32), u16(inp.q[:, hs]), u16(inp.gate[:, hs]),
                                        u16(inp.k), u16(inp.v), dense=True)
        check_outputs(u16(out[:, hs]), ref, "dense")
        assert np.max(np.abs(lse[:, hs].cpu().numpy() - ref_lse)) <= LSE_ABS


def test_separate_stages_equal_fused_prefill(sg):
    """build_block_index + index_topk + sparse_attn_fwd called one by one give the same
    bytes as the fused prefill entry."""
    wl = gen.small_workload(T=700, G=2, Hg=16, B=8, k=12, planted=True)
    inp = _to_cuda(gen.make_inputs(wl, seed=7))
    prm = _prm(sg, wl)
    res = _gpu_prefill(sg, inp, wl, prm)
    kb = torch.zeros_like(res.k_blk)
    sg.sgqa_build_block_index(prm, inp.k_proxy, 0, wl.C, kb)
    idx = torch.empty_like(res.sel_idx)
    cnt = torch.empty_like(res.sel_cnt)
    ws = torch.empty(sg.sgqa_workspace_bytes(prm, sg.SGQA_OP_INDEX_TOPK, wl.T, wl.T), dtype=torch.uint8, device="cuda")
    sg.sgqa_index_topk(prm, inp.q_proxy, 0, kb, idx, cnt, ws)
    out = torch.empty_like(inp.q)
    ws_a = torch.empty(sg.sgqa_workspace_bytes(prm, sg.SGQA_OP_ATTN, wl.T, wl.T), dtype=torch.uint8, device="cuda")
    sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, idx, cnt, 0, out, ws=ws_a)
    torch.cuda.synchronize()
    assert torch.equal(kb, res.k_blk) and torch.equal(idx, res.sel_idx) and torch.equal(cnt, res.sel_cnt)
    assert torch.equal(out, res.out)


def test_small_workspace_many_passes(sg):
    """A workspace that holds only 128 rows forces many indexer/top-k passes; the result
    must not change."""
    wl = gen.small_workload(T=1000, G=2, Hg=16, B=8, k=16, planted=True)
    inp = _to_cuda(gen.make_inputs(wl, seed=8))
    prm = _prm(sg, wl)
    res = _gpu_prefill(sg, inp, wl, prm)
    ld = ((wl.T - 1) // wl.B + 3) // 4 * 4
    ws = torch.empty(wl.G * 128 * ld * 4, dtype=torch.uint8, device="cuda")
    idx = torch.empty_like(res.sel_idx)
    cnt = torch.empty_like(res.sel_cnt)
    sg.sgqa_index_topk(prm, inp.q_proxy, 0, res.k_blk, idx, cnt, ws)
    torch.cuda.synchronize()
    assert torch.equal(idx, res.sel_idx) and torch.equal(cnt, res.sel_cnt)


@pytest.mark.parametrize("q_start,gate_per_dim", [(0, 1), (1000, 1), (1000, 0)])
def test_host_prefill_pipeline_equals_device_prefill(sg, q_start, gate_per_dim):
    """The end-to-end entry sgqa_prefill_host (pinned host tensors, chunks of rows
    pipelined by the library over its copy-in stream, the calling stream and its copy-out
    stream) gives bit-identical outputs, LSE and block index to one prefill call on device
    tensors when its chunks are whole grouping windows (4,096 rows)."""
    wl = gen.small_workload(T=9000, G=2, Hg=16, B=8, k=24, planted=True, q_start=q_start)
    inp = _to_cuda(gen.make_inputs(wl, seed=11))
    prm = _prm(sg, wl, gate_per_dim=gate_per_dim)
    gate = inp.gate if gate_per_dim else inp.gate[:, :, 0].contiguous()
    res = _gpu_prefill(sg, inp, wl, prm, gate=gate)
    hp = sg.HostPrefill(prm, wl.T, wl.C, wl.q_start, chunk_rows=4096, with_lse=True)  # three chunks
    host = {n: getattr(inp, n).cpu().pin_memory() for n in ("q", "k", "v", "q_proxy", "k_proxy")}
    host["gate"] = gate.cpu().pin_memory()
    for _ in range(2):  # a second run reuses every buffer
        hp.out_host.zero_()
        out = hp.run(host)
        torch.cuda.synchronize()
        assert sg.sgqa_get_device_error() == 0
        assert torch.equal(out, res.out.cpu())
        assert torch.equal(hp.lse_host, res.lse.cpu())
        assert torch.equal(hp.d["k_blk"], res.k_blk)


def test_host_prefill_small_chunks_within_tolerance(sg):
    """Chunks of 1,024 rows (smaller than a grouping window): the attention's units differ
    from one call over all rows, so outputs agree within the attention tolerance and LSE
    within its bound; the block index is identical."""
    wl = gen.small_workload(T=2600, G=2, Hg=16, B=8, k=24, planted=True, q_start=1000)
    inp = _to_cuda(gen.make_inputs(wl, seed=11))
    prm = _prm(sg, wl)
    res = _gpu_prefill(sg, inp, wl, prm)
    hp = sg.HostPrefill(prm, wl.T, wl.C, wl.q_start, chunk_rows=1024, with_lse=True)
    host = {n: getattr(inp, n).cpu().pin_memory() for n in ("q", "k", "v", "gate", "q_proxy", "k_proxy")}
    out = hp.run(host)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    assert torch.equal(hp.d["k_blk"], res.k_blk)
    d = (out.float() - res.out.cpu().float()).abs()
    assert float(d.max()) <= 2e-2 and float(d.mean()) <= 1e-3, (float(d.max()), float(d.mean()))
    assert float((hp.lse_host - res.lse.cpu()).abs().max()) <= LSE_ABS


def test_block_index_real_valued_proxies_within_one_ulp(sg):
    """The block mean on arbitrary (non-integer) proxies: the device sums the 8 bf16 token
    proxies in fp32 and rounds once, the oracle takes the fp64 mean and rounds once.  They
    agree exactly unless the fp32 sum itself rounded, and then by at most one bf16 ulp.
    Proxies N(0,1) times 2^e, e uniform in [-12, 11] per token, so most 8-term sums span
    more than 24 bits; the last block is partial (the fp64 division path)."""
    G, C, P, B = 2, 8192 + 5, 256, 8
    g = torch.Generator().manual_seed(31)
    scale = torch.exp2(torch.randint(-12, 12, (G, C, 1), generator=g).float())
    kp = (torch.randn((G, C, P), generator=g) * scale).to(torch.bfloat16)
    prm = sg.params(G=G, Hg=16, P=P, B=B, k=8)
    nb = (C + B - 1) // B
    kb = torch.zeros((G, nb, P), dtype=torch.bfloat16, device="cuda")
    sg.sgqa_build_block_index(prm, kp.cuda(), 0, C, kb)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    ref = oracle.block_index(u16(kp), B, 0, C).astype(np.int32)
    got = u16(kb).astype(np.int32)
    # bf16 payloads as ordered integers: adjacent representable values differ by one
    mono = lambda x: np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    dist = np.abs(mono(got) - mono(ref))
    assert dist.max() <= 1, f"block index more than one bf16 ulp from the fp64 mean ({dist.max()})"
    same = float((dist == 0).mean())
    print(f"bit-identical block proxies: {same:.6f} of {dist.size}")
    assert same > 0.9


# ---------------------------------------------------------------------------------------
# error paths on the device (no fault: bounded waits and checked indices)
# ---------------------------------------------------------------------------------------

def test_bounded_wait_times_out_cleanly(sg):
    assert sg.sgqa_get_device_error() == 0
    sg.sgqa_selftest_wait_timeout(2_000_000)   # 2 ms on a barrier nothing arrives at
    assert sg.sgqa_get_device_error() == 5     # SGQA_ERR_DEVICE_TIMEOUT
    assert sg.sgqa_get_device_error() == 0     # cleared
    # the context is still usable
    wl = gen.small_workload(T=64, G=1, Hg=4, B=8, k=3)
    inp = _to_cuda(gen.make_inputs(wl, seed=9))
    res = _gpu_prefill(sg, inp, wl, _prm(sg, wl))
    _check_prefill(inp, wl, res, np.arange(wl.T))


@pytest.mark.parametrize("kernel", ["union", "warp"])
def test_out_of_range_selection_is_reported_not_read(sg, kernel):
    """Entries outside [0, b_t] are reported and skipped by either attention kernel (forced
    in both runs: in the routed mode a bad entry can change its unit's routing)."""
    wl = gen.small_workload(T=128, G=1, Hg=16, B=8, k=4)
    inp = _to_cuda(gen.make_inputs(wl, seed=10))
    prm = _prm(sg, wl)
    prm.attn_kernel = sg.ATTN_TC_UNION if kernel == "union" else sg.ATTN_WARP
    res = _gpu_prefill(sg, inp, wl, prm)
    idx = res.sel_idx.clone()
    idx[0, 100, 0] = 1_000_000        # far past the cache
    idx[0, 101, 0] = -7
    out = torch.empty_like(inp.q)
    sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, idx, res.sel_cnt, 0, out)
    assert sg.sgqa_get_device_error() == 6     # SGQA_ERR_DEVICE_BOUNDS
    # rows without a bad index are unaffected
    assert torch.equal(out[:100], res.out[:100]) and torch.equal(out[102:], res.out[102:])


# ---------------------------------------------------------------------------------------
# full-size workloads (sampled rows)
# ---------------------------------------------------------------------------------------

def test_l32k_all_selections_and_sampled_attention(sg):
    wl = gen.WORKLOADS["l32k"]
    inp = gen.make_inputs(wl, seed=0, device="cuda")
    res = _gpu_prefill(sg, inp, wl, _prm(sg, wl))
    attn_rows = sample_rows(wl.T, 1024, seed=0, B=wl.B, k=wl.k)
    _check_prefill(inp, wl, res, np.arange(wl.T), attn_rows=attn_rows)
    del inp, res
    gc.collect()
    torch.cuda.empty_cache()


def test_l128k_sampled_rows(sg):
    """The benchmark's workload and launch configuration (fused prefill, default workspace)."""
    wl = gen.WORKLOADS["l128k"]
    inp = gen.make_inputs(wl, seed=0, device="cuda")
    res = _gpu_prefill(sg, inp, wl, _prm(sg, wl))
    rows = sample_rows(wl.T, 1024, seed=1, B=wl.B, k=wl.k)
    _check_prefill(inp, wl, res, rows)
    del inp, res
    gc.collect()
    torch.cuda.empty_cache()


def test_chunk1m_sampled_rows(sg):
    wl = gen.WORKLOADS["chunk1m"]
    inp = gen.make_inputs(wl, seed=0, device="cuda")
    res = _gpu_prefill(sg, inp, wl, _prm(sg, wl))
    rows = sample_rows(wl.T, 96, seed=2, B=wl.B, k=wl.k, q_start=wl.q_start)
    _check_prefill(inp, wl, res, rows)
    del inp, res
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,k", [(8, 12), (1, 96), (2, 48), (4, 24), (16, 6)])
def test_coverage_from_lse_matches_oracle_coverage(sg, B, k):
    """The coverage diagnostic (and its sweep over block sizes at one token budget):
    exp(LSE_sel - LSE_dense) from the GPU equals the oracle's dense-softmax mass on the
    selected tokens, computed from scratch."""
    wl = gen.small_workload(T=600, G=2, Hg=16, B=B, k=k, planted=True)
    inp = _to_cuda(gen.make_inputs(wl, seed=12))
    prm = _prm(sg, wl)
    res = _gpu_prefill(sg, inp, wl, prm)
    lse_d = torch.empty_like(res.lse)
    out = torch.empty_like(inp.q)
    dummy = torch.zeros((wl.G, wl.T, 1), dtype=torch.int32, device="cuda")
    sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, dummy, dummy[:, :, 0].contiguous(), 0, out, lse_d,
                            dense_mode=True)
    torch.cuda.synchronize()
    cov_gpu = torch.exp(res.lse.double() - lse_d.double()).cpu().numpy()
    d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k)
    kb = oracle.block_index(u16(inp.k_proxy), wl.B, 0, wl.C)
    rows = np.arange(wl.T)
    for g in range(wl.G):
        grp = np.full(wl.T, g, np.int32)
        sel, cnt = oracle.select(d, rows, grp, u16(inp.q_proxy[g]), kb)
        hs = slice(g * wl.Hg, (g + 1) * wl.Hg)
        _, _, cov = oracle.attention(d, rows, grp, u16(inp.q[:, hs]), u16(inp.gate[:, hs]), u16(inp.k), u16(inp.v),
                                     sel, cnt, want_coverage=True)
        np.testing.assert_allclose(cov_gpu[:, hs], cov, atol=3e-3, rtol=0)
        assert np.all(cov[: wl.B * (wl.k - 1)] > 1 - 1e-12)  # rows whose every block is kept
