"""Parity of the union attention kernel (8 query rows per unit over the union of their
selected blocks, tcgen05 with Q and P in tensor memory), of the warp-level kernel, of the
routed mode (each 8-row unit to one of the two by the size of its union) and of the
grouped mode (units drawn from 4,096-row windows in MinHash order) against the oracle.  Each is forced through sgqa_params.attn_kernel, and every case first asserts
through sgqa_attention_kernel that the forced kernel is the one the call launches.  The
routed mode is also checked bit for bit: every unit's output is the union kernel's or the
warp-level kernel's, whichever a host restatement of the routing rule picks."""
import numpy as np
import pytest
import torch

from block_sparse_long_18_b300 import inputs as gen
from parity_util import sample_rows
from test_gpu_parity import _check_prefill, _gpu_prefill, _prm, _to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sg():
    from block_sparse_long_18_b300 import build

    build.build()
    from block_sparse_long_18_b300 import sgqa

    assert torch.cuda.is_available()
    return sgqa


def _run_case(sg, kernel, case, seed=21):
    case = dict(case)
    rows_spec = case.pop("rows", "all")
    gpd = case.pop("gate_per_dim", 1)
    wl = gen.small_workload(**case)
    inp = _to_cuda(gen.make_inputs(wl, seed=seed))
    prm = _prm(sg, wl, gate_per_dim=gpd)
    prm.attn_kernel = kernel
    assert sg.sgqa_attention_kernel(prm, wl.T, wl.q_start) == kernel, case
    gate = inp.gate if gpd else inp.gate[:, :, 0].contiguous()
    res = _gpu_prefill(sg, inp, wl, prm, gate=gate)
    rows = np.arange(wl.T) if rows_spec == "all" else sample_rows(wl.T, rows_spec, 5, wl.B, wl.k, wl.q_start)
    _check_prefill(inp, wl, res, rows, gate_per_dim=gpd, gate_rows_all=gate)
    return wl, inp, res


# Every row checked: ragged T, tiles straddling block edges (q_start % 8 != 0), T < 8, a
# per-head gate, unions of every causal block, and many chunks per unit.
UNION_CASES = [
    dict(T=700, G=2, Hg=16, B=8, k=24, planted=True),
    dict(T=400, G=2, Hg=16, B=8, k=40, q_start=1500, planted=True),
    dict(T=5, G=1, Hg=16, B=8, k=8, q_start=3),
    dict(T=333, G=2, Hg=16, B=8, k=16, q_start=77, gate_per_dim=0),
    dict(T=2048, G=1, Hg=16, B=8, k=512),
    dict(T=1000, G=1, Hg=16, B=8, k=1),
]
# Sampled rows: unions near the 4,096-entry capacity (k = 512 far into the context), the
# 32K-style planted layout, several builder windows, and block indices past 16 bits.
UNION_SAMPLED = [
    dict(T=1024, G=1, Hg=16, B=8, k=512, q_start=60000, planted=True, rows=48),
    dict(T=4096, G=2, Hg=16, B=8, k=512, q_start=8192, planted=True, rows=48),
    # block indices past one builder window (16,384 blocks): four windows per unit
    dict(T=256, G=1, Hg=16, B=8, k=512, q_start=400000, planted=True, rows=32),
    # block indices on both sides of 65,536: entries are offsets inside their window
    dict(T=128, G=1, Hg=16, B=8, k=512, q_start=524160, planted=True, rows=32),
    # the 1M-token chunk position: eight windows, the last blocks of a 1,048,576 context
    dict(T=256, G=1, Hg=16, B=8, k=512, q_start=1048576 - 256, planted=True, rows=40),
]


@pytest.mark.parametrize("case", UNION_CASES, ids=[f"T{c['T']}_k{c['k']}_q{c.get('q_start', 0)}" for c in UNION_CASES])
def test_union_attention_all_rows(sg, case):
    _run_case(sg, sg.ATTN_TC_UNION, case)


@pytest.mark.parametrize("case", UNION_SAMPLED, ids=[f"q{c['q_start']}_T{c['T']}" for c in UNION_SAMPLED])
def test_union_attention_sampled_rows_long_context(sg, case):
    _run_case(sg, sg.ATTN_TC_UNION, case)


@pytest.mark.parametrize("case", UNION_CASES, ids=[f"T{c['T']}_k{c['k']}_q{c.get('q_start', 0)}" for c in UNION_CASES])
def test_routed_attention_all_rows(sg, case):
    _run_case(sg, sg.ATTN_ROUTED, case)


@pytest.mark.parametrize("case", UNION_SAMPLED, ids=[f"q{c['q_start']}_T{c['T']}" for c in UNION_SAMPLED])
def test_routed_attention_sampled_rows_long_context(sg, case):
    _run_case(sg, sg.ATTN_ROUTED, case)


@pytest.mark.parametrize("case", UNION_CASES, ids=[f"T{c['T']}_k{c['k']}_q{c.get('q_start', 0)}" for c in UNION_CASES])
def test_grouped_attention_all_rows(sg, case):
    _run_case(sg, sg.ATTN_GROUPED, case)


@pytest.mark.parametrize("case", UNION_SAMPLED, ids=[f"q{c['q_start']}_T{c['T']}" for c in UNION_SAMPLED])
def test_grouped_attention_sampled_rows_long_context(sg, case):
    _run_case(sg, sg.ATTN_GROUPED, case)


def test_grouped_attention_ragged_windows_all_rows(sg):
    """Rows in three 4,096-row grouping windows, the last one ragged, at a position not a
    multiple of 8: every row against the oracle."""
    _run_case(sg, sg.ATTN_GROUPED, dict(T=9000, G=2, Hg=16, B=8, k=128, q_start=6003, planted=True))


def _route_to_union(sel_idx, sel_cnt, q_start, k):
    """Host restatement of the routing rule: per (group, 8-row unit), the distinct valid
    blocks of its rows' selections (counts clamped to [1, min(k, b_t + 1)], entries outside
    [0, b_t] ignored) against its (row, block) pairs; union iff
    100 * windows * |union| <= 55 * pairs, windows = 16,384-block windows its own blocks reach."""
    G, T, _ = sel_idx.shape
    out = np.zeros((G, (T + 7) // 8), dtype=bool)
    for g in range(G):
        for u in range((T + 7) // 8):
            blocks, pairs = set(), 0
            windows = ((q_start + min(T, u * 8 + 8) - 1) // 8) // 16384 + 1
            for i in range(u * 8, min(T, u * 8 + 8)):
                bt = (q_start + i) // 8
                c = int(sel_cnt[g, i])
                c = 1 if c < 1 else min(c, min(k, bt + 1))
                pairs += c
                blocks.update(int(b) for b in sel_idx[g, i, :c] if 0 <= b <= bt)
            out[g, u] = 100 * windows * len(blocks) <= 55 * pairs
    return out


@pytest.mark.parametrize("case", [dict(T=1024, G=2, Hg=16, B=8, k=512, q_start=60000, planted=True),
                                  dict(T=2000, G=1, Hg=16, B=8, k=128, q_start=20003, planted=True)],
                         ids=["q60000_k512", "q20003_k128"])
def test_routed_units_match_the_chosen_kernel_bit_for_bit(sg, case):
    """Routed mode: each unit's outputs and LSE are exactly those of the kernel the rule
    picks for it (both kernels are deterministic), and the call uses both kernels."""
    wl = gen.small_workload(**case)
    inp = _to_cuda(gen.make_inputs(wl, seed=29))
    res = {}
    for kern in (sg.ATTN_TC_UNION, sg.ATTN_WARP, sg.ATTN_ROUTED):
        prm = _prm(sg, wl)
        prm.attn_kernel = kern
        res[kern] = _gpu_prefill(sg, inp, wl, prm)
    assert torch.equal(res[sg.ATTN_ROUTED].sel_idx, res[sg.ATTN_TC_UNION].sel_idx)
    to_union = _route_to_union(res[sg.ATTN_ROUTED].sel_idx.cpu().numpy(), res[sg.ATTN_ROUTED].sel_cnt.cpu().numpy(),
                               wl.q_start, wl.k)
    assert to_union.any() and (~to_union).any(), "the case should use both kernels"
    out = {kk: r.out.view(wl.T, wl.G, wl.Hg, wl.D) for kk, r in res.items()}
    lse = {kk: r.lse.view(wl.T, wl.G, wl.Hg) for kk, r in res.items()}
    for g in range(wl.G):
        for u in range(to_union.shape[1]):
            src = sg.ATTN_TC_UNION if to_union[g, u] else sg.ATTN_WARP
            rows = slice(u * 8, min(wl.T, u * 8 + 8))
            assert torch.equal(out[sg.ATTN_ROUTED][rows, g], out[src][rows, g]), (g, u, src)
            assert torch.equal(lse[sg.ATTN_ROUTED][rows, g], lse[src][rows, g]), (g, u, src)


@pytest.mark.parametrize("case", UNION_CASES[:3], ids=["T700", "T400_q1500", "T5"])
def test_warp_attention_forced(sg, case):
    """The warp-level kernel stays reachable (and correct) when forced."""
    _run_case(sg, sg.ATTN_WARP, case)


def test_auto_choice_at_128k_and_1m(sg):
    """The grouped mode up to where the routing rule can still pick the union kernel; the
    warp-level kernel alone at the 1M chunk (every unit spans eight windows there)."""
    prm = sg.params()
    assert sg.sgqa_attention_kernel(prm, 131072, 0) == sg.ATTN_GROUPED
    assert sg.sgqa_attention_kernel(prm, 8192, 1040384) == sg.ATTN_WARP


def test_union_attention_wait_timeout_is_reported_and_recoverable(sg):
    """Every bounded wait of the union kernel given no time (limit 0): the launch gives up,
    reports SGQA_ERR_DEVICE_TIMEOUT, drains its copies and MMAs and returns; the next call
    in the same context reproduces the normal output bit for bit."""
    wl = gen.small_workload(T=256, G=2, Hg=16, B=8, k=16, planted=True)
    inp = gen.make_inputs(wl, seed=13, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, k=wl.k, attn_kernel=sg.ATTN_TC_UNION)
    res = sg.prefill(prm, inp.q, inp.k, inp.v, inp.gate, inp.q_proxy, inp.k_proxy)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    out = torch.empty_like(inp.q)
    sg.sgqa_set_wait_timeout_ns(0)
    try:
        sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, res.sel_idx, res.sel_cnt, 0, out)
        err = sg.sgqa_get_device_error()
    finally:
        sg.sgqa_set_wait_timeout_ns(1_000_000_000)
    assert err == 5, err
    sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, res.sel_idx, res.sel_cnt, 0, out)
    assert sg.sgqa_get_device_error() == 0
    assert torch.equal(out, res.out)


def test_grouped_attention_wait_timeout_is_reported_and_recoverable(sg):
    """The grouped mode's launches given no time for any bounded wait: the error is
    reported, nothing hangs, and the next call reproduces the normal output bit for bit."""
    wl = gen.small_workload(T=256, G=2, Hg=16, B=8, k=16, planted=True)
    inp = gen.make_inputs(wl, seed=14, device="cuda")
    prm = sg.params(G=wl.G, Hg=wl.Hg, k=wl.k, attn_kernel=sg.ATTN_GROUPED)
    res = sg.prefill(prm, inp.q, inp.k, inp.v, inp.gate, inp.q_proxy, inp.k_proxy)
    torch.cuda.synchronize()
    assert sg.sgqa_get_device_error() == 0
    ws = torch.empty(sg.sgqa_workspace_bytes(prm, sg.SGQA_OP_ATTN, wl.T, wl.T), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(inp.q)
    sg.sgqa_set_wait_timeout_ns(0)
    try:
        sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, res.sel_idx, res.sel_cnt, 0, out, ws=ws)
        err = sg.sgqa_get_device_error()
    finally:
        sg.sgqa_set_wait_timeout_ns(1_000_000_000)
    assert err == 5, err
    sg.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, res.sel_idx, res.sel_cnt, 0, out, ws=ws)
    assert sg.sgqa_get_device_error() == 0
    assert torch.equal(out, res.out)
