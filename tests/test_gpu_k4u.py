"""Parity of the union attention kernel (8 query rows per unit over the union of their
selected blocks, tcgen05 with Q and P in tensor memory) against the oracle, and of the
warp-level kernel it replaces.  Each is forced through sgqa_params.attn_kernel, and every
case first asserts through sgqa_attention_kernel that the forced kernel is the one the
call launches."""
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


@pytest.mark.parametrize("case", UNION_CASES[:3], ids=["T700", "T400_q1500", "T5"])
def test_warp_attention_forced(sg, case):
    """The warp-level kernel stays reachable (and correct) when forced."""
    _run_case(sg, sg.ATTN_WARP, case)


def test_auto_choice_is_the_union_kernel_at_1m(sg):
    prm = sg.params()
    assert sg.sgqa_attention_kernel(prm, 8192, 1040384) == sg.ATTN_TC_UNION


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
