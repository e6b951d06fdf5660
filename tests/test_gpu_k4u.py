"""Parity of the union attention kernel (8 query rows per unit over the union of their
selected blocks, tcgen05 with Q and P in tensor memory) against the oracle, and of the
warp-level kernel it replaces, each forced through SGQA_K4_IMPL.  The library reads the
variable once per process, so every case list runs in a child process, which also asserts
through sgqa_attention_kernel that the forced kernel is the one launched."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
from block_sparse_long_18_b300 import build
build.build()
from block_sparse_long_18_b300 import inputs as gen, sgqa
from parity_util import sample_rows
from test_gpu_parity import _check_prefill, _gpu_prefill, _prm, _to_cuda
want = {want}
for case in {cases!r}:
    case = dict(case)
    rows_spec = case.pop("rows", "all")
    gpd = case.pop("gate_per_dim", 1)
    wl = gen.small_workload(**case)
    inp = _to_cuda(gen.make_inputs(wl, seed=21))
    prm = _prm(sgqa, wl, gate_per_dim=gpd)
    got = sgqa.sgqa_attention_kernel(prm, wl.T, wl.q_start)
    assert got == want, (case, got)
    gate = inp.gate if gpd else inp.gate[:, :, 0].contiguous()
    res = _gpu_prefill(sgqa, inp, wl, prm, gate=gate)
    if rows_spec == "all":
        rows = np.arange(wl.T)
    else:
        rows = sample_rows(wl.T, rows_spec, 5, wl.B, wl.k, wl.q_start)
    _check_prefill(inp, wl, res, rows, gate_per_dim=gpd, gate_rows_all=gate)
    print("case ok", case, flush=True)
print("ok")
"""

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
# 32K-style planted layout, several builder windows, and the largest block index served.
UNION_SAMPLED = [
    dict(T=1024, G=1, Hg=16, B=8, k=512, q_start=60000, planted=True, rows=48),
    dict(T=4096, G=2, Hg=16, B=8, k=512, q_start=8192, planted=True, rows=48),
    # block indices past one builder window (16,384 blocks): four windows per unit
    dict(T=256, G=1, Hg=16, B=8, k=512, q_start=400000, planted=True, rows=32),
    # the last supported block index (65,535): the union tables' 16-bit entries at their limit
    dict(T=128, G=1, Hg=16, B=8, k=512, q_start=524160, planted=True, rows=32),
]


def _run(impl, want, cases):
    env = dict(os.environ, SGQA_K4_IMPL=impl)
    code = CHILD.format(root=ROOT, tests=HERE, want=want, cases=cases)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-3000:] + r.stderr[-3000:]


def test_union_attention_all_rows():
    _run("union", 2, UNION_CASES)


def test_union_attention_sampled_rows_long_context():
    _run("union", 2, UNION_SAMPLED)


def test_warp_attention_forced():
    """The warp-level kernel stays reachable (and correct) when forced."""
    _run("mma", 0, UNION_CASES[:3])


def test_union_attention_wait_timeout_is_reported_and_recoverable():
    """Every bounded wait of the union kernel given no time (limit 0): the launch gives up,
    reports SGQA_ERR_DEVICE_TIMEOUT, drains its copies and MMAs and returns; the next call
    in the same context reproduces the normal output bit for bit."""
    code = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import torch
from block_sparse_long_18_b300 import build
build.build()
from block_sparse_long_18_b300 import inputs as gen, sgqa
wl = gen.small_workload(T=256, G=2, Hg=16, B=8, k=16, planted=True)
inp = gen.make_inputs(wl, seed=13, device="cuda")
prm = sgqa.params(G=wl.G, Hg=wl.Hg, k=wl.k)
assert sgqa.sgqa_attention_kernel(prm, wl.T) == sgqa.ATTN_TC_UNION
res = sgqa.prefill(prm, inp.q, inp.k, inp.v, inp.gate, inp.q_proxy, inp.k_proxy)
torch.cuda.synchronize()
assert sgqa.sgqa_get_device_error() == 0
out = torch.empty_like(inp.q)
sgqa.sgqa_set_wait_timeout_ns(0)
try:
    sgqa.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, res.sel_idx, res.sel_cnt, 0, out)
    err = sgqa.sgqa_get_device_error()
finally:
    sgqa.sgqa_set_wait_timeout_ns(1_000_000_000)
assert err == 5, err
sgqa.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, res.sel_idx, res.sel_cnt, 0, out)
assert sgqa.sgqa_get_device_error() == 0
assert torch.equal(out, res.out)
print("ok")
""".format(root=ROOT, tests=HERE)
    env = dict(os.environ, SGQA_K4_IMPL="union")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-3000:] + r.stderr[-3000:]
