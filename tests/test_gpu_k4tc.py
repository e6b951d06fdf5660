"""Parity of the opt-in tcgen05 attention kernel (keys as the MMA's M, the 16 heads as N;
selected with SGQA_K4_IMPL=tc, blocks of 8 only).  The library reads the variable once per
process, so each case runs in a child process that checks its result against the oracle."""
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
import oracle
from block_sparse_long_18_b300 import build
build.build()
from block_sparse_long_18_b300 import inputs as gen, sgqa
from parity_util import LSE_ABS, check_outputs, u16
wl = gen.small_workload(T={T}, G=2, Hg=16, B=8, k={k}, planted=True, q_start={q_start})
inp = gen.make_inputs(wl, seed=12)
for n in ("q", "k", "v", "gate", "q_proxy", "k_proxy"):
    setattr(inp, n, getattr(inp, n).cuda())
prm = sgqa.params(G=wl.G, Hg=wl.Hg, D=wl.D, P=wl.P, B=wl.B, k=wl.k)
plan = sgqa.PrefillPlan(prm, wl.T, wl.C, wl.q_start)
if wl.q_start:
    sgqa.sgqa_build_block_index(prm, inp.k_proxy, 0, wl.q_start, plan.k_blk)
res = plan.run(inp.q, inp.k, inp.v, inp.gate, inp.q_proxy, inp.k_proxy)
torch.cuda.synchronize()
assert sgqa.sgqa_get_device_error() == 0
d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k)
rows = np.arange(wl.T, dtype=np.int64)
K, V = u16(inp.k), u16(inp.v)
kb = oracle.block_index(u16(inp.k_proxy), wl.B, 0, wl.C)
for g in range(wl.G):
    pos = wl.q_start + rows
    grp = np.full(len(rows), g, np.int32)
    sel, cnt = oracle.select(d, pos, grp, u16(inp.q_proxy[g]), kb)
    hs = slice(g * wl.Hg, (g + 1) * wl.Hg)
    out, lse = oracle.attention(d, pos, grp, u16(inp.q[:, hs]), u16(inp.gate[:, hs]), K, V, sel, cnt)
    check_outputs(u16(res.out[:, hs]), out, "group %d out" % g)
    assert np.max(np.abs(res.lse[:, hs].cpu().numpy() - lse)) <= LSE_ABS
print("ok")
"""


@pytest.mark.parametrize("T,k,q_start", [(700, 24, 0), (400, 40, 1500)])
def test_tcgen05_attention_matches_oracle(T, k, q_start):
    env = dict(os.environ, SGQA_K4_IMPL="tc")
    code = CHILD.format(root=ROOT, tests=HERE, T=T, k=k, q_start=q_start)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
