"""The benchmark's algorithmic work per stage (the numerators of every roofline fraction it
prints) against brute-force counts on small shapes, and against the closed-form totals of
the 128K layer: 2.20e12 indexer FLOPs, 17.2 GB of scores, 2.60e13 attention FLOPs and
1.62 TB of per-(row, group) K/V gathers."""
import numpy as np
import pytest

import bench
from block_sparse_long_18_b300 import inputs as gen


def _brute(wl):
    """Loops over (row, group/head, block) straight from the method's definition: the
    indexer scores every strictly earlier block (2P FLOPs each), the selection keeps
    min(k, b_t + 1) blocks, attention reads the kept blocks' tokens up to t (4 D FLOPs per
    token and head: QK and PV)."""
    k2_flop = k4_flop = n_sum = bt_sum = 0
    for t in range(wl.q_start, wl.q_start + wl.T):
        bt = t // wl.B
        n = min(wl.k, bt + 1)
        tokens = (n - 1) * wl.B + (t - bt * wl.B + 1)  # earlier kept blocks are full
        for _ in range(wl.G):
            k2_flop += 2 * wl.P * bt
            bt_sum += bt
            n_sum += n
        for _ in range(wl.H):
            k4_flop += 4 * wl.D * tokens
    return k2_flop, k4_flop, n_sum, bt_sum


@pytest.mark.parametrize("T,q_start,B,k,G,Hg", [(37, 0, 8, 3, 2, 2), (50, 5, 8, 4, 1, 4), (40, 17, 1, 9, 2, 1),
                                                (33, 100, 16, 2, 4, 16), (9, 0, 4, 64, 1, 1)])
def test_work_model_matches_brute_force(T, q_start, B, k, G, Hg):
    wl = gen.small_workload(T=T, q_start=q_start, B=B, k=k, G=G, Hg=Hg, P=64)
    w = bench.work_model(wl)
    k2_flop, k4_flop, n_sum, bt_sum = _brute(wl)
    assert w["k2_flop"] == k2_flop
    assert w["k4_flop"] == k4_flop
    assert w["sum_n"] * wl.G == n_sum and w["sum_bt"] * wl.G == bt_sum  # per-group sums
    assert w["k3_bytes"] == 4 * bt_sum + 4 * n_sum
    assert w["k4_gather_bytes"] == 2 * 2 * wl.D * wl.B * n_sum


def test_work_model_at_128k_matches_the_closed_forms():
    wl = gen.WORKLOADS["l128k"]
    w = bench.work_model(wl)
    assert w["k2_flop"] == pytest.approx(2.20e12, rel=0.01)
    assert 4 * wl.G * w["sum_bt"] == pytest.approx(17.2e9, rel=0.01)  # fp32 scores, all groups
    assert w["k4_flop"] == pytest.approx(2.60e13, rel=0.01)
    assert w["k4_gather_bytes"] == pytest.approx(1.62e12, rel=0.01)
    # and the exact sums behind them: sum over t of floor(t / 8) for t < 131,072, per group
    T = 131072
    per_group = sum((t // 8) for t in range(0, T, 1))
    assert w["sum_bt"] == per_group
