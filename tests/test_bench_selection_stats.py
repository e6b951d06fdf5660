"""The benchmark's selection statistics (distinct K/V blocks any row selected, union size
of each 8-row unit, and the routing of each unit between the union and the warp-level
attention kernel) against plain Python sets on random selections."""
from types import SimpleNamespace

import numpy as np
import torch

import bench
from block_sparse_long_18_b300 import inputs as gen


def _random_plan(seed, G, T, k, B, q_start):
    rng = np.random.default_rng(seed)
    sel = np.full((G, T, k), -1, np.int32)
    cnt = np.zeros((G, T), np.int32)
    for g in range(G):
        shared = None
        for i in range(T):
            bt = (q_start + i) // B
            n = min(k, bt + 1)
            if i % 8 == 0:  # odd units: every row keeps the same earlier blocks (a small union)
                lo = (q_start + i) // B
                shared = rng.choice(lo, size=min(k, lo + 1) - 1, replace=False)
            if (i // 8) % 2 and n - 1 <= len(shared):
                chosen = shared[:n - 1]
            else:
                chosen = rng.choice(bt, size=n - 1, replace=False) if n > 1 else np.array([], np.int64)
            row = np.sort(np.append(chosen, bt)).astype(np.int32)
            sel[g, i, :n] = row
            cnt[g, i] = n
    return SimpleNamespace(sel_idx=torch.from_numpy(sel), sel_cnt=torch.from_numpy(cnt))


def test_selection_stats_match_sets():
    G, T, k, B, q_start = 2, 64, 12, 8, 8000
    wl = gen.small_workload(T=T, q_start=q_start, B=B, k=k, G=G, Hg=16, P=64)
    plan = _random_plan(7, G, T, k, B, q_start)
    st = bench.selection_stats(plan, wl, units_per_pass=3)  # several passes over the units
    sel, cnt = plan.sel_idx.numpy(), plan.sel_cnt.numpy()
    used = {(g, int(b)) for g in range(G) for i in range(T) for b in sel[g, i, :cnt[g, i]]}
    assert st["kv_blocks_selected"] == len(used)
    sizes, n_union, n_warp = [], 0, 0
    for g in range(G):
        for u in range(T // 8):
            rows = range(8 * u, 8 * u + 8)
            union = {int(b) for i in rows for b in sel[g, i, :cnt[g, i]]}
            pairs = sum(int(cnt[g, i]) for i in rows)
            windows = max((q_start + i) // B for i in rows) // 16384 + 1
            sizes.append(len(union))
            if 100 * windows * len(union) <= 55 * pairs:
                n_union += 1
            else:
                n_warp += 1
    assert st["union_mean_blocks"] == round(sum(sizes) / len(sizes), 1)
    assert st["union_chunks"] == sum((s + 15) // 16 for s in sizes)
    assert (st["routed_union_units"], st["routed_warp_units"]) == (n_union, n_warp)
    assert n_union > 0 and n_warp > 0  # both outcomes of the routing rule occur
