"""The benchmark's restatement of the grouped attention mode's row order (torch, with
packed 64-bit sort keys) against a plain Python one: per group and window of rows, sort the
rows by (least MurmurHash3-finalized block index, high bits of the least hash of the
indices xor 0x5bd1e995, row).  The packed keys flip the sign bit to sort unsigned values
with a signed sort; a slip there reorders rows, which this catches."""
import numpy as np
import torch

import bench
from block_sparse_long_18_b300 import inputs as gen


def _fmix32(h: int) -> int:
    """MurmurHash3's 32-bit finalizer (Appleby, public domain), in Python integers."""
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h ^= h >> 16
    return h


def _python_order(sel, cnt, q_start, B, k, win):
    G, T, _ = sel.shape
    row_bits = win.bit_length() - 1
    perm = np.empty((G, T), np.int64)
    for g in range(G):
        keys = []
        for i in range(T):
            bt = (q_start + i) // B
            c = int(cnt[g, i])
            c = 1 if c < 1 else min(c, bt + 1, k)
            blocks = [int(b) for b in sel[g, i, :c] if 0 <= b <= bt]
            h1 = min((_fmix32(b) for b in blocks), default=0xFFFFFFFF)
            h2 = min((_fmix32(b ^ 0x5BD1E995) for b in blocks), default=0xFFFFFFFF)
            keys.append((i // win, h1, h2 >> row_bits, i))
        perm[g] = [key[3] for key in sorted(keys)]
    return perm


def test_grouped_order_matches_python():
    rng = np.random.default_rng(9)
    G, T, k, B, q_start, win = 2, 200, 6, 8, 4000, 64  # four windows, the last partial
    sel = np.full((G, T, k), -1, np.int32)
    cnt = np.zeros((G, T), np.int32)
    pool = [np.sort(rng.choice(q_start // B, size=k - 1, replace=False)) for _ in range(5)]
    for g in range(G):
        for i in range(T):
            bt = (q_start + i) // B
            earlier = pool[rng.integers(5)] if rng.random() < 0.5 else np.sort(rng.choice(bt, size=k - 1, replace=False))
            sel[g, i] = np.append(earlier, bt)
            cnt[g, i] = k
    wl = gen.small_workload(T=T, q_start=q_start, B=B, k=k, G=G, Hg=16, P=64)
    got = bench.grouped_row_order(torch.from_numpy(sel), torch.from_numpy(cnt), wl, win=win).numpy()
    want = _python_order(sel, cnt, q_start, B, k, win)
    assert np.array_equal(got, want)
    for g in range(G):  # a permutation that keeps every row in its window
        assert np.array_equal(np.sort(got[g]), np.arange(T))
        assert np.array_equal(got[g] // win, np.arange(T) // win)
