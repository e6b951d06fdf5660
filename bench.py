#!/usr/bin/env python3
"""Benchmark of the Sparse GQA layer: prefill tokens/s per layer at 128K tokens on B300,
with the roofline fraction of each stage.

One step = one prefill of the whole layer over one batch of synthetic input (block index
-> indexer + top-k -> gated sparse attention) for T = 131,072 query tokens, 4 KV groups x
16 heads, head_dim 192, proxy_dim 256, block 8, top-k 512 blocks.  Inputs are resident in
HBM when the timed region starts; L2 is flushed (a 256 MB write, twice the L2 size)
before every step, outside the step's event pair.  The three stages are called through
the C ABI one after another on one stream with CUDA events between them (the same kernel
sequence as the fused sgqa_prefill entry), so each stage's device time comes from the
timed steps themselves.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sgqa|reference]

Under torchrun each rank runs its own layer on its own seeded input (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Sparse GQA prefill tokens/s per layer @128K (1×B300); % of roofline per stage"
HBM_FALLBACK_GBS, BF16_FALLBACK_TFS = 6400.0, 1800.0

K4_KERNEL = {1: "k4_sparse_attn", 2: "k4u_sparse_attn", 3: "k4r_count + k4r_compact + k4_sparse_attn + k4u_sparse_attn",
             4: "k4g_signature + k4g_sort + k4r_count + k4r_compact + k4_sparse_attn + k4u_sparse_attn"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None, "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFS, 1400.0, "fallback"


# ---------------------------------------------------------------------------------------
# algorithmic work of each stage (what the method must move or compute)
# ---------------------------------------------------------------------------------------

def work_model(wl):
    T, q0, B, k, G, H, D, P = wl.T, wl.q_start, wl.B, wl.k, wl.G, wl.H, wl.D, wl.P
    t = np.arange(q0, q0 + T, dtype=np.int64)
    bt = t // B
    n = np.minimum(k, bt + 1)                     # kept blocks per (row, group)
    att = B * (n - 1) + (t % B) + 1               # attended tokens (own block causally cut)
    sum_bt, sum_n, sum_att = int(bt.sum()), int(n.sum()), int(att.sum())
    NB_new = (q0 + T + B - 1) // B - q0 // B
    w = {}
    w["k1_bytes"] = 2 * G * P * (T + NB_new)
    w["k2_flop"] = 2 * P * G * sum_bt
    w["k2_bytes"] = G * P * 2 * (T + (q0 + T) // B) + 4 * G * sum_bt
    w["k3_bytes"] = 4 * G * sum_bt + 4 * G * sum_n
    w["k4_flop"] = 4 * D * H * sum_att
    # per-(row, group) gathers: every kept block read once per row that keeps it (a line
    # for a kernel that gathers per row; one that shares gathers across rows moves far less)
    w["k4_gather_bytes"] = 2 * 2 * D * B * G * sum_n
    # bytes every K4 must move: Q, gate and O once, the selection and LSE once, and K/V of
    # every block some row selected once (set by the caller from the selection, else every
    # causal block of the context)
    w["k4_rows_bytes"] = 3 * 2 * T * H * D + 4 * G * sum_n + 4 * G * T + 4 * T * H
    w["k4_kv_once_bytes"] = 2 * 2 * D * B * G * ((q0 + T + B - 1) // B)
    w["sum_n"] = sum_n
    w["sum_bt"] = sum_bt
    return w


_I64_MIN = -(1 << 63)


GROUP_WINDOW = 4096  # rows per grouping window of the library's grouped attention mode
FILTERED_MIN_CAND = 16384  # rows past this many candidates take the library's bound-filtered top-k


def _murmur32(x):
    """The 32-bit MurmurHash3 finalizer on int64 tensors holding 32-bit words, as the
    library's grouping kernel applies it."""
    m = 0xFFFFFFFF
    x = x ^ (x >> 16)
    x = (x * 0x85ebca6b) & m
    x = x ^ (x >> 13)
    x = (x * 0xc2b2ae35) & m
    return x ^ (x >> 16)


def grouped_row_order(sel, cnt, wl, win=GROUP_WINDOW):
    """The grouped attention mode's row order, restated with torch for the benchmark's
    routing statistics: per group and window of `win` rows, the rows sorted by (the least
    32-bit hash of their selected blocks, high bits of a second such hash, row).  Returns
    perm [G, T] (the row at each slot)."""
    G, T, k = sel.shape
    dev = sel.device
    perm = torch.empty((G, T), dtype=torch.int64, device=dev)
    i = torch.arange(T, device=dev)
    bt = (wl.q_start + i) // wl.B
    cap = torch.clamp(bt + 1, max=k)
    j = torch.arange(k, device=dev)
    row_bits = win.bit_length() - 1
    for g in range(G):
        c = cnt[g].long()
        c = torch.where(c < 1, torch.ones_like(c), torch.minimum(c, cap))
        b = sel[g].long()
        valid = (j[None, :] < c[:, None]) & (b >= 0) & (b <= bt[:, None])
        big = torch.full_like(b, 1 << 32)
        h1 = torch.where(valid, _murmur32(b & 0xFFFFFFFF), big).amin(dim=1).clamp(max=0xFFFFFFFF)
        h2 = torch.where(valid, _murmur32((b & 0xFFFFFFFF) ^ 0x5bd1e995), big).amin(dim=1).clamp(max=0xFFFFFFFF)
        # (h1 << 32 | ...) compared as unsigned: flip the sign bit for torch's signed sort
        key = ((h1 << 32) | ((h2 >> row_bits) << row_bits) | (i % win)) ^ _I64_MIN
        nwin = (T + win - 1) // win
        pad = nwin * win - T
        keyw = torch.cat([key, torch.full((pad,), (1 << 63) - 1, device=dev, dtype=torch.int64)])
        srt, _ = torch.sort(keyw.view(nwin, win), dim=1)
        order = ((srt ^ _I64_MIN) & (win - 1)) + torch.arange(nwin, device=dev)[:, None] * win
        perm[g] = order.reshape(-1)[:T]
        del b, valid, big
    return perm


def selection_stats(plan, wl, units_per_pass=4096, grouped=False):
    """From the step's selection: how many distinct (group, block) pairs some row selected
    (the K/V every attention kernel must read at least once), and for units of 8 rows (8
    consecutive rows, or with grouped=True the grouped mode's units) the size of each
    union, the library's routing of the unit, and the MMA work each kernel issues."""
    if wl.T % 8:
        return None
    sel = plan.sel_idx  # [G, T, k], ascending, -1 padded
    cnt_rows = plan.sel_cnt
    G, T, k = sel.shape
    if grouped:
        perm = grouped_row_order(sel, cnt_rows, wl)
        sel = torch.stack([sel[g][perm[g]] for g in range(G)])
        cnt_rows = torch.stack([cnt_rows[g][perm[g]] for g in range(G)])
    nb = (wl.q_start + wl.T + wl.B - 1) // wl.B
    used = torch.zeros((G, nb + 1), dtype=torch.bool, device=sel.device)
    chunks = r_chunks = r_stages = r_union = r_warp = 0
    blocks = 0
    units = sel.reshape(G, T // 8, 8 * k)
    cnt = cnt_rows.reshape(G, T // 8, 8).sum(dim=-1)  # (row, block) pairs per unit
    # the largest own block of each unit (windows of 16,384 blocks it spans)
    pos = wl.q_start + (perm if grouped else torch.arange(T, device=sel.device).expand(G, T))
    bmax = (pos // wl.B).reshape(G, T // 8, 8).amax(dim=-1)
    for u0 in range(0, T // 8, units_per_pass):
        part = units[:, u0:u0 + units_per_pass]
        srt, _ = torch.sort(part, dim=-1)
        valid = srt >= 0
        new = valid.clone()
        new[..., 1:] &= srt[..., 1:] != srt[..., :-1]
        nu = new.sum(dim=-1)  # [G, units]: distinct blocks
        pairs = cnt[:, u0:u0 + units_per_pass]
        # the library's routing rule: union iff 100 * windows * |union| <= 55 * pairs
        windows = bmax[:, u0:u0 + units_per_pass] // 16384 + 1
        to_union = 100 * windows * nu <= 55 * pairs
        blocks += int(nu.sum())
        chunks += int(((nu + 15) // 16).sum())
        r_chunks += int(((nu + 15) // 16)[to_union].sum())
        r_stages += int(((cnt_rows.reshape(G, T // 8, 8)[:, u0:u0 + units_per_pass] + 1) // 2)[~to_union].sum())
        r_union += int(to_union.sum())
        r_warp += int((~to_union).sum())
        for g in range(G):
            used[g].index_fill_(0, (srt[g][valid[g]]).long(), True)
        del srt, valid, new
    n_units = G * (T // 8)
    return {"kv_blocks_selected": int(used.sum()), "union_chunks": chunks,
            "union_mean_blocks": round(blocks / n_units, 1), "routed_union_chunks": r_chunks,
            "routed_warp_stages": r_stages, "routed_union_units": r_union, "routed_warp_units": r_warp}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                pw.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample of the workload
# ---------------------------------------------------------------------------------------

def cpu_oracle_rate(inp_host, wl, n_rows, seed=0, kb_t=None):
    """Oracle time for n_rows query tokens (all groups: indexer + top-k + attention), plus
    its block-index pass prorated to those rows.  kb_t: a block index already built by the
    oracle and the seconds it took (reused across samples).  Returns (tokens/s, seconds,
    rows, cores)."""
    import oracle

    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(wl.T, size=n_rows, replace=False)).astype(np.int64)
    d = oracle.dims(wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.k)
    if kb_t is None:
        t0 = time.perf_counter()
        kb = oracle.block_index(inp_host["k_proxy"], wl.B, 0, wl.C)
        t_k1 = time.perf_counter() - t0
    else:
        kb, t_k1 = kb_t
    t0 = time.perf_counter()
    for g in range(wl.G):
        pos = wl.q_start + rows
        grp = np.full(len(rows), g, np.int32)
        sel, cnt = oracle.select(d, pos, grp, inp_host["q_proxy"][g][rows], kb)
        hs = slice(g * wl.Hg, (g + 1) * wl.Hg)
        oracle.attention(d, pos, grp, inp_host["q"][rows][:, hs], inp_host["gate"][rows][:, hs], inp_host["k"],
                         inp_host["v"], sel, cnt)
    t_rows = time.perf_counter() - t0
    secs = t_rows + t_k1 * len(rows) / wl.T
    return len(rows) / secs, secs, len(rows), oracle.num_threads()


def host_views(inp, rows_needed=None):
    """uint16 host copies of what the oracle reads (whole K/V/k_proxy; q/gate/q_proxy rows)."""
    def u16(t):
        return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    return {"k": u16(inp.k), "v": u16(inp.v), "k_proxy": u16(inp.k_proxy), "q": u16(inp.q), "gate": u16(inp.gate),
            "q_proxy": u16(inp.q_proxy)}


# ---------------------------------------------------------------------------------------
# multi-rank bookkeeping (one process per GPU, replicas of the layer, no data exchange)
# ---------------------------------------------------------------------------------------

def max_over_ranks(x: float, world: int, device=None) -> float:
    """The job's step time is the slowest rank's: all-reduce MAX (gloo on CPU, nccl on GPU)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own tokens_per_rank per step."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


# ---------------------------------------------------------------------------------------
# coverage diagnostic
# ---------------------------------------------------------------------------------------

# Block sizes and selection budgets of the coverage sweep: every block size the kernels
# support at the layer's token budget (B x k = 4,096 tokens), plus single tokens at k = 2,048
# (the pages' token-level comparison point).
COVERAGE_SWEEP = ((8, 512), (1, 2048), (1, 4096), (2, 2048), (4, 1024), (16, 256))


def coverage_diagnostic(sgqa, gen, wl, inp, plan, dev, window=1024):
    """Token coverage on the last `window` query rows: mean over (row, head) of the dense
    causal softmax mass on the selected tokens, exp(LSE_sel - LSE_dense), for each block
    size B and budget k of COVERAGE_SWEEP (block index, indexer + top-k and attention rerun
    at that B on the same inputs).  Also times the indexer + top-k of every setting on the
    window (the pages' claim that token-level indexing costs about 8x).  The pages' own
    figures (78.06 % / 79.09 %) come from the vendor's model and data and are context only."""
    T, r0 = wl.T, wl.T - window
    G, H = wl.G, wl.H
    prm8 = sgqa.params(G=G, Hg=wl.Hg, D=wl.D, P=wl.P, B=8, k=wl.k)
    q, gate = inp.q[r0:], inp.gate[r0:]
    lse_d = torch.empty((window, H), dtype=torch.float32, device=dev)
    out = torch.empty_like(q)
    dummy = torch.zeros((G, window, 1), dtype=torch.int32, device=dev)
    sgqa.sgqa_sparse_attn_fwd(prm8, q, inp.k, inp.v, gate, dummy, dummy[:, :, 0].contiguous(), r0, out, lse_d,
                              dense_mode=True)
    qp = inp.q_proxy[:, r0:].contiguous()
    sweep, same8 = [], None
    for B, k in COVERAGE_SWEEP:
        prm = sgqa.params(G=G, Hg=wl.Hg, D=wl.D, P=wl.P, B=B, k=k)
        nb = (T + B - 1) // B
        kb = torch.empty((G, nb, wl.P), dtype=inp.k_proxy.dtype, device=dev)
        sgqa.sgqa_build_block_index(prm, inp.k_proxy, 0, T, kb)
        idx = torch.empty((G, window, k), dtype=torch.int32, device=dev)
        cnt = torch.empty((G, window), dtype=torch.int32, device=dev)
        ws = torch.empty(sgqa.sgqa_workspace_bytes(prm, sgqa.SGQA_OP_INDEX_TOPK, window, T), dtype=torch.uint8,
                         device=dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for rep in range(2):  # the first pass warms up
            ev[0].record()
            sgqa.sgqa_index_topk(prm, qp, r0, kb, idx, cnt, ws)
            ev[1].record()
        lse = torch.empty((window, H), dtype=torch.float32, device=dev)
        sgqa.sgqa_sparse_attn_fwd(prm, q, inp.k, inp.v, gate, idx, cnt, r0, out, lse)
        torch.cuda.synchronize(dev)
        cov = torch.exp(lse.double() - lse_d.double())
        if B == 8 and k == wl.k:
            same8 = bool(torch.equal(idx, plan.sel_idx[:, r0:]))
        sweep.append({"B": B, "k": k, "tokens": B * k, "coverage": round(float(cov.mean()), 5),
                      "index_topk_ms_window": round(ev[0].elapsed_time(ev[1]), 3)})
        del kb, idx, ws
    by = {(e["B"], e["k"]): e for e in sweep}
    return {
        "rows": f"last {window} query rows of the {wl.name} workload, all {H} heads",
        "b8_k512_blocks": by[(8, 512)]["coverage"],
        "b1_k2048_tokens": by[(1, 2048)]["coverage"],
        "index_topk_ms_window": {"b8_k512": by[(8, 512)]["index_topk_ms_window"],
                                 "b1_k2048": by[(1, 2048)]["index_topk_ms_window"],
                                 "ratio_b1_over_b8": round(by[(1, 2048)]["index_topk_ms_window"] /
                                                           by[(8, 512)]["index_topk_ms_window"], 2)},
        "sweep": sweep,
        "window_selection_matches_full_run": same8,
        "pages_context_only": {"b8_k4096_tokens_pct": 78.06, "b1_k2048_tokens_pct": 79.09},
    }


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------

def run_sgqa(args, rank, world, local_rank):
    from block_sparse_long_18_b300 import build as _build

    _build.build()
    from block_sparse_long_18_b300 import inputs as gen
    from block_sparse_long_18_b300 import sgqa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = gen.WORKLOADS[args.workload]
    hbm, bf16, bf16_sus, peak_src = load_peaks()
    inp = gen.make_inputs(wl, seed=rank, device=dev)
    prm = sgqa.params(G=wl.G, Hg=wl.Hg, D=wl.D, P=wl.P, B=wl.B, k=wl.k)
    plan = sgqa.PrefillPlan(prm, wl.T, wl.C, wl.q_start, device=dev)
    if wl.q_start:
        sgqa.sgqa_build_block_index(prm, inp.k_proxy, 0, wl.q_start, plan.k_blk)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        sgqa.sgqa_build_block_index(prm, inp.k_proxy, wl.q_start, wl.q_start + wl.T, plan.k_blk, stream)
        if evs:
            evs[1].record(stream)
        sgqa.sgqa_index_topk(prm, inp.q_proxy, wl.q_start, plan.k_blk, plan.sel_idx, plan.sel_cnt, plan.ws, stream)
        if evs:
            evs[2].record(stream)
        sgqa.sgqa_sparse_attn_fwd(prm, inp.q, inp.k, inp.v, inp.gate, plan.sel_idx, plan.sel_cnt, wl.q_start,
                                  plan.out, plan.lse, stream=stream, ws=plan.ws)
        if evs:
            evs[3].record(stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    err = sgqa.sgqa_get_device_error()
    if err:
        raise RuntimeError(f"device error {err} during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        t_wall0 = time.perf_counter()
        for s in range(args.steps):
            flush.fill_(s & 0xFF)
            step(events[s])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    err = sgqa.sgqa_get_device_error()
    if err:
        raise RuntimeError(f"device error {err} in the timed region")
    stage_ms = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in events])  # [steps, 3]
    step_ms = stage_ms.sum(axis=1)
    ms = max_over_ranks(float(step_ms.mean()), world, dev)
    value = job_value(wl.T, world, ms)

    # ---- roofline of each stage (max of its FLOPs at the bf16 peak and its algorithmic
    # bytes at the HBM peak, both peaks measured on B300) ----
    w = work_model(wl)
    attn_kind = sgqa.sgqa_attention_kernel(prm, wl.T, wl.q_start)
    sel_stats = selection_stats(plan, wl, grouped=attn_kind == sgqa.ATTN_GROUPED)
    if sel_stats is not None:
        w["k4_kv_once_bytes"] = sel_stats["kv_blocks_selected"] * 2 * 2 * wl.D * wl.B
    k4_compulsory = w["k4_rows_bytes"] + w["k4_kv_once_bytes"]
    k1_ms, ik_ms, k4_ms = (float(x) for x in stage_ms.mean(axis=0))
    hbm_bps, tf = hbm * 1e9, bf16 * 1e12
    k2_scores_bytes = 4 * wl.G * w["sum_bt"]
    roof = {
        "k1_block_index": w["k1_bytes"] / hbm_bps * 1e3,
        "k2k3_index_topk": (max(w["k2_flop"] / tf, w["k2_bytes"] / hbm_bps) + w["k3_bytes"] / hbm_bps) * 1e3,
        "k4_sparse_attn": max(w["k4_flop"] / tf, k4_compulsory / hbm_bps) * 1e3,
    }
    meas = {"k1_block_index": k1_ms, "k2k3_index_topk": ik_ms, "k4_sparse_attn": k4_ms}
    stages = {kname: {"ms": round(meas[kname], 4), "roofline_ms": round(roof[kname], 4),
                      "frac": round(roof[kname] / meas[kname], 4)} for kname in meas}
    stages["k1_block_index"]["bound"] = "hbm"
    stages["k2k3_index_topk"]["bound"] = "hbm (scores written by the indexer and read by the top-k)"
    stages["k2k3_index_topk"]["k2_tflop"] = round(w["k2_flop"] / 1e12, 4)
    stages["k2k3_index_topk"]["score_bytes"] = k2_scores_bytes
    # secondary: scores never leaving the SM (operands, selection out, FLOPs at peak)
    fused_floor = max(w["k2_flop"] / tf, (w["k2_bytes"] - k2_scores_bytes + 4 * wl.G * w["sum_n"]) / hbm_bps) * 1e3
    stages["k2k3_index_topk"]["fused_floor_ms"] = round(fused_floor, 4)
    if wl.q_start // wl.B > FILTERED_MIN_CAND and (wl.q_start + wl.T - 1) // wl.B <= 8 * 16384:
        # every row takes the library's bound-filtered path, which writes no score matrix:
        # the stage's line is then the fused floor (its FLOPs at the bf16 peak, operands and
        # selection once), not the materialised-score line
        roof["k2k3_index_topk"] = fused_floor
        stages["k2k3_index_topk"].update(
            roofline_ms=round(fused_floor, 4), frac=round(fused_floor / ik_ms, 4),
            bound="tensor (bound-filtered selection: no score matrix written; FLOPs of one indexer pass at the bf16 peak)")
    k4s = stages["k4_sparse_attn"]
    k4s["bound"] = "tensor" if w["k4_flop"] / tf >= k4_compulsory / hbm_bps else "hbm"
    k4s["useful_tflop"] = round(w["k4_flop"] / 1e12, 3)
    k4s["useful_tflops"] = round(w["k4_flop"] / (k4_ms / 1e3) / 1e12, 2)
    k4s["compulsory_bytes"] = k4_compulsory
    k4s["frac_vs_sustained_peak"] = (round(max(w["k4_flop"] / (bf16_sus * 1e12), k4_compulsory / hbm_bps) * 1e3
                                           / k4_ms, 4) if bf16_sus else None)
    # secondary lines: the per-(row, group) gather bytes (how much the kernel's sharing of
    # gathers saves) and, for the union kernel, the MMA work it issues including the
    # (row, head) pairs masked out of a union block
    k4s["per_row_gather_bytes"] = w["k4_gather_bytes"] + w["k4_rows_bytes"]
    k4s["per_row_gather_frac_of_hbm"] = round(k4s["per_row_gather_bytes"] / (k4_ms / 1e3) / hbm_bps, 4)
    k4_kernel = K4_KERNEL.get(sgqa.sgqa_attention_kernel(prm, wl.T, wl.q_start), "k4_sparse_attn")
    if sel_stats is not None and ("k4r_count" in k4_kernel):
        # routed: units whose union is small go to the union kernel, the rest to the
        # warp-level kernel (16 heads x 16 keys x 192 x 4 per stage of two blocks)
        issued = (sel_stats["routed_union_chunks"] * 128 * 128 * wl.D * 4
                  + sel_stats["routed_warp_stages"] * 16 * 16 * wl.D * 4)
        k4s["union_mean_blocks"] = sel_stats["union_mean_blocks"]
        k4s["units_to_union_kernel"] = sel_stats["routed_union_units"]
        k4s["units_to_warp_kernel"] = sel_stats["routed_warp_units"]
        k4s["issued_mma_tflop"] = round(issued / 1e12, 3)
        k4s["issued_tflops"] = round(issued / (k4_ms / 1e3) / 1e12, 2)
        k4s["useful_share_of_issued"] = round(w["k4_flop"] / issued, 4)
    elif sel_stats is not None and k4_kernel == "k4u_sparse_attn":
        issued = sel_stats["union_chunks"] * 128 * 128 * wl.D * 4
        k4s["union_mean_blocks"] = sel_stats["union_mean_blocks"]
        k4s["issued_mma_tflop"] = round(issued / 1e12, 3)
        k4s["issued_tflops"] = round(issued / (k4_ms / 1e3) / 1e12, 2)
        k4s["useful_share_of_issued"] = round(w["k4_flop"] / issued, 4)
    layer_roof = sum(roof.values())

    roofline = {
        "kernel": k4_kernel,
        "bound": k4s["bound"],
        "achieved": k4s["useful_tflops"] if k4s["bound"] == "tensor" else round(k4_compulsory / (k4_ms / 1e3) / 1e9, 1),
        "peak": bf16 if k4s["bound"] == "tensor" else hbm,
        "unit": "TFLOP/s" if k4s["bound"] == "tensor" else "GB/s",
        "frac": k4s["frac"],
        "traffic": None,
        "algorithmic": {"useful_flop_per_launch": w["k4_flop"], "compulsory_bytes_per_launch": k4_compulsory},
        "peak_source": f"{peak_src}: bf16 burst (kernel timed alone by its own events)",
        "frac_vs_sustained_peak": k4s["frac_vs_sustained_peak"],
    }

    # ---- end to end through the public API, from pinned host memory ----
    e2e = None
    if not args.no_e2e:
        hp = sgqa.HostPrefill(prm, wl.T, wl.C, wl.q_start, device=dev)
        host = {name: getattr(inp, name).cpu().pin_memory() for name in ("q", "k", "v", "gate", "q_proxy", "k_proxy")}
        for _ in range(max(1, min(args.warmup, 2))):
            hp.run(host)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for s in range(args.steps):
            ev[s][0].record(stream)
            hp.run(host)
            ev[s][1].record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev])), world, dev)
        e2e = {"value": job_value(wl.T, world, e_ms), "unit": "tokens/s", "ms_per_step": round(e_ms, 3),
               "h2d_bytes_per_step": hp.h2d_bytes(), "d2h_bytes_per_step": hp.d2h_bytes(),
               "api": "sgqa_prefill_host (C ABI): pinned host buffers in and out, 4,096-row chunks pipelined by the "
                      "library over its copy-in stream, the calling stream and its copy-out stream"}
        del hp, host

    # ---- CPU baseline (oracle), rank 0 only ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        hv = host_views(inp)
        rate, secs, nrows, cores = cpu_oracle_rate(hv, wl, n_rows=16)
        for attempt in range(3):  # grow the sample towards ~15 s of CPU work
            if secs >= 10.0 or nrows >= wl.T:
                break
            n2 = int(min(wl.T, max(nrows + 1, nrows * 15.0 / max(secs, 1e-3))))
            rate, secs, nrows, cores = cpu_oracle_rate(hv, wl, n_rows=n2, seed=1 + attempt)
        cpu = {"value": round(rate, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
               "nproc": os.cpu_count(),
               "sample": f"{nrows} query tokens drawn uniformly from the {wl.name} workload, all {wl.G} groups "
                         f"(indexer + top-k + attention, fp64) plus the block-index pass prorated; {secs:.1f} s"}

    # ---- coverage diagnostic (rank 0): dense-softmax mass captured by the selection ----
    coverage = None
    if rank == 0 and not args.no_coverage and wl.q_start == 0 and wl.B == 8:
        coverage = coverage_diagnostic(sgqa, gen, wl, inp, plan, dev)

    # ---- decode step (rank 0, one GPU): the decode workload's latency and roofline ----
    decode = None
    if rank == 0 and world == 1 and not args.no_decode:
        del plan
        torch.cuda.empty_cache()
        decode = decode_section(args.steps, args.warmup, dev)

    # K1 once, K2 + top-k per 8,192-row pass (top-k in two launches for rows past 16,384
    # candidates: per-slice selection, then the merge), K4 once
    # (the routed attention: two routing launches and the warp-level kernel besides the union
    # one; the grouped mode two more for the row order)
    kind = sgqa.sgqa_attention_kernel(prm, wl.T, wl.q_start)
    launches_per_step = 2 + {sgqa.ATTN_ROUTED: 3, sgqa.ATTN_GROUPED: 5}.get(kind, 0)
    # per indexer + top-k pass: the indexer and one top-k launch (two for rows past 16,384
    # candidates: slices and merge); a bound-filtered pass (the default workspace holds its
    # buffers) six: indexer maxima, bounds, indexer survivors, selection, and the two
    # launches for rows with too many survivors (they return at once when none has)
    need = wl.k - 1
    max_cand = (wl.q_start + wl.T - 1) // wl.B
    filtered_fits = wl.k >= 2 and need <= 4096 and 8 * need < max_cand <= 8 * 16384
    for r0 in range(0, wl.T, 8192):
        cand_last = (wl.q_start + min(wl.T, r0 + 8192) - 1) // wl.B
        if filtered_fits and (wl.q_start + r0) // wl.B > max(8 * need, FILTERED_MIN_CAND):
            launches_per_step += 6
        else:
            launches_per_step += (1 if cand_last > 0 else 0) + (2 if cand_last > 16384 and wl.k > 1 else 1)
    clocks = clk.summary()
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{wl.name}: prefill T={wl.T} at q_start={wl.q_start}, context {wl.C}, G={wl.G} x Hg={wl.Hg} "
                        f"heads, D={wl.D}, P={wl.P}, block {wl.B}, top-k {wl.k} blocks, planted={wl.planted}",
            "global_batch": 1, "seq_len": wl.T, "parallelism": f"replicas x{world}",
            "l2": "flushed before every step (256 MB write, outside the step events)",
            "wall_ms_per_step_incl_flush": round(t_wall * 1e3 / args.steps, 3),
        },
        "stages": stages,
        "layer_roofline_ms": round(layer_roof, 4),
        "layer_roofline_note": "sum of the stage rooflines (K1 bytes; K2+K3 materialised scores; K4 max of useful "
                               "FLOPs at the bf16 peak and compulsory bytes at HBM) over the step time",
        "layer_roofline_frac": round(layer_roof / ms, 4),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "coverage": coverage,
        "decode": decode,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16_sus, "source": peak_src},
    }
    return out


# ---------------------------------------------------------------------------------------
# decode step timing (not the headline metric; reported for the decode workload)
# ---------------------------------------------------------------------------------------

def decode_measure(sgqa, wl, inp, dev, steps, warmup, fp8=False):
    """Decode step latency over one set of decode inputs; with fp8 the block-proxy cache is
    FP8 E4M3 (sgqa_decode_fp8).  L2 is flushed before every step."""
    prm = sgqa.params(G=wl.G, Hg=wl.Hg, D=wl.D, P=wl.P, B=wl.B, k=wl.k)
    total = inp.k.shape[1]
    batch = len(inp.ctx_len)
    k_blk = torch.zeros((wl.G, total // wl.B, wl.P), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    build_idx = sgqa.sgqa_build_block_index_fp8 if fp8 else sgqa.sgqa_build_block_index
    decode = sgqa.sgqa_decode_fp8 if fp8 else sgqa.sgqa_decode
    for L, off in zip(inp.ctx_len, inp.kv_off):
        build_idx(prm, inp.k_proxy, off, off + L - 1, k_blk)
    sel = torch.empty((wl.G, batch, wl.k), dtype=torch.int32, device=dev)
    cnt = torch.empty((wl.G, batch), dtype=torch.int32, device=dev)
    out = torch.empty((batch, wl.H, wl.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((batch, wl.H), dtype=torch.float32, device=dev)
    ws = torch.empty(sgqa.sgqa_workspace_bytes(prm, sgqa.SGQA_OP_DECODE, 1, max(inp.ctx_len), batch),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        decode(prm, inp.ctx_len, inp.kv_off, inp.q, inp.q_proxy, inp.gate, inp.k, inp.v, inp.k_proxy,
               k_blk, sel, cnt, out, lse, ws)

    for _ in range(warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s in range(steps):
        flush.fill_(s & 0xFF)
        ev[s][0].record()
        step()
        ev[s][1].record()
    torch.cuda.synchronize(dev)
    if sgqa.sgqa_get_device_error():
        raise RuntimeError("device error in decode")
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    nb = sum((L - 1) // wl.B for L in inp.ctx_len)           # blocks scored per group
    idx_bytes = wl.G * nb * wl.P * (1 if fp8 else 2)
    gather = wl.G * sum(min(wl.k, (L - 1) // wl.B + 1) for L in inp.ctx_len) * wl.B * wl.D * 2 * 2
    hbm, _, _, src = load_peaks()
    roof_bytes = idx_bytes + gather + 8 * wl.G * nb        # + scores written and read once
    roof_ms = roof_bytes / (hbm * 1e9) * 1e3
    del k_blk, ws, flush
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(batch / (ms / 1e3), 1),
            "roofline": {"bound": "hbm", "algorithmic_bytes": roof_bytes, "roofline_ms": round(roof_ms, 4),
                         "frac": round(roof_ms / ms, 4), "peak": hbm, "peak_source": src}}


def run_decode(args, local_rank, fp8=False):
    """The decode workload on its own: one JSON line of decode step latency."""
    from block_sparse_long_18_b300 import build as _build

    _build.build()
    from block_sparse_long_18_b300 import inputs as gen
    from block_sparse_long_18_b300 import sgqa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = gen.WORKLOADS["decode"]
    inp = gen.make_decode_inputs(wl, seed=0, device=dev)
    r = decode_measure(sgqa, wl, inp, dev, args.steps, args.warmup, fp8=fp8)
    batch = len(inp.ctx_len)
    return {
        "metric": "Sparse GQA decode step latency (8 sequences, 256K-1M context)",
        "value": r["ms_per_step"], "unit": "ms/step", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "tokens_per_s": r["tokens_per_s"],
        "dtype": "bf16 (block-proxy cache e4m3)" if fp8 else "bf16", "data": "synthetic",
        "config": {"workload": f"decode{'_fp8' if fp8 else ''}: {batch} sequences, ctx_len {inp.ctx_len}, "
                               f"G={wl.G} x Hg={wl.Hg}, D={wl.D}, P={wl.P}, block {wl.B}, top-k {wl.k}"
                               + (", block-proxy cache FP8 E4M3" if fp8 else ""),
                   "l2": "flushed before every step"},
        "roofline": r["roofline"],
    }


def decode_section(steps, warmup, dev):
    """The decode workload (8 sequences, 256K-1M context) measured inside the default run:
    bf16 and FP8 E4M3 block-proxy caches over the same inputs."""
    from block_sparse_long_18_b300 import inputs as gen
    from block_sparse_long_18_b300 import sgqa

    wl = gen.WORKLOADS["decode"]
    inp = gen.make_decode_inputs(wl, seed=0, device=dev)
    out = {"workload": f"decode: {len(inp.ctx_len)} sequences, ctx_len {inp.ctx_len}, top-k {wl.k} blocks of {wl.B}",
           "bf16_cache": decode_measure(sgqa, wl, inp, dev, max(steps, 10), warmup),
           "fp8_e4m3_cache": decode_measure(sgqa, wl, inp, dev, max(steps, 10), warmup, fp8=True)}
    del inp
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------------------

def run_reference(args, rank, world):
    from block_sparse_long_18_b300 import inputs as gen
    import oracle

    wl = gen.WORKLOADS[args.workload]
    inp = gen.make_inputs(wl, seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    hv = host_views(inp)
    del inp
    # the block index is built once (its time is prorated into every sample); each step
    # times the oracle on 64 query tokens drawn uniformly from the workload
    t0 = time.perf_counter()
    kb = oracle.block_index(hv["k_proxy"], wl.B, 0, wl.C)
    kb_t = (kb, time.perf_counter() - t0)
    rates, secs_all, n_rows = [], [], min(64, wl.T)
    for s in range(args.warmup + args.steps):
        rate, secs, nrows, cores = cpu_oracle_rate(hv, wl, n_rows=n_rows, seed=100 + s, kb_t=kb_t)
        if s >= args.warmup:
            rates.append(rate)
            secs_all.append(secs)
    value = float(np.mean(rates))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "tokens/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(float(np.mean(secs_all)) * 1e3, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{wl.name}: prefill T={wl.T}, context {wl.C}, G={wl.G} x Hg={wl.Hg}, D={wl.D}, "
                               f"P={wl.P}, block {wl.B}, top-k {wl.k}", "global_batch": 1, "seq_len": wl.T},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle", "cores": oracle.num_threads(),
                         "cpu_model": cpu_model(), "nproc": os.cpu_count(),
                         "sample": f"{n_rows} query tokens per step drawn uniformly from the {wl.name} workload, all "
                                   f"{wl.G} groups (indexer + top-k + attention, fp64), block-index pass prorated"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["sgqa", "reference"], default="sgqa")
    ap.add_argument("--workload", default="l128k", choices=["tiny", "l32k", "l128k", "l128k_b1", "chunk1m", "l128k_tail", "decode", "decode_fp8"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-coverage", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        if args.workload in ("decode", "decode_fp8"):  # the oracle arm times prefill workloads
            print(json.dumps({"impl": "reference", "unavailable": "the oracle reference arm times the prefill "
                                                                  "workloads only; decode has no reference line"}),
                  flush=True)
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    if args.workload in ("decode", "decode_fp8"):
        if rank == 0:
            print(json.dumps(run_decode(args, local_rank, fp8=args.workload == "decode_fp8")), flush=True)
        return 0
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_sgqa(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
