"""Seeded synthetic inputs for the Sparse GQA layer.

This module is shared by the tests, the benchmark and the CPU oracle's callers.  It
holds none of the layer's arithmetic: it only draws random tensors with the shapes and
value distributions of the workloads below and lays them out in the library's memory
layout.  No public dataset is involved; the pages measure coverage on the vendor's own
data, which these draws stand in for.

Distributions (the pages give none; these are the readings used everywhere):
  * Q, K, V, gate ~ N(0, 1), rounded to bf16.
  * proxies are integers drawn uniformly from [-4, 4] and stored as bf16, so that the
    block means are multiples of 1/8 and every indexer score is exact in fp32.
  * "planted" workloads: per KV group a random unit direction u_g in R^D.  Exactly
    round(0.05 * NB) blocks per group are planted (drawn without replacement); every key
    token in them gets K += alpha * u_g with alpha = sqrt(8 D), so E|K|^2 = 9 D (norm x3).
    Each query token carries the direction with probability 1/2 (drawn once per token,
    shared by all groups); its heads of group g get Q += alpha * u_g.  The proxies share
    the structure: per group a random integer vector w_g in [-4, 4]^P; planted key tokens
    and carrying queries take clamp(w_g + e, -4, 4) with e uniform in {-1, 0, 1}.

Layouts (the library's):
  q, gate  [T, H, D]      (H = G * Hg, heads of group g are g*Hg .. g*Hg+Hg-1)
  k, v     [G, C, D]      (group-major: one block of one group is contiguous)
  q_proxy  [G, T, P]
  k_proxy  [G, C, P]
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int               # query tokens in the call
    C: int               # context tokens (cache length)
    G: int = 4
    Hg: int = 16
    D: int = 192
    P: int = 256
    B: int = 8
    k: int = 512
    q_start: int = 0     # absolute position of query row 0
    planted: bool = True
    batch: int = 1       # decode: number of sequences
    ctx_lo: int = 0      # decode: context length range (inclusive)
    ctx_hi: int = 0

    @property
    def H(self) -> int:
        return self.G * self.Hg


# The five workloads of the layer: shapes from the phantomic12 catalog entry (64 heads,
# 4 KV groups, head_dim 192, sparse indexer topk 512 / proxy_dim 256, 1,048,576
# positions) and the ai4snews item (block size 8).
WORKLOADS = {
    "tiny": Workload("tiny", T=2048, C=2048, G=1, Hg=4, k=32, planted=False),
    "l32k": Workload("l32k", T=32768, C=32768),
    "l128k": Workload("l128k", T=131072, C=131072),
    "l128k_b1": Workload("l128k_b1", T=131072, C=131072, B=1, k=2048),
    "decode": Workload("decode", T=1, C=0, batch=8, ctx_lo=262144, ctx_hi=1048576),
    "chunk1m": Workload("chunk1m", T=8192, C=1048576, q_start=1048576 - 8192),
    # the last 16,384 queries of a 128K context: the 128K gather pattern in ~2 GB of HBM
    # (used for profiler captures, which must stay small)
    "l128k_tail": Workload("l128k_tail", T=16384, C=131072, q_start=131072 - 16384),
}


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _int_proxy(gen, shape, device) -> torch.Tensor:
    return torch.randint(-4, 5, shape, generator=gen, device=device, dtype=torch.int16).to(torch.float32)


@dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    gate: torch.Tensor
    q_proxy: torch.Tensor
    k_proxy: torch.Tensor
    carry: torch.Tensor                      # [T] bool, query carries the planted direction
    planted_blocks: torch.Tensor | None      # [G, n_plant] int64
    # decode only
    ctx_len: list[int] = field(default_factory=list)
    kv_off: list[int] = field(default_factory=list)


def _fill_keys(gen, G, C, D, P, B, planted, device, k_out, v_out, kp_out, u, w, alpha, off=0, n_tok=None):
    """Draw K, V, k_proxy for tokens [off, off + n_tok) of a [G, *, *] cache region."""
    n_tok = C if n_tok is None else n_tok
    for g in range(G):
        k_out[g, off:off + n_tok] = _bf16(torch.randn(n_tok, D, generator=gen, device=device))
        v_out[g, off:off + n_tok] = _bf16(torch.randn(n_tok, D, generator=gen, device=device))
        kp_out[g, off:off + n_tok] = _bf16(_int_proxy(gen, (n_tok, P), device))
    if not planted:
        return None
    NB = (n_tok + B - 1) // B
    n_plant = int(round(0.05 * NB))
    blocks = torch.empty((G, n_plant), dtype=torch.int64, device=device)
    for g in range(G):
        blocks[g] = torch.randperm(NB, generator=gen, device=device)[:n_plant]
        tok = (blocks[g][:, None] * B + torch.arange(B, device=device)[None, :]).reshape(-1)
        tok = tok[tok < n_tok] + off
        kf = k_out[g, tok].float() + alpha * u[g][None, :]
        k_out[g, tok] = _bf16(kf)
        e = torch.randint(-1, 2, (tok.numel(), P), generator=gen, device=device, dtype=torch.int16).float()
        kp_out[g, tok] = _bf16(torch.clamp(w[g][None, :] + e, -4, 4))
    return blocks


def make_inputs(wl: Workload | str, seed: int = 0, device: str | torch.device = "cpu") -> Inputs:
    """Prefill / chunked-prefill inputs (batch 1)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    assert wl.batch == 1, "use make_decode_inputs for decode workloads"
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    G, Hg, D, P, B, T, C = wl.G, wl.Hg, wl.D, wl.P, wl.B, wl.T, wl.C
    H = G * Hg
    alpha = math.sqrt(8.0 * D)
    u = torch.randn(G, D, generator=gen, device=device)
    u = u / u.norm(dim=1, keepdim=True)
    w = _int_proxy(gen, (G, P), device)

    k = torch.empty((G, C, D), dtype=torch.bfloat16, device=device)
    v = torch.empty((G, C, D), dtype=torch.bfloat16, device=device)
    kp = torch.empty((G, C, P), dtype=torch.bfloat16, device=device)
    blocks = _fill_keys(gen, G, C, D, P, B, wl.planted, device, k, v, kp, u, w, alpha)

    q = torch.empty((T, H, D), dtype=torch.bfloat16, device=device)
    gate = torch.empty((T, H, D), dtype=torch.bfloat16, device=device)
    step = 8192
    for t0 in range(0, T, step):
        n = min(step, T - t0)
        q[t0:t0 + n] = _bf16(torch.randn(n, H, D, generator=gen, device=device))
        gate[t0:t0 + n] = _bf16(torch.randn(n, H, D, generator=gen, device=device))
    qp = _bf16(_int_proxy(gen, (G, T, P), device))
    if wl.planted:
        carry = torch.rand(T, generator=gen, device=device) < 0.5
        idx = carry.nonzero().squeeze(1)
        for g in range(G):
            for i0 in range(0, idx.numel(), step):
                sub = idx[i0:i0 + step]
                qf = q[sub, g * Hg:(g + 1) * Hg].float() + alpha * u[g][None, None, :]
                q[sub, g * Hg:(g + 1) * Hg] = _bf16(qf)
            e = torch.randint(-1, 2, (idx.numel(), P), generator=gen, device=device, dtype=torch.int16).float()
            qp[g, idx] = _bf16(torch.clamp(w[g][None, :] + e, -4, 4))
    else:
        carry = torch.zeros(T, dtype=torch.bool, device=device)
    return Inputs(wl, q, k, v, gate, qp, kp, carry, blocks)


def make_decode_inputs(wl: Workload | str = "decode", seed: int = 0, device="cpu") -> Inputs:
    """Decode inputs: `batch` sequences with context lengths uniform in [ctx_lo, ctx_hi],
    packed one after another in the caches at offsets that are multiples of B.  The new
    query of sequence s sits at position ctx_len[s]-1 and its K/V/proxy are already in
    the caches."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    G, Hg, D, P, B = wl.G, wl.Hg, wl.D, wl.P, wl.B
    H = G * Hg
    alpha = math.sqrt(8.0 * D)
    lens = torch.randint(wl.ctx_lo, wl.ctx_hi + 1, (wl.batch,), generator=torch.Generator().manual_seed(seed))
    ctx_len = [int(x) for x in lens]
    kv_off, total = [], 0
    for L in ctx_len:
        kv_off.append(total)
        total += (L + B - 1) // B * B
    u = torch.randn(G, D, generator=gen, device=device)
    u = u / u.norm(dim=1, keepdim=True)
    w = _int_proxy(gen, (G, P), device)
    k = torch.zeros((G, total, D), dtype=torch.bfloat16, device=device)
    v = torch.zeros((G, total, D), dtype=torch.bfloat16, device=device)
    kp = torch.zeros((G, total, P), dtype=torch.bfloat16, device=device)
    for s, L in enumerate(ctx_len):
        _fill_keys(gen, G, L, D, P, B, wl.planted, device, k, v, kp, u, w, alpha, off=kv_off[s], n_tok=L)
    q = _bf16(torch.randn(wl.batch, H, D, generator=gen, device=device))
    gate = _bf16(torch.randn(wl.batch, H, D, generator=gen, device=device))
    qp = _bf16(_int_proxy(gen, (G, wl.batch, P), device))
    carry = torch.rand(wl.batch, generator=gen, device=device) < 0.5
    if wl.planted:
        for s in range(wl.batch):
            if bool(carry[s]):
                for g in range(G):
                    q[s, g * Hg:(g + 1) * Hg] = _bf16(q[s, g * Hg:(g + 1) * Hg].float() + alpha * u[g][None, :])
                    e = torch.randint(-1, 2, (P,), generator=gen, device=device, dtype=torch.int16).float()
                    qp[g, s] = _bf16(torch.clamp(w[g] + e, -4, 4))
    return Inputs(wl, q, k, v, gate, qp, kp, carry, None, ctx_len=ctx_len, kv_off=kv_off)


def small_workload(T: int, C: int | None = None, G: int = 1, Hg: int = 4, B: int = 8, k: int = 8,
                   P: int = 256, D: int = 192, planted: bool = False, q_start: int = 0) -> Workload:
    """An ad-hoc workload for parity cases (ragged T, tiny contexts, edge k)."""
    return Workload(f"small_T{T}", T=T, C=C if C is not None else q_start + T, G=G, Hg=Hg, D=D, P=P, B=B, k=k,
                    planted=planted, q_start=q_start)
