"""Pins of the CPU oracle against things other than itself.

Every check here is independent of the CUDA library: textbook/library routines, exact
integer arithmetic, closed forms and brute force on tiny inputs.  Together they are meant
to fail on any plausible slip in the oracle: a dropped term, a wrong sign, an off-by-one
in the causal mask, a flipped tie rule, a transposed operand, double rounding.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_18_b300 import inputs as gen

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


# ---------------------------------------------------------------------------------------
# bf16 conversions
# ---------------------------------------------------------------------------------------

def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(1)
    b = rng.integers(0, 1 << 16, size=200_000, dtype=np.uint32).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]  # drop inf/nan payloads
    ours = oracle.bf16_to_f64(b)
    ref = _from_bits(b).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_rounding_matches_torch_on_float32_values():
    """For values that are exactly float32, RNE to bf16 is a library routine (torch)."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(100_000).astype(np.float32) * np.float32(3.0)
    # plant exact ties: bf16 value + half its ulp, both parities of the last kept bit
    base = rng.integers(0, 1 << 16, size=20_000, dtype=np.uint32).astype(np.uint16)
    base = base[((base & 0x7F80) != 0x7F80) & ((base & 0x7F80) != 0)]
    ties = ((base.astype(np.uint32) << 16) | 0x8000).view(np.float32)
    subn = (rng.integers(1, 1 << 23, size=2000, dtype=np.uint32)).view(np.float32)  # float32 subnormals
    allx = np.concatenate([x, ties, subn, -ties]).astype(np.float32)
    ours = oracle.f64_to_bf16(allx.astype(np.float64))
    ref = _bits(torch.from_numpy(allx).to(torch.bfloat16))
    assert np.array_equal(ours, ref)


def test_bf16_rounding_is_a_single_rounding():
    # 1 + 2^-8 + 2^-40 is above the tie between 1 and 1+2^-7: rounds UP in one step.
    # Narrowing to float32 first would produce the exact tie 1+2^-8 and round to 1.0.
    assert oracle.f64_to_bf16(np.array([1.0 + 2.0**-8 + 2.0**-40]))[0] == 0x3F81
    assert oracle.f64_to_bf16(np.array([1.0 + 2.0**-8]))[0] == 0x3F80        # tie -> even (1.0)
    assert oracle.f64_to_bf16(np.array([1.0 + 3 * 2.0**-8]))[0] == 0x3F82    # tie -> even (1+2^-6)
    assert oracle.f64_to_bf16(np.array([-2.5]))[0] == 0xC020
    assert oracle.f64_to_bf16(np.array([2.0**128]))[0] == 0x7F80             # overflow -> inf
    assert oracle.f64_to_bf16(np.array([-0.0]))[0] == 0x8000


def _rne_fraction_bf16(fr: Fraction) -> float:
    """Independent exact rounding of a rational to 8 significant bits, ties to even."""
    if fr == 0:
        return 0.0
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 7)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(fl * q)


def _rne_fraction_e4m3(fr: Fraction) -> float:
    """Independent exact rounding of a rational to FP8 E4M3: 4 significant bits, a fixed
    step of 2^-9 below 2^-6 (subnormals), ties to even, magnitude saturating at 448."""
    if fr == 0:
        return 0.0
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (max(e, -6) - 3)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * min(float(fl * q), 448.0)


# ---------------------------------------------------------------------------------------
# FP8 E4M3 (the decode block-proxy cache variant)
# ---------------------------------------------------------------------------------------

def _e4m3_torch_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decoding_matches_torch():
    """Every one of the 256 codes decodes to torch's float8_e4m3fn value (a library routine)."""
    ours = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    ref = _e4m3_torch_values()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.all(np.signbit(ours[ok]) == np.signbit(ref[ok]))


def test_e4m3_rounding_matches_torch_on_float32_values():
    """Round to nearest even below saturation equals torch's conversion: random values,
    every midpoint between adjacent codes (ties) and points just beside them, subnormals."""
    rng = np.random.default_rng(21)
    table = _e4m3_torch_values()
    pos = np.unique(table[(~np.isnan(table)) & (table >= 0)])            # 0 .. 448
    mids = (pos[1:] + pos[:-1]) / 2
    near = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(1e9))]).astype(np.float64)
    x = np.concatenate([rng.standard_normal(50_000) * 3.0, rng.uniform(-464, 464, 20_000),
                        rng.uniform(-2 ** -6, 2 ** -6, 5_000), mids, -mids, near, -near, pos, -pos])
    x = x.astype(np.float32)
    x = x[np.abs(x) <= 464].astype(np.float64)
    ours = oracle.f64_to_e4m3(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturation_and_special_values():
    """Finite values past the largest code (448) saturate (the conversion the GPU uses), NaN
    stays NaN, signed zero keeps its sign, and the first value that rounds up from the
    largest subnormal (7 x 2^-9) lands on the smallest normal 2^-6."""
    big = np.array([465.0, 500.0, 1e6, -470.0, -1e30])
    assert oracle.f64_to_e4m3(big).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.f64_to_e4m3(np.array([np.nan])).tolist() == [0x7F]
    assert oracle.f64_to_e4m3(np.array([0.0, -0.0])).tolist() == [0x00, 0x80]
    assert oracle.e4m3_to_f64(oracle.f64_to_e4m3(np.array([7.5 * 2.0 ** -9]))).tolist() == [2.0 ** -6]


def test_e4m3_cache_of_integer_proxy_means():
    """Integer proxies in [-4, 4] average to multiples of 1/8 over a full block of 8; the
    E4M3 cache holds their round-to-nearest-even values, and its bf16 re-expression is exact
    (so the bf16 scoring path of the oracle scores the E4M3 cache unchanged)."""
    rng = np.random.default_rng(22)
    G, C, P, B = 2, 64, 64, 8
    kp_i = rng.integers(-4, 5, size=(G, C, P))
    kp = _bits(torch.from_numpy(kp_i.astype(np.float32)).to(torch.bfloat16))
    codes = oracle.block_index_e4m3(kp, B, 0, C)
    means = kp_i.reshape(G, C // B, B, P).sum(axis=2) / 8.0                 # exact
    ref = torch.from_numpy(means.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    assert np.array_equal(oracle.bf16_to_f64(oracle.e4m3_as_bf16(codes)), oracle.e4m3_to_f64(codes))
    # the quantisation is visible: 17/8 = 2.125 is a tie between 2 and 2.25 and goes to 2
    assert oracle.e4m3_to_f64(oracle.f64_to_e4m3(np.array([2.125]))).tolist() == [2.0]


# ---------------------------------------------------------------------------------------
# O1: block index
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("B", [1, 2, 8, 16])
def test_block_index_integer_proxies_exact(B):
    rng = np.random.default_rng(3)
    G, C, P = 2, 77, 64   # ragged: the last block is partial
    kp_i = rng.integers(-4, 5, size=(G, C, P))
    kp = _bits(torch.from_numpy(kp_i.astype(np.float32)).to(torch.bfloat16))
    kb = oracle.block_index(kp, B, 0, C)
    NB = (C + B - 1) // B
    kbv = oracle.bf16_to_f64(kb)
    for b in range(NB):
        n = min(B, C - b * B)
        s = kp_i[:, b * B:b * B + n].sum(axis=1)  # exact int64 sums
        if n in (1, 2, 4, 8, 16):
            # power-of-two count: the mean is exact in bf16 (<= 8 significant bits)
            assert np.array_equal(kbv[:, b] * n, s.astype(np.float64))
        else:
            want = np.vectorize(lambda v: _rne_fraction_bf16(Fraction(int(v), n)))(s)
            assert np.array_equal(kbv[:, b], want)


def test_block_index_partial_range_only_touches_its_blocks():
    rng = np.random.default_rng(4)
    G, C, P, B = 1, 64, 64, 8
    kp = _bits(torch.from_numpy(rng.integers(-4, 5, size=(G, C, P)).astype(np.float32)).to(torch.bfloat16))
    sentinel = np.full((G, 8, P), 0x7FC0, dtype=np.uint16)
    out = oracle.block_index(kp, B, 20, 37, k_blk=sentinel.copy(), nb_cap=8)
    touched = {2, 3, 4}          # blocks holding tokens 20..36
    for b in range(8):
        if b in touched:
            assert not np.any(out[0, b] == 0x7FC0)
        else:
            assert np.all(out[0, b] == 0x7FC0)
    # block 4 holds tokens 32..36 only (5 of 8): averaged over the tokens present
    full = oracle.block_index(kp, B, 0, 37)
    assert np.array_equal(out[0, 4], full[0, 4])


def test_block_index_general_values_match_exact_rational_mean():
    rng = np.random.default_rng(5)
    G, C, P, B = 1, 24, 32, 8
    kp = _bits(torch.from_numpy(rng.standard_normal((G, C, P)).astype(np.float32)).to(torch.bfloat16))
    kb = oracle.block_index(kp, B, 0, C)
    vals = oracle.bf16_to_f64(kp)
    for b in range(C // B):
        for p in range(P):
            s = sum(Fraction(float(x)) for x in vals[0, b * B:(b + 1) * B, p])
            assert oracle.bf16_to_f64(kb[0, b, p:p + 1])[0] == _rne_fraction_bf16(s / B)


@pytest.mark.parametrize("fmt", ["bf16", "e4m3"])
def test_partial_block_means_at_rounding_midpoints(fmt):
    """Partial blocks (n = 3, 5, 6, 7 tokens) whose exact sums sit on n times a rounding
    midpoint of bf16 or E4M3, or up to three fp32 steps beside it: the oracle's mean equals
    the exact rational mean rounded once (ties to even only on the midpoints themselves)."""
    from midpoint_sums import midpoint_sums, split_bf16

    rng = np.random.default_rng(41 if fmt == "bf16" else 42)
    G, P, B, nblk = 1, 16, 8, 48
    n = np.array([(3, 5, 6, 7)[i % 4] for i in range(nblk)])
    s = midpoint_sums(rng, np.broadcast_to(n[None, :, None], (G, nblk, P)).astype(np.float64), fmt, max_steps=3)
    t0, t1, t2 = split_bf16(s)
    kp = np.zeros((G, nblk, B, P), np.float32)
    kp[:, :, 0], kp[:, :, 1], kp[:, :, 2] = t0, t1, t2
    kp = _bits(torch.from_numpy(kp.reshape(G, nblk * B, P)).to(torch.bfloat16))
    build = oracle.block_index_e4m3 if fmt == "e4m3" else oracle.block_index
    kb = np.zeros((G, nblk, P), np.uint8 if fmt == "e4m3" else np.uint16)
    for i in range(nblk):
        kb = build(kp, B, i * B, i * B + int(n[i]), k_blk=kb, nb_cap=nblk)
    got = oracle.e4m3_to_f64(kb) if fmt == "e4m3" else oracle.bf16_to_f64(kb)
    rne = _rne_fraction_e4m3 if fmt == "e4m3" else _rne_fraction_bf16
    ties = 0
    for i in range(nblk):
        for p in range(P):
            exact = Fraction(float(s[0, i, p])) / int(n[i])
            assert got[0, i, p] == rne(exact), (i, p)
            ties += rne(exact) != rne(exact * (1 + Fraction(1, 1 << 40)))
    assert ties > 0  # some sums are exact midpoints: the tie rule is exercised


# ---------------------------------------------------------------------------------------
# O2 + O3: indexer scores and selection
# ---------------------------------------------------------------------------------------

def _small_case(seed, T, G=2, P=64, B=8, lo=-4, hi=4):
    rng = np.random.default_rng(seed)
    qp_i = rng.integers(lo, hi + 1, size=(G, T, P))
    kp_i = rng.integers(lo, hi + 1, size=(G, T, P))
    qp = _bits(torch.from_numpy(qp_i.astype(np.float32)).to(torch.bfloat16))
    kp = _bits(torch.from_numpy(kp_i.astype(np.float32)).to(torch.bfloat16))
    return qp_i, kp_i, qp, kp


def test_score_invariant_block_mean_equals_token_scores_over_B():
    """8 * score(q, kb_b) == sum over the block's tokens of q . k_j (exact, int64)."""
    T, G, P, B = 200, 2, 64, 8
    qp_i, kp_i, qp, kp = _small_case(6, T, G, P, B)
    kb = oracle.block_index(kp, B, 0, T)
    d = oracle.dims(G, 4, 192, P, B, k=10)
    pos = np.array([199, 150, 64, 63], dtype=np.int64)
    for g in range(G):
        grp = np.full(pos.shape, g, dtype=np.int32)
        _, _, sc = oracle.select(d, pos, grp, qp[g, pos], kb, want_scores=True)
        for r, t in enumerate(pos):
            bt = t // B
            tok = (qp_i[g, t][None, :] * kp_i[g, :bt * B]).sum(axis=1)      # token-level scores
            want = tok.reshape(bt, B).sum(axis=1)                            # summed per block
            assert np.array_equal((sc[r, :bt] * B).astype(np.int64), want)
            assert np.all(sc[r, :bt] * B == np.round(sc[r, :bt] * B))


def _brute_select(scores, bt, k):
    cand = sorted(range(bt), key=lambda b: (-scores[b], -b))[: k - 1]
    return sorted(cand + [bt])


@pytest.mark.parametrize("seed,lo,hi", [(7, -4, 4), (8, -1, 1), (9, 0, 0)])
def test_selection_matches_full_sort(seed, lo, hi):
    T, G, P, B, k = 300, 2, 32, 8, 9
    _, _, qp, kp = _small_case(seed, T, G, P, B, lo, hi)
    kb = oracle.block_index(kp, B, 0, T)
    d = oracle.dims(G, 4, 192, P, B, k)
    pos = np.arange(T, dtype=np.int64)
    for g in range(G):
        grp = np.full(T, g, dtype=np.int32)
        sel, cnt, sc = oracle.select(d, pos, grp, qp[g], kb, want_scores=True)
        for t in range(T):
            bt = t // B
            want = _brute_select(list(sc[t, :bt]), bt, k)
            assert cnt[t] == len(want)
            assert list(sel[t, :cnt[t]]) == want
            assert np.all(sel[t, cnt[t]:] == -1)


def test_selection_closed_forms():
    T, G, P, B, k = 400, 1, 32, 8, 6
    zero = np.zeros((G, T, P), dtype=np.uint16)           # bf16 +0
    kb = oracle.block_index(zero, B, 0, T)
    pos = np.arange(T, dtype=np.int64)
    grp = np.zeros(T, dtype=np.int32)
    sel, cnt = oracle.select(oracle.dims(G, 4, 192, P, B, k), pos, grp, zero[0], kb)
    for t in range(T):
        bt = t // B
        # all scores tie at 0 -> larger index wins -> a sliding window of the last k blocks
        want = list(range(max(0, bt - k + 1), bt + 1))
        assert list(sel[t, :cnt[t]]) == want
    # k = 1: only the own block
    sel1, cnt1 = oracle.select(oracle.dims(G, 4, 192, P, B, 1), pos, grp, zero[0], kb)
    assert np.all(cnt1 == 1) and np.array_equal(sel1[:, 0], pos // B)


def test_selection_negative_zero_equals_positive_zero():
    # a query proxy with a single -1 against block proxies that are 0 or -0 -> all scores are +-0
    G, T, P, B, k = 1, 64, 8, 8, 3
    kp = np.zeros((G, T, P), dtype=np.uint16)
    kp[0, ::2, 0] = 0x8000  # -0
    qp = np.zeros((G, T, P), dtype=np.uint16)
    qp[0, :, 0] = 0xBF80    # -1
    kb = oracle.block_index(kp, B, 0, T)
    pos = np.arange(T, dtype=np.int64)
    sel, cnt = oracle.select(oracle.dims(G, 1, 192, P, B, k), pos, np.zeros(T, np.int32), qp[0], kb)
    for t in range(T):
        bt = t // B
        assert list(sel[t, :cnt[t]]) == list(range(max(0, bt - k + 1), bt + 1))


# ---------------------------------------------------------------------------------------
# O4: attention
# ---------------------------------------------------------------------------------------

def _dense_numpy(q, K, V, gate, t_list, scale):
    """Independent dense causal attention, matrix form: q [n, Hg, D], K/V [C, D]."""
    out = np.empty(q.shape)
    lse = np.empty(q.shape[:2])
    for r, t in enumerate(t_list):
        S = scale * q[r] @ K[: t + 1].T                       # [Hg, t+1]
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        out[r] = (E @ V[: t + 1]) / E.sum(axis=1, keepdims=True) / (1.0 + np.exp(-gate[r]))
        lse[r] = (m[:, 0] + np.log(E.sum(axis=1)))
    return out, lse


def _rand_bf16(rng, shape, s=1.0):
    return _bits(torch.from_numpy((rng.standard_normal(shape) * s).astype(np.float32)).to(torch.bfloat16))


def test_attention_full_selection_equals_dense_causal():
    rng = np.random.default_rng(10)
    G, Hg, D, P, B = 2, 3, 24, 16, 8
    C = 70
    K = _rand_bf16(rng, (G, C, D), 2.0)
    V = _rand_bf16(rng, (G, C, D))
    pos = np.array([0, 1, 7, 8, 9, 33, 69], dtype=np.int64)
    q = _rand_bf16(rng, (len(pos), Hg, D), 2.0)
    gate = _rand_bf16(rng, (len(pos), Hg, D))
    k = (C + B - 1) // B  # every causal block is selected
    d = oracle.dims(G, Hg, D, P, B, k, scale=1.0 / math.sqrt(D))
    for g in range(G):
        grp = np.full(len(pos), g, np.int32)
        sel = np.full((len(pos), k), -1, np.int32)
        cnt = np.empty(len(pos), np.int32)
        for r, t in enumerate(pos):
            sel[r, : t // B + 1] = np.arange(t // B + 1)
            cnt[r] = t // B + 1
        out, lse = oracle.attention(d, pos, grp, q, gate, K, V, sel, cnt)
        out_d, lse_d = oracle.attention(d, pos, grp, q, gate, K, V, dense=True)
        ref, ref_lse = _dense_numpy(oracle.bf16_to_f64(q), oracle.bf16_to_f64(K[g]), oracle.bf16_to_f64(V[g]),
                                    oracle.bf16_to_f64(gate), pos, d.scale)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out_d, ref, rtol=1e-12, atol=1e-12)


def test_attention_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(11)
    G, Hg, D, P, B, C = 1, 4, 32, 16, 8, 40
    K = _rand_bf16(rng, (G, C, D))
    V = _rand_bf16(rng, (G, C, D))
    q = _rand_bf16(rng, (C, Hg, D))
    gate = np.full((C, Hg, D), 0x4300, np.uint16)   # bf16 128.0 -> sigmoid == 1 in double
    d = oracle.dims(G, Hg, D, P, B, k=64, scale=1.0 / math.sqrt(D))
    pos = np.arange(C, dtype=np.int64)
    out, _ = oracle.attention(d, pos, np.zeros(C, np.int32), q, gate, K, V, dense=True)
    qt = torch.from_numpy(oracle.bf16_to_f64(q)).permute(1, 0, 2)[None]            # [1, Hg, C, D]
    kt = torch.from_numpy(oracle.bf16_to_f64(K[0]))[None, None].expand(1, Hg, C, D)
    vt = torch.from_numpy(oracle.bf16_to_f64(V[0]))[None, None].expand(1, Hg, C, D)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_two_token_worked_example():
    """One head, D = 1, two tokens: out(t=1) = (e^{s0} v0 + e^{s1} v1)/(e^{s0}+e^{s1}) * sigmoid(g)."""
    one = lambda x: _bits(torch.tensor([x], dtype=torch.float32).to(torch.bfloat16))[0]
    K = np.array([[[one(1.0)], [one(-2.0)]]], np.uint16)
    V = np.array([[[one(3.0)], [one(5.0)]]], np.uint16)
    q = np.array([[[one(0.5)]]], np.uint16)
    gate = np.array([[[one(0.0)]]], np.uint16)
    d = oracle.dims(1, 1, 1, 8, 8, k=1, scale=1.0)
    out, lse = oracle.attention(d, np.array([1]), np.array([0]), q, gate, K, V,
                                np.array([[0]], np.int32), np.array([1], np.int32))
    s0, s1 = 0.5, -1.0
    want = (math.exp(s0) * 3 + math.exp(s1) * 5) / (math.exp(s0) + math.exp(s1)) * 0.5
    assert abs(out[0, 0, 0] - want) < 1e-14
    assert abs(lse[0, 0] - math.log(math.exp(s0) + math.exp(s1))) < 1e-14
    # at t = 0 only the first token is visible: out = v0 * sigmoid(0)
    out0, _ = oracle.attention(d, np.array([0]), np.array([0]), q, gate, K, V,
                               np.array([[0]], np.int32), np.array([1], np.int32))
    assert abs(out0[0, 0, 0] - 1.5) < 1e-14


def test_attention_sparse_selection_is_a_subset_softmax():
    """With a proper subset selected, the result equals dense attention restricted to the
    selected tokens (built independently here from the token list)."""
    rng = np.random.default_rng(12)
    G, Hg, D, P, B, C = 1, 2, 16, 16, 4, 64
    K = _rand_bf16(rng, (G, C, D), 2.0)
    V = _rand_bf16(rng, (G, C, D))
    t = 50
    sel_blocks = [1, 5, 9, 12]            # own block 12 = 50 // 4, holds 48..51, visible 48..50
    q = _rand_bf16(rng, (1, Hg, D), 2.0)
    gate = _rand_bf16(rng, (1, Hg, D))
    d = oracle.dims(G, Hg, D, P, B, k=4, scale=0.3)
    out, lse = oracle.attention(d, np.array([t]), np.array([0]), q, gate, K, V,
                                np.array([sel_blocks], np.int32), np.array([4], np.int32))
    toks = [j for b in sel_blocks for j in range(b * B, b * B + B) if j <= t]
    assert toks[-1] == 50 and len(toks) == 15
    qf, Kf, Vf, gf = (oracle.bf16_to_f64(x) for x in (q, K[0], V[0], gate))
    S = 0.3 * qf[0] @ Kf[toks].T
    P_ = np.exp(S - S.max(axis=1, keepdims=True))
    P_ /= P_.sum(axis=1, keepdims=True)
    want = (P_ @ Vf[toks]) / (1 + np.exp(-gf[0]))
    np.testing.assert_allclose(out[0], want, rtol=1e-12, atol=1e-13)


def test_attention_per_head_gate_and_packed_offset():
    rng = np.random.default_rng(13)
    G, Hg, D, P, B = 1, 2, 8, 8, 4
    C = 40
    K = _rand_bf16(rng, (G, C, D))
    V = _rand_bf16(rng, (G, C, D))
    q = _rand_bf16(rng, (1, Hg, D))
    gh = _rand_bf16(rng, (1, Hg))
    gd = np.repeat(gh[:, :, None], D, axis=2)
    sel = np.array([[0, 1, 2]], np.int32)
    cnt = np.array([3], np.int32)
    d1 = oracle.dims(G, Hg, D, P, B, 3, gate_per_dim=0)
    d2 = oracle.dims(G, Hg, D, P, B, 3, gate_per_dim=1)
    # sequence packed at offset 16: position 9 of the sequence reads cache rows 16..25
    a, _ = oracle.attention(d1, np.array([9]), np.array([0]), q, gh, K, V, sel, cnt, kv_off=np.array([16]))
    b, _ = oracle.attention(d2, np.array([9]), np.array([0]), q, gd, K[:, 16:], V[:, 16:], sel, cnt)
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------------------
# O5: coverage
# ---------------------------------------------------------------------------------------

def test_coverage_closed_forms():
    rng = np.random.default_rng(14)
    G, Hg, D, P, B, C = 1, 2, 16, 16, 8, 96
    K = _rand_bf16(rng, (G, C, D), 2.0)
    V = _rand_bf16(rng, (G, C, D))
    pos = np.array([5, 40, 95], dtype=np.int64)
    q = _rand_bf16(rng, (3, Hg, D), 2.0)
    gate = _rand_bf16(rng, (3, Hg, D))
    d = oracle.dims(G, Hg, D, P, B, k=3)
    sel = np.array([[0, -1, -1], [1, 3, 5], [2, 7, 11]], np.int32)
    cnt = np.array([1, 3, 3], np.int32)
    _, lse_s, cov = oracle.attention(d, pos, np.zeros(3, np.int32), q, gate, K, V, sel, cnt, want_coverage=True)
    _, lse_d = oracle.attention(d, pos, np.zeros(3, np.int32), q, gate, K, V, dense=True)
    # row 0 selects every causal block (b_t + 1 <= k) -> coverage 1
    np.testing.assert_allclose(cov[0], 1.0, rtol=0, atol=1e-14)
    # mass on a subset == exp(LSE_subset - LSE_dense)
    np.testing.assert_allclose(cov, np.exp(lse_s - lse_d), rtol=1e-12)
    assert np.all(cov[1:] < 1.0)


# ---------------------------------------------------------------------------------------
# Page constants and the workload table
# ---------------------------------------------------------------------------------------

def test_page_constants_match_workloads():
    with open(os.path.join(HERE, "golden", "page_constants.json")) as f:
        pc = json.load(f)
    wl = gen.WORKLOADS["l128k"]
    assert wl.B == pc["block_size"]["value"]
    assert wl.k == pc["top_k_blocks"]["value"]
    assert wl.k * wl.B == pc["top_k_tokens"]["value"]
    assert wl.P == pc["proxy_dim"]["value"]
    assert wl.G * wl.Hg == pc["num_attention_heads"]["value"]
    assert wl.G == pc["num_kv_groups"]["value"]
    assert wl.D == pc["head_dim"]["value"]
    assert gen.WORKLOADS["chunk1m"].C == pc["max_positions"]["value"]
    b1 = gen.WORKLOADS["l128k_b1"]
    assert b1.B == 1 and b1.k == pc["reference_top_k_tokens_b1"]["value"]
    assert 23 * 2 * wl.G * wl.D * 2 == pc["kv_bytes_per_token_all_full_layers"]["value"]
