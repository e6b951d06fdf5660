"""Seeded fp32 sums placed on, or a few fp32 steps beside, n times a rounding midpoint of
bf16 or FP8 E4M3 -- the hardest cases for rounding a block mean sum / n once -- and their
split into three bf16 token values whose fp32 sum in token order is exact."""
import numpy as np


def _step(s: np.ndarray, k: np.ndarray) -> np.ndarray:
    """s moved by k fp32 steps away from zero (k < 0: toward zero); s is far from zero."""
    return (s.view(np.int32) + k.astype(np.int32)).view(np.float32)


def midpoint_sums(rng: np.random.Generator, n: np.ndarray, fmt: str, max_steps: int = 2) -> np.ndarray:
    """One fp32 sum per entry of n (token counts): n * m + k steps, m a random midpoint of
    `fmt` ("bf16": 9 significant bits ending in 1; "e4m3": 5 such bits in the normal range
    or an odd multiple of 2^-10 below it, at most 448 in magnitude), k in [-max_steps, max_steps]."""
    shape = n.shape
    if fmt == "bf16":
        M = rng.integers(256, 512, size=shape) | 1
        e = rng.integers(-40, 12, size=shape)
        m = M.astype(np.float64) * np.exp2(e - 8.0)
    elif fmt == "e4m3":
        normal = rng.random(shape) < 0.5
        Mn = rng.integers(16, 32, size=shape) | 1
        en = rng.integers(-6, 9, size=shape)
        Ms = rng.integers(1, 16, size=shape) | 1
        m = np.where(normal, Mn * np.exp2(en - 4.0), Ms * 2.0 ** -10)
        m = np.minimum(m, 448.0)
    else:
        raise ValueError(fmt)
    m = m * np.where(rng.random(shape) < 0.5, -1.0, 1.0)
    s = (n * m).astype(np.float32)  # at most 13 significant bits: exact
    k = rng.integers(-max_steps, max_steps + 1, size=shape)
    return _step(s, k)


def split_bf16(s: np.ndarray):
    """Three bf16-representable fp32 arrays t0, t1, t2 with ((t0 + t1) + t2) == s exactly
    in fp32: the leading 8 significant bits, the next 8, the rest."""
    trunc = lambda x: (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    t0 = trunc(s)
    r1 = (s - t0).astype(np.float32)
    t1 = trunc(r1)
    t2 = (r1 - t1).astype(np.float32)
    assert np.array_equal(trunc(t2), t2)
    assert np.array_equal(((t0 + t1) + t2).astype(np.float32), s)
    return t0, t1, t2
