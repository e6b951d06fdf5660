"""CPU oracle of the Sparse GQA layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its Python binding) never
imports it and shares no code with it.

The arithmetic lives in ``sgqa_oracle.c`` (plain C, fp64, OpenMP over rows).  This file
only compiles that source with gcc and marshals numpy arrays to it.  Each function
names the passage of the Step 5 Preview pages it follows; see the C source header for
the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgqa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libsgqa_oracle.so")
_lock = threading.Lock()
_lib = None


class OrcDims(ctypes.Structure):
    _fields_ = [
        ("G", ctypes.c_int64),
        ("Hg", ctypes.c_int64),
        ("D", ctypes.c_int64),
        ("P", ctypes.c_int64),
        ("B", ctypes.c_int64),
        ("k", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("gate_per_dim", ctypes.c_int64),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp).  Returns the library path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_LIB_OVERRIDE or build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.sgqa_oracle_bf16_to_f64.restype = ctypes.c_double
            lib.sgqa_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.sgqa_oracle_f64_to_bf16.restype = ctypes.c_uint16
            lib.sgqa_oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.sgqa_oracle_round_bf16_array.restype = None
            lib.sgqa_oracle_round_bf16_array.argtypes = [P, I64, P]
            lib.sgqa_oracle_block_index.restype = ctypes.c_int
            lib.sgqa_oracle_block_index.argtypes = [I64, I64, I64, P, I64, I64, I64, P, I64]
            lib.sgqa_oracle_select.restype = ctypes.c_int
            lib.sgqa_oracle_select.argtypes = [ctypes.POINTER(OrcDims), I64, P, P, P, P, I64, P, P, P, I64]
            lib.sgqa_oracle_attention.restype = ctypes.c_int
            lib.sgqa_oracle_attention.argtypes = [ctypes.POINTER(OrcDims), I64, P, P, P, P, P, P, P, I64,
                                                  P, P, ctypes.c_int32, P, P, P]
            lib.sgqa_oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.sgqa_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.sgqa_oracle_f64_to_e4m3.restype = ctypes.c_uint8
            lib.sgqa_oracle_f64_to_e4m3.argtypes = [ctypes.c_double]
            lib.sgqa_oracle_round_e4m3_array.restype = None
            lib.sgqa_oracle_round_e4m3_array.argtypes = [P, I64, P]
            lib.sgqa_oracle_block_index_e4m3.restype = ctypes.c_int
            lib.sgqa_oracle_block_index_e4m3.argtypes = [I64, I64, I64, P, I64, I64, I64, P, I64]
            lib.sgqa_oracle_num_threads.restype = ctypes.c_int
            lib.sgqa_oracle_num_threads.argtypes = []
            _lib = lib
    return _lib


class mutated:
    """Context manager for the oracle's own mutation tests: compiles a copy of the oracle
    source with the given (old, new) text replacements into `tmpdir` and routes every
    call of this module to it until exit.  Used only to show that the pins in the test
    suite fail when a plausible mistake is planted in the oracle."""

    def __init__(self, replacements, tmpdir):
        self.replacements = replacements
        self.tmpdir = str(tmpdir)

    def __enter__(self):
        global _lib
        src = open(_SRC).read()
        for old, new in self.replacements:
            if old not in src:
                raise ValueError(f"mutation target not found: {old!r}")
            src = src.replace(old, new)
        path = os.path.join(self.tmpdir, "mut.c")
        lib = os.path.join(self.tmpdir, "libmut.so")
        with open(path, "w") as f:
            f.write(src)
        subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", path, "-o", lib, "-lm"], check=True)
        _get()
        self._saved = _lib
        with _lock:
            _lib = None
        global _LIB_OVERRIDE
        _LIB_OVERRIDE = lib
        _get()
        return self

    def __exit__(self, *exc):
        global _lib, _LIB_OVERRIDE
        with _lock:
            _lib = self._saved
        _LIB_OVERRIDE = None
        return False


_LIB_OVERRIDE = None


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    """bf16 payload as a contiguous uint16 array (accepts uint16 or a torch bf16 tensor)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and "bfloat16" in str(a.dtype):
        import torch  # only for the dtype reinterpretation of caller tensors

        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def dims(G, Hg, D, P, B, k, scale=None, gate_per_dim=1) -> OrcDims:
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    return OrcDims(int(G), int(Hg), int(D), int(P), int(B), int(k), float(scale), int(gate_per_dim))


def num_threads() -> int:
    return int(_get().sgqa_oracle_num_threads())


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 payloads (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """One round-to-nearest-even step from double to bf16 (uint16 payloads)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _get().sgqa_oracle_round_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


def block_index(k_proxy, B: int, tok_begin: int, tok_end: int, k_blk=None, nb_cap=None) -> np.ndarray:
    """Block-mean compression of the proxy keys (ai4snews item, Interpretation para 2;
    ai.info article, "Sparse GQA targets million-token context").  k_proxy: [G, C, P]
    bf16 payloads.  Returns k_blk [G, nb_cap, P] with the blocks touched by
    [tok_begin, tok_end) filled (others left as given, or zero)."""
    kp = _u16(k_proxy)
    G, C, P = kp.shape
    if nb_cap is None:
        nb_cap = (C + B - 1) // B
    if k_blk is None:
        k_blk = np.zeros((G, nb_cap, P), dtype=np.uint16)
    k_blk = np.ascontiguousarray(k_blk, dtype=np.uint16)
    rc = _get().sgqa_oracle_block_index(G, P, B, _ptr(kp), C, tok_begin, tok_end, _ptr(k_blk), nb_cap)
    if rc:
        raise ValueError("oracle block_index: bad arguments")
    return k_blk


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact values of FP8 E4M3 codes (uint8)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    f = _get().sgqa_oracle_e4m3_to_f64
    table = np.array([f(i) for i in range(256)], dtype=np.float64)
    return table[c]


def f64_to_e4m3(x: np.ndarray) -> np.ndarray:
    """One round-to-nearest-even step from double to E4M3 codes, saturating at +-448."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    _get().sgqa_oracle_round_e4m3_array(_ptr(x), x.size, _ptr(out))
    return out


def block_index_e4m3(k_proxy, B: int, tok_begin: int, tok_end: int, k_blk=None, nb_cap=None) -> np.ndarray:
    """The block index of `block_index` stored as FP8 E4M3 codes [G, nb_cap, P] (the decode
    cache variant; the pages deploy in FP8 but do not describe this cache)."""
    kp = _u16(k_proxy)
    G, C, P = kp.shape
    if nb_cap is None:
        nb_cap = (C + B - 1) // B
    if k_blk is None:
        k_blk = np.zeros((G, nb_cap, P), dtype=np.uint8)
    k_blk = np.ascontiguousarray(k_blk, dtype=np.uint8)
    rc = _get().sgqa_oracle_block_index_e4m3(G, P, B, _ptr(kp), C, tok_begin, tok_end, _ptr(k_blk), nb_cap)
    if rc:
        raise ValueError("oracle block_index_e4m3: bad arguments")
    return k_blk


def e4m3_as_bf16(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes re-expressed as bf16 payloads.  Every E4M3 value has at most 4
    significant bits and an exponent inside bf16's range, so this is exact; it lets
    `select` score an E4M3 block index unchanged."""
    return f64_to_bf16(e4m3_to_f64(codes))


def select(d: OrcDims, pos, grp, qp_rows, k_blk, want_scores: bool = False):
    """Indexer scores + top-k block selection for the given (position, group) rows
    (ai4snews item, Interpretation para 2; phantomic12 entry: topk 512, proxy_dim 256).
    qp_rows: [n, P] bf16 payloads.  Returns (sel_idx [n, k] int32, sel_cnt [n] int32[, scores])."""
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    grp = np.ascontiguousarray(grp, dtype=np.int32)
    qp = _u16(qp_rows)
    kb = _u16(k_blk)
    n = pos.shape[0]
    sel = np.empty((n, d.k), dtype=np.int32)
    cnt = np.empty((n,), dtype=np.int32)
    max_cand = int(pos.max() // d.B) if (want_scores and n) else 0
    scores = np.full((n, max(max_cand, 1)), np.nan) if want_scores else None
    rc = _get().sgqa_oracle_select(ctypes.byref(d), n, _ptr(pos), _ptr(grp), _ptr(qp), _ptr(kb), kb.shape[1],
                                   _ptr(sel), _ptr(cnt), _ptr(scores), max_cand)
    if rc:
        raise ValueError("oracle select: bad arguments")
    return (sel, cnt, scores) if want_scores else (sel, cnt)


def attention(d: OrcDims, pos, grp, q_rows, gate_rows, K, V, sel_idx=None, sel_cnt=None,
              dense: bool = False, kv_off=None, want_coverage: bool = False):
    """Gated GQA attention over the selected, causally masked tokens (ai.info article,
    "Why StepFun chose 92 transformer blocks": Gated GQA; ai4snews item, Interpretation
    para 2: sparse flash attention over the selection).  q_rows/gate_rows: [n, Hg, D]
    (gate [n, Hg] when gate_per_dim=0); K, V: [G, C, D].  Returns (out fp64 [n, Hg, D],
    lse fp64 [n, Hg][, coverage fp64 [n, Hg]])."""
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    grp = np.ascontiguousarray(grp, dtype=np.int32)
    q = _u16(q_rows)
    gt = _u16(gate_rows)
    Kh = _u16(K)
    Vh = _u16(V)
    n = pos.shape[0]
    if dense:
        sel_idx = np.zeros((n, d.k), dtype=np.int32)
        sel_cnt = np.zeros((n,), dtype=np.int32)
    sel_idx = np.ascontiguousarray(sel_idx, dtype=np.int32)
    sel_cnt = np.ascontiguousarray(sel_cnt, dtype=np.int32)
    off = None if kv_off is None else np.ascontiguousarray(kv_off, dtype=np.int64)
    out = np.empty((n, d.Hg, d.D), dtype=np.float64)
    lse = np.empty((n, d.Hg), dtype=np.float64)
    cov = np.empty((n, d.Hg), dtype=np.float64) if want_coverage else None
    rc = _get().sgqa_oracle_attention(ctypes.byref(d), n, _ptr(pos), _ptr(grp), _ptr(off), _ptr(q), _ptr(gt),
                                      _ptr(Kh), _ptr(Vh), Kh.shape[1], _ptr(sel_idx), _ptr(sel_cnt),
                                      1 if dense else 0, _ptr(out), _ptr(lse), _ptr(cov))
    if rc:
        raise ValueError("oracle attention: bad arguments")
    return (out, lse, cov) if want_coverage else (out, lse)
