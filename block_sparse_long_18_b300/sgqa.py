"""Python binding of the Sparse GQA C ABI (include/sgqa.h).

Argument marshalling only: every step of the layer runs in the CUDA library
``libsgqa.so`` (built from ``csrc/`` by ``build.py``).  Torch tensors supply device
memory and the current CUDA stream.  Importing this module fails loudly when the library
has not been built; there is no other code path.

The functions carry the C names and raise :class:`SgqaError` on any status but
``SGQA_OK``.  Layouts are the ABI's:

  q, gate       [T, H, D] bf16          k, v            [G, C, D] bf16
  q_proxy       [G, T, P] bf16          k_proxy         [G, C, P] bf16
  k_blk         [G, NB, P] bf16         sel_idx         [G, T, k] int32, sel_cnt [G, T]
  out           [T, H, D] bf16          lse             [T, H] fp32
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsgqa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libsgqa.so is not built ({LIB_PATH}); run `python -m block_sparse_long_18_b300.build`")
_lib = ctypes.CDLL(LIB_PATH)

STATUS = {
    0: "SGQA_OK",
    1: "SGQA_ERR_INVALID_ARGUMENT",
    2: "SGQA_ERR_UNSUPPORTED_SHAPE",
    3: "SGQA_ERR_WORKSPACE_TOO_SMALL",
    4: "SGQA_ERR_CUDA",
    5: "SGQA_ERR_DEVICE_TIMEOUT",
    6: "SGQA_ERR_DEVICE_BOUNDS",
}
SGQA_OP_INDEX_TOPK, SGQA_OP_PREFILL, SGQA_OP_DECODE, SGQA_OP_ATTN, SGQA_OP_PREFILL_HOST = 1, 2, 3, 4, 5

# Every symbol include/sgqa.h declares.
EXPORTS = (
    "sgqa_build_block_index", "sgqa_index_topk", "sgqa_sparse_attn_fwd", "sgqa_prefill", "sgqa_decode",
    "sgqa_workspace_bytes", "sgqa_get_device_error", "sgqa_set_wait_timeout_ns", "sgqa_selftest_wait_timeout",
    "sgqa_status_string", "sgqa_abi_version", "sgqa_index_topk_noalloc", "sgqa_attention_kernel",
    "sgqa_build_block_index_fp8", "sgqa_decode_fp8", "sgqa_prefill_host",
)
ATTN_AUTO, ATTN_WARP, ATTN_TC_UNION, ATTN_ROUTED, ATTN_GROUPED = 0, 1, 2, 3, 4


class SgqaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({_lib.sgqa_status_string(code).decode()})")


class Params(ctypes.Structure):
    _fields_ = [
        ("num_kv_groups", ctypes.c_int32),
        ("heads_per_group", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("proxy_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("top_k_blocks", ctypes.c_int32),
        ("gate_per_dim", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("attn_kernel", ctypes.c_int32),
    ]


def params(G=4, Hg=16, D=192, P=256, B=8, k=512, gate_per_dim=1, scale=0.0, attn_kernel=ATTN_AUTO) -> Params:
    """Layer constants; the defaults are the pages' (phantomic12 entry: 64 heads in 4 KV
    groups, head_dim 192, topk 512, proxy_dim 256; ai4snews item: block size 8).
    attn_kernel: ATTN_AUTO, or ATTN_WARP / ATTN_TC_UNION / ATTN_ROUTED / ATTN_GROUPED to force
    a prefill attention kernel."""
    return Params(G, Hg, D, P, B, k, gate_per_dim, scale, attn_kernel)


class HostTensors(ctypes.Structure):
    """sgqa_host_tensors: host pointers of one end-to-end prefill."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "gate", "q_proxy", "k_proxy", "out", "lse")]


class DeviceTensors(ctypes.Structure):
    """sgqa_device_tensors: the caller's device buffers of one end-to-end prefill."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("gate", ctypes.c_void_p),
                ("k_proxy", ctypes.c_void_p), ("k_blk", ctypes.c_void_p), ("nb_cap", ctypes.c_int64),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("ws", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_PP = ctypes.POINTER(Params)
_lib.sgqa_status_string.restype = ctypes.c_char_p
_lib.sgqa_status_string.argtypes = [ctypes.c_int]
_lib.sgqa_abi_version.restype = ctypes.c_int32
_lib.sgqa_abi_version.argtypes = []
_lib.sgqa_attention_kernel.restype = ctypes.c_int32
_lib.sgqa_attention_kernel.argtypes = [_PP, _I64, _I64, ctypes.c_int32]
_lib.sgqa_build_block_index.argtypes = [_PP, _P, _I64, _I64, _I64, _P, _I64, _P]
_lib.sgqa_index_topk.argtypes = [_PP, _P, _I64, _I64, _P, _I64, _P, _P, _P, ctypes.c_size_t, _P]
_lib.sgqa_index_topk_noalloc.argtypes = [_PP, _P, _I64, _I64, _P, _I64, _P, _P, _P]
_lib.sgqa_sparse_attn_fwd.argtypes = [_PP, _P, _P, _P, _I64, _P, _P, _P, _I64, _I64, _P, _P, ctypes.c_int32, _P,
                                      ctypes.c_size_t, _P]
_lib.sgqa_prefill.argtypes = [_PP, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _P, _P,
                              ctypes.c_size_t, _P]
_lib.sgqa_decode.argtypes = [_PP, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _P,
                             ctypes.c_size_t, _P]
_lib.sgqa_decode_fp8.argtypes = [_PP, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _P,
                             ctypes.c_size_t, _P]
_lib.sgqa_build_block_index_fp8.argtypes = [_PP, _P, _I64, _I64, _I64, _P, _I64, _P]
_lib.sgqa_prefill_host.argtypes = [_PP, ctypes.POINTER(HostTensors), ctypes.POINTER(DeviceTensors), _I64, _I64, _I64,
                                   _I64, _P]
_lib.sgqa_workspace_bytes.restype = ctypes.c_size_t
_lib.sgqa_workspace_bytes.argtypes = [_PP, ctypes.c_int32, _I64, _I64, ctypes.c_int32]
_lib.sgqa_get_device_error.argtypes = [_P]
_lib.sgqa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
_lib.sgqa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _P]
for _f in ("sgqa_build_block_index", "sgqa_index_topk", "sgqa_index_topk_noalloc", "sgqa_sparse_attn_fwd",
           "sgqa_prefill", "sgqa_prefill_host", "sgqa_decode", "sgqa_decode_fp8", "sgqa_build_block_index_fp8",
           "sgqa_get_device_error", "sgqa_set_wait_timeout_ns", "sgqa_selftest_wait_timeout"):
    getattr(_lib, _f).restype = ctypes.c_int


def _check(code: int, where: str):
    if code != 0:
        raise SgqaError(code, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor | None, dtype, name: str, shape=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


BF16, I32, F32 = torch.bfloat16, torch.int32, torch.float32


def abi_version() -> int:
    return int(_lib.sgqa_abi_version())


def sgqa_attention_kernel(prm: Params, T: int, q_start: int = 0, dense_mode: bool = False) -> int:
    """Which attention kernel a call with these arguments launches (ATTN_*); -1 if invalid."""
    return int(_lib.sgqa_attention_kernel(ctypes.byref(prm), T, q_start, 1 if dense_mode else 0))


def sgqa_workspace_bytes(prm: Params, op: int, T: int, ctx_len: int, batch: int = 1) -> int:
    return int(_lib.sgqa_workspace_bytes(ctypes.byref(prm), op, T, ctx_len, batch))


def sgqa_build_block_index(prm: Params, k_proxy, tok_begin: int, tok_end: int, k_blk, stream=None):
    G, C, P = k_proxy.shape
    _check(_lib.sgqa_build_block_index(ctypes.byref(prm), _dev(k_proxy, BF16, "k_proxy"), C, tok_begin, tok_end,
                                       _dev(k_blk, BF16, "k_blk"), k_blk.shape[1], _stream(stream)),
           "sgqa_build_block_index")


def sgqa_build_block_index_fp8(prm: Params, k_proxy, tok_begin: int, tok_end: int, k_blk_e4m3, stream=None):
    """Block index as FP8 E4M3 codes (a uint8 tensor [G, nb_cap, P]) for the decode cache."""
    G, C, P = k_proxy.shape
    _check(_lib.sgqa_build_block_index_fp8(ctypes.byref(prm), _dev(k_proxy, BF16, "k_proxy"), C, tok_begin, tok_end,
                                           _dev(k_blk_e4m3, torch.uint8, "k_blk_e4m3"), k_blk_e4m3.shape[1],
                                           _stream(stream)), "sgqa_build_block_index_fp8")


def sgqa_index_topk(prm: Params, q_proxy, q_start: int, k_blk, sel_idx, sel_cnt, ws, stream=None):
    G, T, P = q_proxy.shape
    _check(_lib.sgqa_index_topk(ctypes.byref(prm), _dev(q_proxy, BF16, "q_proxy"), T, q_start,
                                _dev(k_blk, BF16, "k_blk"), k_blk.shape[1],
                                _dev(sel_idx, I32, "sel_idx", (G, T, prm.top_k_blocks)),
                                _dev(sel_cnt, I32, "sel_cnt", (G, T)), _dev(ws, torch.uint8, "ws"), ws.numel(),
                                _stream(stream)), "sgqa_index_topk")


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def sgqa_index_topk_noalloc(prm: Params, q_proxy, q_start: int, k_blk, sel_idx, sel_cnt, stream=None):
    """sgqa_index_topk for callers that cannot allocate: the library's own fixed scratch
    array (NOALLOC_SCRATCH_BYTES per device) replaces the workspace.  Calls that overlap on
    the GPU race on that array."""
    G, T, P = q_proxy.shape
    _check(_lib.sgqa_index_topk_noalloc(ctypes.byref(prm), _dev(q_proxy, BF16, "q_proxy"), T, q_start,
                                        _dev(k_blk, BF16, "k_blk"), k_blk.shape[1],
                                        _dev(sel_idx, I32, "sel_idx", (G, T, prm.top_k_blocks)),
                                        _dev(sel_cnt, I32, "sel_cnt", (G, T)), _stream(stream)),
           "sgqa_index_topk_noalloc")


def sgqa_sparse_attn_fwd(prm: Params, q, k, v, gate, sel_idx, sel_cnt, q_start: int, out, lse=None,
                         dense_mode: bool = False, stream=None, ws=None):
    """ws: optional uint8 workspace of sgqa_workspace_bytes(prm, SGQA_OP_ATTN, T, q_start + T)
    bytes; it enables the grouped mode (the default where the union kernel's shape holds)."""
    T = q.shape[0]
    _check(_lib.sgqa_sparse_attn_fwd(ctypes.byref(prm), _dev(q, BF16, "q"), _dev(k, BF16, "k"), _dev(v, BF16, "v"),
                                     k.shape[1], _dev(gate, BF16, "gate"), _dev(sel_idx, I32, "sel_idx"),
                                     _dev(sel_cnt, I32, "sel_cnt"), T, q_start, _dev(out, BF16, "out"),
                                     _dev(lse, F32, "lse"), 1 if dense_mode else 0,
                                     _dev(ws, torch.uint8, "ws"), 0 if ws is None else ws.numel(), _stream(stream)),
           "sgqa_sparse_attn_fwd")


def sgqa_prefill(prm: Params, q, k, v, gate, q_proxy, k_proxy, q_start: int, k_blk, sel_idx, sel_cnt, out, lse, ws,
                 stream=None):
    T = q.shape[0]
    _check(_lib.sgqa_prefill(ctypes.byref(prm), _dev(q, BF16, "q"), _dev(k, BF16, "k"), _dev(v, BF16, "v"),
                             _dev(gate, BF16, "gate"), _dev(q_proxy, BF16, "q_proxy"), _dev(k_proxy, BF16, "k_proxy"),
                             k.shape[1], T, q_start, _dev(k_blk, BF16, "k_blk"), k_blk.shape[1],
                             _dev(sel_idx, I32, "sel_idx"), _dev(sel_cnt, I32, "sel_cnt"), _dev(out, BF16, "out"),
                             _dev(lse, F32, "lse"), _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)),
           "sgqa_prefill")


def sgqa_decode(prm: Params, ctx_len, kv_off, q, q_proxy, gate, k_cache, v_cache, k_proxy_cache, k_blk_cache,
                sel_idx, sel_cnt, out, lse, ws, stream=None):
    batch = len(ctx_len)
    cl = (ctypes.c_int64 * batch)(*[int(x) for x in ctx_len])
    ko = (ctypes.c_int64 * batch)(*[int(x) for x in kv_off])
    _check(_lib.sgqa_decode(ctypes.byref(prm), batch, cl, ko, _dev(q, BF16, "q"), _dev(q_proxy, BF16, "q_proxy"),
                            _dev(gate, BF16, "gate"), _dev(k_cache, BF16, "k_cache"), _dev(v_cache, BF16, "v_cache"),
                            _dev(k_proxy_cache, BF16, "k_proxy_cache"), _dev(k_blk_cache, BF16, "k_blk_cache"),
                            k_cache.shape[1], _dev(sel_idx, I32, "sel_idx"), _dev(sel_cnt, I32, "sel_cnt"),
                            _dev(out, BF16, "out"), _dev(lse, F32, "lse"), _dev(ws, torch.uint8, "ws"), ws.numel(),
                            _stream(stream)), "sgqa_decode")


def sgqa_decode_fp8(prm: Params, ctx_len, kv_off, q, q_proxy, gate, k_cache, v_cache, k_proxy_cache,
                    k_blk_cache_e4m3, sel_idx, sel_cnt, out, lse, ws, stream=None):
    """sgqa_decode over an FP8 E4M3 block-proxy cache (uint8 [G, total / B, P])."""
    batch = len(ctx_len)
    cl = (ctypes.c_int64 * batch)(*[int(x) for x in ctx_len])
    ko = (ctypes.c_int64 * batch)(*[int(x) for x in kv_off])
    _check(_lib.sgqa_decode_fp8(ctypes.byref(prm), batch, cl, ko, _dev(q, BF16, "q"), _dev(q_proxy, BF16, "q_proxy"),
                                _dev(gate, BF16, "gate"), _dev(k_cache, BF16, "k_cache"),
                                _dev(v_cache, BF16, "v_cache"), _dev(k_proxy_cache, BF16, "k_proxy_cache"),
                                _dev(k_blk_cache_e4m3, torch.uint8, "k_blk_cache_e4m3"), k_cache.shape[1],
                                _dev(sel_idx, I32, "sel_idx"), _dev(sel_cnt, I32, "sel_cnt"), _dev(out, BF16, "out"),
                                _dev(lse, F32, "lse"), _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)),
           "sgqa_decode_fp8")


def sgqa_get_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the sticky device error code."""
    return int(_lib.sgqa_get_device_error(_stream(stream)))


def sgqa_set_wait_timeout_ns(ns: int):
    _check(_lib.sgqa_set_wait_timeout_ns(int(ns)), "sgqa_set_wait_timeout_ns")


def sgqa_selftest_wait_timeout(limit_ns: int, stream=None):
    _check(_lib.sgqa_selftest_wait_timeout(int(limit_ns), _stream(stream)), "sgqa_selftest_wait_timeout")


# ---------------------------------------------------------------------------------------
# Convenience layer: allocate outputs and workspace with torch, then call the ABI.
# ---------------------------------------------------------------------------------------

@dataclass
class PrefillResult:
    out: torch.Tensor
    lse: torch.Tensor
    sel_idx: torch.Tensor
    sel_cnt: torch.Tensor
    k_blk: torch.Tensor


class PrefillPlan:
    """Preallocated outputs and workspace for repeated prefill calls of one shape."""

    def __init__(self, prm: Params, T: int, ctx_cap: int, q_start: int = 0, device="cuda", ws_bytes: int | None = None):
        self.prm, self.T, self.ctx_cap, self.q_start = prm, T, ctx_cap, q_start
        G, H, D, P, B, k = (prm.num_kv_groups, prm.num_kv_groups * prm.heads_per_group, prm.head_dim, prm.proxy_dim,
                            prm.block_size, prm.top_k_blocks)
        nb = (ctx_cap + B - 1) // B
        self.k_blk = torch.zeros((G, nb, P), dtype=BF16, device=device)
        self.sel_idx = torch.empty((G, T, k), dtype=I32, device=device)
        self.sel_cnt = torch.empty((G, T), dtype=I32, device=device)
        self.out = torch.empty((T, H, D), dtype=BF16, device=device)
        self.lse = torch.empty((T, H), dtype=F32, device=device)
        need = sgqa_workspace_bytes(prm, SGQA_OP_PREFILL, T, q_start + T)
        self.ws = torch.empty((max(need, ws_bytes or 0),), dtype=torch.uint8, device=device)

    def run(self, q, k, v, gate, q_proxy, k_proxy, stream=None) -> PrefillResult:
        sgqa_prefill(self.prm, q, k, v, gate, q_proxy, k_proxy, self.q_start, self.k_blk, self.sel_idx, self.sel_cnt,
                     self.out, self.lse, self.ws, stream)
        return PrefillResult(self.out, self.lse, self.sel_idx, self.sel_cnt, self.k_blk)


def prefill(prm: Params, q, k, v, gate, q_proxy, k_proxy, q_start: int = 0, k_blk=None) -> PrefillResult:
    """One prefill of the layer on device tensors; allocates outputs and workspace."""
    plan = PrefillPlan(prm, q.shape[0], k.shape[1], q_start, device=q.device)
    if k_blk is not None:
        plan.k_blk = k_blk
    return plan.run(q, k, v, gate, q_proxy, k_proxy)


def _host(t: torch.Tensor | None, dtype, name: str, shape=None):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} host tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def sgqa_prefill_host(prm: Params, host: dict, dev: dict, q_start: int = 0, chunk_rows: int = 0, stream=None):
    """End-to-end prefill from host tensors (sgqa_prefill_host).  host: q, k, v, gate,
    q_proxy, k_proxy, out and optionally lse (pinned host tensors); dev: the device
    buffers q, k, v, gate, k_proxy, k_blk, out, lse (or None) and ws."""
    T = host["q"].shape[0]
    ctx_cap = host["k"].shape[1]
    lse_h = host.get("lse")
    ht = HostTensors(*[_host(host[n], BF16, n) for n in ("q", "k", "v", "gate", "q_proxy", "k_proxy", "out")],
                     _host(lse_h, F32, "lse"))
    dv = lambda n, dt=BF16: _dev(dev[n], dt, n)
    dt = DeviceTensors(dv("q"), dv("k"), dv("v"), dv("gate"), dv("k_proxy"), dv("k_blk"), dev["k_blk"].shape[1],
                       dv("out"), _dev(dev.get("lse"), F32, "lse"), _dev(dev["ws"], torch.uint8, "ws"),
                       dev["ws"].numel())
    _check(_lib.sgqa_prefill_host(ctypes.byref(prm), ctypes.byref(ht), ctypes.byref(dt), ctx_cap, T, q_start,
                                  chunk_rows, _stream(stream)), "sgqa_prefill_host")


class HostPrefill:
    """End-to-end prefill from HOST (pinned) tensors through sgqa_prefill_host: the library
    pipelines chunks of query rows over its copy-in stream, the calling stream and its
    copy-out stream.  This class only keeps the device buffers and the pinned output
    between calls.  The calling stream (or the current one) waits for the last copy back,
    so events recorded on it around `run` time the whole job."""

    def __init__(self, prm: Params, T: int, ctx_cap: int, q_start: int = 0, device="cuda", chunk_rows: int = 4096,
                 with_lse: bool = False):
        self.prm, self.T, self.ctx_cap, self.q_start, self.chunk_rows = prm, T, ctx_cap, q_start, chunk_rows
        G, H, D, P = prm.num_kv_groups, prm.num_kv_groups * prm.heads_per_group, prm.head_dim, prm.proxy_dim
        B = prm.block_size
        mk = lambda *s: torch.empty(s, dtype=BF16, device=device)
        gate_shape = (T, H, D) if prm.gate_per_dim else (T, H)
        self.d = dict(q=mk(T, H, D), k=mk(G, ctx_cap, D), v=mk(G, ctx_cap, D), gate=mk(*gate_shape),
                      k_proxy=mk(G, ctx_cap, P), out=mk(T, H, D),
                      k_blk=torch.zeros((G, (ctx_cap + B - 1) // B, P), dtype=BF16, device=device),
                      lse=torch.empty((T, H), dtype=F32, device=device) if with_lse else None)
        need = sgqa_workspace_bytes(prm, SGQA_OP_PREFILL_HOST, T, q_start + T, chunk_rows)
        if need == 0:
            raise ValueError("invalid prefill shape")
        self.d["ws"] = torch.empty(need, dtype=torch.uint8, device=device)
        self.out_host = torch.empty((T, H, D), dtype=BF16, pin_memory=True)
        self.lse_host = torch.empty((T, H), dtype=F32, pin_memory=True) if with_lse else None

    def h2d_bytes(self) -> int:
        G, P, D = self.prm.num_kv_groups, self.prm.proxy_dim, self.prm.head_dim
        ctx = self.q_start + self.T  # cache positions read
        rows = self.d["q"].numel() * 2 + self.d["gate"].numel() * 2 + G * self.T * P * 2
        return rows + G * ctx * (2 * D + P) * 2

    def d2h_bytes(self) -> int:
        n = self.out_host.numel() * self.out_host.element_size()
        return n + (self.lse_host.numel() * 4 if self.lse_host is not None else 0)

    def run(self, host: dict, stream=None) -> torch.Tensor:
        h = dict(host, out=self.out_host)
        if self.lse_host is not None:
            h["lse"] = self.lse_host
        sgqa_prefill_host(self.prm, h, self.d, self.q_start, self.chunk_rows, stream)
        return self.out_host
