"""Host-side checks of the C ABI: the library loads, exports exactly what include/sgqa.h
declares, and rejects bad arguments with the documented status codes before any kernel
is enqueued (no GPU is needed for these paths)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_long_18_b300 import build

    build.build()
    from block_sparse_long_18_b300 import sgqa

    return sgqa


def _declared():
    src = open(os.path.join(ROOT, "include", "sgqa.h")).read()
    return sorted(set(re.findall(r"SGQA_API\s+[\w\s\*]+?\b(sgqa_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports(lib):
    assert _declared() == sorted(lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(sgqa_\w+)", out))
    assert set(_declared()) == exported
    for name in _declared():
        assert hasattr(lib._lib, name)


def test_header_is_plain_c(tmp_path):
    """The header needs no CUDA, torch or C++ headers: it compiles as strict C99 and as C++11,
    and a C program can take the address of every declared entry point."""
    names = _declared()
    src = tmp_path / "use.c"
    src.write_text('#include "sgqa.h"\nint main(void) {\n  void* p[] = {' +
                   ", ".join(f"(void*){n}" for n in names) + "};\n  return p[0] == 0;\n}\n")
    inc = os.path.join(ROOT, "include")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", inc, "-fsyntax-only", str(src)],
                   check=True, capture_output=True)
    cpp = tmp_path / "use.cpp"
    cpp.write_text('#include "sgqa.h"\nint main() { return 0; }\n')
    subprocess.run(["g++", "-std=c++11", "-Wall", "-Wextra", "-Werror", "-I", inc, "-fsyntax-only", str(cpp)],
                   check=True, capture_output=True)


def test_abi_version(lib):
    assert lib.abi_version() == 2


def test_status_strings(lib):
    for code in range(7):
        assert lib._lib.sgqa_status_string(code)
    assert lib._lib.sgqa_status_string(99) == b"unknown status"


def _call_build(lib, prm, kp=1 << 12, ctx=64, b=0, e=64, kb=1 << 12, nb=8):
    return lib._lib.sgqa_build_block_index(ctypes.byref(prm) if prm is not None else None,
                                           ctypes.c_void_p(kp), ctx, b, e, ctypes.c_void_p(kb), nb, None)


def test_validation_codes(lib):
    prm = lib.params(G=1, Hg=4, k=8)
    assert _call_build(lib, None) == 1                                   # null params
    assert _call_build(lib, prm, kp=0) == 1                               # null tensor
    assert _call_build(lib, prm, b=10, e=5) == 1                          # inverted range
    assert _call_build(lib, prm, e=65) == 1                               # past ctx_cap
    assert _call_build(lib, prm, nb=7) == 1                               # blocks beyond nb_cap
    assert _call_build(lib, prm, kp=(1 << 12) + 2) == 1                   # misaligned
    assert _call_build(lib, lib.params(G=1, Hg=4, k=8, D=128)) == 2       # head_dim
    assert _call_build(lib, lib.params(G=1, Hg=32, k=8)) == 2             # heads per group
    assert _call_build(lib, lib.params(G=1, Hg=4, k=8, B=3)) == 2         # block size
    assert _call_build(lib, lib.params(G=1, Hg=4, k=8, P=96)) == 2        # proxy dim
    assert _call_build(lib, lib.params(G=1, Hg=4, k=0)) == 1              # k
    assert _call_build(lib, prm, b=5, e=5) == 0                           # empty range: nothing to do


def test_index_topk_validation(lib):
    prm = lib.params(G=1, Hg=4, k=8)
    f = lib._lib.sgqa_index_topk
    P = ctypes.c_void_p
    a = P(1 << 12)
    # workspace missing / too small
    assert f(ctypes.byref(prm), a, 256, 0, a, 32, a, a, None, 0, None) == 3
    assert f(ctypes.byref(prm), a, 256, 0, a, 32, a, a, a, 16, None) == 3
    # candidates beyond nb_cap
    assert f(ctypes.byref(prm), a, 256, 0, a, 16, a, a, a, 1 << 20, None) == 1
    # T = 0 is a no-op
    assert f(ctypes.byref(prm), a, 0, 0, a, 32, a, a, a, 1 << 20, None) == 0


def test_decode_validation(lib):
    prm = lib.params(G=1, Hg=4, k=8)
    P = ctypes.c_void_p
    a = P(1 << 12)
    cl = (ctypes.c_int64 * 2)(100, 50)
    off_bad = (ctypes.c_int64 * 2)(0, 3)       # not a multiple of B
    off_ok = (ctypes.c_int64 * 2)(0, 104)
    f = lib._lib.sgqa_decode
    assert f(ctypes.byref(prm), 2, cl, off_bad, a, a, a, a, a, None, a, 160, a, a, a, None, a, 1 << 24, None) == 1
    assert f(ctypes.byref(prm), 2, cl, off_ok, a, a, a, a, a, None, a, 150, a, a, a, None, a, 1 << 24, None) == 1
    assert f(ctypes.byref(prm), 0, cl, off_ok, a, a, a, a, a, None, a, 160, a, a, a, None, a, 1 << 24, None) == 1
    assert f(ctypes.byref(prm), 2, cl, off_ok, a, a, a, a, a, None, a, 160, a, a, a, None, a, 16, None) == 3


def test_workspace_sizes(lib):
    prm = lib.params()
    # 128K prefill: one pass of 8,192 rows x 4 groups x 16,384 fp32 candidates
    ws = lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_INDEX_TOPK, 131072, 131072)
    assert ws == 4 * 8192 * 16384 * 4
    # a 16K context (2,047 candidates at most): the same per-candidate layout
    assert lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_INDEX_TOPK, 16384, 16384) == 4 * 8192 * 2048 * 4
    # the 1M limit (rows past 16,384 candidates): the scores (or the survivors' keys in place)
    # [4 x 8,192 x 131,072], the segment + merge pair buffers (8 segments x 511 entries) of
    # the plain top-k, then the bound-filtered top-k's group maxima (a key per 8
    # candidates), bounds, survivor masks (a bit per candidate), row flags and 128-row tile
    # flags
    r = 4 * 8192
    w1 = lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_INDEX_TOPK, 8192, 1 << 20)
    seg = -(-r * 8 * 511 * 4 // 256) * 256
    assert w1 == r * 131072 * 4 + 2 * seg + r * 8 * 4 + r * 16384 * 4 + r * 4 + r * 4096 * 4 + (r * 4 + 4 * 64 * 4)
    # prefill: the indexer's scratch, reused by the grouped attention's sort keys, row order
    # and unit lists (4 groups x 131,072 rows x 13.5 bytes)
    wa = lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_ATTN, 131072, 131072)
    assert wa == 4 * 131072 * (8 + 4) + 3 * 4 * 16384 * 4 + 256
    assert lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_PREFILL, 131072, 131072) == ws
    assert lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_DECODE, 1, 1 << 20, 8) > 0
    assert lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_DECODE, 1, 1 << 20, 0) == 0
    assert lib.sgqa_workspace_bytes(lib.params(B=3), lib.SGQA_OP_PREFILL, 16, 16) == 0


def test_attention_kernel_choice(lib):
    """Which prefill attention kernel a call launches (no device access): the grouped mode
    (units of 8 rows with similar selections, each on the union or the warp-level kernel)
    wherever the union kernel's shape holds, up to 2M positions; the warp-level kernel for other shapes, dense mode and when forced; -1
    for a forced union outside its shape."""
    auto = lib.params()
    assert lib.sgqa_attention_kernel(auto, 131072, 0) == lib.ATTN_GROUPED
    assert lib.sgqa_attention_kernel(auto, 8192, 65536 * 8 - 8192) == lib.ATTN_GROUPED
    # once every unit's blocks span five or more 16,384-block windows the routing rule sends
    # no unit to the union kernel (100 * 5 * |union| > 55 * 8 * |union| >= 55 * pairs): the
    # warp-level kernel alone, without the grouping and routing launches (the 1M chunk)
    assert lib.sgqa_attention_kernel(auto, 8192, 65536 * 8) == lib.ATTN_WARP
    assert lib.sgqa_attention_kernel(auto, 8192, 1040384) == lib.ATTN_WARP
    assert lib.sgqa_attention_kernel(lib.params(attn_kernel=lib.ATTN_GROUPED), 8192, 1040384) == lib.ATTN_GROUPED
    assert lib.sgqa_attention_kernel(lib.params(attn_kernel=lib.ATTN_TC_UNION), 8192, 2097152 - 8192) == lib.ATTN_TC_UNION
    assert lib.sgqa_attention_kernel(lib.params(attn_kernel=lib.ATTN_TC_UNION), 8192, 2097152 - 8191) == -1  # past 2^18 blocks
    assert lib.sgqa_attention_kernel(auto, 1024, 0, dense_mode=True) == lib.ATTN_WARP
    assert lib.sgqa_attention_kernel(lib.params(B=4, k=1024), 1024, 0) == lib.ATTN_WARP
    assert lib.sgqa_attention_kernel(lib.params(Hg=8), 1024, 0) == lib.ATTN_WARP
    assert lib.sgqa_attention_kernel(lib.params(k=513), 1024, 0) == lib.ATTN_WARP
    warp = lib.params(attn_kernel=lib.ATTN_WARP)
    assert lib.sgqa_attention_kernel(warp, 131072, 0) == lib.ATTN_WARP
    union = lib.params(attn_kernel=lib.ATTN_TC_UNION)
    assert lib.sgqa_attention_kernel(union, 131072, 0) == lib.ATTN_TC_UNION
    assert lib.sgqa_attention_kernel(lib.params(B=16, k=256, attn_kernel=lib.ATTN_TC_UNION), 1024, 0) == -1
    assert lib.sgqa_attention_kernel(union, 1024, 0, dense_mode=True) == -1
    routed = lib.params(attn_kernel=lib.ATTN_ROUTED)
    assert lib.sgqa_attention_kernel(routed, 131072, 0) == lib.ATTN_ROUTED
    assert lib.sgqa_attention_kernel(lib.params(B=4, k=1024, attn_kernel=lib.ATTN_ROUTED), 1024, 0) == -1
    grouped = lib.params(attn_kernel=lib.ATTN_GROUPED)
    assert lib.sgqa_attention_kernel(grouped, 4096, 0) == lib.ATTN_GROUPED
    assert lib.sgqa_attention_kernel(lib.params(Hg=8, attn_kernel=lib.ATTN_GROUPED), 4096, 0) == -1
    assert lib.sgqa_attention_kernel(lib.params(attn_kernel=7), 1024, 0) == -1


def test_forced_union_outside_its_shape_is_rejected(lib):
    prm = lib.params(B=16, k=256, attn_kernel=lib.ATTN_TC_UNION)
    a = ctypes.c_void_p(1 << 12)
    f = lib._lib.sgqa_sparse_attn_fwd
    assert f(ctypes.byref(prm), a, a, a, 4096, a, a, a, 1024, 0, a, None, 0, None, 0, None) == 2
    assert f(ctypes.byref(lib.params(attn_kernel=9)), a, a, a, 4096, a, a, a, 1024, 0, a, None, 0, None, 0, None) == 1
    # the routed and grouped modes forced without their workspace (a choice and two lists per
    # 8-row unit, the row order)
    routed = lib.params(attn_kernel=lib.ATTN_ROUTED)
    need = lib.sgqa_workspace_bytes(routed, lib.SGQA_OP_ATTN, 1024, 4096)
    assert need >= 4 * 128 * 12 + 256 + 4 * 1024 * 12
    assert f(ctypes.byref(routed), a, a, a, 4096, a, a, a, 1024, 3072, a, None, 0, a, need - 256, None) == 3
    grouped = lib.params(attn_kernel=lib.ATTN_GROUPED)
    assert f(ctypes.byref(grouped), a, a, a, 4096, a, a, a, 1024, 3072, a, None, 0, None, 0, None) == 3
    # no workspace needed where the union kernel cannot serve
    assert lib.sgqa_workspace_bytes(lib.params(B=4, k=1024), lib.SGQA_OP_ATTN, 1024, 4096) == 256


def test_prefill_host_validation(lib):
    prm = lib.params(G=1, Hg=16, k=8)
    a = 1 << 12
    ht = lib.HostTensors(a, a, a, a, a, a, a, None)
    ws_need = lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_PREFILL_HOST, 1000, 1000, 256)
    assert ws_need > 0
    dt = lambda ws_bytes, lse=None, nb=125: lib.DeviceTensors(a, a, a, a, a, a, nb, a, lse, a, ws_bytes)
    f = lambda h, d, T=1000, q0=0, cap=1000, chunk=256: lib._lib.sgqa_prefill_host(
        ctypes.byref(prm), ctypes.byref(h), ctypes.byref(d), cap, T, q0, chunk, None)
    assert f(ht, dt(ws_need - 1)) == 3                       # workspace too small
    assert f(ht, dt(ws_need), T=1001) == 1                   # rows past the cache
    assert f(ht, dt(ws_need, nb=124)) == 1                   # blocks beyond nb_cap
    assert f(lib.HostTensors(a, a, a, a, a, a, None, None), dt(ws_need)) == 1   # no host output
    assert f(lib.HostTensors(a, a, a, a, a, a, a, a), dt(ws_need)) == 1         # host lse without device lse
    assert f(ht, dt(ws_need), T=0) == 0                      # nothing to do
    # the chunk size moves the workspace: two q_proxy chunks, the chunk's selection, one indexer pass
    assert lib.sgqa_workspace_bytes(prm, lib.SGQA_OP_PREFILL_HOST, 1000, 1000, 512) > ws_need
