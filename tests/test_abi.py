"""The C ABI library builds, loads and exports every entry point that
include/ep_gb300.h declares; host-side argument checks reject bad calls before
anything reaches a GPU.  No compute call is made here."""
import ctypes
import os
import re

import pytest
import torch

import combine_ep_dispatch_gb300 as ep
from combine_ep_dispatch_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep_gb300.h")


@pytest.fixture(scope="module")
def lib():
    _build.build_library()
    return _lib.load_library()


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^EP_API\s+[\w\s\*]+?\b(ep_\w+)\s*\(", txt, re.M)))


def test_header_declares_the_calls():
    assert _declared() == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_enum_values_match_header():
    txt = open(HEADER).read()
    for name in ("EP_OK", "EP_ERR_INVALID_ARG", "EP_ERR_MISALIGNED", "EP_ERR_UNSUPPORTED",
                 "EP_ERR_CUDA", "EP_ERR_WORKSPACE", "EP_STATUS_BAD_EXPERT", "EP_STATUS_CAPACITY",
                 "EP_STATUS_TIMEOUT",
                 "EP_QUANT_BF16", "EP_QUANT_FP8_E4M3_B128"):
        m = re.search(rf"\b{name}\s*=\s*(\d+)", txt)
        assert m and int(m.group(1)) == getattr(_lib, name), name


def test_size_queries(lib):
    assert ep.ep_max_recv_rows(4096, 8, 8) == 32768
    assert ep.ep_max_recv_rows(100, 2, 8) == 200
    assert ep.ep_max_recv_rows(-1, 8, 8) == -1
    assert ep.ep_layout_workspace_bytes(4096, 8, 256) >= 4096 * 4
    assert ep.ep_layout_workspace_bytes(0, 8, 256) > 0
    assert ep.ep_layout_workspace_bytes(10, 33, 66) == 0
    for code in range(6):
        assert ep.ep_status_string(code).startswith("EP_")
    # kernels per ep_dispatch_with_layout call
    L = ep.ep_dispatch_with_layout_launches
    assert L(4096, 7168, 8, 8) == 2      # count + finishing dispatch
    assert L(4096, 7168, 8, 8, 1) == 2   # FP8: count + finishing dispatch
    assert L(1024, 7168, 8, 8, 1) == 2   # one-CTA layout + FP8 dispatch
    assert L(4096, 256, 8, 8) == 3       # rows under 1 KB: count + scan + dispatch
    assert L(1024, 7168, 8, 8) == 2      # one-CTA layout + dispatch
    assert L(512, 7168, 8, 8) == 1       # one-launch dispatch
    assert L(256, 7168, 20, 8) == 2      # k > 16: one-CTA layout + dispatch
    assert L(256, 7168, 8, 8, 1) == 2    # FP8 never takes the one-launch kernel
    assert L(0, 7168, 8, 8) == 1
    assert L(300000, 7168, 8, 8) == 3    # chunk table over 16 KB
    assert L(4096, 7168, 8, 33) == -1


# The calls below pass made-up device addresses that each violate one rule, so
# they must return before any CUDA call.  They are skipped where a GPU exists:
# there the same paths are covered with real tensors by the GPU tests.
cpu_only = pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers: CPU machines only")

A = 0x10000  # a 64 KiB-aligned fake address (never dereferenced)


@cpu_only
@pytest.mark.parametrize("args,code", [
    # (T, k, E, W, workspace_bytes, ptr offsets)
    ((100, 8, 256, 3, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),       # E % W != 0
    ((100, 8, 256, 33, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),      # W > 32
    ((100, 0, 256, 8, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),       # k < 1
    ((-1, 8, 256, 8, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),        # T < 0
    ((100, 8, 16384, 8, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),     # E > 8192
    ((100, 8, 256, 8, 16, 0), _lib.EP_ERR_WORKSPACE),              # workspace too small
    ((100, 8, 256, 8, 1 << 20, 2), _lib.EP_ERR_MISALIGNED),        # slot 2-byte aligned
    ((1 << 29, 8, 256, 8, 1 << 40, 0), _lib.EP_ERR_UNSUPPORTED),   # rows overflow int32
])
def test_layout_rejects(lib, args, code):
    T, k, E, W, wsb, off = args
    rc = lib.ep_dispatch_layout(A, T, k, E, W, A, A, A, A + off, A, wsb, None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(H=7), _lib.EP_ERR_UNSUPPORTED),                       # H % 8 for bf16
    (dict(H=136, quant=1), _lib.EP_ERR_UNSUPPORTED),            # H % 128 for FP8
    (dict(quant=7), _lib.EP_ERR_INVALID_ARG),
    (dict(x_off=8), _lib.EP_ERR_MISALIGNED),                    # x 8-byte aligned
    (dict(recv_off=4), _lib.EP_ERR_MISALIGNED),
    (dict(cap=-1), _lib.EP_ERR_INVALID_ARG),
    (dict(W=0), _lib.EP_ERR_INVALID_ARG),
    (dict(quant=1, H=256, scale_null=True), _lib.EP_ERR_INVALID_ARG),
    (dict(x_null=True), _lib.EP_ERR_INVALID_ARG),
])
def test_dispatch_rejects(lib, kw, code):
    H = kw.get("H", 256)
    quant = kw.get("quant", 0)
    x = None if kw.get("x_null") else A + kw.get("x_off", 0)
    scale = None if kw.get("scale_null") else A
    rc = lib.ep_dispatch(x, A, A, 100, H, 8, kw.get("W", 8), A, kw.get("cap", 800), quant,
                         A + kw.get("recv_off", 0), scale, A, A, A, None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),
    (dict(y_off=2), _lib.EP_ERR_MISALIGNED),
    (dict(out_off=8), _lib.EP_ERR_MISALIGNED),
    (dict(W=40), _lib.EP_ERR_INVALID_ARG),
    (dict(out_null=True), _lib.EP_ERR_INVALID_ARG),
])
def test_combine_rejects(lib, kw, code):
    out = None if kw.get("out_null") else A + kw.get("out_off", 0)
    rc = lib.ep_combine(A + kw.get("y_off", 0), A, 100, kw.get("H", 256), kw.get("W", 8), 800, out,
                        None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(W=33), _lib.EP_ERR_INVALID_ARG),                      # layout's check
    (dict(E=100), _lib.EP_ERR_INVALID_ARG),                     # E % W != 0
    (dict(ws=64), _lib.EP_ERR_WORKSPACE),                       # layout workspace too small
    (dict(slot_off=2), _lib.EP_ERR_MISALIGNED),
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),                      # dispatch's check: H % 8
    (dict(H=200, quant=1), _lib.EP_ERR_UNSUPPORTED),            # FP8 needs H % 128
    (dict(quant=7), _lib.EP_ERR_INVALID_ARG),
    (dict(x_off=8), _lib.EP_ERR_MISALIGNED),
    (dict(scale_null=True, quant=1), _lib.EP_ERR_INVALID_ARG),  # FP8 without recv_scale
])
def test_dispatch_with_layout_rejects(lib, kw, code):
    scale = None if kw.get("scale_null") else A
    rc = lib.ep_dispatch_with_layout(
        A + kw.get("x_off", 0), A, A, 256, kw.get("H", 256), 8, kw.get("E", 256), kw.get("W", 8),
        A, A, A, A + kw.get("slot_off", 0), A, kw.get("ws", 1 << 20), 2048, kw.get("quant", 0), A,
        scale, A, A, A, None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(E=5000), _lib.EP_ERR_INVALID_ARG),                    # expert layout's check
    (dict(ws=64), _lib.EP_ERR_WORKSPACE),
    (dict(k=40), _lib.EP_ERR_UNSUPPORTED),                      # k slot columns > 32
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),                      # dispatch's check
    (dict(x_off=8), _lib.EP_ERR_MISALIGNED),
    (dict(quant=5), _lib.EP_ERR_INVALID_ARG),
])
def test_experts_with_layout_rejects(lib, kw, code):
    rc = lib.ep_dispatch_experts_with_layout(
        A + kw.get("x_off", 0), A, A, 256, kw.get("H", 256), kw.get("k", 8), kw.get("E", 256), A, A,
        A, A, kw.get("ws", 1 << 20), 2048, kw.get("quant", 0), A, A, A, A, A, None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(T=1025), _lib.EP_ERR_UNSUPPORTED),                    # beyond EP_FUSED_MAX_TOKENS
    (dict(k=17), _lib.EP_ERR_UNSUPPORTED),
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),
    (dict(E=100), _lib.EP_ERR_INVALID_ARG),                     # E % W != 0
    (dict(x_off=4), _lib.EP_ERR_MISALIGNED),
])
def test_fused_rejects(lib, kw, code):
    rc = lib.ep_dispatch_fused(A + kw.get("x_off", 0), A, A, kw.get("T", 256), kw.get("H", 256),
                               kw.get("k", 8), kw.get("E", 256), 8, A, A, A, A, 2048, A, A, A, A,
                               None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("args,code", [
    # (T, k, E, workspace_bytes, slot offset)
    ((100, 8, 5000, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),      # E > 4096
    ((100, 0, 256, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),       # k < 1
    ((-3, 8, 256, 1 << 20, 0), _lib.EP_ERR_INVALID_ARG),        # T < 0
    ((100000, 8, 256, 64, 0), _lib.EP_ERR_WORKSPACE),           # workspace too small
    ((100, 8, 256, 1 << 20, 2), _lib.EP_ERR_MISALIGNED),        # slot 2-byte aligned
    ((1 << 29, 8, 256, 1 << 40, 0), _lib.EP_ERR_UNSUPPORTED),   # rows overflow int32
])
def test_layout_experts_rejects(lib, args, code):
    T, k, E, wsb, off = args
    rc = lib.ep_dispatch_layout_experts(A, T, k, E, A, A, A + off, A, wsb, None, None)
    assert rc == code


def test_layout_experts_workspace_size(lib):
    assert ep.ep_layout_experts_workspace_bytes(4096, 8, 256) >= 32 * 256 * 4 + 256 * 4
    assert ep.ep_layout_experts_workspace_bytes(0, 8, 256) > 0
    assert ep.ep_layout_experts_workspace_bytes(10, 0, 256) == 0


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),
    (dict(C=33), _lib.EP_ERR_INVALID_ARG),
    (dict(C=0), _lib.EP_ERR_INVALID_ARG),
    (dict(w_null=True), _lib.EP_ERR_INVALID_ARG),
    (dict(w_off=2), _lib.EP_ERR_MISALIGNED),
    (dict(y_off=4), _lib.EP_ERR_MISALIGNED),
])
def test_combine_weighted_rejects(lib, kw, code):
    w = None if kw.get("w_null") else A + kw.get("w_off", 0)
    rc = lib.ep_combine_weighted(A + kw.get("y_off", 0), A, w, 100, kw.get("H", 256), kw.get("C", 8),
                                 800, A, None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(H=7168 + 128), _lib.EP_ERR_UNSUPPORTED),             # H % 256
    (dict(E=0), _lib.EP_ERR_INVALID_ARG),
    (dict(E=9000), _lib.EP_ERR_INVALID_ARG),
    (dict(t_off=8), _lib.EP_ERR_MISALIGNED),                   # out_t 8-byte aligned
    (dict(scale_null=True), _lib.EP_ERR_INVALID_ARG),
    (dict(cap=-1), _lib.EP_ERR_INVALID_ARG),
])
def test_cast_transpose_rejects(lib, kw, code):
    scale = None if kw.get("scale_null") else A
    rc = lib.ep_cast_transpose_experts(A, A, kw.get("E", 256), kw.get("H", 7168), scale,
                                       kw.get("cap", 1000), A, A + kw.get("t_off", 0), A, None, None)
    assert rc == code


def test_cast_transpose_t_bytes(lib):
    assert ep.ep_cast_transpose_t_bytes(32768, 256, 7168) == 7168 * (32768 + 15 * 256)
    assert ep.ep_cast_transpose_t_bytes(-1, 256, 7168) == 0


def test_binding_rejects_host_tensors(lib):
    idx = torch.zeros(4, 2, dtype=torch.int32)
    with pytest.raises(ValueError):
        ep.ep_dispatch_layout(idx, 4, 2, idx, idx, idx, idx, idx)


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load_library()


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(W=0), _lib.EP_ERR_INVALID_ARG),
    (dict(W=33), _lib.EP_ERR_INVALID_ARG),
    (dict(table_null=True), _lib.EP_ERR_INVALID_ARG),
    (dict(off_null=True), _lib.EP_ERR_INVALID_ARG),
    (dict(rows=-1), _lib.EP_ERR_INVALID_ARG),
    (dict(region_off=8), _lib.EP_ERR_MISALIGNED),               # a region's rows 8-byte aligned
    (dict(quant=1, scale_null=True), _lib.EP_ERR_INVALID_ARG),  # FP8 region without scales
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),
])
def test_dispatch_regions_rejects(lib, kw, code):
    W = kw.get("W", 8)
    n = max(W, 1)
    table = (_lib.RankRegion * n)()
    for r in range(n):
        table[r] = _lib.RankRegion(A + 0x100000 * r + (kw.get("region_off", 0) if r == 3 else 0),
                                   None if kw.get("scale_null") else A, A, A, A,
                                   kw.get("rows", 100))
    rc = lib.ep_dispatch_regions(A, A, A, 100, kw.get("H", 256), 8, W, A,
                                 None if kw.get("off_null") else A,
                                 None if kw.get("table_null") else table, kw.get("quant", 0),
                                 None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(W=33), _lib.EP_ERR_INVALID_ARG),
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),
    (dict(rows=-5), _lib.EP_ERR_INVALID_ARG),
    (dict(y_off=4), _lib.EP_ERR_MISALIGNED),
    (dict(out_off=8), _lib.EP_ERR_MISALIGNED),
    (dict(off_null=True), _lib.EP_ERR_INVALID_ARG),
])
def test_combine_regions_rejects(lib, kw, code):
    W = kw.get("W", 8)
    ptrs = (ctypes.c_void_p * W)(*[A + 0x100000 * r + kw.get("y_off", 0) for r in range(W)])
    rows = (ctypes.c_int64 * W)(*[kw.get("rows", 100)] * W)
    rc = lib.ep_combine_regions(ptrs, rows, A, None if kw.get("off_null") else A, 100,
                                kw.get("H", 256), W, A + kw.get("out_off", 0), None, None)
    assert rc == code


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(W=0), _lib.EP_ERR_INVALID_ARG),
    (dict(W=33), _lib.EP_ERR_INVALID_ARG),
    (dict(E=60), _lib.EP_ERR_INVALID_ARG),                      # E not a multiple of W
    (dict(table_null=True), _lib.EP_ERR_INVALID_ARG),
    (dict(rows=-1), _lib.EP_ERR_INVALID_ARG),
    (dict(region_off=8), _lib.EP_ERR_MISALIGNED),
    (dict(quant=1, scale_null=True), _lib.EP_ERR_INVALID_ARG),
    (dict(H=12), _lib.EP_ERR_UNSUPPORTED),
    (dict(ws_bytes=16), _lib.EP_ERR_WORKSPACE),
])
def test_dispatch_regions_with_layout_rejects(lib, kw, code):
    W = kw.get("W", 8)
    n = max(W, 1)
    table = (_lib.RankRegion * n)()
    for r in range(n):
        table[r] = _lib.RankRegion(A + 0x100000 * r + (kw.get("region_off", 0) if r == 3 else 0),
                                   None if kw.get("scale_null") else A, A, A, A,
                                   kw.get("rows", 100))
    T, E, k = 100, kw.get("E", 64), 8
    ws = kw.get("ws_bytes", ep.ep_layout_workspace_bytes(T, max(min(W, 32), 1), 64) + 4096)
    rc = lib.ep_dispatch_regions_with_layout(
        A, A, A, T, kw.get("H", 256), k, E, W, A, A, A, A, A, ws,
        None if kw.get("table_null") else table, kw.get("quant", 0), None, None)
    assert rc == code
