"""CPU oracle for MoE expert-parallel dispatch / combine (TEST INFRASTRUCTURE).

Only the tests, the package's smoke check and the benchmark's CPU-baseline arm
may import this package.  It wraps ``ep_oracle.c`` (plain single-threaded C)
with ctypes and numpy; it shares no code with the CUDA library and never calls
it.  The C file states what each function computes and which page passage it
follows.

Every function here takes and returns numpy arrays on the host.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from ._build import LIB, build_oracle

__all__ = ["STATUS_BAD_EXPERT", "STATUS_CAPACITY", "QUANT_BF16", "QUANT_FP8",
           "layout", "dispatch", "combine", "localize_ids", "layout_experts", "combine_weighted",
           "cast_transpose", "cast_transpose_t_bytes", "bf16_from_f32", "e4m3_from_f32",
           "f32_from_e4m3", "f32_from_bf16", "run_all"]

STATUS_BAD_EXPERT = 1
STATUS_CAPACITY = 2
QUANT_BF16 = 0
QUANT_FP8 = 1

_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(LIB)
        lib.ep_ref_layout.argtypes = [_P, _I64, _I, _I, _I, _P, _P, _P, _P, _P]
        lib.ep_ref_layout.restype = _I
        lib.ep_ref_dispatch.argtypes = [_P, _P, _P, _I64, _I, _I, _I, _P, _I64, _I,
                                        _P, _P, _P, _P, _P, _P]
        lib.ep_ref_dispatch.restype = _I
        lib.ep_ref_combine.argtypes = [_P, _P, _I64, _I, _I, _I64, _P, _P, _P]
        lib.ep_ref_combine.restype = _I
        lib.ep_ref_bf16_from_f32_array.argtypes = [_P, _I64, _P]
        lib.ep_ref_bf16_from_f32_array.restype = None
        lib.ep_ref_e4m3_from_f32_array.argtypes = [_P, _I64, _P]
        lib.ep_ref_e4m3_from_f32_array.restype = None
        lib.ep_ref_cast_transpose.argtypes = [_P, _P, _I, _I, _P, _P, _P, _P]
        lib.ep_ref_cast_transpose.restype = _I
        lib.ep_ref_layout_experts.argtypes = [_P, _I64, _I, _I, _P, _P, _P, _P, _P]
        lib.ep_ref_layout_experts.restype = _I
        lib.ep_ref_combine_weighted.argtypes = [_P, _P, _P, _I64, _I, _I, _I64, _P, _P, _P]
        lib.ep_ref_combine_weighted.restype = _I
        lib.ep_ref_localize_ids.argtypes = [_P, _I64, _I, _I, _I, _P]
        lib.ep_ref_localize_ids.restype = _I
        lib.ep_ref_f32_from_e4m3.argtypes = [ctypes.c_uint8]
        lib.ep_ref_f32_from_e4m3.restype = ctypes.c_float
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def layout(topk_idx: np.ndarray, E: int, W: int) -> dict:
    """Routing layout: per-expert counts, per-rank counts, rank_offset, slot, status."""
    lib = _load()
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    ne = np.zeros(E, np.int32)
    nr = np.zeros(W, np.int32)
    off = np.zeros(W + 1, np.int32)
    slot = np.zeros((T, W), np.int32)
    st = np.zeros(1, np.int32)
    rc = lib.ep_ref_layout(_ptr(idx), T, k, E, W, _ptr(ne), _ptr(nr), _ptr(off), _ptr(slot), _ptr(st))
    if rc != 0:
        raise ValueError("oracle layout: invalid arguments")
    return {"num_tokens_per_expert": ne, "num_tokens_per_rank": nr, "rank_offset": off,
            "slot": slot, "status": int(st[0])}


def dispatch(x: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray, slot: np.ndarray,
             cap: int, quant: int = QUANT_BF16, fill: int = 0) -> dict:
    """Dispatch into receive buffers of ``cap`` rows (unwritten rows keep ``fill``)."""
    lib = _load()
    x = _c(x, np.uint16)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_w, np.float32)
    slot = _c(slot, np.int32)
    T, H = x.shape
    k = idx.shape[1]
    W = slot.shape[1]
    if quant == QUANT_BF16:
        recv_x = np.full((cap, H), fill, np.uint16)
        recv_scale = np.zeros((0,), np.float32)
    else:
        recv_x = np.full((cap, H), fill & 0xFF, np.uint8)
        recv_scale = np.zeros((cap, H // 128), np.float32)
    ridx = np.full((cap, k), -1, np.int32)
    rw = np.zeros((cap, k), np.float32)
    rsrc = np.full((cap,), -1, np.int32)
    st = np.zeros(1, np.int32)
    rc = lib.ep_ref_dispatch(_ptr(x), _ptr(idx), _ptr(w), T, H, k, W, _ptr(slot), cap, quant,
                             _ptr(recv_x), _ptr(recv_scale), _ptr(ridx), _ptr(rw), _ptr(rsrc), _ptr(st))
    if rc != 0:
        raise ValueError("oracle dispatch: invalid arguments")
    out = {"recv_x": recv_x, "recv_topk_idx": ridx, "recv_topk_w": rw, "recv_src": rsrc,
           "status": int(st[0])}
    if quant == QUANT_FP8:
        out["recv_scale"] = recv_scale
    return out


def localize_ids(recv_topk_idx: np.ndarray, E: int, W: int, rank_offset: np.ndarray) -> np.ndarray:
    """Local-id metadata: ids of rank r's receive rows become e - r*(E/W) for
    experts hosted by r, -1 otherwise (returns a new array)."""
    lib = _load()
    ids = np.array(recv_topk_idx, dtype=np.int32, copy=True, order="C")
    off = _c(rank_offset, np.int32)
    rc = lib.ep_ref_localize_ids(_ptr(ids), ids.shape[0], ids.shape[1], E, W, _ptr(off))
    if rc != 0:
        raise ValueError("oracle localize_ids: invalid arguments")
    return ids


def layout_experts(topk_idx: np.ndarray, E: int) -> dict:
    """Expert-major layout: per-expert counts, expert_offset [E+1], slot [T, k]."""
    lib = _load()
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    ne = np.zeros(E, np.int32)
    off = np.zeros(E + 1, np.int32)
    slot = np.zeros((T, k), np.int32)
    nxt = np.zeros(E, np.int32)
    st = np.zeros(1, np.int32)
    rc = lib.ep_ref_layout_experts(_ptr(idx), T, k, E, _ptr(ne), _ptr(off), _ptr(slot), _ptr(nxt),
                                   _ptr(st))
    if rc != 0:
        raise ValueError("oracle layout_experts: invalid arguments")
    return {"num_tokens_per_expert": ne, "expert_offset": off, "slot": slot, "status": int(st[0])}


def combine_weighted(y: np.ndarray, slot: np.ndarray, w: np.ndarray, cap: int | None = None) -> dict:
    """Weighted combine: fp32 fused multiply-add chain over the slot columns in order."""
    lib = _load()
    y = _c(y, np.uint16)
    slot = _c(slot, np.int32)
    w = _c(w, np.float32)
    T, C = slot.shape
    H = y.shape[1]
    cap = y.shape[0] if cap is None else cap
    out = np.zeros((T, H), np.uint16)
    acc = np.zeros(H, np.float32)
    st = np.zeros(1, np.int32)
    rc = lib.ep_ref_combine_weighted(_ptr(y), _ptr(slot), _ptr(w), T, H, C, cap, _ptr(out),
                                     _ptr(acc), _ptr(st))
    if rc != 0:
        raise ValueError("oracle combine_weighted: invalid arguments")
    return {"out": out, "status": int(st[0])}


def cast_transpose_t_bytes(expert_offset: np.ndarray, H: int) -> int:
    n = np.diff(np.asarray(expert_offset, np.int64))
    return int(H * ((n + 15) // 16 * 16).sum())


def cast_transpose(y: np.ndarray, expert_offset: np.ndarray, scale: np.ndarray,
                   amax: np.ndarray | None = None) -> dict:
    """FP8 cast and per-expert transposed cast of the expert-major rows; amax
    starts from ``amax`` (zeros by default)."""
    lib = _load()
    y = _c(y, np.uint16)
    off = _c(expert_offset, np.int32)
    sc = _c(scale, np.float32)
    E = off.size - 1
    H = y.shape[1]
    R = int(off[-1])
    out_c = np.zeros((R, H), np.uint8)
    out_t = np.zeros(cast_transpose_t_bytes(off, H), np.uint8)
    am = np.zeros(E, np.float32) if amax is None else _c(amax, np.float32).copy()
    rc = lib.ep_ref_cast_transpose(_ptr(y), _ptr(off), E, H, _ptr(sc), _ptr(out_c), _ptr(out_t),
                                   _ptr(am))
    if rc != 0:
        raise ValueError("oracle cast_transpose: invalid arguments")
    return {"out_c": out_c, "out_t": out_t, "amax": am}


def combine(y: np.ndarray, slot: np.ndarray, cap: int | None = None) -> dict:
    """Combine: fp32 ascending-rank sum of each token's rows, rounded to bf16."""
    lib = _load()
    y = _c(y, np.uint16)
    slot = _c(slot, np.int32)
    T, W = slot.shape
    H = y.shape[1]
    cap = y.shape[0] if cap is None else cap
    out = np.zeros((T, H), np.uint16)
    acc = np.zeros(H, np.float32)
    st = np.zeros(1, np.int32)
    rc = lib.ep_ref_combine(_ptr(y), _ptr(slot), T, H, W, cap, _ptr(out), _ptr(acc), _ptr(st))
    if rc != 0:
        raise ValueError("oracle combine: invalid arguments")
    return {"out": out, "status": int(st[0])}


def bf16_from_f32(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().ep_ref_bf16_from_f32_array(_ptr(a), a.size, _ptr(out))
    return out


def e4m3_from_f32(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().ep_ref_e4m3_from_f32_array(_ptr(a), a.size, _ptr(out))
    return out


def f32_from_e4m3(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, np.uint8).ravel()
    return np.array([lib.ep_ref_f32_from_e4m3(int(v)) for v in c], np.float32).reshape(np.shape(codes))


def f32_from_bf16(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def run_all(inputs: dict, quant: int | None = None, y: np.ndarray | None = None,
            cap: int | None = None) -> dict:
    """Layout, dispatch and combine of one input set.  Combine reads ``y`` when
    given, else the dispatched rows themselves (identity experts, bf16 only)."""
    cfg = inputs["cfg"]
    if quant is None:
        quant = QUANT_FP8 if cfg.quant == "fp8" else QUANT_BF16
    lay = layout(inputs["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    cap = R if cap is None else cap
    dis = dispatch(inputs["x"], inputs["topk_idx"], inputs["topk_w"], lay["slot"], cap, quant)
    if y is None and quant == QUANT_BF16:
        y = dis["recv_x"]
    com = combine(y, lay["slot"], cap) if y is not None else None
    return {"layout": lay, "dispatch": dis, "combine": com, "R": R, "cap": cap}
