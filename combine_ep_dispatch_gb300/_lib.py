"""Thin ctypes binding of libep_gb300.so (the C ABI declared in include/ep_gb300.h).

Argument marshalling only: every function takes torch CUDA tensors (and the
caller's stream), passes raw device pointers and sizes to the library, and
raises EPError on a non-zero return code.  All computation happens in the
library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_MISALIGNED = 2
EP_ERR_UNSUPPORTED = 3
EP_ERR_CUDA = 4
EP_ERR_WORKSPACE = 5

EP_STATUS_BAD_EXPERT = 1
EP_STATUS_CAPACITY = 2
EP_STATUS_TIMEOUT = 4

EP_QUANT_BF16 = 0
EP_QUANT_FP8_E4M3_B128 = 1

EXPORTED = ("ep_layout_workspace_bytes", "ep_max_recv_rows", "ep_dispatch_layout", "ep_dispatch",
            "ep_combine", "ep_status_string", "ep_dispatch_layout_noalloc", "ep_dispatch_fused",
            "ep_localize_expert_ids", "ep_layout_experts_workspace_bytes",
            "ep_dispatch_layout_experts", "ep_combine_weighted", "ep_selftest_wait_timeout",
            "ep_cast_transpose_t_bytes", "ep_cast_transpose_experts", "ep_dispatch_with_layout",
            "ep_dispatch_with_layout_launches", "ep_dispatch_experts_with_layout",
            "ep_dispatch_regions", "ep_combine_regions", "ep_dispatch_regions_with_layout")

# Largest batch ep_dispatch_fused takes.
EP_FUSED_MAX_TOKENS = 1024

# Size of the library's built-in layout workspace (ep_dispatch_layout_noalloc).
EP_LAYOUT_NOALLOC_SCRATCH_BYTES = 1 << 20


class RankRegion(ctypes.Structure):
    """ep_rank_region_t: the receive storage of one rank (device pointers)."""
    _fields_ = [("recv_x", ctypes.c_void_p), ("recv_scale", ctypes.c_void_p),
                ("recv_topk_idx", ctypes.c_void_p), ("recv_topk_w", ctypes.c_void_p),
                ("recv_src", ctypes.c_void_p), ("rows", ctypes.c_int64)]


class EPError(RuntimeError):
    """A host-side EP_ERR_* code returned by a library call (``code``)."""
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} failed with code {code}: {text}")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


def load_library() -> ctypes.CDLL:
    """Load libep_gb300.so; raises ImportError when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    lib.ep_layout_workspace_bytes.argtypes = [_I64, _I, _I]
    lib.ep_layout_workspace_bytes.restype = ctypes.c_size_t
    lib.ep_max_recv_rows.argtypes = [_I64, _I, _I]
    lib.ep_max_recv_rows.restype = _I64
    lib.ep_dispatch_layout.argtypes = [_P, _I64, _I, _I, _I, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                       _P, _P]
    lib.ep_dispatch_layout.restype = _I
    lib.ep_dispatch.argtypes = [_P, _P, _P, _I64, _I, _I, _I, _P, _I64, _I, _P, _P, _P, _P, _P,
                                _P, _P]
    lib.ep_dispatch.restype = _I
    lib.ep_dispatch_with_layout.argtypes = [_P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                            ctypes.c_size_t, _I64, _I, _P, _P, _P, _P, _P, _P, _P]
    lib.ep_dispatch_with_layout.restype = _I
    lib.ep_dispatch_experts_with_layout.argtypes = [_P, _P, _P, _I64, _I, _I, _I, _P, _P, _P, _P,
                                                    ctypes.c_size_t, _I64, _I, _P, _P, _P, _P, _P,
                                                    _P, _P]
    lib.ep_dispatch_experts_with_layout.restype = _I
    lib.ep_dispatch_with_layout_launches.argtypes = [_I64, _I, _I, _I, _I]
    lib.ep_dispatch_with_layout_launches.restype = _I
    lib.ep_combine.argtypes = [_P, _P, _I64, _I, _I, _I64, _P, _P, _P]
    lib.ep_combine.restype = _I
    lib.ep_dispatch_layout_noalloc.argtypes = [_P, _I64, _I, _I, _I, _P, _P, _P, _P, _P, _P]
    lib.ep_dispatch_layout_noalloc.restype = _I
    lib.ep_dispatch_fused.argtypes = [_P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _P, _I64, _P,
                                      _P, _P, _P, _P, _P]
    lib.ep_dispatch_fused.restype = _I
    lib.ep_localize_expert_ids.argtypes = [_P, _P, _I64, _I, _I, _I, _P]
    lib.ep_localize_expert_ids.restype = _I
    lib.ep_layout_experts_workspace_bytes.argtypes = [_I64, _I, _I]
    lib.ep_layout_experts_workspace_bytes.restype = ctypes.c_size_t
    lib.ep_dispatch_layout_experts.argtypes = [_P, _I64, _I, _I, _P, _P, _P, _P, ctypes.c_size_t,
                                               _P, _P]
    lib.ep_dispatch_layout_experts.restype = _I
    lib.ep_combine_weighted.argtypes = [_P, _P, _P, _I64, _I, _I, _I64, _P, _P, _P]
    lib.ep_combine_weighted.restype = _I
    lib.ep_cast_transpose_t_bytes.argtypes = [_I64, _I, _I]
    lib.ep_cast_transpose_t_bytes.restype = ctypes.c_size_t
    lib.ep_cast_transpose_experts.argtypes = [_P, _P, _I, _I, _P, _I64, _P, _P, _P, _P, _P]
    lib.ep_cast_transpose_experts.restype = _I
    lib.ep_dispatch_regions.argtypes = [_P, _P, _P, _I64, _I, _I, _I, _P, _P,
                                        ctypes.POINTER(RankRegion), _I, _P, _P]
    lib.ep_dispatch_regions.restype = _I
    lib.ep_dispatch_regions_with_layout.argtypes = [_P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P,
                                                    _P, _P, ctypes.c_size_t,
                                                    ctypes.POINTER(RankRegion), _I, _P, _P]
    lib.ep_dispatch_regions_with_layout.restype = _I
    lib.ep_combine_regions.argtypes = [ctypes.POINTER(ctypes.c_void_p),
                                       ctypes.POINTER(ctypes.c_int64), _P, _P, _I64, _I, _I, _P,
                                       _P, _P]
    lib.ep_combine_regions.restype = _I
    lib.ep_selftest_wait_timeout.argtypes = [_P, _P]
    lib.ep_selftest_wait_timeout.restype = _I
    lib.ep_status_string.argtypes = [_I]
    lib.ep_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(t: torch.Tensor | None):
    # a plain int: ctypes converts it for a c_void_p parameter
    return None if t is None else t.data_ptr()


try:  # the current stream's handle without building a Stream object
    _raw_stream = torch._C._cuda_getCurrentRawStream
except AttributeError:  # pragma: no cover - older or newer torch
    _raw_stream = None


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


try:  # the current device without building a torch.device
    _current_device = torch._C._cuda_getDevice
except AttributeError:  # pragma: no cover - older or newer torch
    _current_device = torch.cuda.current_device


def _check_cuda(name: str, t: torch.Tensor | None, dtype=None, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != _current_device():
        raise ValueError(f"{name} is on {t.device}, not on the current device "
                         f"cuda:{_current_device()} where the kernels run")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _shape(name: str, t: torch.Tensor | None, *shape: int):
    """The kernels trust the sizes they are given: every tensor must have
    exactly the shape the sizes imply (checked before anything is launched)."""
    if t is not None and tuple(t.shape) != shape:
        raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")


def _rows(name: str, t: torch.Tensor | None, *inner: int) -> int | None:
    """Receive tensors: [capacity_rows, *inner]; returns capacity_rows."""
    if t is None:
        return None
    if t.dim() != 1 + len(inner) or tuple(t.shape[1:]) != inner:
        want = ", ".join(["capacity_rows", *map(str, inner)])
        raise ValueError(f"{name} must have shape ({want}), got {tuple(t.shape)}")
    return int(t.shape[0])


def _status(status: torch.Tensor | None):
    if status is not None and status.numel() < 1:
        raise ValueError("status must hold at least one int32")


def _matrix(name: str, t: torch.Tensor) -> tuple[int, int]:
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    return int(t.shape[0]), int(t.shape[1])


def _check_layout_shapes(topk_idx, E, W, ne, nr, off, slot, status):
    T, k = _matrix("topk_idx", topk_idx)
    _shape("num_tokens_per_expert", ne, E)
    _shape("num_tokens_per_rank", nr, W)
    _shape("rank_offset", off, W + 1)
    _shape("slot", slot, T, W)
    _status(status)
    return T, k


def _check_dispatch_shapes(x, topk_idx, topk_w, C, slot, recv_x, recv_topk_idx, recv_topk_w,
                           recv_src, recv_scale, quant, status):
    """Shapes of a dispatch's tensors (C = columns of the slot table); returns
    (T, H, k, capacity_rows)."""
    T, H = _matrix("x", x)
    _, k = _matrix("topk_idx", topk_idx)
    _shape("topk_idx", topk_idx, T, k)
    _shape("topk_w", topk_w, T, k)
    _shape("slot", slot, T, C)
    cap = _rows("recv_x", recv_x, H)
    _rows("recv_topk_idx", recv_topk_idx, k)
    _rows("recv_topk_w", recv_topk_w, k)
    _rows("recv_src", recv_src)
    for n, t in (("recv_topk_idx", recv_topk_idx), ("recv_topk_w", recv_topk_w),
                 ("recv_src", recv_src)):
        if t is not None and t.shape[0] != cap:
            raise ValueError(f"{n} must have capacity_rows = recv_x.shape[0] = {cap} rows, "
                             f"got {t.shape[0]}")
    if quant == EP_QUANT_FP8_E4M3_B128 and recv_scale is not None:
        if H % 128 != 0:
            raise ValueError("FP8 dispatch needs H % 128 == 0")
        _shape("recv_scale", recv_scale, cap, H // 128)
    _status(status)
    return T, H, k, cap


def _raise(fn: str, code: int):
    if code != EP_OK:
        raise EPError(fn, code, ep_status_string(code))


def ep_status_string(code: int) -> str:
    """Name and meaning of an EP_OK / EP_ERR_* code."""
    return load_library().ep_status_string(int(code)).decode()


def ep_layout_workspace_bytes(T: int, W: int, E: int) -> int:
    """Bytes of workspace ep_dispatch_layout needs for these sizes (0: invalid)."""
    return int(load_library().ep_layout_workspace_bytes(T, W, E))


def ep_max_recv_rows(T: int, k: int, W: int) -> int:
    """Worst-case receive rows, T * min(k, W): a capacity that never overflows."""
    return int(load_library().ep_max_recv_rows(T, k, W))


def ep_dispatch_layout(topk_idx: torch.Tensor, E: int, W: int,
                       num_tokens_per_expert: torch.Tensor, num_tokens_per_rank: torch.Tensor,
                       rank_offset: torch.Tensor, slot: torch.Tensor, workspace: torch.Tensor,
                       status: torch.Tensor | None = None, stream=None) -> None:
    """ep_dispatch_layout: per-expert and per-rank counts, rank_offset and the
    slot of every (token, rank) pair for topk_idx [T, k] (int32 CUDA tensors;
    workspace of ep_layout_workspace_bytes(T, W, E) bytes)."""
    T, k = _check_layout_shapes(topk_idx, E, W, num_tokens_per_expert, num_tokens_per_rank,
                                rank_offset, slot, status)
    for n, t in (("topk_idx", topk_idx), ("num_tokens_per_expert", num_tokens_per_expert),
                 ("num_tokens_per_rank", num_tokens_per_rank), ("rank_offset", rank_offset),
                 ("slot", slot)):
        _check_cuda(n, t, torch.int32)
    _check_cuda("workspace", workspace)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_dispatch_layout(
        _ptr(topk_idx), T, k, E, W, _ptr(num_tokens_per_expert), _ptr(num_tokens_per_rank),
        _ptr(rank_offset), _ptr(slot), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _raise("ep_dispatch_layout", rc)


def _check_dispatch_cuda(x, topk_idx, topk_w, slot, recv_x, recv_topk_idx, recv_topk_w, recv_src,
                         recv_scale, quant, status):
    _check_cuda("x", x, torch.bfloat16)
    _check_cuda("topk_idx", topk_idx, torch.int32)
    _check_cuda("topk_w", topk_w, torch.float32)
    _check_cuda("slot", slot, torch.int32)
    _check_cuda("recv_x", recv_x, torch.bfloat16 if quant == EP_QUANT_BF16 else torch.uint8)
    _check_cuda("recv_topk_idx", recv_topk_idx, torch.int32, optional=True)
    _check_cuda("recv_topk_w", recv_topk_w, torch.float32, optional=True)
    _check_cuda("recv_src", recv_src, torch.int32, optional=True)
    _check_cuda("recv_scale", recv_scale, torch.float32, optional=quant == EP_QUANT_BF16)
    _check_cuda("status", status, torch.int32, optional=True)


def ep_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, W: int,
                slot: torch.Tensor, recv_x: torch.Tensor, recv_topk_idx: torch.Tensor | None = None,
                recv_topk_w: torch.Tensor | None = None, recv_src: torch.Tensor | None = None,
                recv_scale: torch.Tensor | None = None, quant: int = EP_QUANT_BF16,
                status: torch.Tensor | None = None, stream=None) -> None:
    """ep_dispatch: rows of x [T, H] bf16 to their receive rows (bf16, or FP8
    codes with recv_scale for EP_QUANT_FP8_E4M3_B128) with the metadata; the
    capacity is recv_x.shape[0]."""
    T, H, k, cap = _check_dispatch_shapes(x, topk_idx, topk_w, W, slot, recv_x, recv_topk_idx,
                                          recv_topk_w, recv_src, recv_scale, quant, status)
    _check_dispatch_cuda(x, topk_idx, topk_w, slot, recv_x, recv_topk_idx, recv_topk_w, recv_src,
                         recv_scale, quant, status)
    rc = load_library().ep_dispatch(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), T, H, k, W, _ptr(slot), cap, quant,
        _ptr(recv_x), _ptr(recv_scale), _ptr(recv_topk_idx), _ptr(recv_topk_w), _ptr(recv_src),
        _ptr(status), _stream(stream))
    _raise("ep_dispatch", rc)


def ep_dispatch_with_layout(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, E: int,
                            W: int, num_tokens_per_expert: torch.Tensor,
                            num_tokens_per_rank: torch.Tensor, rank_offset: torch.Tensor,
                            slot: torch.Tensor, workspace: torch.Tensor, recv_x: torch.Tensor,
                            recv_topk_idx: torch.Tensor | None = None,
                            recv_topk_w: torch.Tensor | None = None,
                            recv_src: torch.Tensor | None = None,
                            recv_scale: torch.Tensor | None = None, quant: int = EP_QUANT_BF16,
                            status: torch.Tensor | None = None, stream=None) -> None:
    """ep_dispatch_layout + ep_dispatch in one call (the dispatch starts
    loading x while the layout runs)."""
    _check_layout_shapes(topk_idx, E, W, num_tokens_per_expert, num_tokens_per_rank, rank_offset,
                         slot, status)
    T, H, k, cap = _check_dispatch_shapes(x, topk_idx, topk_w, W, slot, recv_x, recv_topk_idx,
                                          recv_topk_w, recv_src, recv_scale, quant, status)
    for n, t in (("num_tokens_per_expert", num_tokens_per_expert),
                 ("num_tokens_per_rank", num_tokens_per_rank), ("rank_offset", rank_offset)):
        _check_cuda(n, t, torch.int32)
    _check_cuda("workspace", workspace)
    _check_dispatch_cuda(x, topk_idx, topk_w, slot, recv_x, recv_topk_idx, recv_topk_w, recv_src,
                         recv_scale, quant, status)
    rc = load_library().ep_dispatch_with_layout(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), T, H, k, E, W, _ptr(num_tokens_per_expert),
        _ptr(num_tokens_per_rank), _ptr(rank_offset), _ptr(slot), _ptr(workspace),
        workspace.numel() * workspace.element_size(), cap, quant, _ptr(recv_x),
        _ptr(recv_scale), _ptr(recv_topk_idx), _ptr(recv_topk_w), _ptr(recv_src), _ptr(status),
        _stream(stream))
    _raise("ep_dispatch_with_layout", rc)


def ep_dispatch_experts_with_layout(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                                    E: int, num_tokens_per_expert: torch.Tensor,
                                    expert_offset: torch.Tensor, slot: torch.Tensor,
                                    workspace: torch.Tensor, recv_x: torch.Tensor,
                                    recv_topk_idx: torch.Tensor | None = None,
                                    recv_topk_w: torch.Tensor | None = None,
                                    recv_src: torch.Tensor | None = None,
                                    recv_scale: torch.Tensor | None = None,
                                    quant: int = EP_QUANT_BF16, status: torch.Tensor | None = None,
                                    stream=None) -> None:
    """ep_dispatch_layout_experts + ep_dispatch (W = k) in one call (the
    dispatch starts loading x while the layout runs)."""
    _, k = _matrix("topk_idx", topk_idx)
    T, H, k, cap = _check_dispatch_shapes(x, topk_idx, topk_w, k, slot, recv_x, recv_topk_idx,
                                          recv_topk_w, recv_src, recv_scale, quant, status)
    _shape("num_tokens_per_expert", num_tokens_per_expert, E)
    _shape("expert_offset", expert_offset, E + 1)
    for n, t in (("num_tokens_per_expert", num_tokens_per_expert),
                 ("expert_offset", expert_offset)):
        _check_cuda(n, t, torch.int32)
    _check_cuda("workspace", workspace)
    _check_dispatch_cuda(x, topk_idx, topk_w, slot, recv_x, recv_topk_idx, recv_topk_w, recv_src,
                         recv_scale, quant, status)
    rc = load_library().ep_dispatch_experts_with_layout(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), T, H, k, E, _ptr(num_tokens_per_expert),
        _ptr(expert_offset), _ptr(slot), _ptr(workspace),
        workspace.numel() * workspace.element_size(), cap, quant, _ptr(recv_x),
        _ptr(recv_scale), _ptr(recv_topk_idx), _ptr(recv_topk_w), _ptr(recv_src), _ptr(status),
        _stream(stream))
    _raise("ep_dispatch_experts_with_layout", rc)


def ep_dispatch_with_layout_launches(T: int, H: int, k: int, W: int,
                                     quant: int = EP_QUANT_BF16) -> int:
    """Kernels one ep_dispatch_with_layout call with these sizes launches."""
    return int(load_library().ep_dispatch_with_layout_launches(T, H, k, W, quant))


def _check_combine_shapes(y, slot, out, status):
    T, C = _matrix("slot", slot)
    _, H = _matrix("out", out)
    _shape("out", out, T, H)
    cap = _rows("y", y, H)
    _status(status)
    return T, C, H, cap


def ep_combine(y: torch.Tensor, slot: torch.Tensor, out: torch.Tensor,
               status: torch.Tensor | None = None, stream=None) -> None:
    """ep_combine: out[t] = bf16 of the fp32 sum, in ascending rank order from
    +0, of the rows y[slot[t][r]] (y [capacity_rows, H] bf16)."""
    T, W, H, cap = _check_combine_shapes(y, slot, out, status)
    _check_cuda("y", y, torch.bfloat16)
    _check_cuda("slot", slot, torch.int32)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_combine(_ptr(y), _ptr(slot), T, H, W, cap, _ptr(out), _ptr(status),
                                   _stream(stream))
    _raise("ep_combine", rc)


def ep_dispatch_layout_noalloc(topk_idx: torch.Tensor, E: int, W: int,
                               num_tokens_per_expert: torch.Tensor,
                               num_tokens_per_rank: torch.Tensor, rank_offset: torch.Tensor,
                               slot: torch.Tensor, status: torch.Tensor | None = None,
                               stream=None) -> None:
    """ep_dispatch_layout for callers that cannot allocate device memory: the
    workspace is the library's built-in EP_LAYOUT_NOALLOC_SCRATCH_BYTES array,
    shared by every call (calls that overlap on the GPU race on it)."""
    T, k = _check_layout_shapes(topk_idx, E, W, num_tokens_per_expert, num_tokens_per_rank,
                                rank_offset, slot, status)
    for n, t in (("topk_idx", topk_idx), ("num_tokens_per_expert", num_tokens_per_expert),
                 ("num_tokens_per_rank", num_tokens_per_rank), ("rank_offset", rank_offset),
                 ("slot", slot)):
        _check_cuda(n, t, torch.int32)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_dispatch_layout_noalloc(
        _ptr(topk_idx), T, k, E, W, _ptr(num_tokens_per_expert), _ptr(num_tokens_per_rank),
        _ptr(rank_offset), _ptr(slot), _ptr(status), _stream(stream))
    _raise("ep_dispatch_layout_noalloc", rc)


def ep_dispatch_fused(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, E: int, W: int,
                      num_tokens_per_expert: torch.Tensor, num_tokens_per_rank: torch.Tensor,
                      rank_offset: torch.Tensor, slot: torch.Tensor, recv_x: torch.Tensor,
                      recv_topk_idx: torch.Tensor | None = None,
                      recv_topk_w: torch.Tensor | None = None,
                      recv_src: torch.Tensor | None = None, status: torch.Tensor | None = None,
                      stream=None) -> None:
    """ep_dispatch_layout + bf16 ep_dispatch in one launch (T <= EP_FUSED_MAX_TOKENS)."""
    _check_layout_shapes(topk_idx, E, W, num_tokens_per_expert, num_tokens_per_rank, rank_offset,
                         slot, status)
    T, H, k, cap = _check_dispatch_shapes(x, topk_idx, topk_w, W, slot, recv_x, recv_topk_idx,
                                          recv_topk_w, recv_src, None, EP_QUANT_BF16, status)
    for n, t in (("num_tokens_per_expert", num_tokens_per_expert),
                 ("num_tokens_per_rank", num_tokens_per_rank), ("rank_offset", rank_offset)):
        _check_cuda(n, t, torch.int32)
    _check_dispatch_cuda(x, topk_idx, topk_w, slot, recv_x, recv_topk_idx, recv_topk_w, recv_src,
                         None, EP_QUANT_BF16, status)
    rc = load_library().ep_dispatch_fused(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), T, H, k, E, W, _ptr(num_tokens_per_expert),
        _ptr(num_tokens_per_rank), _ptr(rank_offset), _ptr(slot), cap, _ptr(recv_x),
        _ptr(recv_topk_idx), _ptr(recv_topk_w), _ptr(recv_src), _ptr(status), _stream(stream))
    _raise("ep_dispatch_fused", rc)


def ep_localize_expert_ids(recv_topk_idx: torch.Tensor, rank_offset: torch.Tensor, E: int, W: int,
                           stream=None) -> None:
    """In place: ids of rank r's receive rows become local indices e - r*(E/W), or -1."""
    cap, k = _matrix("recv_topk_idx", recv_topk_idx)
    _shape("rank_offset", rank_offset, W + 1)
    _check_cuda("recv_topk_idx", recv_topk_idx, torch.int32)
    _check_cuda("rank_offset", rank_offset, torch.int32)
    rc = load_library().ep_localize_expert_ids(_ptr(recv_topk_idx), _ptr(rank_offset), cap, k, E, W,
                                               _stream(stream))
    _raise("ep_localize_expert_ids", rc)


def ep_layout_experts_workspace_bytes(T: int, k: int, E: int) -> int:
    """Bytes of workspace ep_dispatch_layout_experts needs for these sizes."""
    return int(load_library().ep_layout_experts_workspace_bytes(T, k, E))


def ep_dispatch_layout_experts(topk_idx: torch.Tensor, E: int, num_tokens_per_expert: torch.Tensor,
                               expert_offset: torch.Tensor, slot: torch.Tensor,
                               workspace: torch.Tensor, status: torch.Tensor | None = None,
                               stream=None) -> None:
    """Expert-major layout: slot [T, k] gives each valid (token, column) pair its
    own row, rows grouped by expert (expert_offset [E + 1])."""
    T, k = _matrix("topk_idx", topk_idx)
    _shape("num_tokens_per_expert", num_tokens_per_expert, E)
    _shape("expert_offset", expert_offset, E + 1)
    _shape("slot", slot, T, k)
    _status(status)
    for n, t in (("topk_idx", topk_idx), ("num_tokens_per_expert", num_tokens_per_expert),
                 ("expert_offset", expert_offset), ("slot", slot)):
        _check_cuda(n, t, torch.int32)
    _check_cuda("workspace", workspace)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_dispatch_layout_experts(
        _ptr(topk_idx), T, k, E, _ptr(num_tokens_per_expert), _ptr(expert_offset), _ptr(slot),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _raise("ep_dispatch_layout_experts", rc)


def ep_combine_weighted(y: torch.Tensor, slot: torch.Tensor, w: torch.Tensor, out: torch.Tensor,
                        status: torch.Tensor | None = None, stream=None) -> None:
    """out[t] = bf16 of the fp32 FMA chain over the columns c of slot[t] >= 0,
    in ascending order, of w[t][c] * y[slot[t][c]]."""
    T, C, H, cap = _check_combine_shapes(y, slot, out, status)
    _shape("w", w, T, C)
    _check_cuda("y", y, torch.bfloat16)
    _check_cuda("slot", slot, torch.int32)
    _check_cuda("w", w, torch.float32)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_combine_weighted(_ptr(y), _ptr(slot), _ptr(w), T, H, C, cap,
                                            _ptr(out), _ptr(status), _stream(stream))
    _raise("ep_combine_weighted", rc)


def ep_selftest_wait_timeout(status: torch.Tensor, stream=None) -> None:
    """Diagnostic: a kernel whose bounded wait must run out (about one second)
    and set EP_STATUS_TIMEOUT in ``status``."""
    _status(status)
    _check_cuda("status", status, torch.int32)
    rc = load_library().ep_selftest_wait_timeout(_ptr(status), _stream(stream))
    _raise("ep_selftest_wait_timeout", rc)


def ep_cast_transpose_t_bytes(capacity_rows: int, E: int, H: int) -> int:
    """Bytes of the transposed FP8 output of ep_cast_transpose_experts."""
    return int(load_library().ep_cast_transpose_t_bytes(capacity_rows, E, H))


def ep_cast_transpose_experts(y: torch.Tensor, expert_offset: torch.Tensor, scale: torch.Tensor,
                              out_c: torch.Tensor, out_t: torch.Tensor, amax: torch.Tensor,
                              status: torch.Tensor | None = None, stream=None) -> None:
    """FP8 cast (out_c) and per-expert transposed cast (out_t) of the
    expert-major rows y, amax[e] = max(amax[e], max |x|)."""
    cap, H = _matrix("y", y)
    if expert_offset.dim() != 1 or expert_offset.numel() < 2:
        raise ValueError("expert_offset must be [E + 1] with E >= 1")
    E = expert_offset.numel() - 1
    _shape("scale", scale, E)
    _shape("amax", amax, E)
    _shape("out_c", out_c, cap, H)
    _status(status)
    _check_cuda("y", y, torch.bfloat16)
    _check_cuda("expert_offset", expert_offset, torch.int32)
    _check_cuda("scale", scale, torch.float32)
    _check_cuda("out_c", out_c, torch.uint8)
    _check_cuda("out_t", out_t, torch.uint8)
    _check_cuda("amax", amax, torch.float32)
    _check_cuda("status", status, torch.int32, optional=True)
    if out_t.numel() < ep_cast_transpose_t_bytes(cap, E, H):
        raise ValueError("out_t is smaller than ep_cast_transpose_t_bytes(capacity_rows, E, H)")
    rc = load_library().ep_cast_transpose_experts(_ptr(y), _ptr(expert_offset), E, H, _ptr(scale),
                                                  cap, _ptr(out_c), _ptr(out_t), _ptr(amax),
                                                  _ptr(status), _stream(stream))
    _raise("ep_cast_transpose_experts", rc)


def _region_table(regions: list[dict], H: int, k: int, quant: int):
    """The C table of per-rank receive regions, after checking every tensor."""
    W = len(regions)
    if W < 1 or W > 32:
        raise ValueError("regions must name 1 to 32 ranks")
    fp8 = quant == EP_QUANT_FP8_E4M3_B128
    table = (RankRegion * W)()
    for r, g in enumerate(regions):
        rx = g["recv_x"]
        rows = _rows(f"regions[{r}].recv_x", rx, H)
        _rows(f"regions[{r}].recv_topk_idx", g.get("recv_topk_idx"), k)
        _rows(f"regions[{r}].recv_topk_w", g.get("recv_topk_w"), k)
        _rows(f"regions[{r}].recv_src", g.get("recv_src"))
        for n in ("recv_topk_idx", "recv_topk_w", "recv_src"):
            t = g.get(n)
            if t is not None and t.shape[0] != rows:
                raise ValueError(f"regions[{r}].{n} must have {rows} rows, got {t.shape[0]}")
        if fp8:
            _shape(f"regions[{r}].recv_scale", g.get("recv_scale"), rows, H // 128)
        _check_cuda(f"regions[{r}].recv_x", rx, torch.uint8 if fp8 else torch.bfloat16)
        _check_cuda(f"regions[{r}].recv_scale", g.get("recv_scale"), torch.float32,
                    optional=not fp8)
        _check_cuda(f"regions[{r}].recv_topk_idx", g.get("recv_topk_idx"), torch.int32,
                    optional=True)
        _check_cuda(f"regions[{r}].recv_topk_w", g.get("recv_topk_w"), torch.float32, optional=True)
        _check_cuda(f"regions[{r}].recv_src", g.get("recv_src"), torch.int32, optional=True)
        table[r] = RankRegion(_ptr(rx), _ptr(g.get("recv_scale") if fp8 else None),
                              _ptr(g.get("recv_topk_idx")), _ptr(g.get("recv_topk_w")),
                              _ptr(g.get("recv_src")), rows)
    return table


def ep_dispatch_regions(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                        slot: torch.Tensor, rank_offset: torch.Tensor, regions: list[dict],
                        quant: int = EP_QUANT_BF16, status: torch.Tensor | None = None,
                        stream=None) -> None:
    """ep_dispatch into per-rank regions: ``regions[r]`` is a dict with rank r's
    receive tensors ``recv_x`` [rows_r, H] (bf16, or uint8 codes for FP8),
    ``recv_scale`` [rows_r, H / 128] (FP8), and optionally ``recv_topk_idx``
    [rows_r, k], ``recv_topk_w`` [rows_r, k], ``recv_src`` [rows_r]; token t's
    row for rank r lands in row slot[t][r] - rank_offset[r] of region r."""
    W = len(regions)
    if W < 1 or W > 32:
        raise ValueError("regions must name 1 to 32 ranks")
    T, H = _matrix("x", x)
    _, k = _matrix("topk_idx", topk_idx)
    _shape("topk_idx", topk_idx, T, k)
    _shape("topk_w", topk_w, T, k)
    _shape("slot", slot, T, W)
    _shape("rank_offset", rank_offset, W + 1)
    _status(status)
    table = _region_table(regions, H, k, quant)
    _check_cuda("x", x, torch.bfloat16)
    _check_cuda("topk_idx", topk_idx, torch.int32)
    _check_cuda("topk_w", topk_w, torch.float32)
    _check_cuda("slot", slot, torch.int32)
    _check_cuda("rank_offset", rank_offset, torch.int32)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_dispatch_regions(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), T, H, k, W, _ptr(slot), _ptr(rank_offset), table,
        quant, _ptr(status), _stream(stream))
    _raise("ep_dispatch_regions", rc)


def ep_dispatch_regions_with_layout(x: torch.Tensor, topk_idx: torch.Tensor,
                                    topk_w: torch.Tensor, E: int,
                                    num_tokens_per_expert: torch.Tensor,
                                    num_tokens_per_rank: torch.Tensor, rank_offset: torch.Tensor,
                                    slot: torch.Tensor, workspace: torch.Tensor,
                                    regions: list[dict], quant: int = EP_QUANT_BF16,
                                    status: torch.Tensor | None = None, stream=None) -> None:
    """ep_dispatch_layout + ep_dispatch_regions in one call (W = len(regions)):
    every layout output is written, region r gets rank r's rows."""
    W = len(regions)
    if W < 1 or W > 32:
        raise ValueError("regions must name 1 to 32 ranks")
    _check_layout_shapes(topk_idx, E, W, num_tokens_per_expert, num_tokens_per_rank, rank_offset,
                         slot, status)
    T, H = _matrix("x", x)
    _, k = _matrix("topk_idx", topk_idx)
    _shape("topk_idx", topk_idx, T, k)
    _shape("topk_w", topk_w, T, k)
    table = _region_table(regions, H, k, quant)
    for n, t in (("num_tokens_per_expert", num_tokens_per_expert),
                 ("num_tokens_per_rank", num_tokens_per_rank), ("rank_offset", rank_offset),
                 ("slot", slot)):
        _check_cuda(n, t, torch.int32)
    _check_cuda("workspace", workspace)
    _check_cuda("x", x, torch.bfloat16)
    _check_cuda("topk_idx", topk_idx, torch.int32)
    _check_cuda("topk_w", topk_w, torch.float32)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_dispatch_regions_with_layout(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), T, H, k, E, W, _ptr(num_tokens_per_expert),
        _ptr(num_tokens_per_rank), _ptr(rank_offset), _ptr(slot), _ptr(workspace),
        workspace.numel() * workspace.element_size(), table, quant, _ptr(status), _stream(stream))
    _raise("ep_dispatch_regions_with_layout", rc)


def ep_combine_regions(y_regions: list[torch.Tensor], slot: torch.Tensor, rank_offset: torch.Tensor,
                       out: torch.Tensor, status: torch.Tensor | None = None, stream=None) -> None:
    """ep_combine with rank r's expert outputs in ``y_regions[r]`` [rows_r, H]
    (bf16): row slot[t][r] - rank_offset[r] of it belongs to token t."""
    W = len(y_regions)
    if W < 1 or W > 32:
        raise ValueError("y_regions must name 1 to 32 ranks")
    T, H = _matrix("out", out)
    _shape("slot", slot, T, W)
    _shape("rank_offset", rank_offset, W + 1)
    _status(status)
    ptrs = (ctypes.c_void_p * W)()
    rows = (ctypes.c_int64 * W)()
    for r, y in enumerate(y_regions):
        rows[r] = _rows(f"y_regions[{r}]", y, H)
        _check_cuda(f"y_regions[{r}]", y, torch.bfloat16)
        ptrs[r] = _ptr(y)
    _check_cuda("slot", slot, torch.int32)
    _check_cuda("rank_offset", rank_offset, torch.int32)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("status", status, torch.int32, optional=True)
    rc = load_library().ep_combine_regions(ptrs, rows, _ptr(slot), _ptr(rank_offset), T, H, W,
                                           _ptr(out), _ptr(status), _stream(stream))
    _raise("ep_combine_regions", rc)
