"""Preallocated buffers for one dispatch/combine shape, and the three calls on them.

PyTorch allocates the device memory once; every step then only enqueues the
library's kernels (layout -> dispatch -> [experts] -> combine) on one stream.
"""
from __future__ import annotations

import torch

from . import _lib


class DispatchCombine:
    """Buffers for T tokens of hidden size H routed top-k over E experts on W ranks.

    ``order`` picks the receive layout:
      - "rank" (default): one row per (token, destination rank), the token's
        experts on a rank share it; combine sums a token's rows unweighted (or
        with per-(token, rank) weights given to ``combine``);
      - "expert": one row per valid (token, expert) pair, rows grouped by
        expert (``expert_offset``), for a grouped expert GEMM; combine takes
        the gate weights ``topk_w`` and forms their FMA-weighted sum.
    ``capacity_rows`` defaults to the worst case (T * min(k, W), or T * k for
    "expert"), so dispatch can never overflow.  ``quant`` selects the dispatch
    payload (bf16 or FP8 e4m3 with 1x128 block scales); combine always reads
    bf16 expert outputs.
    """

    def __init__(self, T: int, H: int, E: int, k: int, W: int, capacity_rows: int | None = None,
                 quant: int = _lib.EP_QUANT_BF16, device: str | torch.device = "cuda",
                 order: str = "rank"):
        if order not in ("rank", "expert"):
            raise ValueError(f"order must be 'rank' or 'expert', got {order!r}")
        self.T, self.H, self.E, self.k, self.W, self.quant = T, H, E, k, W, quant
        self.order = order
        dev = torch.device(device)
        worst = T * k if order == "expert" else _lib.ep_max_recv_rows(T, k, W)
        cap = worst if capacity_rows is None else capacity_rows
        self.capacity_rows = cap
        i32 = dict(dtype=torch.int32, device=dev)
        self.num_tokens_per_expert = torch.empty(E, **i32)
        if order == "rank":
            self.num_tokens_per_rank = torch.empty(W, **i32)
            self.rank_offset = torch.empty(W + 1, **i32)
            self.expert_offset = None
            self.slot = torch.empty(T, W, **i32)
            ws = _lib.ep_layout_workspace_bytes(T, W, E)
        else:
            self.num_tokens_per_rank = None
            self.rank_offset = None
            self.expert_offset = torch.empty(E + 1, **i32)
            self.slot = torch.empty(T, k, **i32)
            ws = _lib.ep_layout_experts_workspace_bytes(T, k, E)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        if quant == _lib.EP_QUANT_BF16:
            self.recv_x = torch.empty(cap, H, dtype=torch.bfloat16, device=dev)
            self.recv_scale = None
        else:
            self.recv_x = torch.empty(cap, H, dtype=torch.uint8, device=dev)
            self.recv_scale = torch.empty(cap, H // 128, dtype=torch.float32, device=dev)
        self.recv_topk_idx = torch.empty(cap, k, **i32)
        self.recv_topk_w = torch.empty(cap, k, dtype=torch.float32, device=dev)
        self.recv_src = torch.empty(cap, **i32)
        self.out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, **i32)

    def layout(self, topk_idx: torch.Tensor, stream=None) -> None:
        """The layout of topk_idx [T, k] into this object's counts, offsets and slot."""
        if self.order == "rank":
            _lib.ep_dispatch_layout(topk_idx, self.E, self.W, self.num_tokens_per_expert,
                                    self.num_tokens_per_rank, self.rank_offset, self.slot,
                                    self.workspace, self.status, stream)
        else:
            _lib.ep_dispatch_layout_experts(topk_idx, self.E, self.num_tokens_per_expert,
                                            self.expert_offset, self.slot, self.workspace,
                                            self.status, stream)

    def dispatch(self, x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                 stream=None) -> None:
        """Rows of x [T, H] bf16 into recv_x (and recv_scale for FP8) with the
        metadata, by the slots of the last layout."""
        _lib.ep_dispatch(x, topk_idx, topk_w, self.slot.shape[1], self.slot, self.recv_x,
                         self.recv_topk_idx, self.recv_topk_w, self.recv_src, self.recv_scale,
                         self.quant, self.status, stream)

    def layout_dispatch(self, x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                        stream=None) -> None:
        """layout() then dispatch() in one library call: the same results, with
        the dispatch loading x while the layout kernels run."""
        if self.order == "expert":
            _lib.ep_dispatch_experts_with_layout(
                x, topk_idx, topk_w, self.E, self.num_tokens_per_expert, self.expert_offset,
                self.slot, self.workspace, self.recv_x, self.recv_topk_idx, self.recv_topk_w,
                self.recv_src, self.recv_scale, self.quant, self.status, stream)
            return
        _lib.ep_dispatch_with_layout(x, topk_idx, topk_w, self.E, self.W,
                                     self.num_tokens_per_expert, self.num_tokens_per_rank,
                                     self.rank_offset, self.slot, self.workspace, self.recv_x,
                                     self.recv_topk_idx, self.recv_topk_w, self.recv_src,
                                     self.recv_scale, self.quant, self.status, stream)

    def dispatch_fused(self, x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                       stream=None) -> None:
        """layout() and dispatch() in one launch (rank order, bf16, T <= EP_FUSED_MAX_TOKENS)."""
        if self.order != "rank":
            raise ValueError("dispatch_fused builds the rank-major layout")
        _lib.ep_dispatch_fused(x, topk_idx, topk_w, self.E, self.W, self.num_tokens_per_expert,
                               self.num_tokens_per_rank, self.rank_offset, self.slot, self.recv_x,
                               self.recv_topk_idx, self.recv_topk_w, self.recv_src, self.status,
                               stream)

    def combine(self, y: torch.Tensor | None = None, w: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
        """Bring each token's expert outputs ``y`` (default: the dispatched rows,
        i.e. identity experts; bf16 dispatch only) back into ``self.out``.
        ``w`` has the slot table's shape: per-(token, rank) weights for "rank"
        (optional: without it the sum is unweighted), the gate weights topk_w
        for "expert" (required)."""
        if y is None:
            if self.quant != _lib.EP_QUANT_BF16:
                raise ValueError("identity experts need a bf16 dispatch")
            y = self.recv_x
        if w is None and self.order == "expert":
            raise ValueError("the expert-major combine needs the gate weights")
        if w is None:
            _lib.ep_combine(y, self.slot, self.out, self.status, stream)
        else:
            _lib.ep_combine_weighted(y, self.slot, w, self.out, self.status, stream)
        return self.out

    def cast_transpose(self, scale: torch.Tensor, amax: torch.Tensor | None = None,
                       stream=None):
        """Expert-major order, bf16 dispatch: the FP8 cast of the received rows
        (``recv_fp8`` [capacity_rows, H]) and their per-expert transposed cast
        (``recv_fp8_t``, one [H][n_e rounded up to 16] block per expert) with
        per-expert scales ``scale`` [E]; ``amax`` [E] (default: zeroed buffer
        ``self.amax``) gets max(amax, max |x|).  Returns (recv_fp8, recv_fp8_t, amax)."""
        if self.order != "expert" or self.quant != _lib.EP_QUANT_BF16:
            raise ValueError("cast_transpose takes the bf16 rows of the expert-major layout")
        if not hasattr(self, "recv_fp8"):
            dev = self.recv_x.device
            self.recv_fp8 = torch.empty(self.capacity_rows, self.H, dtype=torch.uint8, device=dev)
            self.recv_fp8_t = torch.empty(
                max(_lib.ep_cast_transpose_t_bytes(self.capacity_rows, self.E, self.H), 16),
                dtype=torch.uint8, device=dev)
            self.amax = torch.zeros(self.E, dtype=torch.float32, device=dev)
        if amax is None:
            amax = self.amax
            amax.zero_()
        _lib.ep_cast_transpose_experts(self.recv_x, self.expert_offset, scale, self.recv_fp8,
                                       self.recv_fp8_t, amax, self.status, stream)
        return self.recv_fp8, self.recv_fp8_t, amax

    def step(self, x, topk_idx, topk_w, y=None, stream=None) -> torch.Tensor:
        """layout_dispatch() then combine(y) (y defaults to the dispatched rows,
        i.e. identity experts); returns self.out."""
        self.layout_dispatch(x, topk_idx, topk_w, stream)
        return self.combine(y, topk_w if self.order == "expert" else None, stream)
