"""Seeded synthetic inputs for MoE expert-parallel dispatch / combine.

This module only draws random inputs; it holds none of the dispatch or combine
arithmetic, so that the CPU oracle and the CUDA library can both be fed from it
without sharing any of the method's code.

Workload shapes follow the pages' workloads: DeepSeek-V3 (hidden 7168, top-8 of
256 experts; "perf(ep): optimize IntraNode dispatch kernel for MI350X",
Motivation) and a Qwen-MoE shape with 128 experts ("Optimized rocm specific
multicast transpose kernel", Benchmark Results).

Recipe (all draws from ``numpy.random.default_rng(seed)``, in this order):
  1. x: fp32 N(0,1) of shape [T, H], rounded to bf16 by round-to-nearest-even
     (PyTorch's CPU cast); returned as the raw uint16 bit patterns.
  2. routing keys: ``uniform`` = iid U(0,1) per (token, expert); the k experts
     with the smallest keys, in ascending-key order, i.e. the first k entries of
     a uniformly random permutation.  ``zipf`` = Gumbel-top-k over the logits
     log p_e with p_e proportional to (e+1)^-s (expert 0 most popular); the k
     largest perturbed keys in descending order, which is the same law as
     drawing k distinct experts one after another with probability
     proportional to p among those not yet drawn.
  3. gate logits: fp32 N(0,1) of shape [T, k]; weights are their softmax in
     fp32.  Dispatch carries them verbatim, so their exact values never enter
     a comparison.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = ["EPConfig", "CONFIGS", "make_inputs", "make_routing", "make_bf16",
           "bf16_bits_from_f32", "f32_from_bf16_bits"]


@dataclasses.dataclass(frozen=True)
class EPConfig:
    name: str
    T: int          # tokens
    H: int          # hidden size
    E: int          # experts
    W: int          # logical expert-parallel ranks
    k: int          # experts per token
    routing: str    # "uniform" | "zipf"
    quant: str      # "bf16" | "fp8"   (dispatch payload; combine is always bf16)
    zipf_s: float = 1.2

    @property
    def Er(self) -> int:
        return self.E // self.W


CONFIGS = {
    c.name: c
    for c in [
        EPConfig("tiny", T=128, H=256, E=16, W=4, k=4, routing="uniform", quant="bf16"),
        EPConfig("dsv3", T=4096, H=7168, E=256, W=8, k=8, routing="uniform", quant="bf16"),
        EPConfig("dsv3_zipf_fp8", T=4096, H=7168, E=256, W=8, k=8, routing="zipf",
                 quant="fp8", zipf_s=1.2),
        EPConfig("qwen", T=8192, H=4096, E=128, W=8, k=8, routing="uniform", quant="bf16"),
        EPConfig("decode", T=256, H=7168, E=256, W=8, k=8, routing="uniform", quant="bf16"),
    ]
}


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16) by PyTorch's round-to-nearest-even cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of scale * N(0,1) fp32 draws."""
    a = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        a = a * np.float32(scale)
    return bf16_bits_from_f32(a)


def make_routing(rng: np.random.Generator, T: int, E: int, k: int,
                 routing: str = "uniform", zipf_s: float = 1.2) -> np.ndarray:
    """[T, k] int32 expert ids, k distinct per token (step 2 of the recipe)."""
    if not 1 <= k <= E:
        raise ValueError(f"need 1 <= k <= E, got k={k} E={E}")
    if routing == "uniform":
        keys = rng.random((T, E))
        idx = np.argsort(keys, axis=1, kind="stable")[:, :k]
    elif routing == "zipf":
        logp = -zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        u = rng.random((T, E))
        gumbel = -np.log(-np.log(np.clip(u, 1e-300, None)))
        keys = logp[None, :] + gumbel
        idx = np.argsort(-keys, axis=1, kind="stable")[:, :k]
    else:
        raise ValueError(f"unknown routing {routing!r}")
    return np.ascontiguousarray(idx, dtype=np.int32)


def make_inputs(cfg: EPConfig | str, seed: int = 0, T: int | None = None) -> dict:
    """Seeded inputs of one workload.  ``T`` overrides the token count (same recipe).

    Returns a dict with ``x`` (uint16 bf16 bits [T,H]), ``topk_idx`` (int32 [T,k]),
    ``topk_w`` (float32 [T,k]) and ``cfg``.
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    if T is not None:
        cfg = dataclasses.replace(cfg, T=T)
    rng = np.random.default_rng(seed)
    x = make_bf16(rng, (cfg.T, cfg.H))
    topk_idx = make_routing(rng, cfg.T, cfg.E, cfg.k, cfg.routing, cfg.zipf_s)
    logits = rng.standard_normal((cfg.T, cfg.k), dtype=np.float32)
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    topk_w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return {"x": x, "topk_idx": topk_idx, "topk_w": np.ascontiguousarray(topk_w), "cfg": cfg}
