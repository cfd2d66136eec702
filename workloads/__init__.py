"""Seeded synthetic inputs for the MoE expert FFN forward.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.
It only draws random numbers and arranges them into tensors of the right
shape; it performs none of the method's arithmetic (no normalisation, no
softmax, no top-k, no GEMM).  Everything is drawn with a seeded
``torch.Generator`` on the requested device, in a fixed order
(x, norm_w, router_w, router_bias, w13, w2, router_logits), so the same
(config, device, torch version) always yields the same tensors.

Shapes and distributions follow the five workloads the MoE FFN is measured
on (tiny; decode balanced; decode skewed; decode FP8 W8A8; prefill).  The
pages measure on end-to-end serving suites and on model shapes they do not
spell out; these synthetic tensors stand in for them.

Tensor layouts (row-major, last index contiguous):
  x            bf16 [T, H]
  norm_w       bf16 [H]
  router_w     fp32 [H, E]            (None when routing is forced)
  router_bias  fp32 [E]               (None unless the workload is skewed)
  router_logits fp32 [T, E]           (forced routing only, else None)
  w13          bf16 [E, 2I, H]        rows 0..I-1 gate, rows I..2I-1 up
  w2           bf16 [E, H, I]
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

# Large negative logit used to switch an expert off in forced routing.
# exp(FORCED_OFF_LOGIT - max) is exactly 0 in fp32 and fp64, so a softmax over
# all E experts equals the softmax over the k forced ones.
FORCED_OFF_LOGIT = -1.0e4


@dataclasses.dataclass(frozen=True)
class Shape:
    T: int
    H: int
    E: int
    k: int
    I: int


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    shape: Shape
    routing: str          # "learned" | "balanced" | "zipf"
    fp8: bool | str       # False, True (per-channel E4M3) or "block" (128 x 128 tiles)
    seed: int
    eps: float = 1e-6
    description: str = ""
    nvfp4: bool = False   # NVFP4 expert weights (quantised from the drawn bf16 weights)


CONFIGS = {
    "c1_tiny": Config(
        "c1_tiny", Shape(T=4, H=256, E=8, k=2, I=512), "learned", False, 0,
        description="tiny MoE FFN: learned router, softmax then top-2 renorm"),
    "c2_decode_balanced": Config(
        "c2_decode_balanced", Shape(T=16, H=4096, E=64, k=8, I=1536), "balanced", False, 1,
        description="decode, forced balanced routing (token t -> experts (8t+j) mod 64)"),
    "c3_decode_skewed": Config(
        "c3_decode_skewed", Shape(T=64, H=7168, E=256, k=8, I=2048), "zipf", False, 2,
        description="decode, learned router plus Zipf(1.2) per-expert bias scaled to std 2"),
    "c4_decode_fp8": Config(
        "c4_decode_fp8", Shape(T=16, H=4096, E=64, k=8, I=1536), "balanced", True, 3,
        description="decode FP8 W8A8 (E4M3, per-channel weight / per-token activation scales)"),
    "c5_prefill": Config(
        "c5_prefill", Shape(T=4096, H=4096, E=64, k=8, I=1536), "learned", False, 4,
        description="prefill, learned router with natural imbalance"),
    "c6_decode_nvfp4": Config(
        "c6_decode_nvfp4", Shape(T=16, H=4096, E=64, k=8, I=1536), "balanced", False, 5,
        description="decode with NVFP4 expert weights (E2M1 codes, E4M3 block scales of 16, "
                    "fp32 matrix scales) and bf16 activations", nvfp4=True),
    "c7_decode_fp8_block": Config(
        "c7_decode_fp8_block", Shape(T=16, H=4096, E=64, k=8, I=1536), "balanced", "block", 6,
        description="decode with block-wise FP8 (E4M3, one scale per 128 x 128 weight tile and "
                    "per 1 x 128 activation group)"),
    "c8_prefill_fp8": Config(
        "c8_prefill_fp8", Shape(T=4096, H=4096, E=64, k=8, I=1536), "learned", True, 7,
        description="prefill with FP8 W8A8 (E4M3, per-channel weight / per-token activation "
                    "scales)"),
    "c9_prefill_fp8_block": Config(
        "c9_prefill_fp8_block", Shape(T=4096, H=4096, E=64, k=8, I=1536), "learned", "block", 8,
        description="prefill with block-wise FP8 (E4M3, 128 x 128 weight tiles, 1 x 128 "
                    "activation groups)"),
}

CONFIG_ORDER = ["c1_tiny", "c2_decode_balanced", "c3_decode_skewed", "c4_decode_fp8", "c5_prefill"]


def _randn(shape, g, device, std=1.0, mean=0.0, dtype=torch.bfloat16):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def make_inputs(cfg: Config | str, device="cpu", shape: Optional[Shape] = None,
                routing: Optional[str] = None, seed: Optional[int] = None) -> dict:
    """Draw one workload's tensors on ``device``.

    ``shape``/``routing``/``seed`` override the named config (used by the
    parity tests for small ragged shapes with the same recipe)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    s = shape or cfg.shape
    routing = routing or cfg.routing
    seed = cfg.seed if seed is None else seed
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    T, H, E, k, I = s.T, s.H, s.E, s.k, s.I

    x = _randn((T, H), g, device)
    norm_w = _randn((H,), g, device, std=0.1, mean=1.0)
    router_w = None
    router_bias = None
    router_logits = None
    if routing in ("learned", "zipf"):
        router_w = _randn((H, E), g, device, std=0.02, dtype=torch.float32)
    if routing == "zipf":
        # Per-expert popularity 1/rank^1.2 with a seeded random rank order,
        # standardised and scaled to std 2.
        ranks = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
        b = ranks.pow(-1.2)
        b = 2.0 * (b - b.mean()) / b.std()
        router_bias = b.to(torch.float32)
    # Expert weights, drawn expert by expert to bound the fp32 scratch.
    w13 = torch.empty((E, 2 * I, H), device=device, dtype=torch.bfloat16)
    w2 = torch.empty((E, H, I), device=device, dtype=torch.bfloat16)
    for e in range(E):
        w13[e] = _randn((2 * I, H), g, device, std=0.02)
    for e in range(E):
        w2[e] = _randn((H, I), g, device, std=0.02)
    if routing == "balanced":
        # token t uses experts (k*t + j) mod E, j = 0..k-1, with N(0,1) logits;
        # every other expert is switched off with FORCED_OFF_LOGIT.
        vals = torch.randn((T, k), generator=g, device=device, dtype=torch.float32)
        router_logits = torch.full((T, E), FORCED_OFF_LOGIT, device=device, dtype=torch.float32)
        t_idx = torch.arange(T, device=device).unsqueeze(1)
        j_idx = torch.arange(k, device=device).unsqueeze(0)
        ids = (k * t_idx + j_idx) % E
        router_logits.scatter_(1, ids, vals)
    return dict(
        name=cfg.name, T=T, H=H, E=E, k=k, I=I, eps=cfg.eps, fp8=cfg.fp8, nvfp4=cfg.nvfp4,
        routing=routing,
        seed=seed, x=x, norm_w=norm_w, router_w=router_w, router_bias=router_bias,
        router_logits=router_logits, w13=w13, w2=w2,
    )


def weight_bytes_per_expert(H: int, I: int, fp8: bool = False) -> int:
    """Bytes of one expert's FC1 (gate+up) and FC2 weights, plus FP8 scales."""
    elem = 1 if fp8 else 2
    b = 3 * H * I * elem
    if fp8:
        b += (2 * I + H) * 4
    return b
