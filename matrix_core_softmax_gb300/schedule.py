"""Per-step attention precision schedules of a diffusion sampler.

"Fused-Softmax shifts an AI attention bottleneck onto faster GPU hardware",
paragraphs 9-10: the video model runs 20 denoising steps, and the hybrid
schedule uses MXFP6 attention for the first and last three steps and MXFP4
for the fourteen between them.  This module is orchestration only: every
step is one call of the library, the fused MX attention for an MX format or
the BF16 flash-attention kernel for "bf16".
"""
from __future__ import annotations

from . import FORMATS, attention_fwd, bf16_attention_fwd

DENOISING_STEPS = 20
EDGE_STEPS = 3
STEP_FORMATS = tuple(FORMATS) + ("bf16",)


def _check_fmt(fmt: str):
    if fmt not in STEP_FORMATS:
        raise ValueError(f"unknown step format {fmt!r}; expected one of {STEP_FORMATS}")


def hybrid_schedule(n_steps: int = DENOISING_STEPS, n_edge: int = EDGE_STEPS,
                    edge_fmt: str = "mxfp6", mid_fmt: str = "mxfp4") -> list[str]:
    """The format of every denoising step: edge_fmt for the first and last
    n_edge steps, mid_fmt for the steps between (the pages' schedule with the
    defaults: 3 + 3 steps MXFP6, 14 steps MXFP4)."""
    if n_steps < 0 or n_edge < 0:
        raise ValueError("n_steps and n_edge must be non-negative")
    _check_fmt(edge_fmt)
    _check_fmt(mid_fmt)
    return [edge_fmt if (i < n_edge or i >= n_steps - n_edge) else mid_fmt for i in range(n_steps)]


def uniform_schedule(fmt: str, n_steps: int = DENOISING_STEPS) -> list[str]:
    """Every step in one format (the all-MXFP4 and all-BF16 references)."""
    if n_steps < 0:
        raise ValueError("n_steps must be non-negative")
    _check_fmt(fmt)
    return [fmt] * n_steps


def attention_step(q, k, v, fmt: str, threshold: float = 8.0, *, out=None, workspace=None,
                   stream=None):
    """One step's self-attention in the step's format: q, k, v contiguous CUDA
    bf16 [B, H, S, D]; returns the bf16 output (written into `out` if given)."""
    _check_fmt(fmt)
    if fmt == "bf16":
        return bf16_attention_fwd(q, k, v, out=out, stream=stream)
    return attention_fwd(q, k, v, fmt, threshold, out=out, workspace=workspace, stream=stream)
