"""Consumers of the quantizer's outputs: torch FP4 / FP8 views in the layout
block-scaled tensor cores read, and the matrix multiply on them.

"fp4-train" (API: to_fp4_operands, fp4_mm) hands quantized operands to the
native NVFP4 tensor-core matmul; here the codes are viewed as
torch.float4_e2m1fn_x2 (two codes per byte, element 2j in the low nibble, as
the quantizer packs them) and the scales are re-laid out by the library's
nvfp4_scales_to_mma kernel and viewed as torch.float8_e4m3fn.  fp4_mm calls
torch's scaled matrix multiply (a library GEMM, like cuBLAS) and multiplies by
the two per-tensor decode scales.  Not part of the quantization path.
"""
from __future__ import annotations

import torch

from . import nvfp4_global_scales, nvfp4_scales_to_mma


def to_fp4_operands(q: dict) -> dict:
    """{"codes", "scales"} of a rowwise quantize call (device tensors) ->
    {"fp4": codes as float4_e2m1fn_x2 [M, K/2], "scales": float8_e4m3fn in the
    matrix-multiply layout, "scale_dec": the per-tensor decode scale or 1}."""
    codes, scales = q["codes"], q["scales"]
    out = {"fp4": codes.view(torch.float4_e2m1fn_x2),
           "scales": nvfp4_scales_to_mma(scales).view(torch.float8_e4m3fn)}
    g = q.get("gamax")
    out["scale_dec"] = None if g is None else g
    return out


def _scale_dec(g, bound: float) -> torch.Tensor | float:
    """The per-tensor decode scale the library derives from a global amax."""
    if g is None:
        return 1.0
    return nvfp4_global_scales(g.float().reshape(-1)[:1].contiguous(), bound)[1]


def fp4_mm(a: dict, b: dict, *, out_dtype=torch.bfloat16, scale_bound: float = 448.0) -> torch.Tensor:
    """a @ b^T for rowwise-quantized a [M, K] and b [N, K] (each the dict of
    to_fp4_operands): the block-scaled product times both decode scales."""
    y = torch._scaled_mm(a["fp4"], b["fp4"].t(), a["scales"], b["scales"], out_dtype=torch.float32)
    s = _scale_dec(a.get("scale_dec"), scale_bound) * _scale_dec(b.get("scale_dec"), scale_bound)
    return (y * s).to(out_dtype)
