"""Consumers of the quantizer's outputs: torch FP4 / FP8 views in the layout
block-scaled tensor cores read, the matrix multiply on them, and fp4_linear.

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

from . import (nvfp4_dequantize, nvfp4_global_scales, nvfp4_mm, nvfp4_quantize,
               nvfp4_scales_to_mma)


def to_fp4_operands(q, stochastic: bool = False, seed: int = 0, step: int = 0) -> dict:
    """{"codes", "scales"} of a rowwise quantize call (device tensors), or a
    CUDA tensor [M, K] to quantize first with the page's recipe (1x16 blocks,
    no global scale; nearest, or stochastic rounding keyed on (seed, step)) ->
    {"fp4": codes as float4_e2m1fn_x2 [M, K/2], "scales": float8_e4m3fn in the
    matrix-multiply layout, "gamax": the per-tensor amax the codes were made
    with, or None without a global scale}; fp4_mm derives the decode scale
    from it with the library's nvfp4_global_scales."""
    if torch.is_tensor(q):
        q = nvfp4_quantize(q.contiguous(), rounding="sr" if stochastic else "rtn", seed=seed, step=step)
    codes, scales = q["codes"], q["scales"]
    out = {"fp4": codes.view(torch.float4_e2m1fn_x2),
           "scales": nvfp4_scales_to_mma(scales).view(torch.float8_e4m3fn)}
    out["gamax"] = q.get("gamax")
    return out


def _scale_dec(g, bound: float) -> torch.Tensor | float:
    """The per-tensor decode scale the library derives from a global amax."""
    if g is None:
        return 1.0
    return nvfp4_global_scales(g.float().reshape(-1)[:1].contiguous(), bound)[1]


def fp4_mm(a, b, stochastic: bool = False, seed: int = 0, step: int = 0, *, out_dtype=torch.bfloat16,
           scale_bound: float = 448.0) -> torch.Tensor:
    """a @ b^T for rowwise-quantized a [M, K] and b [N, K]: each the dict of
    to_fp4_operands, or a CUDA tensor it quantizes first (stochastic rounding
    keyed on (seed, step) for a and (seed + 1, step) for b, as fp4_matmul and
    fp4_linear do); the block-scaled product times both decode scales."""
    if torch.is_tensor(a):
        a = to_fp4_operands(a, stochastic, seed, step)
    if torch.is_tensor(b):
        b = to_fp4_operands(b, stochastic, seed + 1, step)
    y = torch._scaled_mm(a["fp4"], b["fp4"].t(), a["scales"], b["scales"], out_dtype=torch.float32)
    s = _scale_dec(a.get("gamax"), scale_bound) * _scale_dec(b.get("gamax"), scale_bound)
    return (y * s).to(out_dtype)


# ---- fp4_matmul: the portable product ---------------------------------------------------------
def _dequantized_operand(t: torch.Tensor, stochastic: bool, seed: int, step: int) -> torch.Tensor:
    q = nvfp4_quantize(t.contiguous(), rounding="sr" if stochastic else "rtn", seed=seed, step=step)
    return nvfp4_dequantize(q["codes"], q["scales"], t.shape[0], t.shape[1], out_dtype="bf16")


def fp4_matmul(a: torch.Tensor, b: torch.Tensor, stochastic: bool = False, seed: int = 0,
               step: int = 0) -> torch.Tensor:
    """a @ b^T with FP4 operands by the portable path ("fp4-train", API:
    fp4_matmul, dequantize and a bf16 product).

    Both operands are quantized rowwise in 1x16 blocks with the page's recipe
    as fp4_linear does (no global scale; round-to-nearest, or stochastic
    rounding keyed on (seed, step) for a and (seed + 1, step) for b) and
    dequantized to bf16 by the library.  Those values are exact in bf16 (a
    grid value of two significant bits times a scale of four), and the
    product accumulates them in fp32 (a library GEMM on their fp32 widening,
    at torch's default full fp32 matmul precision) before one rounding to bf16, so it equals the tensor-core
    product (nvfp4_mm, bf16 out) wherever the fp32 sums are exact and
    otherwise differs only in their order.  a [M, K], b [N, K]: CUDA float32
    / bfloat16, K a multiple of 16; returns bf16 [M, N]."""
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("fp4_matmul: a [M, K] and b [N, K]")
    if a.shape[1] % 16:
        raise ValueError("fp4_matmul: K must be a multiple of 16")
    da = _dequantized_operand(a, stochastic, seed, step)
    db = _dequantized_operand(b, stochastic, seed + 1, step)
    return torch.matmul(da.float(), db.float().t()).to(torch.bfloat16)


# ---- fp4_linear -------------------------------------------------------------------------------
def _pad_rows(t: torch.Tensor, mult: int) -> torch.Tensor:
    pad = (-t.shape[0]) % mult
    if pad == 0:
        return t.contiguous()
    return torch.cat([t, t.new_zeros((pad, t.shape[1]))]).contiguous()


def _quantize_operand(t: torch.Tensor, stochastic: bool, seed: int, step: int) -> dict:
    """1x16 rowwise quantization of a [rows, K] operand (rows padded to 128
    with zeros, which quantize to zero codes and add nothing to a product),
    its scales re-laid for the tensor cores, and its dequantized value."""
    rows = t.shape[0]
    tp = _pad_rows(t, 128)
    q = nvfp4_quantize(tp, rounding="sr" if stochastic else "rtn", seed=seed, step=step)
    deq = nvfp4_dequantize(q["codes"], q["scales"], tp.shape[0], tp.shape[1], out_dtype="f32")[:rows]
    return {"codes": q["codes"], "scales_mma": nvfp4_scales_to_mma(q["scales"]), "rows": tp.shape[0], "deq": deq}


class _FP4Linear(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, stochastic, seed, step):
        M, K = x.shape
        N = weight.shape[0]
        qx = _quantize_operand(x, stochastic, seed, step)
        qw = _quantize_operand(weight, stochastic, seed + 1, step)
        y = nvfp4_mm(qx["codes"], qx["scales_mma"], qw["codes"], qw["scales_mma"], qx["rows"], qw["rows"], K,
                     out_dtype="f32")[:M, :N]
        ctx.save_for_backward(qx["deq"], qw["deq"])
        ctx.dtypes = (x.dtype, weight.dtype)
        return y.to(x.dtype)

    @staticmethod
    def backward(ctx, gy):
        dx_q, dw_q = ctx.saved_tensors
        g = gy.float()
        gx = (g @ dw_q).to(ctx.dtypes[0]) if ctx.needs_input_grad[0] else None
        gw = (g.t() @ dx_q).to(ctx.dtypes[1]) if ctx.needs_input_grad[1] else None
        return gx, gw, None, None, None


def fp4_linear(x: torch.Tensor, weight: torch.Tensor, stochastic: bool = False, seed: int = 0,
               step: int = 0) -> torch.Tensor:
    """y = Q(x) Q(weight)^T ("fp4-train", API: fp4_linear, a quantized-operand
    linear with a straight-through gradient).

    Both operands are quantized rowwise in 1x16 blocks (the page's recipe: no
    global scale; round-to-nearest, or stochastic rounding keyed on (seed,
    step) for x and (seed + 1, step) for the weight) and multiplied on the
    block-scaled FP4 tensor cores (nvfp4_mm, fp32 accumulation).  The
    backward pass treats quantization as the identity: dL/dx = dL/dy Q(w)
    and dL/dw = dL/dy^T Q(x), with the dequantized operands.
    x [M, K], weight [N, K]: CUDA float32 / bfloat16, K a multiple of 64."""
    if x.dim() != 2 or weight.dim() != 2 or x.shape[1] != weight.shape[1]:
        raise ValueError("fp4_linear: x [M, K] and weight [N, K]")
    if x.shape[1] % 64:
        raise ValueError("fp4_linear: K must be a multiple of 64")
    return _FP4Linear.apply(x, weight, stochastic, seed, step)
