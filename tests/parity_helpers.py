"""Shared helpers for the GPU parity tests: run the CUDA path (through the C
ABI binding) and the CPU oracle on the same numpy inputs and compare every
output byte.  The tolerance is zero: codes, scale bytes, amaxes, residuals and
dequantized values must be bit-identical."""
import numpy as np
import torch

import oracle

NAMES = {
    "block": {"1x16": oracle.BLOCK_1X16, "16x16": oracle.BLOCK_16X16},
    "rounding": {"rtn": oracle.RTN, "sr": oracle.SR, "rtn_std": oracle.RTN_STD},
    "gamax_mode": {"none": oracle.GAMAX_NONE, "tensor": oracle.GAMAX_TENSOR,
                   "row": oracle.GAMAX_ROW, "tensor_given": oracle.GAMAX_TENSOR_GIVEN,
                   "row_given": oracle.GAMAX_ROW_GIVEN},
    "err_mode": {"none": oracle.ERR_NONE, "mae": oracle.ERR_MAE, "mse": oracle.ERR_MSE},
}


def to_dev(x: np.ndarray) -> torch.Tensor:
    """numpy fp32 -> cuda float32; numpy uint16 (bf16 bits) -> cuda bfloat16."""
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_kwargs(kw: dict) -> dict:
    out = {}
    for k, v in kw.items():
        if k in NAMES:
            out[k] = NAMES[k][v]
        else:
            out[k] = v
    return out


def assert_same(a: np.ndarray, b: np.ndarray, what: str):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    if a.dtype == np.float32:
        # bit-exact, except that any NaN matches any NaN: IEEE 754 fixes no NaN
        # payload (the GPU returns its canonical NaN for NaN - x)
        both_nan = np.isnan(a) & np.isnan(b)
        a, b = a.view(np.uint32).copy(), b.view(np.uint32).copy()
        a[both_nan] = b[both_nan] = 0
    if not np.array_equal(a, b):
        bad = np.argwhere(a != b)
        first = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {a.size} differ; first at {first}: "
                             f"gpu {a[first]!r} oracle {b[first]!r}")


def quantize_both(x: np.ndarray, residual: np.ndarray | None = None, **kw):
    """Run nvfp4_quantize and the oracle; returns (gpu_dict_np, oracle_dict)."""
    import nvfp4_block_quantization_quantize_gb300 as nv
    rd = None if residual is None else to_dev(residual.copy())
    gkw = dict(kw)
    if isinstance(gkw.get("gamax"), np.ndarray):
        gkw["gamax"] = torch.from_numpy(gkw["gamax"].astype(np.float32)).cuda()
    g = nv.nvfp4_quantize(to_dev(x), residual=rd, **gkw)
    torch.cuda.synchronize()
    gpu = {k: to_np(v) for k, v in g.items()}
    if rd is not None:
        gpu["residual"] = to_np(rd)
    okw = oracle_kwargs(kw)
    res_o = None if residual is None else residual.copy()
    o = oracle.quantize(x, residual=res_o, **okw)
    if res_o is not None:
        o["residual"] = res_o
    return gpu, o


def compare_quant(gpu: dict, o: dict, keys=("codes", "scales", "codes_col", "scales_col",
                                             "gamax", "residual")):
    for k in keys:
        if k in o and o[k] is not None:
            assert k in gpu, f"gpu result lacks {k}"
            assert_same(gpu[k], o[k], k)
