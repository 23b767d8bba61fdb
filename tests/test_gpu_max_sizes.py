"""Index arithmetic at the largest sizes, on the GPU against the oracle.

A bf16 tensor past 2^32 elements (65552 x 65552, 8.6 GB; K / 16 = 4097 tiles
and M / 16 = 4097 bands, so every grid has a ragged tail) runs through every
quantize kernel, the amax kernels, dequantize and qdq, and an fp32 copy of it
(17 GB) through the fp32 kernels.  The outputs are compared with the oracle
on five 16-row bands: the first, the ones holding element 2^30 (fp32 byte
2^32), element 2^31 (bf16 byte 2^32) and element 2^32, and the last.  Each
band is checked on its rowwise and columnwise bytes, residual, per-row amax
and dequantized values; the per-row amax is compared on every row.
Stochastic rounding draws on the global element index, so a block read or
written at a wrong offset also draws the wrong words.

The widest input the columnwise kernels take (K = 65535 x 256: 256 columns
per CTA fill a grid's y extent) runs through each columnwise kernel on 16
rows, compared on three column ranges (first, middle, last), with nearest
rounding or four-over-six: their blocks depend on nothing outside their own
columns.

The large tensor is assembled on the device from 256 seeded base rows by
nvfp4_workloads.tiled_row_map (row r = base[p(r)] * 2^e(r), exact), so each
band the oracle takes is rebuilt on the host; the first test checks that the
device tensor holds those values.
"""
import numpy as np
import pytest
import torch

import nvfp4_workloads as W
import oracle
from parity_helpers import assert_same, oracle_kwargs, to_dev, to_np

pytestmark = pytest.mark.gpu

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")

N = 65552                      # rows = columns: 4,297,064,704 elements
P = 256                        # base rows
KMAX = 65535 * 256             # the widest columnwise input


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nv.build()
    nv.load_library()
    with oracle.using_threads(0):
        yield


def _bands():
    b = {0, N // 16 - 1}
    for e in (30, 31, 32):
        b.add(((1 << e) // N) // 16)
    return sorted(b)


BANDS = _bands()               # [0, 1023, 2047, 4095, 4096]


@pytest.fixture(scope="module")
def big():
    base_bits = W.matrix((P, N), seed=93, dtype="bf16", dist="t", outlier_frac=0.01, outlier_factor=50.0)
    p, e = W.tiled_row_map(N, P)
    x = to_dev(base_bits).index_select(0, torch.from_numpy(p).cuda())
    x.mul_(torch.from_numpy(np.exp2(e).astype(np.float32)).cuda().to(torch.bfloat16).view(-1, 1))
    # the oracle's per-row amax of the base rows, scaled exactly by each row's power of two
    rowmax = oracle.amax(base_bits, per_row=True)[p] * np.exp2(e).astype(np.float32)
    d = {"x": x, "base": W.bf16_bits_to_f32(base_bits), "p": p, "e": e, "rowmax": rowmax.astype(np.float32)}
    d["amax"] = np.float32(d["rowmax"].max())
    yield d
    d.clear()
    del x
    torch.cuda.empty_cache()


def _band(big, b):
    """fp32 values of band b (16 rows), rebuilt on the host."""
    return W.tiled_rows(big["base"], big["p"], big["e"], 16 * b, 16 * b + 16)


def _compare_bands(g, kw, band_input, residual=None, res_scale=None):
    """The GPU's full-size outputs against the oracle on each sampled band."""
    okw = oracle_kwargs(kw)
    for b in BANDS:
        r0, r1 = 16 * b, 16 * b + 16
        rb = None if residual is None else (band_input(b, True) * np.float32(res_scale)).astype(np.float32)
        o = oracle.quantize(band_input(b, False), residual=rb, row_offset=r0, **okw)
        assert_same(to_np(g["codes"][r0:r1]), o["codes"], f"codes, band {b}")
        assert_same(to_np(g["scales"][r0:r1]), o["scales"], f"scales, band {b}")
        if "codes_col" in o:
            assert_same(to_np(g["codes_col"][:, 8 * b:8 * b + 8]), o["codes_col"], f"codes_col, band {b}")
            assert_same(to_np(g["scales_col"][:, b:b + 1]), o["scales_col"], f"scales_col, band {b}")
        if okw.get("gamax_mode") == oracle.GAMAX_ROW:
            assert_same(to_np(g["gamax"][r0:r1]), o["gamax"], f"row amax, band {b}")
        if rb is not None:
            assert_same(to_np(residual[r0:r1]), rb, f"residual, band {b}")


def test_device_tensor_holds_the_host_bands(big):
    for b in BANDS:
        assert_same(to_np(big["x"][16 * b:16 * b + 16]), W.to_bf16_bits(_band(big, b)), f"input band {b}")


def test_amax_past_2_32_elements(big):
    A = nv.nvfp4_amax(big["x"])
    R = nv.nvfp4_amax(big["x"], per_row=True)
    torch.cuda.synchronize()
    assert_same(to_np(A), np.array([big["amax"]], np.float32), "tensor amax")
    assert_same(to_np(R), big["rowmax"], "row amax, every row")


BF16_CASES = {
    "rtn 1x16": dict(block="1x16", rounding="rtn"),
    "sr+ef 1x16": dict(block="1x16", rounding="sr", seed=5, step=3),
    "sr+ef 16x16": dict(block="16x16", rounding="sr", seed=5, step=4),
    "rtn 16x16": dict(block="16x16", rounding="rtn"),
    "4o6 mae 1x16 per-row": dict(block="1x16", err_mode="mae", gamax_mode="row"),
    "4o6 mse 16x16 rowwise": dict(block="16x16", err_mode="mse", gamax_mode="tensor_given"),
    "4o6 mae 16x16 row+col": dict(block="16x16", err_mode="mae", gamax_mode="tensor_given", colwise=True),
    "rtn 1x16 row+col": dict(block="1x16", rounding="rtn", colwise=True),
    "sr 16x16 row+col": dict(block="16x16", rounding="sr", seed=9, colwise=True),
    "sr 1x16 row+col": dict(block="1x16", rounding="sr", seed=9, colwise=True),
}


@pytest.mark.parametrize("name", list(BF16_CASES))
def test_bf16_kernels_past_2_32_elements(big, name):
    kw = dict(BF16_CASES[name])
    if kw.get("gamax_mode") == "tensor_given":
        kw["gamax"] = big["amax"]
    ef = name.startswith("sr+ef")
    res = big["x"].float().mul_(2.0 ** -6) if ef else None      # exact: a power of two
    g = nv.nvfp4_quantize(big["x"], residual=res, **kw)
    torch.cuda.synchronize()
    band_input = lambda b, as_f32: _band(big, b) if as_f32 else W.to_bf16_bits(_band(big, b))  # noqa: E731
    _compare_bands(g, kw, band_input, residual=res, res_scale=2.0 ** -6)
    del g, res
    torch.cuda.empty_cache()


def test_dequantize_and_qdq_past_2_32_elements(big):
    q = nv.nvfp4_quantize(big["x"])
    d = nv.nvfp4_dequantize(q["codes"], q["scales"], N, N)
    torch.cuda.synchronize()
    for b in BANDS:
        o = oracle.quantize(W.to_bf16_bits(_band(big, b)), row_offset=16 * b)
        assert_same(to_np(d[16 * b:16 * b + 16]), oracle.dequantize(o["codes"], o["scales"], 16, N),
                    f"dequantized, band {b}")
    del q, d
    torch.cuda.empty_cache()
    out = nv.nvfp4_qdq(big["x"], rounding="sr", seed=2, step=1)["out"]
    torch.cuda.synchronize()
    for b in BANDS:
        o = oracle.qdq(W.to_bf16_bits(_band(big, b)), rounding=oracle.SR, seed=2, step=1, row_offset=16 * b)
        assert_same(to_np(out[16 * b:16 * b + 16]), o["out"], f"qdq, band {b}")
    del out
    torch.cuda.empty_cache()


F32_CASES = {
    "f32 rtn 1x16": dict(block="1x16", rounding="rtn"),
    "f32 4o6 mse 16x16 row+col": dict(block="16x16", err_mode="mse", gamax_mode="tensor_given", colwise=True),
    "f32 sr 1x16 row+col": dict(block="1x16", rounding="sr", seed=11, colwise=True),
}


def test_f32_kernels_past_2_32_elements(big):
    x32 = big["x"].float()                                        # 17 GB, exact
    for name, kw in F32_CASES.items():
        kw = dict(kw)
        if kw.get("gamax_mode") == "tensor_given":
            kw["gamax"] = big["amax"]
        g = nv.nvfp4_quantize(x32, **kw)
        torch.cuda.synchronize()
        _compare_bands(g, kw, lambda b, as_f32: _band(big, b))
        del g
    del x32
    torch.cuda.empty_cache()


WIDE_CASES = {
    "bf16 rtn 1x16": ("bf16", dict(block="1x16", rounding="rtn")),
    "bf16 rtn 16x16": ("bf16", dict(block="16x16", rounding="rtn")),
    "bf16 4o6 mae 16x16": ("bf16", dict(block="16x16", err_mode="mae", gamax_mode="tensor_given")),
    "bf16 4o6 mse 1x16": ("bf16", dict(block="1x16", err_mode="mse", gamax_mode="tensor_given")),
    "f32 rtn 1x16": ("f32", dict(block="1x16", rounding="rtn")),
    "f32 4o6 mse 16x16": ("f32", dict(block="16x16", err_mode="mse", gamax_mode="tensor_given")),
}


def test_columnwise_kernels_at_the_widest_k():
    xb = W.matrix((16, KMAX), seed=94, dtype="bf16")
    x32 = W.bf16_bits_to_f32(xb)
    A = np.float32(oracle.amax(xb)[0])
    dev = {"bf16": to_dev(xb), "f32": to_dev(x32)}
    mid = (KMAX // 2) // 256 * 256 - 2048
    ranges = [(0, 4096), (mid, mid + 4096), (KMAX - 4096, KMAX)]
    for name, (dt, kw) in WIDE_CASES.items():
        kw = dict(kw, colwise=True)
        if kw.get("gamax_mode") == "tensor_given":
            kw["gamax"] = A
        g = nv.nvfp4_quantize(dev[dt], **kw)
        torch.cuda.synchronize()
        okw = oracle_kwargs(kw)
        for c0, c1 in ranges:
            xs = np.ascontiguousarray((xb if dt == "bf16" else x32)[:, c0:c1])
            o = oracle.quantize(xs, **okw)
            what = f"{name}, columns [{c0}, {c1})"
            assert_same(to_np(g["codes"][:, c0 // 2:c1 // 2]), o["codes"], f"codes, {what}")
            assert_same(to_np(g["scales"][:, c0 // 16:c1 // 16]), o["scales"], f"scales, {what}")
            assert_same(to_np(g["codes_col"][c0:c1]), o["codes_col"], f"codes_col, {what}")
            assert_same(to_np(g["scales_col"][c0:c1]), o["scales_col"], f"scales_col, {what}")
        del g
    dev.clear()
    torch.cuda.empty_cache()
