"""GPU parity for the standard-NVFP4 scale association (rounding "rtn_std")
and for stochastic rounding with a columnwise output, keyed on the element's
index in x.  The CUDA path against the CPU oracle, bit for bit.
"""
import itertools
import zlib

import numpy as np
import pytest
import torch

import nvfp4_workloads as W
import oracle
from parity_helpers import assert_same, compare_quant, quantize_both, to_dev, to_np

pytestmark = pytest.mark.gpu

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nv.build()
    nv.load_library()


def _seed(*parts):
    return zlib.crc32("".join(map(str, parts)).encode()) % 1000


# every valid combination: a row-scaled tensor has no 16x16 or columnwise
# form, and a columnwise output takes no residual
STD = [c for c in itertools.product(["f32", "bf16"], ["1x16", "16x16"], [False, True],
                                    ["none", "tensor", "row", "tensor_given"], [False, True])
       if not (c[3] == "row" and (c[1] == "16x16" or c[4])) and not (c[2] and c[4])]


@pytest.mark.parametrize("dtype,block,ef,gm,colwise", STD)
def test_standard_association(dtype, block, ef, gm, colwise):
    x = W.matrix((304, 336), seed=_seed(dtype, block, ef, gm, colwise), dtype=dtype, dist="t",
                 outlier_frac=0.01, outlier_factor=40.0)
    res = (np.random.default_rng(2).standard_normal(x.shape) * 0.05).astype(np.float32) if ef else None
    kw = dict(block=block, rounding="rtn_std", gamax_mode=gm, scale_bound=448.0, colwise=colwise)
    if gm == "tensor_given":
        kw["gamax"] = np.array([3.7], np.float32)
    gpu, o = quantize_both(x, residual=res, **kw)
    compare_quant(gpu, o)


def test_standard_association_near_e4m3_midpoints():
    # block maxima swept around the preimages of E4M3 rounding midpoints, where
    # the two associations round differently on some blocks
    import torch as _t
    tab = _t.arange(256, dtype=_t.int32).to(_t.uint8).view(_t.float8_e4m3fn).to(_t.float32).numpy()[8:0x7F]
    mids = ((tab[:-1].astype(np.float64) + tab[1:]) / 2).astype(np.float32)
    A, bound = np.float32(10.0), np.float32(256.0)
    S_enc = np.float32(6.0) * bound / A
    bs = []
    for mid in mids:
        b0 = np.float32(mid * np.float32(6.0) / S_enc)
        up = dn = b0
        bs.append(b0)
        for _ in range(40):
            up, dn = np.nextafter(up, np.float32(np.inf)), np.nextafter(dn, np.float32(-np.inf))
            bs += [up, dn]
    bs = np.array(bs[: len(bs) // 16 * 16], np.float32)
    x = (bs[:, None] * np.linspace(1.0, 0.25, 16, dtype=np.float32)[None, :]).astype(np.float32)
    x = x.reshape(-1, 256)
    for rounding in ("rtn_std", "rtn"):
        gpu, o = quantize_both(x, rounding=rounding, gamax_mode="tensor_given", gamax=np.array([A]),
                               scale_bound=256.0)
        compare_quant(gpu, o)


def test_standard_association_specials():
    x = W.c4_specials(W.c4(256, 512), with_inf_nan=True)
    for gm in ("none", "tensor"):
        gpu, o = quantize_both(x, block="16x16", rounding="rtn_std", gamax_mode=gm, colwise=True)
        compare_quant(gpu, o)


def test_standard_association_qdq():
    x = W.matrix((256, 512), seed=61, dtype="bf16")
    res_g = to_dev(np.zeros(x.shape, np.float32))
    res_o = np.zeros(x.shape, np.float32)
    q = nv.nvfp4_qdq(to_dev(x), rounding="rtn_std", residual=res_g, gamax_mode="tensor", want_codes=True)
    oq = oracle.qdq(x, rounding=oracle.RTN_STD, residual=res_o, gamax_mode=oracle.GAMAX_TENSOR)
    assert_same(to_np(q["out"]), oq["out"], "qdq out")
    assert_same(to_np(q["codes"]), oq["codes"], "qdq codes")
    assert_same(to_np(res_g), res_o, "residual")


PLAIN_COL = list(itertools.product(["rtn", "sr"], ["f32", "bf16"], ["1x16", "16x16"],
                                   ["none", "tensor", "tensor_given"]))


@pytest.mark.parametrize("rounding,dtype,block,gm", PLAIN_COL)
def test_plain_columnwise(rounding, dtype, block, gm):
    x = W.matrix((304, 336), seed=_seed(rounding, dtype, block, gm), dtype=dtype, dist="t")
    kw = dict(block=block, rounding=rounding, seed=13, step=6, row_offset=48, gamax_mode=gm, colwise=True)
    if gm == "tensor_given":
        kw["gamax"] = np.array([9.25], np.float32)
    gpu, o = quantize_both(x, **kw)
    compare_quant(gpu, o)
    if block == "16x16":                          # Q(x^T) = Q(x)^T
        c = gpu["codes"]
        rows = np.empty((c.shape[0], c.shape[1] * 2), np.uint8)
        rows[:, 0::2], rows[:, 1::2] = c & 15, c >> 4
        cc = gpu["codes_col"]
        cols = np.empty((cc.shape[0], cc.shape[1] * 2), np.uint8)
        cols[:, 0::2], cols[:, 1::2] = cc & 15, cc >> 4
        assert np.array_equal(cols, rows.T)


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_plain_columnwise_specials(rounding):
    x = W.c4_specials(W.c4(256, 512), with_inf_nan=True)
    for dt in (x, W.to_bf16_bits(x)):
        gpu, o = quantize_both(dt, block="1x16", rounding=rounding, seed=2, step=3, colwise=True)
        compare_quant(gpu, o)


@pytest.mark.parametrize("rounding", ["rtn", "rtn_std"])
@pytest.mark.parametrize("shape", [(16, 16), (48, 1552), (272, 528), (80, 48)])
def test_rtn_columnwise_shapes(rounding, shape):
    """1x16 rowwise + columnwise nearest rounding over CTA-sized and ragged
    shapes: one tile; 97 tiles across (four CTA columns, the last ragged);
    17 bands (five CTA rows, the last with one band); fewer tiles than a
    warp's lanes."""
    for dtype in ("bf16", "f32"):
        x = W.matrix(shape, seed=_seed("rtncol", rounding, shape, dtype), dtype=dtype, dist="t")
        for gm in ("none", "tensor"):
            gpu, o = quantize_both(x, block="1x16", rounding=rounding, gamax_mode=gm, colwise=True)
            compare_quant(gpu, o)
