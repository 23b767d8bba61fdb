"""The oracle's worker threads change nothing: every call, run on one thread
and on several, gives the same bytes (each block's arithmetic is the same on
whichever thread runs it; the tensor amax is an order-free maximum).  The
full-size GPU comparisons and the all-core CPU baseline rely on this."""
import numpy as np
import pytest

import nvfp4_workloads as W
import oracle

CASES = [
    ("c1 RTN", lambda: W.c1(), dict()),
    ("c1 SR", lambda: W.c1(), dict(rounding=oracle.SR, seed=3, step=9)),
    ("c3 4o6 MAE tensor", lambda: W.c3()[:256], dict(gamax_mode=oracle.GAMAX_TENSOR, err_mode=oracle.ERR_MAE)),
    ("c3 4o6 MSE row", lambda: W.c3()[:256], dict(gamax_mode=oracle.GAMAX_ROW, err_mode=oracle.ERR_MSE)),
    ("c4 4o6 16x16 row+col", lambda: np.ascontiguousarray(W.c4_specials(W.c4(), with_inf_nan=True)[:256, :1024]),
     dict(block=oracle.BLOCK_16X16, gamax_mode=oracle.GAMAX_TENSOR, err_mode=oracle.ERR_MSE, scale_bound=448.0,
          colwise=True)),
    ("plain 16x16 SR row+col", lambda: W.matrix((128, 320), seed=5, dtype="bf16", dist="t"),
     dict(block=oracle.BLOCK_16X16, rounding=oracle.SR, seed=1, step=2, row_offset=48, colwise=True)),
    ("1x16 RTN_STD tensor", lambda: W.matrix((96, 304), seed=6, dtype="f32", dist="t"),
     dict(rounding=oracle.RTN_STD, gamax_mode=oracle.GAMAX_TENSOR)),
]


def _run(x, kw, threads, ef):
    with oracle.using_threads(threads):
        res = (np.random.default_rng(2).standard_normal(x.shape) * 0.01).astype(np.float32) if ef else None
        o = oracle.quantize(x, residual=res, **kw)
        if res is not None:
            o["residual"] = res
        M, K = x.shape
        gm = kw.get("gamax_mode", oracle.GAMAX_NONE)
        dgm = {oracle.GAMAX_TENSOR: oracle.GAMAX_TENSOR_GIVEN, oracle.GAMAX_ROW: oracle.GAMAX_ROW_GIVEN}.get(gm, gm)
        o["dequant"] = oracle.dequantize(o["codes"], o["scales"], M, K, gamax_mode=dgm, gamax=o["gamax"],
                                         scale_bound=kw.get("scale_bound", 448.0 if "err_mode" not in kw else 256.0),
                                         out_dtype=oracle.F32)
        if gm != oracle.GAMAX_NONE:
            o["amax_row"] = oracle.amax(x, per_row=True)
        return o


@pytest.mark.parametrize("name", [c[0] for c in CASES])
def test_threads_give_the_same_bytes(name):
    _, make, kw = next(c for c in CASES if c[0] == name)
    x = make()
    ef = "err_mode" not in kw and not kw.get("colwise")
    one = _run(x, kw, 1, ef)
    for t in (3, 8):
        many = _run(x, kw, t, ef)
        assert set(one) == set(many)
        for k in one:
            if one[k] is None:
                assert many[k] is None
                continue
            a, b = np.asarray(one[k]), np.asarray(many[k])
            if a.dtype == np.float32:
                a, b = a.view(np.uint32), b.view(np.uint32)
            assert np.array_equal(a, b), f"{name}: {k} differs with {t} threads"


def test_thread_count_is_restored():
    before = oracle.threads()
    with oracle.using_threads(5) as n:
        assert n == 5 and oracle.threads() == 5
    assert oracle.threads() == before


def test_exhaustive_codec_sweep_matches_the_scalar_codec():
    first = np.float32(0.2).view(np.uint32)
    n = 1 << 16
    with oracle.using_threads(4):
        got = oracle.e2m1_encode_rn_bits(int(first), n)
    vals = np.arange(first, first + n, dtype=np.uint32).view(np.float32)
    assert np.array_equal(got, oracle.e2m1_encode_rn(vals))
