"""The five synthetic workloads at full size, GPU against the oracle, tolerance 0.

c1 lives in test_gpu_parity.py.  Every output byte of c2 (the 200-step
stored-weight loop), c3, c4 and c5 is compared with the oracle's: codes, scale
bytes, columnwise outputs, global amaxes, residuals and dequantized values.
The GPU runs each call at full size in the launch configuration the benchmark
times; the oracle runs on all host cores (its result does not depend on the
thread count: tests/test_oracle_threads.py).
"""
import numpy as np
import pytest
import torch

import nvfp4_workloads as W
import oracle
from parity_helpers import (assert_same, compare_quant, oracle_kwargs, quantize_both, to_dev,
                            to_np)

pytestmark = pytest.mark.gpu

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nv.build()
    nv.load_library()
    with oracle.using_threads(0):
        yield


def check_full(x, gpu, kw, residual_before=None, residual_after=None, step=None):
    """The oracle on the whole tensor vs the GPU's full-size outputs."""
    okw = oracle_kwargs(kw)
    if step is not None:
        okw["step"] = step
    res = None if residual_before is None else residual_before.copy()
    o = oracle.quantize(x, residual=res, **okw)
    for k in ("codes", "scales", "codes_col", "scales_col"):
        if k in o:
            assert_same(gpu[k], o[k], k)
    if o.get("gamax") is not None and okw.get("gamax_mode") in (oracle.GAMAX_TENSOR, oracle.GAMAX_ROW):
        assert_same(gpu["gamax"], o["gamax"], "gamax")
    if residual_after is not None:
        assert_same(residual_after, res, "residual")
    return o


def run_gpu(x, residual=None, **kw):
    rd = None if residual is None else to_dev(residual)
    g = nv.nvfp4_quantize(to_dev(x), residual=rd, **kw)
    torch.cuda.synchronize()
    out = {k: to_np(v) for k, v in g.items()}
    return out, (None if rd is None else to_np(rd))


# ---- c2: stored-weight loop -----------------------------------------------------------
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_c2_error_feedback_loop_200_steps(rounding):
    cfg = W.C2()
    Wg = to_dev(cfg.W0)                      # bf16 weight on the GPU
    Wo = cfg.W0.copy()                       # bf16 bits, oracle side
    rg = torch.zeros(cfg.shape, dtype=torch.float32, device="cuda")
    ro = np.zeros(cfg.shape, np.float32)
    ro_rnd = oracle.SR if rounding == "sr" else oracle.RTN
    for t, G in enumerate(cfg.grads()):
        # x_t = float(W_t) - 1e-4 * G_t (multiply, then subtract; host fp32)
        xt = W.bf16_bits_to_f32(Wo) - G * W.C2_LR
        out = nv.nvfp4_qdq(to_dev(xt), residual=rg, rounding=rounding, seed=0, step=t)
        oq = oracle.qdq(xt, residual=ro, rounding=ro_rnd, seed=0, step=t)
        Wg = out["out"]
        assert_same(to_np(Wg), oq["out"], f"W step {t}")
        assert_same(to_np(rg), ro, f"residual step {t}")
        Wo = oq["out"]
    # error feedback keeps the weight moving: it differs from W0 by now
    assert not np.array_equal(Wo, cfg.W0)


def test_c2_rtn_without_feedback_stalls():
    cfg = W.C2(256, 1024)
    Wo = cfg.W0.copy()
    for t, G in zip(range(20), cfg.grads(20)):
        xt = W.bf16_bits_to_f32(Wo) - G * W.C2_LR
        q = nv.nvfp4_qdq(to_dev(xt))
        Wn = to_np(q["out"])
        assert_same(Wn, oracle.qdq(xt)["out"], f"step {t}")
        Wo = Wn
    # most entries never move under round-to-nearest ("fp4-train": RTN discards
    # sub-step updates)
    moved = np.mean(W.bf16_bits_to_f32(Wo) != W.bf16_bits_to_f32(oracle.qdq(
        W.bf16_bits_to_f32(cfg.W0))["out"]))
    assert moved < 0.2


# ---- c3: four-over-six 1x16 -----------------------------------------------------------
@pytest.mark.parametrize("err", ["mae", "mse"])
@pytest.mark.parametrize("gm", ["tensor", "row", "tensor_given", "row_given"])
def test_c3_four_over_six_1x16(err, gm):
    x = _c3()
    kw = dict(gamax_mode=gm, err_mode=err, scale_bound=256.0)
    if gm == "tensor_given":
        kw["gamax"] = oracle.amax(x)
    if gm == "row_given":
        kw["gamax"] = oracle.amax(x, per_row=True)
    gpu, o = quantize_both(x, **kw)
    compare_quant(gpu, o)


_C3 = None


def _c3():
    global _C3
    if _C3 is None:
        _C3 = W.c3()
    return _C3


# ---- c4: four-over-six 16x16, fp32 8192^2, row + col from one read ------------------
_C4 = {}


def _c4(kind):
    if kind not in _C4:
        base = W.c4()
        _C4["plain"] = base
        _C4["specials"] = W.c4_specials(base, with_inf_nan=False)
        _C4["inf_nan"] = W.c4_specials(base, with_inf_nan=True)
    return _C4[kind]


@pytest.mark.parametrize("bound", [256.0, 448.0])
@pytest.mark.parametrize("kind", ["plain", "specials", "inf_nan"])
def test_c4_four_over_six_16x16_row_and_col(bound, kind):
    x = _c4(kind)
    kw = dict(block="16x16", gamax_mode="tensor", err_mode="mse", scale_bound=bound, colwise=True)
    gpu, _ = run_gpu(x, **kw)
    check_full(x, gpu, kw)
    if bound == 256.0 and kind != "inf_nan":
        assert not np.any(gpu["scales"] == 0x7E)      # 256 * 1.5 = 384 < 448: no clipping


# ---- c5: LLM-shaped sweep, bf16 --------------------------------------------------------
_C5 = None


def _c5():
    global _C5
    if _C5 is None:
        _C5 = W.C5()
    return _C5


@pytest.mark.parametrize("name", ["W1", "W2", "A"])
@pytest.mark.parametrize("block", ["1x16", "16x16"])
def test_c5_sr_ef(name, block):
    x = getattr(_c5(), name)
    zeros = np.zeros(x.shape, np.float32)
    kw = dict(block=block, rounding="sr", seed=0)
    # residual = the output of a step-6 call from zeros, then the timed step 7
    g6, r6 = run_gpu(x, residual=zeros, step=6, **kw)
    check_full(x, g6, kw, residual_before=zeros, residual_after=r6, step=6)
    g7, r7 = run_gpu(x, residual=r6, step=7, **kw)
    check_full(x, g7, kw, residual_before=r6, residual_after=r7, step=7)


@pytest.mark.parametrize("kw", [
    dict(gamax_mode="tensor", err_mode="mae", scale_bound=256.0),
    dict(block="16x16", gamax_mode="tensor", err_mode="mae", scale_bound=256.0, colwise=True),
    dict(rounding="rtn"),
    dict(rounding="sr", seed=0, step=7),
])
@pytest.mark.parametrize("name", ["A", "W1", "W2"])
def test_c5_variants(name, kw):
    x = getattr(_c5(), name)
    gpu, _ = run_gpu(x, **kw)
    o = check_full(x, gpu, kw)
    M, K = x.shape
    gm = "tensor_given" if "gamax_mode" in kw else "none"
    dkw = dict(gamax_mode=gm, scale_bound=kw.get("scale_bound", 448.0))
    if gm != "none":
        dkw["gamax"] = to_dev(gpu["gamax"])
    d = to_np(nv.nvfp4_dequantize(to_dev(gpu["codes"]), to_dev(gpu["scales"]), M, K, **dkw))
    okw = oracle_kwargs(dict(gamax_mode=gm))
    e = oracle.dequantize(o["codes"], o["scales"], M, K, gamax=o.get("gamax"),
                          scale_bound=dkw["scale_bound"], **okw)
    assert_same(d, e, "dequantize")
