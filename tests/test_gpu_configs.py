"""The five synthetic workloads at full size, GPU against the oracle, tolerance 0.

c1 lives in test_gpu_parity.py.  c2 (the 200-step stored-weight loop) and c3
are compared in full.  c4 and c5 are quantized on the GPU at full size in the
benchmark's launch configuration; the oracle then recomputes sampled 16-row
bands one by one (with the full tensor's amax given, and row_offset so the SR
draws are the full tensor's) and every byte of those bands must match.  A
16-row band determines its rowwise blocks, its 16x16 tiles and its slice of
the columnwise output, so sampled bands are exact, not approximate, checks.
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


def sample_bands(M, n, seed):
    rng = np.random.default_rng(seed)
    nb = M // 16
    picks = {0, nb - 1} | set(int(v) for v in rng.choice(nb, size=min(n, nb), replace=False))
    return sorted(picks)


def check_bands(x, gpu, bands, kw, residual_before=None, residual_after=None):
    """Oracle on each sampled band vs the GPU's full-size outputs."""
    M, K = x.shape
    okw = oracle_kwargs(kw)
    gm = okw.get("gamax_mode", oracle.GAMAX_NONE)
    if gm == oracle.GAMAX_TENSOR:
        A = oracle.amax(x, residual=residual_before)
        assert_same(gpu["gamax"], A, "gamax")
        okw["gamax_mode"], okw["gamax"] = oracle.GAMAX_TENSOR_GIVEN, A
    colwise = okw.get("colwise", False)
    for b in bands:
        r0 = 16 * b
        res = None if residual_before is None else residual_before[r0:r0 + 16].copy()
        o = oracle.quantize(x[r0:r0 + 16], residual=res, row_offset=r0, **okw)
        assert_same(gpu["codes"][r0:r0 + 16], o["codes"], f"codes band {b}")
        assert_same(gpu["scales"][r0:r0 + 16], o["scales"], f"scales band {b}")
        if colwise:
            assert_same(gpu["codes_col"][:, 8 * b:8 * b + 8], o["codes_col"], f"codes_col band {b}")
            assert_same(gpu["scales_col"][:, b:b + 1], o["scales_col"], f"scales_col band {b}")
        if residual_after is not None:
            assert_same(residual_after[r0:r0 + 16], res, f"residual band {b}")


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
    bands = sorted(set(range(8)) | set(sample_bands(x.shape[0], 10, seed=int(bound))))
    check_bands(x, gpu, bands, kw)
    if bound == 256.0 and kind != "inf_nan":
        assert not np.any(gpu["scales"] == 0x7E)      # 256 * 1.5 = 384 < 448: no clipping


# ---- c5: LLM-shaped sweep, bf16 --------------------------------------------------------
_C5 = None


def _c5():
    global _C5
    if _C5 is None:
        _C5 = W.C5()
    return _C5


@pytest.mark.parametrize("name", ["W1", "W2"])
@pytest.mark.parametrize("block", ["1x16", "16x16"])
def test_c5_sr_ef_weights(name, block):
    x = getattr(_c5(), name)
    zeros = np.zeros(x.shape, np.float32)
    kw = dict(block=block, rounding="sr", seed=0)
    # residual = the output of a step-6 call from zeros, then the timed step 7
    _, r6 = run_gpu(x, residual=zeros, step=6, **kw)
    gpu, r7 = run_gpu(x, residual=r6, step=7, **kw)
    bands = sample_bands(x.shape[0], 12, seed=7)
    for b in bands:
        r0 = 16 * b
        res = np.zeros((16, x.shape[1]), np.float32)
        o6 = oracle.quantize(x[r0:r0 + 16], residual=res, row_offset=r0, step=6,
                             **oracle_kwargs(kw))
        assert_same(r6[r0:r0 + 16], res, f"step-6 residual band {b}")
        o7 = oracle.quantize(x[r0:r0 + 16], residual=res, row_offset=r0, step=7,
                             **oracle_kwargs(kw))
        assert_same(gpu["codes"][r0:r0 + 16], o7["codes"], f"codes band {b}")
        assert_same(gpu["scales"][r0:r0 + 16], o7["scales"], f"scales band {b}")
        assert_same(r7[r0:r0 + 16], res, f"step-7 residual band {b}")


@pytest.mark.parametrize("kw", [
    dict(gamax_mode="tensor", err_mode="mae", scale_bound=256.0),
    dict(block="16x16", gamax_mode="tensor", err_mode="mae", scale_bound=256.0, colwise=True),
    dict(rounding="rtn"),
    dict(rounding="sr", seed=0, step=7),
])
@pytest.mark.parametrize("name", ["A", "W1"])
def test_c5_variants(name, kw):
    x = getattr(_c5(), name)
    gpu, _ = run_gpu(x, **kw)
    check_bands(x, gpu, sample_bands(x.shape[0], 12, seed=3), kw)
    if "err_mode" not in kw:
        M, K = x.shape
        d = to_np(nv.nvfp4_dequantize(to_dev(gpu["codes"]), to_dev(gpu["scales"]), M, K))
        for b in sample_bands(M, 6, seed=5):
            r0 = 16 * b
            e = oracle.dequantize(gpu["codes"][r0:r0 + 16], gpu["scales"][r0:r0 + 16], 16, K)
            assert_same(d[r0:r0 + 16], e, f"dequantize band {b}")
