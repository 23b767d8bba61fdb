"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
element by element, tolerance zero, on seeded inputs from nvfp4_workloads.

Sizes here let the oracle finish in seconds while spanning many CTAs, several
256-column chunks and ragged tails (K not a multiple of 256, M not a multiple
of 128).  The full-size configurations are in test_gpu_configs.py.
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


def mat(shape, seed, dtype="f32", dist="normal", outliers=0.0):
    return W.matrix(shape, seed=seed, dtype=dtype, dist=dist, outlier_frac=outliers,
                    outlier_factor=50.0)


# ---- the fp4-train recipe (no global scale) ----------------------------------------------
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_c1_quantize_dequantize_qdq(rounding):
    x = W.c1()
    gpu, o = quantize_both(x, rounding=rounding, seed=0, step=0)
    compare_quant(gpu, o)
    M, K = x.shape
    for od, ood in (("bf16", oracle.BF16), ("f32", oracle.F32)):
        d = nv.nvfp4_dequantize(to_dev(gpu["codes"]), to_dev(gpu["scales"]), M, K, out_dtype=od)
        assert_same(to_np(d), oracle.dequantize(o["codes"], o["scales"], M, K, out_dtype=ood),
                    f"dequantize {od}")
    q = nv.nvfp4_qdq(to_dev(x), rounding=rounding, want_codes=True)
    oq = oracle.qdq(x, rounding=oracle.SR if rounding == "sr" else oracle.RTN)
    assert_same(to_np(q["out"]), oq["out"], "qdq out")
    assert_same(to_np(q["codes"]), oq["codes"], "qdq codes")


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_c1_scalar_2_3(rounding):
    for x in (W.c1_23(), W.c1_23b()):
        gpu, o = quantize_both(x, rounding=rounding, seed=0, step=0)
        compare_quant(gpu, o)
    dq = to_np(nv.nvfp4_dequantize(to_dev(gpu["codes"]), to_dev(gpu["scales"]), *x.shape,
                                   out_dtype="f32"))
    mean = dq[:, 1:].astype(np.float64).mean()
    if rounding == "sr":
        assert abs(mean - 2.3) <= 0.005      # "fp4-train", Correctness
    else:
        assert mean == 2.0


# every valid combination (a per-row global scale is 1x16 only)
PLAIN = [c for c in itertools.product(["f32", "bf16"], ["1x16", "16x16"], ["rtn", "sr"], [False, True],
                                      ["none", "tensor", "row", "tensor_given"])
         if not (c[1] == "16x16" and c[4] == "row")]


@pytest.mark.parametrize("dtype,block,rounding,ef,gm", PLAIN)
def test_plain_matrix(dtype, block, rounding, ef, gm):
    x = mat((304, 304), seed=zlib.crc32(f"{dtype}{block}{rounding}{ef}{gm}".encode()) % 1000, dtype=dtype,
            dist="t")
    res = (np.random.default_rng(1).standard_normal(x.shape) * 0.05).astype(np.float32) if ef else None
    kw = dict(block=block, rounding=rounding, seed=11, step=5, row_offset=3, gamax_mode=gm,
              scale_bound=448.0)
    if gm == "tensor_given":
        kw["gamax"] = np.array([7.5], np.float32)
    gpu, o = quantize_both(x, residual=res, **kw)
    compare_quant(gpu, o)


# every valid combination (a row-scaled tensor has no 16x16 or columnwise form)
FOUR_SIX = [c for c in itertools.product(["f32", "bf16"], ["mae", "mse"], [256.0, 448.0],
                                         ["1x16", "16x16"], ["tensor", "row"], [False, True])
            if not (c[4] == "row" and (c[3] == "16x16" or c[5]))]


@pytest.mark.parametrize("dtype,err,bound,block,gm,colwise", FOUR_SIX)
def test_four_over_six_matrix(dtype, err, bound, block, gm, colwise):
    for shape in ((128, 128), (256, 512), (304, 304), (128, 320)):
        x = mat(shape, seed=sum(shape), dtype=dtype, outliers=0.02)
        gpu, o = quantize_both(x, block=block, gamax_mode=gm, err_mode=err, scale_bound=bound,
                               colwise=colwise)
        compare_quant(gpu, o)


def _tie_inputs():
    """Inputs on which the two four-over-six candidates' error sums are often
    equal or within a few ulps: small multiples of 1/4 (many values lie on
    both candidates' grids, all-zero blocks included), the same nudged by one
    ulp in random places, and blocks repeating one value."""
    rng = np.random.default_rng(61)
    a = (rng.integers(-6, 7, (256, 512)) * 0.25).astype(np.float32)
    b = a.copy()
    m = rng.random(b.shape) < 0.3
    b[m] = np.nextafter(b[m], np.float32(np.inf) * rng.choice([-1, 1], m.sum()).astype(np.float32))
    c = np.repeat(rng.standard_normal((256, 32)).astype(np.float32), 16, axis=1)
    c[:16] = 0.0
    return a, b, c


@pytest.mark.parametrize("err,bound", [("mae", 256.0), ("mse", 256.0), ("mae", 448.0), ("mse", 448.0)])
def test_four_over_six_ties(err, bound):
    """Where the candidates' sums tie or nearly tie, the decision falls back to
    the exact sums: those blocks and tiles must still match the oracle.  With
    bound 448 every block whose amax equals the tensor's has s6f = 448 and a
    map-to-4 scale that saturates to the same byte: identical candidates,
    equal nonzero sums, so the exact path decides for most blocks of the
    first two inputs (their maximum magnitude recurs in most blocks)."""
    for x in _tie_inputs():
        for kw in (dict(), dict(block="16x16", colwise=True), dict(block="16x16"),
                   dict(colwise=True)):
            for xx in (x, W.to_bf16_bits(x)):
                gpu, o = quantize_both(xx, gamax_mode="tensor", err_mode=err, scale_bound=bound, **kw)
                compare_quant(gpu, o)


@pytest.mark.parametrize("shape", [(16, 16), (1, 16), (3, 48), (32, 272), (48, 4112), (2048, 1024),
                                   (64, 1024)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_and_page_shapes(shape, dtype):
    x = mat(shape, seed=shape[0] * 7 + shape[1], dtype=dtype)
    gpu, o = quantize_both(x, rounding="sr", seed=3, step=1)
    compare_quant(gpu, o)
    if shape[0] % 16 == 0:
        gpu, o = quantize_both(x, block="16x16", gamax_mode="tensor", err_mode="mse",
                               colwise=True)
        compare_quant(gpu, o)
        gpu, o = quantize_both(x, gamax_mode="tensor", err_mode="mae", colwise=True)
        compare_quant(gpu, o)


def test_empty_inputs():
    for M, K in ((0, 64), (16, 0), (0, 0)):
        x = torch.empty((M, K), dtype=torch.float32, device="cuda")
        r = nv.nvfp4_quantize(x, gamax_mode="tensor")
        torch.cuda.synchronize()
        assert r["codes"].numel() == M * K // 2
        assert float(r["gamax"][0]) == 0.0
    r = nv.nvfp4_quantize(torch.empty((8, 0), device="cuda"), gamax_mode="row")
    torch.cuda.synchronize()
    assert np.all(to_np(r["gamax"]) == 0)


def test_special_values():
    x = W.c4_specials(W.c4(256, 512), with_inf_nan=False)
    xi = W.c4_specials(W.c4(256, 512), with_inf_nan=True)
    for xx in (x, xi):
        for kw in (dict(), dict(rounding="sr", seed=5), dict(block="16x16"),
                   dict(gamax_mode="tensor", err_mode="mse", block="16x16", colwise=True),
                   dict(gamax_mode="tensor", err_mode="mse", block="16x16", colwise=True,
                        scale_bound=448.0),
                   dict(gamax_mode="row", err_mode="mae"),
                   dict(gamax_mode="tensor", err_mode="mae"),
                   dict(gamax_mode="tensor", err_mode="mse"),
                   dict(gamax_mode="tensor", err_mode="mae", block="16x16", colwise=True),
                   dict(gamax_mode="tensor", err_mode="mae", colwise=True)):
            gpu, o = quantize_both(xx, **kw)
            compare_quant(gpu, o)
        res = np.zeros(xx.shape, np.float32)
        gpu, o = quantize_both(xx, residual=res, rounding="sr", seed=2, step=9)
        compare_quant(gpu, o)


def test_subnormal_and_large_plain_scales():
    rng = np.random.default_rng(44)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x *= np.exp2(rng.integers(-140, 12, (64, 16))).repeat(16, axis=1).astype(np.float32)
    for kw in (dict(), dict(rounding="sr", seed=9), dict(gamax_mode="tensor"),
               dict(gamax_mode="row"), dict(block="16x16")):
        gpu, o = quantize_both(x, **kw)
        compare_quant(gpu, o)


@pytest.mark.parametrize("block", ["1x16", "16x16"])
def test_sr_bf16_tiny_values(block):
    """Stochastic rounding of bf16 input without a residual or a global scale
    skips the tiny-element check (a nonzero bf16 value over an E4M3 scale
    never gives a zero quotient): blocks mixing bf16 subnormals, zeros and
    values up to 2^20 must still match the oracle, draw for draw."""
    rng = np.random.default_rng(91)
    x = rng.standard_normal((256, 512)).astype(np.float32)
    x *= np.exp2(rng.integers(-140, 20, (256, 512))).astype(np.float32)
    x[rng.random(x.shape) < 0.05] = 0.0
    x[:, :16] = np.float32(2.0 ** -133) * rng.integers(-3, 4, (256, 16)).astype(np.float32)
    xb = W.to_bf16_bits(x)
    for seed, step in ((1, 0), (2, 7)):
        gpu, o = quantize_both(xb, block=block, rounding="sr", seed=seed, step=step)
        compare_quant(gpu, o)


def test_dequantize_global_modes():
    x = mat((128, 256), seed=5, outliers=0.05)
    for gm, given in (("tensor", "tensor_given"), ("row", "row_given")):
        gpu, o = quantize_both(x, gamax_mode=gm, err_mode="mse", scale_bound=256.0)
        compare_quant(gpu, o)
        for od, ood in (("bf16", oracle.BF16), ("f32", oracle.F32)):
            d = nv.nvfp4_dequantize(to_dev(gpu["codes"]), to_dev(gpu["scales"]), *x.shape,
                                    gamax_mode=given, gamax=to_dev(gpu["gamax"]),
                                    scale_bound=256.0, out_dtype=od)
            e = oracle.dequantize(o["codes"], o["scales"], *x.shape,
                                  gamax_mode=oracle.GAMAX_TENSOR_GIVEN if gm == "tensor"
                                  else oracle.GAMAX_ROW_GIVEN, gamax=o["gamax"],
                                  scale_bound=256.0, out_dtype=ood)
            assert_same(to_np(d), e, f"dequantize {gm} {od}")


@pytest.mark.parametrize("kw", [dict(), dict(rounding="sr", seed=4, step=2),
                                dict(gamax_mode="tensor", err_mode="mae"),
                                dict(gamax_mode="row", err_mode="mse"),
                                dict(block="16x16", rounding="sr")])
def test_qdq_matches(kw):
    x = mat((256, 512), seed=8, dtype="bf16", dist="t")
    res = (np.random.default_rng(3).standard_normal(x.shape) * 0.01).astype(np.float32)
    use_res = kw.get("err_mode", "none") == "none"
    rd = to_dev(res) if use_res else None
    q = nv.nvfp4_qdq(to_dev(x), residual=rd, want_codes=True, **kw)
    ro = res.copy() if use_res else None
    from parity_helpers import oracle_kwargs
    oq = oracle.qdq(x, residual=ro, **oracle_kwargs(kw))
    assert_same(to_np(q["out"]), oq["out"], "qdq out")
    assert_same(to_np(q["codes"]), oq["codes"], "qdq codes")
    assert_same(to_np(q["scales"]), oq["scales"], "qdq scales")
    if use_res:
        assert_same(to_np(rd), ro, "qdq residual")


def test_amax_entry_point():
    x = mat((96, 160), seed=9, dtype="bf16", outliers=0.1)
    res = (np.random.default_rng(4).standard_normal(x.shape)).astype(np.float32)
    for per_row in (False, True):
        for r in (None, res):
            g = nv.nvfp4_amax(to_dev(x), residual=None if r is None else to_dev(r), per_row=per_row)
            e = oracle.amax(x, residual=r, per_row=per_row)
            assert_same(to_np(g), e, "amax")


def test_row_shards_match_the_whole_tensor():
    """Row shards quantized with row_offset and the whole tensor's amax
    reproduce the unsharded result, stochastic rounding included."""
    x = mat((512, 256), seed=10, dtype="bf16")
    whole = nv.nvfp4_quantize(to_dev(x), rounding="sr", seed=77, step=3, gamax_mode="tensor")
    A = whole["gamax"]
    parts = [nv.nvfp4_quantize(to_dev(x[r0:r0 + 128]), rounding="sr", seed=77, step=3,
                               row_offset=r0, gamax_mode="tensor_given", gamax=A)
             for r0 in range(0, 512, 128)]
    torch.cuda.synchronize()
    assert_same(np.concatenate([to_np(p["codes"]) for p in parts]), to_np(whole["codes"]), "codes")
    assert_same(np.concatenate([to_np(p["scales"]) for p in parts]), to_np(whole["scales"]), "scales")


def test_host_buffer_path():
    x = mat((64, 128), seed=12)
    r = nv.nvfp4_quantize(torch.from_numpy(x), rounding="sr", seed=1)
    assert r["codes"].device.type == "cpu"
    o = oracle.quantize(x, rounding=oracle.SR, seed=1)
    assert_same(r["codes"].numpy(), o["codes"], "codes")


def test_host_pinned_buffers_and_residual():
    """Host tensors (pinned here) through the staged path: results, the
    in-place residual and a host dequantize match the oracle byte for byte."""
    x = mat((64, 256), seed=14)
    xh = torch.from_numpy(x).pin_memory()
    r0 = mat((64, 256), seed=15) * np.float32(0.01)
    rh = torch.from_numpy(r0.copy()).pin_memory()
    g = nv.nvfp4_quantize(xh, rounding="sr", seed=5, step=2, residual=rh)
    assert g["codes"].device.type == "cpu"
    ro = r0.copy()
    o = oracle.quantize(x, rounding=oracle.SR, seed=5, step=2, residual=ro)
    assert_same(g["codes"].numpy(), o["codes"], "codes")
    assert_same(g["scales"].numpy(), o["scales"], "scales")
    assert_same(rh.numpy(), ro, "residual")
    dq = nv.nvfp4_dequantize(g["codes"], g["scales"], 64, 256)
    assert dq.device.type == "cpu"
    assert_same(dq.view(torch.int16).numpy().view(np.uint16), oracle.dequantize(o["codes"], o["scales"], 64, 256),
                "dequantized")


def test_host_pageable_outputs_and_device_call_refusal():
    x = mat((64, 128), seed=16)
    codes = torch.empty((64, 64), dtype=torch.uint8)
    g = nv.nvfp4_quantize(torch.from_numpy(x), codes=codes)
    assert g["codes"] is codes
    assert_same(codes.numpy(), oracle.quantize(x)["codes"], "codes")
    with pytest.raises(ValueError):
        nv.nvfp4_quantize(to_dev(x), codes=torch.empty((64, 64), dtype=torch.uint8))
    with pytest.raises(ValueError):
        nv.nvfp4_quantize(to_dev(x), rounding="sr", residual=torch.zeros((64, 128)))


def test_mixed_device_tensors_are_checked_or_refused():
    """Tensors whose pointers the kernels take as they are: a device residual
    of a host call is updated in place when it is float32 [M,K] and
    contiguous, and refused otherwise (a zero-stride view would have the
    kernel write M*K floats into K); device codes with host scales, host or
    short operands of the FP4 product, and host probe inputs are refused."""
    x = mat((64, 128), seed=17)
    r0 = mat((64, 128), seed=18) * np.float32(0.01)
    rd = to_dev(r0.copy())
    g = nv.nvfp4_quantize(torch.from_numpy(x), rounding="sr", seed=3, residual=rd)
    ro = r0.copy()
    o = oracle.quantize(x, rounding=oracle.SR, seed=3, residual=ro)
    assert_same(g["codes"].numpy(), o["codes"], "codes")
    assert_same(to_np(rd), ro, "device residual of a host call")
    with pytest.raises(ValueError):
        nv.nvfp4_quantize(torch.from_numpy(x), rounding="sr", residual=torch.zeros((1, 128), device="cuda").expand(64, 128))
    with pytest.raises(ValueError):
        nv.nvfp4_qdq(torch.from_numpy(x), rounding="sr", residual=to_dev(r0).t().contiguous().t())
    with pytest.raises(ValueError):
        nv.nvfp4_amax(torch.from_numpy(x), residual=to_dev(r0).to(torch.bfloat16))
    q = nv.nvfp4_quantize(to_dev(x))
    with pytest.raises(ValueError):
        nv.nvfp4_dequantize(q["codes"], q["scales"].cpu(), 64, 128)
    z = torch.zeros(128 * 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):                      # a host operand
        nv.nvfp4_mm(z, z.cpu(), z, z, 128, 128, 128)
    with pytest.raises(ValueError):                      # codes_a holds 8 KB of the 16 KB it reads
        nv.nvfp4_mm(z[:128 * 64], z, z, z, 128, 128, 256)
    with pytest.raises(ValueError):
        nv.nvfp4_mm(z, z, z, z, 128, 128, 128, out=torch.empty((128, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        nv.nvfp4_probe_divide(torch.ones(4), torch.ones(4, device="cuda"))
    with pytest.raises(ValueError):
        nv.nvfp4_scales_to_mma(q["scales"], out=torch.empty(16, dtype=torch.uint8, device="cuda"))
    host_out = torch.empty((128, 8), dtype=torch.uint8)
    assert nv.nvfp4_scales_to_mma(q["scales"].cpu(), out=host_out) is host_out
    assert_same(host_out.numpy(), to_np(nv.nvfp4_scales_to_mma(q["scales"])), "scales_to_mma into a host tensor")


def _host(x: np.ndarray, pinned: bool = True) -> torch.Tensor:
    t = (torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16) if x.dtype == np.uint16
         else torch.from_numpy(x.copy()))
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_host_pipelined_calls(dtype):
    """Host calls of at least 256 rows run in row chunks on three streams
    (copies in, kernels, copies out overlapping): every byte, the in-place
    residual and the stochastic draws (keyed on row_offset + the chunk's
    first row) must equal the oracle's for the whole tensor."""
    M, K = 1040, 512                                   # chunks of 272 rows and a 224-row tail
    x = mat((M, K), seed=81, dtype=dtype, outliers=0.01)
    r0 = mat((M, K), seed=82) * np.float32(0.01)
    for blk in ("1x16", "16x16"):
        rh = _host(r0)
        g = nv.nvfp4_quantize(_host(x), block=blk, rounding="sr", seed=7, step=3, row_offset=48,
                              residual=rh)
        assert g["codes"].device.type == "cpu"
        ro = r0.copy()
        o = oracle.quantize(x, block=oracle.BLOCK_16X16 if blk == "16x16" else oracle.BLOCK_1X16,
                            rounding=oracle.SR, seed=7, step=3, row_offset=48, residual=ro)
        assert_same(g["codes"].numpy(), o["codes"], f"{blk} codes")
        assert_same(g["scales"].numpy(), o["scales"], f"{blk} scales")
        assert_same(rh.numpy(), ro, f"{blk} residual")
    ga = oracle.amax(x)
    gr = oracle.amax(x, per_row=True)
    for err in ("mae", "mse"):
        for gm, gv, ogm in (("tensor_given", ga, oracle.GAMAX_TENSOR_GIVEN),
                            ("row_given", gr, oracle.GAMAX_ROW_GIVEN)):
            g = nv.nvfp4_quantize(_host(x, pinned=False), gamax_mode=gm, gamax=torch.from_numpy(gv.copy()),
                                  err_mode=err, scale_bound=256.0)
            o = oracle.quantize(x, gamax_mode=ogm, gamax=gv, err_mode=oracle.ERR_MAE if err == "mae"
                                else oracle.ERR_MSE, scale_bound=256.0)
            assert_same(g["codes"].numpy(), o["codes"], f"{err} {gm} codes")
            assert_same(g["scales"].numpy(), o["scales"], f"{err} {gm} scales")
    rh = _host(r0)
    q = nv.nvfp4_qdq(_host(x), rounding="sr", seed=2, step=5, residual=rh, want_codes=True)
    ro = r0.copy()
    oq = oracle.qdq(x, rounding=oracle.SR, seed=2, step=5, residual=ro)
    assert_same(q["out"].view(torch.int16).numpy().view(np.uint16), oq["out"], "qdq out")
    assert_same(q["codes"].numpy(), oq["codes"], "qdq codes")
    assert_same(rh.numpy(), ro, "qdq residual")
    o = oracle.quantize(x, gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=ga, err_mode=oracle.ERR_MAE,
                        scale_bound=256.0)
    for od, ood in (("bf16", oracle.BF16), ("f32", oracle.F32)):
        d = nv.nvfp4_dequantize(torch.from_numpy(o["codes"]), torch.from_numpy(o["scales"]), M, K,
                                gamax_mode="tensor_given", gamax=torch.from_numpy(ga.copy()), scale_bound=256.0,
                                out_dtype=od)
        e = oracle.dequantize(o["codes"], o["scales"], M, K, gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=ga,
                              scale_bound=256.0, out_dtype=ood)
        dn = d.view(torch.int16).numpy().view(np.uint16) if od == "bf16" else d.numpy()
        assert_same(dn, e, f"dequantize {od}")


ROWCOL_SHAPES = [(16, 16), (16, 1040), (48, 528), (80, 240), (272, 48), (64, 512), (208, 784)]


@pytest.mark.parametrize("shape", ROWCOL_SHAPES)
def test_row_col_kernels_shape_sweep(shape):
    """The staged row+col kernels over shapes that start and end inside a
    CTA along both axes (a CTA is 4 bands x 32 tiles for bf16 four-over-six
    and 1x16 nearest rounding, 4 bands x 8 tiles for fp32 four-over-six):
    one tile; one band of 65 tiles; 3 bands x 33 tiles; 5 bands x 15 tiles;
    17 bands x 3 tiles; exactly one CTA; 13 bands x 49 tiles.  Every output
    byte against the oracle, both error modes and both bounds for
    four-over-six, and nearest rounding with either global-scale mode."""
    M, K = shape
    for dtype in ("bf16", "f32"):
        x = mat(shape, seed=zlib.crc32(f"rc{shape}{dtype}".encode()) % 1000, dtype=dtype, dist="t",
                outliers=0.02)
        for err in ("mae", "mse"):
            for bound in (256.0, 448.0):
                gpu, o = quantize_both(x, block="16x16", gamax_mode="tensor", err_mode=err, scale_bound=bound,
                                       colwise=True)
                compare_quant(gpu, o)
        for gm in ("none", "tensor"):
            gpu, o = quantize_both(x, block="1x16", gamax_mode=gm, colwise=True)
            compare_quant(gpu, o)


def test_host_non_blocking_calls():
    """Non-blocking host calls (returning once enqueued, so successive calls
    overlap) give the oracle's bytes: row-chunked calls, whole calls
    (columnwise output, a computed amax, fewer than 256 rows), a residual
    carried from one call to the next, a call whose inputs are a pending
    call's host outputs (codes, scales, gamax), and outputs written into
    given host tensors."""
    M, K = 528, 256
    x = mat((M, K), seed=91, dtype="bf16", outliers=0.01)
    xs = mat((64, 128), seed=92)                       # under 256 rows: one chunk
    r0 = mat((M, K), seed=93) * np.float32(0.01)
    xh, xsh, rh = _host(x), _host(xs), _host(r0)
    ro = r0.copy()
    given = torch.empty((M, K // 2), dtype=torch.uint8).pin_memory()
    sr = []
    for t in range(3):                                 # the residual read by the next call
        sr.append(nv.nvfp4_quantize(xh, rounding="sr", seed=5, step=t, residual=rh,
                                    codes=given if t == 2 else None, non_blocking=True))
    rc = nv.nvfp4_quantize(xh, block="16x16", gamax_mode="tensor", err_mode="mse", scale_bound=256.0,
                           colwise=True, non_blocking=True)
    q1 = nv.nvfp4_quantize(xsh, gamax_mode="tensor", err_mode="mae", scale_bound=256.0, non_blocking=True)
    dq = nv.nvfp4_dequantize(q1["codes"], q1["scales"], 64, 128, gamax_mode="tensor_given",
                             gamax=q1["gamax"], scale_bound=256.0, out_dtype="f32", non_blocking=True)
    qd = nv.nvfp4_qdq(xh, rounding="sr", seed=9, step=1, want_codes=True, non_blocking=True)
    nv.nvfp4_synchronize()
    assert sr[2]["codes"] is given
    for t in range(3):
        o = oracle.quantize(x, rounding=oracle.SR, seed=5, step=t, residual=ro)
        assert_same(sr[t]["codes"].numpy(), o["codes"], f"sr step {t} codes")
        assert_same(sr[t]["scales"].numpy(), o["scales"], f"sr step {t} scales")
    assert_same(rh.numpy(), ro, "residual after three steps")
    ga = oracle.amax(x)
    assert_same(rc["gamax"].numpy(), ga, "computed gamax")
    o = oracle.quantize(x, block=oracle.BLOCK_16X16, gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=ga,
                        err_mode=oracle.ERR_MSE, scale_bound=256.0, colwise=True)
    for k in ("codes", "scales", "codes_col", "scales_col"):
        assert_same(rc[k].numpy(), o[k], f"row+col {k}")
    gs = oracle.amax(xs)
    o1 = oracle.quantize(xs, gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=gs, err_mode=oracle.ERR_MAE,
                         scale_bound=256.0)
    assert_same(q1["codes"].numpy(), o1["codes"], "small call codes")
    e = oracle.dequantize(o1["codes"], o1["scales"], 64, 128, gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=gs,
                          scale_bound=256.0, out_dtype=oracle.F32)
    assert_same(dq.numpy(), e, "dequantize of pending outputs")
    oq = oracle.qdq(x, rounding=oracle.SR, seed=9, step=1)
    assert_same(qd["out"].view(torch.int16).numpy().view(np.uint16), oq["out"], "qdq out")
    assert_same(qd["codes"].numpy(), oq["codes"], "qdq codes")
    with pytest.raises(ValueError):
        nv.nvfp4_quantize(xh, non_blocking=True, stream=torch.cuda.Stream())


def test_stream_argument_is_honoured():
    x = to_dev(mat((256, 256), seed=13))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        r = nv.nvfp4_quantize(x, stream=s)
    s.synchronize()
    ref = nv.nvfp4_quantize(x)
    torch.cuda.synchronize()
    assert torch.equal(r["codes"], ref["codes"])
