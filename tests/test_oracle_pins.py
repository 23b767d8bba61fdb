"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/page_values.json), closed forms, library routines
(torch's fp8/bf16 casts, curand's host Philox generator), brute force on small
inputs, and invariants of the method.  A plausible slip in the oracle (a
dropped term, a wrong tie rule, sign, index or summation order) fails one of
them.

Not pinned by anything outside the oracle ("parity unpinned"): the exact
association of the four-over-six error value ((q*d)*A)/(6*bound) away from the
S_enc = 1 regime, and the S_enc fallback to 1 when the global amax is 0, Inf or
NaN.  The pages name these steps but print no value that fixes them.  The
dequantized value with a global scale, (q*d)*S_dec, is pinned: q*d is exact,
so it is the exact triple product rounded once (checked with rationals).
"""
import ctypes
import json
import os

import numpy as np
import pytest

import nvfp4_workloads as W
import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))
GRID = np.array(GOLD["e2m1_grid"]["value"], np.float64)
f32 = np.float32


# ---- independent brute-force codecs used as pins ---------------------------------------
def brute_e2m1_rn(v):
    """Nearest signed grid point by exhaustive distance comparison (float64,
    exact for the magnitudes used), ties to the even index, |v| >= 6 -> 7,
    NaN -> +6."""
    v = np.asarray(v, np.float32).ravel()
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - GRID[None, :])
    best = d.min(1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(8) % 2 == 0)[None, :]
    idx = np.where(cand.sum(1) > 1, np.argmax(even, 1), np.argmax(cand, 1))
    idx = np.where(a >= 6.0, 7, idx)
    out = (np.signbit(v).astype(np.uint8) << 3) | idx.astype(np.uint8)
    out[np.isnan(v)] = 7
    return out


def torch_e4m3_table():
    import torch
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def brute_e4m3(s):
    """Nearest non-negative finite E4M3 value (from torch's decode table) to s >= 0,
    ties to the even code; s >= 448 saturates."""
    tab = torch_e4m3_table()[:0x7F]                # 0x00..0x7E, all finite
    s = np.asarray(s, np.float32).ravel().astype(np.float64)
    d = np.abs(s[:, None] - tab[None, :])
    best = d.min(1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(0x7F) % 2 == 0)[None, :]
    idx = np.where(cand.sum(1) > 1, np.argmax(even, 1), np.argmax(cand, 1))
    return np.where(s >= 448.0, 0x7E, idx).astype(np.uint8)


def values_near(points, n_ulps=2048):
    """All fp32 values within +-n_ulps of each point (plus the points)."""
    out = []
    for p in points:
        b = np.array([p], np.float32).view(np.uint32)[0].astype(np.int64)
        out.append(np.arange(max(b - n_ulps, 0), b + n_ulps + 1, dtype=np.int64).astype(np.uint32))
    return np.concatenate(out).view(np.float32)


# ---- environment -----------------------------------------------------------------------
def test_fp_environment_keeps_subnormals():
    oracle._load()
    assert oracle._load().orc_fp_env_ok() == 1


# ---- e2m1 ------------------------------------------------------------------------------
def test_e2m1_grid_is_the_pages_grid():
    vals = oracle.e2m1_value(np.arange(16))
    assert np.array_equal(vals[:8].astype(np.float64), GRID)
    assert np.array_equal(vals[8:].astype(np.float64), -GRID)
    assert np.signbit(vals[8])  # code 0x8 is -0


def test_e2m1_rn_page_values():
    # 2.3 rounds to 2 [fp4-train, Correctness]; NaN encodes to +6 [4o6 PR, Design]
    assert oracle.e2m1_encode_rn([2.3])[0] == 4
    assert oracle.e2m1_value(oracle.e2m1_encode_rn([2.3]))[0] == GOLD["rtn_of_2_3"]["value"]
    assert oracle.e2m1_encode_rn([np.nan])[0] == GOLD["nan_encodes_to"]["value"]
    neg_nan = np.array([0xFFC00000], np.uint32).view(np.float32)
    assert oracle.e2m1_encode_rn(neg_nan)[0] == 7
    # saturation and infinities
    assert list(oracle.e2m1_encode_rn([6.0, 7.0, 1e30, np.inf, -np.inf])) == [7, 7, 7, 7, 15]
    # exact midpoints go to the even index
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    assert list(oracle.e2m1_encode_rn(mids)) == [0, 2, 2, 4, 4, 6, 6]
    assert list(oracle.e2m1_encode_rn([-0.0, -0.1])) == [8, 8]


def test_e2m1_rn_brute_force_near_every_boundary():
    pts = [0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0]
    v = values_near(pts, 4096)
    rng = np.random.default_rng(11)
    v = np.concatenate([v, rng.uniform(0, 8, 200_000).astype(np.float32),
                        np.array([2.0 ** -149, 2.0 ** -126, 1e-30, 1e30], np.float32)])
    v = np.concatenate([v, -v])
    assert np.array_equal(oracle.e2m1_encode_rn(v), brute_e2m1_rn(v))


def test_e2m1_sr_probabilities_are_the_fractional_distance():
    # [fp4-train, Method]: the higher point is chosen with probability equal to
    # the fractional distance.  For fixed v the decision is a step in u at p.
    for v, lo, hi in [(2.3, 2.0, 3.0), (0.1, 0.0, 0.5), (4.9, 4.0, 6.0), (1.2, 1.0, 1.5)]:
        p = (float(f32(v)) - lo) / (hi - lo)
        u = np.array([0.0, p * 0.999999, p, p * 1.000001, 0.999999])
        got = oracle.e2m1_value(oracle.e2m1_encode_sr(np.full(5, v, np.float32), u))
        assert list(got) == [hi, hi, lo, lo, lo], (v, got)
    # grid points never move; |v| >= 6 saturates; NaN -> +6; sign is kept
    for g in GRID:
        assert oracle.e2m1_value(oracle.e2m1_encode_sr([g], [0.0]))[0] == g
    assert list(oracle.e2m1_encode_sr([7.0, np.nan, -2.3], [0.0, 0.0, 0.0])) == [7, 7, 13]


# ---- e4m3 ------------------------------------------------------------------------------
def test_e4m3_decode_matches_torch_for_all_bytes():
    tab = torch_e4m3_table()
    mine = oracle.e4m3_decode(np.arange(256)).astype(np.float64)
    nan = np.isnan(tab)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], tab[~nan])
    assert np.nanmax(tab) == GOLD["e4m3_max"]["value"]


def test_e4m3_encode_brute_force_and_torch():
    import torch
    tab = torch_e4m3_table()[:0x7F]
    mids = (tab[:-1] + tab[1:]) / 2
    s = values_near(np.concatenate([tab, mids]).astype(np.float32), 64)
    rng = np.random.default_rng(5)
    s = np.concatenate([s, np.exp2(rng.uniform(-16, 9.5, 200_000)).astype(np.float32),
                        np.array([2.0 ** -10, 447.99997, 448.0, 448.00003, 464.0, 1e30, np.inf],
                                 np.float32)])
    s = s[s >= 0]
    got = oracle.e4m3_encode(s)
    assert np.array_equal(got, brute_e4m3(s))
    ok = s < 464.0   # torch's cast does not saturate beyond that
    t = torch.from_numpy(s[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[ok], t)
    assert oracle.e4m3_encode([np.nan])[0] == 0x7F
    assert oracle.e4m3_encode([2.0 ** -10])[0] == 0x00   # tie at half the smallest subnormal


# ---- bf16 ------------------------------------------------------------------------------
def test_bf16_round_trip_matches_torch():
    import torch
    rng = np.random.default_rng(9)
    bits = rng.integers(0, 2 ** 32, 500_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    mine = oracle.f32_to_bf16(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    widened = W.bf16_bits_to_f32(h)
    got = np.array([oracle._load().orc_bf16_to_f32(int(v)) for v in h[::257]], np.float32)
    assert np.array_equal(got.view(np.uint32), widened[::257].view(np.uint32))


# ---- Philox ----------------------------------------------------------------------------
def _curand_host():
    for path in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    return None


def test_philox_matches_curand_host_generator():
    """curand's host Philox4x32-10 generator (a library routine) lays block b of
    its stream at counter (b // 65536, 0, b % 65536, 0) with key = seed; a
    generator offset advances word 0 and carries into word 1."""
    cur = _curand_host()
    if cur is None:
        pytest.skip("libcurand not loadable")
    PHILOX = 161  # CURAND_RNG_PSEUDO_PHILOX4_32_10
    for seed in (0, 0x0123456789ABCDEF, 0xFEDCBA9876543210):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for offset_blocks, expect_ctr0, expect_ctr1 in ((0, 0, 0), (65536 * 7, 7, 0),
                                                       (65536 * (2 ** 32 + 3), 3, 1)):
            g = ctypes.c_void_p()
            assert cur.curandCreateGeneratorHost(ctypes.byref(g), PHILOX) == 0
            assert cur.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
            assert cur.curandSetGeneratorOffset(g, ctypes.c_ulonglong(4 * offset_blocks)) == 0
            buf = np.zeros(4 * 24, np.uint32)
            assert cur.curandGenerate(g, buf.ctypes.data_as(ctypes.c_void_p),
                                      ctypes.c_size_t(buf.size)) == 0
            cur.curandDestroyGenerator(g)
            for j in range(24):
                ours = oracle.philox4x32_10([expect_ctr0, expect_ctr1, j, 0], key)
                assert np.array_equal(ours, buf[4 * j:4 * j + 4]), (seed, offset_blocks, j)


# ---- scales and blocks: closed forms ------------------------------------------------------
def test_block_of_2_3_closed_form():
    # 2.3/6 = 0.38333 -> e4m3 0.375 (0x2C); 2.3/0.375 = 6.13 saturates to code 7; dq 2.25
    x = np.full((4, 16), 2.3, np.float32)
    for rnd in (oracle.RTN, oracle.SR):
        r = oracle.quantize(x, rounding=rnd)
        assert np.all(r["scales"] == 0x2C) and np.all(r["codes"] == 0x77)
        dq = oracle.dequantize(r["codes"], r["scales"], 4, 16, out_dtype=oracle.F32)
        assert np.all(dq == f32(2.25))


def test_block_with_6_has_unit_scale_and_rtn_bias():
    x = W.c1_23b()[:1000]
    r = oracle.quantize(x)
    assert np.all(r["scales"] == 0x38)             # 6/6 = 1.0
    dq = oracle.dequantize(r["codes"], r["scales"], *x.shape, out_dtype=oracle.F32)
    assert np.all(dq[:, 0] == 6.0)
    assert np.all(dq[:, 1:] == f32(GOLD["rtn_of_2_3"]["value"]))


def test_blocks_below_e4m3_range_quantize_to_zero():
    # [fp4-train, Requirements and limits]: absmax/6 <= 2^-10 gives scale 0 and zero codes
    x = np.zeros((3, 16), np.float32)
    x[0, :] = np.linspace(-2.0 ** -12, 2.0 ** -12, 16)
    x[1, 5] = 6 * 2.0 ** -10          # b/6 == 2^-10 exactly: the tie goes to 0
    x[2, 5] = 6 * 2.0 ** -10 * 1.01   # just above: smallest subnormal scale 2^-9
    r = oracle.quantize(x)
    assert list(r["scales"][:, 0]) == [0x00, 0x00, 0x01]
    assert np.all(r["codes"][:2] == 0)
    res = np.zeros_like(x)
    oracle.quantize(x, residual=res)
    assert np.array_equal(res[:2], x[:2])          # error feedback banks the whole value


def test_single_element_blocks_all_bf16_values():
    """Every bf16 value v as the only nonzero of a 1x16 block: scale = nearest
    e4m3 to fp32(|v|/6) (brute force), code = nearest grid point to fp32(v/d)."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = W.bf16_bits_to_f32(h)
    keep = np.isfinite(v)
    h, v = h[keep], v[keep]
    x = np.zeros((v.size, 16), np.uint16)
    x[:, 3] = h
    r = oracle.quantize(x)
    s6f = np.abs(v) / f32(6.0)
    sf = brute_e4m3(np.minimum(s6f, f32(448.0)))
    assert np.array_equal(r["scales"][:, 0], sf)
    d = torch_e4m3_table()[sf].astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = v / d
    code = np.where(d == 0, 0, brute_e2m1_rn(q))
    got = (r["codes"][:, 1] >> 4)
    assert np.array_equal(got, code.astype(np.uint8))
    assert np.all(r["codes"][:, [0, 2, 3, 4, 5, 6, 7]] == 0)
    assert np.all(r["codes"][:, 1] & 0x0F == 0)


def test_plain_scale_division_is_correctly_rounded_near_e4m3_midpoints():
    """fp32 block amaxes within a few ulps of 6 x (an e4m3 midpoint): the scale
    must use the correctly rounded b / 6 (numpy's IEEE division), not a
    reciprocal multiply, to land on the right side of the midpoint."""
    tab = torch_e4m3_table()[:0x7F]
    mids = ((tab[:-1] + tab[1:]) / 2 * 6).astype(np.float32)
    b = values_near(mids[mids < 2600], 48)
    b = b[b > 0]
    x = np.zeros((b.size, 16), np.float32)
    x[:, 9] = b
    r = oracle.quantize(x)
    assert np.array_equal(r["scales"][:, 0], brute_e4m3(np.minimum(b / f32(6.0), f32(448.0))))


def test_plain_scale_is_nearest_e4m3_random_blocks():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((4000, 16)) * np.exp2(rng.uniform(-14, 12, (4000, 1)))).astype(np.float32)
    r = oracle.quantize(x)
    b = np.abs(x).max(1)
    assert np.array_equal(r["scales"][:, 0], brute_e4m3(np.minimum(b / f32(6.0), f32(448.0))))


# ---- global scale ------------------------------------------------------------------------
def test_global_scale_closed_forms():
    assert oracle.global_scales(1536.0, 256.0) == (1.0, 1.0)
    assert oracle.global_scales(2688.0, 448.0) == (1.0, 1.0)
    assert oracle.global_scales(768.0, 256.0) == (2.0, 0.5)
    for A in (0.0, np.inf, np.nan, -3.0):
        assert oracle.global_scales(A, 256.0) == (1.0, 1.0)
    enc, dec = oracle.global_scales(1e-38, 256.0)
    assert enc == np.finfo(np.float32).max and dec > 0


def rn_f32(fr):
    """The fp32 value nearest to the rational fr (ties to even), computed with
    integers: the plain definition of one correctly rounded fp32 operation."""
    from fractions import Fraction
    fr = Fraction(fr)
    if fr == 0:
        return f32(0.0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = max(e, -126) - 23                      # quantum of the result's binade
    m = a / Fraction(2) ** q                   # significand in units of the quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return f32(sign * float(Fraction(n) * Fraction(2) ** q))


def _frac(v):
    from fractions import Fraction
    return Fraction(float(v))


def test_global_scales_are_correctly_rounded_divisions():
    """S_enc = RN(6*bound / A) (clamped to FLT_MAX) and S_dec = RN(1 / S_enc)
    ("Add NVFP4 four-over-six (row-wise) quantization to the training
    prototype", Design: S_enc / S_dec among the correctly rounded divisions)."""
    from fractions import Fraction
    rng = np.random.default_rng(31)
    As = np.exp2(rng.uniform(-20, 20, 3000)).astype(np.float32) * rng.uniform(1, 2, 3000).astype(np.float32)
    for bound in (256.0, 448.0):
        for A in As:
            enc, dec = oracle.global_scales(float(A), bound)
            want = rn_f32(Fraction(int(6 * bound)) / _frac(A))
            assert enc == want, (A, bound)
            assert dec == rn_f32(1 / _frac(enc)), (A, bound)


def test_dequantize_with_a_global_scale_rounds_the_exact_product_once():
    """Dequantized value = (q * d) * S_dec ("fp4-train", API dequantize; the
    four-over-six page's decode scale S_dec): q * d is exact (a two-bit grid
    significand times a four-bit E4M3 one), so the result is the exact product
    q * d * S_dec rounded once.  Checked with rationals for every code and every
    positive scale byte, at global amaxes whose S_dec is not a power of two;
    the other association q * (d * S_dec) rounds twice and must differ
    somewhere among these cases."""
    from fractions import Fraction
    tab = torch_e4m3_table()
    codes = np.arange(16, dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)      # 16 codes, one row
    M, K = 126, 16
    c = np.tile(packed, (M, 1))
    s = np.arange(1, 127, dtype=np.uint8).reshape(M, 1)                # every positive scale byte
    differs = 0
    for A in (np.float32(1.0), np.float32(3.7), np.float32(1234.5678), np.float32(0.0173)):
        for bound in (256.0, 448.0):
            enc, dec = oracle.global_scales(float(A), bound)
            assert np.float32(dec) != np.exp2(np.round(np.log2(dec)))   # not a power of two
            got = oracle.dequantize(c, s, M, K, gamax_mode=oracle.GAMAX_TENSOR_GIVEN,
                                    gamax=np.array([A], np.float32), scale_bound=bound,
                                    out_dtype=oracle.F32)
            for i in range(M):
                d = Fraction(float(tab[int(s[i, 0])]))
                for j in range(16):
                    q = Fraction(float(oracle.e2m1_value(codes[j])))
                    want = rn_f32(q * d * _frac(dec))
                    if codes[j] == 8:
                        want = f32(-0.0)              # -0 times a positive scale
                    assert got[i, j].view(np.uint32) == want.view(np.uint32), (A, bound, i, j)
                    if rn_f32(q * _frac(rn_f32(d * _frac(dec)))) != want:
                        differs += 1
    assert differs > 0


def test_ef_residual_with_a_global_scale_uses_the_same_dequantized_value():
    """Under error feedback with a global scale the residual is y - (q*d)*S_dec,
    one fp32 subtraction from the once-rounded dequantized value."""
    from fractions import Fraction
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((32, 64)) * 3).astype(np.float32)
    r0 = (rng.standard_normal(x.shape) * 0.05).astype(np.float32)
    A = np.float32(11.3)
    res = r0.copy()
    q = oracle.quantize(x, residual=res, gamax_mode=oracle.GAMAX_TENSOR_GIVEN,
                        gamax=np.array([A], np.float32), scale_bound=448.0)
    enc, dec = oracle.global_scales(float(A), 448.0)
    tab = torch_e4m3_table()
    y = x + r0
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            byte = q["codes"][i, j // 2]
            code = (byte >> 4) if j % 2 else (byte & 0xF)
            qv = Fraction(float(oracle.e2m1_value(np.uint8(code))))
            d = Fraction(float(tab[q["scales"][i, j // 16]]))
            dq = rn_f32(qv * d * _frac(dec))
            assert res[i, j].view(np.uint32) == rn_f32(_frac(y[i, j]) - _frac(dq)).view(np.uint32)


# ---- stochastic rounding -------------------------------------------------------------------
def test_sr_mean_of_2_3_over_a_million_draws():
    g = GOLD["sr_mean_of_2_3"]
    x = W.c1_23b()                                   # 1,000,005 copies of 2.3 at scale 1
    r = oracle.quantize(x, rounding=oracle.SR, seed=0, step=0)
    dq = oracle.dequantize(r["codes"], r["scales"], *x.shape, out_dtype=oracle.F32)
    vals = dq[:, 1:].astype(np.float64)
    assert vals.size >= g["draws_at_least"]
    assert set(np.unique(vals)) == {2.0, 3.0}
    assert abs(vals.mean() - g["value"]) <= g["tolerance"]
    # RTN of the same input is biased to 2.000
    r2 = oracle.quantize(x)
    dq2 = oracle.dequantize(r2["codes"], r2["scales"], *x.shape, out_dtype=oracle.F32)
    assert dq2[:, 1:].mean() == GOLD["rtn_of_2_3"]["value"]


def test_sr_interval_frequencies():
    rng_vals = [0.1, 0.7, 1.2, 1.9, 2.3, 3.3, 4.9, 5.5]
    rows = 4000
    x = np.zeros((rows * len(rng_vals), 16), np.float32)
    x[:, 0] = 6.0
    for i, v in enumerate(rng_vals):
        x[i * rows:(i + 1) * rows, 1:] = v
    r = oracle.quantize(x, rounding=oracle.SR, seed=1234, step=5)
    dq = oracle.dequantize(r["codes"], r["scales"], *x.shape, out_dtype=oracle.F32).astype(np.float64)
    for i, v in enumerate(rng_vals):
        a = float(f32(v))
        k = np.searchsorted(GRID, a, side="right") - 1
        lo, hi = GRID[k], GRID[k + 1]
        p = (a - lo) / (hi - lo)
        cells = dq[i * rows:(i + 1) * rows, 1:]
        assert set(np.unique(cells)) <= {lo, hi}
        n = cells.size
        up = np.count_nonzero(cells == hi)
        z = (up - n * p) / np.sqrt(n * p * (1 - p))
        assert abs(z) < 5, (v, up / n, p)


def test_sr_is_unbiased_per_element_over_steps():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((32, 64)).astype(np.float32)
    steps = 256
    acc = np.zeros(x.shape, np.float64)
    for t in range(steps):
        r = oracle.quantize(x, rounding=oracle.SR, seed=99, step=t)
        acc += oracle.dequantize(r["codes"], r["scales"], *x.shape, out_dtype=oracle.F32)
    mean = acc / steps
    r = oracle.quantize(x)
    d = np.repeat(oracle.e4m3_decode(r["scales"]).astype(np.float64), 16, axis=1)
    gap = np.where(np.abs(x) / d < 2, 0.5, np.where(np.abs(x) / d < 4, 1.0, 2.0)) * d
    z = (mean - x) / (0.5 * gap / np.sqrt(steps))
    assert np.max(np.abs(z)) < 6
    assert abs(z.mean()) < 5 / np.sqrt(z.size)  # aggregate bias ~ 0


def _curand_words(seed, first_block, nblocks):
    """Words of curand's host Philox stream starting at block `first_block`."""
    cur = _curand_host()
    g = ctypes.c_void_p()
    assert cur.curandCreateGeneratorHost(ctypes.byref(g), 161) == 0
    assert cur.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
    assert cur.curandSetGeneratorOffset(g, ctypes.c_ulonglong(4 * first_block)) == 0
    buf = np.zeros(4 * nblocks, np.uint32)
    assert cur.curandGenerate(g, buf.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(buf.size)) == 0
    cur.curandDestroyGenerator(g)
    return buf


def test_sr_draw_layout_against_curand_stream():
    """Element idx at (seed, step) draws word idx % 4 of Philox4x32-10 with
    counter (idx / 4, step) and key seed, keeping its top 24 bits.  curand's
    host stream holds counter (c, 0, s, 0) at block c * 65536 + s."""
    if _curand_host() is None:
        pytest.skip("libcurand not loadable")
    for seed, step in ((0, 0), (0x5EED5EED12345678, 7), (42, 65535)):
        for idx0 in (0, 1000, 4 * 123457):
            idx = np.arange(idx0, idx0 + 4, dtype=np.uint64)
            words = _curand_words(seed, (idx0 // 4) * 65536 + step, 1)
            expect = (words >> 8).astype(np.float64) * 2.0 ** -24
            assert np.array_equal(oracle.sr_uniform(seed, step, idx), expect)
    # inside quantize: element (r, c) of an [R,16] block matrix uses idx = r*16 + c
    seed, step = 0xABCDEF, 3
    x = np.full((4, 16), 2.3, np.float32)
    x[:, 0] = 6.0
    r = oracle.quantize(x, rounding=oracle.SR, seed=seed, step=step, row_offset=2)
    dq = oracle.dequantize(r["codes"], r["scales"], 4, 16, out_dtype=oracle.F32)
    p = float(f32(2.3)) - 2.0
    for row in range(4):
        for blk in range(4):
            g_idx = (2 + row) * 16 + 4 * blk
            w = _curand_words(seed, (g_idx // 4) * 65536 + step, 1)
            u = (w >> 8).astype(np.float64) * 2.0 ** -24
            for j in range(4):
                c = 4 * blk + j
                if c == 0:
                    continue
                assert dq[row, c] == (3.0 if u[j] < p else 2.0)


def test_sr_draw_depends_on_seed_step_and_global_index():
    x = np.full((8, 16), 2.3, np.float32)
    x[:, 0] = 6.0
    base = oracle.quantize(x, rounding=oracle.SR, seed=7, step=3)["codes"]
    assert not np.array_equal(base, oracle.quantize(x, rounding=oracle.SR, seed=8, step=3)["codes"])
    assert not np.array_equal(base, oracle.quantize(x, rounding=oracle.SR, seed=7, step=4)["codes"])
    # row_offset shifts the global index: rows [4,8) alone with offset 4 match
    part = oracle.quantize(x[4:], rounding=oracle.SR, seed=7, step=3, row_offset=4)["codes"]
    assert np.array_equal(part, base[4:])


# ---- error feedback ----------------------------------------------------------------------
def test_ef_time_average_of_2_3():
    g = GOLD["rtn_ef_time_average_of_2_3"]
    blk = np.array([[6.0] + [2.3] * 15], np.float32)
    means = {}
    for T in (10, 37, 64, 100, 101, 1000):
        res = np.zeros_like(blk)
        total = np.zeros(16, np.float64)
        for _ in range(T):
            r = oracle.quantize(blk, residual=res)
            total += oracle.dequantize(r["codes"], r["scales"], 1, 16, out_dtype=oracle.F32)[0]
        means[T] = total[1] / T
        # telescoping: sum_t dq_t = T*x - r_T (up to fp32 rounding of x + r)
        assert abs(total[1] - (T * float(f32(2.3)) - float(res[0, 1]))) < 1e-4 * T
        assert abs(means[T] - 2.3) <= 0.5 / T + 1e-6
    # the page prints 2.297; that is what the average reads at e.g. T = 37, 64, 101
    assert any(round(m, g["printed_digits"]) == g["value"] for m in means.values())


def test_rtn_without_feedback_discards_sub_step_updates():
    # [fp4-train]: under RTN an update below half a quantization step is lost
    W0 = np.array([[6.0] + [2.0] * 15], np.float32)
    Wt = W0.copy()
    for _ in range(50):
        r = oracle.quantize(Wt + f32(0.01))
        Wt = oracle.dequantize(r["codes"], r["scales"], 1, 16, out_dtype=oracle.F32)
    assert np.array_equal(Wt, W0)
    Wt, res = W0.copy(), np.zeros_like(W0)
    for _ in range(50):
        r = oracle.quantize(Wt + f32(0.01), residual=res)
        Wt = oracle.dequantize(r["codes"], r["scales"], 1, 16, out_dtype=oracle.F32)
    assert np.all(Wt[0, 1:] > 2.0)


def test_ef_residual_is_input_minus_dequant():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    r0 = (rng.standard_normal(x.shape) * 0.01).astype(np.float32)
    res = r0.copy()
    q = oracle.quantize(x, residual=res, rounding=oracle.SR, seed=1, step=2)
    dq = oracle.dequantize(q["codes"], q["scales"], *x.shape, out_dtype=oracle.F32)
    assert np.array_equal(res, (x + r0) - dq)


# ---- four-over-six -------------------------------------------------------------------------
def _unit_regime(block, bound=256.0):
    """A = 6*bound makes S_enc = 1 and the error value (q*d*A)/(6*bound) = q*d exactly."""
    return dict(gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=np.array([6 * bound], np.float32),
                scale_bound=bound, block=block)


def test_four_over_six_tie_selects_map_to_6():
    x = np.zeros((2, 16), np.float32)
    x[0, :4] = [6.0, 3.0, 1.5, -6.0]   # exact under both d6 = 1 and d4 = 1.5
    for em in (oracle.ERR_MAE, oracle.ERR_MSE):
        r = oracle.quantize(x, err_mode=em, **_unit_regime(oracle.BLOCK_1X16))
        assert r["scales"][0, 0] == 0x38          # map-to-6 (1.0), not 0x3C (1.5)
        assert r["scales"][1, 0] == 0x00          # all-zero block: both errors 0


def test_four_over_six_picks_map_to_4_when_strictly_better():
    x = np.zeros((1, 16), np.float32)
    x[0, :3] = [6.0, 4.5, -4.5]         # 4.5 = 3 * 1.5 is exact only under map-to-4
    for em in (oracle.ERR_MAE, oracle.ERR_MSE):
        r = oracle.quantize(x, err_mode=em, **_unit_regime(oracle.BLOCK_1X16))
        assert r["scales"][0, 0] == 0x3C
        dq = oracle.dequantize(r["codes"], r["scales"], 1, 16, out_dtype=oracle.F32)
        assert np.array_equal(dq, x)


def test_four_over_six_bound_256_never_clips():
    # [4o6 PR, What]: 256 * 1.5 = 384 < 448
    gold = GOLD["four_over_six_default_bound"]
    x = W.matrix((256, 1024), seed=12, outlier_frac=0.01, outlier_factor=50.0)
    for block in (oracle.BLOCK_1X16, oracle.BLOCK_16X16):
        for gm in (oracle.GAMAX_TENSOR, oracle.GAMAX_ROW):
            if block == oracle.BLOCK_16X16 and gm == oracle.GAMAX_ROW:
                continue
            r = oracle.quantize(x, block=block, gamax_mode=gm, err_mode=oracle.ERR_MAE,
                                scale_bound=gold["value"])
            d = oracle.e4m3_decode(r["scales"])
            assert d.max() <= gold["expanded"] and np.all(r["scales"] != 0x7E)


def test_four_over_six_bound_448_caps_map_to_4_scale():
    x = W.matrix((16, 64), seed=13)
    x[3, 17] = 100.0                   # this block's amax equals the tensor amax
    r = oracle.quantize(x, gamax_mode=oracle.GAMAX_TENSOR, err_mode=oracle.ERR_MSE,
                        scale_bound=448.0)
    assert r["gamax"][0] == 100.0
    assert r["scales"][3, 1] == 0x7E   # both candidates capped at 448: identical, tie -> map-to-6


def _seq(e):
    s = f32(0)
    for v in e:
        s = f32(s + f32(v))
    return s


def _pairwise(e):
    e = [f32(v) for v in e]
    while len(e) > 1:
        e = [f32(e[i] + e[i + 1]) for i in range(0, len(e), 2)]
    return e[0]


def _order_block(rng):
    """A 1x16 block in the S_enc = 1, d6 = 1, d4 = 1.5 regime whose per-element
    MAE errors are known in closed form: 6.0 -> (0, 0); 4.5 -> (0.5, 0);
    2.0 -> (0, 0.25); a tiny delta -> (delta, delta)."""
    ys, e6, e4 = [0.0] * 16, [0.0] * 16, [0.0] * 16
    ys[0] = 6.0
    pos = rng.permutation(np.arange(1, 16))
    ys[pos[0]] = 4.5
    e6[pos[0]] = 0.5
    for p in pos[1:3]:
        ys[p] = 2.0
        e4[p] = 0.25
    for p in pos[3:]:
        d = int(rng.integers(1, 8)) * 2.0 ** -int(rng.integers(25, 29))
        ys[p], e6[p], e4[p] = d, d, d
    return ys, e6, e4


def test_four_over_six_error_sum_is_sequential_in_element_order():
    rng = np.random.default_rng(77)
    blocks, expect = [], []
    while len(blocks) < 64:
        ys, e6, e4 = _order_block(rng)
        seq4 = _seq(e4) < _seq(e6)
        if seq4 != (_pairwise(e4) < _pairwise(e6)) or seq4 != (_seq(e4[::-1]) < _seq(e6[::-1])):
            blocks.append(ys)
            expect.append(0x3C if seq4 else 0x38)
    assert 0x3C in expect and 0x38 in expect
    x = np.array(blocks, np.float32)
    r = oracle.quantize(x, err_mode=oracle.ERR_MAE, **_unit_regime(oracle.BLOCK_1X16))
    assert list(r["scales"][:, 0]) == expect


def test_four_over_six_16x16_uses_the_width16_tree():
    tree = GOLD["tree16"]["value"]

    def tree_sum(R):
        def ev(node):
            if isinstance(node, int):
                return f32(R[node])
            return f32(ev(node[0]) + ev(node[1]))
        return ev(tree)

    rng = np.random.default_rng(5)
    tiles, expect = [], []
    tries = 0
    while len(tiles) < 16 and tries < 200000:
        tries += 1
        rows = [_order_block(rng) for _ in range(16)]
        # only row 0 keeps its 6.0 at column 0; others start with 0 error
        for i in range(1, 16):
            rows[i][0][0] = 0.0
        R6 = [_seq(r[1]) for r in rows]
        R4 = [_seq(r[2]) for r in rows]
        t4 = tree_sum(R4) < tree_sum(R6)
        if t4 != (_seq(R4) < _seq(R6)):
            tiles.append(np.array([r[0] for r in rows], np.float32))
            expect.append(0x3C if t4 else 0x38)
    assert len(tiles) == 16
    x = np.concatenate(tiles, axis=1)            # 16 x 256: 16 tiles side by side
    r = oracle.quantize(x, err_mode=oracle.ERR_MAE, **_unit_regime(oracle.BLOCK_16X16))
    assert list(r["scales"][0, :]) == expect
    assert np.all(r["scales"] == r["scales"][0:1, :])   # the tile's byte on all 16 rows


def test_four_over_six_error_value_in_unit_regime_is_q_times_d():
    # With S_enc = 1 the chosen candidate's dequantized values give exactly the
    # error the selection used: check the choice against brute-force errors.
    rng = np.random.default_rng(8)
    x = np.clip(rng.standard_normal((500, 16)) * 2, -5.9, 5.9).astype(np.float32)
    x[:, 0] = 6.0                                   # block amax 6: d6 = 1, d4 = 1.5
    tab = torch_e4m3_table()
    for em in (oracle.ERR_MAE, oracle.ERR_MSE):
        r = oracle.quantize(x, err_mode=em, **_unit_regime(oracle.BLOCK_1X16))
        E = []
        for d in (1.0, 1.5):
            enc = f32(1.0) / f32(d)
            q = oracle.e2m1_value(brute_e2m1_rn(x * enc)).reshape(x.shape).astype(np.float32)
            diff = q * f32(d) - x
            e = np.abs(diff) if em == oracle.ERR_MAE else diff * diff
            E.append(np.array([_seq(row) for row in e]))
        pick4 = E[1] < E[0]
        assert np.array_equal(r["scales"][:, 0], np.where(pick4, 0x3C, 0x38).astype(np.uint8))
        assert tab[0x3C] == 1.5 and tab[0x38] == 1.0


def test_nan_semantics():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((32, 64)).astype(np.float32)
    xn = x.copy()
    xn[3, 5] = np.nan
    xn[7, 16:32] = np.nan                          # an all-NaN group
    for kw in (dict(), dict(gamax_mode=oracle.GAMAX_TENSOR, err_mode=oracle.ERR_MSE,
                            scale_bound=256.0)):
        a = oracle.quantize(x, **kw)
        b = oracle.quantize(xn, **kw)
        # the NaN element encodes to +6 (code 7 in the odd nibble of byte 2)
        assert (b["codes"][3, 2] >> 4) == 7
        # all-NaN group: amax 0 -> scale 0
        assert b["scales"][7, 1] == 0
        # NaN-free groups are untouched
        mask = np.ones(a["scales"].shape, bool)
        mask[3, 0] = mask[7, 1] = False
        assert np.array_equal(a["scales"][mask], b["scales"][mask])
        cm = np.repeat(mask, 8, axis=1)
        assert np.array_equal(a["codes"][cm], b["codes"][cm])
    assert oracle.amax(xn)[0] == oracle.amax(x)[0]


def test_columnwise_is_rowwise_of_transpose():
    x = W.matrix((64, 96), seed=30, dist="t")
    for em, block in ((oracle.ERR_NONE, oracle.BLOCK_1X16), (oracle.ERR_MSE, oracle.BLOCK_16X16),
                      (oracle.ERR_MAE, oracle.BLOCK_1X16)):
        kw = dict(block=block, err_mode=em, gamax_mode=oracle.GAMAX_TENSOR, scale_bound=256.0)
        r = oracle.quantize(x, colwise=True, **kw)
        t = oracle.quantize(np.ascontiguousarray(x.T), **kw)
        assert np.array_equal(r["codes_col"], t["codes"])
        assert np.array_equal(r["scales_col"], t["scales"])


def test_qdq_is_quantize_then_dequantize_and_exact_in_bf16():
    x = W.matrix((48, 160), seed=31)
    q = oracle.qdq(x)
    r = oracle.quantize(x)
    d = oracle.dequantize(r["codes"], r["scales"], *x.shape, out_dtype=oracle.F32)
    assert np.array_equal(q["out"], oracle.f32_to_bf16(d))
    # without a global scale every dequantized value is exact in bf16
    assert np.array_equal(W.bf16_bits_to_f32(q["out"]), d)


def test_row_mode_equals_per_row_given():
    x = W.matrix((8, 64), seed=32, outlier_frac=0.05, outlier_factor=30)
    r = oracle.quantize(x, gamax_mode=oracle.GAMAX_ROW, err_mode=oracle.ERR_MAE, scale_bound=256.0)
    assert np.array_equal(r["gamax"], np.abs(x).max(1))
    for i in range(8):
        s = oracle.quantize(x[i:i + 1], gamax_mode=oracle.GAMAX_TENSOR_GIVEN,
                            gamax=r["gamax"][i:i + 1], err_mode=oracle.ERR_MAE, scale_bound=256.0)
        assert np.array_equal(s["codes"][0], r["codes"][i])
        assert np.array_equal(s["scales"][0], r["scales"][i])


# ---- the standard NVFP4 association (nearest rounding, b * (S_enc * (1/6))) -------------
def _unpack_codes(c):
    """[R, C/2] packed bytes -> [R, C] 4-bit codes (even column in the low nibble)."""
    c = np.asarray(c, np.uint8)
    out = np.empty((c.shape[0], c.shape[1] * 2), np.uint8)
    out[:, 0::2] = c & 0x0F
    out[:, 1::2] = c >> 4
    return out


def _std_scales_numpy(y, S_enc):
    """Scale bytes of the standard association, evaluated with numpy's fp32
    arithmetic and the brute-force E4M3 encoder (no oracle code)."""
    b = np.abs(y.reshape(y.shape[0], -1, 16)).max(axis=2).astype(f32)
    k6 = f32(S_enc) * f32(1.0 / 6.0)              # S_enc * (1/6), the fp32 constant
    s = (b * k6).astype(f32)
    return brute_e4m3(np.minimum(s, f32(448.0))).reshape(b.shape)


@pytest.mark.parametrize("gmode", ["none", "tensor"])
def test_std_association_scales_match_numpy_fp32(gmode):
    rng = np.random.default_rng(41)
    y = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-6, 6, (64, 1)))).astype(f32)
    if gmode == "none":
        r = oracle.quantize(y, rounding=oracle.RTN_STD)
        S_enc = 1.0
    else:
        A = np.abs(y).max().astype(f32)
        r = oracle.quantize(y, rounding=oracle.RTN_STD, gamax_mode=oracle.GAMAX_TENSOR_GIVEN,
                            gamax=np.array([A], f32), scale_bound=448.0)
        S_enc = np.minimum(f32(6.0) * f32(448.0) / A, np.finfo(f32).max)   # the page's global scale
    assert np.array_equal(r["scales"], _std_scales_numpy(y, S_enc))


@pytest.mark.parametrize("gmode", ["none", "tensor"])
def test_std_association_differs_from_four_over_six_on_a_fraction_of_blocks(gmode):
    # the page: the two associations round differently "on a fraction of
    # blocks" -- blocks whose scale lands next to an E4M3 rounding midpoint.
    # Block maxima b sweep +-40 fp32 steps around each midpoint's preimage.
    tab = torch_e4m3_table()[8:0x7F]              # normal E4M3 values
    mids = ((tab[:-1] + tab[1:]) / 2).astype(f32)
    if gmode == "none":
        S_enc, kw = f32(1.0), {}
    else:
        A, bound = f32(10.0), f32(256.0)
        S_enc = f32(6.0) * bound / A
        kw = dict(gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=np.array([A], f32), scale_bound=256.0)
    bs = []
    for mid in mids:
        b0 = f32(mid * f32(6.0) / S_enc)
        up = dn = b0
        bs.append(b0)
        for _ in range(40):
            up, dn = np.nextafter(up, f32(np.inf)), np.nextafter(dn, f32(-np.inf))
            bs += [up, dn]
    bs = np.array(bs, f32)
    bs = bs[: len(bs) // 4 * 4]
    y = (bs[:, None] * np.linspace(1.0, 0.25, 16, dtype=f32)[None, :]).astype(f32).reshape(-1, 64)
    std = oracle.quantize(y, rounding=oracle.RTN_STD, **kw)
    own = oracle.quantize(y, rounding=oracle.RTN, **kw)
    diff = std["scales"] != own["scales"]
    assert 0 < diff.mean() < 0.1
    assert np.array_equal(std["scales"], _std_scales_numpy(y, S_enc))
    # where the scales agree the element path is the same nearest rounding
    same = np.repeat(~diff, 16, axis=1)
    assert np.array_equal(_unpack_codes(std["codes"])[same], _unpack_codes(own["codes"])[same])


# ---- stochastic rounding of the columnwise output, keyed on the element in x -------------
def test_sr_columnwise_16x16_is_the_transpose_of_rowwise():
    # 16x16 blocks and draws keyed on x's index: Q(x^T) = Q(x)^T ("Stable FP4
    # Training via Transposition-Invariant Block Quantization", abstract)
    x = W.matrix((64, 96), seed=47, outlier_frac=0.02, outlier_factor=30.0)
    r = oracle.quantize(x, block=oracle.BLOCK_16X16, rounding=oracle.SR, seed=9, step=4, colwise=True)
    assert np.array_equal(_unpack_codes(r["codes_col"]), _unpack_codes(r["codes"]).T)
    tiles = r["scales"][::16, :]                  # one byte per tile, repeated on its 16 rows
    assert np.array_equal(r["scales_col"][::16, :], tiles.T)


def test_sr_columnwise_1x16_draws_use_the_x_index():
    x = W.matrix((32, 48), seed=53)
    seed, step, row_offset = 5, 11, 64
    r = oracle.quantize(x, rounding=oracle.SR, seed=seed, step=step, row_offset=row_offset, colwise=True)
    codes_col = _unpack_codes(r["codes_col"])     # [K, M]
    M, K = x.shape
    for c in (0, 17, 47):
        for blk in range(M // 16):
            rows = np.arange(16 * blk, 16 * blk + 16)
            d = float(np.asarray(oracle.e4m3_decode(np.array([r["scales_col"][c, blk]], np.uint8))).ravel()[0])
            v = (x[rows, c] / f32(d)).astype(f32)
            u = oracle.sr_uniform(seed, step, (row_offset + rows) * K + c)
            assert np.array_equal(codes_col[c, rows], oracle.e2m1_encode_sr(v, u))


def test_sr_columnwise_row_shard_is_a_column_slice():
    x = W.matrix((64, 32), seed=59)
    whole = oracle.quantize(x, rounding=oracle.SR, seed=3, step=2, colwise=True)
    part = oracle.quantize(np.ascontiguousarray(x[32:]), rounding=oracle.SR, seed=3, step=2, row_offset=32,
                           colwise=True)
    assert np.array_equal(part["codes_col"], whole["codes_col"][:, 16:])
    assert np.array_equal(part["scales_col"], whole["scales_col"][:, 2:])


# ---- scale layout for the block-scaled matrix multiply -------------------------------------
@pytest.mark.parametrize("rows,cols", [(128, 4), (256, 12), (300, 7), (1, 1), (129, 5)])
def test_scales_to_mma_is_the_blocked_permutation(rows, cols):
    # the layout as a reshape of the zero-padded matrix: [R/128, 4, 32, C/4, 4]
    # (row = 128 a + 32 b + r32, col = 4 t + j) stored as [a, t, r32, b, j]
    rng = np.random.default_rng(rows * 7 + cols)
    s = rng.integers(0, 127, (rows, cols), dtype=np.uint8)
    R, C = -(-rows // 128) * 128, -(-cols // 4) * 4
    pad = np.zeros((R, C), np.uint8)
    pad[:rows, :cols] = s
    want = pad.reshape(R // 128, 4, 32, C // 4, 4).transpose(0, 3, 2, 1, 4).ravel()
    got = oracle.scales_to_mma(s)
    assert np.array_equal(got, want)
    # a bijection of the padded matrix: every byte lands once
    idx = np.arange(R * C, dtype=np.int64).reshape(R, C)
    assert np.array_equal(np.sort(idx.reshape(R // 128, 4, 32, C // 4, 4).transpose(0, 3, 2, 1, 4).ravel()),
                          np.arange(R * C))


def test_four_over_six_encode_is_the_clamped_reciprocal_multiply():
    """[4o6 PR, What + Design]: a candidate encodes each element as y times
    min(1/(d * S_dec), FLT_MAX), rounded to the nearest e2m1 value.  Two kinds
    of blocks take the candidate decision out of the picture, so their codes
    follow from that formula alone (brute-force e2m1 rounding):
    - blocks whose amax is 2x a given global amax A: both candidates' scales
      cap at 448, one scale byte 0x7E; the other elements sit at and next to
      the e2m1 midpoints times the decode scale, where a multiply by the
      rounded reciprocal and a true division round to different codes;
    - blocks far below A: both scales encode to 0, and the FLT_MAX clamp
      keeps zeros at code 0 (0 * inf would be NaN, code 7) while every other
      value saturates."""
    FLT_MAX = np.finfo(np.float32).max
    differ = 0
    for bound in (256.0, 448.0):
        for A in (f32(0.37), f32(3.1), f32(1e-3)):
            Senc, Sdec = oracle.global_scales(float(A), bound)
            D = f32(f32(448.0) * f32(Sdec))
            enc = np.minimum(f32(1.0) / D, FLT_MAX)
            ys = []
            for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
                y = f32(f32(m) * D)
                for _ in range(4):
                    y = np.nextafter(y, f32(0))
                for _ in range(9):
                    differ += int(brute_e2m1_rn(f32(y * enc))[0] != brute_e2m1_rn(f32(y / D))[0])
                    ys += [y, -y]
                    y = np.nextafter(y, f32(10))
            ys += [f32(0.0)] * (-len(ys) % 15)
            body = np.array(ys, np.float32).reshape(-1, 15)
            big = np.concatenate([np.full((body.shape[0], 1), f32(2.0) * A, np.float32), body], axis=1)
            tiny = np.zeros((2, 16), np.float32)
            tiny[0, :4] = [1e-30, 0.0, -0.0, -3e-31]
            tiny[1, 7] = np.float32(-0.0)
            x = np.concatenate([big, tiny]).reshape(1, -1)      # the blocks along one row
            for err in (oracle.ERR_MAE, oracle.ERR_MSE):
                r = oracle.quantize(x, gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=np.array([A]),
                                    err_mode=err, scale_bound=bound)
                blocks = x.reshape(-1, 16)
                sc = r["scales"].reshape(-1)
                codes = np.stack([(r["codes"] & 0xF), (r["codes"] >> 4)], -1).reshape(-1, 16)
                nb = big.shape[0]
                assert np.all(sc[:nb] == 0x7E) and np.all(sc[nb:] == 0)
                assert np.array_equal(codes[:nb], brute_e2m1_rn(f32(blocks[:nb] * enc)).reshape(-1, 16))
                assert np.array_equal(codes[nb:], brute_e2m1_rn(f32(blocks[nb:] * FLT_MAX)).reshape(-1, 16))
                assert codes[nb, 1] == 0 and codes[nb, 2] == 8       # +0 and -0 keep their codes
    assert differ > 0       # the set holds cases a true division would round otherwise


def _near_midpoints(D, reach=4):
    """Values at and next to the e2m1 midpoints times D (both signs), and how
    many of them a division by D and a multiply by RN(1/D) round to
    different codes."""
    ys, differ = [], 0
    r = f32(1.0) / D
    for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
        y = f32(f32(m) * D)
        for _ in range(reach):
            y = np.nextafter(y, f32(0))
        for _ in range(2 * reach + 1):
            differ += int(brute_e2m1_rn(f32(y / D))[0] != brute_e2m1_rn(f32(y * r))[0])
            ys += [y, -y]
            y = np.nextafter(y, f32(10))
    return ys, differ


def test_plain_encode_divides_by_the_decoded_scale():
    """[fp4-train, Method]: every element is divided by the decoded scale and
    rounded to the grid.  A block led by 6d (d an E4M3 value) has scale d
    exactly; its other elements sit at and next to the e2m1 midpoints times d,
    where the division and a multiply by the rounded reciprocal round to
    different codes.  With a global scale the divisor is d * S_dec (d capped
    at 448 by a block amax at the global amax)."""
    tab = torch_e4m3_table()
    differ = 0
    blocks, expect_codes, expect_scales = [], [], []
    for code in (0x39, 0x3B, 0x3D, 0x3F, 0x4B, 0x2D, 0x55, 0x1F):      # significands 9/8 .. 15/8
        d = f32(tab[code])
        ys, n = _near_midpoints(d)
        differ += n
        ys += [f32(0.0)] * (-len(ys) % 15)
        for chunk in np.array(ys, np.float32).reshape(-1, 15):
            blk = np.concatenate([[f32(6.0) * d], chunk]).astype(np.float32)
            blocks.append(blk)
            expect_codes.append(brute_e2m1_rn(f32(blk / d)))
            expect_scales.append(code)
    x = np.array(blocks, np.float32).reshape(1, -1)
    r = oracle.quantize(x)
    codes = np.stack([(r["codes"] & 0xF), (r["codes"] >> 4)], -1).reshape(-1)
    assert np.array_equal(r["scales"].reshape(-1), np.array(expect_scales, np.uint8))
    assert np.array_equal(codes, np.concatenate(expect_codes))
    # with a given global amax A: the block amax A caps d at 448, the divisor is RN(448 * S_dec)
    gdiffer = 0
    for A in (f32(0.37), f32(3.1), f32(1e-3), f32(77.7), f32(0.0123)):
        Senc, Sdec = oracle.global_scales(float(A), 448.0)
        D = f32(f32(448.0) * f32(Sdec))
        gdiffer += int(D != f32(f32(448.0) / f32(Senc)))
        ys, n = _near_midpoints(D)
        differ += n
        ys += [f32(0.0)] * (-len(ys) % 15)
        blk = np.concatenate([np.full((len(ys) // 15, 1), A, np.float32),
                              np.array(ys, np.float32).reshape(-1, 15)], axis=1)
        r = oracle.quantize(blk.reshape(1, -1), gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=np.array([A]))
        codes = np.stack([(r["codes"] & 0xF), (r["codes"] >> 4)], -1).reshape(-1)
        assert np.all(r["scales"] == 0x7E)
        assert np.array_equal(codes, brute_e2m1_rn(f32(blk.reshape(-1) / D)))
    assert differ > 0 and gdiffer > 0     # the sets hold cases the other forms would round otherwise


def test_tensor_amax_under_error_feedback_is_over_x_plus_r():
    """[fp4-train, Method] with the per-tensor scale of the four-over-six page:
    under error feedback the quantized value is x + r, so its amax is
    max |fp32(x + r)|, not max |x|."""
    rng = np.random.default_rng(81)
    x = rng.standard_normal((8, 64)).astype(np.float32)
    res = np.zeros_like(x)
    res[3, 5] = f32(np.abs(x).max() * 2.0)                  # x + r peaks where x does not
    expect = f32(np.max(np.abs(f32(x + res))))
    assert expect != f32(np.max(np.abs(x)))
    for err, rnd in ((oracle.ERR_NONE, oracle.RTN), (oracle.ERR_NONE, oracle.SR)):
        r = oracle.quantize(x, residual=res.copy(), rounding=rnd, gamax_mode=oracle.GAMAX_TENSOR, err_mode=err)
        assert r["gamax"][0] == expect
    # and per row: row 3's amax is the residual's peak
    rows = np.max(np.abs(f32(x + res)), axis=1).astype(np.float32)
    assert rows[3] != f32(np.max(np.abs(x[3])))
    r = oracle.quantize(x, residual=res.copy(), gamax_mode=oracle.GAMAX_ROW)
    assert np.array_equal(r["gamax"], rows)


def test_qdq_is_quantize_then_dequantize():
    """[fp4-train, API: qdq quantizes then dequantizes]: qdq's bf16 output is the
    dequantize (to bf16) of the quantize's codes and scales, with the same
    global amax, in every global-scale mode and with error feedback."""
    rng = np.random.default_rng(83)
    x = (rng.standard_t(3, (32, 64)) * 3.0).astype(np.float32)
    for kw in (dict(), dict(gamax_mode=oracle.GAMAX_TENSOR, err_mode=oracle.ERR_MAE),
               dict(gamax_mode=oracle.GAMAX_ROW, err_mode=oracle.ERR_MSE),
               dict(gamax_mode=oracle.GAMAX_TENSOR, rounding=oracle.SR, seed=4, step=2),
               dict(block=oracle.BLOCK_16X16, gamax_mode=oracle.GAMAX_TENSOR_GIVEN,
                    gamax=np.array([f32(40.0)]), err_mode=oracle.ERR_MAE)):
        q = oracle.quantize(x, **kw)
        o = oracle.qdq(x, **kw)
        bound = 256.0 if kw.get("err_mode", oracle.ERR_NONE) != oracle.ERR_NONE else 448.0
        gm = kw.get("gamax_mode", oracle.GAMAX_NONE)
        dq = oracle.dequantize(q["codes"], q["scales"], 32, 64, gamax_mode=gm,
                               gamax=None if gm == oracle.GAMAX_NONE else q["gamax"], scale_bound=bound)
        assert np.array_equal(o["codes"], q["codes"]) and np.array_equal(o["out"], dq)
    r0 = (rng.standard_normal((32, 64)) * 0.1).astype(np.float32)
    ra, rb = r0.copy(), r0.copy()
    q = oracle.quantize(x, residual=ra, rounding=oracle.SR, seed=1)
    o = oracle.qdq(x, residual=rb, rounding=oracle.SR, seed=1)
    assert np.array_equal(ra, rb)
    assert np.array_equal(o["out"], oracle.dequantize(q["codes"], q["scales"], 32, 64))


def test_row_given_amax_applies_row_by_row():
    """Per-row given amaxes [4o6 PR, What: per-row or per-tensor global scale]:
    row r of a row-given call equals that row quantized (and dequantized)
    alone with its own amax given per tensor (pinned above)."""
    rng = np.random.default_rng(82)
    x = rng.standard_normal((6, 64)).astype(np.float32)
    g = (np.abs(x).max(1) * np.array([1.0, 2.0, 0.5, 3.0, 1.0, 7.0])).astype(np.float32)
    for err in (oracle.ERR_NONE, oracle.ERR_MAE, oracle.ERR_MSE):
        r = oracle.quantize(x, gamax_mode=oracle.GAMAX_ROW_GIVEN, gamax=g, err_mode=err)
        for i in range(6):
            o = oracle.quantize(x[i:i + 1], gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=g[i:i + 1], err_mode=err)
            assert np.array_equal(r["codes"][i], o["codes"][0]) and np.array_equal(r["scales"][i], o["scales"][0])
        bound = 448.0 if err == oracle.ERR_NONE else 256.0
        dq = oracle.dequantize(r["codes"], r["scales"], 6, 64, gamax_mode=oracle.GAMAX_ROW_GIVEN, gamax=g,
                               scale_bound=bound, out_dtype=oracle.F32)
        for i in range(6):
            di = oracle.dequantize(r["codes"][i:i + 1], r["scales"][i:i + 1], 1, 64,
                                   gamax_mode=oracle.GAMAX_TENSOR_GIVEN, gamax=g[i:i + 1], scale_bound=bound,
                                   out_dtype=oracle.F32)
            assert np.array_equal(dq[i], di[0])


def test_amax_of_an_empty_tensor_is_plus_zero():
    """An empty tensor (M = 0 or K = 0) is a valid no-op whose per-tensor amax
    is +0: the identity of a maximum over non-negative magnitudes, which the
    global scale then treats as A = 0 (S_enc falls back to 1)."""
    for shape in ((0, 16), (4, 0), (0, 0)):
        x = np.zeros(shape, np.float32)
        a = oracle.amax(x)
        assert a[0] == 0.0 and not np.signbit(a[0])
        r = oracle.quantize(x, gamax_mode=oracle.GAMAX_TENSOR)
        assert r["gamax"][0] == 0.0 and not np.signbit(r["gamax"][0])
