"""Device probes of the conversion instructions and the generator, run through
the library's own entry points (in-bounds inputs only).

- e2m1, every fp32 value: nvfp4_probe_e2m1 runs the kernels' element encode on
  all 2^32 bit patterns, compared with the oracle's encoder.
- e2m1: blocks [6.0, y1..y15] have scale exactly 1.0 (6/6), so the stored code
  of each y is the hardware's e2m1 rounding of y itself.  Every fp32 value with
  0.125 <= |y| <= 6 (all decision boundaries of the grid) is checked against
  the oracle's encoder, plus signed zeros, tiny values and subnormals.
- e4m3: blocks [b, 0 x 15] give scale E4M3(b / 6); b sweeps +-4096 ulps around
  6x every e4m3 midpoint, plus random values over the whole scale range.
- Philox: stochastic rounding at global indices whose counter uses all four
  words (row_offset beyond 2^32 blocks, steps beyond 2^32, a 64-bit seed).
- the mixed f16/f32 subtract of the certified four-over-six sums rounds once
  (nvfp4_probe_sub_f16 against IEEE fp32 subtraction).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_helpers import assert_same, quantize_both, to_dev, to_np

pytestmark = pytest.mark.gpu

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nv.build()
    nv.load_library()


def blocks_of(values, lead):
    n = (values.size + 14) // 15
    v = np.zeros(n * 15, np.float32)
    v[:values.size] = values
    x = np.empty((n, 16), np.float32)
    x[:, 0] = lead
    x[:, 1:] = v.reshape(n, 15)
    return x, values.size


def unpack_codes(codes):
    lo = codes & 0x0F
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def test_e2m1_conversion_exhaustive_window():
    lo = np.array([0.125], np.float32).view(np.uint32)[0]
    hi = np.array([6.0], np.float32).view(np.uint32)[0]
    pos = np.arange(lo, hi + 1, dtype=np.uint32).view(np.float32)
    extra = np.array([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -149, -(2.0 ** -149), 2.0 ** -126,
                      0.0625, -0.0625], np.float32)
    for vals in (pos, -pos, extra):
        x, n = blocks_of(vals, 6.0)
        r = nv.nvfp4_quantize(to_dev(x))
        torch.cuda.synchronize()
        assert np.all(to_np(r["scales"]) == 0x38)
        got = unpack_codes(to_np(r["codes"]))[:, 1:].reshape(-1)[:n]
        assert_same(got, oracle.e2m1_encode_rn(vals), "e2m1 codes")


def test_e2m1_conversion_every_fp32_value():
    """All 2^32 fp32 bit patterns through the device's element encode (the
    routine every quantize kernel uses) against the oracle's nearest-grid
    encoder, in chunks of 2^28: signs, zeros, subnormals, every decision
    boundary, the saturating range (6, inf], infinities and every NaN."""
    chunk = 1 << 28
    with oracle.using_threads(0):
        for first in range(0, 1 << 32, chunk):
            got = to_np(nv.nvfp4_probe_e2m1(first, chunk))
            c = oracle.e2m1_encode_rn_bits(first, chunk)
            want = (c[0::2] | (c[1::2] << 4)).astype(np.uint8)
            if not np.array_equal(got, want):
                bad = np.flatnonzero(got != want)[:4]
                pats = [hex(first + 2 * int(b)) for b in bad]
                raise AssertionError(f"e2m1 codes differ near patterns {pats}: gpu {got[bad]} oracle {want[bad]}")
            del got, c, want


def test_e2m1_probe_ragged_tail():
    first = int(np.array([1.1], np.float32).view(np.uint32)[0])
    for n in (1, 7, 9, 4099):
        got = to_np(nv.nvfp4_probe_e2m1(first, n))
        c = np.zeros(n + (n & 1), np.uint8)
        c[:n] = oracle.e2m1_encode_rn_bits(first, n)
        assert_same(got, (c[0::2] | (c[1::2] << 4)).astype(np.uint8), f"tail n={n}")


def test_e4m3_conversion_near_midpoints():
    tab = oracle.e4m3_decode(np.arange(0x7F)).astype(np.float64)
    mids = ((tab[:-1] + tab[1:]) / 2 * 6).astype(np.float32)
    b = np.concatenate([
        (mids.view(np.uint32)[:, None].astype(np.int64) + np.arange(-4096, 4097)[None, :])
        .astype(np.uint32).reshape(-1).view(np.float32),
        np.exp2(np.random.default_rng(1).uniform(-12, 12, 2_000_000)).astype(np.float32),
        np.array([6 * 448.0, 6 * 464.0, 1e30, 2.0 ** -130], np.float32)])
    b = b[b > 0]
    x = np.zeros((b.size, 16), np.float32)
    x[:, 0] = b
    r = nv.nvfp4_quantize(to_dev(x))
    torch.cuda.synchronize()
    expect = oracle.e4m3_encode(np.minimum(b / np.float32(6.0), np.float32(448.0)))
    assert_same(to_np(r["scales"])[:, 0], expect, "e4m3 scales")


@pytest.mark.parametrize("block", ["1x16", "16x16"])
def test_philox_all_counter_words(block):
    x = np.full((32, 64), 2.3, np.float32)
    x[:, ::16] = 6.0
    for seed, step, row_offset in ((0xFEDCBA9876543210, 0, 0), (3, (1 << 32) + 5, 0),
                                   (3, 7, (1 << 34) // 64 * 16), (2**64 - 1, 2**64 - 1, 1 << 40)):
        gpu, o = quantize_both(x, block=block, rounding="sr", seed=seed, step=step,
                               row_offset=row_offset)
        assert_same(gpu["codes"], o["codes"], f"sr codes seed={seed} step={step}")


def test_exact_division_routine_exhaustive_mantissas():
    """The plain path divides each element by the decoded scale with a
    reciprocal-and-correction sequence; it must equal IEEE division.  Every fp32
    mantissa of the dividend against every E4M3 divisor mantissa (x 3 divisor
    exponents, 2 dividend exponents), plus divisor 6 (the b / 6 step), plus
    random dividend / divisor pairs across the guarded range and beyond it."""
    mant = (np.arange(1 << 23, dtype=np.uint32) | np.uint32(0x3F800000)).view(np.float32)
    divisors = [np.float32((1 + k / 8) * 2.0 ** e) for k in range(8) for e in (-9, -6, 0, 8)]
    divisors += [np.float32(6.0)]
    for dv in divisors:
        for scale in (np.float32(1.0), np.float32(-2.0 ** -7)):
            a = mant * scale
            b = np.full(a.shape, dv, np.float32)
            got = to_np(nv.nvfp4_probe_divide(to_dev(a), to_dev(b)))
            assert_same(got, a / b, f"divisor {dv} scale {scale}")
    rng = np.random.default_rng(17)
    n = 4_000_000
    a = (rng.standard_normal(n) * np.exp2(rng.uniform(-90, 70, n))).astype(np.float32)
    b = np.exp2(rng.uniform(-30, 30, n)).astype(np.float32) * rng.uniform(1, 2, n).astype(np.float32)
    a[:1000] = np.float32(0.0)
    a[1000:2000] = np.float32(-0.0)
    got = to_np(nv.nvfp4_probe_divide(to_dev(a), to_dev(b)))
    assert_same(got, a / b, "random pairs")


def test_mixed_f16_subtract_rounds_once():
    """The certified four-over-six sums take each element's scaled error as
    RN(q - v), q a grid value held in f16 and v fp32, from one mixed-precision
    subtract; their rounding bound assumes q is taken exactly and the
    difference rounded once to fp32 — the IEEE fp32 subtraction of q and v."""
    rng = np.random.default_rng(93)
    n = 1 << 16
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    q = grid[rng.integers(0, 8, 2 * n)] * rng.choice(np.array([-1, 1], np.float32), 2 * n)
    kind = rng.integers(0, 5, 2 * n)
    v = np.empty(2 * n, np.float32)
    near = q * (1 + rng.standard_normal(2 * n).astype(np.float32) * np.float32(1e-3))
    v[kind == 0] = near[kind == 0]
    v[kind == 1] = (rng.standard_normal(2 * n) * 3).astype(np.float32)[kind == 1]
    v[kind == 2] = (rng.standard_normal(2 * n) * 1e-30).astype(np.float32)[kind == 2]
    v[kind == 3] = (rng.standard_normal(2 * n) * 1e30).astype(np.float32)[kind == 3]
    v[kind == 4] = np.nextafter(q, np.float32(np.inf))[kind == 4]
    h = q.astype(np.float16).view(np.uint16).astype(np.uint32)
    words = (h[0::2] | (h[1::2] << 16)).view(np.int32)
    got = to_np(nv.nvfp4_probe_sub_f16(torch.from_numpy(words.copy()).cuda(), to_dev(v)))
    with np.errstate(over="ignore"):
        want = (q - v).astype(np.float32)
    assert_same(got, want, "q - v")
