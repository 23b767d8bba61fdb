"""The certified four-over-six error sums, checked on the CPU.

With a global scale the kernels first form approximate error sums in the
scaled domain: v = RN(y * enc) is the value the encode rounds to a grid
value q (signed like y), an element's approximate error is |RN(q - v)|
(squared for MSE), and the block's (or tile's) sum S' of those (1x16: two
interleaved chains, then their sum; tiles: column sums in row order, then
the width-16 tree) is scaled back by K (K^2 for MSE), K the error
value of grid value 1, ((1 * d) * A) / C: E^ = RN(K * S').  The comparison of
the two candidates' E^ is accepted only when it is separated by more than a
rounding bound; otherwise the kernels take the exact sums.  The outputs are
the method's as long as |E - E^| <= B for every candidate, E the method's
error sum ("Add NVFP4 four-over-six (row-wise) quantization to the training
prototype", Two load-bearing numeric details: error values ((q*d)*A)/C,
element-order sums, the width-16 tree).  This test computes both in IEEE
fp32 (numpy float32 arithmetic) on many blocks and tiles and checks the
per-candidate bounds the kernels' thresholds are built from (the threshold
is twice the two candidates' bounds together), b the block's amax.  A
16x16 tile's one approximate sum per candidate (x^T's order) is checked
against the exact sums in both orders, since both choices are taken from it:

  1x16 MAE  2^-18 E^ + 2^-16 K + 2^-17 b
  1x16 MSE  2^-17 K sqrt(E^) + 2^-18 b sqrt(E^) + 2^-18 E^
  tile MAE  2^-18 E^ + 2^-12 K + 2^-13 b
  tile MSE  2^-15 K sqrt(E^) + 2^-16 b sqrt(E^) + 2^-18 E^

each plus 2^-121 for subnormal results.
"""
import numpy as np
import pytest

import oracle

f32 = np.float32
FLT_MAX = f32(3.4028234663852886e38)


def _seq(e: np.ndarray) -> np.float32:
    s = f32(0.0)
    for v in e:
        s = f32(s + v)
    return s


def _pairs(d: np.ndarray, err: str) -> np.float32:
    """The 1x16 kernels' approximate sum: two chains over the even and the
    odd elements, then their sum; for MSE each square is fused into its
    chain's addition (emulated in fp64, whose d*d + S is exact or nearly so
    before the one rounding to fp32)."""
    s = [f32(0.0), f32(0.0)]
    for i, x in enumerate(d):
        if err == "mae":
            s[i & 1] = f32(s[i & 1] + abs(x))
        else:
            s[i & 1] = f32(np.float64(x) * np.float64(x) + np.float64(s[i & 1]))
    return f32(s[0] + s[1])


def _tree16(r) -> np.float32:
    a = [f32(r[i] + r[i + 8]) for i in range(8)]
    b = [f32(a[i] + a[i + 4]) for i in range(4)]
    c = [f32(b[i] + b[i + 2]) for i in range(2)]
    return f32(c[0] + c[1])


def _candidates(b, Senc):
    s6f = f32(f32(b / f32(6.0)) * Senc)
    sf6 = oracle.e4m3_encode(np.minimum(np.float32(s6f), f32(448.0)))
    sf4 = oracle.e4m3_encode(np.minimum(f32(s6f * f32(1.5)), f32(448.0)))
    return sf6, sf4


def _block_errors(y, sf, A, Sdec, C, err, signed=False):
    """Exact per-element errors of one candidate on the values y (any shape),
    the approximate ones in the scaled domain (signed: the differences q - v
    themselves), and K."""
    d = oracle.e4m3_decode(sf).astype(f32)
    with np.errstate(divide="ignore", over="ignore"):   # a zero scale: enc = FLT_MAX, the encode saturates
        enc = np.minimum(f32(f32(1.0) / f32(d * Sdec)), FLT_MAX)
        v = (y * enc).astype(f32)
    q = oracle.e2m1_value(oracle.e2m1_encode_rn(v)).astype(f32)
    dq = (((np.abs(q) * d).astype(f32) * A).astype(f32) / C).astype(f32)
    diff_t = (dq - np.abs(y)).astype(f32)
    K = f32(f32(f32(f32(1.0) * d) * A) / C)
    with np.errstate(over="ignore", invalid="ignore"):
        diff_a = (q - v).astype(f32)                              # one rounding, as the mixed subtract
    if signed:
        return (np.abs(diff_t) if err == "mae" else (diff_t * diff_t).astype(f32)), diff_a, K
    if err == "mae":
        return np.abs(diff_t), np.abs(diff_a), K
    with np.errstate(over="ignore"):                          # squares of huge differences: inf, exact path
        return (diff_t * diff_t).astype(f32), (diff_a * diff_a).astype(f32), K


def _scaled(Sp, K, err):
    """E^ from the scaled-domain sum: RN(K * S'), or RN(RN(K * K) * S')."""
    with np.errstate(over="ignore", invalid="ignore"):      # 0 * inf: a NaN the kernels fall back on
        return f32(K * Sp) if err == "mae" else f32(f32(K * K) * Sp)


def _bound(K, E, b, err, tile):
    K, E, b = float(K), float(E), float(b)
    if err == "mae":
        return 2.0 ** -18 * E + 2.0 ** (-12 if tile else -16) * K + 2.0 ** (-13 if tile else -17) * b + 2.0 ** -121
    r = np.sqrt(E)
    return (2.0 ** (-15 if tile else -17) * K * r + 2.0 ** (-16 if tile else -18) * b * r + 2.0 ** -18 * E
            + 2.0 ** -121)


def _inputs(rng, shape):
    n = int(np.prod(shape))
    yield "normal", rng.standard_normal(n).astype(f32).reshape(shape)
    t = rng.standard_t(3, n).astype(f32).reshape(shape)
    t.reshape(-1, shape[-1])[:, :2] *= 50.0                     # outlier columns
    yield "t3 outliers", t
    yield "quarter grid", (rng.integers(-6, 7, n) * 0.25).astype(f32).reshape(shape)
    small = (rng.standard_normal(n) * 1e-30).astype(f32).reshape(shape)
    yield "tiny", small
    mixed = rng.standard_normal(n).astype(f32) * np.exp2(rng.integers(-30, 30, n)).astype(f32)
    yield "wide exponents", mixed.reshape(shape)


@pytest.mark.parametrize("err", ["mae", "mse"])
@pytest.mark.parametrize("bound", [256.0, 448.0])
def test_certified_bound_1x16(err, bound):
    rng = np.random.default_rng(71)
    worst = 0.0
    for name, x in _inputs(rng, (96, 64)):
        A = f32(np.max(np.abs(x)))
        Senc, Sdec = oracle.global_scales(float(A), bound)
        C = f32(f32(6.0) * f32(bound))
        blocks = x.reshape(-1, 16)
        b = np.max(np.abs(blocks), axis=1).astype(f32)
        sf6, sf4 = _candidates(b, Senc)
        for i, y in enumerate(blocks):
            for sf in (sf6[i], sf4[i]):
                with np.errstate(over="ignore", invalid="ignore"):
                    et, da, K = _block_errors(y, np.uint8(sf), A, Sdec, C, err, signed=True)
                    E, Eh = _seq(et), _scaled(_pairs(da, err), K, err)
                if not (np.isfinite(E) and np.isfinite(Eh)):
                    continue                 # the kernels take the exact sums
                gap = abs(float(E) - float(Eh))
                B = _bound(K, Eh, b[i], err, tile=False)
                assert gap <= B, f"{name} block {i}: |E - E^| = {gap} > {B} (K {K}, E^ {Eh})"
                worst = max(worst, gap / B)
    print(err, bound, "worst |E - S| / B:", worst)
    assert 0.0 < worst <= 1.0                # the approximation is not exact everywhere


@pytest.mark.parametrize("err", ["mae", "mse"])
def test_certified_bound_tile(err):
    rng = np.random.default_rng(72)
    worst = 0.0
    for name, x in _inputs(rng, (64, 64)):
        A = f32(np.max(np.abs(x)))
        Senc, Sdec = oracle.global_scales(float(A), 256.0)
        C = f32(f32(6.0) * f32(256.0))
        for t0 in range(0, 64, 16):
            for c0 in range(0, 64, 16):
                y = x[t0:t0 + 16, c0:c0 + 16]
                b = np.array([np.max(np.abs(y))], f32)
                sf6, sf4 = _candidates(b, Senc)
                for sf in (sf6[0], sf4[0]):
                    et, ea, K = _block_errors(y, np.uint8(sf), A, Sdec, C, err)
                    # the kernel's one approximate sum per candidate, in x^T's
                    # order (column sums, then the tree), against the exact
                    # sums in both orders: the rowwise choice uses it too
                    Eh = _scaled(_tree16([_seq(r) for r in ea.T]), K, err)
                    for tr in (False, True):          # rowwise exact sums, then x^T's (columnwise)
                        E = _tree16([_seq(r) for r in (et.T if tr else et)])
                        if not (np.isfinite(E) and np.isfinite(Eh)):
                            continue
                        gap = abs(float(E) - float(Eh))
                        B = _bound(K, Eh, b[0], err, tile=True)
                        assert gap <= B, f"{name} tile ({t0},{c0}) {'col' if tr else 'row'}: {gap} > {B}"
                        worst = max(worst, gap / B)
    assert 0.0 < worst <= 1.0
