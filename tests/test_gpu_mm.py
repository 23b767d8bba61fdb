"""The block-scaled FP4 tensor-core product (nvfp4_mm) against its plain
definition (oracle.mm_reference: the product of the dequantized operands in
float64).

With unit scales and small grid values every partial sum is a multiple of 1/4
below 2^22, so any fp32 accumulation order is exact and the result must equal
the reference bit for bit; with real scales the products are still exact in
fp32 and only the accumulation of K terms can round, which bounds the error
by K * 2^-23 * (|A| |B|^T).
"""
import numpy as np
import pytest
import torch

import nvfp4_workloads as W
import oracle
from parity_helpers import to_dev, to_np

pytestmark = pytest.mark.gpu

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nv.build()
    nv.load_library()


def _mm_both(ca, sa, cb, sb, M, N, K, ga=None, gb=None, out_dtype="f32"):
    y = nv.nvfp4_mm(to_dev(ca), nv.nvfp4_scales_to_mma(to_dev(sa)), to_dev(cb), nv.nvfp4_scales_to_mma(to_dev(sb)),
                    M, N, K, gamax_a=None if ga is None else to_dev(ga), gamax_b=None if gb is None else to_dev(gb),
                    out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = oracle.mm_reference(ca, sa, cb, sb, M, N, K, gamax_a=ga, gamax_b=gb)
    return to_np(y.float()).astype(np.float64), ref


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (128, 256, 192), (256, 128, 512)])
def test_mm_unit_scales_exact(M, N, K):
    rng = np.random.default_rng(M + N + K)
    ca = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = np.full((M, K // 16), 0x38, np.uint8)        # E4M3 1.0
    sb = np.full((N, K // 16), 0x38, np.uint8)
    y, ref = _mm_both(ca, sa, cb, sb, M, N, K)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (256, 384, 1024)])
def test_mm_scales_exact_per_block(M, N, K):
    # one scale per block row, powers of two: still exact in any order
    rng = np.random.default_rng(3 * M + N)
    ca = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = (0x38 + 8 * rng.integers(-2, 3, (M, K // 16))).astype(np.uint8)      # 2^-2 .. 2^2
    sb = (0x38 + 8 * rng.integers(-2, 3, (N, K // 16))).astype(np.uint8)
    y, ref = _mm_both(ca, sa, cb, sb, M, N, K)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("gm", ["none", "tensor"])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_mm_quantized_operands(gm, out_dtype):
    M, N, K = 256, 384, 1024
    a = W.matrix((M, K), seed=83, dtype="bf16", dist="t")
    b = W.matrix((N, K), seed=89, dtype="bf16")
    qa = nv.nvfp4_quantize(to_dev(a), gamax_mode=gm)
    qb = nv.nvfp4_quantize(to_dev(b), gamax_mode=gm)
    ga = None if gm == "none" else to_np(qa["gamax"])
    gb = None if gm == "none" else to_np(qb["gamax"])
    y, ref = _mm_both(to_np(qa["codes"]), to_np(qa["scales"]), to_np(qb["codes"]), to_np(qb["scales"]), M, N, K,
                      ga, gb, out_dtype)
    da = oracle.dequantize(to_np(qa["codes"]), to_np(qa["scales"]), M, K, out_dtype=oracle.F32).astype(np.float64)
    db = oracle.dequantize(to_np(qb["codes"]), to_np(qb["scales"]), N, K, out_dtype=oracle.F32).astype(np.float64)
    scale = abs(ref).max() / max(abs(da @ db.T).max(), 1e-300)
    bound = (np.abs(da) @ np.abs(db).T) * scale * K * 2.0 ** -23
    if out_dtype == "bf16":
        bound = bound + np.abs(ref) * 2.0 ** -8
    err = np.abs(y - ref)
    assert (err <= bound + 1e-30).all(), f"max err {err.max()}"


def test_mm_matches_library_gemm():
    from nvfp4_block_quantization_quantize_gb300.consumers import fp4_mm, to_fp4_operands
    M, N, K = 256, 256, 2048
    a = to_dev(W.matrix((M, K), seed=97, dtype="bf16"))
    b = to_dev(W.matrix((N, K), seed=101, dtype="bf16"))
    qa, qb = nv.nvfp4_quantize(a), nv.nvfp4_quantize(b)
    ours = nv.nvfp4_mm(qa["codes"], nv.nvfp4_scales_to_mma(qa["scales"]), qb["codes"],
                       nv.nvfp4_scales_to_mma(qb["scales"]), M, N, K, out_dtype="f32")
    try:
        lib = fp4_mm(to_fp4_operands(qa), to_fp4_operands(qb), out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError, AttributeError) as e:
        pytest.skip(f"no library block-scaled FP4 GEMM: {e}")
    torch.cuda.synchronize()
    rel = float(((ours - lib).abs().max() / lib.abs().max()).item())
    assert rel < 1e-5


def test_mm_rejects_bad_shapes():
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_mm(z, z, z, z, 100, 128, 64)
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_mm(z, z, z, z, 128, 128, 48)


@pytest.mark.parametrize("stochastic", [False, True])
def test_fp4_linear_forward_and_straight_through_backward(stochastic):
    """fp4_linear's output is the product of the two operands' quantizations
    (each the oracle's, rows padded to the tensor cores' 128 with zeros),
    within the fp32 accumulation bound; its gradients are the straight-through
    ones, dL/dx = g Q(w) and dL/dw = g^T Q(x)."""
    from nvfp4_block_quantization_quantize_gb300.consumers import fp4_linear
    M, N, K = 200, 136, 512                       # neither multiple of 128: padded
    x = W.matrix((M, K), seed=131, dtype="bf16", dist="t")
    w = W.matrix((N, K), seed=137, dtype="bf16")
    xd, wd = to_dev(x).requires_grad_(True), to_dev(w).requires_grad_(True)
    y = fp4_linear(xd, wd, stochastic=stochastic, seed=5, step=3)
    rnd = oracle.SR if stochastic else oracle.RTN
    ox = oracle.quantize(x, rounding=rnd, seed=5, step=3)
    ow = oracle.quantize(w, rounding=rnd, seed=6, step=3)
    dx = oracle.dequantize(ox["codes"], ox["scales"], M, K, out_dtype=oracle.F32).astype(np.float64)
    dw = oracle.dequantize(ow["codes"], ow["scales"], N, K, out_dtype=oracle.F32).astype(np.float64)
    ref = dx @ dw.T
    got = to_np(y.float()).astype(np.float64)
    bound = (np.abs(dx) @ np.abs(dw).T) * K * 2.0 ** -23 + np.abs(ref) * 2.0 ** -8   # bf16 output
    assert (np.abs(got - ref) <= bound + 1e-30).all()
    g = torch.from_numpy(np.random.default_rng(7).standard_normal((M, N)).astype(np.float32)).cuda()
    y.backward(g.to(y.dtype))
    gx_ref = g.double().cpu().numpy() @ dw
    gw_ref = g.double().cpu().numpy().T @ dx
    gx = xd.grad.float().cpu().numpy().astype(np.float64)
    gw = wd.grad.float().cpu().numpy().astype(np.float64)
    gy = np.abs(to_np(g.to(y.dtype).float()).astype(np.float64))
    assert (np.abs(gx - gx_ref) <= (gy @ np.abs(dw)) * (N * 2.0 ** -20 + 2.0 ** -7) + 1e-30).all()
    assert (np.abs(gw - gw_ref) <= (gy.T @ np.abs(dx)) * (M * 2.0 ** -20 + 2.0 ** -7) + 1e-30).all()


def test_fp4_linear_rejects_bad_shapes():
    from nvfp4_block_quantization_quantize_gb300.consumers import fp4_linear
    with pytest.raises(ValueError):
        fp4_linear(torch.zeros(128, 48, device="cuda"), torch.zeros(128, 48, device="cuda"))


def test_fp4_matmul_portable_path():
    """fp4_matmul (dequantize, then the product): with operands on the e2m1
    grid and a 6 in every 16-element block (every scale 1, so the oracle's
    dequantized operands are the inputs) every fp32 partial sum is exact, and
    the result is the exact product rounded once to bf16, bit for bit equal
    to the tensor-core product (nvfp4_mm, bf16 out) on the same codes; with
    stochastic rounding of normal operands it is the product of the oracle's
    dequantized operands within one bf16 rounding and the fp32 accumulation
    bound."""
    from nvfp4_block_quantization_quantize_gb300.consumers import fp4_matmul
    rng = np.random.default_rng(31)
    M, N, K = 256, 384, 512
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)

    def on_grid(rows):
        v = grid[rng.integers(0, 8, (rows, K))] * rng.choice(np.array([-1, 1], np.float32), (rows, K))
        v[:, ::16] = 6.0
        return v

    a, b = on_grid(M), on_grid(N)
    y = fp4_matmul(to_dev(a), to_dev(b))
    qa, qb = nv.nvfp4_quantize(to_dev(a)), nv.nvfp4_quantize(to_dev(b))
    t = nv.nvfp4_mm(qa["codes"], nv.nvfp4_scales_to_mma(qa["scales"]), qb["codes"],
                    nv.nvfp4_scales_to_mma(qb["scales"]), M, N, K, out_dtype="bf16")
    torch.cuda.synchronize()
    oa, ob = oracle.quantize(a), oracle.quantize(b)
    da = oracle.dequantize(oa["codes"], oa["scales"], M, K, out_dtype=oracle.F32).astype(np.float64)
    db = oracle.dequantize(ob["codes"], ob["scales"], N, K, out_dtype=oracle.F32).astype(np.float64)
    exact = W.to_bf16_bits((da @ db.T).astype(np.float32))     # the float64 sums are exact, and so is the cast
    assert np.array_equal(to_np(y), exact)
    assert np.array_equal(to_np(t), exact)

    x = W.matrix((M, K), seed=141)
    w = W.matrix((N, K), seed=143, dist="t")
    y = fp4_matmul(to_dev(x), to_dev(w), stochastic=True, seed=3, step=2)
    torch.cuda.synchronize()
    ox = oracle.quantize(x, rounding=oracle.SR, seed=3, step=2)
    ow = oracle.quantize(w, rounding=oracle.SR, seed=4, step=2)
    dx = oracle.dequantize(ox["codes"], ox["scales"], M, K, out_dtype=oracle.F32).astype(np.float64)
    dw = oracle.dequantize(ow["codes"], ow["scales"], N, K, out_dtype=oracle.F32).astype(np.float64)
    ref = dx @ dw.T
    got = W.bf16_bits_to_f32(to_np(y)).astype(np.float64)
    bound = (np.abs(dx) @ np.abs(dw).T) * K * 2.0 ** -23 + np.abs(ref) * 2.0 ** -8
    assert (np.abs(got - ref) <= bound + 1e-30).all()
    with pytest.raises(ValueError):
        fp4_matmul(to_dev(x[:, :40]), to_dev(w[:, :40]))


def test_fp4_mm_and_operands_take_raw_tensors():
    """fp4_mm(a, b, stochastic, seed, step) on raw tensors quantizes them as
    to_fp4_operands does ((seed, step) for a, (seed + 1, step) for b) and
    gives the same product as on those operands; the codes are the oracle's."""
    from nvfp4_block_quantization_quantize_gb300.consumers import fp4_mm, to_fp4_operands
    M, N, K = 128, 256, 512
    a, b = W.matrix((M, K), seed=151, dtype="bf16"), W.matrix((N, K), seed=157, dtype="bf16")
    oa = to_fp4_operands(to_dev(a), stochastic=True, seed=8, step=1)
    assert np.array_equal(to_np(oa["fp4"].view(torch.uint8)),
                          oracle.quantize(a, rounding=oracle.SR, seed=8, step=1)["codes"])
    ob = to_fp4_operands(to_dev(b), stochastic=True, seed=9, step=1)
    try:
        y_ops = fp4_mm(oa, ob, out_dtype=torch.float32)
        y_raw = fp4_mm(to_dev(a), to_dev(b), stochastic=True, seed=8, step=1, out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError, AttributeError) as e:
        pytest.skip(f"no library block-scaled FP4 GEMM: {e}")
    torch.cuda.synchronize()
    assert torch.equal(y_ops, y_raw)
