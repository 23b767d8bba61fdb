"""The matrix-multiply scale layout: the CUDA re-layout against the oracle,
bit for bit, and the quantized operands through a library block-scaled
matrix multiply against the product of the dequantized operands."""
import numpy as np
import pytest
import torch

import nvfp4_workloads as W
import oracle
from parity_helpers import assert_same, to_dev, to_np

pytestmark = pytest.mark.gpu

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nv.build()
    nv.load_library()


@pytest.mark.parametrize("rows,cols", [(128, 4), (256, 64), (300, 7), (1, 1), (4096, 896), (129, 5)])
def test_scales_to_mma_matches_oracle(rows, cols):
    s = np.random.default_rng(rows + cols).integers(0, 127, (rows, cols), dtype=np.uint8)
    got = to_np(nv.nvfp4_scales_to_mma(to_dev(s))).ravel()
    assert_same(got, oracle.scales_to_mma(s), "scales in the matrix-multiply layout")


def test_scales_to_mma_from_quantize():
    x = W.matrix((384, 1024), seed=71, dtype="bf16")
    q = nv.nvfp4_quantize(to_dev(x))
    got = to_np(nv.nvfp4_scales_to_mma(q["scales"])).ravel()
    assert_same(got, oracle.scales_to_mma(to_np(q["scales"])), "layout of quantizer scales")


@pytest.mark.parametrize("gm", ["none", "tensor"])
def test_fp4_mm_matches_dequantized_product(gm):
    from nvfp4_block_quantization_quantize_gb300.consumers import fp4_mm, to_fp4_operands
    M, N, K = 256, 384, 1024
    a = to_dev(W.matrix((M, K), seed=73, dtype="bf16"))
    b = to_dev(W.matrix((N, K), seed=79, dtype="bf16"))
    qa = nv.nvfp4_quantize(a, gamax_mode=gm)
    qb = nv.nvfp4_quantize(b, gamax_mode=gm)
    kw = dict(gamax_mode="tensor_given", gamax=qa["gamax"]) if gm == "tensor" else {}
    da = nv.nvfp4_dequantize(qa["codes"], qa["scales"], M, K, out_dtype="f32", **kw)
    kw = dict(gamax_mode="tensor_given", gamax=qb["gamax"]) if gm == "tensor" else {}
    db = nv.nvfp4_dequantize(qb["codes"], qb["scales"], N, K, out_dtype="f32", **kw)
    ref = (da.double() @ db.double().t())
    try:
        y = fp4_mm(to_fp4_operands(qa), to_fp4_operands(qb), out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError, TypeError, AttributeError) as e:
        pytest.skip(f"no block-scaled FP4 matrix multiply in this torch build: {e}")
    torch.cuda.synchronize()
    # every product of an e2m1 value and an E4M3 scale pair is exact in fp32; only
    # the order and precision of the K-term accumulation differ from the fp64 sum
    bound = (da.double().abs() @ db.double().abs().t()) * (K * 2.0 ** -23) + 1e-30
    err = (y.double() - ref).abs()
    assert bool((err <= bound).all()), f"max error {float(err.max())}, bound {float(bound.min())}"
