"""The C ABI boundary, checked without a GPU.

The library is built here (nvcc cross-compiles sm_103a), loaded, and every
function include/nvfp4.h declares must be exported.  Argument checks run on
the host before any CUDA call, so calls with bad arguments can be made
without a device: each must return NVFP4_EINVAL with a message.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "nvfp4_block_quantization_quantize_gb300")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_quantization_quantize_gb300 import build, load_library
    build()
    return load_library()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(nvfp4_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"nvfp4_quantize", "nvfp4_dequantize", "nvfp4_qdq", "nvfp4_amax"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_abi_version(lib):
    assert lib.nvfp4_abi_version() == 100
    assert lib.nvfp4_last_error() == b""


def test_binding_names_match_the_abi():
    import nvfp4_block_quantization_quantize_gb300 as nv
    for n in ("nvfp4_quantize", "nvfp4_dequantize", "nvfp4_qdq", "nvfp4_amax", "nvfp4_last_error"):
        assert callable(getattr(nv, n))


def test_missing_library_fails_loudly(tmp_path):
    from nvfp4_block_quantization_quantize_gb300 import load_library
    with pytest.raises(RuntimeError, match="missing"):
        load_library(str(tmp_path / "nope.so"))


# A fake aligned device address: validation rejects before it is ever used.
A16 = ctypes.c_void_p(0x10000)
A4 = ctypes.c_void_p(0x10004)


def q(lib, x=A16, M=64, K=64, dtype=0, block=0, rounding=0, residual=None, gm=0, gamax=None,
      err=0, bound=448.0, codes=A16, scales=A16, ccol=None, scol=None):
    return lib.nvfp4_quantize(x, M, K, dtype, block, rounding, residual, 0, 0, 0, gm, gamax, err,
                              bound, codes, scales, ccol, scol, None)


BAD_QUANT = {
    "K not a multiple of 16": dict(K=40),
    "negative M": dict(M=-1),
    "bad dtype": dict(dtype=7),
    "bad block": dict(block=2),
    "bad rounding": dict(rounding=5),
    "bad rounding 3": dict(rounding=3),
    "bad gamax mode": dict(gm=9, gamax=A16),
    "bad err mode": dict(err=3, gm=1, gamax=A16),
    "bound zero": dict(bound=0.0),
    "bound above 448": dict(bound=449.0),
    "bound NaN": dict(bound=float("nan")),
    "16x16 with M % 16": dict(block=1, M=40),
    "columnwise with M % 16": dict(M=40, ccol=A16, scol=A16),
    "only codes_col": dict(ccol=A16),
    "row gamax with 16x16": dict(block=1, gm=2, gamax=A16),
    "row gamax with columnwise": dict(gm=4, gamax=A16, ccol=A16, scol=A16),
    "4o6 with SR": dict(err=1, rounding=1, gm=1, gamax=A16, bound=256.0),
    "4o6 with standard association": dict(err=1, rounding=2, gm=1, gamax=A16, bound=256.0),
    "4o6 with residual": dict(err=2, residual=A16, gm=1, gamax=A16, bound=256.0),
    "4o6 without global amax": dict(err=1, bound=256.0),
    "4o6 bound 300": dict(err=1, gm=1, gamax=A16, bound=300.0),
    "columnwise with residual": dict(residual=A16, ccol=A16, scol=A16),
    "columnwise with K past the grid": dict(K=65535 * 256 + 16, ccol=A16, scol=A16),
    "x NULL": dict(x=None),
    "codes NULL": dict(codes=None),
    "scales NULL": dict(scales=None),
    "gamax NULL": dict(gm=1, gamax=None),
    "x misaligned": dict(x=ctypes.c_void_p(0x10008)),
    "codes misaligned": dict(codes=ctypes.c_void_p(0x10001)),
    "residual misaligned": dict(residual=ctypes.c_void_p(0x10004)),
    "gamax misaligned": dict(gm=3, gamax=ctypes.c_void_p(0x10002)),
}


@pytest.mark.parametrize("case", sorted(BAD_QUANT))
def test_quantize_rejects(lib, case):
    assert q(lib, **BAD_QUANT[case]) == 1
    assert lib.nvfp4_last_error() != b""


def test_gamax_needs_only_4_byte_alignment(lib):
    # everything else invalid (K=40) so no launch happens; the message names K
    assert q(lib, K=40, gm=3, gamax=A4) == 1
    assert b"K" in lib.nvfp4_last_error()


def test_qdq_rejects(lib):
    f = lib.nvfp4_qdq
    assert f(A16, 64, 64, 0, 0, 0, None, 0, 0, 0, 0, None, 0, 448.0, None, None, None, None) == 1
    assert f(A16, 64, 40, 0, 0, 0, None, 0, 0, 0, 0, None, 0, 448.0, None, None, A16, None) == 1
    assert f(A16, 64, 64, 0, 0, 1, None, 0, 0, 0, 1, A16, 1, 256.0, None, None, A16, None) == 1


def test_dequantize_rejects(lib):
    f = lib.nvfp4_dequantize
    assert f(A16, A16, 64, 40, 0, None, 448.0, A16, 1, None) == 1
    assert f(A16, A16, 64, 64, 0, None, 448.0, A16, 5, None) == 1
    assert f(A16, A16, 64, 64, 3, None, 448.0, A16, 1, None) == 1
    assert f(None, A16, 64, 64, 0, None, 448.0, A16, 1, None) == 1
    assert f(A16, A16, 64, 64, 0, None, 0.0, A16, 1, None) == 1


def test_amax_rejects(lib):
    f = lib.nvfp4_amax
    assert f(A16, 64, 64, 0, None, 0, A16, None) == 1        # NONE is not an amax mode
    assert f(A16, 64, 64, 0, None, 3, A16, None) == 1        # nor is TENSOR_GIVEN
    assert f(None, 64, 64, 0, None, 1, A16, None) == 1
    assert f(A16, 64, 48, 2, None, 1, A16, None) == 1


def test_product_never_touches_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".cpp", ".h")):
            assert "nvfp4_block_quantization_quantize_gb300" not in open(
                os.path.join(ROOT, "oracle", f)).read()


def test_probe_e2m1_rejects(lib):
    f = lib.nvfp4_probe_e2m1
    f.argtypes = [ctypes.c_uint32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert f(0, -1, A16, None) == 1
    assert f(0, (1 << 32) + 1, A16, None) == 1
    assert f(5, 1 << 32, A16, None) == 1                               # runs past 2^32
    assert f(0, 16, None, None) == 1
    assert f(0, 16, ctypes.c_void_p(0x10002), None) == 1
    assert f(0, 0, None, None) == 0


def test_probe_sub_f16_rejects(lib):
    f = lib.nvfp4_probe_sub_f16
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    assert f(A16, A16, A16, -1, None) == 1
    assert f(None, A16, A16, 4, None) == 1
    assert f(A16, ctypes.c_void_p(0x10002), A16, 4, None) == 1          # misaligned
    assert f(None, None, None, 0, None) == 0


def test_scales_to_mma_rejects(lib):
    f = lib.nvfp4_scales_to_mma
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert f(A16, -1, 4, A16, None) == 1
    assert f(None, 128, 4, A16, None) == 1
    assert f(A16, 128, 4, None, None) == 1
    assert f(A16, 128, 4, ctypes.c_void_p(0x10002), None) == 1      # out needs 4-byte alignment
    assert f(None, 0, 4, None, None) == 0                              # empty: a no-op
