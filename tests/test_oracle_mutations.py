"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C++ source
(on the CPU), builds it, and runs the pin suite against that copy: the suite
has to fail.  The committed oracle is never modified.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nvfp4_oracle.cpp")

MUTATIONS = {
    "e2m1 ties round up": ("else pick = (k % 2 == 0) ? k : k + 1;", "else pick = k + 1;"),
    "e2m1 negative zero loses its sign": (
        "const uint8_t sign = std::signbit(v) ? 0x8 : 0x0;\n    const double a = std::fabs(static_cast<double>(v));\n    if (a >= 6.0) return static_cast<uint8_t>(sign | 7);\n    for (int k = 0; k < 7; ++k) {\n        if (a >= kGrid[k] && a < kGrid[k + 1]) {\n            const double twice",
        "const uint8_t sign = (v < 0.0f) ? 0x8 : 0x0;\n    const double a = std::fabs(static_cast<double>(v));\n    if (a >= 6.0) return static_cast<uint8_t>(sign | 7);\n    for (int k = 0; k < 7; ++k) {\n        if (a >= kGrid[k] && a < kGrid[k + 1]) {\n            const double twice"),
    "e4m3 ties round up": ("else pick = (c % 2 == 0) ? c : c + 1;", "else pick = c + 1;"),
    "scale uses a reciprocal multiply": ("return (b / 6.0f) * S_enc;", "return b * (1.0f / 6.0f) * S_enc;"),
    "map-to-4 expansion not 1.5": ("min_nd(s6f * 1.5f, 448.0f)", "min_nd(s6f * 1.25f, 448.0f)"),
    "ties pick map-to-4": ("(E[1] < E[0]) ? 1 : 0", "(E[1] <= E[0]) ? 1 : 0"),
    "error sum in reverse order": ("for (int t = 0; t < 16; ++t) E = E + e[t];",
                                   "for (int t = 15; t >= 0; --t) E = E + e[t];"),
    "16x16 rows summed sequentially": (
        "return (((R[0] + R[8]) + (R[4] + R[12])) + ((R[2] + R[10]) + (R[6] + R[14]))) +",
        "float S = 0.0f; for (int r = 0; r < 16; ++r) S = S + R[r]; return S; return (((R[0] + R[8]) + (R[4] + R[12])) + ((R[2] + R[10]) + (R[6] + R[14]))) +"),
    "block amax propagates NaN": ("float max_nd(float a, float b) { return std::fmax(a, b); }",
                                  "float max_nd(float a, float b) { return (a > b || a != a) ? a : b; }"),
    "SR rounds up on u == p": ("(u < p ? k + 1 : k)", "(u <= p ? k + 1 : k)"),
    "four-over-six encode reciprocal not clamped to FLT_MAX": (
        "const float enc = min_nd(1.0f / (dc[cand] * g.S_dec), FLT_MAX);",
        "const float enc = 1.0f / (dc[cand] * g.S_dec);"),
    "four-over-six encode divides instead of multiplying by the reciprocal": (
        "cc[cand][i] = orc_e2m1_encode_rn(yv * enc);",
        "cc[cand][i] = orc_e2m1_encode_rn(yv / (dc[cand] * g.S_dec));"),
    "plain encode multiplies by the reciprocal": ("const float v = yv / D;", "const float v = yv * (1.0f / D);"),
    "plain divisor d / S_enc instead of d * S_dec": ("const float D = d6 * g.S_dec;", "const float D = d6 / g.S_enc;"),
    "tensor amax over x, not x + residual": (
        "if (gamax_mode == ORC_GAMAX_TENSOR) orc_amax(y.data(), M, K, ORC_F32, nullptr, ORC_GAMAX_TENSOR, gamax);",
        "if (gamax_mode == ORC_GAMAX_TENSOR) orc_amax(x, M, K, dtype, nullptr, ORC_GAMAX_TENSOR, gamax);"),
    "row-given amax takes the first row's": (
        "if (gamax_mode == ORC_GAMAX_ROW || gamax_mode == ORC_GAMAX_ROW_GIVEN) g.A = gamax[r];",
        "if (gamax_mode == ORC_GAMAX_ROW) g.A = gamax[r]; if (gamax_mode == ORC_GAMAX_ROW_GIVEN) g.A = gamax[0];"),
    "row-given dequantize takes the first row's amax": (
        "                orc_global_scales(gamax[r], scale_bound, &S_enc, &S_dec);\n            for (int64_t c = 0;",
        "                orc_global_scales(gamax[0], scale_bound, &S_enc, &S_dec);\n            for (int64_t c = 0;"),
    "qdq dequantizes without the global scale": (
        "return orc_dequantize(codes, scales, M, K, gamax_mode, gamax, scale_bound, out_bf16, ORC_BF16);",
        "return orc_dequantize(codes, scales, M, K, ORC_GAMAX_NONE, gamax, scale_bound, out_bf16, ORC_BF16);"),
    "row amax over x, not x + residual": (
        "if (gamax_mode == ORC_GAMAX_ROW) orc_amax(y.data(), M, K, ORC_F32, nullptr, ORC_GAMAX_ROW, gamax);",
        "if (gamax_mode == ORC_GAMAX_ROW) orc_amax(x, M, K, dtype, nullptr, ORC_GAMAX_ROW, gamax);"),
    "columnwise output without the global scale": (
        "std::vector<GScale> gt(static_cast<size_t>(K > 0 ? K : 1), M > 0 ? gs[0] : GScale{0.0f, 1.0f, 1.0f});",
        "std::vector<GScale> gt(static_cast<size_t>(K > 0 ? K : 1), GScale{0.0f, 1.0f, 1.0f});"),
    "columnwise draws ignore row_offset": ("seed, step, row_offset, codes_col, scales_col, nullptr};",
                                           "seed, step, 0, codes_col, scales_col, nullptr};"),
    "standard association's 1/6 taken in double": (
        "float block_s6f_std(float b, float S_enc) { return b * (S_enc * (1.0f / 6.0f)); }",
        "float block_s6f_std(float b, float S_enc) { return b * static_cast<float>(S_enc / 6.0); }"),
    "e4m3 subnormals one binade low": ("const double mag = (e == 0) ? std::ldexp(static_cast<double>(m), -9)",
                                       "const double mag = (e == 0) ? std::ldexp(static_cast<double>(m), -10)"),
    "fp32 dequantize rounded through bf16": (
        "                else static_cast<float*>(out)[r * K + c] = v;",
        "                else static_cast<float*>(out)[r * K + c] = orc_bf16_to_f32(orc_f32_to_bf16(v));"),
    "empty tensor amax -inf": (
        "        float A = 0.0f;\n        for (int64_t r = 0; r < M; ++r) A = max_nd(A, part[r]);",
        "        float A = -INFINITY;\n        for (int64_t r = 0; r < M; ++r) A = max_nd(A, part[r]);"),
    "S_enc falls back to 1 only for a zero amax": ("if (!(A > 0.0f) || std::isinf(A)) enc = 1.0f;",
                                                   "if (A == 0.0f) enc = 1.0f;"),
    "S_enc not clamped to FLT_MAX": ("else enc = min_nd((6.0f * bound) / A, FLT_MAX);",
                                     "else enc = (6.0f * bound) / A;"),
    "S_dec computed from A instead of 1 / S_enc": (
        "*S_dec = 1.0f / enc;", "*S_dec = (A > 0.0f && !std::isinf(A)) ? A / (6.0f * bound) : 1.0f;"),
    "Philox multipliers swapped": ("const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;",
                                   "const uint32_t M0 = 0xCD9E8D57u, M1 = 0xD2511F53u;"),
    "SR counter uses idx, not idx/4": ("const uint64_t blk = idx >> 2;", "const uint64_t blk = idx;"),
    "residual ignores the previous residual": ("residual[i] = y[i] - dq[i];",
                                               "residual[i] = widen(x, dtype, i) - dq[i];"),
    "standard association grouped like four-over-six": (
        "return b * (S_enc * (1.0f / 6.0f)); }", "return (b * (1.0f / 6.0f)) * S_enc; }"),
    "columnwise SR keyed on the x^T index": (
        "const int64_t xr = P.transposed ? cols[i] : rows[i];\n                const int64_t xc = P.transposed ? rows[i] : cols[i];\n                const int64_t xK = P.transposed ? P.R : P.C;",
        "const int64_t xr = rows[i];\n                const int64_t xc = cols[i];\n                const int64_t xK = P.C;"),
    "dequantize associates q * (d * S_dec)": (
        "const float v = (orc_e2m1_value(code) * d) * S_dec;",
        "const float v = orc_e2m1_value(code) * (d * S_dec);"),
    "residual dequant associates q * (d * S_dec)": (
        "P.dq32[rows[i] * P.C + cols[i]] = (q * d_out) * g.S_dec;",
        "P.dq32[rows[i] * P.C + cols[i]] = q * (d_out * g.S_dec);"),
    "nibbles swapped": ("if (c % 2 == 0) byte = static_cast<uint8_t>((byte & 0xF0) | code);",
                        "if (c % 2 == 1) byte = static_cast<uint8_t>((byte & 0xF0) | code); else if (0) byte = 0;"),
}


def _run_mutation(name: str, work: str):
    """Build the oracle with one planted mistake under work/ and run the pin
    suite against it.  Returns (anchor found, pin-suite exit code, output tail)."""
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    if src.count(old) < 1:
        return False, None, ""
    os.makedirs(work, exist_ok=True)
    cpp = os.path.join(work, "nvfp4_oracle.cpp")
    with open(cpp, "w") as f:
        f.write(src.replace(old, new, 1))
    with open(os.path.join(work, "nvfp4_oracle.h"), "w") as f:
        f.write(open(os.path.join(ROOT, "oracle", "nvfp4_oracle.h")).read())
    so = os.path.join(work, "liboracle_mut.so")
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-w",
                    "-pthread", "-shared", "-fPIC", cpp, "-o", so], check=True)
    env = dict(os.environ, NVFP4_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return True, r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every planted mistake, built and checked concurrently (each one is an
    independent compile and pin-suite process)."""
    base = str(tmp_path_factory.mktemp("mutations"))
    names = sorted(MUTATIONS)
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        runs = ex.map(lambda i: _run_mutation(names[i], os.path.join(base, f"m{i}")), range(len(names)))
        return dict(zip(names, runs))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, outcomes):
    found, rc, tail = outcomes[name]
    assert found, f"mutation anchor not found: {name}"
    # exit code 1 is pytest's "tests failed": an interrupted, crashed or
    # killed pin run (any other code) does not count as a catch
    assert rc == 1, f"pins did not catch: {name} (exit code {rc})\n{tail}"
