"""Planted mistakes in the oracle: each mutant is the oracle's C source with
one plausible slip written into it (ties away from zero, a wrong bias, a
reciprocal where the definition divides, a dropped absolute value or scale,
a transposed scale index, the current tensor leaking into its own delayed
scale, ...), compiled to its own library in a temporary folder.  The pins
in test_oracle_pins.py that guard that part of the definition must fail
against the mutant, and every pin used here must pass against the unchanged
source compiled the same way.  Every mutant keeps its memory accesses in
bounds.  This proves the claim of those pins rather than assuming it."""
import shutil
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins

E4, E5 = oracle.E4M3, oracle.E5M2

# name: (text of the source, its replacement, pins that must catch it)
MUTANTS = {
    "ties_away_from_zero": (
        "if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
        "if (frac >= 0.5) r += 1.0;",
        [("test_encode_midpoints_vs_torch", (E4,)), ("test_encode_midpoints_vs_torch", (E5,))]),
    "ties_toward_zero": (
        "if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
        "if (frac > 0.5) r += 1.0;",
        [("test_encode_midpoints_vs_torch", (E4,)), ("test_encode_every_bf16_vs_torch", (E5,))]),
    "e4m3_bias_8": (
        "d.bias = 7;", "d.bias = 8;",
        [("test_decode_all_bytes_vs_torch", (E4,)), ("test_fixed_codes", ())]),
    "subnormals_on_a_finer_grid": (
        "if (e < emin) e = emin;", "(void)emin;",
        [("test_encode_every_bf16_vs_torch", (E4,)), ("test_encode_every_bf16_vs_torch", (E5,))]),
    "overflow_tested_before_rounding": (
        "if (mag > d.fmax)", "if (a > d.fmax)",
        [("test_encode_every_bf16_vs_torch", (E4,)), ("test_encode_midpoints_vs_torch", (E4,))]),
    "subnormal_decoded_as_normal": (
        "v = ldexp((double)m, 1 - d.bias - d.man_bits);",
        "v = ldexp((double)((1 << d.man_bits) + m), 1 - d.bias - d.man_bits);",
        [("test_decode_all_bytes_vs_torch", (E4,)), ("test_decode_all_bytes_vs_torch", (E5,))]),
    "bf16_widened_by_15_bits": (
        "(uint32_t)((const uint16_t *)x)[i] << 16;", "(uint32_t)((const uint16_t *)x)[i] << 15;",
        [("test_bf16_input_widening", ())]),
    "amax_without_abs": (
        "float a = fabsf(orc_load(x, in_dtype, i));", "float a = orc_load(x, in_dtype, i);",
        [("test_amax_brute_force", ())]),
    "no_scale_floor": (
        "if (s < floor_s) s = floor_s;", "(void)floor_s;",
        [("test_scale_floor", ())]),
    "scale_by_reciprocal": (
        "float s = amax / (float)describe(fmt).fmax;",
        "float s = amax * (1.0f / (float)describe(fmt).fmax);",
        [("test_scale_is_fp32_division", ())]),
    "cast_by_reciprocal": (
        "float v = xv / s;", "float v = xv * (1.0f / s);",
        [("test_cast_is_division_near_fp8_midpoints", (E4,)),
         ("test_cast_is_division_near_fp8_midpoints", (E5,))]),
    "tile_amax_without_abs": (
        "      for (int64_t c = c0; c < c1; ++c) {\n"
        "        float a = fabsf(orc_load(x, in_dtype, r * cols + c));",
        "      for (int64_t c = c0; c < c1; ++c) {\n"
        "        float a = orc_load(x, in_dtype, r * cols + c);",
        [("test_tile_rows_vs_torch_per_tile", (E4, (5, 300)))]),
    "tile_scales_row_major": (
        "scales[(c0 / 128) * rows + r] = s;", "scales[r * ((cols + 127) / 128) + c0 / 128] = s;",
        [("test_tile_rows_vs_torch_per_tile", (E4, (5, 300)))]),
    "block_scales_transposed": (
        "scales[(r0 / 128) * ncb + c0 / 128] = s;",
        "scales[(c0 / 128) * ((rows + 127) / 128) + r0 / 128] = s;",
        [("test_block_is_tensor_per_block", (E4,))]),
    "rowwise_column_amax_over_first_rows": (
        "      for (int64_t r = 0; r < rows; ++r) {\n"
        "        float a = fabsf(orc_load(x, in_dtype, r * cols + c));",
        "      for (int64_t r = 0; r < (rows < 16 ? rows : 16); ++r) {\n"
        "        float a = fabsf(orc_load(x, in_dtype, r * cols + c));",
        [("test_rowwise_is_page_roundtrip_per_row_and_column", (E4,))]),
    "delayed_sees_its_own_amax": (
        "  float s = orc_scale_from_amax(hmax, fmt);\n"
        "  orc_quantize_tensor(x, in_dtype, rows, cols, s, fmt, saturate, q, q_t);\n"
        "  history[*next] = orc_amax(x, in_dtype, rows * cols);",
        "  float cur = orc_amax(x, in_dtype, rows * cols);\n"
        "  if (cur > hmax) hmax = cur;\n"
        "  float s = orc_scale_from_amax(hmax, fmt);\n"
        "  orc_quantize_tensor(x, in_dtype, rows, cols, s, fmt, saturate, q, q_t);\n"
        "  history[*next] = cur;",
        [("test_delayed_ring_bookkeeping", ()),
         ("test_smoke3_delayed_misses_spike_current_holds_it", ())]),
    "gemm_drops_b_scale": (
        "double b = orc_fp8_decode(B->data[n * K + k], B->fmt) * orc_operand_scale(B, n, k);",
        "double b = orc_fp8_decode(B->data[n * K + k], B->fmt);",
        [("test_gemm_vs_numpy_dense", ("tensor",)), ("test_gemm_one_hot_closed_form", ())]),
    "gemm_tile_scale_ignores_k_block": (
        "return op->scale[kb * op->stride_k + row * op->stride_row];",
        "return op->scale[row * op->stride_row];",
        [("test_gemm_vs_numpy_dense", ("tile_tile",)), ("test_gemm_vs_numpy_dense", ("tile_block",))]),
    "gemm_abs_sum_signed": (
        "aacc += fabs(a * b);", "aacc += a * b;",
        [("test_gemm_vs_numpy_dense", ("tensor",))]),
    "tile_cols_scales_column_major": (
        "scales[(r0 / 128) * cols + c] = s;", "scales[c * ((rows + 127) / 128) + r0 / 128] = s;",
        [("test_tile_cols_is_rows_of_transpose", (E4,))]),
    "e5m2_overflow_to_max_instead_of_inf": (
        "uint8_t ovf_code = (uint8_t)(fmt == ORC_E4M3 ? 0x7F : 0x7C);",
        "uint8_t ovf_code = (uint8_t)(fmt == ORC_E4M3 ? 0x7F : 0x7B);",
        [("test_encode_every_bf16_vs_torch", (E5,))]),
    "delayed_ring_never_advances": (
        "*next = (*next + 1) % hist_len;", "*next = *next % hist_len;",
        [("test_delayed_ring_bookkeeping", ())]),
    "amax_ignores_nan": (
        "    if (isnan(a)) return a;\n    if (a > m) m = a;", "    if (a > m) m = a;",
        [("test_amax_brute_force", ())]),
    "tensor_transposed_copy_in_row_layout": (
        "      if (q) q[r * cols + c] = b;\n      if (q_t) q_t[c * rows + r] = b;",
        "      if (q) q[r * cols + c] = b;\n      if (q_t) q_t[r * cols + c] = b;",
        [("test_tensor_matches_page_and_transpose", (E4,))]),
    "e5m2_inf_decoded_as_nan": (
        "v = (m == 0) ? INFINITY : NAN;", "v = NAN;",
        [("test_decode_all_bytes_vs_torch", (E5,))]),
    "saturate_flag_ignored": (
        "(saturate ? max_code : ovf_code)", "(ovf_code)",
        [("test_encode_saturating", (E4,)), ("test_encode_saturating", (E5,))]),
    "gemm_sums_magnitudes": (
        "    acc += a * b;\n", "    acc += fabs(a * b);\n",
        [("test_gemm_vs_numpy_dense", ("tensor",))]),
    "mx_exponent_not_clamped_below": (
        "    if (e < -127) e = -127;\n", "",
        [("test_mx_scale_special_cases", ()), ("test_mx_scale_bracket_in_exact_rationals", (E4,))]),
    "mx_emax_off_by_one": (
        "  return ex - 1;\n}", "  return ex;\n}",
        [("test_emax_elem_from_the_page_constants", (E4,)),
         ("test_mx_scale_bracket_in_exact_rationals", (E5,))]),
    "mx_elements_not_saturating": (
        "out[i * out_stride] = encode_double(v, fmt, 1);",
        "out[i * out_stride] = encode_double(v, fmt, 0);",
        [("test_mx_elements_vs_torch_cast", (E4,))]),
}


def _compile(root, name, old, new):
    src = open(oracle._SRC).read()
    if old is not None:
        assert src.count(old) == 1, f"{name}: the planted text must occur exactly once"
        src = src.replace(old, new)
    d = root / name
    d.mkdir()
    shutil.copy(oracle._HDR, d / "fp8_oracle.h")
    (d / "fp8_oracle.c").write_text(src)
    lib = d / "liboracle.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-o", str(lib), str(d / "fp8_oracle.c"), "-lm"])
    return str(lib)


def _use(monkeypatch, lib):
    """Route every oracle call of this test to `lib` (undone after the test)."""
    monkeypatch.setattr(oracle, "build", lambda force=False: lib)
    monkeypatch.setattr(oracle, "_lib", None)


def _fails(pin, args):
    try:
        getattr(pins, pin)(*args)
    except Exception:          # an assertion, or an error the wrong values lead to
        return True
    return False


def test_pins_pass_on_the_unchanged_source(tmp_path, monkeypatch):
    _use(monkeypatch, _compile(tmp_path, "unchanged", None, None))
    used = sorted({(p, a) for _, _, cases in MUTANTS.values() for p, a in cases},
                  key=repr)
    failing = [(p, a) for p, a in used if _fails(p, a)]
    assert failing == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_the_planted_mistake(name, tmp_path, monkeypatch):
    old, new, cases = MUTANTS[name]
    _use(monkeypatch, _compile(tmp_path, name, old, new))
    survived = [(p, a) for p, a in cases if not _fails(p, a)]
    assert survived == [], f"{name} passes {survived}"


@pytest.mark.parametrize("bits", [7, 9])
def test_bf16_spacing_pin_catches_a_wrong_significand_width(bits, monkeypatch):
    """The GEMM bound's bf16 allowance lives in the Python wrapper: plant a
    spacing for a significand of the wrong width there instead."""
    import numpy as np

    def wrong(v):
        a = np.abs(np.asarray(v, dtype=np.float64))
        e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
        return np.ldexp(1.0, (e - (bits - 1)).astype(np.int64))

    monkeypatch.setattr(oracle, "bf16_ulp", wrong)
    assert _fails("test_bf16_ulp_vs_torch_spacing", ())
