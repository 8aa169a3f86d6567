"""The oracle's pins catch plausible mistakes (CPU only).

Each case edits one expression (always memory-safe for the shapes the pins use) of a copy of the oracle source (a dropped
term, a wrong sign, a swapped index, ties rounded away from even ...),
builds it into a throw-away library, swaps it in, and runs the pin tests.
At least one pin must fail for every planted mistake.  The real oracle is
restored afterwards.
"""
import inspect

import pytest

import oracle
import test_oracle_cast as tc
import test_oracle_codec as tk
import test_oracle_dequant as td
import test_oracle_scale as ts
import test_oracle_swiglu as tw
import test_oracle_tile_cast as tt
import test_oracle_rmsnorm as trn

MUTATIONS = {
    "ties_away_e4m3": ("(dropped == 0x80000u && (keep & 1u))",
                       "(dropped == 0x80000u)"),
    "ties_away_e2m1": ("(dropped == 0x200000u && (keep & 1u))",
                       "(dropped == 0x200000u)"),
    "subnormal_ties_away": ("(frac == 0.5f && (m & 1u))", "(frac == 0.5f)"),
    "no_amax_floor": ("float a = amax > 1e-4f ? amax : 1e-4f;",
                      "float a = amax;"),
    "floor_1e3": ("amax > 1e-4f ? amax : 1e-4f", "amax > 1e-3f ? amax : 1e-3f"),
    "sign_of_zero_lost": ("signbit(q) ? 0x80u : 0u", "q < 0 ? 0x80u : 0u"),
    "pow2_exact_power_bumped": ("(f == 0.5f) ? E - 1 : E", "E"),
    "subnormal_threshold": ("biased >= 127 - 6", "biased >= 127 - 7"),
    "e4m3_bias": ("int e = biased - 127 + 7;", "int e = biased - 127 + 8;"),
    "nibble_order": ("if ((col & 1) == 0)", "if ((col & 1) == 1)"),
    "transposed_rows_paired": ("base[j * ld_scales + m] = sc.s;",
                               "base[j * ld_scales + (m ^ 1)] = sc.s;"),
    "ue8m0_byte_order": ("base[word * 4 + b] = (uint8_t)sc.ue8m0;",
                         "base[word * 4 + (3 - b)] = (uint8_t)sc.ue8m0;"),
    "ue8m0_pad_not_zeroed": ("base[word * 4 + b] = 0;", "(void)word;"),
    "gate_up_swapped": ("row[k] = oracle_swiglu_value(bf16_bits_to_float(xr[k]),\n"
                        "                                         bf16_bits_to_float(xr[N + k]));",
                        "row[k] = oracle_swiglu_value(bf16_bits_to_float(xr[N + k]),\n"
                        "                                         bf16_bits_to_float(xr[k]));"),
    "silu_sign": ("(1.0 + exp(-g))", "(1.0 + exp(g))"),
    "fmt_max_e2m1": ("448.0f : 6.0f", "448.0f : 8.0f"),
    "scale_multiplied": ("float q = yg[k] / sc.s;", "float q = yg[k] * sc.s;"),
    "amax_without_abs": ("float a = fabsf(yg[k]);", "float a = yg[k];"),
    "saturation_dropped": ("if (a > 448.0f)\n        a = 448.0f;", ""),
    "decode_bias": ("mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);",
                    "mag = ldexpf(1.0f + (float)m / 8.0f, e - 8);"),
    "decode_subnormal_step": ("mag = ldexpf((float)m, -9);",
                              "mag = ldexpf((float)m, -10);"),
    "decode_e2m1_subnormal": ("e == 0 ? 0.5f * (float)m", "e == 0 ? 1.0f * (float)m"),
    "bf16_ties_up": ("(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    "bf16_truncates": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))\n        upper += 1;", ""),
    "dequant_nibble_order": ("(k & 1) ? byte >> 4 : byte & 0xF", "(k & 1) ? byte & 0xF : byte >> 4"),
    "dequant_scale_transposed_index": ("                                         : base[j * ld_scales + m];",
                                       "                                         : base[m * 0 + j * ld_scales];"),
}

# Mistakes in the RMSNorm code, run against its pins.
RMS_MUTATIONS = {
    "rms_eps_dropped": ("double rstd = 1.0 / sqrt((double)eps + ss / (double)K);",
                        "double rstd = 1.0 / sqrt(ss / (double)K);"),
    "rms_sum_not_mean": ("double rstd = 1.0 / sqrt((double)eps + ss / (double)K);",
                         "double rstd = 1.0 / sqrt((double)eps + ss);"),
    "rms_no_root": ("double rstd = 1.0 / sqrt((double)eps + ss / (double)K);",
                    "double rstd = 1.0 / ((double)eps + ss / (double)K);"),
    "rms_mean_over_k_minus_1": ("ss / (double)K);", "ss / (double)(K - 1));"),
    "rms_gain_ignored": ("y[m * ld_y + k] = (float)((double)bf16_bits_to_float(w[k]) *",
                         "y[m * ld_y + k] = (float)((double)1.0f *"),
    "rms_abs_not_square": ("ss += v * v;", "ss += fabs(v);"),
    "rms_gain_of_first_channel": ("(double)bf16_bits_to_float(w[k]) *", "(double)bf16_bits_to_float(w[0]) *"),
}

# Mistakes in the per-block / per-channel code, run against those pins.
TILE_MUTATIONS = {
    "block_last_row_dropped": ("int64_t r1 = r0 + block < M ? r0 + block : M;",
                               "int64_t r1 = r0 + block - 1 < M ? r0 + block - 1 : M;"),
    "block_amax_last_column_missed": ("for (int64_t c = c0; c < c1; ++c) {\n                    float v",
                                      "for (int64_t c = c0; c < c1 - 1; ++c) {\n                    float v"),
    "block_scale_columns_reversed": ("put_scale(srow, cb, mode, sc);",
                                     "put_scale(srow, n_cb - 1 - cb, mode, sc);"),
    "block_pad_not_zeroed": ("            zero_word_tail(srow, n_cb);", "            (void)srow;"),
    "block_rows_share_scale_row": ("uint8_t *srow = (uint8_t *)scales + rb * ld_scales * 4;",
                                   "uint8_t *srow = (uint8_t *)scales + (rb / 2) * ld_scales * 4;"),
    "channel_amax_last_row_missed": ("for (int64_t m = 0; m < M; ++m) {\n            float v",
                                     "for (int64_t m = 0; m < M - 1; ++m) {\n            float v"),
    "channel_amax_signed": ("if (fabsf(v) > cmax)\n                cmax = fabsf(v);",
                            "if (v > cmax)\n                cmax = v;"),
    "channel_pad_not_zeroed": ("        zero_word_tail(scales, K);", "        (void)scales;"),
    "tile_nibble_order": ("if (col % 2 == 0)", "if (col % 2 == 1)"),
    "tile_scale_multiplied": ("bf16_bits_to_float(x[m * ld_x + k]) / sc.s);",
                              "bf16_bits_to_float(x[m * ld_x + k]) * sc.s);"),
    "block_dequant_scale_transposed": ("m / block, k / block);", "k / block, m / block);"),
    "channel_dequant_divides": ("code_value(codes + m * ld_codes, k, fmt) * s);\n        }\n    return OR_OK;\n}\n\n/* ---",
                                "code_value(codes + m * ld_codes, k, fmt) / s);\n        }\n    return OR_OK;\n}\n\n/* ---"),
    "dequant_e2m1_nibble_order": ("return e2m1_decode((uint8_t)((k & 1) ? byte >> 4 : byte & 0xF));\n}\n\nstatic void put_output",
                                  "return e2m1_decode((uint8_t)((k & 1) ? byte & 0xF : byte >> 4));\n}\n\nstatic void put_output"),
}


def _pin_functions(mods=None):
    fns = []
    for mod in mods or (tk, ts, tc, tw, td):
        for name, fn in inspect.getmembers(mod, inspect.isfunction):
            if name.startswith("test_") and fn.__module__ == mod.__name__:
                fns.append(fn)
    return fns


def _call_all_params(fn):
    """Run a pin with every parametrisation pytest would give it."""
    marks = getattr(fn, "pytestmark", [])
    combos = [{}]
    for m in marks:
        if m.name != "parametrize":
            continue
        names = [n.strip() for n in m.args[0].split(",")]
        new = []
        for c in combos:
            for v in m.args[1]:
                vals = v if len(names) > 1 else (v,)
                new.append({**c, **dict(zip(names, vals))})
        combos = new
    for kw in combos:
        fn(**kw)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert old in src, f"mutation anchor not found: {old!r}"
    lib = oracle.compile_variant(src.replace(old, new, 1),
                                 str(tmp_path / f"lib_{name}.so"))
    real = oracle._load()
    oracle._lib = lib
    failed = []
    try:
        for fn in _pin_functions():
            try:
                _call_all_params(fn)
            except Exception:  # any failing pin counts
                failed.append(fn.__name__)
    finally:
        oracle._lib = real
    assert failed, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(TILE_MUTATIONS))
def test_planted_tile_mistake_is_caught(name, tmp_path):
    old, new = TILE_MUTATIONS[name]
    src = oracle.source_text()
    assert old in src, f"mutation anchor not found: {old!r}"
    lib = oracle.compile_variant(src.replace(old, new, 1),
                                 str(tmp_path / f"lib_{name}.so"))
    real = oracle._load()
    oracle._lib = lib
    failed = []
    try:
        for fn in _pin_functions((tt,)):
            try:
                _call_all_params(fn)
            except Exception:  # any failing pin counts
                failed.append(fn.__name__)
    finally:
        oracle._lib = real
    assert failed, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(RMS_MUTATIONS))
def test_planted_rmsnorm_mistake_is_caught(name, tmp_path):
    old, new = RMS_MUTATIONS[name]
    src = oracle.source_text()
    assert old in src, f"mutation anchor not found: {old!r}"
    lib = oracle.compile_variant(src.replace(old, new, 1),
                                 str(tmp_path / f"lib_{name}.so"))
    real = oracle._load()
    oracle._lib = lib
    failed = []
    try:
        for fn in _pin_functions((trn,)):
            try:
                _call_all_params(fn)
            except Exception:  # any failing pin counts
                failed.append(fn.__name__)
    finally:
        oracle._lib = real
    assert failed, f"no pin caught the planted mistake {name}"
