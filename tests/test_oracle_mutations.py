"""Plants plausible mistakes in a temporary copy of the CPU oracle and checks that
the oracle's pins (tests/test_oracle_pins.py, tests/test_oracle_pins_glue.py,
tests/test_oracle_pins_q8.py) fail for each one.  The repository's
oracle is never modified; each mutant is compiled and tested in a temp folder."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "nibble_swap": ("out32[j] = (float)(lo - 8) * d;", "out32[j] = (float)(hi - 8) * d;"),
    "offset_7": ("out32[j + 16] = (float)(hi - 8) * d;", "out32[j + 16] = (float)(hi - 7) * d;"),
    "qd_minus_8d": ("out32[j] = (float)(lo - 8) * d;", "out32[j] = (float)lo * d - 8.0f * d;"),
    "scale_big_endian": ("uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));",
                         "uint16_t dbits = (uint16_t)(blk[1] | (blk[0] << 8));"),
    "subnormal_exp": ("v = ldexpf((float)frac, -24);", "v = ldexpf((float)frac, -25);"),
    "ties_to_odd": ("fmod(fl, 2.0) == 1.0", "fmod(fl, 2.0) == 0.0"),
    "max_last_index": ("if (fabsf(x[i]) > amax) {", "if (fabsf(x[i]) >= amax) {"),
    "scale_sign": ("float d32 = x[im] / -8.0f;", "float d32 = x[im] / 8.0f;"),
    "unrounded_scale": ("float t = x[i] / dd;", "float t = x[i] / (x[im] / -8.0f);"),
    "truncating_round": ("float u = t + 8.5f;", "float u = t + 8.0f;"),
    "no_clamp_15": ("if (fq > 15.0f) fq = 15.0f;", "if (fq > 16.0f) fq = 15.0f;"),
    "fp32_accumulate": ("double y = 0.0, s = 0.0;", "float y = 0.0, s = 0.0;"),
    "gather_no_status": ("rc = Q4O_ERR_ID_OUT_OF_RANGE;", "rc = Q4O_OK;"),
    # decoder glue and the repacked layout
    "sigmoid_sign": ("double sig = 1.0 / (1.0 + exp(-a[i]));",
                     "double sig = 1.0 / (1.0 + exp(a[i]));"),
    "gate_on_up": ("double sig = 1.0 / (1.0 + exp(-a[i]));",
                   "double sig = 1.0 / (1.0 + exp(-b[i]));"),
    "no_gate_input": ("out[i] = a[i] * sig * b[i];", "out[i] = sig * b[i];"),
    "argmax_last_tie": ("if (best < 0 || y[i] > y[best]) best = i;",
                        "if (best < 0 || y[i] >= y[best]) best = i;"),
    "argmax_keeps_nan": ("if (isnan(y[i])) continue;", "if (0) continue;"),
    "repack_lane_order": ("int64_t lane = 4 * g + (i % 8) / 2;", "int64_t lane = 4 * g + (i % 4);"),
    "repack_nibble_order": ("int64_t m = hr + 2 * (i / 8) + 4 * (i % 2);",
                            "int64_t m = 2 * hr + (i / 8) + 4 * (i % 2);"),
    "repack_gguf_nibbles": ("if (blk) q = e < 16 ? (blk[2 + e] & 0x0F) : (blk[2 + e - 16] >> 4);",
                            "if (blk) q = (e % 2) ? (blk[2 + e / 2] >> 4) : (blk[2 + e / 2] & 0x0F);"),
    "repack_step_word": ("*code_off = tile + 256 + 512 * (s / 4) + 16 * lane + 4 * (s % 4) + m / 2;",
                         "*code_off = tile + 256 + 512 * (s % 4) + 16 * lane + 4 * (s / 4) + m / 2;"),
    "repack_scale_slot": ("*scale_off = tile + 32 * g + 4 * b + 2 * hr;",
                          "*scale_off = tile + 32 * b + 4 * g + 2 * hr;"),
    "repack_pad_code": ("int q = 8;", "int q = 0;"),
    # the Q4 x Q8 integer path
    "q8_round_half_even": ("c = roundf(t); /* halves away from zero */",
                           "c = rintf(t); /* halves away from zero */"),
    "q8_scale_255": ("float db = amax / 127.0f;", "float db = amax / 255.0f;"),
    "q8_no_offset": ("isum += (int64_t)(lo - 8) * q[32 * b + j];",
                     "isum += (int64_t)lo * q[32 * b + j];"),
    "q8_nibble_order": ("int lo = blk[2 + j] & 0x0F, hi = blk[2 + j] >> 4;",
                        "int hi = blk[2 + j] & 0x0F, lo = blk[2 + j] >> 4;"),
    "q8_signed_max": ("float a = fabsf(xb[j]);", "float a = xb[j];"),
    "f64_rounds_x": ("double p = (double)wrow[kk] * x[kk];",
                     "double p = (double)wrow[kk] * (double)(float)x[kk];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    before, after = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "q4_oracle.c")).read()
    assert before in src, f"mutation site for {name} no longer exists"
    for sub in ("oracle", "tests", "synth"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__", "*.tmp*"))
    (tmp_path / "oracle" / "q4_oracle.c").write_text(src.replace(before, after))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "tests/test_oracle_pins_glue.py",
                        "tests/test_oracle_pins_q8.py"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
