"""The oracle's pins must catch plausible mistakes.

Each case copies memq_oracle.c, plants one mistake (a wrong bias, index, sign, rounding rule,
byte order or a dropped term), compiles the copy to a temporary library and runs the oracle pin
tests against it in a child process: at least one pin must fail.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "memq_oracle.c")

MUTATIONS = {
    "e4m3_bias": ("expo - 7);", "expo - 8);"),
    "e4m3_subnormal_scale": ("ldexp((double)mant, -9)", "ldexp((double)mant, -10)"),
    "e4m3_sign_dropped": ("return sign ? -mag : mag;\n}\n\n/* IEEE", "return mag;\n}\n\n/* IEEE"),
    "f16_bias": ("expo - 15)", "expo - 14)"),
    "f16_subnormal": ("ldexp((double)frac, -24)", "ldexp((double)frac, -23)"),
    "rms_mean_divisor": ("ss / (double)ncols", "ss / (double)(ncols - 1)"),
    "rms_eps_sign": ("+ (double)eps", "- (double)eps"),
    "rms_weight_dropped": ("* rr * (double)w[i]", "* rr"),
    "quant_divisor": ("amax / 127.0", "amax / 128.0"),
    "quant_round_rule": ("(int8_t)round(t)", "(int8_t)floor(t + 0.5)"),
    "quant_amax_signed": ("if (fabs(zb[k]) > amax)\n                    amax = fabs(zb[k]);",
                          "if (zb[k] > amax)\n                    amax = zb[k];"),
    "act_block_index": ("d[j * (in_f / 32) + i / 32]", "d[j * (in_f / 32) + i / 64]"),
    "act_row_index": ("qs[j * in_f + i]", "qs[i]"),
    "e4m3_weight_index": ("tab[w[r * in_f + i]] * act",
                          "tab[w[r * in_f + (in_f - 1 - i)]] * act"),
    "blk_grid_col": ("grid[(r / 128) * gcols + i / 128]", "grid[(r / 128) * gcols + i / 256]"),
    "blk_grid_row": ("grid[(r / 128) * gcols + i / 128]", "grid[(r / 256) * gcols + i / 128]"),
    "q8_0_byte_offset": ("blk[2 + i % 32]", "blk[1 + i % 32]"),
    "q8_0_scale_endianness": ("(blk[0] | (blk[1] << 8))", "(blk[1] | (blk[0] << 8))"),
    "q8_0_unsigned_weights": ("(double)(int8_t)blk[2 + i % 32]", "(double)blk[2 + i % 32]"),
    "sabs_signed": ("s += fabs(p);\n            }\n            y[j * nrows + t] = acc;\n"
                    "            sabs[j * nrows + t] = s;\n        }\n    }\n}\n\n/* ggml",
                    "s += p;\n            }\n            y[j * nrows + t] = acc;\n"
                    "            sabs[j * nrows + t] = s;\n        }\n    }\n}\n\n/* ggml"),
    "silu_sign": ("exp(-gi)", "exp(gi)"),
    "silu_up_dropped": ("(1.0 + exp(-gi)) * (double)u[i];", "(1.0 + exp(-gi));"),
    "f16_ties_up": ("double k = rint(v / q);", "double k = floor(v / q + 0.5);"),
    "f16_subnormal_quantum": ("if (e < -14)\n        e = -14;", "if (e < -15)\n        e = -15;"),
    "repack_grid_col": ("aux[(r / 128) * gcols + i / 128]", "aux[(r / 128) * gcols + i / 256]"),
    # (No tie-rule mutant for the repack: with E4M3 inputs the only reachable tie is
    #  W = amax / 2 -> +-63.5, where ties-away and ties-to-even both give +-64.)
    "repack_divisor": ("amax / 127.0f", "amax / 128.0f"),
    "repack_scale_dropped": ("(float)memq_oracle_e4m3(w[r * in_f + i]) * s;",
                             "(float)memq_oracle_e4m3(w[r * in_f + i]);"),
    "repack_f16_byte_order": ("blk[0] = (uint8_t)(h & 0xFF);\n            blk[1] = (uint8_t)(h >> 8);",
                              "blk[1] = (uint8_t)(h & 0xFF);\n            blk[0] = (uint8_t)(h >> 8);"),
    "mla_gemv_transposed": ("const float *wr = w + ((int64_t)h * rows + i) * cols;\n                for (int k = 0; k < cols; ++k) {\n                    double p = (double)xr[k] * (double)wr[k];",
                            "const float *wr = w + ((int64_t)h * rows) * cols;\n                for (int k = 0; k < cols; ++k) {\n                    double p = (double)xr[k] * (double)wr[(int64_t)k * rows % (rows * cols) + i % cols];"),
    "mla_softmax_no_shift": ("l += exp(s[j] - m);", "l += exp(s[j]);"),
    "mla_scale_dropped": ("s[j] = (double)scale * dot;", "s[j] = dot;"),
    "mla_gather_index": ("const float *c = cache + (int64_t)idx[(int64_t)tt * n_slots + j] * row;\n                double dot",
                         "const float *c = cache + (int64_t)idx[j] * row;\n                double dot"),
}

PIN_TESTS = ["tests/test_oracle_decode.py", "tests/test_oracle_producer.py",
             "tests/test_oracle_gemv.py", "tests/test_oracle_next.py", "tests/test_oracle_mla.py"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so_path),
                           str(c_path), "-lm"])
    env = dict(os.environ, MEMQ_ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutation {name} survived every pin:\n{r.stdout[-2000:]}"
