"""Mutation check of the oracle's pins: each plausible mistake planted in a copy
of the oracle source (a wrong bit order, a transposed scan, a dropped term, a
wrong sign, a dropped padding, a swapped nibble, a wrong tile numbering) must
make the pin suite fail.  Mistakes are planted only in the CPU oracle's source
text, in a temporary directory; the committed oracle is untouched."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "us_oracle.c")

MUTANTS = {
    "bit_order_msb_first": ("if (!dense_nonzero(W, ldw, elem, r, c)) continue;\n                words[p / 64] |= (uint64_t)1 << (p % 64);",
                            "if (!dense_nonzero(W, ldw, elem, r, c)) continue;\n                words[p / 64] |= (uint64_t)1 << (63 - p % 64);"),
    "row_scan_transposed": ("if (order == OR_ROW) { *i = (int)(p / TK); *j = (int)(p % TK); }",
                            "if (order == OR_ROW) { *i = (int)(p % TM); *j = (int)(p / TM); }"),
    "col_scan_transposed": ("else                 { *j = (int)(p / TM); *i = (int)(p % TM); }",
                            "else                 { *j = (int)(p % TK); *i = (int)(p / TK); }"),
    "padding_dropped": ("uint64_t padded = (P + E - 1) / E * E;", "uint64_t padded = P;"),
    "nibble_order_swapped": ("if (e & 1) values[e >> 1] = (uint8_t)((values[e >> 1] & 0x0F) | (nib << 4));",
                             "if (!(e & 1)) values[e >> 1] = (uint8_t)((values[e >> 1] & 0x0F) | (nib << 4));"),
    "int4_sign_wrong": ("return (int8_t)(nib >= 8 ? (int)nib - 16 : (int)nib);",
                        "return (int8_t)(nib >= 8 ? (int)nib - 8 : (int)nib);"),
    "first_term_dropped": ("for (int k = 0; k < K; ++k)\n        acc +=", "for (int k = 1; k < K; ++k)\n        acc +="),
    "scales_swapped": ("float t = a * or_half_to_float(s_w);", "float t = a * or_half_to_float(s_w) * 0.5f + a * or_half_to_float(s_x) * 0.5f;"),
    "abs_dropped_in_skip": ("if (skip && !(fabs(x) > tau)) continue;", "if (skip && !(x > tau)) continue;"),
    "quant_divisor_8": ("uint16_t s16 = or_float_to_half(amax / 7.0f);", "uint16_t s16 = or_float_to_half(amax / 8.0f);"),
    "quant_truncates": ("float q = rintf(v / s);", "float q = truncf(v / s);"),
    "quant_rounds_half_up": ("float q = rintf(v / s);", "float q = floorf(v / s + 0.5f);"),
    "quant_signed_max": ("const float a = fabsf(or_half_to_float(x[k]));", "const float a = or_half_to_float(x[k]);"),
    "colinfo_row_scan": ("const int64_t pos = (int64_t)j * TM + i;          /* COL scan: p = j*TM + i */",
                         "const int64_t pos = (int64_t)i * TK + j;          /* COL scan: p = j*TM + i */"),
    "colinfo_offset_inclusive": ("            colinfo[t * TK + j] = (offset << 16) | nnz;\n            offset += nnz;",
                                 "            offset += nnz;\n            colinfo[t * TK + j] = (offset << 16) | nnz;"),
    "colinfo_fields_swapped": ("colinfo[t * TK + j] = (offset << 16) | nnz;", "colinfo[t * TK + j] = (nnz << 16) | offset;"),
    "ie_stream_offset_dropped": ("const uint64_t e = off + (uint64_t)q * P + rho;", "const uint64_t e = off + rho;"),
    "ie_areas_column_major": ("const int q = a * CA + c;", "const int q = c * RA + a;"),
    "reorder_cost_ignores_union": ("        cost += any;", "        cost += 1;"),
    "reorder_perm_groupwise": ("perm[p * G + g] = (uint8_t)groups[g][p];", "perm[g * RA + p] = (uint8_t)groups[g][p];"),
    "int2_sign_wrong": ("return (int8_t)(c >= 2 ? (int)c - 4 : (int)c);", "return (int8_t)(c >= 2 ? (int)c - 2 : (int)c);"),
    "int2_crumb_order_swapped": ("const int sh = 2 * (int)(e & 3);", "const int sh = 6 - 2 * (int)(e & 3);"),
    "tile_numbering_colmajor": ("            const int64_t t = (int64_t)tm * nTK + tk;\n            uint64_t* words = bitmap + t * words_per_tile;\n"
                                "            for (int64_t w = 0; w < words_per_tile; ++w) words[w] = 0;\n            uint64_t P = 0; ",
                                "            const int64_t t = (int64_t)tk * nTM + tm;\n            uint64_t* words = bitmap + t * words_per_tile;\n"
                                "            for (int64_t w = 0; w < words_per_tile; ++w) words[w] = 0;\n            uint64_t P = 0; "),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=gnu11",
                    "-o", str(lib), str(mut), "-lm"], check=True)
    env = dict(os.environ, US_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake {name} passed every pin:\n{r.stdout[-2000:]}"
