"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins in ``test_oracle.py`` catch every one of them.

Each mutant is a one-line textual change of ``oracle/attn_oracle.c`` compiled
to a temporary library; the original file is never touched.
"""
import os

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "gqa_map_modulo": ("const int hk = h / G;\n    const int64_t n = rows_for",
                       "const int hk = h % n_kv_head;\n    const int64_t n = rows_for"),
    "scale_dropped": ("x[j] = scale * dot;", "x[j] = dot;"),
    "no_normalisation": ("for (int d = 0; d < head_dim; ++d) o[d] /= Z;",
                         "for (int d = 0; d < head_dim; ++d) o[d] /= (Z > 1 ? 1 : Z);"),
    "nkv_off_by_one": ("int64_t n = (int64_t)positions[s] + 1;",
                       "int64_t n = (int64_t)positions[s];"),
    "clamp_missing": ("if (n > cap) n = cap;", "if (n > cap + 0x7fffffff) n = cap;"),
    "k_is_v": ("dot += (double)qh[d] * dec(ks[j * row + d]);\n        x[j]",
               "dot += (double)qh[d] * dec(vs[j * row + d]);\n        x[j]"),
    "exp_sign": ("const double w = exp(x[j] - m);", "const double w = exp(m - x[j]);"),
    "f16_bias": ("ldexp((double)(1024 + frac), expo - 25)",
                 "ldexp((double)(1024 + frac), expo - 24)"),
    "f16_subnormal": ("mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -25);"),
    "f16_sign": ("        mag = ldexp((double)(1024 + frac), expo - 25);\n    return sign ? -mag : mag;",
                 "        mag = ldexp((double)(1024 + frac), expo - 25);\n    return mag;"),
    "bf16_bias": ("ldexp((double)(128 + frac), expo - 134)", "ldexp((double)(128 + frac), expo - 133)"),
    "bf16_fields": ("const int expo = (bits >> 7) & 0xff;", "const int expo = (bits >> 8) & 0xff;"),
    "bf16_as_f16": ("return kv_dtype == 1 ? oracle_bf16_to_double : oracle_f16_to_double;",
                    "return oracle_f16_to_double;"),
    "split_no_corr": ("const double corr = exp(m_ - nmx);", "const double corr = 1.0;"),
    "combine_no_weight": ("exp(mx[sp] - gmx);", "1.0;"),
    "split_chunk_floor": ("(nkv + n_splits - 1) / n_splits", "nkv / n_splits"),
    "causal_off_by_one": ("rows_for(positions, s, cap) - n_q + t + 1;",
                          "rows_for(positions, s, cap) - n_q + t;"),
    "head_stride": ("const float *qh = q + ((int64_t)s * n_head + h) * head_dim;\n    return one_query",
                    "const float *qh = q + ((int64_t)s * n_head + hk) * head_dim;\n    return one_query"),
}

PIN_SUITE = [pins.check_f16_decoder, pins.check_bf16_decoder, pins.check_bruteforce,
             pins.check_bruteforce_bf16, pins.check_closed_forms,
             pins.check_invariants, pins.check_gqa_mapping, pins.check_positions,
             pins.check_split_equivalence, pins.check_stability, pins.check_multi_query]


def _pins_fail(lib) -> bool:
    for pin in PIN_SUITE:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            return True
    return False


def test_unmutated_oracle_passes_every_pin():
    assert not _pins_fail(oracle.load_library())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor for %s not unique" % name
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib_path = oracle.build(str(src), str(tmp_path / "libmutant.so"))
    lib = oracle.load_library(lib_path)
    assert _pins_fail(lib), "pins did not catch mutant %s" % name
