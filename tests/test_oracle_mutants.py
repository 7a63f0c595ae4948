"""Planted mistakes in a copy of the oracle must each fail a pin (CPU only).

Every mutant is a one-line textual change to ``oracle/pda_oracle.cpp``
compiled into a temporary library; the real source is never modified. This
shows the pins in ``oracle_pins.py`` are strong enough to catch a dropped
term, a wrong sign or index, or a transposed operand.
"""

import os

import pytest

import oracle
from tests import oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "pda_oracle.cpp")

MUTANTS = {
    "dropped_k_scale": ("acc += qd[d] * (e4m3[code] * ks);", "acc += qd[d] * e4m3[code];"),
    "dropped_v_scale": ("o[d] += wt * (e4m3[vpage[vi]] * vs);", "o[d] += wt * e4m3[vpage[vi]];"),
    "dropped_softmax_scale": ("z[t] = scale * acc;", "z[t] = acc;"),
    "wrong_sign": ("z[t] = scale * acc;", "z[t] = -scale * acc;"),
    "k_page_token_major": ("kpage[(static_cast<long long>(d / 16) * bs + slot) * 16 + (d % 16)]",
                           "kpage[(slot * (D / 16) + d / 16) * 16 + (d % 16)]"),
    "v_page_token_major": (": static_cast<long long>(d) * bs + slot;", ": slot * D + d;"),
    "gqa_modulo": ("const int kv = h / g;", "const int kv = h % num_kv_heads;"),
    "e4m3_bias_8": ("mag = std::ldexp(1.0 + static_cast<double>(mant) / 8.0, expo - 7);",
                    "mag = std::ldexp(1.0 + static_cast<double>(mant) / 8.0, expo - 8);"),
    "e4m3_subnormal_as_normal": ("mag = std::ldexp(static_cast<double>(mant) / 8.0, -6);",
                                 "mag = std::ldexp(1.0 + static_cast<double>(mant) / 8.0, -7);"),
    "no_max_shift": ("w[t] = std::exp(z[t] - zmax);", "w[t] = std::exp(z[t]);"),
    "table_row_stride_pages": ("const long long b = block_tables[s * MB + t / bs];\n      const long long slot = t % bs;\n      const uint8_t* kpage",
                               "const long long b = block_tables[s * ((L + bs - 1) / bs) + t / bs];\n      const long long slot = t % bs;\n      const uint8_t* kpage"),
    "one_token_short": ("std::vector<double> z(L);\n    for (long long t = 0; t < L; ++t) {",
                        "std::vector<double> z(L);\n    z[L - 1] = -1e300;\n    for (long long t = 0; t + 1 < L; ++t) {"),
    "encode_ties_to_odd": ("(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
    "encode_ties_away": ("(d == best_d && (c & 1) == 0)", "(d == best_d)"),
    "cache_write_divides_in_binary64": ("const float xk = static_cast<float>(bf16_value(key[src])) / k_scale;",
                                        "const double xk = bf16_value(key[src]) / static_cast<double>(k_scale);"),
    "cache_write_multiplies_scale": ("const float xv = static_cast<float>(bf16_value(value[src])) / v_scale;",
                                     "const float xv = static_cast<float>(bf16_value(value[src])) * v_scale;"),
    "cache_write_k_token_major": ("k_cache[page + ((d / 16) * bs + o) * 16 + (d % 16)]",
                                  "k_cache[page + (o * (D / 16) + d / 16) * 16 + (d % 16)]"),
    "cache_write_v_token_major": (": d * bs + o;", ": o * D + d;"),
    "slot_scale_wrong_head": ("k_scales[(b * num_kv_heads + kv) * bs + slot]", "k_scales[(b * num_kv_heads + 0) * bs + slot]"),
    "slot_scale_wrong_slot": ("v_scales[(b * num_kv_heads + kv) * bs + slot]", "v_scales[(b * num_kv_heads + kv) * bs]"),
    "shuffled_v_dim_token_swapped": ("const long long vi = v_shuffled ? ((slot / 16) * D + d) * 16 + (slot % 16)",
                                      "const long long vi = v_shuffled ? ((slot / 16) * D + (slot % 16)) * 16 + d % 16"),
    "sink_carries_value": ("double denom = sinks ? std::exp(zs - zmax) : 0.0;", "double denom = 0.0;"),
}


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, src_text, tmp_path):
    old, new = MUTANTS[name]
    assert src_text.count(old) >= 1, "mutation anchor not found: %s" % name
    mutated = src_text.replace(old, new, 1)
    src = tmp_path / "mutant.cpp"
    src.write_text(mutated)
    lib_path = str(tmp_path / "libmutant.so")
    oracle.build(force=True, src=str(src), out=lib_path)
    lib = oracle.load(lib_path)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError):
            caught.append(pin.__name__)
    assert caught, "mutant %s passed every pin" % name
