"""Plant plausible mistakes in copies of the oracle source and require the
pins to catch each one (CPU only; the real oracle is never modified)."""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, exact text in oracle.c, replacement)
MUTATIONS = [
    ("drop_scale", "scores[j] = scale * dot;", "scores[j] = dot;"),
    ("gqa_modulo", "int64_t hk = h / group;", "int64_t hk = h % Hkv;"),
    ("causal_off_by_one", "last = i + (L - Sq);", "last = i + (L - Sq) + 1;"),
    ("causal_top_left", "if (causal && i + (L - Sq) < last)\n        last = i + (L - Sq);",
     "if (causal && i < last)\n        last = i;"),
    ("ignore_lengths", "L = seqlens_k[b];", "L = Sk;"),
    ("lse_without_max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("no_normalisation", "o_row[c] /= l;", "o_row[c] /= 1.0;"),
    ("transposed_key", "oracle_load(k, kind, kv_head_off + j * d + c);",
     "oracle_load(k, kind, kv_head_off + c * Sk + j);"),
    ("value_from_wrong_key", "o_row[c] += w * oracle_load(v, kind, kv_head_off + j * d + c);",
     "o_row[c] += w * oracle_load(v, kind, kv_head_off + (n - 1 - j) * d + c);"),
    ("bf16_low_half", "uint32_t word = ((uint32_t)bits) << 16;",
     "uint32_t word = ((uint32_t)bits) << 15;"),
    ("max_not_subtracted_in_weights", "double w = exp(scores[j] - m);",
     "double w = exp(scores[j]);"),
    ("window_off_by_one", "first = i + (L - Sq) - window + 1;",
     "first = i + (L - Sq) - window;"),
    ("window_ignored", "if (window > 0 && i + (L - Sq) - window + 1 > first)",
     "if (0 && i + (L - Sq) - window + 1 > first)"),
    ("sink_weight_dropped", "l = (sinks != NULL) ? exp(sink - m) : 0.0;", "l = 0.0;"),
    ("sink_not_in_max", "    m = sink;\n", "    m = -INFINITY;\n"),
    ("empty_row_ignores_sink", "*lse_out = sink;               /* -inf without a sink */",
     "*lse_out = -INFINITY;"),
]


def _caught(lib_path):
    def attn(*a, **kw):
        return oracle.attention_fwd(*a, lib_path=lib_path, **kw)
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(attn)
        except AssertionError as e:
            failures.append(f"{pin.__name__}: {e}")
        except Exception as e:  # a crash of the mutant also counts as caught
            failures.append(f"{pin.__name__}: {type(e).__name__}")
    return failures


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique: {name}"
    mutant_src = tmp_path / f"oracle_{name}.c"
    mutant_src.write_text(text.replace(old, new))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                           "-o", str(lib), str(mutant_src), "-lm"])
    failures = _caught(str(lib))
    assert failures, f"no pin caught mutation {name}"
