"""Each plausible mistake planted in a copy of the oracle fails at least one pin.

The mutants are textual edits of a temporary copy of the oracle's C source,
compiled with the same flags; the committed oracle is untouched. This shows
that the pins constrain the oracle's indexing, group mapping, ragged handling,
decoding and accumulation, not only its shape.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

MUTANTS = {
    "drop_last_context_row": ("for (int64_t c = 0; c < L; ++c)",
                              "for (int64_t c = 0; c + 1 < L; ++c)"),
    "kv_head_modulo": ("const int64_t kv_h = q_h / G;",
                       "const int64_t kv_h = q_h % j->Hkv;"),
    "attn_transposed": ("j->attn[(b * j->Cmax + c) * j->Hq + q_h]",
                        "j->attn[(b * j->Hq + q_h) * j->Cmax + c]"),
    "ignore_seq_lens": ("int64_t L = j->seq_lens ? (int64_t)j->seq_lens[b] : j->Cmax;",
                        "int64_t L = j->Cmax;"),
    "fp16_bias_off_by_one": ("mag = ldexp((double)(m + 1024), e - 25);",
                             "mag = ldexp((double)(m + 1024), e - 24);"),
    "fp16_subnormal_scale": ("mag = ldexp((double)m, -24);",
                             "mag = ldexp((double)m, -25);"),
    "fp16_sign_dropped": ("return sign ? -mag : mag;", "return mag;"),
    "bf16_wrong_half": ("uint32_t w = (uint32_t)bits << 16;",
                        "uint32_t w = (uint32_t)bits << 15;"),
    "accumulator_not_reset": ("acc[d] = 0.0;", "(void)0;"),
    "output_transposed": ("double *o = j->out + (b * j->Hq + q_h) * j->D;",
                          "double *o = j->out + (q_h * j->B + b) * j->D;"),
    "v_row_wrong_stride": ("((b * j->Cmax + c) * j->Hkv + kv_h) * j->D",
                           "((b * j->Cmax + c) + kv_h * j->Cmax * j->B) * j->D"),
    "negative_length_not_clamped": ("if (L < 0) L = 0;", "if (L < 0) L = 1;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(path), str(tmp_path / f"lib_{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            pin(orc)
        except Exception as e:  # an assertion, or a pin that could not even run
            caught.append(f"{pin.__name__}: {type(e).__name__}")
    assert caught, f"mutant {name} passed every pin"
