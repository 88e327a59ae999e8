"""Each plausible mistake planted in a copy of the fused-attention oracle fails a pin.

The mutants are textual edits of the oracle module's source, loaded as a
separate module; the committed oracle is untouched.
"""
import importlib.util

import pytest

from attn_oracle_pins import PINS
from oracle import gqa_attn

MUTANTS = {
    "drop_last_context_row": ("k = decode(k_bits[b, :L, kv_h, :], kv_dtype)       # [L, D]\n            v = decode(v_bits[b, :L, kv_h, :], kv_dtype)",
                              "k = decode(k_bits[b, :L - 1, kv_h, :], kv_dtype)       # [L, D]\n            v = decode(v_bits[b, :L - 1, kv_h, :], kv_dtype)"),
    "kv_head_modulo": ("heads = slice(kv_h * G, (kv_h + 1) * G)",
                       "heads = slice(kv_h, Hq, Hkv)"),
    "v_from_next_head": ("v = decode(v_bits[b, :L, kv_h, :], kv_dtype)",
                         "v = decode(v_bits[b, :L, (kv_h + 1) % Hkv, :], kv_dtype)"),
    "k_from_next_head": ("k = decode(k_bits[b, :L, kv_h, :], kv_dtype)",
                         "k = decode(k_bits[b, :L, (kv_h + 1) % Hkv, :], kv_dtype)"),
    "v_rows_shifted": ("v = decode(v_bits[b, :L, kv_h, :], kv_dtype)",
                       "v = decode(np.roll(v_bits[b, :L, kv_h, :], 1, axis=0), kv_dtype)"),
    "scale_ignored": ("s = scale * (k @ q[b, heads, :].T)", "s = (k @ q[b, heads, :].T)"),
    "softmax_over_heads": ("m = s.max(axis=0)\n            e = np.exp(s - m)\n            w = e / e.sum(axis=0)",
                           "m = s.max(axis=1, keepdims=True)\n            e = np.exp(s - m)\n            w = e / e.sum(axis=1, keepdims=True)"),
    "no_normalisation": ("w = e / e.sum(axis=0)", "w = e"),
    "ignore_seq_lens": ("L = C if seq_lens is None else int(min(max(int(seq_lens[b]), 0), C))",
                        "L = C"),
    "negative_length_not_clamped": ("int(min(max(int(seq_lens[b]), 0), C))",
                                    "int(min(max(int(seq_lens[b]), 1), C))"),
    "bf16_wrong_half": ("(bits.astype(np.uint32) << 16)", "(bits.astype(np.uint32) << 15)"),
    "fp16_read_as_bf16": ('if dtype == "fp16":\n            return bits.view(np.float16).astype(np.float64)',
                          'if dtype == "fp16":\n            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)'),
    "query_heads_reversed": ("s = scale * (k @ q[b, heads, :].T)",
                             "s = scale * (k @ q[b, heads, :][::-1].T)"),
    "weights_transposed_heads": ("out[b, heads, :] = w.T @ v", "out[b, heads, :] = w[:, ::-1].T @ v"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_attn_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(gqa_attn.__file__) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"attn_mutant_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"attn_mutant_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception as e:
            caught.append(f"{pin.__name__}: {type(e).__name__}")
    assert caught, f"mutant {name} passed every pin"
