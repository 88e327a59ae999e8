"""The seeded input generator: shapes, determinism, lengths and padding (CPU)."""
import math

import pytest
import torch

from gqa_attention_weighted_gb300 import workloads as W


def test_five_decode_shapes():
    names = [W.get(a).name for a in ("small", "llama", "phi", "mqa", "large")]
    assert len(set(names)) == 5
    assert W.get("mqa").G == 16 and W.get("phi").G == 3 and W.get("large").G == 8


def test_deterministic_and_seeded():
    w = W.custom(2, 40, 6, 2, 16, len_lo=5, len_hi=40)
    a = W.generate(w)
    b = W.generate(w)
    c = W.generate(w, seed=1)
    for k in ("attn", "v", "seq_lens"):
        assert torch.equal(a[k].view(torch.uint8) if a[k].is_floating_point() else a[k],
                           b[k].view(torch.uint8) if b[k].is_floating_point() else b[k])
    assert not torch.equal(a["v"], c["v"])


@pytest.mark.parametrize("pad", ["zero", "nan"])
def test_lengths_softmax_and_padding(pad):
    w = W.custom(4, 64, 8, 2, 8, v_dtype="fp16", len_lo=0, len_hi=64)
    x = W.generate(w, pad=pad)
    assert x["attn"].shape == (4, 64, 8) and x["attn"].dtype == torch.float32
    assert x["v"].shape == (4, 64, 2, 8) and x["v"].dtype == torch.float16
    assert x["seq_lens"].dtype == torch.int32
    for b, L in enumerate(x["seq_lens"].tolist()):
        assert 0 <= L <= 64
        if L:
            s = x["attn"][b, :L].double().sum(0)
            assert torch.allclose(s, torch.ones_like(s), atol=1e-5)
            assert torch.all(x["attn"][b, :L] >= 0)
        tail_a, tail_v = x["attn"][b, L:], x["v"][b, L:]
        if pad == "zero":
            assert torch.all(tail_a == 0) and torch.all(tail_v == 0)
        else:
            assert torch.all(torch.isnan(tail_a)) and torch.all(torch.isnan(tail_v))


def test_value_spread():
    w = W.custom(1, 4096, 4, 1, 64, v_sigma=0.5)
    x = W.generate(w)
    std = x["v"].float().std().item()
    assert abs(std - 0.5) < 0.01


def test_compulsory_bytes_of_the_two_dense_shapes():
    small, llama = W.get("small"), W.get("llama")
    assert W.compulsory_bytes(small, [512]) == 149_508
    assert W.compulsory_bytes(llama, [8192]) == 17_842_180
    assert W.flops(llama, [8192]) == 2 * 8192 * 32 * 128
