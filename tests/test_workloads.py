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


@pytest.mark.parametrize("pad", ["zero", "nan"])
def test_fused_attention_inputs(pad):
    """generate_qkv: V and lengths as generate() draws them, K of the same
    shape and type from the next seed with the same padding, q spread like the
    workload's logits; deterministic."""
    w = W.custom(3, 80, 8, 2, 16, v_dtype="bf16", logit_sigma=3.0, len_lo=0, len_hi=80)
    x = W.generate_qkv(w, pad=pad)
    g = W.generate(w, pad=pad)
    assert set(x) == {"q", "k", "v", "seq_lens"}
    assert torch.equal(x["seq_lens"], g["seq_lens"])
    assert torch.equal(x["v"].view(torch.int16), g["v"].view(torch.int16))
    assert x["k"].shape == x["v"].shape and x["k"].dtype == x["v"].dtype
    assert not torch.equal(x["k"].view(torch.int16), x["v"].view(torch.int16))
    assert x["q"].shape == (3, 8, 16) and x["q"].dtype == torch.float32
    for b, L in enumerate(x["seq_lens"].tolist()):
        tail = x["k"][b, L:].float()
        assert torch.all(tail == 0) if pad == "zero" else torch.all(torch.isnan(tail))
        assert not torch.isnan(x["k"][b, :L].float()).any()
    y = W.generate_qkv(w, pad=pad)
    for k in ("q", "k", "v", "seq_lens"):
        a, b = x[k], y[k]
        if a.is_floating_point():
            a, b = a.view(torch.uint8), b.view(torch.uint8)
        assert torch.equal(a, b)
    big = W.generate_qkv(W.custom(1, 2048, 16, 1, 64, logit_sigma=2.0))
    assert abs(big["q"].std().item() - 2.0) < 0.1


def test_fused_attention_compulsory_bytes():
    llama = W.get("llama")
    # K and V rows once (2 x 8192 x 8 x 128 x 2 B), q and out (2 x 32 x 128 x 4 B), seq_lens.
    assert W.attention_compulsory_bytes(llama, [8192]) == 33_587_204
    assert W.attention_flops(llama, [8192]) == 4 * 8192 * 32 * 128
