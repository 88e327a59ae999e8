"""The fused decode-attention oracle against its pins (CPU only)."""
import numpy as np
import pytest
import torch

from attn_oracle_pins import PINS
from helpers import bits
from oracle import gqa_attn, gqa_qk


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_attn_oracle_pin(pin):
    pin(gqa_attn)


def test_attn_oracle_matches_score_then_av_oracles():
    """The fused definition against the two separately pinned oracles chained
    (score-step softmax in fp64, rounded to fp32 as the AV call takes it, then
    the AV sum): they agree to the fp32 rounding of the weights."""
    import oracle
    rng = np.random.default_rng(26)
    B, C, Hq, Hkv, D = 3, 50, 8, 2, 16
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    k = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(torch.bfloat16)
    v = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(torch.bfloat16)
    lens = np.array([50, 17, 0], dtype=np.int32)
    fused = gqa_attn.gqa_attention(q, bits(k), bits(v), "bf16", lens, 0.25)
    attn = gqa_qk.gqa_qk_softmax(q, bits(k), "bf16", lens, 0.25).astype(np.float32)
    chained = oracle.gqa_av(attn, bits(v), "bf16", lens)
    vmax = np.abs(v.to(torch.float64).numpy()).max()
    assert np.allclose(fused, chained, rtol=0, atol=1e-6 * vmax)
    assert np.all(fused[2] == 0.0)
