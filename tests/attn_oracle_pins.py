"""Pins of the fused decode-attention oracle against facts fixed outside it.

Each pin takes the oracle (a module or an object with ``decode`` and
``gqa_attention``) and raises AssertionError on a disagreement.
``test_attn_oracle_pins.py`` runs them on the committed oracle;
``test_attn_oracle_mutants.py`` on copies with a planted mistake, each of
which must fail at least one pin.

What pins what:
- brute force: the definition evaluated with 50-digit decimal arithmetic
  (decimal.Decimal.exp) on tiny shapes.
- G = 1: scipy.special.softmax of a matrix-vector product, then the weighted
  sum of V rows, per head.
- closed forms: a zero query gives the column mean of V (numpy.mean); one
  score far above the others returns that V row exactly; V rows that are all
  equal come back unchanged (the weights sum to 1).
- the group mapping: V of KV head j holds the constant j + 1 and K makes
  every query head prefer a different row, so each output is its KV head's
  constant; a second case makes K and V disagree on the head if either is
  taken from the wrong one.
- invariants: joint permutation of positions; ragged equals truncated; a
  constant added to every score changes nothing; scale folding into q;
  lengths clamp to [0, Cmax] and a zero length gives zeros.
"""
from decimal import Decimal, getcontext

import numpy as np
import torch

from helpers import TORCH_V, bits


def _kv(rng, B, C, Hkv, D, kd, sigma=1.0):
    t = torch.tensor(rng.standard_normal((B, C, Hkv, D)) * sigma, dtype=torch.float32)
    return t.to(TORCH_V[kd])


def _q(rng, B, Hq, D, sigma=1.0):
    return (rng.standard_normal((B, Hq, D)) * sigma).astype(np.float32)


def pin_decimal_brute_force(orc):
    getcontext().prec = 50
    rng = np.random.default_rng(21)
    for B, C, Hq, Hkv, D, kd in ((1, 5, 2, 1, 4, "bf16"), (2, 7, 4, 2, 8, "fp16"),
                                 (2, 3, 6, 3, 2, "bf16")):
        q = _q(rng, B, Hq, D)
        k = _kv(rng, B, C, Hkv, D, kd)
        v = _kv(rng, B, C, Hkv, D, kd)
        lens = rng.integers(1, C + 1, size=B)
        scale = 0.375
        got = orc.gqa_attention(q, bits(k), bits(v), kd, lens, scale)
        kf = k.to(torch.float64).numpy()
        vf = v.to(torch.float64).numpy()
        G = Hq // Hkv
        for b in range(B):
            L = int(lens[b])
            for h in range(Hq):
                s = [Decimal(scale) * sum(Decimal(float(q[b, h, d])) * Decimal(float(kf[b, c, h // G, d]))
                                          for d in range(D)) for c in range(L)]
                m = max(s)
                e = [(x - m).exp() for x in s]
                tot = sum(e)
                for d in range(D):
                    want = float(sum(e[c] * Decimal(float(vf[b, c, h // G, d])) for c in range(L)) / tot)
                    assert abs(got[b, h, d] - want) <= 1e-15 * max(1.0, abs(want)), (b, h, d, got[b, h, d], want)


def pin_mha_matches_scipy(orc):
    from scipy.special import softmax
    rng = np.random.default_rng(22)
    B, C, H, D = 2, 40, 3, 16
    q = _q(rng, B, H, D)
    k = _kv(rng, B, C, H, D, "bf16")
    v = _kv(rng, B, C, H, D, "bf16")
    got = orc.gqa_attention(q, bits(k), bits(v), "bf16", None, 0.25)
    kf = k.to(torch.float64).numpy()
    vf = v.to(torch.float64).numpy()
    for b in range(B):
        for h in range(H):
            w = softmax(0.25 * (kf[b, :, h, :] @ q[b, h].astype(np.float64)))
            want = np.einsum("c,cd->d", w, vf[b, :, h, :])
            assert np.allclose(got[b, h], want, rtol=1e-13, atol=1e-15)


def pin_closed_forms(orc):
    rng = np.random.default_rng(23)
    B, C, Hq, Hkv, D = 2, 24, 4, 2, 8
    k = _kv(rng, B, C, Hkv, D, "bf16")
    v = _kv(rng, B, C, Hkv, D, "bf16")
    lens = np.array([24, 16])
    vf = v.to(torch.float64).numpy()
    G = Hq // Hkv
    zero = orc.gqa_attention(np.zeros((B, Hq, D), np.float32), bits(k), bits(v), "bf16", lens, 1.0)
    for b in range(B):
        for h in range(Hq):
            want = np.mean(vf[b, :lens[b], h // G, :], axis=0)
            assert np.allclose(zero[b, h], want, rtol=0, atol=1e-15), "zero query is not the mean"
    # One position far above the others: that V row, exactly.
    big = k.clone()
    big[:, 5] = 64.0
    ones = np.ones((B, Hq, D), np.float32)
    oh = orc.gqa_attention(ones, bits(big), bits(v), "bf16", lens, 1.0)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(oh[b, h], vf[b, 5, h // G]), "one dominant score"
    # Equal V rows: out is that row whatever the weights.
    same = v.clone()
    same[:, :, :, :] = same[:, :1, :, :]
    q = _q(rng, B, Hq, D)
    eq = orc.gqa_attention(q, bits(k), bits(same), "bf16", lens, 1.0)
    sf = same.to(torch.float64).numpy()
    for b in range(B):
        for h in range(Hq):
            assert np.allclose(eq[b, h], sf[b, 0, h // G], rtol=1e-14, atol=0), "equal rows"


def pin_group_mapping(orc):
    B, C, Hkv, G, D = 1, 8, 3, 2, 4    # C a power of two: the uniform weights are exact
    k = torch.zeros((B, C, Hkv, D), dtype=torch.float32)
    v = torch.zeros((B, C, Hkv, D), dtype=torch.float32)
    for j in range(Hkv):
        v[0, :, j, :] = j + 1.0        # KV head j holds the constant j + 1
    q = np.ones((B, Hkv * G, D), np.float32)
    out = orc.gqa_attention(q, bits(k.to(torch.bfloat16)), bits(v.to(torch.bfloat16)), "bf16", None, 1.0)
    for h in range(Hkv * G):
        assert np.all(out[0, h] == h // G + 1.0), f"query head {h} reads the wrong V head"
    # K of KV head j peaks at row j and V row c holds c: each output is its KV head's row.
    for j in range(Hkv):
        k[0, j, j, :] = 64.0
    vr = torch.arange(C, dtype=torch.float32).view(1, C, 1, 1).expand(B, C, Hkv, D).contiguous()
    # (scale 4: the other rows' scores are 1024 lower, so their weights underflow to 0)
    out = orc.gqa_attention(q, bits(k.to(torch.bfloat16)), bits(vr.to(torch.bfloat16)), "bf16", None, 4.0)
    for h in range(Hkv * G):
        assert np.all(out[0, h] == float(h // G)), f"query head {h} takes K from the wrong head"


def pin_invariants(orc):
    rng = np.random.default_rng(24)
    B, C, Hq, Hkv, D = 2, 30, 6, 2, 8
    q = _q(rng, B, Hq, D)
    k = _kv(rng, B, C, Hkv, D, "fp16")
    v = _kv(rng, B, C, Hkv, D, "fp16")
    base = orc.gqa_attention(q, bits(k), bits(v), "fp16", None, 0.5)
    perm = rng.permutation(C)
    pk = orc.gqa_attention(q, bits(k[:, perm]), bits(v[:, perm]), "fp16", None, 0.5)
    assert np.allclose(pk, base, rtol=1e-12, atol=1e-15), "permutation"
    lens = np.array([17, 30])
    rag = orc.gqa_attention(q, bits(k), bits(v), "fp16", lens, 0.5)
    trunc = orc.gqa_attention(q[:1], bits(k[:1, :17]), bits(v[:1, :17]), "fp16", None, 0.5)
    assert np.array_equal(rag[0], trunc[0]) and np.array_equal(rag[1], base[1]), "ragged"
    # A constant added to every score through an extra K column (V gets one too).
    k2 = torch.cat([k, torch.full((B, C, Hkv, 1), 2.0, dtype=k.dtype)], dim=3)
    v2 = torch.cat([v, torch.zeros((B, C, Hkv, 1), dtype=v.dtype)], dim=3)
    q2 = np.concatenate([q, np.full((B, Hq, 1), 3.0, np.float32)], axis=2)
    shifted = orc.gqa_attention(q2, bits(k2), bits(v2), "fp16", None, 0.5)
    assert np.allclose(shifted[:, :, :D], base, rtol=1e-12, atol=1e-15), "shift invariance"
    folded = orc.gqa_attention(q * 2.0, bits(k), bits(v), "fp16", None, 0.25)
    assert np.array_equal(folded, base), "scale folding"


def pin_lengths_clamped(orc):
    rng = np.random.default_rng(25)
    B, C, Hq, Hkv, D = 3, 10, 2, 1, 8
    q = _q(rng, B, Hq, D)
    k = _kv(rng, B, C, Hkv, D, "bf16")
    v = _kv(rng, B, C, Hkv, D, "bf16")
    full = orc.gqa_attention(q, bits(k), bits(v), "bf16", None, 1.0)
    over = orc.gqa_attention(q, bits(k), bits(v), "bf16", np.array([10, 11, 1 << 30]), 1.0)
    assert np.array_equal(over, full), "lengths above Cmax"
    neg = orc.gqa_attention(q, bits(k), bits(v), "bf16", np.array([0, -3, -(1 << 30)]), 1.0)
    assert np.all(neg == 0.0), "non-positive lengths"
    one = orc.gqa_attention(q, bits(k), bits(v), "bf16", np.array([1, 1, 1]), 1.0)
    vf = v.to(torch.float64).numpy()
    assert np.array_equal(one, np.repeat(vf[:, 0], Hq, axis=1)), "one row is that row"


PINS = [pin_decimal_brute_force, pin_mha_matches_scipy, pin_closed_forms, pin_group_mapping,
        pin_invariants, pin_lengths_clamped]
