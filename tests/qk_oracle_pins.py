"""Pins of the score-step oracle against facts fixed outside the oracle itself.

Each pin takes the oracle's two functions (``decode``, ``gqa_qk_softmax``, as a
module or an object with those attributes) and raises AssertionError on a
disagreement. ``test_qk_oracle_pins.py`` runs them on the committed oracle;
``test_qk_oracle_mutants.py`` on copies with a planted mistake, each of which
must fail at least one pin.

What pins what:
- decoding: every 16-bit pattern against torch's bf16/fp16 conversion.
- brute force: the definition evaluated with 50-digit decimal arithmetic
  (decimal.Decimal.exp) on tiny shapes.
- G = 1: scipy.special.softmax of a numpy matrix-vector product per head.
- closed forms: a zero query or equal K rows give 1/L; one score far above
  the others gives a one-hot row; every row sums to 1.
- the group mapping: K rows built so that KV head j peaks at position j.
- invariants: joint permutation of positions; ragged equals truncated; a
  constant added to every score (through an extra K column) changes nothing;
  scale s with q equals scale 1 with s*q (s a power of two); lengths clamp
  to [0, Cmax] and a zero length leaves zeros.
"""
from decimal import Decimal, getcontext

import numpy as np
import torch

from helpers import TORCH_V, bits


def _k(rng, B, C, Hkv, D, kd, sigma=1.0):
    t = torch.tensor(rng.standard_normal((B, C, Hkv, D)) * sigma, dtype=torch.float32)
    return t.to(TORCH_V[kd])


def _q(rng, B, Hq, D, sigma=1.0):
    return (rng.standard_normal((B, Hq, D)) * sigma).astype(np.float32)


def pin_decode_all_patterns(orc):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for kd in ("bf16", "fp16"):
        ref = torch.from_numpy(allbits.view(np.int16).copy()).view(TORCH_V[kd]).to(torch.float64).numpy()
        got = orc.decode(allbits, kd)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan), f"{kd}: NaN patterns differ"
        assert np.array_equal(got[~nan], ref[~nan]), f"{kd}: decoded values differ"


def pin_decimal_brute_force(orc):
    getcontext().prec = 50
    rng = np.random.default_rng(11)
    for B, C, Hq, Hkv, D, kd in ((1, 5, 2, 1, 4, "bf16"), (2, 7, 4, 2, 8, "fp16"),
                                 (2, 3, 6, 3, 2, "bf16")):
        q = _q(rng, B, Hq, D)
        k = _k(rng, B, C, Hkv, D, kd)
        lens = rng.integers(1, C + 1, size=B)
        scale = 0.375
        got = orc.gqa_qk_softmax(q, bits(k), kd, lens, scale)
        kv = k.to(torch.float64).numpy()
        G = Hq // Hkv
        for b in range(B):
            L = int(lens[b])
            for h in range(Hq):
                s = [Decimal(scale) * sum(Decimal(float(q[b, h, d])) * Decimal(float(kv[b, c, h // G, d]))
                                          for d in range(D)) for c in range(L)]
                m = max(s)
                e = [(x - m).exp() for x in s]
                tot = sum(e)
                for c in range(L):
                    want = float(e[c] / tot)
                    assert abs(got[b, c, h] - want) <= 4e-16, (B, C, Hq, b, c, h, got[b, c, h], want)
                assert np.all(got[b, L:, h] == 0.0)


def pin_mha_matches_scipy_softmax(orc):
    from scipy.special import softmax
    rng = np.random.default_rng(12)
    B, C, H, D = 2, 40, 3, 16
    q = _q(rng, B, H, D)
    k = _k(rng, B, C, H, D, "bf16")
    got = orc.gqa_qk_softmax(q, bits(k), "bf16", None, 0.25)
    kv = k.to(torch.float64).numpy()
    for b in range(B):
        for h in range(H):
            want = softmax(0.25 * (kv[b, :, h, :] @ q[b, h].astype(np.float64)))
            assert np.allclose(got[b, :, h], want, rtol=1e-13, atol=1e-16)


def pin_closed_forms(orc):
    rng = np.random.default_rng(13)
    B, C, Hq, Hkv, D = 2, 24, 4, 2, 8
    k = _k(rng, B, C, Hkv, D, "bf16")
    lens = np.array([24, 16])
    zero = orc.gqa_qk_softmax(np.zeros((B, Hq, D), np.float32), bits(k), "bf16", lens, 1.0)
    for b in range(B):
        assert np.all(zero[b, :lens[b]] == 1.0 / lens[b]), "zero query is not uniform"
    same = k.clone()
    same[:, :, :, :] = same[:, :1, :, :]
    q = _q(rng, B, Hq, D)
    eq = orc.gqa_qk_softmax(q, bits(same), "bf16", lens, 1.0)
    for b in range(B):
        assert np.allclose(eq[b, :lens[b]], 1.0 / lens[b], rtol=0, atol=1e-15), "equal rows"
    a = orc.gqa_qk_softmax(q, bits(k), "bf16", lens, 1.0)
    for b in range(B):
        assert np.allclose(a[b, :lens[b]].sum(axis=0), 1.0, rtol=0, atol=1e-14), "rows do not sum to 1"
    # One position far above the others: a one-hot row.
    big = k.clone()
    big[:, 5] = 64.0
    ones = np.ones((B, Hq, D), np.float32)
    oh = orc.gqa_qk_softmax(ones, bits(big), "bf16", lens, 1.0)
    assert np.all(oh[:, 5] == 1.0) and np.all(oh[:, :5] < 1e-100), "one-hot row"


def pin_group_mapping(orc):
    B, C, Hkv, G, D = 1, 6, 3, 2, 4
    k = torch.zeros((B, C, Hkv, D), dtype=torch.float32)
    for j in range(Hkv):
        k[0, j, j, :] = 8.0           # KV head j peaks at position j
    k = k.to(torch.bfloat16)
    q = np.ones((B, Hkv * G, D), np.float32)
    a = orc.gqa_qk_softmax(q, bits(k), "bf16", None, 1.0)
    for h in range(Hkv * G):
        assert int(np.argmax(a[0, :, h])) == h // G, f"query head {h} reads the wrong KV head"


def pin_invariants(orc):
    rng = np.random.default_rng(14)
    B, C, Hq, Hkv, D = 2, 30, 6, 2, 8
    q = _q(rng, B, Hq, D)
    k = _k(rng, B, C, Hkv, D, "fp16")
    base = orc.gqa_qk_softmax(q, bits(k), "fp16", None, 0.5)
    perm = rng.permutation(C)
    pk = orc.gqa_qk_softmax(q, bits(k[:, perm]), "fp16", None, 0.5)
    assert np.allclose(pk, base[:, perm], rtol=1e-13, atol=1e-16), "permutation"
    lens = np.array([17, 30])
    rag = orc.gqa_qk_softmax(q, bits(k), "fp16", lens, 0.5)
    trunc = orc.gqa_qk_softmax(q[:1], bits(k[:1, :17]), "fp16", None, 0.5)
    assert np.array_equal(rag[0, :17], trunc[0]) and np.all(rag[0, 17:] == 0), "ragged"
    # A constant added to every score through an extra K column.
    k2 = torch.cat([k, torch.full((B, C, Hkv, 1), 2.0, dtype=k.dtype)], dim=3)
    q2 = np.concatenate([q, np.full((B, Hq, 1), 3.0, np.float32)], axis=2)
    shifted = orc.gqa_qk_softmax(q2, bits(k2), "fp16", None, 0.5)
    assert np.allclose(shifted, base, rtol=1e-12, atol=1e-16), "shift invariance"
    folded = orc.gqa_qk_softmax(q * 2.0, bits(k), "fp16", None, 0.25)
    assert np.array_equal(folded, base), "scale folding"


def pin_lengths_clamped(orc):
    rng = np.random.default_rng(15)
    B, C, Hq, Hkv, D = 3, 10, 2, 1, 8
    q = _q(rng, B, Hq, D)
    k = _k(rng, B, C, Hkv, D, "bf16")
    full = orc.gqa_qk_softmax(q, bits(k), "bf16", None, 1.0)
    over = orc.gqa_qk_softmax(q, bits(k), "bf16", np.array([10, 11, 1 << 30]), 1.0)
    assert np.array_equal(over, full), "lengths above Cmax"
    neg = orc.gqa_qk_softmax(q, bits(k), "bf16", np.array([0, -3, -(1 << 30)]), 1.0)
    assert np.all(neg == 0.0), "non-positive lengths"


PINS = [pin_decode_all_patterns, pin_decimal_brute_force, pin_mha_matches_scipy_softmax,
        pin_closed_forms, pin_group_mapping, pin_invariants, pin_lengths_clamped]
