"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each pin is a function of one compiled oracle (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees. ``test_oracle_pins.py`` runs them on
the oracle as committed; ``test_oracle_mutants.py`` runs them on copies with a
planted mistake and requires every mutant to fail at least one pin.

What pins what (definition on the page "pytorch/executorch pull 21063",
summary paragraph, and the GQA-reuse paragraph after it):
- bf16/fp16 decoding: every 16-bit pattern against torch / numpy conversion.
- hand-worked fixture: exact values derived by hand (tests/golden).
- brute force: exact rational sums (fractions.Fraction) on tiny shapes.
- one-hot weights: the output is the selected V row, exactly.
- uniform weights 1/L: the column mean computed by numpy.
- G = 1: a plain per-head GEMV computed with numpy matmul.
- invariants: identical weights within a group give identical outputs;
  linearity in attn; joint permutation of context positions; ragged equals
  truncated; zero length gives zeros; lengths are clamped to [0, Cmax].
"""
from fractions import Fraction

import numpy as np
import torch

from helpers import bits, decoded, load_golden, rand_case, TORCH_V


def _run(orc, attn, v, seq_lens, v_dtype, nthreads=1):
    sl = None if seq_lens is None else seq_lens.numpy()
    return orc.gqa_av(attn.numpy(), bits(v), v_dtype, sl, nthreads)


def pin_decode_all_patterns(orc):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for vd in ("bf16", "fp16"):
        ref = torch.from_numpy(allbits.view(np.int16).copy()).view(TORCH_V[vd]).to(torch.float64).numpy()
        got = np.array([orc.decode(int(b), vd) for b in allbits])
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan), f"{vd}: NaN patterns differ"
        assert np.array_equal(got[~nan], ref[~nan]), f"{vd}: decoded values differ"
        # Through the reduction: one context row with weight 1, D = 65536 columns.
        v = torch.from_numpy(allbits.view(np.int16).copy()).view(TORCH_V[vd]).reshape(1, 1, 1, 65536)
        attn = torch.ones((1, 1, 1), dtype=torch.float32)
        out = _run(orc, attn, v, None, vd)[0, 0]
        assert np.array_equal(np.isnan(out), nan)
        assert np.array_equal(out[~nan], ref[~nan]), f"{vd}: 1*V through the sum differs"


def pin_hand_worked(orc):
    for vd in ("bf16", "fp16"):
        g = load_golden("hand_worked_b2_c3_hq4_hkv2_d2.json", vd)
        out = _run(orc, g["attn"], g["v"], g["seq_lens"], vd)
        assert np.array_equal(out, g["out"]), f"{vd}: hand-worked values differ:\n{out}"


def pin_brute_force(orc):
    rng = np.random.default_rng(1234)
    shapes = [(1, 1, 1, 1, 1), (2, 5, 4, 2, 3), (2, 9, 6, 3, 8), (1, 7, 6, 1, 4),
              (2, 4, 6, 6, 2), (2, 8, 4, 4, 5)]
    for (B, C, Hq, Hkv, D) in shapes:
        for vd in ("bf16", "fp16"):
            lens = rng.integers(-1, C + 2, size=B)  # includes clamped values
            attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, vd, lens)
            out = _run(orc, attn, v, sl, vd)
            a = attn.numpy().astype(np.float64)
            vv = decoded(v)
            G = Hq // Hkv
            for b in range(B):
                L = max(0, min(int(lens[b]), C))
                for q in range(Hq):
                    for d in range(D):
                        terms = [Fraction(float(a[b, c, q])) * Fraction(float(vv[b, c, q // G, d]))
                                 for c in range(L)]
                        exact = sum(terms, Fraction(0))
                        bound = (L + 1) * 2.0 ** -53 * float(sum(abs(t) for t in terms))
                        assert np.isfinite(out[b, q, d]), "non-finite oracle output"
                        err = abs(Fraction(float(out[b, q, d])) - exact)
                        assert err <= Fraction(bound), (
                            f"brute force mismatch at {(B, C, Hq, Hkv, D, vd)} b={b} q={q} d={d}: "
                            f"{out[b, q, d]} vs {float(exact)}")


def pin_one_hot(orc):
    rng = np.random.default_rng(7)
    B, C, Hq, Hkv, D = 2, 13, 12, 3, 16
    for vd in ("bf16", "fp16"):
        attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, vd, [13, 9])
        vv = decoded(v)
        G = Hq // Hkv
        for c0 in (0, 4, 8):
            a = torch.zeros((B, C, Hq), dtype=torch.float32)
            a[:, c0, :] = 1.0
            out = _run(orc, a, v, sl, vd)
            for b in range(B):
                for q in range(Hq):
                    assert np.array_equal(out[b, q], vv[b, c0, q // G]), (vd, c0, b, q)


def pin_uniform_mean(orc):
    rng = np.random.default_rng(8)
    B, C, Hq, Hkv, D = 2, 20, 8, 2, 24
    for vd in ("bf16", "fp16"):
        for L in (1, 4, 16):
            attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, vd, [L, L])
            a = torch.zeros((B, C, Hq), dtype=torch.float32)
            a[:, :L, :] = 1.0 / L
            out = _run(orc, a, v, sl, vd)
            vv = decoded(v)
            G = Hq // Hkv
            for b in range(B):
                for q in range(Hq):
                    mean = vv[b, :L, q // G, :].mean(axis=0)
                    assert np.allclose(out[b, q], mean, rtol=1e-12, atol=1e-14), (vd, L, b, q)


def pin_g1_is_mha_gemv(orc):
    rng = np.random.default_rng(9)
    B, C, H, D = 3, 17, 5, 12
    for vd in ("bf16", "fp16"):
        attn, v, sl = rand_case(rng, B, C, H, H, D, vd, [17, 3, 11])
        out = _run(orc, attn, v, sl, vd)
        a = attn.numpy().astype(np.float64)
        vv = decoded(v)
        for b in range(B):
            L = int(sl[b])
            for h in range(H):
                ref = a[b, :L, h] @ vv[b, :L, h, :]
                assert np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-13), (vd, b, h)


def pin_identical_weights_identical_outputs(orc):
    rng = np.random.default_rng(10)
    B, C, Hq, Hkv, D = 2, 11, 12, 3, 8
    G = Hq // Hkv
    for vd in ("bf16", "fp16"):
        attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, vd, [11, 6])
        for k in range(Hkv):
            for g in range(1, G):
                attn[:, :, k * G + g] = attn[:, :, k * G]
        out = _run(orc, attn, v, sl, vd)
        for k in range(Hkv):
            for g in range(1, G):
                assert np.array_equal(out[:, k * G + g], out[:, k * G]), (vd, k, g)
        # And different weights within a group give different outputs.
        attn2 = attn.clone()
        attn2[:, :6, 1] += 1.0
        out2 = _run(orc, attn2, v, sl, vd)
        assert not np.array_equal(out2[:, 1], out2[:, 0])


def pin_linearity(orc):
    rng = np.random.default_rng(11)
    B, C, Hq, Hkv, D = 2, 15, 6, 2, 8
    for vd in ("bf16", "fp16"):
        _, v, sl = rand_case(rng, B, C, Hq, Hkv, D, vd, [15, 10], pad_nan=False)
        # Weights k/1024 with |k| < 2^12: 2*a1 - 0.5*a2 is exact in fp32.
        a1 = torch.tensor(rng.integers(-4095, 4096, (B, C, Hq)) / 1024.0, dtype=torch.float32)
        a2 = torch.tensor(rng.integers(-4095, 4096, (B, C, Hq)) / 1024.0, dtype=torch.float32)
        a3 = 2.0 * a1 - 0.5 * a2
        assert torch.equal(a3.double(), 2.0 * a1.double() - 0.5 * a2.double())
        f1, f2, f3 = (_run(orc, a, v, sl, vd) for a in (a1, a2, a3))
        assert np.allclose(f3, 2.0 * f1 - 0.5 * f2, rtol=1e-12, atol=1e-12)


def pin_permutation(orc):
    rng = np.random.default_rng(12)
    B, C, Hq, Hkv, D = 1, 19, 8, 4, 8
    for vd in ("bf16", "fp16"):
        attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, vd, [19])
        perm = torch.from_numpy(rng.permutation(C))
        out = _run(orc, attn, v, sl, vd)
        outp = _run(orc, attn[:, perm], v[:, perm], sl, vd)
        assert np.allclose(out, outp, rtol=1e-12, atol=1e-13)
        assert not np.array_equal(_run(orc, attn[:, perm], v, sl, vd), out)


def pin_ragged_equals_truncated(orc):
    rng = np.random.default_rng(13)
    B, C, Hq, Hkv, D = 3, 16, 6, 3, 8
    lens = [16, 5, 0]
    for vd in ("bf16", "fp16"):
        attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, vd, lens)  # NaN padding
        out = _run(orc, attn, v, sl, vd)
        assert np.all(np.isfinite(out))
        for b, L in enumerate(lens):
            ref = _run(orc, attn[b:b + 1, :L].contiguous(), v[b:b + 1, :L].contiguous(), None, vd)
            assert np.array_equal(out[b], ref[0]), (vd, b)
        assert np.array_equal(out[2], np.zeros((Hq, D)))


def pin_length_clamping(orc):
    rng = np.random.default_rng(14)
    B, C, Hq, Hkv, D = 2, 6, 4, 2, 8
    attn, v, _ = rand_case(rng, B, C, Hq, Hkv, D, "bf16", [6, 6], pad_nan=False)
    full = _run(orc, attn, v, None, "bf16")
    over = _run(orc, attn, v, torch.tensor([7, 1 << 30], dtype=torch.int32), "bf16")
    assert np.array_equal(full, over)
    neg = _run(orc, attn, v, torch.tensor([-1, -(1 << 30)], dtype=torch.int32), "bf16")
    assert np.array_equal(neg, np.zeros_like(neg))


def pin_threads_bitwise(orc):
    rng = np.random.default_rng(15)
    attn, v, sl = rand_case(rng, 3, 33, 8, 2, 16, "fp16")
    one = _run(orc, attn, v, sl, "fp16", 1)
    many = _run(orc, attn, v, sl, "fp16", 7)
    assert np.array_equal(one, many)


PINS = [pin_decode_all_patterns, pin_hand_worked, pin_brute_force, pin_one_hot,
        pin_uniform_mean, pin_g1_is_mha_gemv, pin_identical_weights_identical_outputs,
        pin_linearity, pin_permutation, pin_ragged_equals_truncated, pin_length_clamping,
        pin_threads_bitwise]
