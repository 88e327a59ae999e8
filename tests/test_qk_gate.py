"""The score-step parity gate (tests/helpers.py, qk_gate) is a real check.

Run on the oracle's own output for a workload-length case, with no GPU: the
output rounded to fp32 (what the kernels return) passes, and the same output
with the weights of one context split scaled by 1.01 (what a split-merge bug
that mis-weights one split would produce) fails, although it stays within an
absolute 1e-4 of the oracle everywhere.
"""
import numpy as np
import torch

from oracle import gqa_qk
from helpers import bits, qk_gate, qk_gate_errors

import pytest


@pytest.fixture(scope="module")
def case():
    rng = np.random.default_rng(21)
    B, C, Hq, Hkv, D = 2, 8192, 8, 2, 64
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    k = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(torch.bfloat16)
    lens = np.array([8192, 5000], dtype=np.int32)
    ref = gqa_qk.gqa_qk_softmax(q, bits(k), "bf16", lens, D ** -0.5)
    return ref, lens


def test_gate_accepts_the_oracle_rounded_to_fp32(case):
    ref, lens = case
    got = ref.astype(np.float32).astype(np.float64)
    e = qk_gate(got, ref, lens, "fp32-rounded oracle")
    assert e["rel"] < 1e-7


@pytest.mark.parametrize("split", [(0, 448), (3584, 4032), (4800, 5000)])
def test_gate_rejects_one_split_scaled_by_one_percent(case, split):
    ref, lens = case
    got = ref.astype(np.float32).astype(np.float64)
    s0, s1 = split
    got[1, s0:s1] *= 1.01
    # An absolute 1e-4 bound would not see it: the probabilities are ~1e-4.
    assert float(np.abs(got - ref).max()) < 1e-4
    e = qk_gate_errors(got, ref, lens)
    assert e["ratio"] > 1.0 and e["rel"] > 0.009
    with pytest.raises(AssertionError):
        qk_gate(got, ref, lens, "one split scaled by 1.01")


def test_gate_rejects_a_row_that_does_not_sum_to_one(case):
    ref, lens = case
    got = ref.astype(np.float32).astype(np.float64)
    # Every probability of one row 3e-5 high: inside the element bound, but
    # the row then sums to 1 + 3e-5.
    got[0, :, 3] *= 1.0 + 3e-5
    e = qk_gate_errors(got, ref, lens)
    assert e["ratio"] <= 1.0 and e["row_sum"] > 1e-5
    with pytest.raises(AssertionError):
        qk_gate(got, ref, lens, "a row scaled by 1 + 3e-5")
