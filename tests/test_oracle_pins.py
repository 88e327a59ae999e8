"""The committed oracle passes every pin (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_rejects_bad_arguments(orc):
    attn = np.zeros((1, 2, 6), np.float32)
    v = np.zeros((1, 2, 4, 8), np.uint16)  # Hq=6 is not a multiple of Hkv=4
    with pytest.raises(ValueError):
        orc.gqa_av(attn, v, "bf16")
    rc = orc.lib.oracle_gqa_av(None, None, 0, None, None, 1, 1, 1, 1, 1, 1)
    assert rc == -1
    rc = orc.lib.oracle_gqa_av(attn.ctypes.data, v.ctypes.data, 5, None,
                               np.zeros(8).ctypes.data, 1, 2, 4, 4, 2, 1)
    assert rc == -1  # unknown v_dtype


def test_empty_batch(orc):
    out = orc.gqa_av(np.zeros((0, 4, 2), np.float32), np.zeros((0, 4, 1, 8), np.uint16), "bf16")
    assert out.shape == (0, 2, 8)


def test_zero_context(orc):
    out = orc.gqa_av(np.zeros((2, 0, 4), np.float32), np.zeros((2, 0, 2, 8), np.uint16), "fp16")
    assert np.array_equal(out, np.zeros((2, 4, 8)))
