"""Test helpers: tensor <-> numpy marshalling and the golden fixtures."""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TORCH_V = {"bf16": torch.bfloat16, "fp16": torch.float16}


def bits(v: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a bf16/fp16 tensor as a numpy uint16 array."""
    return v.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def decoded(v: torch.Tensor) -> np.ndarray:
    """Values of a bf16/fp16 tensor in float64, converted by torch."""
    return v.detach().cpu().to(torch.float64).numpy()


def _num(x):
    return float("nan") if x == "nan" else float(x)


def load_golden(name: str, v_dtype: str = "bf16"):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    v = torch.tensor(np.vectorize(_num)(np.array(g["v"], dtype=object)).astype(np.float64),
                     dtype=torch.float64).to(TORCH_V[v_dtype])
    attn = torch.tensor(np.vectorize(_num)(np.array(g["attn"], dtype=object)).astype(np.float64),
                        dtype=torch.float32)
    seq_lens = torch.tensor(g["seq_lens"], dtype=torch.int32)
    out = np.array(g["out"], dtype=np.float64)
    return {"attn": attn, "v": v, "seq_lens": seq_lens, "out": out, "shape": g["shape"]}


def rand_case(rng: np.random.Generator, B, C, Hq, Hkv, D, v_dtype="bf16", lens=None,
              pad_nan=True):
    """Small random case drawn with numpy (for oracle pins)."""
    v = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(TORCH_V[v_dtype])
    attn = torch.tensor(rng.standard_normal((B, C, Hq)), dtype=torch.float32)
    if lens is None:
        lens = rng.integers(0, C + 1, size=B)
    seq_lens = torch.tensor(np.asarray(lens), dtype=torch.int32)
    if pad_nan:
        for b in range(B):
            L = max(0, min(int(lens[b]), C))
            v[b, L:] = float("nan")
            attn[b, L:] = float("nan")
    return attn, v, seq_lens


# Gate of the decode score step. Its outputs are softmax probabilities, which
# at workload lengths are of order 1/L (2e-5 at L = 32768): an absolute bound
# near 1e-4 would let most of them be wrong by more than 100 %. Each written
# probability is therefore held to a bound relative to itself, and each row
# (b, q_h) over c < L_b must still sum to 1.
QK_RTOL = 1e-4      # per element, relative to the oracle's value
QK_ATOL = 1e-12     # floor for probabilities that are exactly or nearly zero
QK_SUM_TOL = 1e-5   # |sum_c attn[b, c, q_h] - 1| for every row with L_b > 0


def qk_gate_errors(got, ref, lens):
    """Errors of a score-step result against the oracle's over the written rows
    (c < L_b): a dict with `ratio`, the largest |got - ref| / (QK_RTOL * |ref| +
    QK_ATOL) (the gate holds at <= 1), `rel`, the largest |got - ref| / |ref|
    over ref != 0, `where`, the index of the worst ratio, `row_sum`, the largest
    |sum_c got - 1| over rows with L_b > 0, and `finite`."""
    B, C, _ = got.shape
    res = {"ratio": 0.0, "rel": 0.0, "where": None, "row_sum": 0.0, "finite": True}
    for b in range(B):
        L = max(0, min(int(lens[b]), C)) if lens is not None else C
        if L == 0:
            continue
        g, r = got[b, :L], ref[b, :L]
        res["finite"] = res["finite"] and bool(np.all(np.isfinite(g)))
        diff = np.abs(g - r)
        ratio = diff / (QK_RTOL * np.abs(r) + QK_ATOL)
        i = int(np.argmax(ratio))
        if ratio.flat[i] > res["ratio"]:
            res["ratio"] = float(ratio.flat[i])
            res["where"] = (b,) + tuple(int(x) for x in np.unravel_index(i, ratio.shape))
        nz = r != 0
        if np.any(nz):
            res["rel"] = max(res["rel"], float((diff[nz] / np.abs(r[nz])).max()))
        res["row_sum"] = max(res["row_sum"],
                             float(np.abs(g.sum(axis=0, dtype=np.float64) - 1.0).max()))
    return res


def qk_gate(got, ref, lens, what):
    """Asserts the score-step gate: |got - ref| <= QK_RTOL * |ref| + QK_ATOL for
    every written probability, and every row sums to 1 within QK_SUM_TOL."""
    e = qk_gate_errors(got, ref, lens)
    assert e["finite"], f"{what}: non-finite probabilities"
    assert e["ratio"] <= 1.0, (f"{what}: |gpu - oracle| is {e['ratio']:.3g} x the bound "
                               f"{QK_RTOL:.0e} * |oracle| + {QK_ATOL:.0e} at {e['where']}")
    assert e["row_sum"] <= QK_SUM_TOL, \
        f"{what}: a row sums to 1 +- {e['row_sum']:.3e} (> {QK_SUM_TOL:.0e})"
    return e
