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
