"""CPU fp64 oracle for fused decode attention (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU legs may import this
module; the product path never does. It shares no code with the CUDA path.

Definition. The AV coop-GEMV of LLM decode (page "pytorch/executorch pull
21063", summary paragraph) consumes softmax weights over the context; taking
the weights as the softmax of the scaled query-key products of the same step,
with the same query-to-KV-head mapping, the whole decode attention of one
step is

    s[b, c, q_h]   = scale * sum_d q[b, q_h, d] * K[b, c, q_h // G, d]
    w[b, c, q_h]   = exp(s[b, c, q_h] - max_c' s[b, c', q_h])
                     / sum_c'' exp(s[b, c'', q_h] - max_c' s[b, c', q_h])
    out[b, q_h, d] = sum_c w[b, c, q_h] * V[b, c, q_h // G, d]

for c, c', c'' < L_b = clamp(seq_lens[b], 0, Cmax). With L_b = 0 the sum is
empty and out is 0. The weights are never rounded: the arithmetic is binary64
throughout (the fp32 query and the bf16/fp16 K and V widen exactly; numpy
matrix products, exp, max and sum).
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 / fp16 bit patterns (uint16) -> float64, exactly."""
    bits = np.ascontiguousarray(bits)
    if bits.dtype != np.uint16:
        bits = bits.view(np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to NaN
        if dtype == "bf16":
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        if dtype == "fp16":
            return bits.view(np.float16).astype(np.float64)
    raise ValueError("dtype must be 'bf16' or 'fp16'")


def gqa_attention(q: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, kv_dtype: str,
                  seq_lens: Optional[np.ndarray] = None, scale: float = 1.0) -> np.ndarray:
    """q [B,Hq,D] fp32, k_bits / v_bits [B,C,Hkv,D] uint16 patterns -> out [B,Hq,D] fp64."""
    q = np.asarray(q, dtype=np.float32).astype(np.float64)
    k_bits = np.asarray(k_bits)
    v_bits = np.asarray(v_bits)
    if q.ndim != 3 or k_bits.ndim != 4 or v_bits.shape != k_bits.shape:
        raise ValueError("q must be [B,Hq,D], k and v [B,C,Hkv,D]")
    B, Hq, D = q.shape
    B2, C, Hkv, D2 = k_bits.shape
    if B2 != B or D2 != D or Hq % Hkv:
        raise ValueError("q and k disagree on B or D, or Hq % Hkv != 0")
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = C if seq_lens is None else int(min(max(int(seq_lens[b]), 0), C))
        if L == 0:
            continue
        for kv_h in range(Hkv):
            k = decode(k_bits[b, :L, kv_h, :], kv_dtype)       # [L, D]
            v = decode(v_bits[b, :L, kv_h, :], kv_dtype)       # [L, D]
            heads = slice(kv_h * G, (kv_h + 1) * G)             # q_h // G == kv_h
            s = scale * (k @ q[b, heads, :].T)                  # [L, G]
            m = s.max(axis=0)
            e = np.exp(s - m)
            w = e / e.sum(axis=0)                               # softmax over c, per head
            out[b, heads, :] = w.T @ v                          # [G, D]
    return out
