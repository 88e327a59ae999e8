"""CPU fp64 oracle for the decode score step (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU legs may import this
module; the product path never does. It shares no code with the CUDA path.

Definition (the step before the AV reduction of LLM decode: the page
"pytorch/executorch pull 21063", summary paragraph, names the AV coop-GEMV of
decode; the scores it consumes are the softmax-normalised products of the
query with the K cache, with the same query-to-KV-head mapping):

    s[b, c, q_h]    = scale * sum_d q[b, q_h, d] * K[b, c, q_h // G, d]
    attn[b, c, q_h] = exp(s[b, c, q_h] - max_c' s[b, c', q_h])
                      / sum_c'' exp(s[b, c'', q_h] - max_c' s[b, c', q_h])

for c, c', c'' < L_b = clamp(seq_lens[b], 0, Cmax). Entries at c >= L_b are
not defined by the operation; this oracle returns 0 there. Arithmetic in
binary64: the fp32 query and the bf16/fp16 K widen exactly; the dot products
are numpy matrix products, the softmax numpy exp / max / sum.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def decode(bits: np.ndarray, k_dtype: str) -> np.ndarray:
    """bf16 / fp16 bit patterns (uint16) -> float64, exactly."""
    bits = np.ascontiguousarray(bits)
    if bits.dtype != np.uint16:
        bits = bits.view(np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to NaN
        if k_dtype == "bf16":
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        if k_dtype == "fp16":
            return bits.view(np.float16).astype(np.float64)
    raise ValueError("k_dtype must be 'bf16' or 'fp16'")


def gqa_qk_softmax(q: np.ndarray, k_bits: np.ndarray, k_dtype: str,
                   seq_lens: Optional[np.ndarray] = None, scale: float = 1.0) -> np.ndarray:
    """q [B,Hq,D] fp32, k_bits [B,C,Hkv,D] uint16 patterns -> attn [B,C,Hq] fp64."""
    q = np.asarray(q, dtype=np.float32).astype(np.float64)
    k_bits = np.asarray(k_bits)
    if q.ndim != 3 or k_bits.ndim != 4:
        raise ValueError("q must be [B,Hq,D] and k [B,C,Hkv,D]")
    B, Hq, D = q.shape
    B2, C, Hkv, D2 = k_bits.shape
    if B2 != B or D2 != D or Hq % Hkv:
        raise ValueError("q and k disagree on B or D, or Hq % Hkv != 0")
    G = Hq // Hkv
    out = np.zeros((B, C, Hq), dtype=np.float64)
    for b in range(B):
        L = C if seq_lens is None else int(min(max(int(seq_lens[b]), 0), C))
        if L == 0:
            continue
        for kv_h in range(Hkv):
            k = decode(k_bits[b, :L, kv_h, :], k_dtype)       # [L, D]
            heads = slice(kv_h * G, (kv_h + 1) * G)             # q_h // G == kv_h
            s = scale * (k @ q[b, heads, :].T)                  # [L, G]
            m = s.max(axis=0)
            e = np.exp(s - m)
            out[b, :L, heads] = e / e.sum(axis=0)
    return out
