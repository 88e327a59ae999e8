"""Seeded synthetic inputs for the GQA AV decode reduction.

This module only draws inputs; it computes nothing of the reduction itself, so
the CUDA path and the CPU oracle can both be fed from it without sharing any of
the method's arithmetic.

Shapes follow the decode step of grouped-query attention described on the page
"pytorch/executorch pull 21063" (summary paragraph): Hq = G * Hkv query heads,
the V cache holds one D-wide row per (context position, KV head), and the
attention weights hold one scalar per (context position, query head). A batch
dimension B and per-sequence lengths seq_lens[b] are added in front.

Recipe (one ``torch.Generator`` seeded with ``seed``, draws in this order):

1. ``seq_lens[b]`` ~ integers uniform on [len_lo, len_hi], both ends inclusive.
2. For b = 0..B-1: ``V[b]`` ~ N(0, v_sigma^2) drawn in fp32, then rounded to
   bf16/fp16 (round-to-nearest-even, torch ``.to``).
3. For b = 0..B-1: logits ~ N(0, logit_sigma^2) drawn in fp64 with shape
   [Cmax, Hq]; ``attn[b, :L_b, q]`` = softmax over c < L_b of the logits in
   fp64, then rounded to fp32.

Positions c >= L_b are padding: zero by default, NaN with ``pad="nan"`` so a
kernel that reads and uses them poisons its output.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

V_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Cmax: int
    Hq: int
    Hkv: int
    D: int
    v_dtype: str = "bf16"
    v_sigma: float = 1.0
    logit_sigma: float = 2.0
    len_lo: Optional[int] = None  # None -> Cmax
    len_hi: Optional[int] = None  # None -> Cmax
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def lo(self) -> int:
        return self.Cmax if self.len_lo is None else self.len_lo

    @property
    def hi(self) -> int:
        return self.Cmax if self.len_hi is None else self.len_hi

    def describe(self) -> Dict[str, object]:
        return {
            "workload": self.name, "B": self.B, "Cmax": self.Cmax, "Hq": self.Hq,
            "Hkv": self.Hkv, "G": self.G, "D": self.D, "v_dtype": self.v_dtype,
            "seq_lens": f"uniform[{self.lo},{self.hi}]", "seed": self.seed,
        }


# The five decode shapes the method is measured on. Names say what they are.
WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    # The small case: G=4, D=64, one short sequence.
    Workload("small_b1_c512_hq8_hkv2_d64", 1, 512, 8, 2, 64, "bf16", 1.0, 2.0),
    # Llama-style decode, G=4, full-length context.
    Workload("llama_b1_c8192_hq32_hkv8_d128", 1, 8192, 32, 8, 128, "bf16", 1.0, 2.0),
    # Phi-style decode, G=3, peaked weights, ragged lengths in [C/2, C].
    Workload("phi_b4_c16384_hq24_hkv8_d128_ragged", 4, 16384, 24, 8, 128, "bf16",
             1.0, 3.0, 8192, 16384),
    # Multi-query attention beyond a group cap of 8: G=16, D=256, fp16, lengths in [1, C].
    Workload("mqa_b8_c32768_hq16_hkv1_d256_fp16_ragged", 8, 32768, 16, 1, 256, "fp16",
             0.5, 2.0, 1, 32768),
    # Large batch, G=8, ~8.6 GB of V, lengths in [C/4, C].
    Workload("large_b32_c131072_hq64_hkv8_d128_ragged", 32, 131072, 64, 8, 128, "bf16",
             1.0, 2.0, 32768, 131072),
    # V-traffic comparison shape: Llama-style heads (G=4) with 537 MB of V, four
    # times the L2, so per-head re-reads of V cannot all be L2 hits.
    Workload("traffic_b8_c32768_hq32_hkv8_d128", 8, 32768, 32, 8, 128, "bf16", 1.0, 2.0),
    # The large-batch shape at an eighth of the context (~1.07 GB of V, lengths
    # in [C/4, C]): the same 256 tiles and split rule, small enough to profile.
    Workload("ragged_b32_c16384_hq64_hkv8_d128", 32, 16384, 64, 8, 128, "bf16",
             1.0, 2.0, 4096, 16384),
    # The Llama-style shape with a head dimension of 100 (a multiple of the
    # page's 4-wide texel, not of 8): the calls the TMA kernels cannot take.
    Workload("odd_b1_c8192_hq32_hkv8_d100", 1, 8192, 32, 8, 100, "bf16", 1.0, 2.0),
]}

# Short aliases, in the order above.
ALIASES = {
    "small": "small_b1_c512_hq8_hkv2_d64",
    "llama": "llama_b1_c8192_hq32_hkv8_d128",
    "phi": "phi_b4_c16384_hq24_hkv8_d128_ragged",
    "mqa": "mqa_b8_c32768_hq16_hkv1_d256_fp16_ragged",
    "large": "large_b32_c131072_hq64_hkv8_d128_ragged",
    "traffic": "traffic_b8_c32768_hq32_hkv8_d128",
    "ragged": "ragged_b32_c16384_hq64_hkv8_d128",
    "odd": "odd_b1_c8192_hq32_hkv8_d100",
}


def get(name: str) -> Workload:
    return WORKLOADS[ALIASES.get(name, name)]


def custom(B, Cmax, Hq, Hkv, D, v_dtype="bf16", v_sigma=1.0, logit_sigma=2.0,
           len_lo=None, len_hi=None, seed=0) -> Workload:
    name = f"b{B}_c{Cmax}_hq{Hq}_hkv{Hkv}_d{D}_{v_dtype}"
    return Workload(name, B, Cmax, Hq, Hkv, D, v_dtype, v_sigma, logit_sigma,
                    len_lo, len_hi, seed)


def generate(w: Workload, device="cpu", pad: str = "zero",
             seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw (attn, v, seq_lens) for workload ``w`` on ``device``.

    Returns contiguous tensors: attn [B, Cmax, Hq] fp32, v [B, Cmax, Hkv, D]
    bf16/fp16, seq_lens [B] int32. The same seed on the same device type gives
    the same bits; CPU and CUDA draws differ from each other.
    """
    if pad not in ("zero", "nan"):
        raise ValueError("pad must be 'zero' or 'nan'")
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    B, C, Hq, Hkv, D = w.B, w.Cmax, w.Hq, w.Hkv, w.D
    vt = V_DTYPES[w.v_dtype]
    padv = 0.0 if pad == "zero" else float("nan")

    seq_lens = torch.randint(w.lo, w.hi + 1, (B,), generator=g, device=device,
                             dtype=torch.int64).to(torch.int32)
    lens = seq_lens.cpu().tolist()

    v = torch.empty((B, C, Hkv, D), dtype=vt, device=device)
    for b in range(B):
        vb = torch.randn((C, Hkv, D), generator=g, device=device, dtype=torch.float32)
        vb.mul_(w.v_sigma)
        v[b].copy_(vb.to(vt))
        if lens[b] < C:
            v[b, lens[b]:].fill_(padv)
        del vb

    attn = torch.empty((B, C, Hq), dtype=torch.float32, device=device)
    for b in range(B):
        logits = torch.randn((C, Hq), generator=g, device=device, dtype=torch.float64)
        logits.mul_(w.logit_sigma)
        L = lens[b]
        if L > 0:
            attn[b, :L].copy_(torch.softmax(logits[:L], dim=0).to(torch.float32))
        if L < C:
            attn[b, L:].fill_(padv)
        del logits
    return {"attn": attn, "v": v, "seq_lens": seq_lens}


def generate_qkv(w: Workload, device="cpu", pad: str = "zero",
                 seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Inputs of the fused decode attention for workload ``w``: (q, k, v, seq_lens).

    ``seq_lens`` and ``v`` are those of ``generate`` with the same seed. A second
    generator seeded with seed + 1 then draws, for b = 0..B-1, ``K[b]`` ~
    N(0, v_sigma^2) in fp32 rounded to the cache type, and after that
    ``q`` [B, Hq, D] ~ N(0, logit_sigma^2) in fp32, so that the scores
    q . K / sqrt(D) spread like the workload's logits. K rows c >= L_b are
    padding like V's.
    """
    x = generate(w, device, pad, seed)
    del x["attn"]
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 1)
    B, C, Hkv, D = w.B, w.Cmax, w.Hkv, w.D
    lens = x["seq_lens"].cpu().tolist()
    padv = 0.0 if pad == "zero" else float("nan")
    k = torch.empty((B, C, Hkv, D), dtype=V_DTYPES[w.v_dtype], device=device)
    for b in range(B):
        kb = torch.randn((C, Hkv, D), generator=g, device=device, dtype=torch.float32)
        kb.mul_(w.v_sigma)
        k[b].copy_(kb.to(k.dtype))
        if lens[b] < C:
            k[b, lens[b]:].fill_(padv)
        del kb
    q = torch.randn((B, w.Hq, D), generator=g, device=device, dtype=torch.float32)
    q.mul_(w.logit_sigma)
    return {"q": q, "k": k, "v": x["v"], "seq_lens": x["seq_lens"]}


def attention_compulsory_bytes(w: Workload, seq_lens) -> int:
    """Bytes the fused decode attention must move at least once: every in-range
    K row and V row once, q once, out once, and seq_lens."""
    total_L = int(sum(int(x) for x in seq_lens))
    return total_L * w.Hkv * w.D * 2 * 2 + 2 * w.B * w.Hq * w.D * 4 + 4 * w.B


def attention_flops(w: Workload, seq_lens) -> int:
    """Multiply-adds x 2 of the two products (scores and the weighted sum)."""
    total_L = int(sum(int(x) for x in seq_lens))
    return 4 * total_L * w.Hq * w.D


def compulsory_bytes(w: Workload, seq_lens) -> int:
    """Bytes the reduction must move at least once: every in-range V row once,
    every in-range attn weight once, out once, and seq_lens."""
    esz = 2
    total_L = int(sum(int(x) for x in seq_lens))
    return (total_L * (w.Hkv * w.D * esz + w.Hq * 4)
            + w.B * w.Hq * w.D * 4 + 4 * w.B)


def flops(w: Workload, seq_lens) -> int:
    """Multiply-add count x 2 over in-range positions."""
    total_L = int(sum(int(x) for x in seq_lens))
    return 2 * total_L * w.Hq * w.D
