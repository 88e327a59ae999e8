"""CPU fp64 oracle for the GQA AV decode reduction (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package. The product path never does. The arithmetic lives in
``gqa_av_oracle.c`` (plain C, pthreads, binary64); this module compiles it with
gcc on first use and marshals numpy arrays through ctypes.

Definition (page "pytorch/executorch pull 21063", summary paragraph):
``out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, q_h // G, d]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gqa_av_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle_gqa_av.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread"]

V_DTYPE_CODES = {"bf16": 0, "fp16": 1}


def compile_library(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` into the shared library ``output`` with gcc."""
    cmd = ["gcc", *CFLAGS, source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def _stale(lib: str, src: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


class Oracle:
    """ctypes handle on one compiled copy of the oracle."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_gqa_av.restype = ctypes.c_int
        lib.oracle_gqa_av.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_fp16.restype = ctypes.c_double
        lib.oracle_decode_fp16.argtypes = [ctypes.c_uint16]
        self.lib = lib

    def gqa_av(self, attn: np.ndarray, v_bits: np.ndarray, v_dtype: str,
               seq_lens: Optional[np.ndarray] = None, nthreads: int = 1) -> np.ndarray:
        """attn [B,C,Hq] fp32, v_bits [B,C,Hkv,D] uint16 patterns -> out [B,Hq,D] fp64."""
        attn = np.ascontiguousarray(attn, dtype=np.float32)
        v_bits = np.ascontiguousarray(v_bits)
        if v_bits.dtype != np.uint16:
            v_bits = v_bits.view(np.uint16)
        if attn.ndim != 3 or v_bits.ndim != 4:
            raise ValueError("attn must be [B,C,Hq] and v [B,C,Hkv,D]")
        B, C, Hq = attn.shape
        B2, C2, Hkv, D = v_bits.shape
        if (B, C) != (B2, C2):
            raise ValueError("attn and v disagree on B or C")
        sl_ptr = None
        if seq_lens is not None:
            seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
            if seq_lens.shape != (B,):
                raise ValueError("seq_lens must be [B]")
            sl_ptr = seq_lens.ctypes.data
        out = np.empty((B, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_gqa_av(attn.ctypes.data, v_bits.ctypes.data,
                                    V_DTYPE_CODES[v_dtype], sl_ptr, out.ctypes.data,
                                    B, C, Hq, Hkv, D, int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_gqa_av rejected its arguments (rc={rc})")
        return out

    def decode(self, bits: int, v_dtype: str) -> float:
        if v_dtype == "bf16":
            return self.lib.oracle_decode_bf16(bits)
        return self.lib.oracle_decode_fp16(bits)


_default: Optional[Oracle] = None


def load() -> Oracle:
    """The oracle built from this directory's source (compiled if stale)."""
    global _default
    if _default is None:
        if _stale(LIBRARY, SOURCE):
            compile_library()
        _default = Oracle(LIBRARY)
    return _default


def gqa_av(attn, v_bits, v_dtype, seq_lens=None, nthreads=1) -> np.ndarray:
    return load().gqa_av(attn, v_bits, v_dtype, seq_lens, nthreads)


def host_cores() -> int:
    return len(os.sched_getaffinity(0))
