"""ctypes binding of libgqa_av.so (include/gqa_av.h).

Argument marshalling only: every step of the reduction runs in the CUDA
library. Import fails loudly when the library has not been built; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_PKG, "libgqa_av.so")

GQA_AV_OK = 0
GQA_AV_ERR_INVALID = 1
GQA_AV_ERR_UNSUPPORTED = 2
GQA_AV_ERR_CUDA = 3
GQA_AV_ERR_NOMEM = 4
GQA_AV_ERR_DEVICE_TIMEOUT = 5

GQA_AV_BF16 = 0
GQA_AV_FP16 = 1
MODE_AUTO, MODE_PER_HEAD, MODE_GQA = -1, 0, 1

_V_DTYPE = {torch.bfloat16: GQA_AV_BF16, torch.float16: GQA_AV_FP16}


class GqaAvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class Tuning(ctypes.Structure):
    _fields_ = [("nsplit", ctypes.c_int), ("dtile", ctypes.c_int),
                ("rows_per_stage", ctypes.c_int), ("stages", ctypes.c_int),
                ("early_stages", ctypes.c_int), ("engine", ctypes.c_int),
                ("split_mode", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "mode", "heads_per_cta", "head_chunk", "dtile", "rows_per_stage", "stages",
        "early_stages", "engine", "split_mode", "nsplit",
        "combine_ctas", "rows_per_split", "tiles", "ctas", "threads_per_cta", "smem_bytes",
        "ctas_per_sm")] + [
        ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIBRARY):
        raise ImportError(
            f"{LIBRARY} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIBRARY)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sizes = [I, I, I, I, I]
    lib.gqa_av_decode.argtypes = [P, P, P, P, *sizes, I, I, P]
    lib.gqa_av_decode_per_head.argtypes = [P, P, P, P, *sizes, I, P]
    lib.gqa_av_decode_tuned.argtypes = [P, P, P, P, *sizes, I, I, ctypes.POINTER(Tuning), P]
    lib.gqa_av_decode_noalloc.argtypes = [P, P, P, P, *sizes, I, I, P]
    lib.gqa_av_decode_paged.argtypes = [P, P, P, P, P, *sizes, I, I, I, I, I,
                                        ctypes.POINTER(Tuning), P]
    lib.gqa_av_plan.argtypes = [*sizes, I, I, ctypes.POINTER(Tuning), ctypes.POINTER(PlanInfo)]
    lib.gqa_av_selftest_wait_timeout.argtypes = [P, P, P, P, *sizes, I, ctypes.c_longlong, I, P]
    lib.gqa_av_workspace_bytes.argtypes = [*sizes, I, I]
    lib.gqa_av_workspace_bytes.restype = S
    lib.gqa_av_set_workspace.argtypes = [P, S]
    lib.gqa_av_device_status.argtypes = [P, I]
    lib.gqa_av_status_string.argtypes = [I]
    lib.gqa_av_status_string.restype = ctypes.c_char_p
    lib.gqa_av_last_error.argtypes = []
    lib.gqa_av_last_error.restype = ctypes.c_char_p
    lib.gqa_av_version.argtypes = []
    lib.gqa_qk_softmax_decode.argtypes = [P, P, P, P, *sizes, I, ctypes.c_float, I, P]
    lib.gqa_qk_softmax_decode_tuned.argtypes = [P, P, P, P, *sizes, I, ctypes.c_float, I, I, P]
    lib.gqa_qk_device_status.argtypes = [P, I]
    lib.gqa_qk_last_error.argtypes = []
    lib.gqa_qk_last_error.restype = ctypes.c_char_p
    lib.gqa_attn_decode.argtypes = [P, P, P, P, P, *sizes, I, ctypes.c_float, I, P]
    lib.gqa_attn_decode_tuned.argtypes = [P, P, P, P, P, *sizes, I, ctypes.c_float, I, I, I, I, I,
                                          P]
    lib.gqa_attn_plan.argtypes = [*sizes, I, I, I, I, I, I, I, ctypes.POINTER(ctypes.c_int), I]
    lib.gqa_attn_device_status.argtypes = [P, I]
    lib.gqa_attn_last_error.argtypes = []
    lib.gqa_attn_last_error.restype = ctypes.c_char_p
    for f in ("gqa_attn_decode", "gqa_attn_decode_tuned", "gqa_attn_plan", "gqa_attn_device_status"):
        getattr(lib, f).restype = I
    for f in ("gqa_av_decode", "gqa_av_decode_per_head", "gqa_av_decode_tuned", "gqa_av_decode_paged",
              "gqa_av_decode_noalloc", "gqa_av_plan", "gqa_av_selftest_wait_timeout",
              "gqa_av_set_workspace", "gqa_av_device_status", "gqa_av_version",
              "gqa_qk_softmax_decode", "gqa_qk_softmax_decode_tuned", "gqa_qk_device_status"):
        getattr(lib, f).restype = I
    return lib


lib = _load()


def _check(status: int) -> None:
    if status != GQA_AV_OK:
        name = lib.gqa_av_status_string(status).decode()
        msg = lib.gqa_av_last_error().decode()
        raise GqaAvError(status, f"{name}: {msg}")


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _shapes(attn: torch.Tensor, v_cache: torch.Tensor, seq_lens, out: torch.Tensor):
    if attn.dim() != 3 or v_cache.dim() != 4 or out.dim() != 3:
        raise ValueError("attn must be [B,Cmax,Hq], v_cache [B,Cmax,Hkv,D], out [B,Hq,D]")
    B, Cmax, Hq = attn.shape
    B2, C2, Hkv, D = v_cache.shape
    if (B2, C2) != (B, Cmax) or tuple(out.shape) != (B, Hq, D):
        raise ValueError(f"inconsistent shapes: attn {tuple(attn.shape)}, v "
                         f"{tuple(v_cache.shape)}, out {tuple(out.shape)}")
    for name, t in (("attn", attn), ("v_cache", v_cache), ("out", out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if attn.dtype != torch.float32 or out.dtype != torch.float32:
        raise ValueError("attn and out must be float32")
    if v_cache.dtype not in _V_DTYPE:
        raise ValueError("v_cache must be bfloat16 or float16")
    if seq_lens is not None:
        if (not seq_lens.is_cuda or seq_lens.dtype != torch.int32 or seq_lens.numel() != B
                or not seq_lens.is_contiguous()):
            raise ValueError("seq_lens must be a contiguous CUDA int32 tensor of B elements")
    return B, Cmax, Hq, Hkv, D, _V_DTYPE[v_cache.dtype]


def _ptr(t):
    return None if t is None else t.data_ptr()


def gqa_av_decode(attn, v_cache, seq_lens, out, mode: int = MODE_AUTO, stream=None) -> torch.Tensor:
    """out[b,q,d] = sum_{c<L_b} attn[b,c,q] * v_cache[b,c,q//G,d]; writes and returns ``out``."""
    B, C, Hq, Hkv, D, vd = _shapes(attn, v_cache, seq_lens, out)
    _check(lib.gqa_av_decode(_ptr(attn), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                             B, C, Hq, Hkv, D, vd, int(mode), _stream_handle(stream)))
    return out


def gqa_av_decode_per_head(attn, v_cache, seq_lens, out, stream=None) -> torch.Tensor:
    B, C, Hq, Hkv, D, vd = _shapes(attn, v_cache, seq_lens, out)
    _check(lib.gqa_av_decode_per_head(_ptr(attn), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                                      B, C, Hq, Hkv, D, vd, _stream_handle(stream)))
    return out


def gqa_av_decode_noalloc(attn, v_cache, seq_lens, out, mode: int = MODE_AUTO,
                          stream=None) -> torch.Tensor:
    """gqa_av_decode for callers that may not allocate device memory: the
    library's fixed scratch array is used and no call allocates. The first call
    on a device looks up that array's address; make it before any capture."""
    B, C, Hq, Hkv, D, vd = _shapes(attn, v_cache, seq_lens, out)
    _check(lib.gqa_av_decode_noalloc(_ptr(attn), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                                     B, C, Hq, Hkv, D, vd, int(mode), _stream_handle(stream)))
    return out


def _tuning(t) -> Optional[Tuning]:
    if t is None:
        return None
    if isinstance(t, Tuning):
        return t
    return Tuning(int(t.get("nsplit", 0)), int(t.get("dtile", 0)),
                  int(t.get("rows_per_stage", 0)), int(t.get("stages", 0)),
                  int(t.get("early_stages", 0)), int(t.get("engine", 0)),
                  int(t.get("split_mode", 0)))


def gqa_av_decode_tuned(attn, v_cache, seq_lens, out, mode=MODE_AUTO, tuning=None,
                        stream=None) -> torch.Tensor:
    B, C, Hq, Hkv, D, vd = _shapes(attn, v_cache, seq_lens, out)
    t = _tuning(tuning)
    _check(lib.gqa_av_decode_tuned(_ptr(attn), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                                   B, C, Hq, Hkv, D, vd, int(mode),
                                   ctypes.byref(t) if t is not None else None,
                                   _stream_handle(stream)))
    return out


def gqa_av_decode_paged(attn, v_pool, block_table, seq_lens, out, mode=MODE_AUTO, tuning=None,
                        stream=None) -> torch.Tensor:
    """gqa_av_decode over a paged V cache: v_pool [num_blocks, block_size, Hkv, D],
    block_table [B, max_blocks] int32 (row c of sequence b in block
    block_table[b, c // block_size])."""
    if attn.dim() != 3 or v_pool.dim() != 4 or out.dim() != 3 or block_table.dim() != 2:
        raise ValueError("attn [B,Cmax,Hq], v_pool [blocks,block_size,Hkv,D], block_table "
                         "[B,max_blocks], out [B,Hq,D]")
    B, Cmax, Hq = attn.shape
    num_blocks, block_size, Hkv, D = v_pool.shape
    if tuple(out.shape) != (B, Hq, D) or block_table.shape[0] != B:
        raise ValueError("inconsistent shapes")
    for name, t in (("attn", attn), ("v_pool", v_pool), ("out", out), ("block_table", block_table)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if attn.dtype != torch.float32 or out.dtype != torch.float32:
        raise ValueError("attn and out must be float32")
    if v_pool.dtype not in _V_DTYPE or block_table.dtype != torch.int32:
        raise ValueError("v_pool must be bfloat16 or float16 and block_table int32")
    if seq_lens is not None and (not seq_lens.is_cuda or seq_lens.dtype != torch.int32
                                 or seq_lens.numel() != B or not seq_lens.is_contiguous()):
        raise ValueError("seq_lens must be a contiguous CUDA int32 tensor of B elements")
    t = _tuning(tuning)
    _check(lib.gqa_av_decode_paged(_ptr(attn), _ptr(v_pool), _ptr(block_table), _ptr(seq_lens),
                                   _ptr(out), B, Cmax, Hq, Hkv, D, _V_DTYPE[v_pool.dtype],
                                   block_size, num_blocks, block_table.shape[1], int(mode),
                                   ctypes.byref(t) if t is not None else None,
                                   _stream_handle(stream)))
    return out


def gqa_av_plan(B, Cmax, Hq, Hkv, D, v_dtype=GQA_AV_BF16, mode=MODE_AUTO, tuning=None) -> dict:
    info = PlanInfo()
    t = _tuning(tuning)
    _check(lib.gqa_av_plan(B, Cmax, Hq, Hkv, D, v_dtype, mode,
                           ctypes.byref(t) if t is not None else None, ctypes.byref(info)))
    return info.as_dict()


def gqa_av_workspace_bytes(B, Cmax, Hq, Hkv, D, v_dtype=GQA_AV_BF16, mode=MODE_AUTO) -> int:
    return int(lib.gqa_av_workspace_bytes(B, Cmax, Hq, Hkv, D, v_dtype, mode))


def gqa_av_set_workspace(buffer: Optional[torch.Tensor]) -> None:
    if buffer is None:
        _check(lib.gqa_av_set_workspace(None, 0))
    else:
        _check(lib.gqa_av_set_workspace(buffer.data_ptr(), buffer.numel() * buffer.element_size()))


def gqa_av_device_status(stream=None, clear: bool = True) -> None:
    _check(lib.gqa_av_device_status(_stream_handle(stream), 1 if clear else 0))


def gqa_av_status_string(status: int) -> str:
    return lib.gqa_av_status_string(status).decode()


def gqa_av_last_error() -> str:
    return lib.gqa_av_last_error().decode()


def v_dtype_code(dtype: torch.dtype) -> int:
    return _V_DTYPE[dtype]


# ------------------------------------------------------------ score step
def _check_qk(status: int) -> None:
    if status != GQA_AV_OK:
        name = lib.gqa_av_status_string(status).decode()
        raise GqaAvError(status, f"{name}: {lib.gqa_qk_last_error().decode()}")


def gqa_qk_softmax_decode(q, k_cache, seq_lens, attn, mode: int = MODE_AUTO, scale=None,
                          stream=None, engine: int = 0) -> torch.Tensor:
    """attn[b,c,q] = softmax over c < L_b of scale * q[b,q,:] . k_cache[b,c,q//G,:]
    (scale defaults to 1/sqrt(D)); rows c >= L_b of ``attn`` are left as they are."""
    if q.dim() != 3 or k_cache.dim() != 4 or attn.dim() != 3:
        raise ValueError("q must be [B,Hq,D], k_cache [B,Cmax,Hkv,D], attn [B,Cmax,Hq]")
    B, Hq, D = q.shape
    B2, Cmax, Hkv, D2 = k_cache.shape
    if (B2, D2) != (B, D) or tuple(attn.shape) != (B, Cmax, Hq):
        raise ValueError(f"inconsistent shapes: q {tuple(q.shape)}, k {tuple(k_cache.shape)}, "
                         f"attn {tuple(attn.shape)}")
    for name, t in (("q", q), ("k_cache", k_cache), ("attn", attn)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if q.dtype != torch.float32 or attn.dtype != torch.float32:
        raise ValueError("q and attn must be float32")
    if k_cache.dtype not in _V_DTYPE:
        raise ValueError("k_cache must be bfloat16 or float16")
    if seq_lens is not None and (not seq_lens.is_cuda or seq_lens.dtype != torch.int32
                                 or seq_lens.numel() != B or not seq_lens.is_contiguous()):
        raise ValueError("seq_lens must be a contiguous CUDA int32 tensor of B elements")
    sc = float(D) ** -0.5 if scale is None else float(scale)
    _check_qk(lib.gqa_qk_softmax_decode_tuned(_ptr(q), _ptr(k_cache), _ptr(seq_lens), _ptr(attn),
                                              B, Cmax, Hq, Hkv, D, _V_DTYPE[k_cache.dtype], sc,
                                              int(mode), int(engine), _stream_handle(stream)))
    return attn


def gqa_qk_device_status(stream=None, clear: bool = True) -> None:
    _check_qk(lib.gqa_qk_device_status(_stream_handle(stream), 1 if clear else 0))


# ------------------------------------------------------- fused attention
def _check_attn(status: int) -> None:
    if status != GQA_AV_OK:
        name = lib.gqa_av_status_string(status).decode()
        raise GqaAvError(status, f"{name}: {lib.gqa_attn_last_error().decode()}")


def gqa_attn_decode(q, k_cache, v_cache, seq_lens, out, mode: int = MODE_AUTO, scale=None,
                    stream=None, consumer_warps: int = 0, nsplit: int = 0,
                    split_mode: int = 0, column_blocks: int = 0) -> torch.Tensor:
    """out[b,q,:] = sum over c < L_b of softmax_c(scale * q[b,q,:] . k_cache[b,c,q//G,:])
    * v_cache[b,c,q//G,:] (scale defaults to 1/sqrt(D)); writes and returns ``out``."""
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.dim() != 4 or out.dim() != 3:
        raise ValueError("q [B,Hq,D], k_cache and v_cache [B,Cmax,Hkv,D], out [B,Hq,D]")
    B, Hq, D = q.shape
    B2, Cmax, Hkv, D2 = k_cache.shape
    if ((B2, D2) != (B, D) or tuple(v_cache.shape) != tuple(k_cache.shape)
            or tuple(out.shape) != (B, Hq, D)):
        raise ValueError(f"inconsistent shapes: q {tuple(q.shape)}, k {tuple(k_cache.shape)}, "
                         f"v {tuple(v_cache.shape)}, out {tuple(out.shape)}")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if q.dtype != torch.float32 or out.dtype != torch.float32:
        raise ValueError("q and out must be float32")
    if k_cache.dtype not in _V_DTYPE or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must both be bfloat16 or both float16")
    if seq_lens is not None and (not seq_lens.is_cuda or seq_lens.dtype != torch.int32
                                 or seq_lens.numel() != B or not seq_lens.is_contiguous()):
        raise ValueError("seq_lens must be a contiguous CUDA int32 tensor of B elements")
    sc = float(D) ** -0.5 if scale is None else float(scale)
    _check_attn(lib.gqa_attn_decode_tuned(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                          _ptr(out), B, Cmax, Hq, Hkv, D, _V_DTYPE[k_cache.dtype],
                                          sc, int(mode), int(consumer_warps), int(nsplit),
                                          int(split_mode), int(column_blocks),
                                          _stream_handle(stream)))
    return out


def gqa_attn_plan(B, Cmax, Hq, Hkv, D, kv_dtype=GQA_AV_BF16, mode=MODE_AUTO, consumer_warps=0,
                  nsplit=0, split_mode=0, ragged=True, column_blocks=0) -> dict:
    info = (ctypes.c_int * 11)()
    _check_attn(lib.gqa_attn_plan(B, Cmax, Hq, Hkv, D, kv_dtype, mode, consumer_warps, nsplit,
                                  split_mode, column_blocks, 1 if ragged else 0, info, 11))
    keys = ("mode", "heads_per_cta", "consumer_warps", "stages", "rows_per_split", "nsplit",
            "tiles", "smem_bytes", "split_mode", "ctas", "column_blocks")
    return dict(zip(keys, list(info)))


def gqa_attn_device_status(stream=None, clear: bool = True) -> None:
    _check_attn(lib.gqa_attn_device_status(_stream_handle(stream), 1 if clear else 0))
