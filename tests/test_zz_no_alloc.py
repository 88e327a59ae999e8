"""gqa_av_decode_noalloc, the entry point for callers that may not allocate
device memory (engine plug-ins whose host owns all device memory, loops that
must not risk an allocation's implicit synchronisation, fixed memory budgets).

It is called through the C ABI and must match the fp64 oracle, and gqa_av_decode
(the allocating entry point), within the parity tolerance on two calls in a row
(the second with different inputs, so stale scratch contents would show). Its
status word must be reported by gqa_av_device_status. This file is collected
last so a stop-at-first-failure run has already run everything else; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gqa_attention_weighted_gb300 import workloads as W
from helpers import bits

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def native():
    from gqa_attention_weighted_gb300 import build
    build.build()
    from gqa_attention_weighted_gb300 import _native
    return _native


def _inputs(w, seed):
    x = W.generate(w, "cpu", pad="nan", seed=seed)
    ref = oracle.gqa_av(x["attn"].numpy(), bits(x["v"]), w.v_dtype, x["seq_lens"].numpy(),
                        nthreads=oracle.host_cores())
    return {k: t.cuda() for k, t in x.items()}, ref


def _call_noalloc(native, x, out, w, mode):
    vd = native.v_dtype_code(x["v"].dtype)
    stream = torch.cuda.current_stream().cuda_stream
    return native.lib.gqa_av_decode_noalloc(
        x["attn"].data_ptr(), x["v"].data_ptr(), x["seq_lens"].data_ptr(), out.data_ptr(),
        w.B, w.Cmax, w.Hq, w.Hkv, w.D, vd, mode, ctypes.c_void_p(stream))


SHAPES = [
    W.custom(1, 8192, 32, 8, 128, "bf16"),                       # Llama-style, split combine
    W.custom(3, 2000, 24, 8, 128, "bf16", len_lo=0, len_hi=2000),  # G=3, ragged, empty rows
    W.custom(2, 4096, 16, 1, 256, "fp16", len_lo=1, len_hi=4096),  # G=16 MQA, fp16
]


@pytest.mark.parametrize("w", SHAPES, ids=[w.name for w in SHAPES])
@pytest.mark.parametrize("mode", [-1, 0])
def test_noalloc_matches_allocating_entry_point(native, w, mode):
    for seed in (11, 12):  # two calls in a row, different inputs
        x, exact = _inputs(w, seed)
        ref = torch.empty((w.B, w.Hq, w.D), device="cuda")
        native.gqa_av_decode(x["attn"], x["v"], x["seq_lens"], ref, mode=mode)
        out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        rc = _call_noalloc(native, x, out, w, mode)
        assert rc == 0, native.gqa_av_last_error()
        torch.cuda.synchronize()
        assert native.lib.gqa_av_device_status(None, 0) == 0, "a bounded wait ran out"
        r, o = ref.double().cpu().numpy(), out.double().cpu().numpy()
        tol = TOL * max(1.0, float(np.abs(exact).max()))
        assert np.all(np.isfinite(o))
        assert float(np.abs(o - exact).max()) <= tol, "no-allocation call vs the oracle"
        assert float(np.abs(r - exact).max()) <= tol, "gqa_av_decode vs the oracle"
        assert float(np.abs(o - r).max()) <= tol, "no-allocation call vs gqa_av_decode"


def test_noalloc_rejects_shapes_beyond_its_scratch(native):
    # G = 128 heads on one KV head: a plan with many split partials of 128 x D floats.
    B, C, Hq, Hkv, D = 1, 65536, 128, 1, 256
    plan = native.gqa_av_plan(B, C, Hq, Hkv, D, native.GQA_AV_BF16, 1)
    partials = plan["workspace_bytes"] - 256
    cap = (8 << 20) - 256
    if partials <= cap:
        pytest.skip(f"plan needs only {partials} B of partials on this GPU")
    attn = torch.zeros((B, C, Hq), device="cuda")
    v = torch.zeros((B, C, Hkv, D), dtype=torch.bfloat16, device="cuda")
    sl = torch.full((B,), C, dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, D), 3.0, device="cuda")
    w = W.custom(B, C, Hq, Hkv, D)
    rc = _call_noalloc(native, {"attn": attn, "v": v, "seq_lens": sl}, out, w, 1)
    assert rc == native.GQA_AV_ERR_UNSUPPORTED
    assert "scratch" in native.gqa_av_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
