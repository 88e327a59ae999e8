"""A bounded wait inside the kernel that runs out is reported, and the next
call is correct (failure detection without a GPU fault).

gqa_av_selftest_wait_timeout runs the CUDA-core FMA kernel with the producer
withholding each split's last stage (nothing of it is issued, so nothing is in
flight) and the consumers' wait for a stage limited to 200 us. Their wait for
the withheld stage runs out: they set the device status word and leave. The
host then reads GQA_AV_ERR_DEVICE_TIMEOUT from gqa_av_device_status, once for
the workspace's word and once for the no-allocation call's fixed array, clears
it, and the next normal call matches the oracle.
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
WAIT_NS = 200_000


@pytest.fixture(scope="module")
def native():
    from gqa_attention_weighted_gb300 import build
    build.build()
    from gqa_attention_weighted_gb300 import _native
    return _native


def _args(x, out, w, vd, stream):
    return (x["attn"].data_ptr(), x["v"].data_ptr(), x["seq_lens"].data_ptr(), out.data_ptr(),
            w.B, w.Cmax, w.Hq, w.Hkv, w.D, vd)


@pytest.mark.parametrize("scratch", [0, 1], ids=["workspace", "noalloc_array"])
def test_wait_that_runs_out_is_reported_and_cleared(native, scratch):
    # Llama-style heads, full lengths: every split has four stages.
    w = W.custom(1, 8192, 32, 8, 128, "bf16")
    xc = W.generate(w, "cpu", pad="nan", seed=31)
    x = {k: t.cuda() for k, t in xc.items()}
    vd = native.v_dtype_code(x["v"].dtype)
    stream = torch.cuda.current_stream().cuda_stream
    lib = native.lib
    native.gqa_av_device_status()  # start from a clear status word (raises if set)
    if scratch == 1:  # the fixed array is set up by the first no-allocation call
        out0 = torch.empty((w.B, w.Hq, w.D), device="cuda")
        assert lib.gqa_av_decode_noalloc(*_args(x, out0, w, vd, stream), -1,
                                         ctypes.c_void_p(stream)) == 0
        assert lib.gqa_av_device_status(ctypes.c_void_p(stream), 0) == 0

    out = torch.zeros((w.B, w.Hq, w.D), device="cuda")
    rc = lib.gqa_av_selftest_wait_timeout(*_args(x, out, w, vd, stream), WAIT_NS, scratch,
                                          ctypes.c_void_p(stream))
    assert rc == 0, native.gqa_av_last_error()
    # Reported, and still reported until cleared.
    assert lib.gqa_av_device_status(ctypes.c_void_p(stream), 0) == native.GQA_AV_ERR_DEVICE_TIMEOUT
    assert "0x1" in native.gqa_av_last_error()  # the consumers' stage wait
    assert lib.gqa_av_device_status(ctypes.c_void_p(stream), 1) == native.GQA_AV_ERR_DEVICE_TIMEOUT
    assert lib.gqa_av_device_status(ctypes.c_void_p(stream), 0) == 0

    # The context is intact: the next normal call is correct.
    exact = oracle.gqa_av(xc["attn"].numpy(), bits(xc["v"]), "bf16", xc["seq_lens"].numpy(),
                          nthreads=oracle.host_cores())
    got = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
    if scratch == 1:
        assert lib.gqa_av_decode_noalloc(*_args(x, got, w, vd, stream), -1,
                                         ctypes.c_void_p(stream)) == 0
    else:
        native.gqa_av_decode(x["attn"], x["v"], x["seq_lens"], got)
    native.gqa_av_device_status()
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g))
    assert float(np.abs(g - exact).max()) <= TOL * max(1.0, float(np.abs(exact).max()))


def test_selftest_rejects_bad_arguments(native):
    w = W.custom(1, 64, 8, 2, 64, "bf16")
    x = {k: t.cuda() for k, t in W.generate(w, "cpu").items()}
    out = torch.empty((w.B, w.Hq, w.D), device="cuda")
    vd = native.v_dtype_code(x["v"].dtype)
    lib = native.lib
    for wait_ns, scratch in ((10, 0), (3_000_000_000, 0), (WAIT_NS, 2)):
        assert lib.gqa_av_selftest_wait_timeout(*_args(x, out, w, vd, None), wait_ns, scratch,
                                                None) == native.GQA_AV_ERR_INVALID
    torch.cuda.synchronize()
    assert native.lib.gqa_av_device_status(None, 0) == 0
