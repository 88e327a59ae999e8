"""The C-ABI library loads and exports every entry point its header declares;
host-side argument checks reject bad calls before any CUDA call (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("gqa_av.h", "gqa_qk.h", "gqa_attn.h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(gqa_(?:av|qk|attn)_\w+)\s*\(", text, re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def native():
    from gqa_attention_weighted_gb300 import build
    build.build()
    from gqa_attention_weighted_gb300 import _native
    return _native


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("gqa_av_decode", "gqa_av_decode_per_head", "gqa_av_status_string",
              "gqa_av_workspace_bytes", "gqa_qk_softmax_decode", "gqa_qk_device_status",
              "gqa_attn_decode", "gqa_attn_decode_tuned", "gqa_attn_plan",
              "gqa_attn_device_status", "gqa_attn_last_error"):
        assert f in names


def test_library_exports_every_declared_symbol(native):
    lib = ctypes.CDLL(native.LIBRARY)
    missing = [f for f in declared_functions() if not hasattr(lib, f)]
    assert not missing, f"declared but not exported: {missing}"


def test_status_strings(native):
    assert native.gqa_av_status_string(0) == "GQA_AV_OK"
    assert native.gqa_av_status_string(1) == "GQA_AV_ERR_INVALID"
    assert native.gqa_av_status_string(5) == "GQA_AV_ERR_DEVICE_TIMEOUT"
    assert native.gqa_av_status_string(99) == "GQA_AV_ERR_UNKNOWN"
    assert native.lib.gqa_av_version() == 1


# (attn, v, out) as fake non-NULL 16-byte-aligned addresses: every case below
# is rejected by the host checks before any pointer is touched or CUDA called.
FAKE = 1 << 20


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, None, FAKE, 1, 8, 6, 4, 8, 0, -1), 1),   # Hq % Hkv != 0
    ((FAKE, FAKE, None, FAKE, 0, 8, 4, 4, 8, 0, -1), 1),   # B == 0
    ((FAKE, FAKE, None, FAKE, 1, -3, 4, 4, 8, 0, -1), 1),  # Cmax < 0
    ((FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 8, 2, -1), 1),   # unknown dtype
    ((FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 8, 0, 3), 1),    # unknown mode
    ((None, FAKE, None, FAKE, 1, 8, 4, 4, 8, 0, -1), 1),   # NULL attn
    ((FAKE, FAKE, None, None, 1, 8, 4, 4, 8, 0, 1), 1),    # NULL out
    ((FAKE, FAKE + 1, None, FAKE, 1, 8, 4, 4, 12, 0, 1), 1),  # v not 2-byte aligned
    ((FAKE + 2, FAKE, None, FAKE, 1, 8, 4, 4, 8, 0, 0), 1),  # attn not 4-byte aligned
    ((FAKE, FAKE, None, FAKE + 2, 1, 8, 4, 4, 8, 0, 0), 1),  # out not 4-byte aligned
    ((FAKE, FAKE, FAKE + 2, FAKE, 1, 8, 4, 4, 8, 0, 0), 1),  # misaligned seq_lens
])
def test_host_checks_reject_before_launch(native, args, status):
    rc = native.lib.gqa_av_decode(*args, None)
    assert rc == status, native.gqa_av_last_error()
    assert native.gqa_av_last_error() != ""


def test_tunings_need_the_tma_kernels(native):
    # D % 8 != 0 runs the generic kernel, which takes no launch-shape tuning.
    t = native.Tuning(3, 0, 0, 0, 0, 0, 0)
    rc = native.lib.gqa_av_decode_tuned(FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 12, 0, -1,
                                        ctypes.byref(t), None)
    assert rc == 2 and "TMA" in native.gqa_av_last_error()


def test_per_head_entry_checks(native):
    rc = native.lib.gqa_av_decode_per_head(FAKE, FAKE, None, FAKE, 1, 8, 6, 4, 8, 0, None)
    assert rc == 1 and "multiple" in native.gqa_av_last_error()


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, None, FAKE, 1, 8, 6, 4, 64, 0, 1.0, -1), 1),    # Hq % Hkv != 0
    ((FAKE, FAKE, None, FAKE, 0, 8, 4, 4, 64, 0, 1.0, -1), 1),    # B == 0
    ((FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 64, 2, 1.0, -1), 1),    # unknown dtype
    ((FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0, 3), 1),     # unknown mode
    ((None, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0, -1), 1),    # NULL q
    ((FAKE, FAKE, None, None, 1, 8, 4, 4, 64, 0, 1.0, 1), 1),     # NULL attn
    ((FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 96, 0, 1.0, 1), 2),     # D % 64 != 0
    ((FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 320, 0, 1.0, 1), 2),    # D > 256
    ((FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 192, 0, 1.0, 1), 2),    # D = 192
    ((FAKE, FAKE, None, FAKE, 1, 8, 128, 1, 64, 0, 1.0, 1), 2),   # 128 heads on one KV head
    ((FAKE + 4, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0, 0), 2),  # misaligned q
])
def test_score_step_host_checks_reject_before_launch(native, args, status):
    rc = native.lib.gqa_qk_softmax_decode(*args, None)
    assert rc == status, native.lib.gqa_qk_last_error()
    assert native.lib.gqa_qk_last_error() != b""


# (q, k, v, seq_lens, out, B, Cmax, Hq, Hkv, D, kv_dtype, scale, mode)
@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, FAKE, None, FAKE, 1, 8, 6, 4, 64, 0, 1.0, -1), 1),    # Hq % Hkv != 0
    ((FAKE, FAKE, FAKE, None, FAKE, 0, 8, 4, 4, 64, 0, 1.0, -1), 1),    # B == 0
    ((FAKE, FAKE, FAKE, None, FAKE, 1, 0, 4, 4, 64, 0, 1.0, -1), 1),    # Cmax == 0
    ((FAKE, FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 64, 2, 1.0, -1), 1),    # unknown dtype
    ((FAKE, FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0, 3), 1),     # unknown mode
    ((None, FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0, -1), 1),    # NULL q
    ((FAKE, FAKE, None, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0, -1), 1),    # NULL v
    ((FAKE, FAKE, FAKE, None, None, 1, 8, 4, 4, 64, 0, 1.0, 1), 1),     # NULL out
    ((FAKE, FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, float("inf"), 1), 1),  # scale not finite
    ((FAKE, FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 96, 0, 1.0, 1), 2),     # D % 64 != 0
    ((FAKE, FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 512, 0, 1.0, 1), 2),    # D > 256
    ((FAKE, FAKE + 8, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0, 0), 2),  # misaligned k
])
def test_attention_host_checks_reject_before_launch(native, args, status):
    rc = native.lib.gqa_attn_decode(*args, None)
    assert rc == status, native.lib.gqa_attn_last_error()
    assert native.lib.gqa_attn_last_error() != b""


def test_attention_tuning_range_checked(native):
    for warps, splits, smode, ncol in ((9, 0, 0, 0), (-1, 0, 0, 0), (0, -2, 0, 0), (0, 0, 3, 0),
                                       (0, 0, 0, -1)):
        rc = native.lib.gqa_attn_decode_tuned(FAKE, FAKE, FAKE, None, FAKE, 1, 8, 4, 4, 64, 0, 1.0,
                                              -1, warps, splits, smode, ncol, None)
        assert rc == 1 and b"out of range" in native.lib.gqa_attn_last_error()


@pytest.mark.parametrize("wait_ns,scratch,D,status", [
    (10, 0, 64, 1),              # wait limit below 1 us
    (3_000_000_000, 0, 64, 1),   # above the 2 s every other wait has
    (200_000, 2, 64, 1),         # unknown scratch
    (200_000, 0, 12, 2),         # the self-test runs the TMA kernels only (D % 8 == 0)
])
def test_wait_timeout_selftest_checks_arguments(native, wait_ns, scratch, D, status):
    rc = native.lib.gqa_av_selftest_wait_timeout(FAKE, FAKE, None, FAKE, 1, 64, 8, 2, D, 0,
                                                 wait_ns, scratch, None)
    assert rc == status, native.gqa_av_last_error()
