"""GPU parity of the AV reduction on shapes and pointers the TMA kernels do not
take: any head dimension (D % 8 != 0, the page's 4-wide texels and below) and
attn / V / out that are aligned only to their element type. Those calls run the
generic kernel; the gate is the AV call's, max|gpu - oracle| <= 1e-4 *
max(1, max|oracle|), with NaN in every padding row.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import bits, rand_case

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def gq():
    from gqa_attention_weighted_gb300 import build
    build.build()
    import gqa_attention_weighted_gb300 as pkg
    return pkg


def ref_of(attn, v, sl, vd):
    return oracle.gqa_av(attn.numpy(), bits(v), vd, None if sl is None else sl.numpy(),
                         nthreads=oracle.host_cores())


def check(got, ref, what):
    tol = TOL * max(1.0, float(np.abs(ref).max()))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max())
    assert err <= tol, f"{what}: max|gpu-oracle| = {err:.3e} > {tol:.3e}"


def shifted(t, k, dev):
    """A copy of `t` on `dev` that starts k elements into its allocation."""
    store = torch.empty(t.numel() + 8, dtype=t.dtype, device=dev)
    view = store[k:k + t.numel()].view(t.shape)
    view.copy_(t.to(dev))
    return view


DS = [1, 2, 4, 12, 36, 100, 260, 300]


@pytest.mark.parametrize("D", DS)
@pytest.mark.parametrize("G", [1, 3, 4, 12])
def test_any_head_dim(gq, D, G):
    rng = np.random.default_rng(10 * D + G)
    Hkv = 2
    B, C = 3, 700
    lens = [700, 1, 0]
    dev = torch.device("cuda")
    for vd in ("bf16", "fp16"):
        attn, v, sl = rand_case(rng, B, C, G * Hkv, Hkv, D, vd, lens)
        ref = ref_of(attn, v, sl, vd)
        plan = gq.gqa_av_plan(B, C, G * Hkv, Hkv, D, gq.native.v_dtype_code(v.dtype))
        assert plan["engine"] == 3 if D % 8 else plan["engine"] in (1, 2)
        for mode in (0, 1):
            out = torch.full((B, G * Hkv, D), 7.0, device=dev)
            gq.gqa_av_decode(attn.to(dev), v.to(dev), sl.to(dev), out, mode=mode)
            gq.gqa_av_device_status()
            got = out.cpu().double().numpy()
            check(got, ref, f"D={D} G={G} {vd} mode={mode}")
            assert np.all(got[2] == 0.0)


@pytest.mark.parametrize("ka,kv,ko", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 5, 2), (2, 4, 2)])
def test_element_aligned_pointers(gq, ka, kv, ko):
    """attn, V and out that start ka, kv, ko elements into their allocations
    (16-byte aligned only when all three are multiples of 4 / 8 / 4)."""
    rng = np.random.default_rng(100 + ka + 7 * kv + 31 * ko)
    B, C, Hq, Hkv, D = 2, 900, 16, 4, 128
    attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, "bf16", [900, 333])
    ref = ref_of(attn, v, sl, "bf16")
    dev = torch.device("cuda")
    a, vv = shifted(attn, ka, dev), shifted(v, kv, dev)
    out = shifted(torch.full((B, Hq, D), 7.0), ko, dev)
    for mode in (0, 1):
        gq.gqa_av_decode(a, vv, sl.to(dev), out, mode=mode)
        gq.gqa_av_device_status()
        check(out.cpu().double().numpy(), ref, f"shifts {ka},{kv},{ko} mode={mode}")


def test_generic_long_context_and_determinism(gq):
    """Many splits over a long ragged batch; repeated calls agree bitwise."""
    rng = np.random.default_rng(7)
    B, C, Hq, Hkv, D = 2, 20000, 8, 2, 20
    attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, "fp16", [20000, 12345])
    ref = ref_of(attn, v, sl, "fp16")
    dev = torch.device("cuda")
    outs = []
    for _ in range(2):
        out = torch.empty((B, Hq, D), device=dev)
        gq.gqa_av_decode(attn.to(dev), v.to(dev), sl.to(dev), out)
        gq.gqa_av_device_status()
        outs.append(out.cpu().double().numpy())
    check(outs[0], ref, "long context")
    assert np.array_equal(outs[0], outs[1])
    assert gq.gqa_av_plan(B, C, Hq, Hkv, D, 1)["nsplit"] > 1


def test_generic_clamped_and_null_lengths(gq):
    rng = np.random.default_rng(8)
    B, C, Hq, Hkv, D = 3, 64, 6, 3, 10
    attn, v, _ = rand_case(rng, B, C, Hq, Hkv, D, "bf16", [C, C, C], pad_nan=False)
    dev = torch.device("cuda")
    out = torch.empty((B, Hq, D), device=dev)
    gq.gqa_av_decode(attn.to(dev), v.to(dev), None, out)
    check(out.cpu().double().numpy(), ref_of(attn, v, None, "bf16"), "null lengths")
    sl = torch.tensor([500, -2, 17], dtype=torch.int32)
    gq.gqa_av_decode(attn.to(dev), v.to(dev), sl.to(dev), out)
    got = out.cpu().double().numpy()
    check(got, ref_of(attn, v, sl, "bf16"), "clamped lengths")
    assert np.all(got[1] == 0.0)
