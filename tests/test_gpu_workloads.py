"""GPU parity on the five decode workloads, in the launch configuration the
benchmark times (the library's default plan).

The four workloads that fit the oracle in seconds are compared element by
element on inputs drawn on the CPU. The ~8.6 GB large-batch workload (and its
1/8-context profiling twin) is drawn on the GPU and compared element by element
too, one sequence at a time: the oracle runs on that sequence's in-range
context (all heads), so every output row, every split seam of the
length-balanced splits and every head of every group is checked. Properties
that hold at any size (determinism, per-head vs GQA-reuse agreement, the other
engine) are checked on the whole output as well.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_attention_weighted_gb300 import workloads as W
from helpers import bits

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def gq():
    from gqa_attention_weighted_gb300 import build
    build.build()
    import gqa_attention_weighted_gb300 as pkg
    return pkg


def _gate(got, ref, what):
    tol = TOL * max(1.0, float(np.abs(ref).max()))
    assert np.all(np.isfinite(got)), what
    err = float(np.abs(got - ref).max())
    assert err <= tol, f"{what}: max|gpu-oracle| = {err:.3e} > {tol:.3e}"


_REFS = {}


def _dense_case(name):
    """Inputs (NaN padding) and the oracle's result, drawn once per workload."""
    if name not in _REFS:
        w = W.get(name)
        x = W.generate(w, "cpu", pad="nan")
        ref = oracle.gqa_av(x["attn"].numpy(), bits(x["v"]), w.v_dtype, x["seq_lens"].numpy(),
                            nthreads=oracle.host_cores())
        _REFS[name] = (w, x, ref)
    return _REFS[name]


@pytest.mark.parametrize("engine", [0, 1, 2, 3], ids=["auto", "fma", "tensor", "stream"])
@pytest.mark.parametrize("name", ["small", "llama", "phi", "mqa"])
def test_workload_dense(gq, name, engine):
    w, x, ref = _dense_case(name)
    dev = torch.device("cuda")
    attn, v, sl = x["attn"].to(dev), x["v"].to(dev), x["seq_lens"].to(dev)
    tuning = (dict(engine=2, split_mode=3) if engine == 3 else
              dict(engine=engine) if engine else None)

    def call(out, mode=gq.MODE_AUTO):
        if tuning is None:
            gq.gqa_av_decode(attn, v, sl, out, mode=mode)
        else:
            gq.gqa_av_decode_tuned(attn, v, sl, out, mode=mode, tuning=tuning)

    outs = []
    for mode in (gq.MODE_AUTO, gq.MODE_GQA, gq.MODE_PER_HEAD):
        out = torch.full((w.B, w.Hq, w.D), float("nan"), device=dev)
        call(out, mode)
        gq.gqa_av_device_status()
        got = out.cpu().double().numpy()
        _gate(got, ref, f"{name} mode={mode} engine={engine}")
        outs.append(got)
    again = torch.empty((w.B, w.Hq, w.D), device=dev)
    call(again)
    assert np.array_equal(again.cpu().double().numpy(), outs[0]), "not bitwise reproducible"


@pytest.mark.parametrize("name", ["large", "ragged"])
def test_workload_large_full(gq, name):
    w = W.get(name)
    dev = torch.device("cuda")
    x = W.generate(w, dev, pad="zero")
    attn, v, sl = x["attn"], x["v"], x["seq_lens"]
    out = torch.empty((w.B, w.Hq, w.D), device=dev)
    gq.gqa_av_decode(attn, v, sl, out)
    gq.gqa_av_device_status()
    got = out.cpu().double().numpy()
    lens = sl.cpu().tolist()
    ref = np.empty_like(got)
    for b in range(w.B):  # one sequence at a time keeps the host copy small
        L = lens[b]
        a_b = attn[b:b + 1, :L].contiguous().cpu().numpy()
        v_b = v[b:b + 1, :L].contiguous().cpu()
        ref[b] = oracle.gqa_av(a_b, bits(v_b), w.v_dtype, None,
                               nthreads=oracle.host_cores())[0]
    for b in range(w.B):
        _gate(got[b], ref[b], f"{name} b={b} (L={lens[b]})")
    _gate(got, ref, f"{name} whole output")
    again = torch.empty_like(out)
    gq.gqa_av_decode(attn, v, sl, again)
    assert torch.equal(again, out), "not bitwise reproducible"
    per = torch.empty_like(out)
    gq.gqa_av_decode(attn, v, sl, per, mode=gq.MODE_PER_HEAD)
    gq.gqa_av_device_status()
    tol = TOL * max(1.0, float(out.abs().max()))
    assert float((per - out).abs().max()) <= tol
    # The other kernels on the whole output (the library picks tensor cores here).
    for tun in (dict(engine=1), dict(engine=2, split_mode=3), dict(engine=2, split_mode=2)):
        other = torch.empty_like(out)
        gq.gqa_av_decode_tuned(attn, v, sl, other, tuning=tun)
        gq.gqa_av_device_status()
        assert float((other - out).abs().max()) <= tol, tun
