"""GPU parity of the decode score step (through the C ABI) against its fp64 oracle.

Gate (tests/helpers.py, qk_gate): every written probability (c < L_b) within
1e-4 of the oracle's value relative to that value (plus 1e-12), and every row
summing to 1 within 1e-5. Softmax probabilities at workload lengths are of
order 1/L, so an absolute bound would not check them. Rows c >= L_b must keep
the value they had. K rows past a length hold NaN, so a kernel that uses an
out-of-range row fails.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import gqa_qk
from helpers import TORCH_V, bits, qk_gate

pytestmark = pytest.mark.gpu

TOL = 1e-4
SENTINEL = 7.0


@pytest.fixture(scope="module")
def gq():
    from gqa_attention_weighted_gb300 import build
    build.build()
    import gqa_attention_weighted_gb300 as pkg
    return pkg


def qk_case(rng, B, C, Hq, Hkv, D, kd, lens, pad_nan=True):
    q = torch.tensor(rng.standard_normal((B, Hq, D)), dtype=torch.float32)
    k = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(TORCH_V[kd])
    sl = torch.tensor(np.asarray(lens), dtype=torch.int32)
    if pad_nan:
        for b in range(B):
            k[b, max(0, min(int(lens[b]), C)):] = float("nan")
    return q, k, sl


def run_qk(gq, q, k, sl, mode=-1, scale=None, engine=0):
    dev = torch.device("cuda")
    B, Hq, D = q.shape
    C = k.shape[1]
    attn = torch.full((B, C, Hq), SENTINEL, dtype=torch.float32, device=dev)
    gq.gqa_qk_softmax_decode(q.to(dev), k.to(dev), None if sl is None else sl.to(dev), attn,
                             mode=mode, scale=scale, engine=engine)
    gq.gqa_qk_device_status()
    return attn.cpu().double().numpy()


def check(got, ref, lens, what):
    B, C, _ = got.shape
    qk_gate(got, ref, lens, what)
    for b in range(B):
        L = max(0, min(int(lens[b]), C)) if lens is not None else C
        assert np.all(got[b, L:] == SENTINEL), f"{what}: rows past L_b={L} were written"


SWEEP = [(g, d) for g in (1, 2, 3, 4, 8, 16, 32, 64) for d in (64, 128, 256)] + [(5, 256), (12, 128), (24, 64)]


ENGINES = [0, 1, 2, 3]
ENGINE_IDS = ["auto", "fma", "tensor", "stream"]


@pytest.mark.parametrize("engine", ENGINES, ids=ENGINE_IDS)
@pytest.mark.parametrize("G,D", SWEEP, ids=[f"G{g}-D{d}" for g, d in SWEEP])
def test_score_step_shape_sweep(gq, G, D, engine):
    rng = np.random.default_rng(100 * G + D)
    Hkv = 2 if G <= 16 else 1
    B, C = 3, 517
    lens = [517, 1, 200]
    for kd in ("bf16", "fp16"):
        q, k, sl = qk_case(rng, B, C, G * Hkv, Hkv, D, kd, lens)
        scale = D ** -0.5
        ref = gqa_qk.gqa_qk_softmax(q.numpy(), bits(k), kd, sl.numpy(), scale)
        for mode in (0, 1):
            if engine == 3 and mode == 1 and G == 64 and D == 256:
                # 64 heads at D = 256: the streamed kernel's double-buffered
                # queries and two 64 KiB stages exceed shared memory; auto
                # takes the fixed-split kernel there (checked with engine 0).
                with pytest.raises(gq.GqaAvError) as e:
                    run_qk(gq, q, k, sl, mode, engine=engine)
                assert e.value.status == 2 and "shared memory" in str(e.value)
                continue
            got = run_qk(gq, q, k, sl, mode, engine=engine)
            check(got, ref, lens, f"G={G} D={D} {kd} mode={mode} engine={engine}")


@pytest.mark.parametrize("engine", [1, 2, 3], ids=["fma", "tensor", "stream"])
@pytest.mark.parametrize("L", [0, 1, 2, 31, 32, 33, 127, 128, 129, 255, 256, 257, 1000, 4095, 4096])
def test_score_step_lengths(gq, L, engine):
    rng = np.random.default_rng(L + 3)
    B, C, Hq, Hkv, D = 2, 4096, 8, 2, 128
    lens = [L, 4096 - L]
    q, k, sl = qk_case(rng, B, C, Hq, Hkv, D, "bf16", lens)
    ref = gqa_qk.gqa_qk_softmax(q.numpy(), bits(k), "bf16", sl.numpy(), D ** -0.5)
    check(run_qk(gq, q, k, sl, engine=engine), ref, lens, f"L={L} engine={engine}")


@pytest.mark.parametrize("engine", [1, 2, 3], ids=["fma", "tensor", "stream"])
def test_score_step_null_lengths_clamping_scale_and_determinism(gq, engine):
    rng = np.random.default_rng(7)
    B, C, Hq, Hkv, D = 3, 300, 8, 2, 64
    q, k, _ = qk_case(rng, B, C, Hq, Hkv, D, "fp16", [C] * B, pad_nan=False)
    full = gqa_qk.gqa_qk_softmax(q.numpy(), bits(k), "fp16", None, 0.3)
    a = run_qk(gq, q, k, None, scale=0.3, engine=engine)
    check(a, full, None, "seq_lens=NULL")
    over = torch.tensor([300, 301, 1 << 30], dtype=torch.int32)
    check(run_qk(gq, q, k, over, scale=0.3, engine=engine), full, [300, 300, 300],
          "lengths above Cmax")
    neg = run_qk(gq, q, k, torch.tensor([0, -4, -(1 << 30)], dtype=torch.int32), scale=0.3,
                 engine=engine)
    assert np.all(neg == SENTINEL), "non-positive lengths wrote rows"
    assert np.array_equal(run_qk(gq, q, k, None, scale=0.3, engine=engine), a), \
        "not bitwise reproducible"
    # The two modes agree.
    check(run_qk(gq, q, k, None, 0, 0.3, engine=engine), full, None, "per-head")


@pytest.mark.parametrize("engine", [1, 2, 3], ids=["fma", "tensor", "stream"])
@pytest.mark.parametrize("name", ["small", "llama", "phi", "mqa"])
def test_score_step_workload_shapes(gq, name, engine):
    """The AV workloads' shapes, with K drawn like V, and the chained call:
    the AV reduction on the score step's weights against the oracles' chain."""
    from gqa_attention_weighted_gb300 import workloads as W
    w = W.get(name)
    rng = np.random.default_rng(5)
    gen = torch.Generator().manual_seed(w.seed)
    lens = torch.randint(w.lo, w.hi + 1, (w.B,), generator=gen).to(torch.int32).numpy()
    q, k, sl = qk_case(rng, w.B, w.Cmax, w.Hq, w.Hkv, w.D, w.v_dtype, lens)
    scale = w.D ** -0.5
    ref = gqa_qk.gqa_qk_softmax(q.numpy(), bits(k), w.v_dtype, sl.numpy(), scale)
    got = run_qk(gq, q, k, sl, engine=engine)
    check(got, ref, lens, f"{name} engine={engine}")
    # Chain: out = AV(attn from the score step, V); V reuses K's shape.
    dev = torch.device("cuda")
    v = torch.tensor(rng.standard_normal((w.B, w.Cmax, w.Hkv, w.D)),
                     dtype=torch.float32).to(TORCH_V[w.v_dtype])
    attn = torch.tensor(got, dtype=torch.float32)
    for b in range(w.B):
        attn[b, int(lens[b]):] = 0.0
    out = torch.empty((w.B, w.Hq, w.D), device=dev)
    gq.gqa_av_decode(attn.to(dev), v.to(dev), sl.to(dev), out)
    gq.gqa_av_device_status()
    ref_attn = ref.astype(np.float32)
    ref_out = oracle.gqa_av(ref_attn, bits(v), w.v_dtype, sl.numpy(), nthreads=oracle.host_cores())
    o = out.cpu().double().numpy()
    tol = TOL * max(1.0, float(np.abs(ref_out).max()))
    assert float(np.abs(o - ref_out).max()) <= tol, "chained score step + AV"


def test_score_step_errors_launch_nothing(gq):
    dev = torch.device("cuda")
    q = torch.zeros((1, 4, 96), device=dev)
    k = torch.zeros((1, 16, 2, 96), dtype=torch.bfloat16, device=dev)
    attn = torch.full((1, 16, 4), SENTINEL, device=dev)
    with pytest.raises(gq.GqaAvError) as e:
        gq.gqa_qk_softmax_decode(q, k, None, attn)
    assert e.value.status == 2
    torch.cuda.synchronize()
    assert torch.all(attn == SENTINEL)


# The streamed kernel over batches past one and several warps of lengths (its
# first stage is found by a warp scan over the lengths), empty sequences, one
# long sequence among short ones, and fewer stages than CTAs.
@pytest.mark.parametrize("B,kind", [(33, "mix"), (70, "mix"), (40, "one_long"), (5, "all_empty"),
                                    (3, "short")])
def test_score_step_streamed_over_the_batch(gq, B, kind):
    rng = np.random.default_rng(B)
    C, Hq, Hkv, D = 700, 16, 4, 64
    if kind == "one_long":
        lens = [3] * B
        lens[B // 2] = C
    elif kind == "all_empty":
        lens = [0] * B
    elif kind == "short":
        lens = [1, 0, 5]
    else:
        lens = list(rng.integers(0, C + 1, size=B))
        lens[3] = 0
        lens[7 % B] = C
    q, k, sl = qk_case(rng, B, C, Hq, Hkv, D, "bf16", lens)
    ref = gqa_qk.gqa_qk_softmax(q.numpy(), bits(k), "bf16", sl.numpy(), D ** -0.5)
    for mode in (0, 1):
        a = run_qk(gq, q, k, sl, mode, engine=3)
        check(a, ref, lens, f"B={B} {kind} mode={mode}")
        assert np.array_equal(run_qk(gq, q, k, sl, mode, engine=3), a), "not reproducible"


# Calls long enough that each normalise CTA rewrites its rows in several
# batches (the grid is capped near ten CTAs an SM on these), with 16-byte
# loads (Hq % 4 == 0) and with 4-byte loads (Hq = 6), ragged lengths with
# empty and full sequences, on both score kernels and their normalise steps.
@pytest.mark.parametrize("engine", [2, 3], ids=["tensor", "stream"])
@pytest.mark.parametrize("B,C,Hq,Hkv", [(64, 16384, 8, 1), (48, 16384, 6, 1)], ids=["vec4", "scalar"])
def test_score_step_normalise_in_batches(gq, B, C, Hq, Hkv, engine):
    D = 64
    rng = np.random.default_rng(B + Hq)
    lens = rng.integers(0, C + 1, size=B)
    lens[0], lens[1], lens[2] = 0, C, 1
    q = torch.from_numpy(rng.standard_normal((B, Hq, D), dtype=np.float32))
    k = torch.from_numpy(rng.standard_normal((B, C, Hkv, D), dtype=np.float32)).to(torch.bfloat16)
    for b in range(B):
        k[b, int(lens[b]):] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    ref = gqa_qk.gqa_qk_softmax(q.numpy(), bits(k), "bf16", sl.numpy(), D ** -0.5)
    got = run_qk(gq, q, k, sl, engine=engine)
    check(got, ref, lens, f"B={B} Hq={Hq} engine={engine}")


# One sequence over many splits or groups: more than 32 (max, sum) pairs a
# head, so the normalise step merges them with the shared-memory path
# (Hq = 8: 1024 pairs staged) or reads them from global memory (Hq = 32:
# 4096 pairs, past the staging buffer), on both score kernels.
@pytest.mark.parametrize("engine", [2, 3], ids=["tensor", "stream"])
@pytest.mark.parametrize("Hq", [8, 32])
@pytest.mark.parametrize("L", [16384, 9001])
def test_score_step_many_segments(gq, Hq, L, engine):
    C, Hkv, D = 16384, 1, 64
    rng = np.random.default_rng(Hq + L)
    q, k, sl = qk_case(rng, 1, C, Hq, Hkv, D, "bf16", [L])
    ref = gqa_qk.gqa_qk_softmax(q.numpy(), bits(k), "bf16", sl.numpy(), D ** -0.5)
    got = run_qk(gq, q, k, sl, engine=engine)
    check(got, ref, [L], f"Hq={Hq} L={L} engine={engine}")
    assert np.array_equal(run_qk(gq, q, k, sl, engine=engine), got), "not reproducible"
