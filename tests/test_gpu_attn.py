"""GPU parity of the fused decode attention (through the C ABI) against its fp64 oracle.

Gate: max|gpu - oracle| <= 1e-4 * max(1, max|oracle|) per case. K and V rows
past a sequence's length hold NaN, so a kernel that uses an out-of-range row
fails. Cases span several 32-row stages and context splits with ragged tails,
empty and one-row sequences, G from 1 to 32 (past one 16-head tile), every
supported D, both cache types and both modes.
"""
import numpy as np
import pytest
import torch

from oracle import gqa_attn
from helpers import TORCH_V, bits

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def gq():
    from gqa_attention_weighted_gb300 import build
    build.build()
    import gqa_attention_weighted_gb300 as pkg
    return pkg


def attn_case(rng, B, C, Hq, Hkv, D, kd, lens, q_sigma=1.0, pad_nan=True):
    q = torch.tensor(rng.standard_normal((B, Hq, D)) * q_sigma, dtype=torch.float32)
    k = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(TORCH_V[kd])
    v = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(TORCH_V[kd])
    sl = torch.tensor(np.asarray(lens), dtype=torch.int32)
    if pad_nan:
        for b in range(B):
            L = max(0, min(int(lens[b]), C))
            k[b, L:] = float("nan")
            v[b, L:] = float("nan")
    return q, k, v, sl


def run_attn(gq, q, k, v, sl, mode=-1, scale=None, warps=0, nsplit=0, split_mode=0, ncol=0):
    dev = torch.device("cuda")
    B, Hq, D = q.shape
    out = torch.full((B, Hq, D), 7.0, dtype=torch.float32, device=dev)
    gq.gqa_attn_decode(q.to(dev), k.to(dev), v.to(dev), None if sl is None else sl.to(dev), out,
                       mode=mode, scale=scale, consumer_warps=warps, nsplit=nsplit,
                       split_mode=split_mode, column_blocks=ncol)
    gq.gqa_attn_device_status()
    return out.cpu().double().numpy()


def oracle_of(q, k, v, sl, kd, scale):
    return gqa_attn.gqa_attention(q.numpy(), bits(k), bits(v), kd,
                                  None if sl is None else sl.numpy(), scale)


def check(got, ref, what):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max())
    tol = TOL * max(1.0, float(np.abs(ref).max()))
    assert err <= tol, f"{what}: max|gpu-oracle| = {err:.3e} > {tol:.3e}"


SWEEP = [(g, d) for g in (1, 2, 3, 4, 8, 16) for d in (64, 128, 256)] + [(5, 128), (12, 64),
                                                                         (24, 128), (32, 64)]


@pytest.mark.parametrize("G,D", SWEEP, ids=[f"G{g}-D{d}" for g, d in SWEEP])
def test_attention_shape_sweep(gq, G, D):
    rng = np.random.default_rng(1000 * G + D)
    Hkv = 2 if G <= 16 else 1
    B, C = 4, 517
    lens = [517, 1, 200, 0]
    scale = D ** -0.5
    for kd in ("bf16", "fp16"):
        q, k, v, sl = attn_case(rng, B, C, G * Hkv, Hkv, D, kd, lens, q_sigma=2.0)
        ref = oracle_of(q, k, v, sl, kd, scale)
        assert np.all(ref[3] == 0.0)
        for mode in (0, 1):
            for nsplit, smode in ((0, 0), (1, 1), (5, 1), (1, 2), (5, 2)):
                for ncol in ((0, 1, 2) if D == 256 else (0,)):
                    got = run_attn(gq, q, k, v, sl, mode, scale, nsplit=nsplit, split_mode=smode,
                                   ncol=ncol)
                    what = (f"G={G} D={D} {kd} mode={mode} nsplit={nsplit} split_mode={smode} "
                            f"column_blocks={ncol}")
                    check(got, ref, what)
                    assert np.all(got[3] == 0.0), f"{what}: an empty context must give out = 0"


@pytest.mark.parametrize("warps", [1, 2, 3, 4, 5, 6, 7, 8])
def test_attention_consumer_warps(gq, warps):
    """Every consumer-warp count (ring slots per warp, the warp merge, both
    compiled register bounds) gives the same result; D = 256 takes at most 6
    consumer warps and refuses more."""
    rng = np.random.default_rng(7 + warps)
    q, k, v, sl = attn_case(rng, 2, 1000, 8, 2, 64, "bf16", [1000, 333], q_sigma=2.0)
    ref = oracle_of(q, k, v, sl, "bf16", 64 ** -0.5)
    for nsplit, smode in ((0, 0), (1, 1), (3, 1), (3, 2)):
        check(run_attn(gq, q, k, v, sl, 1, 64 ** -0.5, warps=warps, nsplit=nsplit,
                       split_mode=smode), ref, f"warps={warps} nsplit={nsplit} split_mode={smode}")
    for D, kd, G in ((128, "bf16", 6), (256, "fp16", 16)):
        q, k, v, sl = attn_case(rng, 2, 700, 2 * G, 2, D, kd, [700, 90], q_sigma=2.0)
        if warps > 6 and D == 256:
            with pytest.raises(gq.GqaAvError):
                run_attn(gq, q, k, v, sl, 1, D ** -0.5, warps=warps)
            continue
        ref = oracle_of(q, k, v, sl, kd, D ** -0.5)
        for nsplit, smode in ((0, 0), (1, 1), (4, 2)):
            for ncol in ((1, 2) if D == 256 else (0,)):
                check(run_attn(gq, q, k, v, sl, 1, D ** -0.5, warps=warps, nsplit=nsplit,
                               split_mode=smode, ncol=ncol), ref,
                      f"D={D} warps={warps} split_mode={smode} column_blocks={ncol}")
    with pytest.raises(gq.GqaAvError):  # two column blocks need D = 256
        run_attn(gq, q[:, :, :64].contiguous(), k[..., :64].contiguous(), v[..., :64].contiguous(),
                 sl, ncol=2)


def test_attention_balanced_splits_many_sequences(gq):
    """Balanced splits over a batch of more sequences than a warp has lanes,
    with empty, one-row, full and clamped lengths mixed."""
    rng = np.random.default_rng(21)
    B, C = 40, 300
    lens = rng.integers(0, C + 1, size=B)
    lens[:6] = [0, 1, C, 5000, -3, 33]
    q, k, v, _ = attn_case(rng, B, C, 8, 2, 64, "bf16", np.clip(lens, 0, C), q_sigma=2.0)
    sl = torch.tensor(lens, dtype=torch.int32)
    ref = oracle_of(q, k, v, sl, "bf16", 0.125)
    for nsplit in (0, 1, 2, 9):
        check(run_attn(gq, q, k, v, sl, -1, 0.125, nsplit=nsplit, split_mode=2), ref,
              f"balanced nsplit={nsplit}")
        check(run_attn(gq, q, k, v, sl, -1, 0.125, nsplit=nsplit, split_mode=1), ref,
              f"fixed nsplit={nsplit}")


def test_attention_one_hot_scores_return_the_row(gq):
    """A score far above the others puts all the weight on one row: out = V row
    (exactly representable: every other weight underflows to 0)."""
    rng = np.random.default_rng(3)
    B, C, Hq, Hkv, D = 1, 300, 4, 1, 64
    k = torch.zeros((B, C, Hkv, D), dtype=torch.bfloat16)
    c0 = 217
    k[0, c0, 0, 0] = 1.0
    q = torch.zeros((B, Hq, D), dtype=torch.float32)
    q[0, :, 0] = 1000.0
    v = torch.tensor(rng.standard_normal((B, C, Hkv, D)), dtype=torch.float32).to(torch.bfloat16)
    got = run_attn(gq, q, k, v, None, 1, 1.0)
    want = v[0, c0, 0].double().numpy()
    for h in range(Hq):
        assert np.array_equal(got[0, h], want)


def test_attention_defaults_and_scale(gq):
    """scale=None means 1/sqrt(D); seq_lens=None means every length is Cmax."""
    rng = np.random.default_rng(5)
    q, k, v, _ = attn_case(rng, 2, 260, 6, 2, 64, "fp16", [260, 260], pad_nan=False)
    ref = oracle_of(q, k, v, None, "fp16", 64 ** -0.5)
    check(run_attn(gq, q, k, v, None), ref, "defaults")
    ref2 = oracle_of(q, k, v, None, "fp16", 0.3)
    check(run_attn(gq, q, k, v, None, scale=0.3), ref2, "scale 0.3")


def test_attention_lengths_clamped(gq):
    """seq_lens beyond Cmax act as Cmax, negative ones as 0."""
    rng = np.random.default_rng(6)
    q, k, v, _ = attn_case(rng, 3, 100, 4, 2, 64, "bf16", [100, 100, 100], pad_nan=False)
    sl = torch.tensor([1000, -5, 37], dtype=torch.int32)
    ref = oracle_of(q, k, v, sl, "bf16", 0.125)
    got = run_attn(gq, q, k, v, sl, scale=0.125)
    check(got, ref, "clamped")
    assert np.all(got[1] == 0.0)


def test_attention_deterministic(gq):
    rng = np.random.default_rng(8)
    q, k, v, sl = attn_case(rng, 3, 3000, 16, 4, 128, "bf16", [3000, 1777, 64])
    for smode in (1, 2):
        a = run_attn(gq, q, k, v, sl, nsplit=7, split_mode=smode)
        b = run_attn(gq, q, k, v, sl, nsplit=7, split_mode=smode)
        assert np.array_equal(a, b)


def test_attention_matches_chained_score_and_av_calls(gq):
    """The fused call against the score-step call followed by the AV call."""
    rng = np.random.default_rng(9)
    B, C, Hq, Hkv, D = 2, 900, 12, 4, 128
    q, k, v, sl = attn_case(rng, B, C, Hq, Hkv, D, "bf16", [900, 450])
    dev = torch.device("cuda")
    qd, kd_, vd, sld = q.to(dev), k.to(dev), v.to(dev), sl.to(dev)
    attn = torch.zeros((B, C, Hq), dtype=torch.float32, device=dev)
    gq.gqa_qk_softmax_decode(qd, kd_, sld, attn)
    chained = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    gq.gqa_av_decode(attn, vd, sld, chained)
    fused = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    gq.gqa_attn_decode(qd, kd_, vd, sld, fused)
    gq.gqa_attn_device_status()
    err = float((fused - chained).abs().max())
    assert err <= 2 * TOL * max(1.0, float(chained.abs().max()))


def _workload_inputs(name, dev):
    from gqa_attention_weighted_gb300 import workloads as W
    w = W.get(name)
    x = W.generate_qkv(w, dev, pad="nan")
    return w, x["q"], x["k"], x["v"], x["seq_lens"]


@pytest.mark.parametrize("name", ["small", "llama", "phi", "mqa"])
def test_attention_workloads_full(gq, name):
    """Every output of the decode workloads against the oracle at full size, in
    the launch configuration the benchmark times."""
    dev = torch.device("cuda")
    w, q, k, v, sl = _workload_inputs(name, dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    gq.gqa_attn_decode(q, k, v, sl, out)
    gq.gqa_attn_device_status()
    ref = oracle_of(q.cpu(), k.cpu(), v.cpu(), sl.cpu(), w.v_dtype, w.D ** -0.5)
    check(out.cpu().double().numpy(), ref, name)


def test_attention_large_batch_sampled(gq):
    """The large batch (B=32, C=131072, G=8) at full size: every head of a
    sample of (sequence, KV head) pairs against the oracle on that slice."""
    dev = torch.device("cuda")
    free, _ = torch.cuda.mem_get_info()
    if free < 40e9:
        pytest.skip("needs about 40 GB of free device memory")
    w, q, k, v, sl = _workload_inputs("large", dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    gq.gqa_attn_decode(q, k, v, sl, out)
    gq.gqa_attn_device_status()
    got = out.cpu().double().numpy()
    G = w.G
    rng = np.random.default_rng(11)
    for b, kv_h in [(0, 0), (31, 7)] + [tuple(x) for x in zip(rng.integers(0, w.B, 4),
                                                              rng.integers(0, w.Hkv, 4))]:
        L = int(sl[b])
        heads = slice(kv_h * G, (kv_h + 1) * G)
        ref = oracle_of(q[b:b + 1, heads].cpu(), k[b:b + 1, :L, kv_h:kv_h + 1].cpu(),
                        v[b:b + 1, :L, kv_h:kv_h + 1].cpu(), None, w.v_dtype, w.D ** -0.5)
        check(got[b:b + 1, heads], ref, f"large b={b} kv_h={kv_h}")


@pytest.mark.parametrize("D,kd", [(64, "bf16"), (128, "bf16"), (256, "fp16")])
def test_attention_many_splits(gq, D, kd):
    """More splits per sequence than a warp has lanes and than one batch of
    combine loads covers, on fixed and balanced splits."""
    rng = np.random.default_rng(300 + D)
    q, k, v, sl = attn_case(rng, 2, 6000, 8, 2, D, kd, [6000, 2500], q_sigma=2.0)
    ref = oracle_of(q, k, v, sl, kd, D ** -0.5)
    for nsplit, smode in ((150, 1), (150, 2)):
        plan = gq.gqa_attn_plan(2, 6000, 8, 2, D, gq.native.v_dtype_code(k.dtype), -1, 0,
                                nsplit, smode)
        assert plan["nsplit"] > 64
        check(run_attn(gq, q, k, v, sl, -1, D ** -0.5, nsplit=nsplit, split_mode=smode), ref,
              f"D={D} nsplit={nsplit} split_mode={smode}")
