"""GPU parity of the paged-V entry point (gqa_av_decode_paged) against the
fp64 oracle on the equivalent contiguous cache.

The pool's blocks are a random permutation; blocks the table does not use,
rows past each length and past Cmax hold NaN; table entries of blocks past a
length are garbage (negative, past the pool, or some other block).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import TORCH_V, bits, rand_case

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def gq():
    from gqa_attention_weighted_gb300 import build
    build.build()
    import gqa_attention_weighted_gb300 as pkg
    return pkg


def make_paged(rng, v, lens, bs):
    B, C, Hkv, D = v.shape
    maxb = math.ceil(C / bs)
    nblocks = B * maxb + 3
    pool = torch.full((nblocks, bs, Hkv, D), float("nan"), dtype=v.dtype)
    perm = rng.permutation(nblocks)
    table = np.empty((B, maxb), dtype=np.int32)
    for b in range(B):
        used = math.ceil(max(0, min(int(lens[b]), C)) / bs)
        for j in range(maxb):
            blk = int(perm[b * maxb + j])
            if j < used:
                rows = min(bs, C - j * bs)
                pool[blk, :rows] = v[b, j * bs:j * bs + rows]
                table[b, j] = blk
            else:
                table[b, j] = (-1, nblocks + 5, blk)[(b + j) % 3]
    return pool, torch.from_numpy(table)


def run_paged(gq, attn, pool, table, sl, mode, tuning=None):
    dev = torch.device("cuda")
    B, C, Hq = attn.shape
    out = torch.full((B, Hq, pool.shape[3]), float("nan"), device=dev)
    gq.gqa_av_decode_paged(attn.to(dev), pool.to(dev), table.to(dev), sl.to(dev), out,
                           mode=mode, tuning=tuning)
    gq.gqa_av_device_status()
    return out.cpu().double().numpy()


CASES = [(4, 128, 16), (4, 128, 64), (1, 64, 8), (8, 128, 32), (16, 256, 16), (3, 128, 256),
         (16, 64, 128), (2, 256, 48)]


@pytest.mark.parametrize("engine", [0, 1, 2], ids=["auto", "fma", "tensor"])
@pytest.mark.parametrize("G,D,bs", CASES, ids=[f"G{g}-D{d}-bs{b}" for g, d, b in CASES])
def test_paged_matches_contiguous_oracle(gq, G, D, bs, engine):
    rng = np.random.default_rng(G * 1000 + D + bs)
    Hkv = 2
    B, C = 3, 517
    lens = [517, 0, 300]
    for vd in ("bf16", "fp16"):
        attn, v, sl = rand_case(rng, B, C, G * Hkv, Hkv, D, vd, lens)
        ref = oracle.gqa_av(attn.numpy(), bits(v), vd, sl.numpy(), nthreads=oracle.host_cores())
        pool, table = make_paged(rng, v, lens, bs)
        for mode in (0, 1):
            heads = G if mode == 1 else 1
            if engine == 2 and not (heads <= 64 and D >= 64):
                continue
            tun = dict(engine=engine) if engine else None
            got = run_paged(gq, attn, pool, table, sl, mode, tun)
            tol = TOL * max(1.0, float(np.abs(ref).max()))
            assert np.all(np.isfinite(got)), (G, D, bs, vd, mode)
            err = float(np.abs(got - ref).max())
            assert err <= tol, f"G={G} D={D} bs={bs} {vd} mode={mode} engine={engine}: {err:.3e}"


@pytest.mark.parametrize("split_mode", [1, 2], ids=["fixed", "balanced"])
def test_paged_split_rules_and_large_batch(gq, split_mode):
    rng = np.random.default_rng(77)
    B, C, Hq, Hkv, D, bs = 40, 700, 16, 2, 128, 32
    lens = list(rng.integers(0, C + 1, size=B))
    attn, v, sl = rand_case(rng, B, C, Hq, Hkv, D, "bf16", lens)
    ref = oracle.gqa_av(attn.numpy(), bits(v), "bf16", sl.numpy(), nthreads=oracle.host_cores())
    pool, table = make_paged(rng, v, lens, bs)
    got = run_paged(gq, attn, pool, table, sl, 1, dict(engine=2, split_mode=split_mode, nsplit=3))
    tol = TOL * max(1.0, float(np.abs(ref).max()))
    assert float(np.abs(got - ref).max()) <= tol
    again = run_paged(gq, attn, pool, table, sl, 1, dict(engine=2, split_mode=split_mode, nsplit=3))
    assert np.array_equal(got, again), "not bitwise reproducible"


def test_paged_argument_checks(gq):
    dev = torch.device("cuda")
    attn = torch.zeros((1, 64, 4), device=dev)
    pool = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    out = torch.full((1, 4, 64), 3.0, device=dev)
    short = torch.zeros((1, 2), dtype=torch.int32, device=dev)      # 2 x 16 < Cmax = 64
    with pytest.raises(gq.GqaAvError) as e:
        gq.gqa_av_decode_paged(attn, pool, short, None, out)
    assert e.value.status == 1
    odd = torch.zeros((4, 12, 2, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(gq.GqaAvError) as e:
        gq.gqa_av_decode_paged(attn, odd, torch.zeros((1, 6), dtype=torch.int32, device=dev),
                               None, out)
    assert e.value.status == 1                                     # block_size % 8 != 0
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
