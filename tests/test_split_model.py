"""A CPU model of how the split kernels cover a batch (no GPU).

The fused attention kernel and the tensor-core AV kernel spread a batch's
context rows over CTAs in one of two ways, and a combine kernel finds each
tile's split partials again. This model restates those rules with plain
integers and checks the properties the kernels rely on, over many random
batches:

- fixed splits: CTA (tile, split) covers rows [split * rps, (split + 1) * rps)
  of its sequence; splits at or past ceil(L / rps) have no work, except that
  an empty sequence keeps split 0 (which writes zeros);
- balanced splits: sequence b with s_b = ceil(L_b / R) stages gets
  n_b = max(1, ceil(s_b / sps)) splits of sps = ceil(K * sum_b s_b / units)
  stages; CTA u takes tile-in-sequence u % K and batch split u / K, the
  partial of CTA u is slot u, and the combine reads split s of sequence b at
  slot (P_b + s) * K + k, P_b = n_0 + ... + n_{b-1};
- at most units + K * B CTAs have work, which sizes the grid and the
  workspace.

Every (sequence, tile, row) must be covered exactly once, by a CTA inside the
grid, and the combine must find exactly the slots written for its tile.
"""
import random

R = 32  # rows per stage


def clamp(L, C):
    return max(0, min(L, C))


def fixed_cover(lens, C, K, rps):
    nsplit = -(-C // rps)
    cover = {}
    writes = {}
    for k in range(K):
        for b, L0 in enumerate(lens):
            L = clamp(L0, C)
            nsb = -(-L // rps) if L > 0 else 1
            tile = k * len(lens) + b
            for split in range(nsplit):
                if split >= nsb:
                    continue
                c0, c1 = split * rps, min((split + 1) * rps, L)
                if c1 > c0:
                    cover.setdefault((b, k), []).append((c0, c1))
                if nsb > 1:
                    writes[(b, k, split)] = tile * nsplit + split
    return cover, writes, K * len(lens) * nsplit


def balanced_cover(lens, C, K, units):
    B = len(lens)
    Ls = [clamp(L, C) for L in lens]
    stages = [-(-L // R) for L in Ls]
    sps = max(1, -(-(sum(stages) * K) // units))
    n = [max(1, -(-s // sps)) for s in stages]
    prefix = [sum(n[:b]) for b in range(B)]
    grid = units + K * B
    cover, writes = {}, {}
    used = 0
    for u in range(grid):
        k, q = u % K, u // K
        # the sequence whose splits contain batch split q
        found = None
        for b in range(B):
            if prefix[b] <= q < prefix[b] + n[b]:
                found = b
                break
        if found is None:
            continue
        used = max(used, u + 1)
        b, split = found, q - prefix[found]
        c0, c1 = split * sps * R, min((split + 1) * sps * R, Ls[b])
        if c1 > c0:
            cover.setdefault((b, k), []).append((c0, c1))
        if n[b] > 1:
            writes[(b, k, split)] = u
    # what the combine reads
    reads = {(b, k, s): (prefix[b] + s) * K + k for b in range(B) for k in range(K)
             for s in range(n[b]) if n[b] > 1}
    return cover, writes, reads, used, grid


def tiles_exactly(cover, lens, C, K):
    """The row intervals of every (sequence, tile) are disjoint and make up
    [0, L_b) exactly."""
    for b, L0 in enumerate(lens):
        L = clamp(L0, C)
        for k in range(K):
            iv = sorted(cover.get((b, k), []))
            pos = 0
            for c0, c1 in iv:
                if c0 != pos:
                    return False
                pos = c1
            if pos != L:
                return False
    return set(cover) <= {(b, k) for b in range(len(lens)) for k in range(K)}


def random_batches(seed, count):
    rnd = random.Random(seed)
    for _ in range(count):
        B = rnd.choice([1, 2, 3, 5, 8, 31, 32, 33, 40, 70])
        C = rnd.choice([1, 31, 32, 33, 100, 517, 4096, 6000])
        lens = [rnd.choice([0, 1, C, rnd.randint(0, C), C + 7, -3]) for _ in range(B)]
        K = rnd.choice([1, 2, 3, 8, 16])
        yield B, C, lens, K, rnd


def test_fixed_splits_cover_every_row_once():
    for B, C, lens, K, rnd in random_batches(1, 300):
        rps = R * rnd.randint(1, max(1, -(-C // R)))
        cover, writes, grid = fixed_cover(lens, C, K, rps)
        assert tiles_exactly(cover, lens, C, K)
        assert all(0 <= slot < grid for slot in writes.values())
        assert len(set(writes.values())) == len(writes)


def test_balanced_splits_cover_every_row_once_and_the_combine_finds_them():
    for B, C, lens, K, rnd in random_batches(2, 300):
        tiles = K * B
        nsplit = rnd.randint(1, 40)
        units = tiles * nsplit
        cover, writes, reads, used, grid = balanced_cover(lens, C, K, units)
        assert tiles_exactly(cover, lens, C, K)
        assert used <= grid == units + tiles          # the grid and workspace bound
        assert writes == reads                        # the combine reads what was written
        assert all(0 <= slot < grid for slot in writes.values())


def test_balanced_splits_even_out_ragged_lengths():
    # One long sequence among short ones (the MQA shape's spread): balanced
    # splits cut the long one into many equal splits, where fixed splits
    # would give the CTAs of the short ones almost nothing to do.
    lens = [32768] + [64] * 7
    K, units = 1, 152
    cover, writes, reads, used, grid = balanced_cover(lens, 32768, K, units)
    assert tiles_exactly(cover, lens, 32768, K)
    sizes = [c1 - c0 for iv in cover.values() for c0, c1 in iv]
    assert max(sizes) <= 32 * R          # no CTA gets more than sps stages
    assert used <= grid
    assert len(cover[(0, 0)]) > units // 2  # the long sequence takes most CTAs
