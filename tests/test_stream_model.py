"""A CPU model of the streamed tensor-core schedule and its combine (no GPU).

The streamed kernel (gqa_av_stream.cuh): sequence b has
n_b = max(1, ceil(L_b / R)) stages in each of its K tiles; tile column k
lists tile k of every sequence, sequence after sequence, T = sum_b n_b stages.
The grid is U = K * Ug CTAs; CTA u takes column k = u % K and, with
Ug' = min(Ug, T), stages [floor(T g / Ug'), floor(T (g + 1) / Ug')) of it,
g = u / K (at least one each; none for g >= Ug'). Every run of one tile's
stages inside a CTA (a segment) is written to `out` when it covers the whole
tile, else to workspace slot 2u (the CTA's first segment) or 2u + 1 (its
last). The combine finds, for each tile (b, k), the groups g0..g1 whose
ranges hold its first and last stage and sums slots 2 (g K + k) in group
order, except that g0's slot is 2 (g0 K + k) + 1 when the tile does not start
g0's range.

This model restates those integer rules the way the device code computes
them (the warp scan that finds a CTA's first stage, the cursor that walks
the stages, the segment ends, the combine's owner formula) and checks over
many random calls that:
- every (sequence, tile, stage) is streamed exactly once;
- every tile is either written whole by exactly one CTA, or has its partial
  slots written exactly once each and the combine reads exactly those slots,
  in CTA order;
- slot indices stay inside [0, 2U) and the cursor never reads a length past
  the batch.
"""
import random


def stages_of(L, R):
    return max(1, -(-L // R))


M32 = (1 << 32) - 1


def first_stage(T, g, Ug):
    """floor(T g / Ug), as the producer warp computes it: in unsigned 32-bit
    arithmetic with T = q Ug + r0 when T < 2^31 and Ug < 2^15, else in 64-bit."""
    if T < (1 << 31) and Ug < (1 << 15):
        q = (T & M32) // Ug
        r0 = (T - q * Ug) & M32
        return ((q * g) & M32) + ((r0 * g) & M32) // Ug & M32
    return T * g // Ug


def stream_range(lens, R, g, Ug):
    """(count, b, j) of group g in a column, as the producer warp finds them."""
    T = sum(stages_of(L, R) for L in lens)
    Ug = min(Ug, T)
    if g >= Ug:
        return 0, 0, 0
    s0, s1 = first_stage(T, g, Ug), first_stage(T, g + 1, Ug)
    count = s1 - s0
    assert count >= 1
    base = 0
    for b, L in enumerate(lens):  # the warp scan, one sequence at a time
        n = stages_of(L, R)
        if base <= s0 < base + n:
            return count, b, s0 - base
        base += n
    raise AssertionError("s0 past the stage list")


def walk(lens, R, K, u, U):
    """The stages CTA u streams, and what its accumulators write at each
    segment end: ('out', b, k) or ('slot', slot, b, k)."""
    B = len(lens)
    k, g = u % K, u // K
    count, b, j = stream_range(lens, R, g, U // K)
    n = stages_of(lens[b], R) if count else 1
    streamed, writes = [], []
    first_segment, seg_j0 = True, j
    for it in range(count):
        assert 0 <= b < B, "cursor past the batch while streaming"
        streamed.append((b, k, j))
        tile_end = j == n - 1
        if tile_end or it == count - 1:
            if seg_j0 == 0 and tile_end:
                writes.append(("out", b, k))
            else:
                writes.append(("slot", 2 * u + (0 if first_segment else 1), b, k))
            first_segment, seg_j0 = False, 0
        # stream_advance
        j += 1
        if j >= n:
            j = 0
            b += 1
            n = stages_of(lens[b], R) if b < B else 1
    return streamed, writes


def combine_slots(lens, R, K, U, b, k):
    """The slots the combine sums for tile (b, k), in order (empty: whole)."""
    T = sum(stages_of(L, R) for L in lens)
    pre = sum(stages_of(L, R) for L in lens[:b])
    nb = stages_of(lens[b], R)
    Ug = min(U // K, T)
    owner = lambda x: ((x + 1) * Ug - 1) // T
    g0, g1 = owner(pre), owner(pre + nb - 1)
    if g0 == g1:
        return []
    first = T * g0 // Ug
    slots = [2 * (g0 * K + k) + (0 if first == pre else 1)]
    slots += [2 * (g * K + k) for g in range(g0 + 1, g1 + 1)]
    return slots


def grid_of(K, want):
    """The planner's grid: K CTAs a group, as many groups as fit `want`."""
    return K * max(1, want // K)


def check(lens, R, K, want):
    U = grid_of(K, want)
    B = len(lens)
    streamed, out_writes, slot_writes = {}, {}, {}
    for u in range(U):
        st, wr = walk(lens, R, K, u, U)
        for key in st:
            streamed[key] = streamed.get(key, 0) + 1
        for w in wr:
            if w[0] == "out":
                out_writes[(w[1], w[2])] = out_writes.get((w[1], w[2]), 0) + 1
            else:
                slot, tb, tk = w[1], w[2], w[3]
                assert 0 <= slot < 2 * U
                assert slot not in slot_writes, "slot written twice"
                slot_writes[slot] = (tb, tk)
    for b in range(B):
        for k in range(K):
            for j in range(stages_of(lens[b], R)):
                assert streamed.get((b, k, j), 0) == 1, (b, k, j)
            slots = combine_slots(lens, R, K, U, b, k)
            if not slots:
                assert out_writes.get((b, k), 0) == 1, ("whole tile not written", b, k)
                assert all(v != (b, k) for v in slot_writes.values())
            else:
                assert (b, k) not in out_writes
                assert len(set(slots)) == len(slots)
                written = sorted(s for s, v in slot_writes.items() if v == (b, k))
                assert written == sorted(slots), ("combine reads other slots", b, k, slots, written)
                # CTA order: the slots' CTAs increase.
                assert [x // 2 for x in slots] == sorted(x // 2 for x in slots)
    assert sum(streamed.values()) == K * sum(stages_of(L, R) for L in lens)


def test_stream_schedule_random_calls():
    rng = random.Random(7)
    for _ in range(600):
        B = rng.choice([1, 2, 3, 5, 8, 31, 32, 33, 64, 70])
        C = rng.choice([1, 16, 64, 100, 512, 4096, 32768])
        R = rng.choice([16, 32, 48, 64, 128])
        K = rng.choice([1, 2, 3, 8, 16, 64])
        U = rng.choice([1, 2, 7, 152, 304, 456])
        kind = rng.random()
        if kind < 0.2:
            lens = [C] * B
        elif kind < 0.3:
            lens = [0] * B
        else:
            lens = [rng.randint(0, C) for _ in range(B)]
        check(lens, R, K, U)


def test_stream_schedule_workload_shapes():
    rng = random.Random(3)
    # The decode workloads' shapes: (B, C, K) with K = head groups x column tiles.
    for B, C, K, lo in ((1, 512, 2, 512), (1, 8192, 8, 8192), (4, 16384, 8, 8192),
                        (8, 32768, 2, 1), (32, 131072, 8, 32768)):
        lens = [rng.randint(lo, C) for _ in range(B)]
        for U in (152, 304, 456):
            check(lens, 64, K, U)


def test_more_ctas_than_stages():
    # Fewer stages than CTAs: most CTAs have none; each stage still once.
    check([5, 0, 17], 16, 1, 152)
    check([0], 64, 1, 304)


def test_first_stage_32bit_path():
    # The 32-bit path is floor(T g / Ug) exactly, with nothing wrapping, up to
    # its bounds (T < 2^31, Ug < 2^15, g <= Ug); the 64-bit path takes the rest.
    rng = random.Random(11)
    cases = [((1 << 31) - 1, (1 << 15) - 1), ((1 << 31) - 1, 1), (1, 1), (12345, 304)]
    for _ in range(20000):
        Ug = rng.choice([1, 2, 3, 7, 19, 38, 152, 304, 4096, (1 << 15) - 1, rng.randint(1, (1 << 15) - 1)])
        T = rng.choice([Ug, Ug + 1, rng.randint(Ug, (1 << 31) - 1), (1 << 31) - 1 - rng.randint(0, 99)])
        cases.append((max(T, Ug), Ug))
    for T, Ug in cases:
        for g in {0, 1, Ug // 2, Ug - 1, Ug, rng.randint(0, Ug)}:
            q, r0 = T // Ug, T % Ug
            assert q * g < (1 << 32) and r0 * g < (1 << 30) + (1 << 15)
            assert first_stage(T, g, Ug) == T * g // Ug, (T, g, Ug)
    assert first_stage(1 << 40, 5, 7) == (1 << 40) * 5 // 7
