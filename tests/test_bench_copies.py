"""The end-to-end step's host-to-device copies (bench.in_range_copies, CPU):
for [B, Cmax, ...] tensors exactly rows c < L_b of each sequence are copied,
each piece contiguous and at most 1 GiB, other tensors whole."""
import os
import sys
from types import SimpleNamespace

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_in_range_copies_cover_exactly_the_rows_read():
    w = SimpleNamespace(B=3, Cmax=10)
    lens = [10, 0, 4]
    v = torch.arange(3 * 10 * 2 * 4, dtype=torch.float32).reshape(3, 10, 2, 4)
    attn = torch.arange(3 * 10 * 6, dtype=torch.float32).reshape(3, 10, 6) + 1000
    sl = torch.tensor(lens, dtype=torch.int32)
    dv, da, ds = torch.full_like(v, -1), torch.full_like(attn, -1), torch.full_like(sl, -1)
    chunks = bench.in_range_copies([(dv, v), (da, attn), (ds, sl)], w, lens)
    for d, h in chunks:
        assert d.is_contiguous() and h.is_contiguous() and d.numel() == h.numel()
        d.copy_(h)
    for b, L in enumerate(lens):
        assert torch.equal(dv[b, :L], v[b, :L]) and torch.all(dv[b, L:] == -1)
        assert torch.equal(da[b, :L], attn[b, :L]) and torch.all(da[b, L:] == -1)
    assert torch.equal(ds, sl)
    copied = sum(h.numel() * h.element_size() for _, h in chunks)
    assert copied == sum(lens) * (2 * 4 + 6) * 4 + 3 * 4
    # Everything whole when no lengths are given (a paged cache).
    whole = bench.in_range_copies([(dv, v)], w, None)
    assert len(whole) == 1 and whole[0][1].numel() == v.numel()
