"""A model of the attention kernels' stream-K schedule (attn_common.cuh:
build_prefix, working_ctas, slice_begin, decode_segment and the producer's
walk over its slice), run on the CPU over random calls.

The work of a call is the flattened list of (group, item) pairs, sequence
major, where a group (sequence, kv head, row group) holds seg_items items
standing for a segment's fixed cost followed by its visible pages in items
of ppi pages (1 on the CUDA-core kernel, 8-page tiles on the tcgen05
kernel).  CTA c takes items [c T / n, (c + 1) T / n) and walks them as
segments.  The model checks what the kernels and the merge rely on:

* every visible page of every group is read by exactly one segment;
* a segment starts on an item boundary of its group (a tile boundary when
  ppi = 8), and no segment is empty;
* the owners f and l that every segment of a group records are the first
  and last CTAs holding the group's pages, and the CTAs in between hold
  pages of it too;
* a split group is the last segment of its first CTA (slot 1) and the
  first segment of every other contributor (slot 0), so no two split
  groups share a CTA's partial slot;
* the slices' item counts differ by at most one.
"""
import random

import pytest

BLOCK = 16


def visible_pages(L, q_len, n_sink, window):
    nblk = (L + BLOCK - 1) // BLOCK
    if window == 0:
        return 0, 0, nblk
    t0 = L - q_len
    lo = max(0, t0 - window + 1)
    sink_end = min(n_sink, L)
    na = (sink_end + BLOCK - 1) // BLOCK
    bs = lo // BLOCK
    if bs <= na:
        return 0, 0, nblk
    return na, bs, na + (nblk - bs)


def schedule(seq_lens, q_len, n_sink, window, groups_per_seq, n_rg, ppi,
             seg_items, grid, min_items):
    """The segments every CTA walks: (cta, b, g, rg, page0, n_pages, f, l,
    slot) in walk order, and each slice's item count."""
    prefix = [0]
    for L in seq_lens:
        np_ = visible_pages(L, q_len, n_sink, window)[2]
        prefix.append(prefix[-1] + ((np_ + ppi - 1) // ppi + seg_items) *
                      groups_per_seq)
    total = prefix[-1]
    n_ctas = max(1, min(total // max(min_items, 1), grid))

    def slice_begin(c):
        return c * total // n_ctas if c < n_ctas else total

    segs, sizes = [], []
    for cta in range(grid):
        begin = slice_begin(cta)
        end = slice_begin(cta + 1) if cta < n_ctas else total
        sizes.append(end - begin)
        pos = begin
        while pos < end:
            b = max(i for i in range(len(seq_lens)) if prefix[i] <= pos)
            per = (prefix[b + 1] - prefix[b]) // groups_per_seq
            nt = per - seg_items
            qoff = pos - prefix[b]
            gi, off = divmod(qoff, per)
            gfirst = prefix[b] + gi * per + seg_items
            t0 = 0 if off < seg_items else off - seg_items
            np_ = visible_pages(seq_lens[b], q_len, n_sink, window)[2]
            page0 = t0 * ppi
            item0 = gfirst + t0
            n_pages = min(min(end - item0, nt - t0) * ppi, np_ - page0)
            if n_pages <= 0:
                break
            f = ((gfirst + 1) * n_ctas - 1) // total
            l_ = ((gfirst + nt) * n_ctas - 1) // total
            segs.append((cta, b, gi // n_rg, gi % n_rg, page0, n_pages, f, l_,
                         1 if cta == f else 0))
            pos = item0 + (n_pages + ppi - 1) // ppi
    return segs, sizes[:n_ctas]


def random_call(rnd):
    batch = rnd.randint(1, 40)
    q_len = rnd.randint(1, 8)
    if rnd.random() < 0.3:
        n_sink, window = rnd.randint(0, 40), rnd.randint(1, 300)
    else:
        n_sink, window = 0, 0
    seq_lens = [rnd.randint(q_len, rnd.choice([40, 600, 5000])) for _ in range(batch)]
    hkv, n_rg = rnd.randint(1, 8), rnd.randint(1, 3)
    ppi, seg_items = rnd.choice([(1, 0), (1, 12), (8, 2), (8, 0)])
    grid = rnd.randint(1, 500)
    min_items = rnd.randint(1, 16)
    return (seq_lens, q_len, n_sink, window, hkv * n_rg, n_rg, ppi, seg_items,
            grid, min_items)


@pytest.mark.parametrize("seed", range(6))
def test_every_page_once_and_split_bookkeeping(seed):
    rnd = random.Random(seed)
    for _ in range(60):
        call = random_call(rnd)
        (seq_lens, q_len, n_sink, window, gps, n_rg, ppi, seg_items, grid,
         min_items) = call
        segs, sizes = schedule(*call)
        assert max(sizes) - min(sizes) <= 1, call
        seen = {}
        holders = {}
        for cta, b, g, rg, page0, n_pages, f, l_, slot in segs:
            assert n_pages > 0 and page0 % ppi == 0, call
            for k in range(page0, page0 + n_pages):
                key = (b, g, rg, k)
                assert key not in seen, (call, key)
                seen[key] = cta
            holders.setdefault((b, g, rg), []).append((cta, f, l_, slot))
        want = sum(visible_pages(L, q_len, n_sink, window)[2] * gps
                   for L in seq_lens)
        assert len(seen) == want, call
        first_seg, last_seg = {}, {}
        for i, s in enumerate(segs):
            first_seg.setdefault(s[0], i)
            last_seg[s[0]] = i
        for grp, hs in holders.items():
            ctas = [h[0] for h in hs]
            assert ctas == list(range(ctas[0], ctas[-1] + 1)), (call, grp)
            assert all(h[1] == ctas[0] and h[2] == ctas[-1] for h in hs), (call, grp)
            if len(hs) > 1:  # a split group: slots as the merge expects
                for i, s in enumerate(segs):
                    if (s[1], s[2], s[3]) != grp:
                        continue
                    if s[8] == 1:
                        assert last_seg[s[0]] == i, (call, grp)
                    else:
                        assert first_seg[s[0]] == i, (call, grp)


def test_tile_items_start_every_segment_on_a_tile():
    """ppi = 8 with slices cutting groups: every cut is a tile boundary, so
    a group split over several CTAs has one partial tile, its last."""
    call = ([4096 + 16 * 37] * 3, 5, 0, 0, 8, 1, 8, 2, 152, 1)
    segs, _ = schedule(*call)
    by_group = {}
    for s in segs:
        by_group.setdefault(s[1:4], []).append(s)
    splits = [v for v in by_group.values() if len(v) > 1]
    assert splits
    for v in splits:
        partial = [s for s in v if s[5] % 8]
        assert len(partial) <= 1 and (not partial or partial[0] is v[-1])
