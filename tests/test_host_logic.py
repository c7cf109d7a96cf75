"""CPU mirror of the device-side work partition and tile walk.

Re-derives, in Python, what mla_partition_kernel and mla_split_kernel's tile
iterator compute, and checks the invariants every launch relies on: every
token row is visited exactly once, all reads stay inside [0, kv_indptr[batch])
rows and inside the caller's scale bytes, every smem copy fits its stage, and
partial slots (range g's first segment -> slot 2g, its last -> 2g + 1) are
unique, below the workspace bound of 2 slots per CTA, and exactly the slots
the merge kernel derives for each split sequence from the tile prefix alone.
"""
import random

import pytest

TILE, PACKED, NSCALE = 128, 288, 18
FP8_TILE = 96
STAGE_SCALE_BYTES = 2432


def partition(indptr, G, kv_null=False, tile=TILE):
    """ipc (sanitised kv_indptr), tp (tiles before each sequence), T, geff, the ranges' first
    rows (and the end) and their first sequences, and the malformed-input flag."""
    B = len(indptr) - 1
    hi = 0 if kv_null else max(indptr[B], 0)
    ipc, pm, bad = [], None, False
    for i, v in enumerate(indptr):
        if v < 0 or v > hi or (i > 0 and v < indptr[i - 1]):
            bad = True
        pm = v if pm is None else max(pm, v)
        ipc.append(min(max(pm, 0), hi))
    tp = [0]
    for b in range(B):
        tp.append(tp[-1] + -(-(ipc[b + 1] - ipc[b]) // tile))
    T = tp[B]
    geff = min(G, T)
    cuts, firsts = [], []
    for g in range(geff):
        x = g * T // geff  # range g holds tiles [x_g, x_{g+1})
        b = next(b for b in range(B) if tp[b] <= x < tp[b + 1])
        cuts.append(ipc[b] + (x - tp[b]) * tile)
        firsts.append(b)
    cuts.append(ipc[B])
    return ipc, tp, T, geff, cuts, firsts, bad


def merge_slots(ipc, tp, T, geff, b):
    """Slots the merge kernel reads for sequence b (None: whole or empty sequence)."""
    if ipc[b + 1] <= ipc[b]:
        return None
    t0, t1 = tp[b], tp[b + 1]
    f, l = ((t0 + 1) * geff - 1) // T, (t1 * geff - 1) // T
    if f == l:
        return None
    shift0 = 1 if f * T // geff != t0 else 0
    return [2 * (f + i) + (shift0 if i == 0 else 0) for i in range(l - f + 1)]


def tiles(ipc, B, r0, r1, first_seq, tile=TILE):
    """The split kernel's tile walk of range [r0, r1) (TileIterT)."""
    b = first_seq
    t0 = max(r0, ipc[b])
    s1 = min(r1, ipc[b + 1])
    out, seg, first = [], 0, True
    while True:
        n = min(tile, s1 - t0)
        assert n > 0
        out.append((b, seg, t0, n, first, t0 + n >= s1))
        if t0 + n < s1:
            t0 += n
            first = False
            continue
        b += 1
        while b < B and ipc[b] == ipc[b + 1]:
            b += 1
        if b >= B or ipc[b] >= r1:
            return out
        t0, s1, seg, first = ipc[b], min(r1, ipc[b + 1]), seg + 1, True


def scale_copy_plan(t0, n, mis, scale_end):
    """The producer's plan for a tile's scale bytes, offsets from the 16-byte boundary at or
    below kv_scale (kv_scale itself at offset mis): (a0, plain byte offsets, bulk range)."""
    b0, b1 = mis + t0 * NSCALE, mis + (t0 + n) * NSCALE
    a0 = b0 & ~15
    head16 = (mis + 15) & ~15
    c0 = max(a0, head16)
    a1 = min((b1 + 15) & ~15, scale_end & ~15)
    plain = [(b0, min(b1, c0)), (max(a1, c0), b1)]  # [lo, hi) intervals, possibly empty
    plain = [(lo, hi) for lo, hi in plain if hi > lo]
    bulk = (c0, a1) if a1 > c0 else None
    return b0, b1, a0, plain, bulk


def check(indptr, G=152, kv_null=False, mis=0, tile=TILE):
    B = len(indptr) - 1
    ipc, tp, T, geff, cuts, firsts, bad = partition(indptr, G, kv_null, tile)
    rows_limit = 0 if kv_null else max(indptr[B], 0)  # caller guarantees indptr[batch] rows
    assert all(ipc[i] <= ipc[i + 1] for i in range(B))
    assert geff <= G
    seen = set()
    used_slots = set()
    slots_of = {}
    scale_end = mis + ipc[B] * NSCALE  # the buffer is [mis, mis + 18 * rows) from the boundary below it
    for g in range(geff):
        tl = tiles(ipc, B, cuts[g], cuts[g + 1], firsts[g], tile)
        # ranges are cut in whole tiles: range g walks exactly its tiles, and none holds more
        # than ceil(T / geff) of them
        assert len(tl) == (g + 1) * T // geff - g * T // geff, g
        assert len(tl) <= -(-T // geff)
        for (b, seg, t0, n, first, last) in tl:
            if first:
                seg_start = t0
            assert 0 <= ipc[b] <= t0 and t0 + n <= ipc[b + 1] <= rows_limit
            assert 1 <= n <= tile
            for r in range(t0, t0 + n):
                assert r not in seen
                seen.add(r)
            # scale bytes: 16-byte chunks inside the buffer by bulk copy, the rest by plain
            # loads; together exactly the tile's bytes, never a byte outside the buffer
            b0, b1, a0, plain, bulk = scale_copy_plan(t0, n, mis, scale_end)
            pieces = list(plain)
            if bulk:
                c0, a1 = bulk
                assert c0 % 16 == 0 and a1 % 16 == 0 and mis <= c0 < a1 <= scale_end
                pieces.append(bulk)
            assert all(mis <= lo and hi <= scale_end and hi - lo <= 16 for lo, hi in plain)
            pieces.sort()
            assert pieces[0][0] <= b0 and pieces[-1][1] >= b1  # no gap inside [b0, b1):
            assert all(pieces[i][1] >= pieces[i + 1][0] for i in range(len(pieces) - 1))
            assert all(lo - a0 >= 0 and hi - a0 <= STAGE_SCALE_BYTES for lo, hi in pieces)
            if last:
                whole = seg_start == ipc[b] and t0 + n == ipc[b + 1]
                if not whole:
                    slot = 2 * g + (1 if seg > 0 else 0)
                    assert slot not in used_slots and 0 <= slot < 2 * G
                    used_slots.add(slot)
                    slots_of.setdefault(b, []).append(slot)
    assert sorted(seen) == list(range(ipc[0], ipc[B]))
    for b in range(B):
        assert merge_slots(ipc, tp, T, geff, b) == slots_of.get(b), b
    return bad


@pytest.mark.parametrize("G", [1, 2, 152, 304])
def test_partition_covers_every_row_once(G):
    rng = random.Random(G)
    cases = [
        [0, 256], [0, 1024, 2048, 3072, 4096], [0, 0, 0], [0, 1], [0, 0, 5, 5, 6],
        [0] + [4096 * (i + 1) for i in range(128)],
        [7, 7, 300, 301, 301, 900],  # non-zero base
    ]
    for _ in range(30):
        B = rng.randint(1, 70)
        lens = [rng.choice([0, 1, 2, 127, 128, 129, rng.randint(0, 40000)]) for _ in range(B)]
        ip = [0]
        for x in lens:
            ip.append(ip[-1] + x)
        cases.append(ip)
    for i, ip in enumerate(cases):
        assert not check(ip, G, mis=(0, 1, 7, 15)[i % 4], tile=(TILE, FP8_TILE)[i % 2])


def test_ragged_workload_partition():
    import torch
    g = torch.Generator().manual_seed(4)
    lens = torch.randint(1, 32769, (64,), generator=g).tolist()
    ip = [0]
    for x in lens:
        ip.append(ip[-1] + x)
    assert not check(ip, 152)
    assert not check(ip, 152, tile=FP8_TILE)


def test_uniform_ranges_hold_whole_tiles():
    # 128 sequences of 4096 rows: 4096 tiles over 152 ranges, none cut inside a tile
    ip = [4096 * i for i in range(129)]
    ipc, tp, T, geff, cuts, firsts, bad = partition(ip, 152)
    assert T == 4096 and geff == 152
    assert all((c - ipc[b]) % TILE == 0 for c, b in zip(cuts, firsts))
    assert max((g + 1) * T // geff - g * T // geff for g in range(geff)) == 27


def test_malformed_indptr_is_clamped_and_flagged():
    for ip in ([5, 3, 10], [-4, 2, 8], [0, 10, 4, 12], [0, 50, 20]):
        assert check(ip) is True


def test_absent_kv_buffers_read_nothing():
    assert check([0, 0, 0], kv_null=True) is False
    assert check([0, 5, 9], kv_null=True) is True
