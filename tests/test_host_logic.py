"""CPU mirror of the device-side work partition and tile walk.

Re-derives, in Python, what mla_partition_kernel and mla_split_kernel's tile
iterator compute, and checks the invariants every launch relies on: every
token row is visited exactly once, all reads stay inside [0, kv_indptr[batch])
rows and inside the caller's scale bytes, every smem copy fits its stage, and
partial slots (range g's first segment -> slot 2g, its last -> 2g + 1) are
unique, below the workspace bound of 2 slots per CTA, and exactly the slots
the merge kernel derives for each split sequence from kv_indptr alone.
"""
import random

import pytest

TILE, PACKED, NSCALE, MIN_PER = 128, 288, 18, 64
STAGE_SCALE_BYTES = 2432


def partition(indptr, G, kv_null=False):
    B = len(indptr) - 1
    hi = 0 if kv_null else max(indptr[B], 0)
    ipc, pm, bad = [], None, False
    for i, v in enumerate(indptr):
        if v < 0 or v > hi or (i > 0 and v < indptr[i - 1]):
            bad = True
        pm = v if pm is None else max(pm, v)
        ipc.append(min(max(pm, 0), hi))
    N = ipc[B] - ipc[0]
    per = max(MIN_PER, -(-N // G))
    geff = -(-N // per) if N > 0 else 0
    cta_first = []
    for g in range(geff):
        r0 = ipc[0] + g * per
        cta_first.append(max(b for b in range(B) if ipc[b] <= r0))
    return ipc, per, geff, cta_first, bad


def merge_slots(ipc, per, b):
    """Slots the merge kernel reads for sequence b (None: whole or empty sequence)."""
    a0, a1, rbase = ipc[b], ipc[b + 1], ipc[0]
    if a1 <= a0:
        return None
    f, l = (a0 - rbase) // per, (a1 - 1 - rbase) // per
    if f == l:
        return None
    shift0 = 1 if a0 != rbase + f * per else 0
    return [2 * (f + i) + (shift0 if i == 0 else 0) for i in range(l - f + 1)]


def tiles(ipc, B, g, per, first_seq):
    rend = ipc[B]
    r0 = ipc[0] + g * per
    if r0 >= rend:
        return []
    r1 = min(rend, r0 + per)
    b = first_seq
    t0 = max(r0, ipc[b])
    s1 = min(r1, ipc[b + 1])
    out, seg, first = [], 0, True
    while True:
        n = min(TILE, s1 - t0)
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


def check(indptr, G=152, kv_null=False, mis=0):
    B = len(indptr) - 1
    ipc, per, geff, cta_first, bad = partition(indptr, G, kv_null)
    rows_limit = 0 if kv_null else max(indptr[B], 0)  # caller guarantees indptr[batch] rows
    assert all(ipc[i] <= ipc[i + 1] for i in range(B))
    assert geff <= G
    seen = set()
    used_slots = set()
    slots_of = {}
    scale_end = mis + ipc[B] * NSCALE  # the buffer is [mis, mis + 18 * rows) from the boundary below it
    for g in range(geff):
        tl = tiles(ipc, B, g, per, cta_first[g])
        assert tl, g
        for (b, seg, t0, n, first, last) in tl:
            if first:
                seg_start = t0
            assert 0 <= ipc[b] <= t0 and t0 + n <= ipc[b + 1] <= rows_limit
            assert 1 <= n <= TILE
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
        assert merge_slots(ipc, per, b) == slots_of.get(b), b
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
        assert not check(ip, G, mis=(0, 1, 7, 15)[i % 4])


def test_ragged_workload_partition():
    import torch
    g = torch.Generator().manual_seed(4)
    lens = torch.randint(1, 32769, (64,), generator=g).tolist()
    ip = [0]
    for x in lens:
        ip.append(ip[-1] + x)
    assert not check(ip, 152)


def test_malformed_indptr_is_clamped_and_flagged():
    for ip in ([5, 3, 10], [-4, 2, 8], [0, 10, 4, 12], [0, 50, 20]):
        assert check(ip) is True


def test_absent_kv_buffers_read_nothing():
    assert check([0, 0, 0], kv_null=True) is False
    assert check([0, 5, 9], kv_null=True) is True
