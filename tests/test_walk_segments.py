"""The decode kernel's tile walk as its producer and MMA warps now issue it,
checked against the ring order on the CPU (no GPU involved).

Both warps of decode_kv_cache_gb300/csrc/lf_decode_tc.cuh run the walk one
step per item k = 0 .. nitems (the last step only flushes) and issue each
step as up to five segments through a single issue loop:
  0  a V block still pending from two or more items back (the flush),
  1  (producer only) unit k's norms and positions,
  2  unit k's first K tiles: all of them when no V block is pending, else
     the first L (the lookahead),
  3  the pending V block of the unit before,
  4  the rest of unit k's K tiles.
The MMA warp writes unit k's query operand before it issues the step, so a
flushed V block now follows that write (it used to precede it); the query
buffer's wait looks at MMAs issued two non-empty units back, which complete
on their own, so the order of the two cannot deadlock.

The reference is the ring order the pipeline model derives from the unit list
(tests/test_pipeline_model.py): K of the first non-empty unit, then for each
next non-empty unit its first L K tiles, the V tiles of the unit before it,
and its remaining K tiles; a V block two items behind the walk is issued
alone first.  The producer's norm/position loads must come after the flush
and before the unit's own tiles.  Planted mistakes (no final flush step, the
pending V block placed after all of the unit's K tiles) must fail.
"""
import random

import pytest

from test_pipeline_model import ntiles, ring_order


def walk_segments(rows, lookahead, final_step=True, v_last=False):
    """(kind, item, tile) in the order the kernel's single issue loop emits them;
    kind "A" is the producer's norm/position load of an item (segment 1)."""
    out = []
    prev = -1
    prev_rows = 0
    nitems = len(rows)
    last = nitems if final_step else nitems - 1
    for k in range(last + 1):
        flush = prev >= 0 and (k == nitems or prev <= k - 2)
        fk, frows = prev, prev_rows
        if flush:
            prev = -1
        r = rows[k] if k < nitems else 0
        nt = ntiles(r)
        L = nt if prev < 0 else min(nt, lookahead)
        pend = prev >= 0 and r > 0
        for si in range(5):
            if si == 0:
                if flush:
                    out += [("V", fk, t) for t in range(ntiles(frows))]
            elif si == 1:
                if k < nitems:
                    out.append(("A", k, 0))
            elif si == 3:
                if pend:
                    seg = ("V", prev, ntiles(prev_rows))
                    if v_last:
                        continue
                    out += [("V", prev, t) for t in range(seg[2])]
            else:
                t0, t1 = (0, L) if si == 2 else (L, nt)
                out += [("K", k, t) for t in range(t0, t1)]
                if si == 4 and v_last and pend:
                    out += [("V", prev, t) for t in range(ntiles(prev_rows))]
        if k < nitems and r > 0:
            prev, prev_rows = k, r
    return out


def tiles_only(order):
    return [x for x in order if x[0] != "A"]


def patterns(seed, count):
    rng = random.Random(seed)
    for _ in range(count):
        n = rng.randint(1, 12)
        rows = []
        for _ in range(n):
            u = rng.random()
            rows.append(0 if u < 0.3 else rng.choice([1, 16, 127, 128, 129, 256, 300, 1000]))
        yield rows, rng.choice([0, 1, 2, 3, 8])


@pytest.mark.parametrize("seed", range(4))
def test_segments_give_the_ring_order(seed):
    for rows, L in patterns(seed, 400):
        got = tiles_only(walk_segments(rows, L))
        assert got == ring_order(rows, L, flush=True), (rows, L)


def test_norm_loads_follow_the_flush_and_precede_the_unit():
    for rows, L in patterns(7, 400):
        order = walk_segments(rows, L)
        pos = {x: i for i, x in enumerate(order)}
        prev = None
        for k, r in enumerate(rows):
            a = pos[("A", k, 0)]
            # every tile of unit k comes after its norm load
            assert all(i > a for x, i in pos.items() if x[0] == "K" and x[1] == k), (rows, k)
            # a flushed V block (two or more items back) comes before it
            if prev is not None and prev <= k - 2:
                assert all(i < a for x, i in pos.items() if x[0] == "V" and x[1] == prev), (rows, k)
                prev = None
            if r > 0:
                prev = k


def test_planted_mistakes_are_caught():
    no_final = any(tiles_only(walk_segments(rows, L, final_step=False)) !=
                   ring_order(rows, L, flush=True) for rows, L in patterns(11, 200))
    v_late = any(tiles_only(walk_segments(rows, L, v_last=True)) !=
                 ring_order(rows, L, flush=True) for rows, L in patterns(12, 200))
    assert no_final and v_late
