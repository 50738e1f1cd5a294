"""The R-KV compression's pass-2 buffer schedule, modelled on the CPU.

Pass 2 takes the row blocks in pairs (I0 = 2p, I1 = 2p + 1) and streams every
column tile J > I1 once through a ring of shared-memory stages for both row
blocks; the pair's last two tiles (I1 + 2, then I1 + 1) are kept as the next
pair's row blocks, and the old row-block buffers take their places in the ring.
Three roles track the buffers on their own:

* the producer swaps a stage with a row-block buffer when it loads a kept tile
  (its next load into that stage waits for the stage to be handed back);
* the MMA warps swap when the pair is done with its old row blocks;
* the epilogue hands a stage back after the tile's second block, and the stage
  of the next pair's row block 1 only after the pair's last block.

This model replays the three sequences and checks that every MMA operand read
finds the tile it needs in its buffer at that point, with every load gated by
the hand-back it waits for, and that the blocks cover each pair of row blocks
(J >= I) exactly once.  A planted mistake (handing the kept stage back at its
own second block) must fail the check.
"""
import pytest


def pair_tiles(i1, nb):
    return nb - i1 - 1 if i1 < nb else 0


def pair_kept(m):
    return m if m < 2 else 2


def pair_tile(i1, k, m):
    if k < m - pair_kept(m):
        return i1 + 3 + k
    return i1 + 1 if k == m - 1 else i1 + 2


def blocks(nb):
    """(row block, column block) in the order the MMA warps issue them."""
    out, p = [], 0
    while 2 * p < nb:
        i0, i1 = 2 * p, 2 * p + 1
        out.append((i0, i0))
        if i1 < nb:
            out += [(i0, i1), (i1, i1)]
        m = pair_tiles(i1, nb)
        for k in range(m):
            j = pair_tile(i1, k, m)
            out += [(i0, j), (i1, j)]
        p += 1
    return out


def replay(nb, stages=3, defer_kept=True):
    # producer: ring loads (pass 1 tiles, then each pair's column tiles), with swaps
    seq = [(t, -1) for t in range(nb)]
    p = 0
    while 2 * p + 1 < nb:
        i1 = 2 * p + 1
        m = pair_tiles(i1, nb)
        for k in range(m):
            keep = 0 if k == m - 1 else (1 if pair_kept(m) == 2 and k == m - 2 else -1)
            seq.append((pair_tile(i1, k, m), keep))
        p += 1
    stage, a = ["S%d" % i for i in range(stages)], ["A0", "A1"]
    loads = []
    for tt, (t, keep) in enumerate(seq):
        st = tt % stages
        loads.append((tt, st, stage[st], t))
        if keep >= 0:
            stage[st], a[keep] = a[keep], stage[st]
    # MMA reads and epilogue hand-backs, in block order
    stage, a = ["S%d" % i for i in range(stages)], ["A0", "A1"]
    ev, rt = [], 0
    for t in range(nb):   # pass 1: the epilogue reads the tile, then hands it back
        st = rt % stages
        ev += [("read", stage[st], t), ("back", st)]
        rt += 1
    p = 0
    while 2 * p < nb:
        i0, i1 = 2 * p, 2 * p + 1
        has1 = i1 < nb
        m = pair_tiles(i1, nb)
        ev.append(("read", a[0], i0))                 # importance of I0
        if has1:
            ev.append(("read", a[1], i1))             # importance of I1
        ev.append(("read", a[0], i0))                 # (I0, I0)
        if has1:
            ev += [("read", a[0], i0), ("read", a[1], i1), ("read", a[1], i1)]
        kept_st, held = [-1, -1], -1
        for k in range(m):
            j, st = pair_tile(i1, k, m), rt % stages
            keep1 = pair_kept(m) == 2 and k == m - 2
            ev += [("read", a[0], i0), ("read", stage[st], j),
                   ("read", a[1], i1), ("read", stage[st], j)]
            if not (keep1 and defer_kept):
                ev.append(("back", st))
            if k == m - 1 and held >= 0:
                ev.append(("back", held))
            if keep1:
                held = st
            keep = 0 if k == m - 1 else (1 if keep1 else -1)
            if keep >= 0:
                kept_st[keep] = st
            rt += 1
        if kept_st[1] >= 0:
            stage[kept_st[1]], a[1] = a[1], stage[kept_st[1]]
        if kept_st[0] >= 0:
            stage[kept_st[0]], a[0] = a[0], stage[kept_st[0]]
        p += 1
    # a load into a stage may happen once that stage's previous tile was handed back
    back_at, count = {}, [0] * stages
    for i, e in enumerate(ev):
        if e[0] == "back":
            back_at[(e[1], count[e[1]])] = i
            count[e[1]] += 1
    contents = {"A0": [(-1, 0)], "A1": [(-1, 1)] if nb > 1 else []}
    for tt, st, buf, tile in loads:
        gate = back_at.get((st, tt // stages - 1)) if tt >= stages else -1
        if gate is None:
            return False
        contents.setdefault(buf, []).append((gate, tile))
    for buf in contents:
        contents[buf].sort()
    for i, e in enumerate(ev):
        if e[0] != "read":
            continue
        landed = [c for c in contents.get(e[1], []) if c[0] < i]
        if not landed or landed[-1][1] != e[2]:
            return False
    return True


@pytest.mark.parametrize("stages", [3, 4])
def test_every_read_finds_its_tile(stages):
    for nb in range(1, 33):
        assert replay(nb, stages), nb


def test_blocks_cover_each_pair_once():
    for nb in range(1, 40):
        got = sorted(blocks(nb))
        assert got == [(i, j) for i in range(nb) for j in range(i, nb)], nb


def test_early_hand_back_of_the_kept_tile_is_caught():
    assert not all(replay(nb, 3, defer_kept=False) for nb in range(1, 33))
