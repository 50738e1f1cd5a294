"""The host's launch planner (CPU only: lf_launch_plan_for needs no GPU).

A planned launch of the tensor-core decode kernel gives every cluster a few
whole rounds of units and one contiguous range of the units past them; a unit
cut inside a range is shared by the clusters whose ranges meet it.  The kernel
derives each cluster's items from the cut points (its parts of shared units,
then the units wholly inside its range, then its rounds) and sizes its
exchange buffers, item table and part counts from them.  Here a model of that
derivation checks, over many shapes and occupancies, the facts the kernel
relies on:

* every unit is visited exactly once, whole or as parts that tile its slots
  [0, n) in cluster order;
* cut points are on 4-slot boundaries (16-byte aligned loads of the norms and
  positions), inside [0, n), and never go backwards;
* every part's exchange row (its unit's first inner cut) is a valid row,
  below the number of clusters;
* no unit is shared by more than 16 CTAs, no cluster holds more than two
  parts, and no cluster visits more items than the item table holds.
"""
import math
import random

import pytest

from decode_kv_cache_gb300 import longflow as lf

MAX_PARTS = 16


def derive(plan, n, cluster, nc):
    """The kernel's items per cluster: [(unit, lo, hi, row, index, clusters)]
    for parts, [(unit,)] for whole units (hi None: to the occupied count)."""
    rounds, cuts = plan
    units = len(n)

    def inner(c, u):
        return 1 <= c < nc and cuts[c][0] == u and cuts[c][1] > 0

    out = []
    for j in range(nc):
        (u0, s0), (u1, s1) = cuts[j], cuts[j + 1]
        items = []
        if s0 > 0:
            jmin = jmax = j
            while inner(jmin - 1, u0):
                jmin -= 1
            while inner(jmax + 1, u0):
                jmax += 1
            items.append((u0, s0, s1 if u1 == u0 else None, jmin, j - jmin + 1, jmax - jmin + 2))
        if s1 > 0 and not (s0 > 0 and u1 == u0):
            jmax = j + 1
            while inner(jmax + 1, u1):
                jmax += 1
            items.append((u1, 0, s1, j + 1, 0, jmax - j + 1))
        w0 = u0 + 1 if s0 > 0 else u0
        items += [(w,) for w in range(w0, max(w0, u1))]
        items += [(j + k * nc,) for k in range(rounds)]
        out.append(items)
    return out


def check(plan, n, cluster, nc, max_items):
    rounds, cuts = plan
    units = len(n)
    assert len(cuts) == nc + 1 and cuts[0] == (rounds * nc, 0) and cuts[-1] == (units, 0)
    assert all(a <= b for a, b in zip(cuts, cuts[1:]))
    for u, s in cuts[1:-1]:
        assert s % 4 == 0 and (s == 0 or s < n[u])
    items = derive(plan, n, cluster, nc)
    whole, parts = [], {}
    for j, it in enumerate(items):
        assert len(it) <= max_items
        assert sum(1 for x in it if len(x) > 1) <= 2
        for x in it:
            if len(x) == 1:
                whole.append(x[0])
            else:
                u, lo, hi, row, idx, ncl = x
                assert 1 <= row < nc and 0 <= idx < ncl and ncl * cluster <= MAX_PARTS
                parts.setdefault(u, []).append((idx, lo, hi, row, ncl, j))
    assert len(whole) == len(set(whole)) and not set(whole) & set(parts)
    assert set(whole) | set(parts) == set(range(units))
    for u, ps in parts.items():
        ps.sort()
        assert [p[0] for p in ps] == list(range(len(ps))) and len(ps) == ps[0][4] >= 2
        assert len({p[3] for p in ps}) == 1                 # one exchange row per unit
        assert ps[0][1] == 0 and ps[-1][2] is None           # from slot 0 to the end
        assert all(a[2] == b[1] for a, b in zip(ps, ps[1:]))  # contiguous
        assert [p[5] for p in ps] == list(range(ps[0][5], ps[0][5] + len(ps)))
    rows = [ps[0][3] for ps in parts.values()]
    assert len(rows) == len(set(rows))                       # no two units share a row


SHAPES = [  # (batch, kv_heads, occupancy or per-sequence list, cluster, clusters)
    (64, 8, 3276, 2, 76), (32, 8, 3276, 2, 76), (12, 8, 3276, 2, 76), (4, 8, 3276, 2, 76),
    (2, 8, 3276, 2, 76), (1, 8, 3276, 2, 76), (48, 8, 3276, 2, 76), (2, 8, 3200, 4, 38),
    (24, 8, (2048, 3276, 2560), 2, 76), (256, 8, (512, 1024, 2048, 3276), 2, 76),
    (64, 8, 16384, 4, 38), (128, 8, 2048, 1, 152), (3, 3, 130, 16, 9),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"b{s[0]}x{s[1]}-c{s[3]}")
def test_plans_cover_every_unit_once(shape):
    batch, heads, occ, cluster, nc = shape
    per_seq = [occ[b % len(occ)] for b in range(batch)] if isinstance(occ, tuple) else [occ] * batch
    n = [x for x in per_seq for _ in range(heads)]
    max_items = math.ceil(len(n) / nc) + 2
    plan = lf.lf_launch_plan_for(n, cluster, nc, max_items)
    if plan is not None:
        check(plan, n, cluster, nc, max_items)


def test_plans_of_random_occupancies():
    rng = random.Random(11)
    planned = 0
    for _ in range(800):
        cluster = rng.choice([1, 2, 4])
        nc = max(1, rng.choice([152, 76, 38, 19]) // cluster)
        units = rng.randint(1, 600)
        n = [rng.choice([0, rng.randint(1, 64), rng.randint(1, 4096), 3276]) for _ in range(units)]
        max_items = math.ceil(units / nc) + 2
        plan = lf.lf_launch_plan_for(n, cluster, nc, max_items)
        if plan is not None:
            planned += 1
            check(plan, n, cluster, nc, max_items)
    assert planned > 40


def test_batch_64_and_32_take_plans():
    """The two steady shapes at budget 3276 on 76 two-CTA clusters: batch 64
    (six whole rounds, 56 units past them) and batch 32 (three rounds, 28)
    take plans in which no cluster streams much more than the average (the
    planner levels cost, so a range that meets two shared units is shorter,
    and the last ranges may come out short or empty)."""
    for batch, rounds in ((64, 6), (32, 3)):
        n = [3276] * (batch * 8)
        plan = lf.lf_launch_plan_for(n, 2, 76, math.ceil(len(n) / 76) + 2)
        assert plan is not None and plan[0] == rounds
        work = []
        for it in derive(plan, n, 2, 76):
            w = 0
            for x in it:
                w += n[x[0]] if len(x) == 1 else (x[2] if x[2] is not None else n[x[0]]) - x[1]
            work.append(w)
        assert max(work) - sum(work) / len(work) <= 3276 // 4, (max(work), min(work))
        assert max(work) < (rounds + 1) * 3276


def test_bad_arguments():
    with pytest.raises(lf.LFError):
        lf.lf_launch_plan_for([], 2, 76, 4)
    with pytest.raises(lf.LFError):
        lf.lf_launch_plan_for([100], 2, 153, 4)
    with pytest.raises(lf.LFError):
        lf.lf_launch_plan_for([-1, 5], 2, 2, 4)
