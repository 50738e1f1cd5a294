"""The tie rule on the GPU: an exact tie of the lowest score goes to the lowest
slot index, wherever the tied slots sit -- in one CTA, in different CTAs of a
cluster, or in different clusters that share a unit in a planned launch.

The rule comes from the guide ("LongFlow Guide: KV Cache Compression for
Reasoning AI"), section "Static Memory Pre-Allocation and In-Place Eviction",
step 2 (the argmin), with ties read as going to the lowest slot.  Ties are
planted: several candidate slots of every unit get the same stored key and
value, the value scaled down so that these slots hold the lowest scores, and
the query is zero, so every weight is uniform in both the fp32 kernel and the
fp64 oracle and the tied scores are bit-equal on both sides.  Each step then
evicts one tied slot, the lowest one left; the harness requires the oracle's
slot at every exact tie (no resync) and the test checks the order directly.

The H2O variant has a closed form under a zero query (the oracle pin
``check_h2o_zero_query_closed_form``): at the t-th evicting step from a full
prompt the victim is slot t mod (W + 1).  Its first W + 2 steps are exact
ties (among the prompt tokens, then between them and the first decoded token,
which has received the same mass); it is replayed here through lf_decode_step
and checked on every unit.
"""
import pytest
import torch

import oracle
from gpu_harness import ParityRun
from synth.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


def _chunk_edges(n, parts):
    """Slot ranges of `parts` equal pieces of n occupied slots (multiples of 4),
    as the kernels split a unit over a cluster."""
    per = ((n + parts - 1) // parts + 3) & ~3
    return [(r * per, min(n, (r + 1) * per)) for r in range(parts) if r * per < n]


def _tie_slots(n, parts, window, sinks=0):
    """Candidate slots on both sides of every piece boundary, plus two slots
    inside one piece, all older than the protected window (pos = slot)."""
    top = n - window - 1
    slots = {sinks + 3, sinks + 5}
    for lo, hi in _chunk_edges(n, parts):
        slots.update({lo - 1, lo, lo + 7, (lo + hi) // 2, hi - 1, hi})
    return sorted(s for s in slots if sinks <= s < top)


def _tie_run(wl, slots, steps, **kw):
    sample = kw.pop("sample", None)
    run = ParityRun(wl, layers=(0,), sample=sample, **kw)
    try:
        run.plant_tie(0, slots)
        seen = []
        for _ in range(steps):
            run.step(check=True, zero_query=True)
            seen.append(run.ev[0].clone())
        run.compare_state()
        run.check_invariants()
        st = run.stats
        print(f"\nties: {st.unit_steps} unit-steps, {st.exact_ties} exact ties, "
              f"{st.near_ties} near-ties, {st.resyncs} resyncs, "
              f"{len(st.hard_mismatches)} mismatches")
        st.assert_ok()
        assert st.resyncs == 0
        return run, seen
    except Exception:
        run.close()
        raise


@pytest.mark.parametrize("kernel,cluster", [
    ("simt", 1), ("simt", 2), ("simt", 4), ("simt", 16),
    ("tc", 1), ("tc", 2), ("tc", 4), ("tc", 16)])
def test_exact_ties_go_to_the_lowest_slot(kernel, cluster):
    """Tied slots on both sides of every CTA boundary of the cluster: each
    step evicts the lowest tied slot left, on every unit."""
    budget = 1500 if cluster == 1 else 3276
    wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, batch=2, budget=budget, prefill=budget)
    parts = max(1, cluster)
    slots = _tie_slots(budget, parts, wl.window)
    steps = len(slots) + 2
    run, seen = _tie_run(wl, slots, steps, cluster=cluster, kernel=kernel,
                         sample=[(0, 0, 0), (0, 1, 5), (0, 1, 7)])
    try:
        assert run.cache.layout.cluster == cluster
        for t, s in enumerate(slots):
            assert bool((seen[t] == s).all()), (t, s, seen[t].unique().tolist())
        # an exact tie while two or more planted slots are left, none after
        assert run.stats.exact_ties == 3 * (len(slots) - 1)
    finally:
        run.close()


def test_exact_ties_planned_launch():
    """Batch 32 at budget 3276 on two-CTA clusters takes a launch plan: three
    whole rounds, and the 28 units past them cut into 76 ranges, so each is
    shared by two to four clusters, which exchange their lowest (score, slot)
    through global memory.  Tied slots sit on both sides of the cut points of
    three shared units and of the CTA boundaries inside their parts -- inside
    one CTA, across the CTAs of a cluster, and across clusters."""
    from test_gpu_parity import _check_plan
    wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, prefill=3276)
    units = wl.batch * wl.kv_heads
    probe = ParityRun(wl, layers=(0,), sample=[(0, 0, 0)])
    try:
        plan = probe.cache.plan(0)
        C = probe.cache.layout.cluster
        nc = probe.cache.layout.split_units
    finally:
        probe.close()
    assert plan is not None
    shared = _check_plan(plan, units, nc)
    cuts = plan[1]
    chosen = sorted(shared, key=lambda u: -len(shared[u]))[:2] + [max(shared)]
    slots = {3, 5}
    for u in chosen:
        bounds = [0] + [cuts[q][1] for q in shared[u][1:]] + [wl.budget]
        for lo, hi in zip(bounds, bounds[1:]):
            per = ((hi - lo + C - 1) // C + 3) & ~3
            for x in (lo - 1, lo, lo + per - 1, lo + per):
                slots.add(x)
    top = wl.budget - wl.window - 1
    slots = sorted(x for x in slots if 0 <= x < top)
    steps = len(slots) + 2
    sample = [(0,) + divmod(u, wl.kv_heads) for u in chosen] + [(0, 0, 0), (0, 13, 6)]
    run, seen = _tie_run(wl, slots, steps, sample=sample)
    try:
        assert run.cache.plan(0) == plan
        for t, s in enumerate(slots):
            assert bool((seen[t] == s).all()), (t, s, seen[t].unique().tolist())
        assert run.stats.exact_ties == len(sample) * (len(slots) - 1)
    finally:
        run.close()


def test_exact_ties_planned_launch_deferred():
    """The same planned launch (batch 32 at budget 3276, two-CTA clusters)
    with the deferred victim: the step that fills each buffer chooses the
    lowest tied slot, and every later step overwrites the slot chosen one step
    before, across the cut points of shared units and the CTA boundaries
    inside their parts."""
    from test_gpu_parity import _check_plan
    pol = oracle.Policy(deferred=True)
    wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, prefill=3275)
    units = wl.batch * wl.kv_heads
    probe = ParityRun(wl, layers=(0,), sample=[(0, 0, 0)], policy=pol)
    try:
        plan = probe.cache.plan(0)
        C = probe.cache.layout.cluster
        nc = probe.cache.layout.split_units
    finally:
        probe.close()
    assert plan is not None
    shared = _check_plan(plan, units, nc)
    cuts = plan[1]
    chosen = sorted(shared, key=lambda u: -len(shared[u]))[:2] + [max(shared)]
    slots = {3, 5}
    for u in chosen:
        bounds = [0] + [cuts[q][1] for q in shared[u][1:]] + [wl.budget]
        for lo, hi in zip(bounds, bounds[1:]):
            per = ((hi - lo + C - 1) // C + 3) & ~3
            for x in (lo - 1, lo, lo + per - 1, lo + per):
                slots.add(x)
    top = wl.budget - wl.window - 1
    slots = sorted(x for x in slots if 0 <= x < top)
    steps = len(slots) + 2
    sample = [(0,) + divmod(u, wl.kv_heads) for u in chosen] + [(0, 0, 0), (0, 13, 6)]
    run, seen = _tie_run(wl, slots, steps, sample=sample, policy=pol)
    try:
        assert run.cache.plan(0) is not None
        for t, s in enumerate(slots):
            assert bool((seen[t + 1] == s).all()), (t, s, seen[t + 1].unique().tolist())
        assert run.stats.exact_ties >= len(slots) - 1
    finally:
        run.close()


POLICIES = {
    "deferred": oracle.Policy(deferred=True),
    "layer": oracle.Policy(scope="layer"),
    "l2_sinks4": oracle.Policy(norm=2, sinks=4),
}


@pytest.mark.parametrize("name", sorted(POLICIES))
def test_exact_ties_policies(name):
    """The deferred order (the tie decides the slot the next token takes), the
    layer-wide victim (heads' tied scores summed, the selection kernel's
    argmin) and the l2 norm with sinks, on two-CTA clusters."""
    pol = POLICIES[name]
    wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, batch=2, budget=1200, window=8,
                                         prefill=1199 if pol.deferred else 1200)
    slots = _tie_slots(wl.budget - 1, 2, wl.window, sinks=pol.sinks)
    steps = len(slots) + 2
    run, seen = _tie_run(wl, slots, steps, cluster=2, kernel="tc", policy=pol)
    try:
        if pol.deferred:
            # the first step fills the buffer and chooses; each later step
            # overwrites the slot chosen one step before
            for t, s in enumerate(slots):
                assert bool((seen[t + 1] == s).all()), (t, s, seen[t + 1].unique().tolist())
        else:
            for t, s in enumerate(slots):
                assert bool((seen[t] == s).all()), (t, s, seen[t].unique().tolist())
        assert run.stats.exact_ties >= len(slots) - 1
    finally:
        run.close()


@pytest.mark.parametrize("kernel,cluster", [("simt", 2), ("tc", 1), ("tc", 2), ("tc", 16)])
def test_h2o_zero_query_closed_form(kernel, cluster):
    """H2O from a full prompt under a zero query: the t-th evicting step
    evicts slot t mod (W + 1) on every unit (not only the sampled ones)."""
    W = 6
    wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, batch=2, q_heads=8, kv_heads=2, budget=300,
                                         window=W, prefill=300)
    run = ParityRun(wl, layers=(0,), cluster=cluster, kernel=kernel,
                    policy=oracle.Policy(score="h2o"))
    try:
        for t in range(3 * (W + 1) + 2):
            run.step(check=True, zero_query=True)
            assert bool((run.ev[0] == t % (W + 1)).all()), (t, run.ev[0].tolist())
        run.compare_state()
        run.check_invariants()
        st = run.stats
        st.assert_ok()
        # every step until the first decoded token leaves the window is an exact
        # tie (prompt tokens, then that token, all with the same mass); later
        # victims are unique minima
        assert st.resyncs == 0 and st.exact_ties == (W + 2) * wl.batch * wl.kv_heads
    finally:
        run.close()
