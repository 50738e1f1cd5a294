"""CUDA path vs the fp64 oracle, element by element on the same seeded inputs.

Small cases run every unit through the oracle.  The large workloads run one or
two layers at their full per-layer size (batch, heads, budget, window: the
launch configuration the benchmark times) and replay a sample of units.
"""
import os

import numpy as np
import pytest
import torch

from gpu_harness import ParityRun
from synth.workloads import WORKLOADS, InputStream

pytestmark = pytest.mark.gpu


def _run(wl, steps, **kw):
    run = ParityRun(wl, **kw)
    try:
        run.run(steps)
        run.compare_state()
        run.check_invariants()
        st = run.stats
        # one line per case (shown with pytest -s): the parity counts of the run
        case = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        print(f"\nparity {case}: {st.unit_steps} unit-steps, {st.evictions} evictions, "
              f"{st.near_ties} near-ties, {st.resyncs} resyncs, "
              f"{len(st.hard_mismatches)} mismatches, max output error "
              f"{st.max_out_violation:.3f} of tolerance")
        st.assert_ok()
        return st
    finally:
        run.close()


@pytest.mark.parametrize("cluster", [0, 2, 4])
def test_tiny_fp32_full_workload(cluster):
    """The tiny fp32 workload end to end (8-token prompt, 64 steps: 24 fill, 40 evict)."""
    st = _run(WORKLOADS["tiny-fp32"], 64, cluster=cluster)
    assert st.evictions == 40


def test_qwen3_06b_shape_two_layers():
    wl = WORKLOADS["qwen3-0.6b"]
    sample = [(li, b, g) for li in range(2) for b in (0, 3, 7) for g in (0, 5)]
    st = _run(wl, 600, layers=(0, 13), sample=sample)
    assert st.evictions > 0


def test_r1_llama_shape_fill_phase():
    """Prompt 512 of budget 3276: the first steps of the fill phase at full size."""
    wl = WORKLOADS["r1-llama-8b"]
    _run(wl, 40, layers=(5,), sample=[(0, 0, 0), (0, 31, 7), (0, 17, 3)])


def test_r1_llama_shape_eviction_phase():
    """Same launch shape with the prompt near the budget, so steps evict."""
    wl = WORKLOADS["r1-llama-8b"].scaled(prefill=3240)
    st = _run(wl, 160, layers=(2,), sample=[(0, 0, 0), (0, 13, 6), (0, 31, 7)])
    assert st.evictions >= 3 * 120


def test_r1_llama_full_generation():
    """The R1-Llama-8B-shaped workload end to end on one layer at full batch:
    prompt 512, then all 16384 decode steps (2764 fill steps up to the 3276-slot
    budget, then 13620 evicting steps), two sampled units replayed throughout."""
    wl = WORKLOADS["r1-llama-8b"]
    st = _run(wl, 16384, layers=(7,), sample=[(0, 0, 0), (0, 31, 7)])
    assert st.evictions == 2 * (16384 - (3276 - 512))


def test_qwen3_06b_full_generation():
    """The Qwen3-0.6B-shaped workload end to end on one layer: prompt 256, all
    4096 decode steps (256 fill, then evictions at budget 512)."""
    wl = WORKLOADS["qwen3-0.6b"]
    st = _run(wl, 4096, layers=(20,), sample=[(0, 2, 1), (0, 7, 6)])
    assert st.evictions == 2 * (4096 - (512 - 256))


def test_qwen3_8b_steady_state():
    wl = WORKLOADS["qwen3-8b-steady"]
    st = _run(wl, 120, layers=(0,), sample=[(0, 0, 0), (0, 63, 7), (0, 40, 2)])
    assert st.evictions == 3 * 120


def test_qwen3_8b_steady_long_run():
    """600 steps of the benchmark's layer launch (every step evicts): no drift
    between the fp32 GPU path and the fp64 oracle over many evictions."""
    wl = WORKLOADS["qwen3-8b-steady"]
    st = _run(wl, 600, layers=(0,), sample=[(0, 1, 3), (0, 62, 0)])
    assert st.evictions == 2 * 600


def test_full_kv_read_only():
    """Eviction off at the full 16384-token capacity: every step attends over
    all slots plus the new token and writes nothing."""
    wl = WORKLOADS["qwen3-8b-steady"].scaled(prefill=16384, batch=16)
    st = _run(wl, 12, layers=(0,), sample=[(0, 0, 0), (0, 15, 7)], evict=False, capacity=16384)
    assert st.evictions == 0


def test_ragged_serving_shape():
    """Mixed budgets and prompts at full batch, 1100 steps.  A sequence whose
    prompt is longer than its budget prefills the budget and feeds the rest of
    its prompt as decode steps, each with the query drawn for that step, while
    the batch advances in lock-step.  The sampled sequences include, per budget
    value, the first one drawn, and sequences whose prompt remainder ends after
    30, 109 and 996 steps or outlasts the run, so the run crosses the end of
    the prompt remainder and the first abrupt query reset (every 1000 steps)."""
    wl = WORKLOADS["ragged-serving"]
    ins = InputStream(wl, seed=0, device="cpu", layers=[0])  # the same seeded draw
    budgets, prompts = ins.budgets, ins.prompt_lens
    picks = []
    seqs = [budgets.index(B) for B in sorted(set(budgets))]
    extra = {b: P - B for b, (P, B) in enumerate(zip(prompts, budgets)) if P > B}
    remainders = sorted(extra.values())
    for want in (30, 109, 996):   # a remainder of about this length
        seqs.append(min(extra, key=lambda b: abs(extra[b] - want)))
    seqs.append(max(extra, key=extra.get))
    for b in dict.fromkeys(seqs):
        picks += [(0, b, 0), (0, b, 7)]
    run = ParityRun(wl, layers=(0,), sample=picks)
    try:
        fed = run.overflow[0]
        assert sum(0 < fed[b] < 1100 for b in seqs) >= 3 and max(fed) > 1100
        assert fed == [max(0, P - B) for P, B in zip(prompts, budgets)]
        assert remainders and min(remainders) > 0
        run.run(1100)
        run.compare_state()
        run.check_invariants()
        st = run.stats
        print(f"\nparity ragged: {st.unit_steps} unit-steps, {st.evictions} evictions, "
              f"{st.near_ties} near-ties, {st.resyncs} resyncs, "
              f"{len(st.hard_mismatches)} mismatches, max output error "
              f"{st.max_out_violation:.3f} of tolerance")
        st.assert_ok()
        assert st.unit_steps == 1100 * len(picks)
    finally:
        run.close()


@pytest.mark.parametrize("case", [
    # name, overrides, capacity, cluster
    ("g1_d64_empty_start_ragged_tail", dict(q_heads=4, kv_heads=4, head_dim=64, budget=37,
                                            window=3, prefill=0, batch=3), None, 4),
    ("g8_d32_f32_single_candidate", dict(q_heads=8, kv_heads=1, head_dim=32, budget=100,
                                         window=99, prefill=100, batch=2, dtype="f32"), None, 0),
    ("g4_d128_sparse_cluster16", dict(q_heads=8, kv_heads=2, head_dim=128, budget=130,
                                      window=5, prefill=120, batch=2), None, 16),
    ("g2_d16_window0", dict(q_heads=4, kv_heads=2, head_dim=16, budget=64, window=0,
                            prefill=64, batch=2), None, 2),
    ("g4_d128_f32", dict(q_heads=8, kv_heads=2, head_dim=128, budget=200, window=8,
                         prefill=150, batch=2, dtype="f32"), None, 0),
], ids=lambda c: c[0])
def test_edge_cases(case):
    name, over, cap, cluster = case
    wl = WORKLOADS["qwen3-0.6b"].scaled(layers=1, steps=80, v_lognormal_sigma=0.5, **over)
    _run(wl, 80, cluster=cluster, capacity=cap)


@pytest.mark.parametrize("kernel,cluster,stages", [
    ("simt", 1, 4), ("simt", 2, 2), ("simt", 4, 8), ("simt", 8, 3), ("simt", 16, 16),
    ("tc", 1, 2), ("tc", 2, 2), ("tc", 4, 3), ("tc", 8, 4), ("tc", 16, 3)])
def test_launch_shapes_agree(kernel, cluster, stages):
    """Both kernels, every cluster size and ring depth give the oracle's results."""
    # cluster 1 keeps every slot of a unit in one CTA: use a budget that fits
    budget = 1500 if cluster == 1 else 3276
    wl = WORKLOADS["r1-llama-8b"].scaled(batch=2, budget=budget, prefill=budget - 76)
    _run(wl, 100, cluster=cluster, stages=stages, kernel=kernel, sample=[(0, 0, 0), (0, 1, 5)])


@pytest.mark.parametrize("case", [
    # name, overrides, cluster: tensor-core kernel (bf16, d = 128) edge cases
    ("g1_empty_start", dict(q_heads=3, kv_heads=3, budget=37, window=3, prefill=0, batch=2), 4),
    ("g2_multi_tile_ragged", dict(q_heads=4, kv_heads=2, budget=300, window=6, prefill=290,
                                  batch=2), 1),
    ("g8_single_candidate", dict(q_heads=8, kv_heads=1, budget=140, window=139, prefill=140,
                                 batch=2), 2),
    ("g4_sparse_cluster16", dict(q_heads=8, kv_heads=2, budget=130, window=5, prefill=120,
                                 batch=2), 16),
    ("g4_tail_of_one", dict(q_heads=8, kv_heads=2, budget=129, window=2, prefill=129,
                            batch=2), 1),
], ids=lambda c: c[0])
def test_tensor_core_edge_cases(case):
    name, over, cluster = case
    wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, v_lognormal_sigma=0.5, **over)
    _run(wl, 60, cluster=cluster, kernel="tc")


def test_simt_kernel_full_size_eviction():
    """The CUDA-core kernel at the full r1-llama-8b launch shape."""
    wl = WORKLOADS["r1-llama-8b"].scaled(prefill=3240)
    st = _run(wl, 80, layers=(1,), kernel="simt", sample=[(0, 4, 1), (0, 30, 6)])
    assert st.evictions >= 2 * 40


def test_nonfinite_query_sets_error_word():
    from decode_kv_cache_gb300.longflow import LF_DEVERR_NONFINITE, LFCache
    wl = WORKLOADS["tiny-fp32"]
    c = LFCache(1, 1, 1, 2, 16, 32, 4, dtype="f32")
    k = torch.randn(1, 1, 8, 16, device="cuda")
    c.prefill(0, k, k.clone(), [8])
    q = torch.randn(1, 2, 16, device="cuda")
    kn = torch.randn(1, 1, 16, device="cuda")
    c.decode_step(0, q, kn, kn.clone())
    assert c.check() == 0
    q[0, 1, 3] = float("nan")
    c.decode_step(0, q, kn, kn.clone())
    assert c.check() & LF_DEVERR_NONFINITE
    assert c.check() == 0  # cleared by the read
    c.close()


@pytest.mark.parametrize("kernel,budget,cluster", [
    ("simt", 1, 0), ("simt", 2, 2), ("tc", 1, 0), ("tc", 2, 2), ("tc", 3, 16)])
def test_degenerate_budgets(kernel, budget, cluster):
    """Budgets of 1-3 slots with window 0, batch 1: every step past the prompt
    evicts one of a handful of candidates (budget 1: the only cached slot), and
    most CTAs of a cluster own no slot at all."""
    if kernel == "tc":
        wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, batch=1, q_heads=8, kv_heads=2,
                                              budget=budget, window=0, prefill=1,
                                              v_lognormal_sigma=0.5)
    else:
        wl = WORKLOADS["tiny-fp32"].scaled(budget=budget, window=0, prefill=1)
    st = _run(wl, 40, cluster=cluster, kernel=kernel)
    assert st.evictions == 40 * wl.kv_heads - (budget - 1) * wl.kv_heads


def _plan_items(plan, units, nc):
    """The items of every cluster of a launch plan (lf_launch_plan), in the
    kernel's order: its parts of shared units (of the unit its range starts
    inside, then of the unit it ends inside), the units wholly inside its
    range, then its whole rounds.  Each item is (unit, shared)."""
    rounds, cuts = plan
    items = []
    for j in range(nc):
        (u0, s0), (u1, s1) = cuts[j], cuts[j + 1]
        it = []
        if s0 > 0:
            it.append((u0, True))
        if s1 > 0 and not (s0 > 0 and u1 == u0):
            it.append((u1, True))
        it += [(w, False) for w in range(u0 + 1 if s0 > 0 else u0, u1)]
        it += [(j + k * nc, False) for k in range(rounds)]
        items.append(it)
    return items


def _check_plan(plan, units, nc):
    """A launch plan covers the layer once: whole rounds round-robin, then
    contiguous ranges over the units past them, with cut points on 4-slot
    boundaries.  Returns, per shared unit, the clusters holding its parts."""
    rounds, cuts = plan
    first = rounds * nc
    assert len(cuts) == nc + 1 and cuts[0] == (first, 0) and cuts[-1] == (units, 0)
    assert all(a <= b for a, b in zip(cuts, cuts[1:]))           # cuts never go back
    assert all(s % 4 == 0 for _, s in cuts)
    items = _plan_items(plan, units, nc)
    whole = sorted(u for it in items for u, sh in it if not sh)
    shared = {}
    for j, it in enumerate(items):
        for u, sh in it:
            if sh:
                shared.setdefault(u, []).append(j)
    assert len(whole) == len(set(whole)) and not set(whole) & set(shared)
    assert set(whole) | set(shared) == set(range(units))          # every unit, once
    assert all(len(js) >= 2 and js == list(range(js[0], js[-1] + 1)) for js in shared.values())
    return shared


def test_planned_launch_choice():
    """A layer whose sequences all hold >= 2048 tokens takes a launch plan when
    the host's cost model prefers it to whole units: batches 64, 32 and 4 at
    budget 3276 on two-CTA clusters do (units shared by two clusters, and by
    three or more).  The plan covers every unit once.  An empty layer never
    takes one; the deferred order, the H2O score and the layer scope do."""
    from decode_kv_cache_gb300.longflow import LFCache
    clusters = torch.cuda.get_device_properties(0).multi_processor_count // 2
    for batch in (32, 4):
        cache = LFCache(2, batch, 8, 32, 128, 3276, 64, cluster=2)
        try:
            lay = cache.layout
            assert lay.cluster == 2 and lay.split_units == clusters
            assert cache.plan(0) is None                          # empty
            k = torch.zeros(batch, 8, 3276, 128, dtype=torch.bfloat16, device="cuda")
            cache.prefill(0, k, k, [3276] * batch)
            plan = cache.plan(0)
            assert plan is not None and cache.plan(1) is None
            shared = _check_plan(plan, batch * 8, clusters)
            widest = max(len(p) for p in shared.values())
            assert widest >= 3, widest
        finally:
            cache.close()
    # 64 sequences: 512 units on 76 clusters, six whole rounds and the 56
    # units past them cut into 76 ranges
    cache = LFCache(1, 64, 8, 32, 128, 3276, 64)
    try:
        k = torch.zeros(64, 8, 3276, 128, dtype=torch.bfloat16, device="cuda")
        cache.prefill(0, k, k, [3276] * 64)
        plan = cache.plan(0)
        assert plan is not None and plan[0] == 6
        _check_plan(plan, 512, clusters)
    finally:
        cache.close()
    for kw, prompt in ((dict(deferred=True), 3275), (dict(score="h2o"), 3276),
                       (dict(scope="layer"), 3276)):
        cache = LFCache(1, 32, 8, 32, 128, 3276, 64, **kw)
        try:
            k = torch.zeros(32, 8, 3276, 128, dtype=torch.bfloat16, device="cuda")
            cache.prefill(0, k, k, [prompt] * 32)    # deferred: at most budget - 1
            assert cache.layout.split_units == clusters
            plan = cache.plan(0)
            assert plan is not None
            _check_plan(plan, 256, clusters)
        finally:
            cache.close()


def test_planned_launch_transition_with_policy():
    """r1-llama-8b's launch shape (256 units): a prompt of 2038, so the first
    10 steps run whole units and the rest take a plan, here with the l2 norm
    and 4 sinks; sampled units among the shared ones and whole ones."""
    import oracle
    wl = WORKLOADS["r1-llama-8b"].scaled(prefill=2038)
    run = ParityRun(wl, layers=(1,), sample=[(0, 31, 7), (0, 29, 0), (0, 2, 3), (0, 13, 4)],
                    policy=oracle.Policy(norm=2, sinks=4))
    try:
        for t in range(60):
            assert (run.cache.plan(0) is None) == (t < 10), t
            run.step()
        run.compare_state()
        run.check_invariants()
        run.stats.assert_ok()
        assert run.stats.unit_steps == 60 * 4
    finally:
        run.close()


@pytest.mark.parametrize("batch,budgets", [(4, None), (24, (2048, 3276, 2560))])
def test_planned_launch_parity(batch, budgets):
    """Planned launches at full head geometry: batch 4 (32 units on 76 clusters,
    so every unit is shared by three or more clusters, up to 16 CTAs) and a
    ragged batch of budgets 2048 / 3276 / 2560, all full, every step evicts.
    Every unit is replayed by the oracle."""
    wl = WORKLOADS["r1-llama-8b"].scaled(batch=batch, prefill=3276)
    bud = [budgets[b % len(budgets)] for b in range(batch)] if budgets else None
    run = ParityRun(wl, layers=(0,), budgets=bud, cluster=2)
    try:
        plan = run.cache.plan(0)
        assert plan is not None
        shared = _check_plan(plan, batch * 8, len(plan[1]) - 1)
        assert max(len(p) for p in shared.values()) >= 3
        run.run(40)
        run.compare_state()
        run.check_invariants()
        st = run.stats
        print(f"\nparity planned b{batch}: {st.unit_steps} unit-steps, {st.evictions} evictions, "
              f"{st.near_ties} near-ties, {st.resyncs} resyncs, {len(st.hard_mismatches)} "
              f"mismatches, max output error {st.max_out_violation:.3f} of tolerance")
        st.assert_ok()
        assert st.evictions == 40 * batch * 8
    finally:
        run.close()


def test_split_exchange_timeout_recovers():
    """A planned launch whose exchange through global memory can never
    complete: the waits give up after their bound, the shared unit skips the
    step (state, count and position unchanged, evicted = -1),
    LF_DEVERR_TIMEOUT is reported, lf_cache_check zeroes the counters, and the
    context stays usable.  The failure is made on the host: the first
    exchange's arrival count of one shared unit is set so low that the arrivals
    never reach the target.  Batch 12 at budget 3276 on 2-CTA clusters takes a
    plan (one whole round of 76 units, the other 20 cut into 76 ranges, so
    every one of them is shared by three to five clusters).  A CTA whose wait
    ran out skips the rest of its launch, so the items after the shared unit
    in its cluster's list skip the step too; every other unit matches the
    oracle."""
    import time
    from decode_kv_cache_gb300.longflow import LF_DEVERR_TIMEOUT
    wl = WORKLOADS["r1-llama-8b"].scaled(layers=1, batch=12, prefill=3276)
    units = wl.batch * wl.kv_heads
    probe = ParityRun(wl, layers=(0,), sample=[(0, 0, 0)], cluster=2)
    try:
        plan = probe.cache.plan(0)
        nc = probe.cache.layout.split_units
    finally:
        probe.close()
    assert plan is not None
    shared = _check_plan(plan, units, nc)
    items = _plan_items(plan, units, nc)
    bad_unit = min(shared)                     # the first shared unit
    xi = shared[bad_unit][1]                   # its exchange row: its first inner cut
    skipped_units = {bad_unit}
    for j in shared[bad_unit]:                 # the clusters holding its parts skip
        it = [u for u, _ in items[j]]          # every item after it
        skipped_units.update(it[it.index(bad_unit):])
    skipped = [divmod(u, wl.kv_heads) for u in sorted(skipped_units)]
    sample = [(0, b, g) for b in range(wl.batch) for g in range(wl.kv_heads)
              if (b, g) not in skipped]
    run = ParityRun(wl, layers=(0,), sample=sample, cluster=2)
    try:
        assert run.cache.layout.cluster == 2 and run.cache.plan(0) == plan
        run.run(3)
        assert run.cache.check() == 0
        vw = run.views
        cnt = vw["split_cnt"]
        assert int(cnt.abs().sum()) == 0
        names = ("k", "v", "vnorm", "pos", "count", "next_pos")
        before = {(bg, n): vw[n][0][bg].clone() for bg in skipped for n in names}
        cnt[xi, 0] = -(1 << 20)
        torch.cuda.synchronize()
        t0 = time.monotonic()
        run.step(check=True)  # every sampled unit against the oracle as usual
        bits = run.cache.check()
        elapsed = time.monotonic() - t0
        assert bits == LF_DEVERR_TIMEOUT, bits
        assert elapsed < 30.0
        assert int(cnt.abs().sum()) == 0
        for (bg, n), t in before.items():
            assert torch.equal(vw[n][0][bg], t), (bg, n)
        for bg in skipped:
            assert int(run.ev[0][bg]) == -1
        run.run(4)
        assert run.cache.check() == 0
        run.compare_state()
        run.stats.assert_ok()
    finally:
        run.close()
