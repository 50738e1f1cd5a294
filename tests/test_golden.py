"""The oracle against the values the guide prints for its own validation run.

"LongFlow Guide: KV Cache Compression for Reasoning AI", section "Functional
Validation Benchmark": 8 heads of dimension 64, a 1000-token budget, 2500
decode steps with fresh standard-normal q, k and v, starting from an empty
buffer.  The guide prints the number of finished steps and a final cache length
of 1000, which it says can never exceed the budget.  The fixture in
tests/golden/guide_functional_validation.json holds those printed values.

The run uses the guide listing's own choices (section "End-to-End
Implementation"): 4 sink slots, one victim per step chosen from the sum over
all heads, overwritten by the next token (deferred, window 1: only the newest
token is protected), and also the method as read here (a victim per KV head,
decided in the same step).
"""
import json
import os

import numpy as np
import pytest

import oracle

FIXTURE = os.path.join(os.path.dirname(__file__), "golden", "guide_functional_validation.json")


def _golden():
    with open(FIXTURE) as fh:
        return json.load(fh)


@pytest.mark.parametrize("policy,window", [
    (oracle.Policy(sinks=4, deferred=True, scope="layer"), 1),
    (oracle.Policy(), 1),
], ids=["listing", "per_kv_head"])
def test_guide_validation_run(policy, window):
    g = _golden()
    cfg, printed = g["config"], g["printed"]
    H, d, B, steps = cfg["num_heads"], cfg["head_dim"], cfg["cache_budget"], cfg["total_gen_steps"]
    if policy.sinks:
        assert policy.sinks == cfg["sink_size"]
    rng = np.random.default_rng(2500)
    seq = oracle.OracleSequence(H, H, B, d, B, window, True, policy)
    finished = 0
    for t in range(steps):
        q = rng.standard_normal((H, d))
        _, res = seq.step(q, rng.standard_normal((H, d)), rng.standard_normal((H, d)))
        finished += 1
        for u, r in zip(seq.units, res):
            assert u.n == min(B, t + 1)          # fills one slot per step, then stays capped
            live = u.pos[:u.n]
            assert len(np.unique(live)) == u.n   # no slot holds two tokens, none is lost
            if policy.sinks and t >= policy.sinks:
                assert set(range(policy.sinks)) <= set(live.tolist())
        if policy.scope == "layer" and t >= B:
            # one victim per step, the same slot in every head
            assert len({r.evicted for r in res}) == 1
    assert finished == printed["steps_finished"]
    for u in seq.units:
        assert u.n == printed["final_cache_length"]
        assert u.p == steps
