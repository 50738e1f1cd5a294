"""The library against the values the guide prints for its own validation run.

"LongFlow Guide: KV Cache Compression for Reasoning AI", section "Functional
Validation Benchmark": 8 heads of dimension 64, a 1000-token budget, 2500
decode steps with fresh standard-normal q, k and v (fp32), starting from an
empty buffer; the guide prints the number of finished steps and a final cache
length of 1000 (tests/golden/guide_functional_validation.json).  Run here
through lf_decode_step with the guide listing's choices (4 sinks, one victim
per step summed over all heads, overwritten by the next token) and with the
method as read here (a victim per KV head, same step).
"""
import json
import os

import pytest
import torch

from decode_kv_cache_gb300 import longflow as lf

pytestmark = pytest.mark.gpu

FIXTURE = os.path.join(os.path.dirname(__file__), "golden", "guide_functional_validation.json")


@pytest.mark.parametrize("policy", [dict(sinks=4, deferred=True, scope="layer"), dict()],
                         ids=["listing", "per_kv_head"])
def test_guide_validation_run_on_gpu(policy):
    with open(FIXTURE) as fh:
        g = json.load(fh)
    cfg, printed = g["config"], g["printed"]
    H, d, B, steps = cfg["num_heads"], cfg["head_dim"], cfg["cache_budget"], cfg["total_gen_steps"]
    gen = torch.Generator(device="cuda").manual_seed(2500)
    with lf.LFCache(1, 1, H, H, d, B, 1, dtype="f32", **policy) as cache:
        views = cache.views()
        out = torch.empty(1, H, d, device="cuda")
        ev = torch.empty(1, H, dtype=torch.int32, device="cuda")
        finished = 0
        for t in range(steps):
            q, k, v = (torch.randn(1, H, d, generator=gen, device="cuda") for _ in range(3))
            cache.decode_step(0, q, k, v, out, ev)
            finished += 1
            if t in (B - 2, B - 1, B, steps - 1):
                torch.cuda.synchronize()
                assert bool((views["count"][0, 0] == min(B, t + 1)).all())
        assert cache.check() == 0
        torch.cuda.synchronize()
        assert finished == printed["steps_finished"]
        count = views["count"][0, 0].cpu()
        assert count.tolist() == [printed["final_cache_length"]] * H
        assert views["next_pos"][0, 0].cpu().tolist() == [steps] * H
        pos = views["pos"][0, 0, :, :B].cpu()
        for h in range(H):
            live = pos[h].tolist()
            assert len(set(live)) == B and min(live) >= 0 and max(live) < steps
            if policy.get("sinks"):
                assert set(range(policy["sinks"])) <= set(live)
            assert steps - 1 in live                   # the newest token is cached
        if policy.get("scope") == "layer":
            # one victim per step for the whole layer: every head holds the same positions
            assert all(pos[h].tolist() == pos[0].tolist() for h in range(H))
