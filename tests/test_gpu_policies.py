"""Policy variants on the GPU against the fp64 oracle (same harness rules as
test_gpu_parity.py): the l2 norm, attention sinks, the deferred victim, the
layer-wide victim and the H2O cumulative score, alone and combined, on both
decode kernels -- small cases with every unit replayed, then the benchmark's
full launch shape with sampled units.

Sources: "LongFlow Guide: KV Cache Compression for Reasoning AI" -- section
"Mathematical Derivation of the LongFlow Score" (the l1 or l2 norm of the
contribution vector), section "End-to-End Implementation" (sink slots, a score
summed over all heads, the victim overwritten at the next step), section
"The Long-Output Reasoning Crisis" and the comparison table (H2O's cumulative
attention statistics).
"""
import pytest

import oracle
from test_gpu_parity import _run
from synth.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

POLICIES = {
    "l2_sinks4": oracle.Policy(norm=2, sinks=4),
    "deferred": oracle.Policy(deferred=True),
    "layer": oracle.Policy(scope="layer"),
    "h2o": oracle.Policy(score="h2o"),
    "h2o_sinks_deferred": oracle.Policy(score="h2o", sinks=2, deferred=True),
    # the guide listing's choices together: sinks 4, one slot for all heads,
    # chosen now and overwritten by the next token (window 1: the new token)
    "listing": oracle.Policy(sinks=4, deferred=True, scope="layer"),
    "h2o_layer_l2": oracle.Policy(score="h2o", scope="layer", norm=2),
}


def _small(kernel):
    if kernel == "tc":   # bf16, d = 128: several 128-slot tiles, a ragged tail, G = 4
        return WORKLOADS["r1-llama-8b"].scaled(layers=1, batch=2, q_heads=8, kv_heads=2,
                                               budget=300, window=6, prefill=280,
                                               v_lognormal_sigma=0.5), 2
    # CUDA cores: fp32, d = 32, G = 2, a chunk boundary inside the buffer
    return WORKLOADS["qwen3-0.6b"].scaled(layers=1, batch=2, q_heads=4, kv_heads=2, head_dim=32,
                                          budget=90, window=5, prefill=70, dtype="f32",
                                          v_lognormal_sigma=0.5), 2


@pytest.mark.parametrize("kernel", ["simt", "tc"])
@pytest.mark.parametrize("name", sorted(POLICIES))
def test_policy_small(kernel, name):
    pol = POLICIES[name]
    wl, cluster = _small(kernel)
    if name == "listing":
        wl = wl.scaled(window=1)
    st = _run(wl, 90, cluster=cluster, kernel=kernel, policy=pol)
    assert st.evictions > 0


@pytest.mark.parametrize("name", ["deferred", "layer", "h2o", "listing"])
def test_policy_cluster_shapes(name):
    """The tensor-core kernel with 1 and 4 CTAs per unit (different slot splits)."""
    wl, _ = _small("tc")
    if name == "listing":
        wl = wl.scaled(window=1)
    for cluster in (1, 4):
        _run(wl, 40, cluster=cluster, kernel="tc", policy=POLICIES[name])


@pytest.mark.parametrize("name", ["l2_sinks4", "deferred", "layer", "h2o", "listing"])
def test_policy_full_size(name):
    """qwen3-8b-steady's per-layer launch (batch 64, 8 KV heads, budget 3276) with
    the variant, on sampled units (layer scope: whole sampled sequences)."""
    wl = WORKLOADS["qwen3-8b-steady"]
    if name == "listing":
        wl = wl.scaled(window=1)
    st = _run(wl, 40, layers=(0,), sample=[(0, 0, 0), (0, 63, 7), (0, 40, 2)],
              policy=POLICIES[name])
    assert st.evictions > 0


def test_eviction_off_ignores_policy():
    """Full-KV mode has nothing to evict: the variants leave it unchanged."""
    wl, cluster = _small("tc")
    _run(wl, 30, cluster=cluster, kernel="tc", evict=False, capacity=512,
         policy=oracle.Policy(norm=2))


def test_h2o_full_size_long():
    """The H2O accumulators of a qwen3-8b-steady layer over 300 steps: fp32 on
    the GPU stays within 1e-4 relative of the fp64 sums, victims exact outside
    near-ties."""
    wl = WORKLOADS["qwen3-8b-steady"]
    st = _run(wl, 300, layers=(0,), sample=[(0, 5, 1), (0, 50, 6)], policy=POLICIES["h2o"])
    assert st.evictions == 2 * 300


def test_policy_ragged_deferred_sinks():
    """Per-sequence budgets 512..3276 with the deferred victim and 4 sinks."""
    from synth.workloads import InputStream
    wl = WORKLOADS["ragged-serving"]
    budgets = InputStream(wl, seed=0, device="cpu", layers=[0]).budgets
    picks = []
    for B in sorted(set(budgets)):
        b = budgets.index(B)
        picks += [(0, b, 0), (0, b, 5)]
    st = _run(wl, 150, layers=(0,), sample=picks,
              policy=oracle.Policy(deferred=True, sinks=4))
    assert st.unit_steps == 150 * len(picks)
