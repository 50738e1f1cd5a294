"""Checks that pin the fp64 oracle to things other than itself.

Each ``check_*`` takes the oracle module (or a deliberately broken copy of it,
see ``test_oracle_mutants.py``) and raises AssertionError on a violation.

The pages print no worked numeric example, so every pin here is one of:

* a library routine the method reduces to: torch's scaled_dot_product_attention
  in float64 on the CPU (textbook softmax attention, scale 1/sqrt(d)), used both
  for outputs and -- with one-hot values -- for the attention weights;
* brute force: deleting a token and recomputing attention from scratch;
* closed forms and invariants the pages fix: weights sum to one, the cache
  stays at exactly B occupied slots once full, the victim is the lowest
  alpha_i * ||v_i||_1 among the unprotected slots;
* special cases: a zero query (uniform weights, so the victim is a plain
  argmin of ||v||_1), one dominant key, a single candidate.

Citations: "LongFlow Guide: KV Cache Compression for Reasoning AI" (the guide),
"LongFlow: Efficient KV Cache Compression for Reasoning M" (the summary).
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

RNG_SEED = 1234


def sdpa(q_heads: np.ndarray, keys: np.ndarray, values: np.ndarray) -> np.ndarray:
    """torch SDPA, float64, CPU: q [H][d], keys/values [H][m][d] -> [H][dv]."""
    q = torch.from_numpy(np.array(q_heads, dtype=np.float64))[None, :, None, :]
    k = torch.from_numpy(np.array(keys, dtype=np.float64))[None]
    v = torch.from_numpy(np.array(values, dtype=np.float64))[None]
    return F.scaled_dot_product_attention(q, k, v)[0, :, 0, :].numpy()


def sdpa_weights(q_heads: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Attention weights from the library: attend to one-hot values."""
    H, m, _ = keys.shape
    eye = np.broadcast_to(np.eye(m), (H, m, m))
    return sdpa(q_heads, keys, eye)


def _unit_inputs(rng, n, d, G):
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d)) * np.exp(0.5 * rng.standard_normal((n, 1)))
    q = rng.standard_normal((G, d))
    k_new = rng.standard_normal(d)
    v_new = rng.standard_normal(d)
    return K, V, q, k_new, v_new


def _filled_unit(orc, rng, cap, d, budget, window, n, evict=True):
    u = orc.OracleUnit(cap, d, budget, window, evict)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d)) * np.exp(0.5 * rng.standard_normal((n, 1)))
    u.prefill(K, V)
    return u


# ---------------------------------------------------------------------------
# Attention (guide, "Mathematical Derivation of the LongFlow Score": alpha, o)
# ---------------------------------------------------------------------------

def check_weights_sum_to_one(orc):
    """sum_i alpha_{h,i} = 1 over the cached slots plus the new token."""
    rng = np.random.default_rng(RNG_SEED)
    for n, d, G in [(1, 4, 1), (7, 16, 2), (40, 32, 4)]:
        K, V, q, kn, vn = _unit_inputs(rng, n, d, G)
        u = orc.OracleUnit(64, d, 64, 4)
        u.prefill(K, V)
        r = u.step(q, kn, vn)
        assert r.alpha.shape == (G, n + 1), r.alpha.shape
        assert np.allclose(r.alpha.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def check_gqa_output_matches_library(orc):
    """Fill phase: a (layer, seq) step equals textbook GQA softmax attention
    (torch SDPA, fp64) over the prompt plus the new token, with query head h
    reading KV head h // G and scale 1/sqrt(d)."""
    rng = np.random.default_rng(RNG_SEED + 1)
    for hkv, G, d, P in [(1, 2, 16, 8), (2, 2, 8, 5), (2, 4, 32, 11)]:
        hq = hkv * G
        seq = orc.OracleSequence(hkv, hq, capacity=64, head_dim=d, budget=64, window=4)
        k = rng.standard_normal((hkv, P, d))
        v = rng.standard_normal((hkv, P, d))
        seq.prefill(k, v)
        keys, vals = k, v
        for _ in range(3):
            q = rng.standard_normal((hq, d))
            kn = rng.standard_normal((hkv, d))
            vn = rng.standard_normal((hkv, d))
            out, res = seq.step(q, kn, vn)
            keys = np.concatenate([keys, kn[:, None]], axis=1)
            vals = np.concatenate([vals, vn[:, None]], axis=1)
            ref = sdpa(q, np.repeat(keys, G, axis=0), np.repeat(vals, G, axis=0))
            assert np.allclose(out, ref, rtol=1e-12, atol=1e-12), np.abs(out - ref).max()
            assert all(r.evicted == -1 for r in res)


def check_deletion_identity(orc):
    """Brute force (summary, section 2.2, the denominator approximation):
    deleting token i and recomputing attention changes the output by exactly
    alpha_i / (1 - alpha_i) * (o - v_i).  Removing it while keeping the old
    denominator changes it by -alpha_i v_i, whose l1 norm is the score (G = 1)."""
    rng = np.random.default_rng(RNG_SEED + 2)
    for n, d in [(5, 8), (24, 16)]:
        K, V, q, kn, vn = _unit_inputs(rng, n, d, 1)
        u = orc.OracleUnit(n, d, n, 1)
        u.prefill(K, V)
        r = u.step(q, kn, vn)                      # n == budget: an eviction step
        keys = np.vstack([K, kn[None]])
        vals = np.vstack([V, vn[None]])
        o = r.out[0]
        for i in range(n):
            a = r.alpha[0, i]
            # a softmax over n + 1 >= 2 finite logits puts every weight strictly
            # inside (0, 1), so the identity's factor alpha / (1 - alpha) is finite
            assert 0.0 < a < 1.0, (i, a)
            keep = [j for j in range(n + 1) if j != i]
            o_del = sdpa(q, keys[keep][None], vals[keep][None])[0]
            pred = a / (1 - a) * (o - vals[i])
            assert np.allclose(o_del - o, pred, rtol=1e-10, atol=1e-12), (i, o_del - o, pred)
            # Fixed denominator: o_del * (1 - alpha_i) is the unrenormalised remainder.
            contrib = o - o_del * (1 - a)
            assert np.allclose(contrib, a * vals[i], rtol=1e-10, atol=1e-13)
            assert math.isclose(np.abs(contrib).sum(), r.scores[i], rel_tol=1e-9, abs_tol=1e-15)


def check_small_weight_change_is_first_order(orc):
    """As alpha_i -> 0 the exact deletion change divided by alpha_i tends to
    o - v_i, i.e. the change is O(alpha_i) and vanishes with the weight."""
    rng = np.random.default_rng(RNG_SEED + 3)
    d, n = 8, 6
    K, V, q, kn, vn = _unit_inputs(rng, n, d, 1)
    prev = None
    for shift in [2.0, 4.0, 6.0]:   # alpha_0 ~ 1e-3, 1e-5, 1e-7 (cancellation stays small)
        K2 = K.copy()
        K2[0] = -shift * q[0] / np.linalg.norm(q[0]) * math.sqrt(d)   # push alpha_0 down
        u = orc.OracleUnit(n, d, n, 1)
        u.prefill(K2, V)
        r = u.step(q, kn, vn)
        a = r.alpha[0, 0]
        keys = np.vstack([K2, kn[None]])
        vals = np.vstack([V, vn[None]])
        o_del = sdpa(q, keys[1:][None], vals[1:][None])[0]
        ratio = (o_del - r.out[0]) / a
        err = np.abs(ratio - (r.out[0] - vals[0])).max()
        if prev is not None:
            assert a < prev[0]
            assert err <= prev[1] + 1e-12
        prev = (a, err)
    assert prev[0] < 1e-5 and prev[1] < 1e-5


# ---------------------------------------------------------------------------
# Score and victim (guide, "Mathematical Derivation ..." and "Static Memory
# Pre-Allocation and In-Place Eviction"; summary, sections 2.1 and 2.3)
# ---------------------------------------------------------------------------

def check_victim_is_argmin_of_library_scores(orc):
    """Over a long run, every victim is the lowest sum_h alpha_{h,i} ||v_i||_1
    among slots older than the window, with alpha taken from the library (SDPA
    on one-hot values) and ||v||_1 summed directly; exact ties -> lowest slot."""
    rng = np.random.default_rng(RNG_SEED + 4)
    for G, d, B, W in [(1, 8, 12, 3), (2, 16, 16, 4), (4, 8, 10, 2)]:
        u = orc.OracleUnit(B, d, B, W)
        u.prefill(rng.standard_normal((B // 2, d)), rng.standard_normal((B // 2, d)))
        evictions = 0
        for t in range(40):
            q = rng.standard_normal((G, d))
            kn = rng.standard_normal(d)
            vn = rng.standard_normal(d) * math.exp(0.5 * rng.standard_normal())
            n_before = u.n
            K0, V0, pos0, p0 = u.K[:n_before].copy(), u.V[:n_before].copy(), u.pos[:n_before].copy(), u.p
            r = u.step(q, kn, vn)
            if n_before < B:
                assert r.evicted == -1 and r.written == n_before
                continue
            keys = np.vstack([K0, kn[None]])
            alpha = sdpa_weights(q, np.broadcast_to(keys, (G,) + keys.shape))   # [G][n+1]
            l1 = np.abs(V0).sum(axis=1)
            score = alpha[:, :n_before].sum(axis=0) * l1
            cand = np.nonzero(pos0 < p0 - W)[0]
            expect = cand[np.argmin(score[cand])]          # first minimum = lowest slot
            assert r.evicted == expect, (t, r.evicted, expect)
            assert np.allclose(r.scores, score, rtol=1e-10, atol=1e-300)
            evictions += 1
        assert evictions > 10


def check_zero_query_evicts_min_l1(orc):
    """q = 0 gives uniform weights 1/(n+1), so the victim is the candidate with
    the smallest ||v||_1 (a plain argmin)."""
    rng = np.random.default_rng(RNG_SEED + 5)
    B, W, d = 20, 5, 8
    K = rng.standard_normal((B, d))
    V = rng.standard_normal((B, d)) * np.exp(0.5 * rng.standard_normal((B, 1)))
    u = orc.OracleUnit(B, d, B, W)
    u.prefill(K, V)
    r = u.step(np.zeros((2, d)), rng.standard_normal(d), rng.standard_normal(d))
    assert np.allclose(r.alpha, 1.0 / (B + 1), rtol=0, atol=1e-15)
    l1 = np.abs(V).sum(axis=1)
    # prompt positions are 0..B-1 and the new token is at p = B, so positions
    # B-W..B-1 are protected and slots 0..B-W-1 are the candidates
    assert r.evicted == int(np.argmin(l1[:B - W]))


def check_dominant_key_survives(orc):
    """A key aligned with every query gets alpha -> 1 and is never evicted."""
    rng = np.random.default_rng(RNG_SEED + 6)
    B, W, d = 12, 2, 16
    u = _filled_unit(orc, rng, B, d, B, W, B)
    direction = rng.standard_normal(d)
    direction /= np.linalg.norm(direction)
    u.K[0] = 12.0 * math.sqrt(d) * direction
    for _ in range(30):
        q = direction[None] + 0.05 * rng.standard_normal((1, d))
        r = u.step(q, rng.standard_normal(d), rng.standard_normal(d))
        assert r.evicted != 0
        assert r.alpha[0, 0] > 0.99
    assert u.pos[0] == 0


def check_single_candidate(orc):
    """W = B - 1 leaves exactly one unprotected slot, which must go."""
    rng = np.random.default_rng(RNG_SEED + 7)
    B, d = 8, 4
    u = _filled_unit(orc, rng, B, d, B, B - 1, B)
    for t in range(12):
        oldest = int(np.argmin(u.pos[:B]))
        r = u.step(rng.standard_normal((1, d)), rng.standard_normal(d), rng.standard_normal(d))
        assert r.evicted == oldest
        assert math.isinf(r.second)


def check_exact_tie_lowest_slot(orc):
    """Identical keys and values give identical scores: the lowest slot wins."""
    rng = np.random.default_rng(RNG_SEED + 8)
    B, W, d = 6, 1, 4
    K = rng.standard_normal((B, d)) * 0.1
    V = np.ones((B, d)) * 5.0
    K[2] = K[4] = np.array([-3.0, -3.0, -3.0, -3.0])
    V[2] = V[4] = np.full(d, 0.01)
    u = orc.OracleUnit(B, d, B, W)
    u.prefill(K, V)
    r = u.step(np.ones((1, d)), np.zeros(d), np.ones(d))
    assert r.evicted == 2
    assert r.lowest == r.second


def check_cap_and_window_invariants(orc):
    """Functional validation in the spirit of the guide's "Functional Validation
    Benchmark" (2500 steps, budget 1000, d = 64, several heads): once full the
    occupied count stays at exactly B, positions stay unique, the W most recent
    positions are always cached, and every victim was older than the window."""
    rng = np.random.default_rng(RNG_SEED + 9)
    B, W, d, G, steps = 1000, 16, 64, 2, 2500
    u = orc.OracleUnit(B, d, B, W)
    u.prefill(rng.standard_normal((100, d)), rng.standard_normal((100, d)))
    q = rng.standard_normal((G, d))
    for t in range(steps):
        q = 0.9 * q + 0.44 * rng.standard_normal((G, d))
        p = u.p
        pos_before = u.pos.copy()
        r = u.step(q, rng.standard_normal(d), rng.standard_normal(d))
        assert u.n == min(B, 100 + t + 1)
        if r.evicted >= 0:
            assert pos_before[r.evicted] < p - W
        live = u.pos[:u.n]
        assert len(np.unique(live)) == u.n
        recent = set(range(max(0, u.p - W), u.p))
        assert recent <= set(live.tolist())
    assert u.n == B


def check_fill_then_evict_slots(orc):
    """Initial fill writes slots in order; the new token lands in the victim's
    slot with its position and its stored ||v||_1 (guide, steps 1 and 3)."""
    rng = np.random.default_rng(RNG_SEED + 10)
    B, W, d = 6, 1, 4
    u = orc.OracleUnit(B, d, B, W)
    u.prefill(rng.standard_normal((3, d)), rng.standard_normal((3, d)))
    assert u.n == 3 and u.p == 3 and list(u.pos[:3]) == [0, 1, 2]
    for expect_slot in [3, 4, 5]:
        kn, vn = rng.standard_normal(d), rng.standard_normal(d)
        r = u.step(rng.standard_normal((1, d)), kn, vn)
        assert r.written == expect_slot and r.evicted == -1
        assert np.array_equal(u.K[expect_slot], kn) and np.array_equal(u.V[expect_slot], vn)
    kn, vn = rng.standard_normal(d), rng.standard_normal(d)
    r = u.step(rng.standard_normal((1, d)), kn, vn)
    assert r.evicted >= 0 and r.written == r.evicted
    assert np.array_equal(u.K[r.evicted], kn) and np.array_equal(u.V[r.evicted], vn)
    assert u.pos[r.evicted] == 6
    assert u.vnorm[r.evicted] == np.abs(vn).sum()
    assert u.n == B and u.p == 7


def check_budget_below_capacity(orc):
    """A per-sequence budget below the slab's capacity (the ragged serving
    workload): the buffer fills to the budget, never further, and then every
    step evicts among the budget's slots; the slots above the budget are never
    written; a prompt longer than the budget is refused (guide, "Static Memory
    Pre-Allocation and In-Place Eviction": the fixed budget B is the buffer)."""
    rng = np.random.default_rng(RNG_SEED + 17)
    cap, d, B, W = 12, 8, 7, 2
    for deferred in (False, True):
        pol = orc.Policy(deferred=deferred)
        u = orc.OracleUnit(cap, d, B, W, True, pol)
        u.prefill(rng.standard_normal((3, d)), rng.standard_normal((3, d)))
        for t in range(30):
            r = u.step(rng.standard_normal((1, d)), rng.standard_normal(d), rng.standard_normal(d))
            assert u.n == min(B, 3 + t + 1), (deferred, t, u.n)
            assert 0 <= r.written < B
            if not deferred and 3 + t >= B:
                assert 0 <= r.evicted < B
        assert np.all(u.pos[B:] == -1) and not u.K[B:].any() and not u.V[B:].any()
        assert sorted(u.pos[:B].tolist()) == sorted(set(u.pos[:B].tolist()))
        long_prompt = B if deferred else B + 1
        v = orc.OracleUnit(cap, d, B, W, True, pol)
        try:
            v.prefill(np.zeros((long_prompt, d)), np.zeros((long_prompt, d)))
        except ValueError:
            pass
        else:
            raise AssertionError("a prompt longer than the buffer was accepted")


def check_eviction_off_full_cache(orc):
    """Eviction off: tokens append up to the capacity, then the cache is read
    only -- every step still attends over all cached slots plus the new token."""
    rng = np.random.default_rng(RNG_SEED + 11)
    cap, d = 5, 4
    u = orc.OracleUnit(cap, d, cap, 0, evict=False)
    K = rng.standard_normal((cap, d))
    V = rng.standard_normal((cap, d))
    u.prefill(K, V)
    before = u.snapshot()
    q = rng.standard_normal((1, d))
    kn, vn = rng.standard_normal(d), rng.standard_normal(d)
    r = u.step(q, kn, vn)
    assert r.evicted == -1 and r.written == -1
    ref = sdpa(q, np.vstack([K, kn[None]])[None], np.vstack([V, vn[None]])[None])
    assert np.allclose(r.out, ref, rtol=1e-12, atol=1e-13)
    after = u.snapshot()
    for a, b in zip(before[:4], after[:4]):
        assert np.array_equal(a, b)
    assert after[5] == before[5] + 1


# ---------------------------------------------------------------------------
# Policy variants (guide, "Mathematical Derivation ..." -- the l1 or l2 norm;
# "End-to-End Implementation" -- sinks, a layer-wide score, the victim written
# at the next step; "The Long-Output Reasoning Crisis" and the comparison table
# -- H2O's cumulative attention)
# ---------------------------------------------------------------------------

def _policy_run(orc, policy, rng, G, d, B, W, steps, prompt, hkv=1):
    """Drive an OracleSequence; yield (state before, q, k_new, v_new, results) per step."""
    seq = orc.OracleSequence(hkv, hkv * G, B, d, B, W, True, policy)
    seq.prefill(rng.standard_normal((hkv, prompt, d)),
                rng.standard_normal((hkv, prompt, d)) * np.exp(0.5 * rng.standard_normal((hkv, prompt, 1))))
    for _ in range(steps):
        q = rng.standard_normal((hkv * G, d))
        kn = rng.standard_normal((hkv, d))
        vn = rng.standard_normal((hkv, d)) * np.exp(0.5 * rng.standard_normal((hkv, 1)))
        before = [(u.K[:u.n].copy(), u.V[:u.n].copy(), u.pos[:u.n].copy(), u.n, u.p)
                  for u in seq.units]
        _, res = seq.step(q, kn, vn)
        yield seq, before, q, kn, vn, res


def check_l2_norm_and_sinks_against_library(orc):
    """norm = 2 and s sinks: every victim is the lowest sum_h alpha_{h,i} ||v_i||_2
    (weights from SDPA, norm from numpy) among slots with s <= pos < p - W; the
    first s positions are never evicted."""
    rng = np.random.default_rng(RNG_SEED + 12)
    for G, d, B, W, s in [(1, 8, 12, 2, 3), (2, 16, 16, 4, 4)]:
        pol = orc.Policy(norm=2, sinks=s)
        evictions = 0
        for seq, before, q, kn, vn, res in _policy_run(orc, pol, rng, G, d, B, W, 50, B - 3):
            K0, V0, pos0, n0, p0 = before[0]
            r = res[0]
            if n0 < B:
                continue
            keys = np.vstack([K0, kn[0][None]])
            alpha = sdpa_weights(q, np.broadcast_to(keys, (G,) + keys.shape))
            score = alpha[:, :n0].sum(axis=0) * np.linalg.norm(V0, axis=1)
            cand = np.nonzero((pos0 < p0 - W) & (pos0 >= s))[0]
            assert r.evicted == cand[np.argmin(score[cand])], (r.evicted, cand)
            assert np.allclose(r.scores, score, rtol=1e-10, atol=1e-300)
            assert pos0[r.evicted] >= s
            evictions += 1
        assert evictions > 20
        assert sorted(seq.units[0].pos[seq.units[0].pos < s].tolist()) == list(range(s))


def check_deferred_equals_same_step_one_slot_larger(orc):
    """Choosing the victim at step t and overwriting it at t + 1 with a buffer of
    B + 1 and a window of W + 1 (the new token counts) attends over exactly the
    tokens that same-step eviction with B slots and window W attends over, and
    drops the same tokens: outputs agree to rounding and victims by position.
    Holds for every score, norm, sink count and scope."""
    rng = np.random.default_rng(RNG_SEED + 13)
    for score, norm, sinks, scope, hkv in [("longflow", 1, 0, "kv_head", 1),
                                           ("longflow", 2, 2, "kv_head", 2),
                                           ("h2o", 1, 1, "kv_head", 1),
                                           ("longflow", 1, 1, "layer", 2),
                                           ("h2o", 1, 0, "layer", 3)]:
        G, d, B, W, P = 2, 8, 10, 2, 6
        same = orc.OracleSequence(hkv, hkv * G, B, d, B, W, True,
                                  orc.Policy(score=score, norm=norm, sinks=sinks, scope=scope))
        defer = orc.OracleSequence(hkv, hkv * G, B + 1, d, B + 1, W + 1, True,
                                   orc.Policy(score=score, norm=norm, sinks=sinks, scope=scope,
                                              deferred=True))
        k = rng.standard_normal((hkv, P, d))
        v = rng.standard_normal((hkv, P, d))
        same.prefill(k, v)
        defer.prefill(k, v)
        dropped = 0
        for t in range(40):
            q = rng.standard_normal((hkv * G, d))
            kn = rng.standard_normal((hkv, d))
            vn = rng.standard_normal((hkv, d))
            o1, r1 = same.step(q, kn, vn)
            o2, r2 = defer.step(q, kn, vn)
            assert np.allclose(o1, o2, rtol=1e-12, atol=1e-13), (score, t, np.abs(o1 - o2).max())
            for g in range(hkv):
                assert (r1[g].evicted >= 0) == (r2[g].chosen >= 0), (score, t)
            # the token same-step eviction dropped is the one deferred eviction marked
            for g in range(hkv):
                if r2[g].chosen >= 0:
                    marked = defer.units[g].pos[r2[g].chosen]
                    live = set(same.units[g].pos[:same.units[g].n].tolist())
                    live_d = set(defer.units[g].pos[:defer.units[g].n].tolist()) - {marked}
                    assert live == live_d, (score, t)
                    dropped += 1
        assert dropped > 20


def check_deferred_order(orc):
    """Deferred: the slot chosen at step t is the slot written at step t + 1
    (guide, fused kernel step 4), the new token is attended from the buffer
    (weights sum to one over n slots), never chosen in its own step, and the
    first victim is chosen by the step that fills the buffer."""
    rng = np.random.default_rng(RNG_SEED + 14)
    G, d, B, W = 2, 8, 9, 1
    pol = orc.Policy(deferred=True, sinks=2)
    prev_chosen = None
    for seq, before, q, kn, vn, res in _policy_run(orc, pol, rng, G, d, B, W, 30, 5):
        r = res[0]
        u = seq.units[0]
        n0 = before[0][3]
        assert np.allclose(r.alpha.sum(axis=1), 1.0, atol=1e-12)
        assert r.alpha.shape[1] == u.n
        if n0 < B:
            assert r.written == n0 and r.evicted == -1
        else:
            assert r.written == prev_chosen and r.evicted == prev_chosen
        if u.n == B:
            assert r.chosen >= 0 and r.chosen != r.written
            assert u.pos[r.chosen] >= 2
        else:
            assert r.chosen == -1
        prev_chosen = r.chosen


def check_layer_scope(orc):
    """One victim per sequence: (a) it is the lowest sum over every query head of
    alpha_{h,i} ||v_{kv(h),i}||_1 (weights from SDPA); (b) all KV heads keep the
    same positions; (c) with identical KV heads it equals the per-head victim."""
    rng = np.random.default_rng(RNG_SEED + 15)
    G, d, B, W, hkv = 2, 8, 12, 2, 3
    evictions = 0
    for seq, before, q, kn, vn, res in _policy_run(orc, orc.Policy(scope="layer"), rng, G, d, B,
                                                   W, 40, 8, hkv=hkv):
        n0, p0 = before[0][3], before[0][4]
        if n0 < B:
            continue
        score = np.zeros(n0)
        for g in range(hkv):
            K0, V0 = before[g][0], before[g][1]
            keys = np.vstack([K0, kn[g][None]])
            alpha = sdpa_weights(q[g * G:(g + 1) * G], np.broadcast_to(keys, (G,) + keys.shape))
            score += alpha[:, :n0].sum(axis=0) * np.abs(V0).sum(axis=1)
        cand = np.nonzero(before[0][2] < p0 - W)[0]
        expect = cand[np.argmin(score[cand])]
        assert all(r.evicted == expect for r in res), ([r.evicted for r in res], expect)
        for u in seq.units[1:]:
            assert np.array_equal(u.pos, seq.units[0].pos)
        evictions += 1
    assert evictions > 20
    # (c) identical heads: the summed score is hkv times each head's
    same = orc.OracleSequence(hkv, hkv * G, B, d, B, W, True, orc.Policy(scope="layer"))
    per = orc.OracleSequence(1, G, B, d, B, W, True)
    k = rng.standard_normal((1, B, d))
    v = rng.standard_normal((1, B, d))
    same.prefill(np.repeat(k, hkv, 0), np.repeat(v, hkv, 0))
    per.prefill(k, v)
    for _ in range(15):
        q = rng.standard_normal((G, d))
        kn = rng.standard_normal((1, d))
        vn = rng.standard_normal((1, d))
        _, r_all = same.step(np.tile(q, (hkv, 1)), np.repeat(kn, hkv, 0), np.repeat(vn, hkv, 0))
        _, r_one = per.step(q, kn, vn)
        assert r_all[0].evicted == r_one[0].evicted


def check_h2o_accumulates_library_weights(orc):
    """H2O: each slot's accumulator is the sum of the SDPA weights (over the
    group's heads) its token received at every step since it entered, its own
    entry step included, prompt tokens from zero; the victim is the lowest
    accumulator among the candidates."""
    rng = np.random.default_rng(RNG_SEED + 16)
    G, d, B, W = 2, 8, 10, 2
    mass = {}   # token position -> accumulated weight
    evictions = 0
    for seq, before, q, kn, vn, res in _policy_run(orc, orc.Policy(score="h2o"), rng, G, d, B,
                                                   W, 60, 7):
        K0, V0, pos0, n0, p0 = before[0]
        r = res[0]
        keys = np.vstack([K0, kn[0][None]])
        alpha = sdpa_weights(q, np.broadcast_to(keys, (G,) + keys.shape)).sum(axis=0)
        for i in range(n0):
            mass[int(pos0[i])] = mass.get(int(pos0[i]), 0.0) + alpha[i]
        mass[p0] = alpha[n0]
        if n0 >= B:
            cand = np.nonzero(pos0 < p0 - W)[0]
            acc = np.array([mass[int(x)] for x in pos0])
            assert r.evicted == cand[np.argmin(acc[cand])], (r.evicted, cand)
            evictions += 1
        u = seq.units[0]
        expect = np.array([mass[int(x)] for x in u.pos[:u.n]])
        assert np.allclose(u.acc[:u.n], expect, rtol=1e-12, atol=1e-15)
    assert evictions > 40


def check_h2o_zero_query_closed_form(orc):
    """H2O with q = 0 on a full prompt: weights are uniform, so a token's mass
    is proportional to the steps it has been cached.  Prompt tokens tie until a
    decode token leaves the window; from then on the victim is the decode token
    cached W + 1 steps earlier.  Exact ties go to the lowest slot, so the victim
    of eviction step t is slot t mod (W + 1)."""
    rng = np.random.default_rng(RNG_SEED + 17)
    for B, W, G in [(9, 2, 1), (12, 3, 2)]:
        u = orc.OracleUnit(B, 4, B, W, True, orc.Policy(score="h2o"))
        u.prefill(rng.standard_normal((B, 4)), rng.standard_normal((B, 4)))
        for t in range(30):
            r = u.step(np.zeros((G, 4)), rng.standard_normal(4), rng.standard_normal(4))
            assert r.evicted == t % (W + 1), (B, W, t, r.evicted)


ALL_CHECKS = [
    check_weights_sum_to_one,
    check_gqa_output_matches_library,
    check_deletion_identity,
    check_small_weight_change_is_first_order,
    check_victim_is_argmin_of_library_scores,
    check_zero_query_evicts_min_l1,
    check_dominant_key_survives,
    check_single_candidate,
    check_exact_tie_lowest_slot,
    check_cap_and_window_invariants,
    check_fill_then_evict_slots,
    check_budget_below_capacity,
    check_eviction_off_full_cache,
    check_l2_norm_and_sinks_against_library,
    check_deferred_equals_same_step_one_slot_larger,
    check_deferred_order,
    check_layer_scope,
    check_h2o_accumulates_library_weights,
    check_h2o_zero_query_closed_form,
]
