"""Checks that pin the R-KV oracle to things other than itself (CPU only).

Each ``check_*`` takes the oracle module (or a deliberately broken copy, see
``test_rkv_oracle.py``) and raises AssertionError on a violation.  The README
("GitHub - Zefan-Cai/R-KV", section "Method") prints no worked example, so
the pins are library routines (torch SDPA weights, pairwise cosines written
as loops), closed forms and invariants.
"""
from __future__ import annotations

import math

import numpy as np

from oracle_pins import sdpa, sdpa_weights

SEED = 4321


def _params(orc, budget, **kw):
    return orc.RKVParams(budget=budget, **kw)


def check_importance_is_mean_library_weight(orc):
    """I_i = mean over the observation queries of their SDPA weight on i."""
    rng = np.random.default_rng(SEED)
    for Q, n, d in [(1, 5, 4), (8, 40, 16), (32, 200, 32)]:
        q = rng.standard_normal((Q, d))
        k = rng.standard_normal((n, d))
        got = orc.importance(q, k, 1.0 / math.sqrt(d))
        w = sdpa_weights(q, np.broadcast_to(k, (Q, n, d)))     # [Q][n]
        assert np.allclose(got, w.mean(axis=0), rtol=1e-12, atol=1e-15)
        assert math.isclose(got.sum(), 1.0, rel_tol=1e-12)


def check_redundancy_pairwise(orc):
    """R_i from explicit pair loops: count later tokens with cosine >= tau."""
    rng = np.random.default_rng(SEED + 1)
    for n, d, tau, beta in [(12, 8, 0.9, 1), (30, 16, 0.8, 2), (25, 4, 0.5, 3)]:
        k = rng.standard_normal((n, d))
        # plant near-duplicates of a few earlier keys
        for i in rng.choice(n, size=n // 3, replace=False):
            src = rng.integers(0, n)
            k[i] = k[src] + 0.05 * rng.standard_normal(d)
        pos = rng.permutation(n) * 3
        got = orc.redundancy(k, pos, tau, beta)
        for i in range(n):
            cnt = 0
            for j in range(n):
                if pos[j] > pos[i]:
                    c = float(np.dot(k[i], k[j]) / (np.linalg.norm(k[i]) * np.linalg.norm(k[j])))
                    cnt += c >= tau
            assert got[i] == (1.0 if cnt >= beta else 0.0), (i, cnt, got[i])


def check_identical_keys_keep_the_newest(orc):
    """All keys equal: every token but the beta latest is redundant."""
    n, d = 10, 8
    k = np.ones((n, d))
    pos = np.arange(n)[::-1].copy()      # slot 0 is the latest
    for beta in (1, 2, 4):
        r = orc.redundancy(k, pos, 0.99, beta)
        newest = set(np.argsort(-pos)[:beta].tolist())
        for i in range(n):
            assert r[i] == (0.0 if i in newest else 1.0)


def check_selection_threshold_and_observation_tokens(orc):
    """The alpha latest positions always stay; every token kept on score has z
    at least that of every dropped token; equal z goes to the later token."""
    rng = np.random.default_rng(SEED + 2)
    for n, B, alpha in [(20, 12, 3), (100, 64, 8)]:
        z = rng.standard_normal(n).round(1)      # rounding makes ties
        pos = rng.permutation(n)
        keep = orc.select_keep(z, pos, B, alpha)
        assert len(keep) == B and len(set(keep.tolist())) == B
        latest = set(np.argsort(-pos)[:alpha].tolist())
        assert latest <= set(keep.tolist())
        scored = [i for i in keep if i not in latest]
        dropped = [i for i in range(n) if i not in set(keep.tolist())]
        for i in scored:
            for j in dropped:
                assert z[i] > z[j] or (z[i] == z[j] and pos[i] > pos[j])


def check_zero_query_no_redundancy_is_a_sliding_window(orc):
    """q = 0: uniform importance; distinct random keys: no redundancy.  All z
    tie, so the kept set is the `budget` latest tokens, and every compression
    keeps exactly positions p - budget .. p - 1."""
    rng = np.random.default_rng(SEED + 3)
    d, G = 16, 2
    prm = orc.RKVParams(budget=24, buffer=8, alpha=4)
    u = orc.RKVUnit(d, prm)
    u.prefill(rng.standard_normal((20, d)), rng.standard_normal((20, d)))
    compressions = 0
    for t in range(60):
        if u.n == u.capacity:
            r = u.compress(np.zeros((prm.alpha, G, d)))
            assert r is not None and np.allclose(r.imp, 1.0 / len(r.imp))
            assert r.red.sum() == 0
            compressions += 1
            assert sorted(u.pos[:u.n].tolist()) == list(range(u.p - prm.budget, u.p))
        u.step(np.zeros((G, d)), rng.standard_normal(d), rng.standard_normal(d))
    assert compressions >= 4


def check_decode_step_is_library_attention(orc):
    """Decode steps attend over every staged and retained token plus the new one."""
    rng = np.random.default_rng(SEED + 4)
    d, G = 8, 2
    u = orc.RKVUnit(d, orc.RKVParams(budget=10, buffer=4, alpha=2))
    K = rng.standard_normal((6, d))
    V = rng.standard_normal((6, d))
    u.prefill(K, V)
    keys, vals = K, V
    for _ in range(8):
        q = rng.standard_normal((G, d))
        kn, vn = rng.standard_normal(d), rng.standard_normal(d)
        out = u.step(q, kn, vn)
        keys = np.vstack([keys, kn[None]])
        vals = np.vstack([vals, vn[None]])
        ref = sdpa(q, np.broadcast_to(keys, (G,) + keys.shape), np.broadcast_to(vals, (G,) + vals.shape))
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)


def check_compression_layout(orc):
    """After a compression: budget slots full; retained tokens that stay keep
    their slots; the kept buffer tokens fill the freed slots in slot order; the
    kept set is the oracle's own threshold choice on library scores."""
    rng = np.random.default_rng(SEED + 5)
    d, G = 16, 4
    prm = orc.RKVParams(budget=40, buffer=16, alpha=8, tau=0.7)
    u = orc.RKVUnit(d, prm)
    k = rng.standard_normal((prm.budget, d))
    k[5] = k[30] + 0.01 * rng.standard_normal(d)       # slot 5 older near-duplicate of 30
    u.prefill(k, rng.standard_normal((prm.budget, d)))
    qs = []
    for _ in range(prm.buffer):
        q = rng.standard_normal((G, d))
        qs.append(q)
        u.step(q, rng.standard_normal(d), rng.standard_normal(d))
    before = (u.K.copy(), u.V.copy(), u.pos.copy())
    r = u.compress(np.array(qs[-prm.alpha:]))
    assert u.n == prm.budget
    # library scores
    n = prm.budget + prm.buffer
    qo = np.array(qs[-prm.alpha:]).reshape(-1, d)
    w = sdpa_weights(qo, np.broadcast_to(before[0][:n], (len(qo), n, d))).mean(axis=0)
    assert np.allclose(r.imp, w, rtol=1e-12)
    assert r.red[5] == 1.0
    kept = set(r.keep.tolist())
    for s in range(prm.budget):
        if s in kept:
            assert u.pos[s] == before[2][s] and np.array_equal(u.K[s], before[0][s])
    movers = [s for s in range(prm.budget, n) if s in kept]
    freed = [s for s in range(prm.budget) if s not in kept]
    assert r.moves == list(zip(movers, freed))
    for src, dst in r.moves:
        assert np.array_equal(u.K[dst], before[0][src]) and u.pos[dst] == before[2][src]
    assert sorted(u.pos[:u.n].tolist()) == sorted(before[2][sorted(kept)].tolist())


def check_long_run_invariants(orc):
    """Steps with a compression whenever the buffer fills: occupancy stays in
    [budget, budget + buffer], positions unique, the alpha latest kept."""
    rng = np.random.default_rng(SEED + 6)
    d, G = 8, 2
    prm = orc.RKVParams(budget=32, buffer=8, alpha=4, tau=0.6)
    u = orc.RKVUnit(d, prm)
    u.prefill(rng.standard_normal((32, d)), rng.standard_normal((32, d)))
    qs = [rng.standard_normal((G, d)) for _ in range(prm.alpha)]
    for t in range(200):
        if u.n == u.capacity:
            u.compress(np.array(qs[-prm.alpha:]))
            latest = set(range(u.p - prm.alpha, u.p))
            assert latest <= set(u.pos[:u.n].tolist())
        q = rng.standard_normal((G, d))
        qs.append(q)
        kn = rng.standard_normal(d) if rng.random() > 0.3 else u.K[rng.integers(0, u.n)] * 1.01
        u.step(q, kn, rng.standard_normal(d))
        assert prm.budget <= u.n <= u.capacity
        live = u.pos[:u.n]
        assert len(np.unique(live)) == u.n


def check_redundant_goes_before_important(orc):
    """lambda = 0.1: a redundant token scores at most 0.1 - 0.9 < 0 and every
    other token at least 0, so an older near-duplicate is dropped first even
    when the observation queries attend to it most."""
    rng = np.random.default_rng(SEED + 7)
    d, n = 16, 12
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    k = 0.3 * rng.standard_normal((n, d))
    k[0] = 4.0 * math.sqrt(d) * u                     # oldest, dominant attention
    k[5] = k[0] + 0.01 * rng.standard_normal(d)       # its newer near-duplicate
    pos = np.arange(n)
    q = np.tile(u, (8, 1))
    imp = orc.importance(q, k, 1.0 / math.sqrt(d))
    red = orc.redundancy(k, pos, 0.9, 1)
    assert red[0] == 1.0 and red[5] == 0.0 and imp[0] > 0.3
    prm = orc.RKVParams(budget=n - 1, buffer=4, alpha=2)
    unit = orc.RKVUnit(d, prm)
    unit.prefill(k, rng.standard_normal((n, d)))
    r = unit.compress(q.reshape(8, 1, d))
    assert 0 not in set(r.keep.tolist()) and 5 in set(r.keep.tolist())
    assert r.z[0] < 0 <= min(r.z[i] for i in range(1, n))


ALL_CHECKS = [
    check_importance_is_mean_library_weight,
    check_redundancy_pairwise,
    check_identical_keys_keep_the_newest,
    check_selection_threshold_and_observation_tokens,
    check_zero_query_no_redundancy_is_a_sliding_window,
    check_decode_step_is_library_attention,
    check_compression_layout,
    check_long_run_invariants,
    check_redundant_goes_before_important,
]
