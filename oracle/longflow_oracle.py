"""Plain, slow fp64 CPU oracle for the LongFlow fused decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this module.  The
product path (the C-ABI library and its Python binding) never does, and this
module imports nothing from it: the two share no kernels, headers, helpers,
tables or constants.

What it computes, one cache unit at a time (one layer, one sequence, one KV
head with its group of G query heads), in float64 on the exact stored values:

* attention weights and output of a single query over the cached tokens plus
  the new token -- "LongFlow Guide: KV Cache Compression for Reasoning AI"
  (aifetchly blog), section "Mathematical Derivation of the LongFlow Score",
  the equations for alpha_{t,i} and o_t;
* the LongFlow importance score alpha_i * ||v_i||_1 -- same section, the
  contribution vector c_{t,i} = alpha_{t,i} v_i and its l1 norm; the same
  formula, printed cleanly, is in "LongFlow: Efficient KV Cache Compression for
  Reasoning M" (gist.science summary), section 2.1 "Zero-Cost Estimation";
* the static buffer: initial fill, then argmin eviction with an in-place
  overwrite -- guide, section "Static Memory Pre-Allocation and In-Place
  Eviction", steps 1-3; summary, section 2.3 "Static KV Cache".

Readings where the pages are silent or ambiguous:

* GQA: query head h reads KV head floor(h / G); each KV head keeps its own
  slots and evicts its own victim, scored by the sum over its G query heads.
* The new token attends to itself: the softmax runs over the n cached slots
  plus the new token (the guide's reference step also writes the token before
  attending).  Eviction is decided in the same step, among the cached slots,
  and the new token is written into the victim's slot.
* The W most recent cached positions (pos >= p - W, p = the new token's
  position) are never evicted; exact score ties go to the lowest slot index.
* Softmax scale 1/sqrt(d).  The cached ||v||_1 is taken from the stored value.

Policy variants (``Policy``), each a plain reading of a passage:

* ``norm=2``: the score uses ||v_i||_2 -- the guide lets the importance be
  either the l1 or the l2 norm of c_{t,i} ("Mathematical Derivation ...").
* ``sinks=s``: positions 0..s-1 are never evicted -- the guide's reference step
  ("End-to-End Implementation") protects its first sink_size slots.
* ``deferred=True``: the order of the guide's reference step and of its fused
  kernel's step 4, whose output is the slot that the following step
  overwrites: the new token is first written into the slot chosen at the
  previous step (or the next free slot while filling), the query attends over
  the buffer, and the lowest-score slot outside the window becomes the slot
  the next token overwrites.  The window then counts the new token: slots with
  pos >= p + 1 - W are protected (W >= 1 keeps the new token itself).
* ``scope="layer"``: one victim per (layer, sequence), shared by all KV heads,
  scored by the sum over every query head -- the guide's reference step sums
  |c| over heads and feature dimensions.
* ``score="h2o"``: cumulative attention mass -- the comparison the guide draws
  with H2O, which scores tokens by the attention they have accumulated
  (section "The Long-Output Reasoning Crisis" and H2O's row of the comparison
  table).
  Each slot keeps the sum of the attention weights its token has received
  (over the group's query heads) at every decode step since it entered the
  buffer, its own entry step included; a prompt token starts at zero.  The
  victim is the lowest such sum among the candidates.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

__all__ = ["attention", "value_norm", "longflow_scores", "choose_victim", "Policy",
           "OracleUnit", "StepResult", "OracleSequence"]


def attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float):
    """Single-query softmax attention for G query heads sharing one KV head.

    q [G][d], keys/values [m][d] -> (alpha [G][m], out [G][d]).
    alpha_{h,i} = exp(s_{h,i}) / sum_j exp(s_{h,j}) with s_{h,i} = scale * q_h . k_i
    and out_h = sum_i alpha_{h,i} v_i  (guide, "Mathematical Derivation of the
    LongFlow Score", the alpha_{t,i} and o_t equations).  The row maximum is
    subtracted before exp only to avoid overflow; it cancels in the ratio.
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    logits = (q @ keys.T) * scale                      # [G][m]
    shifted = logits - logits.max(axis=1, keepdims=True)
    w = np.exp(shifted)
    alpha = w / w.sum(axis=1, keepdims=True)
    out = alpha @ values                               # [G][d]
    return alpha, out


def value_norm(v: np.ndarray, norm: int = 1) -> float:
    """||v||_1 (default) or ||v||_2 of one stored value vector."""
    v = np.asarray(v, np.float64)
    if norm == 1:
        return float(np.abs(v).sum())
    if norm == 2:
        return float(math.sqrt((v * v).sum()))
    raise ValueError("norm must be 1 or 2")


def longflow_scores(alpha_cached: np.ndarray, vnorm1: np.ndarray) -> np.ndarray:
    """LongFlow score of every cached slot of one KV head.

    score_i = sum_{h in group} ||c_{h,i}||_1 = sum_h alpha_{h,i} * ||v_i||_1
    (guide, "Mathematical Derivation of the LongFlow Score", the Score_LongFlow
    equation; summary, section 2.1, LongFlowScore(t_i) = alpha_i^t ||v_i||_1),
    summed over the group's query heads (GQA reading).
    alpha_cached [G][n], vnorm1 [n] -> [n].
    """
    return np.asarray(alpha_cached, np.float64).sum(axis=0) * np.asarray(vnorm1, np.float64)


def choose_victim(scores: np.ndarray, pos: np.ndarray, next_pos: int, window: int,
                  sinks: int = 0):
    """Lowest-score slot among the candidates (guide, "Static Memory
    Pre-Allocation and In-Place Eviction", step 2).

    Candidates are slots whose position is older than the protected window,
    pos_i < next_pos - window, and not one of the first `sinks` positions.
    They are sorted by score with a stable sort, so equal scores stay in slot
    order and an exact tie goes to the lowest slot.
    Returns (victim slot, lowest score, second-lowest score or inf).
    """
    scores = np.asarray(scores, np.float64)
    pos = np.asarray(pos)
    cand = np.flatnonzero((pos < next_pos - window) & (pos >= sinks))
    if cand.size == 0:
        raise ValueError("no eviction candidate: window and sinks cover every cached slot")
    order = cand[np.argsort(scores[cand], kind="stable")]
    best = int(order[0])
    second = float(scores[order[1]]) if order.size > 1 else math.inf
    return best, float(scores[best]), second


@dataclass(frozen=True)
class Policy:
    """How a cache scores and evicts (the defaults are the method as read here)."""
    score: str = "longflow"   # "longflow": alpha * ||v||; "h2o": cumulative attention
    norm: int = 1             # norm of v in the LongFlow score: 1 or 2
    sinks: int = 0            # positions < sinks are never evicted
    deferred: bool = False    # pick now, overwrite with the next token
    scope: str = "kv_head"    # "kv_head": a victim per KV head; "layer": one per sequence

    def validate(self):
        if self.score not in ("longflow", "h2o"):
            raise ValueError("score must be 'longflow' or 'h2o'")
        if self.norm not in (1, 2):
            raise ValueError("norm must be 1 or 2")
        if self.sinks < 0:
            raise ValueError("sinks must be >= 0")
        if self.scope not in ("kv_head", "layer"):
            raise ValueError("scope must be 'kv_head' or 'layer'")


@dataclass
class StepResult:
    out: np.ndarray          # [G][d] attention output of the group's query heads
    evicted: int             # slot whose token left the buffer this step, or -1
    written: int             # slot the new token went to, or -1 (read-only full cache)
    alpha: np.ndarray        # [G][m] weights (same step: n cached then the new token;
                             #         deferred: the buffer's n slots, new token included)
    scores: Optional[np.ndarray]  # [n] the scores a victim was chosen from this step
    lowest: float            # lowest candidate score (nan when nothing was chosen)
    second: float            # second-lowest candidate score (nan when nothing was chosen)
    chosen: int = -1         # victim chosen this step (same step: == evicted;
                             # deferred: the slot the next token overwrites)

    @property
    def rel_gap(self) -> float:
        """(second - lowest) / second: how far the chosen victim is from a tie."""
        if not (self.chosen >= 0) or not math.isfinite(self.second) or self.second <= 0:
            return math.inf if self.chosen >= 0 else math.nan
        return (self.second - self.lowest) / self.second


class OracleUnit:
    """One cache unit: a KV head's static slot buffer for one layer and sequence.

    State (summary, section 2.3 "Static KV Cache"; guide, "Static Memory
    Pre-Allocation and In-Place Eviction"): K/V [capacity][d], the cached
    ||v|| per slot, the token position per slot, the occupied count n and the
    next token position p; with the H2O score, the accumulated attention per
    slot; when deferred, the slot the next token overwrites.  Nothing is ever
    moved or compacted.
    """

    def __init__(self, capacity: int, head_dim: int, budget: int, window: int,
                 evict: bool = True, policy: Optional[Policy] = None):
        policy = policy or Policy()
        policy.validate()
        if not (0 < budget <= capacity):
            raise ValueError("need 0 < budget <= capacity")
        if evict:
            if not (0 <= window and window + policy.sinks < budget):
                raise ValueError("need 0 <= window and window + sinks < budget")
            if policy.deferred and window < 1:
                raise ValueError("deferred eviction needs window >= 1")
        self.capacity, self.d, self.budget, self.window = capacity, head_dim, budget, window
        self.evict = evict
        self.policy = policy
        self.K = np.zeros((capacity, head_dim))
        self.V = np.zeros((capacity, head_dim))
        self.vnorm = np.zeros(capacity)
        self.pos = np.full(capacity, -1, dtype=np.int64)
        self.acc = np.zeros(capacity)   # H2O: attention received so far
        self.pending = -1               # deferred: slot the next token overwrites
        self.n = 0
        self.p = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def limit(self) -> int:
        return self.budget if self.evict else self.capacity

    def _write(self, slot: int, k, v, position: int):
        # In-place overwrite of one slot (guide, step 3 "Direct In-Place Overwrite").
        self.K[slot] = k
        self.V[slot] = v
        self.vnorm[slot] = value_norm(v, self.policy.norm)
        self.pos[slot] = position
        self.acc[slot] = 0.0

    def prefill(self, k: np.ndarray, v: np.ndarray):
        """Initial fill: prompt tokens take slots 0..P-1 in order (guide, step 1).

        k, v [P][d] with P <= budget (eviction on; < budget when deferred, so
        that the step that fills the buffer picks the first victim) or
        <= capacity (eviction off).
        """
        P = len(k)
        limit = self.limit
        if self.evict and self.policy.deferred:
            limit -= 1
        if P > limit:
            raise ValueError("prompt longer than the buffer")
        for i in range(P):
            self._write(i, k[i], v[i], i)
        self.n = P
        self.p = P

    def slot_scores(self, alpha_slots: np.ndarray, n: int) -> np.ndarray:
        """This unit's score of each of its n slots (alpha over those slots)."""
        if self.policy.score == "h2o":
            return self.acc[:n].copy()
        return longflow_scores(alpha_slots, self.vnorm[:n])

    def step(self, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray) -> StepResult:
        """One decode step for this unit; q [G][d], k_new/v_new [d]."""
        if self.policy.scope != "kv_head" and self.evict:
            raise ValueError("a layer-wide victim needs OracleSequence")
        return group_step([self], [q], [k_new], [v_new])[0]

    def snapshot(self):
        return (self.K.copy(), self.V.copy(), self.vnorm.copy(), self.pos.copy(), self.n, self.p)


def group_step(units: Sequence[OracleUnit], qs, k_news, v_news) -> List[StepResult]:
    """One decode step of units that share one eviction decision.

    With the per-KV-head scope the group is one unit; with the layer scope it is
    every KV head of the sequence, and a slot's score is the sum of the units'
    scores for it.  Returns one StepResult per unit.
    """
    u0 = units[0]
    pol = u0.policy
    n, p = u0.n, u0.p
    for u in units:
        if (u.n, u.p) != (n, p) or u.pending != u0.pending:
            raise ValueError("units of one group must share occupancy and positions")
    if pol.deferred and u0.evict:
        return _deferred_group_step(units, qs, k_news, v_news)

    # Same-step order: attend over the n cached slots plus the new token, update
    # the accumulated attention, pick the victim among the cached slots, write.
    alphas, outs = [], []
    for u, q, kn, vn in zip(units, qs, k_news, v_news):
        keys = np.vstack([u.K[:n], np.asarray(kn, np.float64)[None]])
        values = np.vstack([u.V[:n], np.asarray(vn, np.float64)[None]])
        alpha, out = attention(q, keys, values, u.scale)
        if pol.score == "h2o":
            u.acc[:n] += alpha[:, :n].sum(axis=0)
        alphas.append(alpha)
        outs.append(out)
    scores, lowest, second = None, math.nan, math.nan
    evicted = -1
    if u0.evict and n >= u0.budget:
        scores = sum(u.slot_scores(a[:, :n], n) for u, a in zip(units, alphas))
        evicted, lowest, second = choose_victim(scores, u0.pos[:n], p, u0.window, pol.sinks)
        written = evicted
    elif n < u0.limit:
        written = n            # initial fill: next free slot
        for u in units:
            u.n = n + 1
    else:
        written = -1           # eviction off and the buffer is full: read-only
    results = []
    for u, kn, vn, a, out in zip(units, k_news, v_news, alphas, outs):
        if written >= 0:
            u._write(written, kn, vn, p)
            if pol.score == "h2o":
                u.acc[written] = a[:, n].sum()   # the new token's own weight
        u.p = p + 1
        results.append(StepResult(out=out, evicted=evicted, written=written, alpha=a,
                                  scores=scores, lowest=lowest, second=second, chosen=evicted))
    return results


def _deferred_group_step(units, qs, k_news, v_news) -> List[StepResult]:
    """Deferred order: write the new token into the next free slot or the slot
    chosen at the previous step, attend over the buffer, and once the buffer is
    full choose the slot the next token overwrites."""
    u0 = units[0]
    pol = u0.policy
    n, p = u0.n, u0.p
    if n < u0.budget:
        written, evicted, n_after = n, -1, n + 1
    else:
        if u0.pending < 0:
            raise ValueError("full buffer without a chosen slot")
        written, evicted, n_after = u0.pending, u0.pending, n
    alphas, outs = [], []
    for u, q, kn, vn in zip(units, qs, k_news, v_news):
        u._write(written, kn, vn, p)
        u.n = n_after
        alpha, out = attention(q, u.K[:n_after], u.V[:n_after], u.scale)
        if pol.score == "h2o":
            u.acc[:n_after] += alpha.sum(axis=0)
        alphas.append(alpha)
        outs.append(out)
    scores, lowest, second = None, math.nan, math.nan
    chosen = -1
    if n_after >= u0.budget:
        scores = sum(u.slot_scores(a, n_after) for u, a in zip(units, alphas))
        chosen, lowest, second = choose_victim(scores, u0.pos[:n_after], p + 1, u0.window,
                                               pol.sinks)
    results = []
    for u, a, out in zip(units, alphas, outs):
        u.pending = chosen
        u.p = p + 1
        results.append(StepResult(out=out, evicted=evicted, written=written, alpha=a,
                                  scores=scores, lowest=lowest, second=second, chosen=chosen))
    return results


class OracleSequence:
    """All KV heads of one (layer, sequence): q [H_q][d] -> out [H_q][d]."""

    def __init__(self, kv_heads: int, q_heads: int, capacity: int, head_dim: int,
                 budget: int, window: int, evict: bool = True, policy: Optional[Policy] = None):
        if q_heads % kv_heads:
            raise ValueError("q_heads must be a multiple of kv_heads")
        self.G = q_heads // kv_heads
        self.policy = policy or Policy()
        self.units = [OracleUnit(capacity, head_dim, budget, window, evict, self.policy)
                      for _ in range(kv_heads)]

    def prefill(self, k: np.ndarray, v: np.ndarray):
        """k, v [H_kv][P][d]."""
        for g, u in enumerate(self.units):
            u.prefill(k[g], v[g])

    def step(self, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray):
        """q [H_q][d], k_new/v_new [H_kv][d] -> (out [H_q][d], [StepResult per KV head])."""
        qs = [q[g * self.G:(g + 1) * self.G] for g in range(len(self.units))]
        if self.policy.scope == "layer":
            results = group_step(self.units, qs, k_new, v_new)
        else:
            results = [group_step([u], [qs[g]], [k_new[g]], [v_new[g]])[0]
                       for g, u in enumerate(self.units)]
        return np.vstack([r.out for r in results]), results
