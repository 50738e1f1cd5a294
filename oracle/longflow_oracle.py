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

Readings where the pages are silent or ambiguous (each listed in the design doc):

* GQA: query head h reads KV head floor(h / G); each KV head keeps its own
  slots and evicts its own victim, scored by the sum over its G query heads.
* The new token attends to itself: the softmax runs over the n cached slots
  plus the new token (the guide's reference step also writes the token before
  attending).  Eviction is decided in the same step, among the cached slots,
  and the new token is written into the victim's slot.
* The W most recent cached positions (pos >= p - W, p = the new token's
  position) are never evicted; exact score ties go to the lowest slot index.
* Softmax scale 1/sqrt(d).  The cached ||v||_1 is taken from the stored value.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

__all__ = ["attention", "longflow_scores", "choose_victim", "OracleUnit", "StepResult",
           "OracleSequence"]


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


def longflow_scores(alpha_cached: np.ndarray, vnorm1: np.ndarray) -> np.ndarray:
    """LongFlow score of every cached slot of one KV head.

    score_i = sum_{h in group} ||c_{h,i}||_1 = sum_h alpha_{h,i} * ||v_i||_1
    (guide, "Mathematical Derivation of the LongFlow Score", the Score_LongFlow
    equation; summary, section 2.1, LongFlowScore(t_i) = alpha_i^t ||v_i||_1),
    summed over the group's query heads (GQA reading).
    alpha_cached [G][n], vnorm1 [n] -> [n].
    """
    return np.asarray(alpha_cached, np.float64).sum(axis=0) * np.asarray(vnorm1, np.float64)


def choose_victim(scores: np.ndarray, pos: np.ndarray, next_pos: int, window: int):
    """Lowest-score slot among the candidates (guide, "Static Memory
    Pre-Allocation and In-Place Eviction", step 2).

    Candidates are slots whose position is older than the protected window,
    pos_i < next_pos - window.  They are sorted by score with a stable sort, so
    equal scores stay in slot order and an exact tie goes to the lowest slot.
    Returns (victim slot, lowest score, second-lowest score or inf).
    """
    scores = np.asarray(scores, np.float64)
    cand = np.flatnonzero(np.asarray(pos) < next_pos - window)
    if cand.size == 0:
        raise ValueError("no eviction candidate: window covers every cached slot")
    order = cand[np.argsort(scores[cand], kind="stable")]
    best = int(order[0])
    second = float(scores[order[1]]) if order.size > 1 else math.inf
    return best, float(scores[best]), second


@dataclass
class StepResult:
    out: np.ndarray          # [G][d] attention output of the group's query heads
    evicted: int             # overwritten slot, or -1 (fill phase / eviction off)
    written: int             # slot the new token went to, or -1 (read-only full cache)
    alpha: np.ndarray        # [G][n+1] weights over cached slots then the new token
    scores: Optional[np.ndarray]  # [n] LongFlow scores when an eviction happened
    lowest: float            # lowest candidate score (nan when no eviction)
    second: float            # second-lowest candidate score (nan when no eviction)

    @property
    def rel_gap(self) -> float:
        """(second - lowest) / second: how far the victim is from a tie."""
        if not (self.evicted >= 0) or not math.isfinite(self.second) or self.second <= 0:
            return math.inf if self.evicted >= 0 else math.nan
        return (self.second - self.lowest) / self.second


class OracleUnit:
    """One cache unit: a KV head's static slot buffer for one layer and sequence.

    State (summary, section 2.3 "Static KV Cache"; guide, "Static Memory
    Pre-Allocation and In-Place Eviction"): K/V [capacity][d], the cached
    ||v||_1 per slot, the token position per slot, the occupied count n and the
    next token position p.  Nothing is ever moved or compacted.
    """

    def __init__(self, capacity: int, head_dim: int, budget: int, window: int,
                 evict: bool = True):
        if not (0 < budget <= capacity):
            raise ValueError("need 0 < budget <= capacity")
        if evict and not (0 <= window < budget):
            raise ValueError("need 0 <= window < budget")
        self.capacity, self.d, self.budget, self.window = capacity, head_dim, budget, window
        self.evict = evict
        self.K = np.zeros((capacity, head_dim))
        self.V = np.zeros((capacity, head_dim))
        self.vnorm = np.zeros(capacity)
        self.pos = np.full(capacity, -1, dtype=np.int64)
        self.n = 0
        self.p = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def _write(self, slot: int, k, v, position: int):
        # In-place overwrite of one slot (guide, step 3 "Direct In-Place Overwrite").
        self.K[slot] = k
        self.V[slot] = v
        self.vnorm[slot] = np.abs(np.asarray(v, np.float64)).sum()
        self.pos[slot] = position

    def prefill(self, k: np.ndarray, v: np.ndarray):
        """Initial fill: prompt tokens take slots 0..P-1 in order (guide, step 1).

        k, v [P][d] with P <= budget (eviction on) or <= capacity (eviction off).
        """
        P = len(k)
        limit = self.budget if self.evict else self.capacity
        if P > limit:
            raise ValueError("prompt longer than the buffer")
        for i in range(P):
            self._write(i, k[i], v[i], i)
        self.n = P
        self.p = P

    def step(self, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray) -> StepResult:
        """One decode step for this unit; q [G][d], k_new/v_new [d]."""
        n = self.n
        keys = np.vstack([self.K[:n], np.asarray(k_new, np.float64)[None]])
        values = np.vstack([self.V[:n], np.asarray(v_new, np.float64)[None]])
        alpha, out = attention(q, keys, values, self.scale)
        scores, lowest, second = None, math.nan, math.nan
        evicted = -1
        if self.evict and n >= self.budget:
            scores = longflow_scores(alpha[:, :n], self.vnorm[:n])
            evicted, lowest, second = choose_victim(scores, self.pos[:n], self.p, self.window)
            written = evicted
        elif n < (self.budget if self.evict else self.capacity):
            written = n            # initial fill: next free slot
            self.n = n + 1
        else:
            written = -1           # eviction off and the buffer is full: read-only
        if written >= 0:
            self._write(written, k_new, v_new, self.p)
        self.p += 1
        return StepResult(out=out, evicted=evicted, written=written, alpha=alpha,
                          scores=scores, lowest=lowest, second=second)

    def snapshot(self):
        return (self.K.copy(), self.V.copy(), self.vnorm.copy(), self.pos.copy(), self.n, self.p)


class OracleSequence:
    """All KV heads of one (layer, sequence): q [H_q][d] -> out [H_q][d]."""

    def __init__(self, kv_heads: int, q_heads: int, capacity: int, head_dim: int,
                 budget: int, window: int, evict: bool = True):
        if q_heads % kv_heads:
            raise ValueError("q_heads must be a multiple of kv_heads")
        self.G = q_heads // kv_heads
        self.units = [OracleUnit(capacity, head_dim, budget, window, evict)
                      for _ in range(kv_heads)]

    def prefill(self, k: np.ndarray, v: np.ndarray):
        """k, v [H_kv][P][d]."""
        for g, u in enumerate(self.units):
            u.prefill(k[g], v[g])

    def step(self, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray):
        """q [H_q][d], k_new/v_new [H_kv][d] -> (out [H_q][d], [StepResult per KV head])."""
        results = []
        outs = []
        for g, u in enumerate(self.units):
            r = u.step(q[g * self.G:(g + 1) * self.G], k_new[g], v_new[g])
            results.append(r)
            outs.append(r.out)
        return np.vstack(outs), results
