"""Plain, slow fp64 CPU oracle for R-KV's buffered compression step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this module; the
product path never does, and this module imports nothing from it.

R-KV is the baseline the LongFlow pages compare against.  Its README
("GitHub - Zefan-Cai/R-KV", section "Method -- Redundancy-aware KV Cache
Compression (R-KV)", the four-stage table) describes one compression step:

1. decoding-time staging: new tokens go to a buffer of B_buffer slots next to
   the retained cache of B_budget slots;
2. importance: the attention weights of the last alpha observation queries
   score every candidate token;
3. redundancy: cosine similarity between key vectors; of highly similar
   tokens at most beta of the most recent are kept, older near-duplicates are
   marked redundant;
4. joint selection: Z = lambda * Importance - (1 - lambda) * Redundancy; the
   top-scoring tokens plus the alpha observation tokens stay, within B_budget.

Defaults from the same README ("Default Hyper-parameters"): B_buffer = 128,
alpha = 8, lambda = 0.1.

Readings where the README is silent:

* one cache unit = one (layer, sequence, KV head), as for LongFlow; the
  observation queries are the group's G query heads at each of the alpha most
  recent decode steps;
* importance I_i = the mean over those alpha * G queries of their softmax
  weight on candidate i, the softmax taken over every candidate (scale
  1/sqrt(d));
* two keys count as near-duplicates when their cosine is >= tau; token i is
  redundant (R_i = 1) when at least beta candidates with a later position are
  near-duplicates of it, else R_i = 0.  The README gives no tau or beta:
  tau = 0.9, beta = 1 here;
* the alpha most recent positions are the observation tokens and always stay;
  the other B_budget - alpha places go to the highest Z, exact ties to the
  more recent token;
* the cache stays a static slab: a kept token in a retained slot (< B_budget)
  stays where it is; kept buffer tokens move into the freed retained slots,
  both taken in increasing slot order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

__all__ = ["RKVParams", "importance", "redundancy", "select_keep", "RKVUnit", "CompressResult"]


@dataclass(frozen=True)
class RKVParams:
    budget: int            # B_budget: slots kept after a compression
    buffer: int = 128      # B_buffer: staged tokens before a compression
    alpha: int = 8         # observation queries (and always-kept newest tokens)
    lam: float = 0.1       # lambda: importance / redundancy trade-off
    tau: float = 0.9       # cosine at or above which two keys are near-duplicates
    beta: int = 1          # near-duplicates kept among the most recent

    def validate(self):
        if not (0 < self.alpha < self.budget):
            raise ValueError("need 0 < alpha < budget")
        if self.buffer < 1 or self.beta < 1:
            raise ValueError("need buffer >= 1 and beta >= 1")


def importance(q_obs: np.ndarray, keys: np.ndarray, scale: float) -> np.ndarray:
    """Mean softmax weight of the observation queries on every candidate.

    q_obs [Q][d] (alpha * G query vectors), keys [n][d] -> I [n];
    w_{j,i} = exp(s_{j,i}) / sum_k exp(s_{j,k}), s = scale * q_j . k_i,
    I_i = (1/Q) sum_j w_{j,i}  (README, stage 2).
    """
    q = np.asarray(q_obs, np.float64)
    k = np.asarray(keys, np.float64)
    s = (q @ k.T) * scale
    w = np.exp(s - s.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    return w.mean(axis=0)


def redundancy(keys: np.ndarray, pos: np.ndarray, tau: float, beta: int) -> np.ndarray:
    """R_i = 1 if at least beta later tokens have cosine >= tau with token i.

    keys [n][d], pos [n] -> R [n] in {0, 1} (README, stage 3).
    """
    k = np.asarray(keys, np.float64)
    norms = np.sqrt((k * k).sum(axis=1))
    cos = (k @ k.T) / np.outer(norms, norms)
    pos = np.asarray(pos)
    newer = pos[None, :] > pos[:, None]            # [i][j]: j is later than i
    near = (cos >= tau) & newer
    return (near.sum(axis=1) >= beta).astype(np.float64)


def select_keep(z: np.ndarray, pos: np.ndarray, budget: int, alpha: int) -> np.ndarray:
    """Indices kept: the alpha latest positions, then the highest z (ties to
    the later position) until `budget` are kept (README, stage 4)."""
    pos = np.asarray(pos)
    n = len(pos)
    if n <= budget:
        return np.arange(n)
    by_recency = np.argsort(-pos, kind="stable")
    obs = set(by_recency[:alpha].tolist())
    rest = [i for i in range(n) if i not in obs]
    # highest z first; equal z: later position first
    rest.sort(key=lambda i: (-z[i], -pos[i]))
    keep = sorted(list(obs) + rest[:budget - alpha])
    return np.array(keep, dtype=np.int64)


@dataclass
class CompressResult:
    keep: np.ndarray         # kept candidate slots (before the moves), sorted
    imp: np.ndarray          # [n] importance
    red: np.ndarray          # [n] redundancy (0/1)
    z: np.ndarray            # [n] joint score
    moves: list              # [(from_slot, to_slot)] buffer tokens moved into freed slots
    cut: float               # z of the last token kept on score (nan if none)
    next_z: float            # z of the first token dropped (nan if none)


class RKVUnit:
    """One cache unit under R-KV: a static slab of budget + buffer slots.

    Decode steps append (the new token attends to itself, scale 1/sqrt(d));
    `compress` runs the four stages when more than `budget` slots are full.
    """

    def __init__(self, head_dim: int, params: RKVParams):
        params.validate()
        self.d = head_dim
        self.prm = params
        cap = params.budget + params.buffer
        self.K = np.zeros((cap, head_dim))
        self.V = np.zeros((cap, head_dim))
        self.pos = np.full(cap, -1, dtype=np.int64)
        self.n = 0
        self.p = 0

    @property
    def capacity(self) -> int:
        return self.prm.budget + self.prm.buffer

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def prefill(self, k: np.ndarray, v: np.ndarray):
        P = len(k)
        if P > self.capacity:
            raise ValueError("prompt longer than the slab")
        self.K[:P] = k
        self.V[:P] = v
        self.pos[:P] = np.arange(P)
        self.n = P
        self.p = P

    def step(self, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray) -> np.ndarray:
        """Attend over the n occupied slots plus the new token, then stage the
        token in slot n.  q [G][d] -> out [G][d]."""
        if self.n >= self.capacity:
            raise ValueError("buffer full: compress first")
        n = self.n
        keys = np.vstack([self.K[:n], np.asarray(k_new, np.float64)[None]])
        vals = np.vstack([self.V[:n], np.asarray(v_new, np.float64)[None]])
        s = (np.asarray(q, np.float64) @ keys.T) * self.scale
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        out = w @ vals
        self.K[n] = k_new
        self.V[n] = v_new
        self.pos[n] = self.p
        self.n = n + 1
        self.p += 1
        return out

    def compress(self, q_obs: np.ndarray) -> Optional[CompressResult]:
        """q_obs [alpha][G][d]: the observation queries.  Reduces the unit to
        `budget` slots; returns None when nothing is above the budget."""
        prm, n = self.prm, self.n
        if n <= prm.budget:
            return None
        keys = self.K[:n]
        pos = self.pos[:n]
        q = np.asarray(q_obs, np.float64).reshape(-1, self.d)
        imp = importance(q, keys, self.scale)
        red = redundancy(keys, pos, prm.tau, prm.beta)
        z = prm.lam * imp - (1.0 - prm.lam) * red
        keep = select_keep(z, pos, prm.budget, prm.alpha)
        kept = np.zeros(n, dtype=bool)
        kept[keep] = True
        # the z cut among tokens kept on score (not the observation tokens)
        obs = set(np.argsort(-pos, kind="stable")[:prm.alpha].tolist())
        scored = sorted([i for i in range(n) if i not in obs], key=lambda i: (-z[i], -pos[i]))
        m = prm.budget - prm.alpha
        cut = float(z[scored[m - 1]]) if m >= 1 else math.nan
        next_z = float(z[scored[m]]) if m < len(scored) else math.nan
        # static slab: kept buffer tokens fill the freed retained slots in order
        freed = [s for s in range(prm.budget) if s < n and not kept[s]]
        movers = [s for s in range(prm.budget, n) if kept[s]]
        assert len(freed) == len(movers)
        moves = list(zip(movers, freed))
        for src, dst in moves:
            self.K[dst] = self.K[src]
            self.V[dst] = self.V[src]
            self.pos[dst] = self.pos[src]
        self.K[prm.budget:] = 0.0
        self.V[prm.budget:] = 0.0
        self.pos[prm.budget:] = -1
        self.n = prm.budget
        return CompressResult(keep=keep, imp=imp, red=red, z=z, moves=moves, cut=cut,
                              next_z=next_z)
