"""GPU-vs-oracle parity harness (used by the ``-m gpu`` tests and smoke()).

The CUDA path runs every unit of the chosen layers; a sample of
(layer, sequence, KV head) units is replayed in lock-step by the fp64 oracle on
the exact stored-precision inputs the kernels consumed.

Comparison rules:

* evicted slots are bit-exact wherever the oracle's two lowest candidate
  scores differ by more than ``NEAR_TIE`` relative; a step within that band is
  a near-tie.  A near-tie on which the two sides pick different slots is
  counted and resynchronised: the oracle's state of that unit (K, V, ||v||_1,
  positions) is written over the GPU's through the slab layout, so both
  continue from the oracle's state;
* outputs: fp32 storage -- |x - y| <= 1e-5 * max(|y|, max |y| of that head);
  bf16 storage -- |x - y| <= 2e-2 + 1e-2 |y| (fp32 accumulation on the GPU);
* after the run, every sampled unit's slab state equals the oracle's: K, V and
  positions exactly, ||v||_1 to fp32 rounding, count and next position.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

import oracle
from decode_kv_cache_gb300.longflow import LFCache
from synth.workloads import InputStream, Workload

NEAR_TIE = 1e-3
TINY_SCORE = 1e-30


def out_violation(gpu: np.ndarray, ref: np.ndarray, dtype: str) -> float:
    """Largest |x - y| / allowed over one unit's [G][d] output (<= 1 passes)."""
    err = np.abs(gpu - ref)
    if dtype == "f32":
        scale = np.maximum(np.abs(ref), np.abs(ref).max(axis=1, keepdims=True))
        allowed = 1e-5 * np.maximum(scale, 1e-30)
    else:
        allowed = 2e-2 + 1e-2 * np.abs(ref)
    return float((err / allowed).max())


@dataclass
class ParityStats:
    steps: int = 0
    unit_steps: int = 0
    evictions: int = 0
    near_ties: int = 0
    resyncs: int = 0
    hard_mismatches: List[Tuple] = field(default_factory=list)
    max_out_violation: float = 0.0
    worst_out: Optional[Tuple] = None
    state_errors: List[str] = field(default_factory=list)

    def assert_ok(self):
        assert not self.hard_mismatches, f"evicted-slot mismatches: {self.hard_mismatches[:5]}"
        assert self.max_out_violation <= 1.0, f"output tolerance exceeded: {self.worst_out}"
        assert not self.state_errors, self.state_errors[:5]


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class ParityRun:
    """One cache on the GPU + oracle units for a sample of its units."""

    def __init__(self, wl: Workload, layers: Sequence[int] = (0,), seed: int = 0,
                 sample: Optional[Sequence[Tuple[int, int, int]]] = None, cluster: int = 0,
                 stages: int = 0, evict: bool = True, capacity: Optional[int] = None,
                 budgets: Optional[Sequence[int]] = None, device="cuda", kernel: str = "auto"):
        self.wl = wl
        self.layers = list(layers)
        self.stream = InputStream(wl, seed=seed, device=device, layers=self.layers)
        self.budgets = list(budgets) if budgets is not None else list(self.stream.budgets)
        cap = capacity if capacity is not None else max(self.budgets)
        self.capacity = cap
        self.evict = evict
        self.G = wl.q_heads // wl.kv_heads
        self.cache = LFCache(len(self.layers), wl.batch, wl.kv_heads, wl.q_heads, wl.head_dim,
                             cap, wl.window, dtype=wl.dtype, evict=evict,
                             budgets=self.budgets if evict else None, cluster=cluster,
                             stages=stages, kernel=kernel)
        if sample is None:
            sample = [(li, b, g) for li in range(len(self.layers)) for b in range(wl.batch)
                      for g in range(wl.kv_heads)]
        self.sample = list(sample)
        self.units = {}
        limit = lambda b: self.budgets[b] if evict else cap
        for li, l in enumerate(self.layers):
            k, v, lens = self.stream.prompt(l)
            lens = [min(P, limit(b)) for b, P in enumerate(lens)]
            self.cache.prefill(li, k, v, lens)
            for (sli, b, g) in self.sample:
                if sli != li:
                    continue
                u = oracle.OracleUnit(cap, wl.head_dim, self.budgets[b] if evict else cap,
                                      wl.window, evict)
                P = lens[b]
                u.prefill(to64(k[b, g, :P]), to64(v[b, g, :P]))
                self.units[(li, b, g)] = u
        torch.cuda.synchronize()
        dev = torch.device(device)
        self.out = [torch.empty(wl.batch, wl.q_heads, wl.head_dim, dtype=self.cache.dtype,
                                device=dev) for _ in self.layers]
        self.ev = [torch.empty(wl.batch, wl.kv_heads, dtype=torch.int32, device=dev)
                   for _ in self.layers]
        self.views = self.cache.views()
        self.stats = ParityStats()
        self._pos_before = {}

    def close(self):
        self.cache.close()

    def _was_candidate(self, li, b, g, slot, u: oracle.OracleUnit) -> bool:
        # u has already advanced one step: its p is the new token's position + 1
        return bool(self._pos_before[(li, b, g)][slot] < (u.p - 1) - self.wl.window)

    def _resync(self, li, b, g, u: oracle.OracleUnit):
        vw = self.views
        dt = self.cache.dtype
        cap = self.capacity
        vw["k"][li, b, g, :cap] = torch.from_numpy(u.K).to(dt).to(vw["k"].device)
        vw["v"][li, b, g, :cap] = torch.from_numpy(u.V).to(dt).to(vw["v"].device)
        vw["vnorm"][li, b, g, :cap] = torch.from_numpy(u.vnorm).to(torch.float32).to(vw["k"].device)
        vw["pos"][li, b, g, :cap] = torch.from_numpy(u.pos).to(torch.int32).to(vw["k"].device)

    def step(self, check: bool = True):
        qs, ks, vs = self.stream.next_step()
        for li in range(len(self.layers)):
            self.cache.decode_step(li, qs[li], ks[li], vs[li], self.out[li], self.ev[li])
        self.stats.steps += 1
        if not check:
            return
        G = self.G
        # Pull only the sampled units' inputs and results to the host.
        host = {}
        for li in range(len(self.layers)):
            idx = [(b, g) for (sli, b, g) in self.sample if sli == li]
            if not idx:
                continue
            bi = torch.tensor([b for b, _ in idx], device=qs[li].device)
            gi = torch.tensor([g for _, g in idx], device=qs[li].device)
            qg = qs[li].view(self.wl.batch, self.wl.kv_heads, G, self.wl.head_dim)[bi, gi]
            og = self.out[li].view(self.wl.batch, self.wl.kv_heads, G, self.wl.head_dim)[bi, gi]
            host[li] = (idx, to64(qg), to64(ks[li][bi, gi]), to64(vs[li][bi, gi]), to64(og),
                        self.ev[li][bi, gi].cpu().numpy())
        for li, (idx, q, k, v, o, ev) in host.items():
            for j, (b, g) in enumerate(idx):
                u = self.units[(li, b, g)]
                self._pos_before[(li, b, g)] = u.pos.copy()
                r = u.step(q[j], k[j], v[j])
                self.stats.unit_steps += 1
                viol = out_violation(o[j], r.out, self.wl.dtype)
                if viol > self.stats.max_out_violation:
                    self.stats.max_out_violation = viol
                    self.stats.worst_out = (self.stats.steps, li, b, g, viol)
                if r.evicted >= 0:
                    self.stats.evictions += 1
                near = (r.rel_gap <= NEAR_TIE) or (r.evicted >= 0 and r.second < TINY_SCORE)
                if near:
                    self.stats.near_ties += 1
                e_gpu = int(ev[j])
                if e_gpu != r.evicted:
                    # A different pick is acceptable only at a near-tie, and only
                    # if the GPU's slot was a candidate within the tie band.
                    ok_pick = (near and r.scores is not None and 0 <= e_gpu < len(r.scores)
                               and self._was_candidate(li, b, g, e_gpu, u)
                               and r.scores[e_gpu] <= r.lowest * (1 + 2 * NEAR_TIE) + TINY_SCORE)
                    if ok_pick:
                        self.stats.resyncs += 1
                        self._resync(li, b, g, u)
                    else:
                        self.stats.hard_mismatches.append(
                            (self.stats.steps, li, b, g, e_gpu, r.evicted, r.rel_gap))
                        self._resync(li, b, g, u)

    def run(self, steps: int, check_every: int = 1) -> ParityStats:
        for t in range(steps):
            self.step(check=True)
        torch.cuda.synchronize()
        return self.stats

    def compare_state(self):
        """Sampled units' slab state against the oracle's."""
        vw = self.views
        cap = self.capacity
        for (li, b, g), u in self.units.items():
            n = u.n
            k = to64(vw["k"][li, b, g, :n])
            v = to64(vw["v"][li, b, g, :n])
            pos = vw["pos"][li, b, g, :n].cpu().numpy()
            vn = vw["vnorm"][li, b, g, :n].cpu().numpy().astype(np.float64)
            cnt = int(vw["count"][li, b, g])
            nxt = int(vw["next_pos"][li, b, g])
            tag = (li, b, g)
            if cnt != u.n or nxt != u.p:
                self.stats.state_errors.append(f"{tag}: count/next {cnt}/{nxt} vs {u.n}/{u.p}")
                continue
            if not np.array_equal(pos, u.pos[:n]):
                self.stats.state_errors.append(f"{tag}: positions differ")
            if not (np.array_equal(k, u.K[:n]) and np.array_equal(v, u.V[:n])):
                self.stats.state_errors.append(f"{tag}: K/V differ")
            if not np.allclose(vn, u.vnorm[:n], rtol=2e-6, atol=1e-6):
                self.stats.state_errors.append(f"{tag}: ||v||_1 differs "
                                               f"{np.abs(vn - u.vnorm[:n]).max()}")
        return self.stats

    def check_invariants(self):
        """Every unit (sampled or not): count within its buffer, the occupied
        positions unique, and the W most recent positions present."""
        vw = self.views
        cnt = vw["count"].cpu().numpy()
        nxt = vw["next_pos"].cpu().numpy()
        pos = vw["pos"].cpu().numpy()
        W = self.wl.window
        for li in range(len(self.layers)):
            for b in range(self.wl.batch):
                lim = self.budgets[b] if self.evict else self.capacity
                for g in range(self.wl.kv_heads):
                    n, p = int(cnt[li, b, g]), int(nxt[li, b, g])
                    if not (0 <= n <= lim):
                        self.stats.state_errors.append(f"count {n} outside [0,{lim}]")
                        continue
                    live = pos[li, b, g, :n]
                    if len(np.unique(live)) != n or (n and (live.min() < 0 or live.max() >= p)):
                        self.stats.state_errors.append(f"({li},{b},{g}): bad positions")
                    if self.evict:
                        recent = np.arange(max(0, p - W), p)
                        if not np.isin(recent, live).all():
                            self.stats.state_errors.append(f"({li},{b},{g}): window lost")
        return self.stats
