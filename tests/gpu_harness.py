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
* an exact tie -- the oracle's two lowest candidate scores equal in fp64,
  which takes identical stored values -- has one right answer, the lowest
  tied slot (the tie rule), so there the slot must be bit-exact too: a
  different pick is a mismatch, never a resync;
* outputs: fp32 storage -- |x - y| <= 1e-5 * max(|y|, max |y| of that head);
  bf16 storage -- |x - y| <= 2e-2 + 1e-2 |y| (fp32 accumulation on the GPU);
* after the run, every sampled unit's slab state equals the oracle's: K, V and
  positions exactly, ||v||_1 to fp32 rounding, count and next position; with
  the H2O score the accumulators to fp32 accumulation (rtol 1e-4), and when
  deferred the chosen slot exactly.

Long prompts: a sequence's prompt tokens past its buffer are fed as its first
decode tokens, each with the query the stream draws for that step
(``InputStream.prompt_split``); the oracle receives the same tokens.

Policy variants: with the deferred order the slot chosen at a step is compared
through the cache's `pending` state (near-tie rule as above) and the slot the
step overwrote exactly; with the layer scope the oracle replays every KV head of
a sampled sequence as one group sharing one victim.
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
    exact_ties: int = 0
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
                 budgets: Optional[Sequence[int]] = None, device="cuda", kernel: str = "auto",
                 policy: Optional["oracle.Policy"] = None):
        self.wl = wl
        self.layers = list(layers)
        self.policy = pol = policy or oracle.Policy()
        self.stream = InputStream(wl, seed=seed, device=device, layers=self.layers)
        self.budgets = list(budgets) if budgets is not None else list(self.stream.budgets)
        cap = capacity if capacity is not None else max(self.budgets)
        self.capacity = cap
        self.evict = evict
        self.deferred = evict and pol.deferred
        self.h2o = evict and pol.score == "h2o"
        self.G = wl.q_heads // wl.kv_heads
        self.cache = LFCache(len(self.layers), wl.batch, wl.kv_heads, wl.q_heads, wl.head_dim,
                             cap, wl.window, dtype=wl.dtype, evict=evict,
                             budgets=self.budgets if evict else None, cluster=cluster,
                             stages=stages, kernel=kernel, score=pol.score, norm=pol.norm,
                             sinks=pol.sinks, deferred=pol.deferred, scope=pol.scope)
        if sample is None:
            sample = [(li, b, g) for li in range(len(self.layers)) for b in range(wl.batch)
                      for g in range(wl.kv_heads)]
        layer_scope = evict and pol.scope == "layer"
        if layer_scope:   # a sampled sequence brings all its KV heads
            sample = [(li, b, g) for (li, b) in sorted({(x[0], x[1]) for x in sample})
                      for g in range(wl.kv_heads)]
        self.sample = sorted(set(sample))
        self.groups = {}
        for (li, b, g) in self.sample:
            self.groups.setdefault((li, b) if layer_scope else (li, b, g), []).append((li, b, g))
        self.units = {}

        def limit(b):
            if not evict:
                return cap
            return self.budgets[b] - (1 if self.deferred else 0)

        self.overflow = []   # per layer: prompt tokens each sequence feeds as decode tokens
        for li, l in enumerate(self.layers):
            k, v, lens = self.stream.prompt_split(l, [limit(b) for b in range(wl.batch)])
            self.overflow.append(self.stream.overflow_lengths(l))
            self.cache.prefill(li, k, v, lens)
            for (sli, b, g) in self.sample:
                if sli != li:
                    continue
                u = oracle.OracleUnit(cap, wl.head_dim, self.budgets[b] if evict else cap,
                                      wl.window, evict, pol)
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

    def close(self):
        self.cache.close()

    def _resync(self, members):
        """Write the oracle's state of these units over the GPU's."""
        vw = self.views
        dt = self.cache.dtype
        cap = self.capacity
        for (li, b, g) in members:
            u = self.units[(li, b, g)]
            dev = vw["k"].device
            vw["k"][li, b, g, :cap] = torch.from_numpy(u.K).to(dt).to(dev)
            vw["v"][li, b, g, :cap] = torch.from_numpy(u.V).to(dt).to(dev)
            vw["vnorm"][li, b, g, :cap] = torch.from_numpy(u.vnorm).to(torch.float32).to(dev)
            vw["pos"][li, b, g, :cap] = torch.from_numpy(u.pos).to(torch.int32).to(dev)
            if self.h2o:
                vw["acc"][li, b, g, :cap] = torch.from_numpy(u.acc).to(torch.float32).to(dev)
            if self.deferred:
                vw["pending"][li, b, g] = int(u.pending)

    def _candidate(self, u: oracle.OracleUnit, pos_before, slot: int) -> bool:
        """Was `slot` a candidate at the step the oracle unit just took?"""
        pol, W = self.policy, self.wl.window
        p = u.p - 1                     # the step's token position
        if self.deferred:               # after the write; the window counts the new token
            ps = u.pos[slot]
            return bool(pol.sinks <= ps < p + 1 - W)
        ps = pos_before[slot]
        return bool(pol.sinks <= ps < p - W)

    def plant_tie(self, li: int, slots: Sequence[int], src: Optional[int] = None,
                  scale: float = 0.05):
        """Make `slots` of every unit of layer index `li` hold the same stored
        key and value: slot `src`'s (default: the first of `slots`), with the
        value scaled by `scale` so that a small ||v|| puts them at the bottom
        of the LongFlow score.  The GPU slab and the oracle units get the same
        bytes; each slot keeps its position."""
        vw = self.views
        src = slots[0] if src is None else src
        sl = torch.tensor(list(slots), device=vw["k"].device)
        krow = vw["k"][li, :, :, src].clone()
        vrow = (vw["v"][li, :, :, src].float() * scale).to(self.cache.dtype)
        norm = vrow.float().abs().sum(-1) if self.policy.norm == 1 else vrow.float().norm(dim=-1)
        n_s = len(slots)
        vw["k"][li][:, :, sl] = krow.unsqueeze(2).expand(-1, -1, n_s, -1)
        vw["v"][li][:, :, sl] = vrow.unsqueeze(2).expand(-1, -1, n_s, -1)
        vw["vnorm"][li][:, :, sl] = norm.unsqueeze(2).expand(-1, -1, n_s)
        torch.cuda.synchronize()
        for (sli, b, g), u in self.units.items():
            if sli != li:
                continue
            kk, vv = to64(krow[b, g]), to64(vrow[b, g])
            for s in slots:
                u.K[s] = kk
                u.V[s] = vv
                u.vnorm[s] = oracle.value_norm(vv, self.policy.norm)

    def step(self, check: bool = True, zero_query: bool = False):
        qs, ks, vs = self.stream.next_step()
        if zero_query:   # every weight uniform: the score is ||v|| (or the H2O mass) alone
            qs = [torch.zeros_like(q) for q in qs]
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
            pend = (self.views["pending"][li][bi, gi].cpu().numpy() if self.deferred else None)
            host[li] = ({bg: j for j, bg in enumerate(idx)}, to64(qg), to64(ks[li][bi, gi]),
                        to64(vs[li][bi, gi]), to64(og), self.ev[li][bi, gi].cpu().numpy(), pend)
        for key, members in self.groups.items():
            li = members[0][0]
            jmap, q, k, v, o, ev, pend = host[li]
            js = [jmap[(b, g)] for (_, b, g) in members]
            units = [self.units[m] for m in members]
            pos_before = [u.pos.copy() for u in units]
            res = oracle.group_step(units, [q[j] for j in js], [k[j] for j in js],
                                    [v[j] for j in js])
            self.stats.unit_steps += len(units)
            for m, j, r in zip(members, js, res):
                viol = out_violation(o[j], r.out, self.wl.dtype)
                if viol > self.stats.max_out_violation:
                    self.stats.max_out_violation = viol
                    self.stats.worst_out = (self.stats.steps,) + m + (viol,)
            r0 = res[0]
            if r0.evicted >= 0:
                self.stats.evictions += len(units)
            # The slot the GPU chose this step (same step: the one it overwrote;
            # deferred: its pending choice), and what the step overwrote.
            gpu_chosen = [int(pend[j]) if self.deferred else int(ev[j]) for j in js]
            if self.deferred:
                for m, j, r in zip(members, js, res):
                    if int(ev[j]) != r.evicted:
                        self.stats.hard_mismatches.append(
                            (self.stats.steps,) + m + (int(ev[j]), r.evicted, "overwritten"))
            exact = (r0.chosen >= 0 and r0.lowest == r0.second and r0.lowest >= TINY_SCORE)
            near = not exact and ((r0.rel_gap <= NEAR_TIE) or
                                  (r0.chosen >= 0 and r0.second < TINY_SCORE))
            if exact:
                self.stats.exact_ties += 1
            if near:
                self.stats.near_ties += 1
            if any(c != r0.chosen for c in gpu_chosen):
                e_gpu = gpu_chosen[0]
                if exact:   # one right answer: the lowest tied slot
                    self.stats.hard_mismatches.append(
                        (self.stats.steps,) + members[0] + (e_gpu, r0.chosen, "exact tie"))
                    self._resync(members)
                    continue
                ok_pick = (near and r0.scores is not None and all(c == e_gpu for c in gpu_chosen)
                           and 0 <= e_gpu < len(r0.scores)
                           and self._candidate(units[0], pos_before[0], e_gpu)
                           and r0.scores[e_gpu] <= r0.lowest * (1 + 2 * NEAR_TIE) + TINY_SCORE)
                if ok_pick:
                    self.stats.resyncs += 1
                else:
                    self.stats.hard_mismatches.append(
                        (self.stats.steps,) + members[0] + (e_gpu, r0.chosen, r0.rel_gap))
                self._resync(members)

    def run(self, steps: int, zero_query: bool = False) -> ParityStats:
        for t in range(steps):
            self.step(check=True, zero_query=zero_query)
        torch.cuda.synchronize()
        return self.stats

    def compare_state(self):
        """Sampled units' slab state against the oracle's."""
        vw = self.views
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
                self.stats.state_errors.append(f"{tag}: ||v|| differs "
                                               f"{np.abs(vn - u.vnorm[:n]).max()}")
            if self.h2o:
                acc = vw["acc"][li, b, g, :n].cpu().numpy().astype(np.float64)
                if not np.allclose(acc, u.acc[:n], rtol=1e-4, atol=1e-7):
                    self.stats.state_errors.append(f"{tag}: H2O accumulators differ "
                                                   f"{np.abs(acc - u.acc[:n]).max()}")
            if self.deferred and int(vw["pending"][li, b, g]) != u.pending:
                self.stats.state_errors.append(
                    f"{tag}: pending {int(vw['pending'][li, b, g])} vs {u.pending}")
        return self.stats

    def check_invariants(self):
        """Every unit (sampled or not): count within its buffer, the occupied
        positions unique, the W most recent positions and the sinks present,
        the deferred choice outside both; with the layer scope every KV head of
        a sequence holds the same positions."""
        vw = self.views
        cnt = vw["count"].cpu().numpy()
        nxt = vw["next_pos"].cpu().numpy()
        pos = vw["pos"].cpu().numpy()
        pend = vw["pending"].cpu().numpy() if self.deferred else None
        W, S = self.wl.window, self.policy.sinks
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
                        if not np.isin(np.arange(min(S, p)), live).all():
                            self.stats.state_errors.append(f"({li},{b},{g}): sink lost")
                    if self.deferred and n == lim:
                        e = int(pend[li, b, g])
                        if not (0 <= e < n and S <= pos[li, b, g, e] < p - W):
                            self.stats.state_errors.append(f"({li},{b},{g}): bad pending {e}")
                    if self.evict and self.policy.scope == "layer" and g > 0:
                        if not np.array_equal(live, pos[li, b, 0, :n]):
                            self.stats.state_errors.append(f"({li},{b}): heads disagree")
        return self.stats
