"""GPU-vs-oracle harness for R-KV's compression (used by test_gpu_rkv.py and smoke()).

A cache in R-KV mode appends every decode step's token into its staging
buffer; whenever the buffer is full the harness calls lf_rkv_compress with the
queries of the last alpha steps and replays the same on oracle units.

Rules: outputs as for LongFlow (bf16: |x - y| <= 2e-2 + 1e-2 |y|); after a
compression the set of kept positions is exact, except at a near-tie of the
joint score Z at the budget cut (relative gap under 1e-4), where the GPU's
pick must come from the tied band and the oracle's state is written over the
GPU's; when the sets agree the slot layout (K, V, positions per slot) is
exact.  Source: "GitHub - Zefan-Cai/R-KV", section "Method".
"""
import numpy as np
import torch

from decode_kv_cache_gb300.longflow import LFCache
from gpu_harness import out_violation, to64
from oracle import rkv_oracle
from synth.workloads import InputStream

NEAR = 1e-4


class RKVRun:
    def __init__(self, wl, sample=None, seed=0):
        self.wl = wl
        self.B, self.buf, self.alpha = wl.budget, wl.rkv_buffer, wl.rkv_alpha
        self.cap = self.B + self.buf
        self.G = wl.q_heads // wl.kv_heads
        self.stream = InputStream(wl, seed=seed, device="cuda", layers=[0])
        self.cache = LFCache(1, wl.batch, wl.kv_heads, wl.q_heads, wl.head_dim, self.cap, 0,
                             dtype=wl.dtype, evict="rkv", rkv_buffer=self.buf,
                             rkv_alpha=self.alpha, rkv_beta=wl.rkv_beta,
                             rkv_lambda=wl.rkv_lambda, rkv_tau=wl.rkv_tau)
        self.prm = rkv_oracle.RKVParams(budget=self.B, buffer=self.buf, alpha=self.alpha,
                                        lam=wl.rkv_lambda, tau=wl.rkv_tau, beta=wl.rkv_beta)
        k, v, lens = self.stream.prompt(0)
        lens = [min(P, self.cap) for P in lens]
        self.cache.prefill(0, k, v, lens)
        self.sample = sample or [(b, g) for b in range(wl.batch) for g in range(wl.kv_heads)]
        self.units = {}
        for (b, g) in self.sample:
            u = rkv_oracle.RKVUnit(wl.head_dim, self.prm)
            u.prefill(to64(k[b, g, :lens[b]]), to64(v[b, g, :lens[b]]))
            self.units[(b, g)] = u
        self.views = self.cache.views()
        self.out = torch.empty(wl.batch, wl.q_heads, wl.head_dim, dtype=self.cache.dtype,
                               device="cuda")
        self.ev = torch.empty(wl.batch, wl.kv_heads, dtype=torch.int32, device="cuda")
        self.qhist = []   # the last alpha queries, [b][H_q][d] each
        self.max_viol = 0.0
        self.compressions = 0
        self.near_ties = 0
        self.redundant = 0
        self.errors = []

    def step(self):
        qs, ks, vs = self.stream.next_step()
        q, k, v = qs[0], ks[0], vs[0]
        self.cache.decode_step(0, q, k, v, self.out, self.ev)
        self.qhist = (self.qhist + [q])[-self.alpha:]
        G = self.G
        qh = to64(q).reshape(self.wl.batch, self.wl.kv_heads, G, -1)
        kh, vh, oh = to64(k), to64(v), to64(self.out).reshape(self.wl.batch, self.wl.kv_heads, G, -1)
        for (b, g), u in self.units.items():
            ref = u.step(qh[b, g], kh[b, g], vh[b, g])
            self.max_viol = max(self.max_viol, out_violation(oh[b, g], ref, self.wl.dtype))

    def compress(self):
        q_obs = torch.stack(self.qhist, dim=1).contiguous()   # [b][alpha][H_q][d]
        self.cache.rkv_compress(0, q_obs)
        torch.cuda.synchronize()
        self.compressions += 1
        qo = to64(q_obs).reshape(self.wl.batch, self.alpha, self.wl.kv_heads, self.G, -1)
        vw = self.views
        for (b, g), u in self.units.items():
            before_pos = u.pos[:u.n].copy()
            r = u.compress(qo[b, :, g])
            self.redundant += int(r.red.sum())
            gpu_pos = vw["pos"][0, b, g, :self.B].cpu().numpy()
            cnt = int(vw["count"][0, b, g])
            if cnt != self.B:
                self.errors.append(f"({b},{g}): count {cnt}")
                continue
            if set(gpu_pos.tolist()) != set(u.pos[:self.B].tolist()):
                # the kept sets differ: only tokens whose Z ties at the cut may swap
                gap = abs(r.cut - r.next_z) / max(abs(r.cut), 1e-30)
                zpos = dict(zip(before_pos.tolist(), r.z.tolist()))
                lo, hi = min(r.cut, r.next_z), max(r.cut, r.next_z)
                band = NEAR * max(abs(r.cut), 1e-30)
                diff = set(gpu_pos.tolist()) ^ set(u.pos[:self.B].tolist())
                ok = gap <= NEAR and all(lo - band <= zpos.get(p, np.inf) <= hi + band
                                         for p in diff)
                if ok:
                    self.near_ties += 1
                else:
                    self.errors.append(f"({b},{g}) compression {self.compressions}: kept sets "
                                       f"differ by {sorted(diff)[:6]} (cut gap {gap:.2e})")
                self._resync(b, g, u)
                continue
            # same set: the layout is exact
            if not np.array_equal(gpu_pos, u.pos[:self.B]):
                self.errors.append(f"({b},{g}): slot layout differs")
            elif not (np.array_equal(to64(vw["k"][0, b, g, :self.B]), u.K[:self.B]) and
                      np.array_equal(to64(vw["v"][0, b, g, :self.B]), u.V[:self.B])):
                self.errors.append(f"({b},{g}): K/V after the moves differ")

    def _resync(self, b, g, u):
        vw = self.views
        dev = vw["k"].device
        n = u.capacity
        vw["k"][0, b, g, :n] = torch.from_numpy(u.K).to(self.cache.dtype).to(dev)
        vw["v"][0, b, g, :n] = torch.from_numpy(u.V).to(self.cache.dtype).to(dev)
        vw["pos"][0, b, g, :n] = torch.from_numpy(u.pos).to(torch.int32).to(dev)

    def run(self, steps):
        for t in range(steps):
            if int(self.views["count"][0, 0, 0]) == self.cap:
                self.compress()
            self.step()
        torch.cuda.synchronize()
        bits = self.cache.check()
        assert bits == 0, f"device error word {bits}"
        assert self.max_viol <= 1.0, self.max_viol
        assert not self.errors, self.errors[:4]
        return self

    def close(self):
        self.cache.close()
