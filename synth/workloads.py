"""Seeded synthetic workloads for the LongFlow fused decode step.

This module only *draws inputs*: prompt keys/values, per-step queries and new
keys/values, and the per-sequence prompt lengths, budgets and AR(1) rates of the
ragged workload.  It contains none of the method's arithmetic (no attention, no
score, no eviction), so the fp64 oracle and the CUDA path can both consume its
output without sharing any code of the method.

The five workloads mirror the shapes of the pages' experiments (DeepSeek-R1-
Distill-Llama-8B and Qwen3-0.6B/8B head geometry, a 16k-token generation kept
at a 20% budget of 3276 slots).  The pages measure on AIME24 / MATH-500 /
GSM8K / LiveCodeBench with trained weights; none of those are available, so
these seeded streams stand in for them and reproduce only shapes, sizes and the
temporal correlation of consecutive queries that the pages' query approximation
relies on.

Every draw comes from a ``torch.Generator`` seeded from ``(seed, purpose,
layer)``, so a stream is reproducible on a given device and torch build.  The
parity tests generate on the device that runs the kernels and copy the exact
stored-precision bytes of the sampled units to the host for the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import List, Optional, Sequence, Tuple

import torch

__all__ = ["Workload", "WORKLOADS", "InputStream", "get_workload", "torch_dtype"]


@dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic decode workload."""

    name: str
    layers: int
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    budget: int              # per-sequence slot budget B (max over sequences when ragged)
    window: int              # W most recent cached positions are never evicted
    prefill: int             # prompt length P (max when ragged)
    steps: int               # decode steps of the full workload
    dtype: str               # "f32" or "bf16": storage and I/O type of q, K, V, out
    rho: float = 0.9         # AR(1) coefficient of consecutive queries
    innovation: Optional[float] = None   # AR(1) innovation std; None -> sqrt(1 - rho^2)
    v_lognormal_sigma: float = 0.0       # v_i *= exp(sigma * z_i), z_i ~ N(0,1) per token
    sink_prob: float = 0.0   # probability that a token's keys get the shared sink direction
    sink_sigmas: float = 3.0  # sink shift = sink_sigmas * sqrt(d) * u (u unit vector)
    ragged: bool = False
    budget_choices: Tuple[int, ...] = ()
    prompt_range: Tuple[int, int] = (0, 0)
    rho_range: Tuple[float, float] = (0.0, 0.0)
    reset_every: int = 0     # fresh N(0,1) query every `reset_every` steps (0: never)
    full_kv_capacity: int = 0  # capacity of the eviction-off full-KV comparison (0: none)
    # Near-duplicate keys: with probability dup_prob a token's key is one of
    # dup_bank seeded pattern vectors of its (layer, KV head) plus relative noise
    # dup_noise, so tokens sharing a pattern are near-duplicates of each other.
    dup_prob: float = 0.0
    dup_bank: int = 64
    dup_noise: float = 0.02
    # R-KV compression (0: not an R-KV workload): staging buffer, observation
    # queries, lambda, cosine threshold and near-duplicates kept.
    rkv_buffer: int = 0
    rkv_alpha: int = 8
    rkv_lambda: float = 0.1
    rkv_tau: float = 0.9
    rkv_beta: int = 1

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def scaled(self, **kw) -> "Workload":
        """Same recipe with some sizes replaced (used for small parity cases)."""
        return replace(self, **kw)


WORKLOADS = {
    # Tiny fp32 case the oracle finishes in well under a second.
    "tiny-fp32": Workload(
        name="tiny-fp32", layers=1, batch=1, q_heads=2, kv_heads=1, head_dim=16,
        budget=32, window=4, prefill=8, steps=64, dtype="f32",
        rho=0.9, innovation=0.44),
    # Qwen3-0.6B attention geometry: 16 query / 8 KV heads, d=128.
    "qwen3-0.6b": Workload(
        name="qwen3-0.6b", layers=28, batch=8, q_heads=16, kv_heads=8, head_dim=128,
        budget=512, window=16, prefill=256, steps=4096, dtype="bf16",
        rho=0.9, v_lognormal_sigma=0.5),
    # DeepSeek-R1-Distill-Llama-8B geometry, 20% budget of a 16k generation, sink keys.
    "r1-llama-8b": Workload(
        name="r1-llama-8b", layers=32, batch=32, q_heads=32, kv_heads=8, head_dim=128,
        budget=3276, window=64, prefill=512, steps=16384, dtype="bf16",
        rho=0.9, innovation=0.44, sink_prob=0.01),
    # Qwen3-8B geometry in steady state: cache pre-filled to the budget.
    "qwen3-8b-steady": Workload(
        name="qwen3-8b-steady", layers=36, batch=64, q_heads=32, kv_heads=8, head_dim=128,
        budget=3276, window=64, prefill=3276, steps=2048, dtype="bf16",
        rho=0.9, innovation=0.44, sink_prob=0.01, full_kv_capacity=16384),
    # Ragged serving stress: per-sequence prompts, budgets and query correlation.
    "ragged-serving": Workload(
        name="ragged-serving", layers=32, batch=256, q_heads=32, kv_heads=8, head_dim=128,
        budget=3276, window=32, prefill=2048, steps=8192, dtype="bf16",
        ragged=True, budget_choices=(512, 1024, 2048, 3276), prompt_range=(64, 2048),
        rho_range=(0.6, 0.98), reset_every=1000),
    # R-KV, the pages' baseline, on the R1-Llama-8B geometry: 3276 retained slots
    # plus a 128-token staging buffer, compressed whenever the buffer is full;
    # 5% of tokens are near-duplicates of a per-head pattern (repeated
    # reasoning), the redundancy R-KV removes.  Prefilled to the budget.
    "rkv-r1-llama-8b": Workload(
        name="rkv-r1-llama-8b", layers=32, batch=32, q_heads=32, kv_heads=8, head_dim=128,
        budget=3276, window=0, prefill=3276, steps=16384, dtype="bf16",
        rho=0.9, innovation=0.44, v_lognormal_sigma=0.5, dup_prob=0.05, rkv_buffer=128),
}


def get_workload(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


# Purposes keep independent draws in independent streams.
_PURPOSE = {"seq": 1, "q0": 2, "step": 3, "prompt": 4, "sinkdir": 5, "dupbank": 6}


def _gen(seed: int, purpose: str, layer: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + _PURPOSE[purpose] * 10_007 + int(layer)) % (2**63))
    return g


class InputStream:
    """Seeded stream of prompts and per-step decode inputs for one workload.

    ``layers`` selects the layer indices that are drawn (default: all); each
    layer's streams depend only on ``(seed, layer)``, so a subset reproduces the
    same values as the full run for those layers.
    """

    def __init__(self, wl: Workload, seed: int = 0, device="cpu",
                 layers: Optional[Sequence[int]] = None):
        self.wl = wl
        self.seed = int(seed)
        self.device = torch.device(device)
        self.layer_ids: List[int] = list(range(wl.layers)) if layers is None else list(layers)
        self.dtype = torch_dtype(wl.dtype)
        b, hq, d = wl.batch, wl.q_heads, wl.head_dim

        # Per-sequence parameters (ragged workload); identical for every layer.
        gs = _gen(seed, "seq", 0, "cpu")
        if wl.ragged:
            lo, hi = wl.prompt_range
            self.prompt_lens = torch.randint(lo, hi + 1, (b,), generator=gs).tolist()
            idx = torch.randint(0, len(wl.budget_choices), (b,), generator=gs)
            self.budgets = [wl.budget_choices[i] for i in idx.tolist()]
            r0, r1 = wl.rho_range
            self.rhos = (r0 + (r1 - r0) * torch.rand(b, generator=gs, dtype=torch.float64)).tolist()
        else:
            self.prompt_lens = [wl.prefill] * b
            self.budgets = [wl.budget] * b
            self.rhos = [wl.rho] * b
        if wl.innovation is not None and not wl.ragged:
            self.innovations = [wl.innovation] * b
        else:
            self.innovations = [math.sqrt(max(0.0, 1.0 - r * r)) for r in self.rhos]
        self._rho_t = torch.tensor(self.rhos, dtype=torch.float32, device=self.device).view(b, 1, 1)
        self._sig_t = torch.tensor(self.innovations, dtype=torch.float32,
                                   device=self.device).view(b, 1, 1)

        # Per-layer state: AR(1) query state and the shared sink direction.
        self._gstep = {l: _gen(seed, "step", l, self.device) for l in self.layer_ids}
        self._q = {}
        self._sink_u = {}
        self._bank = {}
        for l in self.layer_ids:
            if wl.dup_prob > 0:
                gb = _gen(seed, "dupbank", l, self.device)
                self._bank[l] = torch.randn(wl.kv_heads, wl.dup_bank, d, generator=gb,
                                            device=self.device)
            g0 = _gen(seed, "q0", l, self.device)
            self._q[l] = torch.randn(b, hq, d, generator=g0, device=self.device)
            if wl.sink_prob > 0:
                gu = _gen(seed, "sinkdir", l, self.device)
                u = torch.randn(wl.kv_heads, d, generator=gu, device=self.device)
                self._sink_u[l] = u / u.norm(dim=-1, keepdim=True)
        self.t = 0  # decode steps drawn so far
        # Prompt tokens past a sequence's buffer limit, fed as its next decode
        # tokens (see prompt_split): layer -> (k [b][H_kv][n][d], v, lengths [b]).
        self._overflow = {}

    # -- token K/V recipe shared by prompt and decode tokens -----------------
    def _tokens(self, g: torch.Generator, layer: int, n: int):
        """Draw K, V for `n` tokens of every sequence: [b][H_kv][n][d] fp32."""
        wl = self.wl
        shape = (wl.batch, wl.kv_heads, n, wl.head_dim)
        k = torch.randn(shape, generator=g, device=self.device)
        v = torch.randn(shape, generator=g, device=self.device)
        if wl.v_lognormal_sigma > 0:
            z = torch.randn(wl.batch, 1, n, 1, generator=g, device=self.device)
            v = v * torch.exp(wl.v_lognormal_sigma * z)
        if wl.sink_prob > 0:
            is_sink = (torch.rand(wl.batch, 1, n, 1, generator=g, device=self.device)
                       < wl.sink_prob).to(torch.float32)
            shift = wl.sink_sigmas * math.sqrt(wl.head_dim) * self._sink_u[layer]
            k = k + is_sink * shift.view(1, wl.kv_heads, 1, wl.head_dim)
        if wl.dup_prob > 0:
            is_dup = (torch.rand(wl.batch, wl.kv_heads, n, 1, generator=g, device=self.device)
                      < wl.dup_prob)
            pick = torch.randint(0, wl.dup_bank, (wl.batch, wl.kv_heads, n), generator=g,
                                 device=self.device)
            bank = self._bank[layer]                                   # [H_kv][bank][d]
            pattern = torch.stack([bank[h][pick[:, h]] for h in range(wl.kv_heads)], dim=1)
            noise = torch.randn(shape, generator=g, device=self.device)
            k = torch.where(is_dup, pattern + wl.dup_noise * noise, k)
        return k, v

    def prompt(self, layer: int):
        """Prompt K/V of one layer: ([b][H_kv][P_max][d], same, prompt_lens list).

        Entries past a sequence's own prompt length are drawn too but unused.
        """
        g = _gen(self.seed, "prompt", layer, self.device)
        pmax = max(self.prompt_lens)
        k, v = self._tokens(g, layer, pmax)
        return k.to(self.dtype).contiguous(), v.to(self.dtype).contiguous(), list(self.prompt_lens)

    def prompt_split(self, layer: int, limits: Sequence[int]):
        """Prompt of one layer cut at each sequence's buffer limit.

        Returns (k, v, lens) like ``prompt`` with lens[b] = min(P_b, limits[b]):
        the part that prefills the buffer.  The rest of a longer prompt,
        positions limits[b] .. P_b - 1, is kept and comes out of ``next_step``
        as that sequence's k_new / v_new for its first P_b - limits[b] decode
        steps, each with the query the stream draws for that step.  The batch
        advances in lock-step: sequences without such a remainder take drawn
        tokens from the first step on.  Every step draws the same random
        numbers either way, so the other sequences' streams are unchanged.
        """
        k, v, lens = self.prompt(layer)
        cut = [min(P, int(lim)) for P, lim in zip(lens, limits)]
        extra = [P - c for P, c in zip(lens, cut)]
        if max(extra) > 0:
            n = max(extra)
            ok = torch.zeros(k.shape[0], k.shape[1], n, k.shape[3], dtype=k.dtype,
                             device=k.device)
            ov = torch.zeros_like(ok)
            for b, (c, e) in enumerate(zip(cut, extra)):
                if e > 0:
                    ok[b, :, :e] = k[b, :, c:c + e]
                    ov[b, :, :e] = v[b, :, c:c + e]
            self._overflow[layer] = (ok, ov, torch.tensor(extra, device=self.device))
        else:
            self._overflow.pop(layer, None)
        return k, v, cut

    def overflow_lengths(self, layer: int) -> List[int]:
        """Prompt tokens of each sequence still to be fed as decode tokens
        (counted from the start of decoding)."""
        if layer not in self._overflow:
            return [0] * self.wl.batch
        return self._overflow[layer][2].tolist()

    def next_step(self):
        """Advance one decode step for every drawn layer.

        Returns (q, k_new, v_new), each a list over ``layer_ids`` of tensors
        [b][H_q][d], [b][H_kv][d], [b][H_kv][d] in the workload dtype.
        """
        wl = self.wl
        self.t += 1
        qs, ks, vs = [], [], []
        for l in self.layer_ids:
            g = self._gstep[l]
            eps = torch.randn(self._q[l].shape, generator=g, device=self.device)
            if wl.reset_every and self.t % wl.reset_every == 0:
                self._q[l] = eps  # abrupt query reset (topic shift)
            else:
                self._q[l] = self._rho_t * self._q[l] + self._sig_t * eps
            k, v = self._tokens(g, l, 1)
            k = k[:, :, 0].to(self.dtype)
            v = v[:, :, 0].to(self.dtype)
            if l in self._overflow:
                ok, ov, extra = self._overflow[l]
                i = self.t - 1
                if i < ok.shape[2]:   # prompt tokens past the buffer come first
                    use = (extra > i).view(-1, 1, 1)
                    k = torch.where(use, ok[:, :, i], k)
                    v = torch.where(use, ov[:, :, i], v)
            qs.append(self._q[l].to(self.dtype).contiguous())
            ks.append(k.contiguous())
            vs.append(v.contiguous())
        return qs, ks, vs
