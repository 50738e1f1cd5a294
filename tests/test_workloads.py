"""The seeded input streams follow the stated recipe (CPU only): reproducible
draws, the AR(1) query correlation, the per-token log-normal value scale, the
1% sink keys shared across KV heads, the ragged workload's per-sequence draws
and its abrupt query resets.  Tolerances are several standard errors of each
statistic at the sample sizes used."""
import math

import torch

from synth.workloads import WORKLOADS, InputStream


def _steps(stream, n):
    out = [stream.next_step() for _ in range(n)]
    return ([o[0][0].float() for o in out], [o[1][0].float() for o in out],
            [o[2][0].float() for o in out])


def test_streams_are_reproducible_and_per_layer():
    wl = WORKLOADS["r1-llama-8b"].scaled(batch=2, layers=4, prefill=16)
    a = InputStream(wl, seed=3, layers=[0, 2])
    b = InputStream(wl, seed=3, layers=[2])
    c = InputStream(wl, seed=4, layers=[2])
    assert torch.equal(a.prompt(2)[0], b.prompt(2)[0])
    for _ in range(3):
        qa, qb, qc = a.next_step()[0][1], b.next_step()[0][0], c.next_step()[0][0]
        assert torch.equal(qa, qb)          # layer 2 does not depend on layer 0 being drawn
        assert not torch.equal(qb, qc)      # another seed, another stream


def test_query_ar1_correlation_and_variance():
    wl = WORKLOADS["tiny-fp32"].scaled(batch=16, q_heads=8, kv_heads=1, head_dim=64)
    s = InputStream(wl, seed=1)
    qs, _, _ = _steps(s, 400)
    q = torch.stack(qs[100:])                       # past the start-up transient
    x, y = q[:-1].flatten(), q[1:].flatten()
    rho = float(((x - x.mean()) * (y - y.mean())).mean() / (x.std() * y.std()))
    assert abs(rho - 0.9) < 0.01, rho
    stationary = 0.44 ** 2 / (1 - 0.9 ** 2)        # ~1.02
    assert abs(float(q.var()) - stationary) < 0.08, float(q.var())


def test_value_lognormal_scale():
    wl = WORKLOADS["qwen3-0.6b"].scaled(batch=8, prefill=512)
    k, v, _ = InputStream(wl, seed=2, layers=[0]).prompt(0)
    v = v.float()
    # v = n * exp(0.5 z): E[v^2] = E[exp(z)] = e^{1/2}; one z per token, shared by its KV heads
    assert abs(float((v * v).mean()) - math.exp(0.5)) < 0.1
    per_token = (v * v).mean(dim=3)                 # [b][H_kv][n]
    logs = torch.log(per_token).mean(dim=1)         # the shared log-scale shows as a token effect
    assert float(logs.std()) > 0.7                  # 2 sigma = 1 on top of chi-square noise
    assert abs(float(k.float().var()) - 1.0) < 0.02


def test_sink_keys_one_percent_shared_across_heads():
    wl = WORKLOADS["r1-llama-8b"].scaled(batch=16, prefill=2048)
    s = InputStream(wl, seed=5, layers=[0])
    k, _, _ = s.prompt(0)
    u = s._sink_u[0]                                # [H_kv][d], unit vectors
    proj = torch.einsum("bhnd,hd->bhn", k.float(), u)
    shift = 3.0 * math.sqrt(wl.head_dim)            # ~34 against N(0,1) noise
    is_sink = proj > shift / 2
    frac = float(is_sink.float().mean())
    assert abs(frac - 0.01) < 0.003, frac
    # a token is a sink in every KV head or in none
    assert torch.equal(is_sink.all(dim=1), is_sink.any(dim=1))


def test_ragged_draws_and_query_resets():
    wl = WORKLOADS["ragged-serving"].scaled(q_heads=8, kv_heads=2, head_dim=32)
    s = InputStream(wl, seed=0, layers=[0])
    assert len(s.budgets) == wl.batch and set(s.budgets) <= {512, 1024, 2048, 3276}
    assert len(set(s.budgets)) == 4
    assert all(64 <= p <= 2048 for p in s.prompt_lens)
    assert all(0.6 <= r <= 0.98 for r in s.rhos)
    assert all(abs(i - math.sqrt(1 - r * r)) < 1e-12 for r, i in zip(s.rhos, s.innovations))
    prev = None
    corr = {}
    for t in range(1, 1003):
        q = s.next_step()[0][0].float()
        if prev is not None and t in (999, 1000, 1001):
            x, y = prev.flatten(), q.flatten()
            corr[t] = float(((x - x.mean()) * (y - y.mean())).mean() / (x.std() * y.std()))
        prev = q
    assert corr[999] > 0.6 and corr[1001] > 0.6      # AR(1) with rho in [0.6, 0.98]
    assert abs(corr[1000]) < 0.05                     # step 1000 draws a fresh query


def test_prompt_remainder_fed_as_decode_tokens():
    """A prompt longer than its sequence's buffer: the buffer takes its first
    tokens, the rest come out as that sequence's next decode tokens in prompt
    order (one per step, with the step's own query), then drawn tokens
    follow; other sequences and the queries see the same draws as without
    the cut."""
    wl = WORKLOADS["ragged-serving"].scaled(batch=6, layers=1, prompt_range=(40, 90))
    a = InputStream(wl, seed=5, layers=[0])
    b = InputStream(wl, seed=5, layers=[0])
    limits = [50, 100, 60, 10, 100, 45]
    k, v, cut = a.prompt_split(0, limits)
    kb, vb, lens = b.prompt(0)
    assert torch.equal(k, kb) and lens == a.prompt_lens
    assert cut == [min(P, m) for P, m in zip(lens, limits)]
    extra = [P - c for P, c in zip(lens, cut)]
    assert a.overflow_lengths(0) == extra and max(extra) > 0 and min(extra) == 0
    for t in range(max(extra) + 2):
        qa, ka, va = a.next_step()
        qb, kb_t, vb_t = b.next_step()
        assert torch.equal(qa[0], qb[0])
        for s in range(wl.batch):
            if t < extra[s]:   # the prompt's token at position cut + t
                assert torch.equal(ka[0][s], k[s, :, cut[s] + t])
                assert torch.equal(va[0][s], v[s, :, cut[s] + t])
            else:              # a drawn token, the same as without the cut
                assert torch.equal(ka[0][s], kb_t[0][s])
                assert torch.equal(va[0][s], vb_t[0][s])
