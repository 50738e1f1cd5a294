"""R-KV's compression step on the GPU against the fp64 R-KV oracle (rules in
gpu_rkv_harness.py).  Source: "GitHub - Zefan-Cai/R-KV", section "Method"."""
import pytest

from gpu_rkv_harness import RKVRun
from synth.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


def _small(**over):
    base = dict(layers=1, batch=2, q_heads=8, kv_heads=2, budget=300, prefill=300,
                rkv_buffer=64, dup_prob=0.2)
    base.update(over)
    return WORKLOADS["rkv-r1-llama-8b"].scaled(**base)


@pytest.mark.parametrize("case", [
    ("g4_two_compressions", dict()),
    ("g1_ragged_tail", dict(q_heads=2, kv_heads=2, budget=201, prefill=150, rkv_buffer=37)),
    ("g8_alpha8", dict(q_heads=16, kv_heads=2, budget=250, prefill=260, rkv_buffer=50)),
    ("g2_beta2_tau085", dict(q_heads=4, kv_heads=2, rkv_beta=2, rkv_tau=0.85)),
], ids=lambda c: c[0])
def test_rkv_small(case):
    name, over = case
    wl = _small(**over)
    run = RKVRun(wl)
    try:
        first = (wl.budget + wl.rkv_buffer) - min(wl.prefill, wl.budget + wl.rkv_buffer)
        run.run(first + 2 * wl.rkv_buffer + 3)   # fill the buffer, then two more cycles
        assert run.compressions >= 2
        assert run.redundant > 0 or name == "g1_ragged_tail"
    finally:
        run.close()


def test_rkv_full_size():
    """The rkv-r1-llama-8b launch shape (batch 32, 8 KV heads, budget 3276 +
    buffer 128, 3404 tokens per compression) on sampled units."""
    wl = WORKLOADS["rkv-r1-llama-8b"].scaled(layers=1)
    run = RKVRun(wl, sample=[(0, 0), (31, 7), (17, 3)])
    try:
        run.run(4 * wl.rkv_buffer + 2)
        assert run.compressions == 4
        assert run.redundant > 0
    finally:
        run.close()
