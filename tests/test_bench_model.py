"""bench.py's algorithmic byte model against the per-unit formula, written out.

Per (layer, sequence) unit at steady state, with H_kv KV heads, H_q query
heads, B occupied slots, head dim d and e bytes per element: K and V of every
slot (2 H_kv B d e), each slot's cached norm and position (8 H_kv B), q read
and out written (2 H_q d e), the new token read and written into its slot
(4 H_kv d e), and per KV head the new norm, position and evicted index
(12 H_kv).  Fill steps write the token but pick no victim; eviction-off steps
read only.
"""
import bench
from synth.workloads import WORKLOADS


def _formula(hkv, hq, B, d, e, writes=True):
    b = 2 * hkv * B * d * e + 8 * hkv * B + 2 * hq * d * e + 2 * hkv * d * e + 4 * hkv
    if writes:
        b += 2 * hkv * d * e + 8 * hkv
    return b


def test_steady_unit_bytes_qwen3_8b():
    wl = WORKLOADS["qwen3-8b-steady"]
    assert bench.unit_bytes(wl, 3276) == 13_652_832
    assert bench.unit_bytes(wl, 3276) == _formula(8, 32, 3276, 128, 2)
    # one launch of the bench line: 64 sequences
    assert 64 * bench.unit_bytes(wl, 3276) == 873_781_248


def test_other_shapes_and_modes():
    for name in ("tiny-fp32", "qwen3-0.6b", "r1-llama-8b", "ragged-serving"):
        wl = WORKLOADS[name]
        e = wl.elem_bytes
        for n in (1, 17, wl.budget):
            assert bench.unit_bytes(wl, n) == _formula(wl.kv_heads, wl.q_heads, n, wl.head_dim, e)
            assert bench.unit_bytes(wl, n, writes_slot=False) == _formula(
                wl.kv_heads, wl.q_heads, n, wl.head_dim, e, writes=False)


def test_h2o_adds_the_accumulators():
    wl = WORKLOADS["qwen3-8b-steady"]
    extra = bench.unit_bytes(wl, 3276, h2o=True) - bench.unit_bytes(wl, 3276)
    # each slot's running sum is read in place of its norm and written back: 4 B per slot,
    # plus the new token's
    assert extra == 4 * 8 * 3276 + 4 * 8
