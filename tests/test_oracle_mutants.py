"""Plant plausible mistakes in a copy of the oracle (CPU only) and show that
the pins catch every one of them.

Each mutant is the oracle's own source with one textual edit, loaded as a
separate module; the real oracle is untouched.
"""
import importlib.util
import os
import sys
import types

import pytest

import oracle_pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "longflow_oracle.py")

MUTANTS = {
    "new_token_not_attended": (
        "keys = np.vstack([self.K[:n], np.asarray(k_new, np.float64)[None]])",
        "keys = np.vstack([self.K[:n], 0.0 * np.asarray(k_new, np.float64)[None]])"),
    "scale_1_over_d": ("return 1.0 / math.sqrt(self.d)", "return 1.0 / self.d"),
    "logit_sign": ("logits = (q @ keys.T) * scale", "logits = -(q @ keys.T) * scale"),
    "softmax_wrong_axis": ("alpha = w / w.sum(axis=1, keepdims=True)",
                           "alpha = w / w.sum(axis=0, keepdims=True)"),
    "gqa_interleaved": ("q[g * self.G:(g + 1) * self.G]", "q[g::len(self.units)]"),
    "score_without_vnorm": (
        "return np.asarray(alpha_cached, np.float64).sum(axis=0) * np.asarray(vnorm1, np.float64)",
        "return np.asarray(alpha_cached, np.float64).sum(axis=0)"),
    "score_max_over_heads": (
        "return np.asarray(alpha_cached, np.float64).sum(axis=0) *",
        "return np.asarray(alpha_cached, np.float64).max(axis=0) *"),
    "score_index_shift": ("longflow_scores(alpha[:, :n], self.vnorm[:n])",
                          "longflow_scores(alpha[:, 1:], self.vnorm[:n])"),
    "argmax_not_argmin": ('np.argsort(scores[cand], kind="stable")',
                          'np.argsort(-scores[cand], kind="stable")'),
    "ties_to_highest": ("cand = np.flatnonzero(np.asarray(pos) < next_pos - window)",
                        "cand = np.flatnonzero(np.asarray(pos) < next_pos - window)[::-1]"),
    "window_off_by_one": ("np.asarray(pos) < next_pos - window", "np.asarray(pos) <= next_pos - window"),
    "vnorm_l2": ("self.vnorm[slot] = np.abs(np.asarray(v, np.float64)).sum()",
                 "self.vnorm[slot] = np.sqrt((np.asarray(v, np.float64) ** 2).sum())"),
    "fill_wrong_slot": ("written = n            # initial fill: next free slot",
                        "written = (n + 1) % self.capacity"),
    "position_off_by_one": ("self._write(written, k_new, v_new, self.p)",
                            "self._write(written, k_new, v_new, self.p + 1)"),
    "no_write_on_evict": ("            written = evicted\n", "            written = -1\n"),
}


def _load_mutant(name, old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    src = src.replace(old, new)
    mod = types.ModuleType(f"oracle_mutant_{name}")
    mod.__dict__["__name__"] = mod.__name__
    sys.modules[mod.__name__] = mod     # dataclasses look the module up by name
    try:
        exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    except Exception:
        del sys.modules[mod.__name__]
        raise
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new)
    caught = []
    try:
        for check in oracle_pins.ALL_CHECKS:
            try:
                check(mod)
            except (AssertionError, ValueError, IndexError) as e:
                caught.append(check.__name__)
    finally:
        sys.modules.pop(mod.__name__, None)
    assert caught, f"no pin caught mutant {name}"
