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
        "keys = np.vstack([u.K[:n], np.asarray(kn, np.float64)[None]])",
        "keys = np.vstack([u.K[:n], 0.0 * np.asarray(kn, np.float64)[None]])"),
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
    "score_index_shift": ("u.slot_scores(a[:, :n], n)", "u.slot_scores(a[:, 1:], n)"),
    "argmax_not_argmin": ('np.argsort(scores[cand], kind="stable")',
                          'np.argsort(-scores[cand], kind="stable")'),
    "ties_to_highest": ("cand = np.flatnonzero((pos < next_pos - window) & (pos >= sinks))",
                        "cand = np.flatnonzero((pos < next_pos - window) & (pos >= sinks))[::-1]"),
    "window_off_by_one": ("(pos < next_pos - window)", "(pos <= next_pos - window)"),
    "vnorm_l2": ("self.vnorm[slot] = value_norm(v, self.policy.norm)",
                 "self.vnorm[slot] = value_norm(v, 2)"),
    "fill_wrong_slot": ("written = n            # initial fill: next free slot",
                        "written = (n + 1) % u0.capacity"),
    "position_off_by_one": ("u._write(written, kn, vn, p)", "u._write(written, kn, vn, p + 1)"),
    "no_write_on_evict": ("        written = evicted\n", "        written = -1\n"),
    "budget_ignored": ("if u0.evict and n >= u0.budget:", "if u0.evict and n >= u0.capacity:"),
    "limit_is_capacity": ("return self.budget if self.evict else self.capacity",
                          "return self.capacity"),
    "deferred_budget_ignored": ("    if n < u0.budget:\n", "    if n < u0.capacity:\n"),
    # policy variants
    "sinks_ignored": ("& (pos >= sinks)", "& (pos >= 0)"),
    "sinks_off_by_one": ("& (pos >= sinks)", "& (pos > sinks)"),
    "l2_without_sqrt": ("return float(math.sqrt((v * v).sum()))", "return float((v * v).sum())"),
    "l2_is_l1": ("if norm == 1:", "if norm in (1, 2):"),
    "deferred_window_excludes_new": ("p + 1, u0.window,", "p, u0.window,"),
    "deferred_attends_before_write": (
        "        u._write(written, kn, vn, p)\n        u.n = n_after\n",
        "        u.n = n_after\n"),
    "deferred_choice_not_carried": ("        u.pending = chosen\n", "        u.pending = -1 if chosen < 0 else 0\n"),
    "layer_scope_first_head_only": (
        "scores = sum(u.slot_scores(a[:, :n], n) for u, a in zip(units, alphas))",
        "scores = units[0].slot_scores(alphas[0][:, :n], n)"),
    "layer_scope_is_per_head": ('if self.policy.scope == "layer":', "if False:"),
    "h2o_no_self_weight": ("u.acc[written] = a[:, n].sum()   # the new token's own weight",
                           "u.acc[written] = 0.0"),
    "h2o_not_accumulated": ("u.acc[:n] += alpha[:, :n].sum(axis=0)",
                            "u.acc[:n] = alpha[:, :n].sum(axis=0)"),
    "h2o_scores_are_longflow": ('if self.policy.score == "h2o":\n            return',
                                'if False:\n            return'),
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
            except (AssertionError, ValueError, IndexError, KeyError):
                caught.append(check.__name__)
    finally:
        sys.modules.pop(mod.__name__, None)
    assert caught, f"no pin caught mutant {name}"
