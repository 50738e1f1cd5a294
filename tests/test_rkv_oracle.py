"""The R-KV oracle against its pins, and planted mistakes in copies of it (CPU only)."""
import os
import sys
import types

import pytest

from oracle import rkv_oracle
import rkv_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "rkv_oracle.py")

MUTANTS = {
    "importance_mean_over_candidates": ("return w.mean(axis=0)", "return w.mean(axis=1).repeat(w.shape[1])[:w.shape[1]]"),
    "importance_softmax_wrong_axis": ("w /= w.sum(axis=1, keepdims=True)", "w /= w.sum(axis=0, keepdims=True)"),
    "cosine_unnormalised": ("cos = (k @ k.T) / np.outer(norms, norms)", "cos = (k @ k.T)"),
    "older_not_newer": ("newer = pos[None, :] > pos[:, None]", "newer = pos[None, :] < pos[:, None]"),
    "beta_strict": ("return (near.sum(axis=1) >= beta)", "return (near.sum(axis=1) > beta)"),
    "tau_strict": ("near = (cos >= tau) & newer", "near = (cos > tau + 0.05) & newer"),
    "lambda_swapped": ("z = prm.lam * imp - (1.0 - prm.lam) * red", "z = (1.0 - prm.lam) * imp - prm.lam * red"),
    "ties_to_older": ("rest.sort(key=lambda i: (-z[i], -pos[i]))", "rest.sort(key=lambda i: (-z[i], pos[i]))"),
    "no_observation_tokens": ("obs = set(by_recency[:alpha].tolist())", "obs = set()"),
    "moves_reversed": ("moves = list(zip(movers, freed))", "moves = list(zip(movers, freed[::-1]))"),
    "new_token_not_attended": ("keys = np.vstack([self.K[:n], np.asarray(k_new, np.float64)[None]])",
                               "keys = np.vstack([self.K[:n], 0 * np.asarray(k_new, np.float64)[None]])"),
}


@pytest.mark.parametrize("check", rkv_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_rkv_pin(check):
    check(rkv_oracle)


def _mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mod = types.ModuleType(f"rkv_mutant_{name}")
    sys.modules[mod.__name__] = mod
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_rkv_pins_catch_mutant(name):
    mod = _mutant(name, *MUTANTS[name])
    caught = []
    try:
        for check in rkv_pins.ALL_CHECKS:
            try:
                check(mod)
            except (AssertionError, ValueError, IndexError, KeyError):
                caught.append(check.__name__)
    finally:
        sys.modules.pop(mod.__name__, None)
    assert caught, f"no pin caught mutant {name}"
