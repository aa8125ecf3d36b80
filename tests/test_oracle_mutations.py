"""The pins must be able to fail: plant plausible mistakes in a CPU copy of the
recurrence and check that at least one pin rejects each of them.

The planted copies live here, on the CPU; the oracle itself is untouched.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import chunkwise as cw
from oracle import recurrence

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def recur_py(q, k, v, g, beta, scale, S0, mutation=None):
    """Per-pair recurrence in NumPy with an optional planted mistake."""
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.zeros((q.shape[0], v.shape[1]))
    for t in range(q.shape[0]):
        a = np.exp(g[t]) if mutation != "gate_sign" else np.exp(-g[t])
        b = beta[t] if mutation != "beta_erase_dropped" else 1.0
        if mutation == "decay_after_readout":
            r = S.T @ k[t]
            S = a * S
        else:
            S = a * S
            r = S.T @ k[t]
        if mutation == "transposed_readout":
            r = S @ k[t]
        sign = -1.0 if mutation == "erase_sign" else 1.0
        S_prev = S.copy()
        S = S + np.outer(k[t], beta[t] * v[t] - sign * b * r)
        src = S_prev if mutation == "pre_update_output" else S
        o[t] = (1.0 if mutation == "scale_dropped" else scale) * (src.T @ q[t])
    return o, S


MUTATIONS = ["decay_after_readout", "gate_sign", "beta_erase_dropped", "transposed_readout",
             "erase_sign", "pre_update_output", "scale_dropped"]


def _pins_pass(impl):
    """Run a battery of the oracle pins on ``impl``; True iff all hold."""
    rng = np.random.default_rng(0)
    T, K, V = 70, 8, 8
    q = rng.standard_normal((T, K))
    k = rng.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, V))
    g = np.log(1 / (1 + np.exp(-(3 + rng.standard_normal(T)))))
    beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    S0 = 0.1 * rng.standard_normal((K, V))
    ok = True
    # (1) chunk forms of the pages
    o, S = impl(q, k, v, g, beta, 0.35, S0)
    for form in (cw.fla_form, cw.qla_form):
        o2, S2 = form(q, k, v, g, beta, 0.35, S0, 16)
        ok &= np.allclose(o, o2, atol=1e-10) and np.allclose(S, S2, atol=1e-10)
    # (2) hand-worked golden (scalar case)
    case = json.load(open(os.path.join(GOLDEN, "recurrence_cases.json")))["cases"][0]
    F = lambda x: np.array([[float(Fraction(s)) for s in r] for r in x]) if isinstance(x[0], list) \
        else np.array([float(Fraction(s)) for s in x])
    o, S = impl(F(case["q"]), F(case["k"]), F(case["v"]), np.log(F(case["alpha"])),
                F(case["beta"]), float(Fraction(case["scale"])), F(case["S0"]))
    ok &= np.allclose(o, F(case["o"]), atol=1e-13) and np.allclose(S, F(case["S_T"]), atol=1e-13)
    # (3) orthonormal retrieval
    kk = np.eye(K)[:6]
    vv = rng.standard_normal((6, V))
    o, S = impl(kk, kk, vv, np.zeros(6), np.ones(6), 0.5, np.zeros((K, V)))
    ok &= np.allclose(o, 0.5 * vv, atol=1e-13)
    return bool(ok)


def test_clean_copy_passes_and_matches_oracle():
    assert _pins_pass(lambda *a: recur_py(*a))
    rng = np.random.default_rng(1)
    T, K, V = 30, 8, 4
    x = [rng.standard_normal((T, K)), rng.standard_normal((T, K)), rng.standard_normal((T, V)),
         -rng.uniform(0, 0.2, T), rng.uniform(0, 1, T)]
    S0 = rng.standard_normal((K, V))
    o, S = recur_py(*x, 0.3, S0)
    o2, S2 = recurrence(x[0][None, :, None], x[1][None, :, None], x[2][None, :, None],
                        x[3][None, :, None], x[4][None, :, None], 0.3, S0[None, None])
    assert np.allclose(o, o2[0, :, 0], atol=1e-12) and np.allclose(S, S2[0, 0], atol=1e-12)


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_planted_mistake_is_caught(mutation):
    assert not _pins_pass(lambda *a: recur_py(*a, mutation=mutation))
