"""Pins of the gradient oracle (oracle.recurrence_backward), independent of it.

* Adjoint (dot-product) identities, exact up to rounding: o is linear in q (the states do not
  depend on q), and (o, ht) is jointly linear in (v, h0).  So for any direction X,
  <forward(X), (do, dht)> = <X, gradient>, with the forward oracle on the left.
* Central finite differences of the forward oracle for every input, along random directions and
  for single entries, across a checkpoint block boundary (T = 70 > 64), packed sequences, GVA and
  both gate kinds.
* The beta = 0 closed form: the state only decays, S_t = exp(G_t) h0, so o_t = scale exp(G_t) h0^T q_t
  and every gradient is a short sum written out here by hand.
"""
import numpy as np
import pytest

from oracle import recurrence, recurrence_backward

pytestmark = pytest.mark.filterwarnings("ignore")


def _inputs(seed, B=2, T=70, H=1, HV=2, K=4, V=5, gate="scalar", varlen=None, beta_zero=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, HV, V))
    gshape = (B, T, HV) if gate == "scalar" else (B, T, HV, K)
    g = -np.abs(rng.standard_normal(gshape)) * 0.3
    beta = np.zeros((B, T, HV)) if beta_zero else rng.uniform(0.1, 0.9, (B, T, HV))
    cu = None
    if varlen is not None:
        cu = np.asarray(varlen, dtype=np.int64)
    N = B if cu is None else len(cu) - 1
    h0 = rng.standard_normal((N, HV, K, V)) * 0.5
    do = rng.standard_normal((B, T, HV, V))
    dht = rng.standard_normal((N, HV, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, do=do, dht=dht, cu=cu, gate=gate, scale=K ** -0.5)


def _loss(x, **over):
    y = dict(x)
    y.update(over)
    o, ht = recurrence(y["q"], y["k"], y["v"], y["g"], y["beta"], y["scale"], y["h0"], y["cu"], gate=y["gate"])
    return float((o * x["do"]).sum() + (ht * x["dht"]).sum())


def _grads(x):
    return recurrence_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["do"], x["h0"],
                               x["dht"], x["cu"], gate=x["gate"])


CASES = [
    dict(gate="scalar"),
    dict(gate="channel"),
    dict(gate="scalar", B=1, T=75, varlen=[0, 5, 70, 70, 75]),  # packed, with an empty sequence
    dict(gate="channel", B=1, T=75, varlen=[0, 66, 75], H=2, HV=4),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_adjoint_identities_for_the_linear_inputs(case):
    x = _inputs(10 + case, **CASES[case])
    dq, dk, dv, dbeta, dg, dh0 = _grads(x)
    rng = np.random.default_rng(99)
    # o is linear in q: <o(Q'), do> (h0, dht terms are independent of q: zero them)
    Qp = rng.standard_normal(x["q"].shape)
    o, _ = recurrence(Qp, x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["cu"], gate=x["gate"])
    lhs = (o * x["do"]).sum()
    assert abs(lhs - (Qp * dq).sum()) <= 1e-10 * (1 + abs(lhs))
    # (o, ht) is linear in (v, h0)
    Vp, Hp = rng.standard_normal(x["v"].shape), rng.standard_normal(x["h0"].shape)
    o, ht = recurrence(x["q"], x["k"], Vp, x["g"], x["beta"], x["scale"], Hp, x["cu"], gate=x["gate"])
    lhs = (o * x["do"]).sum() + (ht * x["dht"]).sum()
    assert abs(lhs - (Vp * dv).sum() - (Hp * dh0).sum()) <= 1e-10 * (1 + abs(lhs))


@pytest.mark.parametrize("case", range(len(CASES)))
def test_finite_differences_along_random_directions(case):
    x = _inputs(20 + case, **CASES[case])
    grads = dict(zip(["q", "k", "v", "beta", "g", "h0"], _grads(x)))
    rng = np.random.default_rng(7)
    eps = 1e-5
    for name in ["q", "k", "v", "beta", "g", "h0"]:
        for _ in range(2):
            u = rng.standard_normal(x[name].shape)
            fd = (_loss(x, **{name: x[name] + eps * u}) - _loss(x, **{name: x[name] - eps * u})) / (2 * eps)
            an = float((grads[name] * u).sum())
            assert abs(fd - an) <= 1e-6 * (1 + abs(fd)), (name, fd, an)


def test_finite_differences_single_entries():
    x = _inputs(31, gate="scalar", B=1, T=70, H=1, HV=1)
    grads = dict(zip(["q", "k", "v", "beta", "g", "h0"], _grads(x)))
    eps = 1e-6
    for name, idx in [("k", (0, 3, 0, 1)), ("k", (0, 66, 0, 2)), ("beta", (0, 0, 0)), ("beta", (0, 64, 0)),
                      ("g", (0, 0, 0)), ("g", (0, 63, 0)), ("g", (0, 69, 0)), ("q", (0, 10, 0, 3)),
                      ("v", (0, 65, 0, 4)), ("h0", (0, 0, 2, 1))]:
        d = np.zeros_like(x[name])
        d[idx] = 1.0
        fd = (_loss(x, **{name: x[name] + eps * d}) - _loss(x, **{name: x[name] - eps * d})) / (2 * eps)
        assert abs(fd - grads[name][idx]) <= 1e-6 * (1 + abs(fd)), (name, idx, fd, grads[name][idx])


def test_beta_zero_closed_form():
    """beta = 0: S_t = exp(G_t) h0 with G_t the inclusive sum of g over the sequence, so
    o_t = scale exp(G_t) h0^T q_t and ht = exp(G_T) h0.  By hand:
      dq_t = scale exp(G_t) h0 do_t,  dv = 0,
      dh0 = sum_t scale exp(G_t) q_t do_t^T + exp(G_T) dht,
      dg_s = sum_{t >= s} scale exp(G_t) q_t^T h0 do_t + exp(G_T) <dht, h0>,
      dk_t = dS_t (beta d_t) + ... = 0 (every term carries beta_t or d_t = 0), and
      dbeta_t = k_t^T dS_t (v_t - exp(G_t) h0^T k_t) with dS_t = sum_{t' >= t} scale exp(G_t' - G_t)
                q_t' do_t'^T + exp(G_T - G_t) dht (the gradient reaching S_t)."""
    x = _inputs(41, gate="scalar", B=1, T=70, H=1, HV=1, beta_zero=True)
    dq, dk, dv, dbeta, dg, dh0 = _grads(x)
    q, k, v, g, do, h0, dht, sc = (x["q"][0, :, 0], x["k"][0, :, 0], x["v"][0, :, 0], x["g"][0, :, 0],
                                   x["do"][0, :, 0], x["h0"][0, 0], x["dht"][0, 0], x["scale"])
    T = q.shape[0]
    G = np.cumsum(g)
    e_dq = np.stack([sc * np.exp(G[t]) * h0 @ do[t] for t in range(T)])
    e_dh0 = sum(sc * np.exp(G[t]) * np.outer(q[t], do[t]) for t in range(T)) + np.exp(G[-1]) * dht
    c = np.array([sc * np.exp(G[t]) * q[t] @ h0 @ do[t] for t in range(T)])
    e_dg = np.array([c[s:].sum() for s in range(T)]) + np.exp(G[-1]) * (dht * h0).sum()
    e_db = np.zeros(T)
    for t in range(T):
        dS = sum(sc * np.exp(G[u] - G[t]) * np.outer(q[u], do[u]) for u in range(t, T)) + np.exp(G[-1] - G[t]) * dht
        e_db[t] = k[t] @ dS @ (v[t] - np.exp(G[t]) * h0.T @ k[t])
    np.testing.assert_allclose(dq[0, :, 0], e_dq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dh0[0, 0], e_dh0, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg[0, :, 0], e_dg, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dbeta[0, :, 0], e_db, rtol=1e-10, atol=1e-12)
    assert np.abs(dk).max() == 0.0 and np.abs(dv).max() == 0.0


def test_planted_mistake_is_caught():
    """A sign error in dg (a plausible slip: dg = -<dSb, Sb>) fails the finite-difference pin."""
    x = _inputs(51, gate="scalar", B=1, T=20, H=1, HV=1)
    dg = _grads(x)[4]
    rng = np.random.default_rng(3)
    u = rng.standard_normal(x["g"].shape)
    eps = 1e-5
    fd = (_loss(x, g=x["g"] + eps * u) - _loss(x, g=x["g"] - eps * u)) / (2 * eps)
    assert abs(fd - float((dg * u).sum())) <= 1e-6 * (1 + abs(fd))
    assert abs(fd - float((-dg * u).sum())) > 1e-3 * (1 + abs(fd))
