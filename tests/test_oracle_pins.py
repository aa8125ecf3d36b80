"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with a retyped copy of itself: each test
uses an independent formulation (the chunk forms the pages give, evaluated
naively), a closed form of a special case, an invariant, a hand-worked
fixture, or exact rational brute force.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from gdn_inputs import Workload, make_inputs, to_f64
from oracle import recurrence
from oracle import chunkwise as cw
from oracle.exact import exact_recurrence

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_case(seed, B=2, T=150, H=2, HV=None, K=16, V=8, gate="scalar", h0=True,
               varlen=0, g_mu=3.0, g_sigma=1.0):
    w = Workload("small", B=B, T=T, H=H, HV=HV, K=K, V=V, dtype="f32", gate=gate, h0=h0,
                 varlen=varlen, seed=seed, g_mu=g_mu, g_sigma=g_sigma)
    x = make_inputs(w)
    return {key: (to_f64(val) if hasattr(val, "dtype") and key != "cu_seqlens" else val)
            for key, val in x.items()}


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def run_oracle(x, **kw):
    return recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"],
                      x["cu_seqlens"], gate=x["gate"], **kw)


# ---------------------------------------------------------------- P-chunk
@pytest.mark.parametrize("C", [1, 2, 4, 8, 16, 64])
@pytest.mark.parametrize("form", ["fla", "qla"])
def test_chunk_forms_match_recurrence(C, form):
    x = small_case(seed=11 + C)
    o, ht = run_oracle(x)
    f = cw.fla_form if form == "fla" else cw.qla_form
    o2, ht2 = cw.run_pairs(f, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], C=C)
    assert rel(o2, o) < 1e-10 and rel(ht2, ht) < 1e-10


@pytest.mark.parametrize("C", [1, 16, 64])
def test_channel_form_matches_recurrence(C):
    x = small_case(seed=21 + C, gate="channel")
    o, ht = run_oracle(x)
    o2, ht2 = cw.run_pairs(cw.channel_form, x["q"], x["k"], x["v"], x["g"], x["beta"],
                           x["scale"], x["h0"], C=C)
    assert rel(o2, o) < 1e-10 and rel(ht2, ht) < 1e-10


def test_gva_head_mapping():
    # HV = 2H: value heads 2j and 2j+1 read query/key head j.
    x = small_case(seed=5, H=2, HV=4, T=70)
    o, ht = run_oracle(x)
    o2, ht2 = cw.run_pairs(cw.qla_form, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                           x["h0"], C=64)
    assert rel(o2, o) < 1e-10 and rel(ht2, ht) < 1e-10
    # and it equals running each value head against an explicitly repeated q/k
    q = np.repeat(x["q"], 2, axis=2)
    k = np.repeat(x["k"], 2, axis=2)
    o3, ht3 = recurrence(q, k, x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    assert rel(o3, o) < 1e-14 and rel(ht3, ht) < 1e-14


# ---------------------------------------------------------------- P-beta0 / GLA reductions
def _gla_closed_form(q, k, v, g, beta, scale, h0):
    """Gated linear attention, per pair: o = scale [(Q K^T * D) diag(beta) V + diag(e^G) Q h0],
    D_ij = exp(G_i - G_j) for j <= i, G the global inclusive cumsum."""
    G = np.cumsum(g)
    D = np.tril(np.exp(G[:, None] - G[None, :]))
    return scale * ((q @ k.T * D) @ (beta[:, None] * v) + np.exp(G)[:, None] * (q @ h0))


def test_beta_zero_only_decays_h0():
    x = small_case(seed=31, B=1, H=1)
    x["beta"][:] = 0.0
    o, ht = run_oracle(x)
    G = np.cumsum(x["g"][0, :, 0])
    h0 = x["h0"][0, 0]
    exp_o = x["scale"] * np.exp(G)[:, None] * (x["q"][0, :, 0] @ h0)
    assert rel(o[0, :, 0], exp_o) < 1e-12
    assert rel(ht[0, 0], math.exp(G[-1]) * h0) < 1e-12


def test_small_beta_limit_is_gated_linear_attention():
    # First order in beta the erase term vanishes: o(eps b)/eps -> GLA with values b*v.
    x = small_case(seed=32, B=1, H=1, T=40)
    eps = 1e-7
    b = x["beta"].copy()
    x["beta"] = eps * b
    x["h0"] = np.zeros_like(x["h0"])
    o, _ = run_oracle(x)
    gla = _gla_closed_form(x["q"][0, :, 0], x["k"][0, :, 0], x["v"][0, :, 0], x["g"][0, :, 0],
                           b[0, :, 0], x["scale"], np.zeros((16, 8)))
    assert rel(o[0, :, 0] / eps, gla) < 1e-5


def test_orthogonal_keys_give_gated_linear_attention_exactly():
    rng = np.random.default_rng(7)
    T, K, V = 12, 16, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm[:T]                               # orthonormal rows
    q = rng.standard_normal((T, K))
    v = rng.standard_normal((T, V))
    g = -rng.uniform(0.0, 0.5, T)
    beta = rng.uniform(0.1, 1.0, T)
    o, ht = recurrence(q[None, :, None], k[None, :, None], v[None, :, None], g[None, :, None],
                       beta[None, :, None], 0.5)
    assert rel(o[0, :, 0], _gla_closed_form(q, k, v, g, beta, 0.5, np.zeros((K, V)))) < 1e-12


# ---------------------------------------------------------------- delta-rule retrieval
def test_orthonormal_retrieval():
    rng = np.random.default_rng(3)
    T, K, V = 10, 16, 6
    perm = rng.permutation(K)[:T]
    k = np.zeros((T, K))
    k[np.arange(T), perm] = 1.0
    v = rng.standard_normal((T, V))
    src = np.array([rng.integers(0, t + 1) for t in range(T)])
    q = k[src]
    g = np.zeros(T)
    beta = np.ones(T)
    o, ht = recurrence(q[None, :, None], k[None, :, None], v[None, :, None], g[None, :, None],
                       beta[None, :, None], 0.25)
    assert np.allclose(o[0, :, 0], 0.25 * v[src], atol=1e-14, rtol=0)
    assert np.allclose(ht[0, 0], k.T @ v, atol=1e-14, rtol=0)


def test_same_key_overwrites():
    rng = np.random.default_rng(4)
    K, V = 8, 4
    kk = rng.standard_normal(K)
    kk /= np.linalg.norm(kk)
    k = np.stack([kk, kk])
    v = rng.standard_normal((2, V))
    q = np.stack([kk, kk])
    o, ht = recurrence(q[None, :, None], k[None, :, None], v[None, :, None], np.zeros((1, 2, 1)),
                       np.ones((1, 2, 1)), 1.0)
    assert np.allclose(o[0, 1, 0], v[1], atol=1e-13)
    assert np.allclose(ht[0, 0], np.outer(kk, v[1]), atol=1e-13)


def test_householder_preserves_state_norm():
    rng = np.random.default_rng(5)
    T, K, V = 50, 16, 8
    k = rng.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    h0 = rng.standard_normal((1, 1, K, V))
    o, ht = recurrence(rng.standard_normal((1, T, 1, K)), k[None, :, None],
                       np.zeros((1, T, 1, V)), np.zeros((1, T, 1)), 2.0 * np.ones((1, T, 1)),
                       1.0, h0)
    assert abs(np.linalg.norm(ht) - np.linalg.norm(h0)) < 1e-12 * np.linalg.norm(h0)


# ---------------------------------------------------------------- exact brute force + golden
def _frac_case(rng, T, dk, dv, channel):
    def r(den=8, lo=-8, hi=8):
        return Fraction(int(rng.integers(lo, hi + 1)), den)
    q = [[r() for _ in range(dk)] for _ in range(T)]
    k = [[r(4, -4, 4) for _ in range(dk)] for _ in range(T)]
    v = [[r() for _ in range(dv)] for _ in range(T)]
    if channel:
        alpha = [[Fraction(int(rng.integers(1, 9)), 8) for _ in range(dk)] for _ in range(T)]
    else:
        alpha = [Fraction(int(rng.integers(1, 9)), 8) for _ in range(T)]
    beta = [Fraction(int(rng.integers(0, 9)), 8) for _ in range(T)]
    S0 = [[r(4) for _ in range(dv)] for _ in range(dk)]
    return q, k, v, alpha, beta, S0


@pytest.mark.parametrize("channel", [False, True])
@pytest.mark.parametrize("seed", range(4))
def test_exact_rational_bruteforce(seed, channel):
    rng = np.random.default_rng(100 + seed)
    T, dk, dv = int(rng.integers(1, 9)), int(rng.integers(1, 5)), int(rng.integers(1, 5))
    q, k, v, alpha, beta, S0 = _frac_case(rng, T, dk, dv, channel)
    scale = Fraction(1, 2)
    eo, eS = exact_recurrence(q, k, v, alpha, beta, scale, S0)
    f = lambda a: np.array(a, dtype=np.float64)
    g = np.log(f(alpha))
    o, ht = recurrence(f(q)[None, :, None], f(k)[None, :, None], f(v)[None, :, None],
                       g[None, :, None], f(beta)[None, :, None], 0.5, f(S0)[None, None],
                       gate="channel" if channel else "scalar")
    tol = 1e-13 * max(1.0, float(np.max(np.abs(f(eo)))))
    assert np.max(np.abs(o[0, :, 0] - f(eo))) < tol
    assert np.max(np.abs(ht[0, 0] - f(eS))) < 1e-13 * max(1.0, float(np.max(np.abs(f(eS)))))


def test_golden_hand_worked_cases():
    with open(os.path.join(GOLDEN, "recurrence_cases.json")) as fh:
        cases = json.load(fh)["cases"]
    F = lambda x: [[Fraction(s) for s in row] for row in x] if isinstance(x[0], list) else [Fraction(s) for s in x]
    for c in cases:
        q, k, v, S0 = F(c["q"]), F(c["k"]), F(c["v"]), F(c["S0"])
        alpha, beta, scale = F(c["alpha"]), F(c["beta"]), Fraction(c["scale"])
        eo, eS = exact_recurrence(q, k, v, alpha, beta, scale, S0)
        assert eo == F(c["o"]) and eS == F(c["S_T"]), c["name"]
        f = lambda a: np.array(a, dtype=np.float64)
        o, ht = recurrence(f(q)[None, :, None], f(k)[None, :, None], f(v)[None, :, None],
                           np.log(f(alpha))[None, :, None], f(beta)[None, :, None],
                           float(scale), f(S0)[None, None], gate=c["gate"])
        assert np.max(np.abs(o[0, :, 0] - f(F(c["o"])))) < 1e-14, c["name"]
        assert np.max(np.abs(ht[0, 0] - f(F(c["S_T"])))) < 1e-14, c["name"]


def test_one_token_scalar_by_hand():
    # dk = dv = 1: S1 = alpha (1 - beta k^2) S0 + beta k v = 1.5,  o = scale S1 q = 0.5*1.5*5.
    alpha, beta, k, v, S0, q, scale = 0.5, 0.25, 2.0, 3.0, 4.0, 5.0, 0.5
    S1 = alpha * (1 - beta * k * k) * S0 + beta * k * v          # = 0.5*0*4 + 1.5 = 1.5
    o, ht = recurrence(np.full((1, 1, 1, 1), q), np.full((1, 1, 1, 1), k), np.full((1, 1, 1, 1), v),
                       np.full((1, 1, 1), math.log(alpha)), np.full((1, 1, 1), beta), scale,
                       np.full((1, 1, 1, 1), S0))
    assert S1 == 1.5
    assert abs(ht[0, 0, 0, 0] - 1.5) < 1e-15 and abs(o[0, 0, 0, 0] - 3.75) < 1e-15


# ---------------------------------------------------------------- structure: linearity, continuation, varlen
def test_linear_in_values_and_initial_state():
    x = small_case(seed=41)
    x2 = dict(x)
    rng = np.random.default_rng(1)
    v2, h2 = rng.standard_normal(x["v"].shape), rng.standard_normal(x["h0"].shape)
    a, b = 0.7, -1.3
    o1, s1 = run_oracle(x)
    x2["v"], x2["h0"] = v2, h2
    o2, s2 = run_oracle(x2)
    x3 = dict(x)
    x3["v"], x3["h0"] = a * x["v"] + b * v2, a * x["h0"] + b * h2
    o3, s3 = run_oracle(x3)
    assert rel(o3, a * o1 + b * o2) < 1e-12 and rel(s3, a * s1 + b * s2) < 1e-12


def test_continuation_from_final_state():
    x = small_case(seed=42, T=200)
    o, ht = run_oracle(x)
    T1 = 77
    xa = {kk: (vv[:, :T1] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in x.items()}
    oa, sa = run_oracle(xa)
    xb = {kk: (vv[:, T1:] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in x.items()}
    xb["h0"] = sa
    ob, sb = run_oracle(xb)
    assert rel(np.concatenate([oa, ob], axis=1), o) < 1e-12 and rel(sb, ht) < 1e-12


def test_varlen_equals_independent_runs():
    x = small_case(seed=43, varlen=5, T=90)
    o, ht = run_oracle(x)
    cu = x["cu_seqlens"].numpy()
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        on, hn = recurrence(x["q"][:, s:e], x["k"][:, s:e], x["v"][:, s:e], x["g"][:, s:e],
                            x["beta"][:, s:e], x["scale"], x["h0"][n:n + 1])
        assert rel(on, o[:, s:e]) < 1e-14 and rel(hn[0], ht[n]) < 1e-14


def test_channel_gate_with_equal_channels_equals_scalar():
    x = small_case(seed=44)
    o, ht = run_oracle(x)
    xc = dict(x)
    xc["g"] = np.repeat(x["g"][..., None], x["q"].shape[-1], axis=-1)
    xc["gate"] = "channel"
    oc, hc = run_oracle(xc)
    assert rel(oc, o) < 1e-13 and rel(hc, ht) < 1e-13


def test_thread_count_does_not_change_result():
    x = small_case(seed=45, B=3, H=2)
    o1, s1 = run_oracle(x, nthreads=1)
    o4, s4 = run_oracle(x, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)


# ---------------------------------------------------------------- triangular inverse
@pytest.mark.parametrize("n", [16, 37, 64])
def test_blocked_inverse(n):
    rng = np.random.default_rng(n)
    k = rng.standard_normal((n, 32))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    beta = rng.uniform(0, 1, n)
    Lm = np.tril(beta[:, None] * (k @ k.T), -1)
    Ainv = cw.blocked_inverse(Lm)
    assert np.max(np.abs((np.eye(n) + Lm) @ Ainv - np.eye(n))) < 1e-12
    assert np.max(np.abs(Ainv - np.linalg.inv(np.eye(n) + Lm))) < 1e-12
    assert np.max(np.abs(cw.forward_substitution(Lm) - Ainv)) < 1e-12
    assert np.allclose(np.tril(Ainv), Ainv) and np.allclose(np.diag(Ainv), 1.0)


# ---------------------------------------------------------------- chunk-parallel split
@pytest.mark.parametrize("seg", [1, 2, 3])
def test_cp_exact_forms_match_serial(seg):
    x = small_case(seed=51, B=1, H=1, T=300, K=16, V=8, g_mu=5.0)
    o, ht = run_oracle(x)
    for f in (cw.cp_exact_deltanet, cw.cp_exact_qla):
        o2, ht2 = cw.run_pairs(f, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"],
                               C=16, seg_chunks=seg)
        assert rel(o2, o) < 1e-10 and rel(ht2, ht) < 1e-10


def test_cp_warmup_error_within_bound():
    x = small_case(seed=52, B=1, H=1, T=640, K=16, V=8, g_mu=3.0)
    o, ht = run_oracle(x)
    log_eps = math.log(2.0 ** -24)
    o2, ht2 = cw.run_pairs(cw.cp_warmup, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                           x["h0"], C=16, seg_chunks=8, log_eps=log_eps)
    # the dropped start state is attenuated by at least eps; outputs inherit that bound
    assert rel(ht2, ht) < 1e-6
    assert rel(o2, o) < 1e-6
    # a weaker threshold gives a visibly larger (but still bounded) error
    o3, _ = cw.run_pairs(cw.cp_warmup, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                         x["h0"], C=16, seg_chunks=8, log_eps=math.log(1e-2))
    assert rel(o3, o) < 1e-1


def test_warmup_start_walk():
    sums = [-1.0, -2.0, -0.5, -4.0, -0.1]
    # walking back from chunk 5: -0.1, -4.1, -4.6, -6.6, -7.6
    assert cw.warmup_start(sums, 5, -6.5) == 1
    assert cw.warmup_start(sums, 5, -4.0) == 3
    assert cw.warmup_start(sums, 2, -100.0) == 0


def test_transition_norm_is_bounded_by_the_slowest_channel():
    """||(I - beta k k^T) Diag(alpha)||_2 <= max_d alpha_d for ||k|| = 1, beta in [0, 2] (the
    inequality behind the warmup split's gate statistics), checked by SVD, beta = 0 and 2 included;
    with beta = 0 it is attained."""
    rng = np.random.default_rng(61)
    for trial in range(200):
        K = int(rng.integers(2, 17))
        kv = rng.standard_normal(K)
        kv /= np.linalg.norm(kv)
        beta = [0.0, 2.0, float(rng.uniform(0, 2))][trial % 3]
        alpha = rng.uniform(0.0, 1.0, K)
        A = (np.eye(K) - beta * np.outer(kv, kv)) @ np.diag(alpha)
        nrm = np.linalg.norm(A, 2)
        assert nrm <= alpha.max() * (1 + 1e-12)
        if beta == 0.0:
            assert abs(nrm - alpha.max()) <= 1e-12


def test_per_channel_products_are_not_a_decay_bound():
    """Two channels that take turns decaying, and a reflection (beta = 2, k = (e0 - e1)/sqrt 2) that swaps
    them every token: every channel's own product decays by 0.1 every other token, yet the state keeps
    its norm, since it always sits in the channel that does not decay.  chunk_decay_bounds (per token the
    slowest channel) gives no decay here, as it must."""
    T = 16
    kv = np.array([1.0, -1.0]) / np.sqrt(2.0)
    P = np.eye(2) - 2.0 * np.outer(kv, kv)
    assert np.allclose(P, [[0.0, 1.0], [1.0, 0.0]])
    g = np.log(np.array([[1.0, 0.1] if t % 2 == 0 else [0.1, 1.0] for t in range(T)]))
    S = np.array([1.0, 0.0])
    for t in range(T):
        S = P @ (np.exp(g[t]) * S)
    assert abs(np.linalg.norm(S) - 1.0) < 1e-12
    per_channel = g.sum(axis=0)
    assert per_channel.max() < -18.0  # each channel alone would claim a decay of 1e-8
    assert cw.chunk_decay_bounds(g, C=T) == [0.0]


def test_chunk_decay_bounds_scalar_is_the_gate_sum():
    g = np.array([-0.5, -1.0, -0.25, -2.0, -0.125])
    assert cw.chunk_decay_bounds(g, C=2) == [-1.5, -2.25, -0.125]
    gc = np.array([[-0.5, -3.0], [-2.0, -1.0], [-0.25, -0.75]])
    assert cw.chunk_decay_bounds(gc, C=2) == [-1.5, -0.25]


def test_cp_warmup_channel_error_within_bound():
    """The warmup split with per-channel gates, windows chosen on the slowest-channel bound: within
    the bound's attenuation of the exact result, and exact when every window reaches the sequence start."""
    x = small_case(seed=53, B=1, H=1, T=640, K=16, V=8, gate="channel", g_mu=0.0)
    o, ht = run_oracle(x)
    log_eps = math.log(2.0 ** -24)
    o2, ht2 = cw.run_pairs(cw.cp_warmup, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                           x["h0"], C=16, seg_chunks=8, log_eps=log_eps)
    assert rel(ht2, ht) < 1e-6 and rel(o2, o) < 1e-6
    # the windows are truncated here (the bound reaches 2^-24 within the sequence), so the split is not
    # the exact recurrence
    g0 = np.asarray(x["g"])[0, :, 0]
    sums = cw.chunk_decay_bounds(g0, 16)
    assert cw.warmup_start(sums, 32, log_eps) > 0
    # with a threshold no window reaches, every segment starts from the true initial state: exact
    o3, ht3 = cw.run_pairs(cw.cp_warmup, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                           x["h0"], C=16, seg_chunks=8, log_eps=-1e9)
    assert rel(o3, o) < 1e-10 and rel(ht3, ht) < 1e-10


# ---------------------------------------------------------------- step a1: the chunk-local gate cumsum
def test_local_cumsum_golden():
    """Hand-worked cumsums ("Flash Linear Attention" page, sec. 3, chunk_local_cumsum; sec. 2 for
    the restart at every packed sequence start): exact binary values, compared exactly."""
    with open(os.path.join(GOLDEN, "gate_cumsum_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = cw.local_cumsum(np.array(c["g"]), c["C"], c["cu_seqlens"])
        assert np.array_equal(got, np.array(c["expected"])), c["name"]


def test_local_cumsum_restarts_match_per_sequence_runs():
    """Packed input equals the sequences cumsummed one by one, and each chunk's sum ends at
    the sum of the chunk's gates."""
    rng = np.random.default_rng(5)
    cu = np.array([0, 70, 70, 200, 201, 330])
    g = -rng.random((330, 3))
    got = cw.local_cumsum(g, 64, cu)
    for s, e in zip(cu[:-1], cu[1:]):
        assert np.array_equal(got[s:e], cw.local_cumsum(g[s:e], 64))
        for c0 in range(s, e, 64):
            c1 = min(c0 + 64, e)
            assert np.allclose(got[c1 - 1], g[c0:c1].sum(axis=0), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- input activations (f3)
def test_activation_closed_forms():
    """softplus, sigmoid, the two gate forms and the L2 norm against values they must take."""
    from oracle import activations as act
    assert act.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-15)
    assert act.sigmoid(0.0) == 0.5
    z = np.linspace(-50, 50, 101)
    assert np.allclose(act.softplus(z) - act.softplus(-z), z, atol=1e-12)       # softplus(z) - softplus(-z) = z
    assert np.allclose(act.sigmoid(z) + act.sigmoid(-z), 1.0, atol=1e-15)
    assert act.softplus(800.0) == 800.0 and act.softplus(-800.0) == 0.0            # no overflow
    # gate without a lower bound: -exp(A) * ln 2 at x + bias = 0; with one: lb / 2 there, lb and 0 at the ends
    A_log = np.array([0.0, math.log(3.0)])
    x = np.zeros((1, 1, 2))
    assert np.allclose(act.gate(x, A_log), [[[-math.log(2.0), -3 * math.log(2.0)]]], atol=1e-15)
    assert np.allclose(act.gate(x, A_log, lower_bound=-5.0), -2.5)
    assert np.allclose(act.gate(np.full((1, 1, 2), 1e3), A_log, lower_bound=-5.0), -5.0)
    assert np.allclose(act.gate(np.full((1, 1, 2), -1e3), A_log, lower_bound=-5.0), 0.0)
    # per-channel bias: the bias of channel d shifts channel d only
    xb = np.zeros((1, 1, 1, 3))
    bias = np.array([[0.0, 1.0, -1.0]])
    g = act.gate(xb, np.array([0.0]), bias)
    assert np.allclose(g[0, 0, 0], -np.logaddexp(0.0, bias[0]), atol=1e-15)
    # L2 norm: unit length, same direction; the zero vector stays zero
    v = np.array([[3.0, 4.0], [0.0, 0.0]])
    assert np.allclose(act.l2norm(v), [[0.6, 0.8], [0.0, 0.0]])
