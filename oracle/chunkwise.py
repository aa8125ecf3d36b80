"""Naive fp64 NumPy statements of the chunk forms of the gated delta rule.

TEST INFRASTRUCTURE ONLY.  Each function follows one passage of the pages, in
their order and notation, with ``numpy.linalg`` as the only library step.  No
blocking, fusion or reordering beyond what the passage states.  Notation for
one chunk (rows = tokens of the chunk, at most C of them):

* ``G``  inclusive cumulative natural-log gate inside the chunk (restarts at
  every chunk and sequence), ``gam = exp(G)``, ``gC = gam[-1]`` (the last
  *valid* token of a partial chunk);
* ``Gam[i, j] = exp(G_i - G_j)`` (the relative decay);
* ``StrictLower`` / ``Lower`` keep j < i / j <= i.

Per-pair functions take q, k [L, K], v [L, V], g [L] (scalar gate) or [L, K]
(per-key-channel gate), beta [L], S0 [K, V] and return (o [L, V], S_end [K, V]).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "local_cumsum", "fla_form", "qla_form", "channel_form", "forward_substitution",
    "blocked_inverse", "cp_exact_deltanet", "cp_exact_qla", "cp_warmup",
    "warmup_start", "chunk_decay_bounds", "run_pairs",
]


def local_cumsum(g, C, cu_seqlens=None):
    """Chunk-local inclusive cumsum of the log-gate.

    "Flash Linear Attention" page, sec. 3 (chunk_local_cumsum): inside a chunk
    g_t <- sum of g_s for s in the chunk, s <= t; nothing carries across chunks.
    Packed input ("Flash Linear Attention" page, sec. 2, varlen): chunks are
    counted from each sequence's first token, so the sum also restarts at every
    sequence start ``cu_seqlens[n]``.  Works on the leading (token) axis, so it
    covers the per-channel gate too.
    """
    g = np.asarray(g, dtype=np.float64)
    out = np.empty_like(g)
    bounds = [0, g.shape[0]] if cu_seqlens is None else [int(b) for b in cu_seqlens]
    for bos, eos in zip(bounds[:-1], bounds[1:]):
        for s in range(bos, eos, C):
            out[s:min(s + C, eos)] = np.cumsum(g[s:min(s + C, eos)], axis=0)
    return out


def _strict_lower(M):
    return np.tril(M, -1)


def _lower(M):
    return np.tril(M, 0)


def fla_form(q, k, v, g, beta, scale, S0, C):
    """FLA's four-step chunk form (FlashQLA blog, "Key problems in FLA's GDN
    chunked prefill", the four update lines; GDN-in-FLA notes, forward Steps
    2-5).

        A  = (I + StrictLower(diag(beta)(Gam * K K^T)))^-1
        W  = A diag(beta) diag(gam) K,   U = A diag(beta) V
        V' = U - W S
        O  = scale [diag(gam) Q S + (Lower(Gam) * Q K^T) V']
        S  <- gC S + K^T diag(gC / gam) V'

    ``scale`` multiplies both output terms (the FLA output kernel scales both,
    "Flash Linear Attention" page, sec. 3).
    """
    L = q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.zeros((L, v.shape[1]))
    for s in range(0, L, C):
        Q, K, Vc, b = q[s:s + C], k[s:s + C], v[s:s + C], beta[s:s + C]
        G = np.cumsum(g[s:s + C])
        gam = np.exp(G)
        gC = gam[-1]
        Gam = np.exp(G[:, None] - G[None, :])
        n = Q.shape[0]
        A = np.linalg.inv(np.eye(n) + _strict_lower(np.diag(b) @ (Gam * (K @ K.T))))
        W = A @ np.diag(b) @ np.diag(gam) @ K
        U = A @ np.diag(b) @ Vc
        Vp = U - W @ S
        o[s:s + C] = scale * (np.diag(gam) @ Q @ S + (_lower(Gam) * (Q @ K.T)) @ Vp)
        S = gC * S + K.T @ np.diag(gC / gam) @ Vp
    return o, S


def qla_form(q, k, v, g, beta, scale, S0, C):
    """FlashQLA's restructured chunk form (FlashQLA blog, "A balanced
    solution", steps 1 and 3): A carries no gate,

        A0  = (I + StrictLower(diag(beta) K K^T))^-1
        VD  = V - diag(gam) K S
        V'  = (Gam * A0) diag(beta) VD
        S   <- gC S + K^T diag(gC / gam) V'
        O   = scale [diag(gam) Q S + (Lower(Gam) * Q K^T) V']
    """
    L = q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.zeros((L, v.shape[1]))
    for s in range(0, L, C):
        Q, K, Vc, b = q[s:s + C], k[s:s + C], v[s:s + C], beta[s:s + C]
        G = np.cumsum(g[s:s + C])
        gam = np.exp(G)
        gC = gam[-1]
        Gam = np.exp(G[:, None] - G[None, :])
        n = Q.shape[0]
        A0 = np.linalg.inv(np.eye(n) + _strict_lower(np.diag(b) @ (K @ K.T)))
        VD = Vc - np.diag(gam) @ K @ S
        Vp = (Gam * A0) @ np.diag(b) @ VD
        o[s:s + C] = scale * (np.diag(gam) @ Q @ S + (_lower(Gam) * (Q @ K.T)) @ Vp)
        S = gC * S + K.T @ np.diag(gC / gam) @ Vp
    return o, S


def channel_form(q, k, v, g, beta, scale, S0, C):
    """Per-key-channel gate (KDA) chunk form ("KDA source walkthrough":
    Akk/Aqk with exp(g_id - g_jd) in chunk_kda_fwd_intra, w = A(beta k e^g),
    u = A(beta v) in recompute_w_u_fwd, kg = k e^(g_C - g) and the per-row
    state decay in chunk_gated_delta_rule_fwd_h, qg = q e^g in the output):

        Akk[i,j] = beta_i sum_d k_id k_jd exp(G_id - G_jd)   (j < i)
        A        = (I + Akk)^-1
        U = A diag(beta) V,  W = A diag(beta) (K * exp(G)),  V' = U - W S
        O_i = scale [ (q_i * e^G_i)^T S + sum_{j<=i} Aqk[i,j] V'_j ],
              Aqk[i,j] = sum_d q_id k_jd exp(G_id - G_jd)
        S  <- Diag(e^G_C) S + (K * exp(G_C - G))^T V'
    """
    L = q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.zeros((L, v.shape[1]))
    for s in range(0, L, C):
        Q, K, Vc, b = q[s:s + C], k[s:s + C], v[s:s + C], beta[s:s + C]
        G = np.cumsum(g[s:s + C], axis=0)                  # [n, K]
        D = np.exp(G[:, None, :] - G[None, :, :])          # [n, n, K], D[i,j,d]
        n = Q.shape[0]
        Akk = np.einsum("id,jd,ijd->ij", K, K, D)
        Aqk = np.einsum("id,jd,ijd->ij", Q, K, D)
        A = np.linalg.inv(np.eye(n) + _strict_lower(np.diag(b) @ Akk))
        U = A @ np.diag(b) @ Vc
        W = A @ np.diag(b) @ (K * np.exp(G))
        Vp = U - W @ S
        o[s:s + C] = scale * ((Q * np.exp(G)) @ S + _lower(Aqk) @ Vp)
        S = np.diag(np.exp(G[-1])) @ S + (K * np.exp(G[-1][None, :] - G)).T @ Vp
    return o, S


def forward_substitution(Lm):
    """(I + Lm)^-1 for strictly lower Lm, row by row ("Flash Linear Attention"
    page, sec. 4: row i absorbs the rows above it)."""
    n = Lm.shape[0]
    X = np.eye(n)
    for i in range(1, n):
        X[i, :i] = -Lm[i, :i] @ X[:i, :i]
    return X


def blocked_inverse(Lm, block=16):
    """(I + Lm)^-1 by forward substitution on block x block diagonal blocks and
    the exact block merge  [[A00,0],[A10,A11]]^-1 = [[A00^-1,0],
    [-A11^-1 A10 A00^-1, A11^-1]]  ("Flash Linear Attention" page, sec. 4,
    16 -> 32 -> 64)."""
    n = Lm.shape[0]
    if n <= block:
        return forward_substitution(Lm)
    h = n // 2
    if h % block:
        h = ((n + 2 * block - 1) // (2 * block)) * block
        h = min(h, n - 1)
    inv00 = blocked_inverse(Lm[:h, :h], block)
    inv11 = blocked_inverse(Lm[h:, h:], block)
    out = np.zeros((n, n))
    out[:h, :h] = inv00
    out[h:, h:] = inv11
    out[h:, :h] = -inv11 @ Lm[h:, :h] @ inv00
    return out


def _chunk_bounds(L, C):
    return [(s, min(s + C, L)) for s in range(0, L, C)]


def cp_exact_deltanet(q, k, v, g, beta, scale, S0, C, seg_chunks):
    """Chunk-parallel split with the S*/M correction in the DeltaNet form
    (FlashQLA blog, "Key problems", the CP pre-processing for rank j):

        S*_{i+1} = gC S*_i + K^T diag(gC/gam) V'_i      (V' computed from S*)
        M_{i+1}  = (gC I - K^T diag(gC/gam) W_i) M_i
        S_{j,0}  = S*_{j,0} + M_{j,0} S_{j-1,0}

    Reading: segment j starts from S* = 0 and M = I; after its chunks,
    S_end = S*_end + M_end S_start, and S_start(j+1) = S_end(j).
    Returns (o, S_end, starts) where starts[j] is the combined start state.
    """
    bounds = _chunk_bounds(q.shape[0], C)
    segs = [bounds[i:i + seg_chunks] for i in range(0, len(bounds), seg_chunks)]
    Kd = q.shape[1]
    pre = []
    for seg in segs:
        Ss = np.zeros((Kd, v.shape[1]))
        M = np.eye(Kd)
        for (s, e) in seg:
            K, Vc, b = k[s:e], v[s:e], beta[s:e]
            G = np.cumsum(g[s:e])
            gam, n = np.exp(G), e - s
            gC = gam[-1]
            Gam = np.exp(G[:, None] - G[None, :])
            A = np.linalg.inv(np.eye(n) + _strict_lower(np.diag(b) @ (Gam * (K @ K.T))))
            W = A @ np.diag(b) @ np.diag(gam) @ K
            U = A @ np.diag(b) @ Vc
            Vp = U - W @ Ss
            Ss = gC * Ss + K.T @ np.diag(gC / gam) @ Vp
            M = (gC * np.eye(Kd) - K.T @ np.diag(gC / gam) @ W) @ M
        pre.append((Ss, M))
    starts = [np.array(S0, dtype=np.float64)]
    for (Ss, M) in pre[:-1]:
        starts.append(Ss + M @ starts[-1])
    o = np.zeros((q.shape[0], v.shape[1]))
    S_end = None
    for j, seg in enumerate(segs):
        s0, e1 = seg[0][0], seg[-1][1]
        o[s0:e1], S_end = fla_form(q[s0:e1], k[s0:e1], v[s0:e1], g[s0:e1], beta[s0:e1],
                                   scale, starts[j], C)
    return o, S_end, starts


def cp_exact_qla(q, k, v, g, beta, scale, S0, C, seg_chunks):
    """Chunk-parallel pre-processing in FlashQLA's X/Y/Z form (FlashQLA blog,
    "A balanced solution", step 2.1 and 2.2), with A' read as the gate-free
    A0 of step 1:

        X = -diag(beta) A0^T K
        Y = gC K S* - diag(gC / gam) V
        Z = K M
        S* <- gC S* + X^T Y
        M  <- gC (M + X^T Z)
        S_{j,0} = S*_{j,0} + M_{j,0} S_{j-1,0}
    """
    bounds = _chunk_bounds(q.shape[0], C)
    segs = [bounds[i:i + seg_chunks] for i in range(0, len(bounds), seg_chunks)]
    Kd = q.shape[1]
    pre = []
    for seg in segs:
        Ss = np.zeros((Kd, v.shape[1]))
        M = np.eye(Kd)
        for (s, e) in seg:
            K, Vc, b = k[s:e], v[s:e], beta[s:e]
            G = np.cumsum(g[s:e])
            gam, n = np.exp(G), e - s
            gC = gam[-1]
            A0 = np.linalg.inv(np.eye(n) + _strict_lower(np.diag(b) @ (K @ K.T)))
            X = -np.diag(b) @ A0.T @ K
            Y = gC * (K @ Ss) - np.diag(gC / gam) @ Vc
            Z = K @ M
            Ss = gC * Ss + X.T @ Y
            M = gC * (M + X.T @ Z)
        pre.append((Ss, M))
    starts = [np.array(S0, dtype=np.float64)]
    for (Ss, M) in pre[:-1]:
        starts.append(Ss + M @ starts[-1])
    o = np.zeros((q.shape[0], v.shape[1]))
    S_end = None
    for j, seg in enumerate(segs):
        s0, e1 = seg[0][0], seg[-1][1]
        o[s0:e1], S_end = qla_form(q[s0:e1], k[s0:e1], v[s0:e1], g[s0:e1], beta[s0:e1],
                                   scale, starts[j], C)
    return o, S_end, starts


def warmup_start(chunk_gate_sums, seg_first_chunk, log_eps, max_chunks=None):
    """First chunk from which a segment starting at ``seg_first_chunk`` must be
    warmed up from a zero state (FlashQLA blog, "Further optimisation via gate
    decay": start W chunks early from S = 0; W from the gate statistics).

    Reading of the open threshold: walk back from the segment start adding the
    per-chunk gate sums; stop at the first chunk where the accumulated log-decay
    is <= log_eps.  If the sequence start is reached first, return 0 (warm up
    from the true initial state, which is exact).  With ||k|| <= 1 and beta in
    [0, 2] each transition has spectral norm <= its decay, so the dropped
    start state contributes at most exp(accumulated log-decay) ||S_true||.
    """
    acc = 0.0
    c = seg_first_chunk
    while c > 0:
        c -= 1
        acc += chunk_gate_sums[c]
        if acc <= log_eps:
            return c
        if max_chunks is not None and seg_first_chunk - c >= max_chunks:
            return 0
    return 0


def chunk_decay_bounds(g, C):
    """Per chunk, the log of a bound on how far the chunk's transitions contract
    the state (the gate statistics of the warmup split).  One token's transition
    A_t = (I - beta_t k_t k_t^T) Diag(alpha_t) has spectral norm at most
    max_d alpha_{t,d}, since ||k|| <= 1 and beta in [0, 2] keep the first factor's
    norm at most 1; a chunk therefore contracts the state by at most the product of
    those maxima.  In logs: the sum over the chunk's tokens of the largest
    per-channel log-gate; for a scalar gate, of the gate itself.  (Reading for
    per-channel gates: the per-channel products over a chunk are not a bound,
    because the delta-rule factor moves state between channels.)"""
    gt = g if g.ndim == 1 else g.max(axis=1)
    return [float(np.sum(gt[s:e])) for (s, e) in _chunk_bounds(gt.shape[0], C)]


def cp_warmup(q, k, v, g, beta, scale, S0, C, seg_chunks, log_eps):
    """Gate-driven warmup split: each segment j > 0 recomputes its start state
    from zero over the warmup chunks chosen by :func:`warmup_start` on the
    :func:`chunk_decay_bounds` (or from the true initial state when the walk
    reaches the sequence start), then emits its own chunks.  Scalar gate
    (:func:`qla_form`) or per-key-channel gate (:func:`channel_form`)."""
    bounds = _chunk_bounds(q.shape[0], C)
    sums = chunk_decay_bounds(g, C)
    form = qla_form if g.ndim == 1 else channel_form
    o = np.zeros((q.shape[0], v.shape[1]))
    S_end = None
    starts = []
    for c0 in range(0, len(bounds), seg_chunks):
        c1 = min(c0 + seg_chunks, len(bounds))
        w = warmup_start(sums, c0, log_eps) if c0 > 0 else 0
        S = np.array(S0, dtype=np.float64) if w == 0 else np.zeros_like(S0, dtype=np.float64)
        ws, s0, e1 = bounds[w][0], bounds[c0][0], bounds[c1 - 1][1]
        if s0 > ws:
            _, S = form(q[ws:s0], k[ws:s0], v[ws:s0], g[ws:s0], beta[ws:s0], scale, S, C)
        starts.append(S)
        o[s0:e1], S_end = form(q[s0:e1], k[s0:e1], v[s0:e1], g[s0:e1], beta[s0:e1],
                               scale, S, C)
    return o, S_end, starts


def run_pairs(form, q, k, v, g, beta, scale, h0=None, cu_seqlens=None, C=64, **kw):
    """Apply a per-pair chunk form to every (sequence, value head) pair of a
    batch laid out like the chunk API (q,k [B,T,H,K], v [B,T,HV,V], g [B,T,HV]
    or [B,T,HV,K], beta [B,T,HV], h0 [N,HV,K,V], cu_seqlens [N+1])."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, Kd = q.shape
    HV, Vd = v.shape[2], v.shape[3]
    cu = (np.arange(B + 1) * T) if cu_seqlens is None else np.asarray(cu_seqlens)
    N = len(cu) - 1
    qf, kf, vf = q.reshape(B * T, H, Kd), k.reshape(B * T, H, Kd), v.reshape(B * T, HV, Vd)
    gf = g.reshape((B * T,) + g.shape[2:])
    bf = beta.reshape(B * T, HV)
    o = np.zeros((B * T, HV, Vd))
    ht = np.zeros((N, HV, Kd, Vd))
    for n in range(N):
        s, e = int(cu[n]), int(cu[n + 1])
        for h in range(HV):
            hq = h // (HV // H)
            S0 = np.zeros((Kd, Vd)) if h0 is None else np.asarray(h0, dtype=np.float64)[n, h]
            if e == s:
                ht[n, h] = S0
                continue
            res = form(qf[s:e, hq], kf[s:e, hq], vf[s:e, h], gf[s:e, h], bf[s:e, h],
                       scale, S0, C, **kw)
            o[s:e, h], ht[n, h] = res[0], res[1]
    return o.reshape(B, T, HV, Vd), ht
