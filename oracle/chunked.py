"""Chunked (WY/UT) form of the gated delta rule, numpy fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Shares no code with the CUDA path
nor with the token-by-token C oracle; it exists to pin the chunk algebra against the
token recurrence.

The recurrence is the one of "Qwen3.5-27B GPTQ Garbage Inference -- Root Cause
Analysis", "Why abliteration failed on Qwen3.5", item 3, S_t = exp(g_t) S_{t-1}
(I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = scale * S_t q_t, with the state kept as
h = S^T of shape [dk, dv].  Chunks are anchored at each sequence start and have length
``chunk`` (the last one may be shorter), following "[Feature] Add batch invariance support
to GDN_ATTN backend - #45819", Birol's comment, part 3(a): chunk boundaries on
multiples of the delta-rule block.

Within one chunk with tokens r = 0..L-1, gamma_r = sum_{s<=r} g_s (inclusive), and
entering state h0:

    A[r,s]  = beta_r exp(gamma_r - gamma_s) (k_r . k_s)        for s < r, else 0
    Tinv    = (I + A)^-1
    W       = Tinv diag(beta exp(gamma)) K
    U       = Tinv diag(beta) V
    Vnew    = U - W h0                       (the per-token delta vectors u_r)
    Mqk[r,s]= exp(gamma_r - gamma_s) (q_r . k_s)               for s <= r, else 0
    O       = scale * ( diag(exp(gamma)) Q h0 + Mqk Vnew )
    h       = exp(gamma_{L-1}) h0 + K^T diag(exp(gamma_{L-1} - gamma)) Vnew

Only differences gamma_r - gamma_s with s <= r are exponentiated, so nothing overflows.
"""
from __future__ import annotations

import numpy as np

_EPS = 1e-6


def _norm(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + _EPS)


def _as64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def chunk_step(Qc, Kc, Vc, gc, bc, h0, scale):
    """One chunk of the WY/UT form for one (sequence, v-head).  Returns (O, h)."""
    L = Kc.shape[0]
    gam = np.cumsum(gc)
    diff = gam[:, None] - gam[None, :]
    lower_strict = np.tril(np.ones((L, L), bool), -1)
    lower_incl = np.tril(np.ones((L, L), bool), 0)
    decay = np.where(lower_incl, np.exp(np.where(lower_incl, diff, 0.0)), 0.0)
    A = np.where(lower_strict, bc[:, None] * decay * (Kc @ Kc.T), 0.0)
    Tinv = np.linalg.solve(np.eye(L) + A, np.eye(L))
    W = Tinv @ ((bc * np.exp(gam))[:, None] * Kc)
    U = Tinv @ (bc[:, None] * Vc)
    Vnew = U - W @ h0
    Mqk = np.where(lower_incl, decay * (Qc @ Kc.T), 0.0)
    O = scale * (np.exp(gam)[:, None] * (Qc @ h0) + Mqk @ Vnew)
    tail = np.exp(gam[-1] - gam)
    h = np.exp(gam[-1]) * h0 + Kc.T @ (tail[:, None] * Vnew)
    return O, h


def chunked_gated_delta_rule(q, k, v, g, beta, cu_seqlens, chunk=64, scale=1.0,
                             l2norm=False, initial_state=None):
    """Chunked WY/UT gated delta rule.  Shapes as ``oracle.gated_delta_rule``."""
    q, k, v, g, beta = (_as64(a) for a in (q, k, v, g, beta))
    cu = np.asarray(_as64(cu_seqlens), dtype=np.int64)
    T, Hk, dk = q.shape
    _, Hv, dv = v.shape
    N = cu.shape[0] - 1
    G = Hv // Hk
    if l2norm:
        q, k = _norm(q), _norm(k)
    h_all = _as64(initial_state)
    o = np.zeros((T, Hv, dv))
    hT = np.zeros((N, Hv, dk, dv))
    for n in range(N):
        s0, s1 = int(cu[n]), int(cu[n + 1])
        for hv in range(Hv):
            hk = hv // G
            h = np.zeros((dk, dv)) if h_all is None else h_all[n, hv].copy()
            for c0 in range(s0, s1, chunk):
                c1 = min(c0 + chunk, s1)
                O, h = chunk_step(q[c0:c1, hk], k[c0:c1, hk], v[c0:c1, hv],
                                  g[c0:c1, hv], beta[c0:c1, hv], h, scale)
                o[c0:c1, hv] = O
            hT[n, hv] = h
    return o, hT
