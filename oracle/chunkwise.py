"""Naive fp64 chunkwise (WY/UT) form of the channelwise gated delta rule.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Pure numpy; shares
nothing with the C oracle or the CUDA library.

Follows the chunked path of "Add parallel chunked prefill for channelwise
gated delta rule" (executorch PR #21061), Summary: per chunk, per-channel
log-decay prefixes, causal query/key terms, the beta-folded triangular
transform, WY pseudo-keys and pseudo-values, and the inter-chunk state carry;
the ragged final chunk runs through the same code.  The pages give the names
of these steps, not their formulas; the formulas below are the plain algebra
that makes the chunked form equal to the token recurrence (obtained by
unrolling the recurrence over one chunk; the tests check it against the
recurrence):

  gamma_r   = sum_{s<=r} g_s                   (per channel, inside the chunk)
  A_rs      = beta_r sum_i k_ri k_si exp(gamma_ri - gamma_si),  s < r
  P_rs      =        sum_i q_ri k_si exp(gamma_ri - gamma_si),  s <= r
  Tm        = (I + A)^{-1} Diag(beta)          (forward substitution)
  W         = Tm (K * exp(gamma))              (pseudo-keys)
  Ut        = Tm V                             (pseudo-values)
  U         = Ut - W S
  O         = (Q * exp(gamma)) S + P U
  S        <- Diag(exp(gamma_C)) S + (K * exp(gamma_C - gamma))^T U

Pairwise exponents are formed as exp(gamma_r - gamma_s) directly, never as a
product exp(gamma_r) * exp(-gamma_s), so no anchoring is needed here.
"""
from __future__ import annotations

import numpy as np


def _softplus(x):
    return np.where(x > 20.0, x, np.log1p(np.exp(np.minimum(x, 20.0))))


def _prep(q, k, v, g, beta, a, b, A_log, dt_bias, l2norm, q_scale, eps):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, T, Hk, dk = q.shape
    Hv = v.shape[2]
    rep = Hv // Hk
    # head repeat: v-head h reads q/k head h // rep
    qh = np.repeat(q, rep, axis=2)
    kh = np.repeat(k, rep, axis=2)
    if l2norm:
        qh = qh / np.sqrt((qh * qh).sum(-1, keepdims=True) + eps)
        kh = kh / np.sqrt((kh * kh).sum(-1, keepdims=True) + eps)
    qh = qh * (q_scale if q_scale is not None else 1.0 / np.sqrt(dk))
    if g is not None:
        gg = np.asarray(g, dtype=np.float64)
        bb = np.asarray(beta, dtype=np.float64)
    else:
        a = np.asarray(a, dtype=np.float64)
        b = np.asarray(b, dtype=np.float64)
        gs = -np.exp(np.asarray(A_log, dtype=np.float64)) * _softplus(a + np.asarray(dt_bias, dtype=np.float64))
        gg = np.repeat(gs[..., None], dk, axis=-1)
        bb = 1.0 / (1.0 + np.exp(-b))
    return qh, kh, v, gg, bb


def chunkwise(q, k, v, *, chunk, g=None, beta=None, a=None, b=None, A_log=None, dt_bias=None,
              S0=None, l2norm=True, q_scale=None, eps=1e-6):
    """Chunked fp64 evaluation; same inputs and outputs as ``oracle.recurrence``."""
    qh, kh, v, gg, bb = _prep(q, k, v, g, beta, a, b, A_log, dt_bias, l2norm, q_scale, eps)
    B, T, Hv, dk = kh.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, Hv, dv))
    S_out = np.zeros((B, Hv, dk, dv))
    for bi in range(B):
        for h in range(Hv):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[bi, h], dtype=np.float64)
            for c0 in range(0, T, chunk):
                c1 = min(T, c0 + chunk)
                L = c1 - c0
                Q = qh[bi, c0:c1, h]          # [L, dk]
                K = kh[bi, c0:c1, h]          # [L, dk]
                V = v[bi, c0:c1, h]           # [L, dv]
                G = gg[bi, c0:c1, h]          # [L, dk]
                be = bb[bi, c0:c1, h]         # [L]
                gam = np.cumsum(G, axis=0)    # per-channel log-decay prefix
                A = np.zeros((L, L))
                P = np.zeros((L, L))
                for r in range(L):
                    for s in range(r + 1):
                        dec = np.exp(gam[r] - gam[s])
                        if s < r:
                            A[r, s] = be[r] * np.sum(K[r] * K[s] * dec)
                        P[r, s] = np.sum(Q[r] * K[s] * dec)
                # Tm = (I + A)^{-1} Diag(beta) by forward substitution, row by row
                Tm = np.zeros((L, L))
                for r in range(L):
                    row = np.zeros(L)
                    row[r] = be[r]
                    for s in range(r):
                        row -= A[r, s] * Tm[s]
                    Tm[r] = row
                W = Tm @ (K * np.exp(gam))
                Ut = Tm @ V
                U = Ut - W @ S
                o[bi, c0:c1, h] = (Q * np.exp(gam)) @ S + P @ U
                S = np.exp(gam[-1])[:, None] * S + (K * np.exp(gam[-1] - gam)).T @ U
            S_out[bi, h] = S
    return o, S_out
