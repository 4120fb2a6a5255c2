"""The chunked (WY/UT) form of Gated Delta Rule prefill in numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is a second,
independent CPU statement of the same result as the token recurrence; the
tests check the two against each other to fp64 round-off.

Derivation (the chunk-parallel delta-rule form of Yang et al., "Parallelizing
Linear Transformers with the Delta Rule over Sequence Length", with the gated
extension of "Gated Delta Networks"): writing the recurrence
``S_t = g_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T`` as
``S_t = g_t S_{t-1} + u_t k_t^T`` with ``u_t = b_t (v_t - g_t S_{t-1} k_t)``
and unrolling over a chunk of C rows with ``G = cumsum(log g)``:

    gamma_i   = exp(G_i),   Gam_ij = exp(G_i - G_j) for i >= j, else 0
    A         = strictly_lower(diag(b) (K K^T * Gam))
    T         = (I + A)^-1
    W         = T diag(b * gamma) K,     U = T diag(b) V
    V_new     = U - W S^T                 (row i is u_i)
    O         = scale (diag(gamma) Q S^T + (Q K^T * Gam) V_new)
    S        <- gamma_C S + V_new^T diag(exp(G_C - G)) K

with S the state entering the chunk.  Requires g > 0.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
from scipy.linalg import solve_triangular

CHUNK = 64


def chunked_unit(q, k, v, g, beta, scale: float, use_qk_l2norm: bool, s0,
                 chunk: int = CHUNK, eps: float = 1e-6):
    """One (sequence, head): q, k ``[L, Dk]``, v ``[L, Dv]``, g, beta ``[L]``
    or None, s0 ``[Dv, Dk]`` or None.  Returns (o ``[L, Dv]``, S ``[Dv, Dk]``)."""
    L, dk = q.shape
    dv = v.shape[1]
    if use_qk_l2norm:
        q = q / np.sqrt((q * q).sum(1, keepdims=True) + eps)
        k = k / np.sqrt((k * k).sum(1, keepdims=True) + eps)
    g = np.ones(L) if g is None else np.asarray(g, dtype=np.float64)
    b = np.ones(L) if beta is None else np.asarray(beta, dtype=np.float64)
    S = np.zeros((dv, dk)) if s0 is None else np.array(s0, dtype=np.float64)
    o = np.zeros((L, dv))
    for c0 in range(0, L, chunk):
        c1 = min(c0 + chunk, L)
        n = c1 - c0
        Q, K, V, bc = q[c0:c1], k[c0:c1], v[c0:c1], b[c0:c1]
        G = np.cumsum(np.log(g[c0:c1]))
        gamma = np.exp(G)
        lower_incl = np.tril(np.ones((n, n), dtype=bool))
        diff = np.where(lower_incl, G[:, None] - G[None, :], 0.0)
        Gam = np.where(lower_incl, np.exp(diff), 0.0)
        A = np.tril(bc[:, None] * (K @ K.T) * Gam, -1)
        T = solve_triangular(np.eye(n) + A, np.eye(n), lower=True, unit_diagonal=True)
        W = T @ ((bc * gamma)[:, None] * K)
        U = T @ (bc[:, None] * V)
        V_new = U - W @ S.T
        o[c0:c1] = scale * (gamma[:, None] * (Q @ S.T) + ((Q @ K.T) * Gam) @ V_new)
        S = gamma[-1] * S + V_new.T @ (np.exp(G[-1] - G)[:, None] * K)
    return o, S


def chunked(q, k, v, g=None, beta=None, scale=None, initial_state=None,
            state_indices=None, cu_seqlens=None, use_qk_l2norm=False,
            units: Optional[Sequence[tuple]] = None, chunk: int = CHUNK):
    """Whole-problem chunked form with the same signature and results layout as
    :func:`oracle.recurrence`."""
    from . import Units, resolve_scale, scatter, L2NORM_EPS

    if cu_seqlens is None:
        cu_seqlens = [0, int(q.shape[0])]
    U = Units(q, k, v, g, beta, initial_state, state_indices, cu_seqlens, units)
    sc = resolve_scale(scale, U.dk)
    rows = np.zeros((int(U.len.sum()) if len(U.len) else 0, U.dv))
    sf = np.zeros((len(U.units), U.dv, U.dk))
    for i in range(len(U.units)):
        a, L = int(U.off[i]), int(U.len[i])
        sl = slice(a, a + L)
        o_u, s_u = chunked_unit(
            U.q[sl], U.k[sl], U.v[sl], None if U.g is None else U.g[sl],
            None if U.beta is None else U.beta[sl], sc, use_qk_l2norm,
            None if U.s0 is None else U.s0[i], chunk=chunk, eps=L2NORM_EPS)
        rows[sl] = o_u
        sf[i] = s_u
    o, fs = scatter(U, rows, sf, cu_seqlens)
    final = np.full((U.N, U.H, U.dv, U.dk), np.nan)
    for (n, h), s in fs.items():
        final[n, h] = s
    return o, final
