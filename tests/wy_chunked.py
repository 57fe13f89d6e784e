"""fp64 numpy chunked (WY / UT) form of the gated delta rule, used only to
check that the chunked algebra the CUDA prefill kernel follows equals the
token-by-token oracle.  Written from the recurrence itself:

  within a chunk with inclusive log-decay prefix G (G_i = g_1 + ... + g_i),
  Gamma_ij = exp(G_i - G_j) for i >= j, the state after token i is
      S_i = exp(G_i) S_0 + sum_{j <= i} Gamma_ij k_j u_j^T
  where the pseudo-values u solve the unit-lower system
      (I + A) U = diag(beta) V - diag(beta exp(G)) K S_0,
      A = strict_lower(diag(beta) (K K^T * Gamma)).
  Hence, with T = (I + A)^-1, W = T diag(beta exp(G)) K, U_v = T diag(beta) V:
      U = U_v - W S_0
      O = diag(exp(G)) Q S_0 + (Q K^T * Gamma * causal) U
      S_C = exp(G_C) S_0 + (K * exp(G_C - G))^T U
  (S is the stored transpose St[k][v]).  exp(-G) is never formed.
"""
import numpy as np
from scipy.linalg import solve_triangular


def chunked_recurrence(q, k, v, g, beta, S0, chunk):
    T, dk = q.shape
    dv = v.shape[1]
    S = np.array(S0, dtype=np.float64, copy=True)
    O = np.zeros((T, dv))
    for s in range(0, T, chunk):
        e = min(s + chunk, T)
        Q, K, V = q[s:e], k[s:e], v[s:e]
        G = np.cumsum(g[s:e])
        b = beta[s:e]
        n = e - s
        diff = G[:, None] - G[None, :]
        lower_incl = np.tril(np.ones((n, n), dtype=bool))
        Gam = np.where(lower_incl, np.exp(np.where(lower_incl, diff, 0.0)), 0.0)
        A = np.tril(b[:, None] * (K @ K.T) * Gam, -1)
        I = np.eye(n)
        W = solve_triangular(I + A, (b * np.exp(G))[:, None] * K, lower=True, unit_diagonal=True)
        Uv = solve_triangular(I + A, b[:, None] * V, lower=True, unit_diagonal=True)
        U = Uv - W @ S
        O[s:e] = np.exp(G)[:, None] * (Q @ S) + ((Q @ K.T) * Gam) @ U
        S = np.exp(G[-1]) * S + (K * np.exp(G[-1] - G)[:, None]).T @ U
    return O, S
