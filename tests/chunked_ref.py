"""Float64 chunked (WY/UT) form of the gated delta rule -- a test helper.

The pages run the recurrence one token at a time.  The GPU prefill instead
re-associates it over chunks of C tokens.  This module writes that
re-association out in numpy so a test can show, on the CPU, that it equals the
sequential oracle to float64 rounding (a re-association, not an approximation).
It is test infrastructure: the CUDA path neither imports nor mirrors it.

Per chunk, with S0 the state entering it, g_i, beta_i the gates and
G_i = g_1 + ... + g_i, gamma_i = exp(G_i):
  delta_i = beta_i (v_i - gamma_i S0^T k_i - sum_{j<i} e^{G_i-G_j} (k_i.k_j) delta_j)
so (I + A) Delta = diag(beta) V - diag(beta gamma) K S0 with the strictly lower
A_ij = beta_i e^{G_i-G_j} k_i.k_j, hence Delta = U - W S0 for
  T = (I + A)^-1,  W = T diag(beta gamma) K,  U = T diag(beta) V.
Outputs: O = scale (diag(gamma) Q S0 + P Delta), P_ij = e^{G_i-G_j} q_i.k_j (j <= i).
Carry:   S_C = gamma_C S0 + (diag(e^{G_C - G}) K)^T Delta.
"""
import numpy as np


def chunked_unit(q, k, v, g, beta, S0, scale, C=64):
    """q,k [L, d_k]; v [L, d_v]; g, beta [L]; S0 [d_k, d_v] -> (o [L, d_v], S)."""
    L = q.shape[0]
    S = S0.copy()
    o = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        c1 = min(c0 + C, L)
        Q, K, V = q[c0:c1], k[c0:c1], v[c0:c1]
        gc, bc = g[c0:c1], beta[c0:c1]
        n = c1 - c0
        G = np.cumsum(gc)
        gamma = np.exp(G)
        decay = np.exp(np.minimum(G[:, None] - G[None, :], 0.0))   # only j <= i is used
        A = np.tril(bc[:, None] * decay * (K @ K.T), -1)
        Tm = np.linalg.inv(np.eye(n) + A)
        W = Tm @ ((bc * gamma)[:, None] * K)
        U = Tm @ (bc[:, None] * V)
        Delta = U - W @ S
        P = np.tril(decay * (Q @ K.T))
        o[c0:c1] = scale * (gamma[:, None] * (Q @ S) + P @ Delta)
        Ktil = np.exp(G[-1] - G)[:, None] * K
        S = gamma[-1] * S + Ktil.T @ Delta
    return o, S


def chunked_unit_per_key(q, k, v, g, beta, S0, scale, C=64):
    """The same with one log decay per key dimension, g [L, d_k] (Step 1 scales row i of
    S by e^{g_i}).  G_t = g_1 + ... + g_t per dimension; inside a chunk
      S_t = diag(e^{G_t}) S0 + sum_{s<=t} diag(e^{G_t - G_s}) k_s delta_s^T,
    so A_ts = beta_t sum_i k_ti k_si e^{G_ti - G_si} (s < t) and P likewise with q_t
    (s <= t), W = T diag(beta) (K o e^G), U = T diag(beta) V, and
      O = scale ((Q o e^G) S0 + P Delta),  S_C = diag(e^{G_C}) S0 + (K o e^{G_C - G})^T Delta."""
    L = q.shape[0]
    S = S0.copy()
    o = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        c1 = min(c0 + C, L)
        Q, K, V = q[c0:c1], k[c0:c1], v[c0:c1]
        bc = beta[c0:c1]
        n = c1 - c0
        G = np.cumsum(g[c0:c1], axis=0)                              # [n, d_k]
        E = np.exp(np.minimum(G[:, None, :] - G[None, :, :], 0.0))   # [t, s, i], s <= t used
        A = np.tril(bc[:, None] * np.einsum("ti,si,tsi->ts", K, K, E), -1)
        P = np.tril(np.einsum("ti,si,tsi->ts", Q, K, E))
        Tm = np.linalg.inv(np.eye(n) + A)
        W = Tm @ (bc[:, None] * (K * np.exp(G)))
        U = Tm @ (bc[:, None] * V)
        Delta = U - W @ S
        o[c0:c1] = scale * ((Q * np.exp(G)) @ S + P @ Delta)
        S = np.exp(G[-1])[:, None] * S + (K * np.exp(G[-1] - G)).T @ Delta
    return o, S
