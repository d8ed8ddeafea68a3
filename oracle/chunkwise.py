"""The oracle's chunkwise/WY formulation, in fp64 numpy.

TEST INFRASTRUCTURE (see oracle/__init__.py). Independent of the token scan in
kda_scan.c: it shares no code with it and is checked against it.

It follows "Understanding Kimi Delta Attention", sections "The triangular
system", "Putting the chunks together" and Figure 04, step by step, for one
chunk of n <= C tokens with incoming state S0 (d_k x d_v):

  G_i      = sum_{r <= i} log alpha_r              cumulative log-decay
  Gamma_i  = Diag(exp(G_i))                        decay from chunk start
  Gamma_{j->i} = Diag(exp(G_i - G_j))              decay from token j to i
  A_ij     = -beta_i k_i^T Gamma_{j->i} k_j        for j < i, else 0
  T        = (I - A)^{-1}                          via a triangular solve
  L_i      = (Gamma_i k_i)^T
  R = T B L,  U = T B V,  Z = U - R S0             B = Diag(beta)
  Qbar_i   = (Gamma_i q_i)^T  (q already multiplied by the query scale)
  H_ij     = q_i^T Gamma_{j->i} k_j                for j <= i, else 0
  O        = Qbar S0 + H Z
  S_out    = Gamma_n S0 + Kbar^T Z,  Kbar_j = (Gamma_{j->n} k_j)^T

The per-pair decay is formed the plain way, as an n x n x d_k tensor of
exp(G_i - G_j) with the non-causal pairs removed before exponentiating (the
size "Kimi Delta Attention: a half-life per channel", section "What changes in
the kernel", warns a kernel against; an oracle can afford it).

A sequence whose length is not a multiple of C ends with a shorter chunk; the
formulas above hold for any n, so no padding is involved.
"""
import numpy as np
from scipy.linalg import solve_triangular


def chunk_factors(k, g, beta):
    """For one chunk: returns (G, A, T) with G the cumulative log-decay
    [n, d_k], A the strictly lower correction matrix [n, n] and T = (I-A)^{-1}.
    """
    k = np.asarray(k, dtype=np.float64)
    n = k.shape[0]
    G = np.cumsum(np.asarray(g, dtype=np.float64), axis=0)
    diff = G[:, None, :] - G[None, :, :]                 # [i, j, c] = G_i - G_j
    strict = np.tril(np.ones((n, n), dtype=bool), -1)
    decay = np.where(strict[:, :, None], np.exp(np.where(strict[:, :, None], diff, 0.0)), 0.0)
    A = -np.asarray(beta, dtype=np.float64)[:, None] * np.einsum("ic,ijc,jc->ij", k, decay, k)
    T = solve_triangular(np.eye(n) - A, np.eye(n), lower=True, unit_diagonal=True)
    return G, A, T


def chunk_step(q, k, v, g, beta, S0):
    """One chunk of the chunkwise form. q already carries the query scale.
    Returns (O [n, d_v], S_out [d_k, d_v])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    n = k.shape[0]
    G, A, T = chunk_factors(k, g, beta)
    L = np.exp(G) * k
    R = T @ (beta[:, None] * L)
    U = T @ (beta[:, None] * v)
    Z = U - R @ S0
    Qbar = np.exp(G) * q
    diff = G[:, None, :] - G[None, :, :]
    causal = np.tril(np.ones((n, n), dtype=bool), 0)
    decay = np.where(causal[:, :, None], np.exp(np.where(causal[:, :, None], diff, 0.0)), 0.0)
    Hm = np.einsum("ic,ijc,jc->ij", q, decay, k)
    O = Qbar @ S0 + Hm @ Z
    Kbar = np.exp(G[-1][None, :] - G) * k
    S_out = np.exp(G[-1])[:, None] * S0 + Kbar.T @ Z
    return O, S_out


def chunkwise_scan(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, C=64):
    """Same contract and shapes as ``oracle.scan`` but computed chunk by chunk
    with chunk size C (C = 1 degenerates to the token recurrence)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        seqs = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        seqs = [(0, int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]
    out = np.zeros((B, T, H, dv))
    final = np.zeros((len(seqs), H, dk, dv))
    for n, (b, bos, eos) in enumerate(seqs):
        for h in range(H):
            S = np.zeros((dk, dv)) if init_state is None else np.array(init_state[n, h], dtype=np.float64)
            for s in range(bos, eos, C):
                e = min(s + C, eos)
                O, S = chunk_step(scale * q[b, s:e, h], k[b, s:e, h], v[b, s:e, h],
                                  g[b, s:e, h], beta[b, s:e, h], S)
                out[b, s:e, h] = O
            final[n, h] = S
    return out, final
