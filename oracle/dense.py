"""The oracle's dense transition-product formulation, in fp64 numpy, for tiny T.

TEST INFRASTRUCTURE (see oracle/__init__.py).

"Understanding Kimi Delta Attention", box "KDA as a structured state
transition", writes one token as an affine map of the state,

    S_t = F_t S_{t-1} + beta_t k_t v_t^T,   F_t = (I - beta_t k_t k_t^T) D_t,

with D_t = Diag(a_t). This module builds every F_t as an explicit d_k x d_k
matrix, forms the prefix transitions P_t = F_t ... F_1 and the accumulated
writes W_t = sum_{s <= t} F_t ... F_{s+1} beta_s k_s v_s^T, and reads
S_t = P_t S_0 + W_t and o_t = S_t^T (scale q_t). No state is updated in place
token by token; the state at t is always rebuilt from the products.
"""
import numpy as np


def transition(k, g, beta):
    """F = (I - beta k k^T) Diag(exp(g)) as a dense d_k x d_k matrix."""
    k = np.asarray(k, dtype=np.float64)
    dk = k.shape[0]
    return (np.eye(dk) - beta * np.outer(k, k)) @ np.diag(np.exp(np.asarray(g, dtype=np.float64)))


def dense_scan(q, k, v, g, beta, scale, S0):
    """One sequence, one head: q, k, g [T, d_k]; v [T, d_v]; beta [T];
    S0 [d_k, d_v]. Returns (out [T, d_v], S_T)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    Fs = [transition(k[t], g[t], float(beta[t])) for t in range(T)]
    out = np.zeros((T, dv))
    S_t = np.array(S0, dtype=np.float64)
    for t in range(T):
        P = np.eye(dk)
        for s in range(t + 1):
            P = Fs[s] @ P
        W = np.zeros((dk, dv))
        for s in range(t + 1):
            M = np.eye(dk)
            for r in range(s + 1, t + 1):
                M = Fs[r] @ M
            W = W + M @ (float(beta[s]) * np.outer(k[s], v[s]))
        S_t = P @ np.asarray(S0, dtype=np.float64) + W
        out[t] = S_t.T @ (scale * q[t])
    return out, S_t
