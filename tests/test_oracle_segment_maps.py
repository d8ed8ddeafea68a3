"""Pins of the chunk-level parallel prefix's reading on the fp64 oracle: the
state after a run of tokens is an affine function of the state entering it,
S_out = M S_in + E ("Understanding Kimi Delta Attention": each token's
transition S -> (I - beta k k^T) Diag(a) S + beta k v^T is affine, so runs of
tokens compose as affine maps). M is the run started from the identity with
v = 0, E the run started from a zero state; composing the maps of consecutive
runs in order reproduces the scan over all of them. These are the quantities
the segmented state pass computes (identity tiles with U = 0, d_v tiles from
zero) and combines."""
import numpy as np
import pytest

import oracle


def _inputs(rng, T, H, d):
    q = rng.normal(size=(1, T, H, d))
    k = rng.normal(size=(1, T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(1, T, H, d))
    g = -np.log1p(np.exp(rng.normal(size=(1, T, H, d)) - 2.0))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=(1, T, H))))
    return q, k, v, g, beta


def _run(q, k, v, g, beta, init, t0, t1):
    sl = slice(t0, t1)
    return oracle.scan(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], 0.3, init)


def _maps(q, k, v, g, beta, t0, t1, H, d):
    eye = np.broadcast_to(np.eye(d), (1, H, d, d)).copy()
    M = _run(q, k, np.zeros_like(v), g, beta, eye, t0, t1)[1]
    E = _run(q, k, v, g, beta, None, t0, t1)[1]
    return M, E


@pytest.mark.parametrize("T,cuts", [(40, (0, 13, 40)), (75, (0, 1, 30, 64, 75))])
def test_segment_maps_compose_to_the_scan(T, cuts):
    H, d = 2, 5
    rng = np.random.default_rng(T)
    q, k, v, g, beta = _inputs(rng, T, H, d)
    S0 = rng.normal(size=(1, H, d, d)) * 0.3
    out_full, S_full = oracle.scan(q, k, v, g, beta, 0.3, S0)
    S = S0
    for t0, t1 in zip(cuts[:-1], cuts[1:]):
        M, E = _maps(q, k, v, g, beta, t0, t1, H, d)
        # The run's own scan from S equals its affine map applied to S ...
        assert np.allclose(_run(q, k, v, g, beta, S, t0, t1)[1], M @ S + E, rtol=1e-12, atol=1e-12)
        # ... and the outputs rerun from the composed entering state are the
        # full scan's outputs for those tokens.
        assert np.allclose(_run(q, k, v, g, beta, S, t0, t1)[0], out_full[:, t0:t1], rtol=1e-12,
                           atol=1e-12)
        S = M @ S + E
    assert np.allclose(S, S_full, rtol=1e-12, atol=1e-12)


def test_transition_map_is_the_dense_product():
    # M of a run equals the ordered product of the per-token transitions
    # (I - beta_t k_t k_t^T) Diag(a_t), written out densely here.
    T, H, d = 6, 1, 4
    rng = np.random.default_rng(5)
    q, k, v, g, beta = _inputs(rng, T, H, d)
    M, _ = _maps(q, k, v, g, beta, 0, T, H, d)
    P = np.eye(d)
    for t in range(T):
        kt = k[0, t, 0]
        A = (np.eye(d) - beta[0, t, 0] * np.outer(kt, kt)) @ np.diag(np.exp(g[0, t, 0]))
        P = A @ P
    assert np.allclose(M[0, 0], P, rtol=1e-12, atol=1e-13)


def test_dropping_the_zero_value_run_breaks_composition():
    # A composition that forgets E (or takes M from the run with values) must
    # fail: the check above is not vacuous.
    T, H, d = 20, 1, 3
    rng = np.random.default_rng(9)
    q, k, v, g, beta = _inputs(rng, T, H, d)
    S0 = rng.normal(size=(1, H, d, d))
    _, S_full = oracle.scan(q, k, v, g, beta, 0.3, S0)
    M, E = _maps(q, k, v, g, beta, 0, T, H, d)
    assert np.allclose(M @ S0 + E, S_full, rtol=1e-12, atol=1e-12)
    assert not np.allclose(M @ S0, S_full, rtol=1e-6, atol=1e-6)
    eye = np.eye(d).reshape(1, 1, d, d)
    M_wrong = _run(q, k, v, g, beta, eye, 0, T)[1]
    assert not np.allclose(M_wrong @ S0 + E, S_full, rtol=1e-6, atol=1e-6)
