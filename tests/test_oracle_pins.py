"""Pins the oracle to facts other than itself: worked examples the pages print,
closed forms, special cases that reduce to simpler rules, identities of the
chunkwise derivation, and agreement between three independent formulations.

Each test names the mistake it is there to catch. All run on CPU.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle.chunkwise import chunk_factors, chunkwise_scan
from oracle.dense import dense_scan, transition

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def rand_inputs(rng, B, T, H, dk, dv, init=True, gate_shift=2.0):
    q = rng.standard_normal((B, T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H, dk)) - gate_shift))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    S0 = 0.3 * rng.standard_normal((B, H, dk, dv)) if init else None
    return q, k, v, g, beta, S0


def one_token(S0, k, v, beta, a, q=None, scale=1.0):
    """Runs the oracle scan on a single token of a single head."""
    k = np.asarray(k, float)
    q = k if q is None else np.asarray(q, float)
    dk, dv = np.asarray(S0).shape
    g = np.log(np.broadcast_to(np.asarray(a, float), (dk,)))
    out, fin = oracle.scan(q[None, None, None], k[None, None, None],
                           np.asarray(v, float)[None, None, None], g[None, None, None],
                           np.array([[[beta]]]), scale, np.asarray(S0, float)[None, None])
    return out[0, 0, 0], fin[0, 0]


# ---------------------------------------------------------------- worked examples

def test_fig01_delta_write_reads_value_not_sum():
    """Figure 01 of "Understanding Kimi Delta Attention": a memory reading 2 at
    a unit key, written with value 2, reads 4 under an additive write; the
    delta rule with beta = 1 reads 2. Catches an additive (linear-attention)
    write in place of the corrective one."""
    ex = GOLDEN["additive_vs_delta_write"]
    rng = np.random.default_rng(1)
    dk, dv = 5, 3
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    # Any state whose read at k is 2 in every value channel.
    S0 = rng.standard_normal((dk, dv))
    S0 += np.outer(k, ex["read_before"] - S0.T @ k)
    assert np.allclose(S0.T @ k, ex["read_before"])
    o, _ = one_token(S0, k, np.full(dv, ex["value_written"]), 1.0, 1.0)
    assert np.allclose(o, ex["delta_rule_beta1_read_after"], atol=1e-12)
    # The additive write of the same value would read the page's 4.
    additive = (S0 + np.outer(k, np.full(dv, ex["value_written"]))).T @ k
    assert np.allclose(additive, ex["additive_read_after"])
    assert not np.allclose(o, ex["additive_read_after"])


def test_try_it_with_numbers_halfway_correction():
    """"Try it with numbers": prediction 2, target 6, beta 0.5 -> error 4,
    next prediction 4. Catches a wrong beta placement or a write of v
    instead of the error."""
    ex = GOLDEN["halfway_correction"]
    o, S = one_token([[ex["prediction"]]], [1.0], [ex["target"]], ex["beta"], 1.0)
    assert o[0] == pytest.approx(ex["next_prediction"], abs=1e-14)
    assert ex["target"] - ex["prediction"] == ex["error"]


def test_decay_range_order_of_magnitude():
    """"What changes in the kernel": with a = 0.9 the inverse cumulative decay
    1/gamma reaches ~1e3 over 64 positions and ~1e6 over 128. Run with
    beta = 0 (pure decay) and read the state ratio. Catches decay applied
    per token more or fewer times than once."""
    ex = GOLDEN["decay_range_a0p9"]
    for case in ex["inverse_gamma_order_of_magnitude"]:
        T = case["positions"]
        dk = dv = 2
        g = np.full((1, T, 1, dk), np.log(ex["a"]))
        S0 = np.ones((1, 1, dk, dv))
        _, fin = oracle.scan(np.zeros((1, T, 1, dk)), np.zeros((1, T, 1, dk)),
                             np.zeros((1, T, 1, dv)), g, np.zeros((1, T, 1)), 1.0, S0)
        ratio = fin[0, 0, 0, 0]  # gamma: the part of the initial state kept after T tokens
        assert 0.0 < ratio < 1.0
        assert round(-np.log10(ratio)) == case["log10"]  # log10(1 / gamma)


def test_half_lives():
    """Opening of "a half-life per channel": a = 0.9999 keeps half of a fact
    for about seven thousand tokens; a = 0.9 for under seven. The half-life
    is read off the oracle's pure-decay run (beta = 0): after T tokens the
    state keeps a ratio r, so the half-life is T ln 2 / (-ln r)."""
    slow, fast = GOLDEN["half_lives"]["cases"]

    def half_life(a, T):
        g = np.full((1, T, 1, 1), np.log(a))
        out, fin = oracle.scan(np.ones((1, T, 1, 1)), np.zeros((1, T, 1, 1)),
                               np.zeros((1, T, 1, 1)), g, np.zeros((1, T, 1)), 1.0,
                               np.ones((1, 1, 1, 1)))
        r = fin[0, 0, 0, 0]
        assert out[0, -1, 0, 0] == pytest.approx(r, rel=1e-15)
        assert 0.0 < r < 1.0  # a strict decay keeps part of the state
        return T * np.log(2.0) / -np.log(r)

    hl = half_life(slow["a"], 1000)
    assert abs(hl - slow["approx_tokens"]) <= slow["rel_band"] * slow["approx_tokens"]
    assert half_life(fast["a"], 20) < fast["below_tokens"]


def test_naive_decay_tensor_size_claim():
    """The page's ~500 000 is the element count of a C x C x d_k pair tensor
    for C = 64, d_k = 128 (exactly 524 288); the chunkwise oracle builds
    exactly that tensor per chunk."""
    ex = GOLDEN["naive_pair_decay_tensor"]
    n = ex["C"] * ex["C"] * ex["d_k"]
    assert abs(n - ex["approx_elements"]) / ex["approx_elements"] < 0.05


# ---------------------------------------------------------------- closed forms

def test_overwrite_beta1_any_decay():
    """"Does the write work?": with beta = 1 and a unit key the updated state
    returns v exactly at that key, whatever the per-channel decay, because the
    decay happens before the prediction. Catches decay applied after the write
    and predictions against the undecayed state."""
    rng = np.random.default_rng(2)
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, 24, 2, 6, 4)
    beta[:] = 1.0
    # Query each token with its own key, scale 1: o_t = S_t^T k_t.
    out, _ = oracle.scan(k, k, v, g, beta, 1.0, S0)
    assert np.allclose(out, v, atol=1e-12)


def test_overwrite_general_beta_moves_partway():
    """"Does the write work?": S_t^T k_t = (1 - beta) vhat + beta v, with vhat
    the prediction of the decayed state. Catches a beta applied twice or to
    the wrong term."""
    rng = np.random.default_rng(3)
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, 9, 1, 5, 3)
    t = 8
    _, S_prev = oracle.scan(k[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t], 1.0, S0)
    vhat = (np.exp(g[0, t, 0])[:, None] * S_prev[0, 0]).T @ k[0, t, 0]
    out, _ = oracle.scan(k[:, : t + 1], k[:, : t + 1], v[:, : t + 1], g[:, : t + 1],
                         beta[:, : t + 1], 1.0, S0)
    b = beta[0, t, 0]
    assert np.allclose(out[0, t, 0], (1 - b) * vhat + b * v[0, t, 0], atol=1e-12)


def test_beta0_pure_decay_closed_form():
    """With beta = 0 nothing is written: S_t = Diag(prod_{r<=t} a_r) S_0 and
    o_t = S_t^T (scale q_t). Uses d_k != d_v and a non-symmetric S_0, so it
    catches decay applied to value columns instead of key rows, a transposed
    read, a wrong exp sign, and the scale applied anywhere but q."""
    rng = np.random.default_rng(4)
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, 11, 2, 6, 3)
    beta[:] = 0.0
    scale = 0.37
    out, fin = oracle.scan(q, k, v, g, beta, scale, S0)
    cum = np.cumsum(g[0], axis=0)                       # [T, H, dk]
    for h in range(2):
        for t in range(11):
            S_t = np.exp(cum[t, h])[:, None] * S0[0, h]
            assert np.allclose(out[0, t, h], S_t.T @ (scale * q[0, t, h]), atol=1e-12)
        assert np.allclose(fin[0, h], np.exp(cum[-1, h])[:, None] * S0[0, h], atol=1e-12)


def test_deltanet_orthonormal_dictionary():
    """a = 1 (no decay) is DeltaNet ("Learning to overwrite"). With orthonormal
    keys and beta = 1 the memory is an exact dictionary: each key reads the
    last value written at it, and keys never written read the initial state."""
    rng = np.random.default_rng(5)
    dk, dv = 8, 3
    Q, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Q.T                                        # rows are orthonormal keys
    order = [0, 3, 5, 3, 1, 0]                        # keys 3 and 0 rewritten
    T = len(order)
    k = keys[order][None, :, None, :]
    v = rng.standard_normal((1, T, 1, dv))
    S0 = rng.standard_normal((1, 1, dk, dv))
    _, fin = oracle.scan(k, k, v, np.zeros((1, T, 1, dk)), np.ones((1, T, 1)), 1.0, S0)
    last = {key: t for t, key in enumerate(order)}
    for key in range(dk):
        read = fin[0, 0].T @ keys[key]
        expect = v[0, last[key], 0] if key in last else S0[0, 0].T @ keys[key]
        assert np.allclose(read, expect, atol=1e-12)


def test_gated_deltanet_is_rescaled_deltanet():
    """With a decay constant across channels (Gated DeltaNet, "Learning what to
    forget"), S_t = gamma_t S'_t where S' is DeltaNet (a = 1) run on values
    v_t / gamma_t and gamma_t = prod_{r<=t} alpha_r. The identity holds only if
    the decay multiplies the whole state before the prediction, so it catches
    decay-after-predict and decay on the write."""
    rng = np.random.default_rng(6)
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, 17, 1, 5, 4)
    alpha_log = g[..., :1]                             # one decay per token
    g_scalar = np.broadcast_to(alpha_log, g.shape).copy()
    scale = 0.5
    out_gdn, fin_gdn = oracle.scan(q, k, v, g_scalar, beta, scale, S0)
    gamma = np.exp(np.cumsum(alpha_log[0, :, 0, 0]))   # [T]
    v_resc = v / gamma[None, :, None, None]
    out_dn, fin_dn = oracle.scan(q, k, v_resc, np.zeros_like(g), beta, scale, S0)
    assert np.allclose(out_gdn, gamma[None, :, None, None] * out_dn, atol=1e-12)
    assert np.allclose(fin_gdn, gamma[-1] * fin_dn, atol=1e-12)


def test_linearity_in_values_and_state():
    """For fixed keys, queries, decays and write strengths the map
    (V, S_0) -> (O, S_T) is linear, and O is proportional to the query scale."""
    rng = np.random.default_rng(7)
    q, k, v1, g, beta, S1 = rand_inputs(rng, 2, 13, 2, 4, 3)
    v2 = rng.standard_normal(v1.shape)
    S2 = rng.standard_normal(S1.shape)
    a, b = 0.7, -1.3
    o1, f1 = oracle.scan(q, k, v1, g, beta, 0.5, S1)
    o2, f2 = oracle.scan(q, k, v2, g, beta, 0.5, S2)
    o3, f3 = oracle.scan(q, k, a * v1 + b * v2, g, beta, 0.5, a * S1 + b * S2)
    assert np.allclose(o3, a * o1 + b * o2, atol=1e-12)
    assert np.allclose(f3, a * f1 + b * f2, atol=1e-12)
    o4, f4 = oracle.scan(q, k, v1, g, beta, 1.5, S1)
    assert np.allclose(o4, 3.0 * o1, atol=1e-12)
    assert np.allclose(f4, f1, atol=0)


# ---------------------------------------------------------------- dense DPLR form

def test_two_transition_expansion():
    """"Two transitions already reveal the pattern": F2 F1 = I - b1 k1 k1^T -
    b2 k2 k2^T + b2 b1 k2 (k2^T k1) k1^T (no decay). Pins the dense module."""
    rng = np.random.default_rng(8)
    k1, k2 = rng.standard_normal(5), rng.standard_normal(5)
    b1, b2 = 0.3, 0.8
    lhs = transition(k2, np.zeros(5), b2) @ transition(k1, np.zeros(5), b1)
    rhs = (np.eye(5) - b1 * np.outer(k1, k1) - b2 * np.outer(k2, k2)
           + b2 * b1 * np.outer(k2, k1) * (k2 @ k1))
    assert np.allclose(lhs, rhs, atol=1e-14)


def test_decay_and_rank_one_do_not_commute():
    """"KDA as a structured state transition": D and k k^T generally do not
    commute, so (I - b k k^T) D != D (I - b k k^T). Catches a transition built
    with the factors swapped (the dense module must use (I - b k k^T) D)."""
    rng = np.random.default_rng(9)
    k = rng.standard_normal(4)
    g = np.log(np.array([0.9, 0.5, 0.2, 0.99]))
    F = transition(k, g, 0.7)
    assert np.allclose(F, (np.eye(4) - 0.7 * np.outer(k, k)) @ np.diag(np.exp(g)))
    assert not np.allclose(F, np.diag(np.exp(g)) @ (np.eye(4) - 0.7 * np.outer(k, k)))


def test_scan_matches_dense_transition_products():
    """The token scan equals the explicit product of (I - b k k^T) D
    transitions plus accumulated writes, on tiny T."""
    rng = np.random.default_rng(10)
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, 7, 2, 5, 4)
    out, fin = oracle.scan(q, k, v, g, beta, 0.8, S0)
    for h in range(2):
        o_d, S_d = dense_scan(q[0, :, h], k[0, :, h], v[0, :, h], g[0, :, h], beta[0, :, h],
                              0.8, S0[0, h])
        assert np.allclose(out[0, :, h], o_d, atol=1e-12)
        assert np.allclose(fin[0, h], S_d, atol=1e-12)


# ---------------------------------------------------------------- chunkwise form

@pytest.mark.parametrize("C", [1, 3, 8, 16, 32, 64])
def test_chunkwise_equals_scan(C):
    """Figure 04: chunkwise processing with a carried state gives the token
    recurrence's result, for chunk sizes that divide T and ones that leave a
    ragged last chunk."""
    rng = np.random.default_rng(11)
    q, k, v, g, beta, S0 = rand_inputs(rng, 2, 70, 2, 6, 5)
    o1, f1 = oracle.scan(q, k, v, g, beta, 0.6, S0)
    o2, f2 = chunkwise_scan(q, k, v, g, beta, 0.6, S0, C=C)
    assert np.allclose(o1, o2, atol=1e-11)
    assert np.allclose(f1, f2, atol=1e-11)


def test_nilpotent_series_and_unit_triangular():
    """"The triangular system appears": A is strictly lower triangular, so
    A^C = 0 and (I - A)^{-1} = I + A + ... + A^{C-1}. Pins the solve."""
    rng = np.random.default_rng(12)
    n, dk = 12, 6
    k = rng.standard_normal((n, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    g = -np.log1p(np.exp(rng.standard_normal((n, dk))))
    beta = rng.uniform(0, 1, n)
    _, A, T = chunk_factors(k, g, beta)
    assert np.allclose(np.triu(A), 0)
    assert np.allclose(np.linalg.matrix_power(A, n), 0, atol=1e-14)
    series = sum(np.linalg.matrix_power(A, p) for p in range(n))
    assert np.allclose(T, series, atol=1e-12)
    # Entry check of one coefficient against its definition with explicit decay.
    i, j = 7, 3
    Gam = np.exp(np.cumsum(g, 0))
    assert A[i, j] == pytest.approx(-beta[i] * k[i] @ (Gam[i] / Gam[j] * k[j]), rel=1e-12)


def test_wy_identity_without_decay():
    """"Where did WY go?": with every retention factor 1 the boundary update is
    S_out = (I - K^T T B K) S_0 + K^T T B V."""
    rng = np.random.default_rng(13)
    n, dk, dv = 10, 6, 4
    q, k, v, _, beta, S0 = rand_inputs(rng, 1, n, 1, dk, dv)
    k, v, beta, S0 = k[0, :, 0], v[0, :, 0], beta[0, :, 0], S0[0, 0]
    _, _, T = chunk_factors(k, np.zeros((n, dk)), beta)
    Bm = np.diag(beta)
    expect = (np.eye(dk) - k.T @ T @ Bm @ k) @ S0 + k.T @ T @ Bm @ v
    _, fin = oracle.scan(k[None, :, None], k[None, :, None],
                         v[None, :, None], np.zeros((1, n, 1, dk)), beta[None, :, None], 1.0,
                         S0[None, None])
    assert np.allclose(fin[0, 0], expect, atol=1e-12)


def test_first_corrections_unrolled():
    """"First correction" and "Second correction": z_1 = b_1 (v_1 - S_0^T
    Gamma_1 k_1) and z_2 = b_2 (v_2 - S_0^T Gamma_2 k_2) - b_2 (k_2^T
    Gamma_{1->2} k_1) z_1; the state after two tokens is Gamma_2 S_0 +
    Gamma_{1->2} k_1 z_1^T + k_2 z_2^T."""
    rng = np.random.default_rng(14)
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, 2, 1, 5, 3)
    k1, k2 = k[0, 0, 0], k[0, 1, 0]
    v1, v2 = v[0, 0, 0], v[0, 1, 0]
    b1, b2 = beta[0, 0, 0], beta[0, 1, 0]
    G1 = np.exp(g[0, 0, 0])
    G2 = G1 * np.exp(g[0, 1, 0])
    G12 = np.exp(g[0, 1, 0])
    S = S0[0, 0]
    z1 = b1 * (v1 - S.T @ (G1 * k1))
    z2 = b2 * (v2 - S.T @ (G2 * k2)) - b2 * (k2 @ (G12 * k1)) * z1
    S2 = G2[:, None] * S + np.outer(G12 * k1, z1) + np.outer(k2, z2)
    _, fin = oracle.scan(q, k, v, g, beta, 1.0, S0)
    assert np.allclose(fin[0, 0], S2, atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_varlen_packed_equals_separate():
    """Packed sequences (cu_seqlens) give the same results as separate runs;
    a zero-length sequence returns its initial state."""
    rng = np.random.default_rng(15)
    lens = [5, 0, 9, 1]
    T = sum(lens)
    q, k, v, g, beta, _ = rand_inputs(rng, 1, T, 2, 4, 3)
    S0 = rng.standard_normal((len(lens), 2, 4, 3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    out, fin = oracle.scan(q, k, v, g, beta, 0.5, S0, cu_seqlens=cu)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        o_n, f_n = oracle.scan(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], beta[:, s:e], 0.5,
                               S0[n:n + 1])
        assert np.allclose(out[:, s:e], o_n, atol=0)
        assert np.allclose(fin[n], f_n[0], atol=0)
    assert np.array_equal(fin[1], S0[1])


def test_split_resume_equals_whole():
    """Feeding one run's final state as the next run's initial state continues
    the sequence exactly (the state is the whole checkpoint)."""
    rng = np.random.default_rng(16)
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, 30, 2, 4, 4)
    o, f = oracle.scan(q, k, v, g, beta, 0.5, S0)
    oa, fa = oracle.scan(q[:, :13], k[:, :13], v[:, :13], g[:, :13], beta[:, :13], 0.5, S0)
    ob, fb = oracle.scan(q[:, 13:], k[:, 13:], v[:, 13:], g[:, 13:], beta[:, 13:], 0.5, fa)
    assert np.allclose(np.concatenate([oa, ob], 1), o, atol=0)
    assert np.allclose(fb, f, atol=0)


def test_decode_steps_equal_prefill():
    """T single-token decode steps reproduce a T-token prefill."""
    rng = np.random.default_rng(17)
    q, k, v, g, beta, S0 = rand_inputs(rng, 3, 6, 2, 4, 5)
    o, f = oracle.scan(q, k, v, g, beta, 0.5, S0)
    S = S0
    for t in range(6):
        ot, S = oracle.decode_step(q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], 0.5, S)
        assert np.allclose(ot, o[:, t], atol=0)
    assert np.allclose(S, f, atol=0)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(18)
    q, k, v, g, beta, S0 = rand_inputs(rng, 3, 20, 4, 4, 4)
    a = oracle.scan(q, k, v, g, beta, 0.5, S0, nthreads=1)
    b = oracle.scan(q, k, v, g, beta, 0.5, S0, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
