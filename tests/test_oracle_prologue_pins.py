"""Pins of the oracle's prologue (oracle/prologue.py) against closed forms,
limits and special cases, independent of the oracle's own code paths:

* the log-sigmoid gate against the sigmoid's definition a = 1 / (1 + e^-z)
  ("Kimi Delta Attention: a half-life per channel", "Promote the scalar to a
  diagonal"), including far into both tails;
* the bounded gate's midpoint, range and limits;
* L2 normalisation on a 3-4-5 example, on zero vectors, and the scan's
  invariance under rescaling q and k when normalisation is on;
* the scalar-decay family against a two-token closed form of the gated delta
  rule with orthonormal keys (the decay multiplies the earlier write only),
  per head with different decays ("Kimi Delta Attention: How It Works, Step by
  Step", section 6);
* the no-decay family (DeltaNet) against the same closed form with a = 1.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.prologue import L2_EPS, l2normalize, log_decay, prepare


def test_logsigmoid_is_log_of_sigmoid():
    for z in (-30.0, -5.0, -1.0, -1e-3, 0.0, 0.5, 3.0, 40.0):
        a = 1.0 / (1.0 + math.exp(-z))
        assert float(np.exp(log_decay(z, "logsigmoid"))) == pytest.approx(a, rel=1e-12)
    # Far tails stay finite: log sigmoid(-800) = -800 - log(1 + e^-800), log sigmoid(800) -> 0-.
    assert float(log_decay(-800.0, "logsigmoid")) == pytest.approx(-800.0, rel=1e-12)
    assert -1e-300 <= float(log_decay(800.0, "logsigmoid")) <= 0.0
    assert float(log_decay(0.0, "logsigmoid")) == pytest.approx(-math.log(2.0), rel=1e-15)


def test_bounded_gate():
    lo = -5.0
    assert float(log_decay(0.0, "bounded", lo)) == pytest.approx(-2.5, rel=1e-15)
    assert float(log_decay(60.0, "bounded", lo)) == pytest.approx(lo, rel=1e-12)
    assert abs(float(log_decay(-60.0, "bounded", lo))) < 1e-20
    z = np.linspace(-8, 8, 33)
    g = log_decay(z, "bounded", lo)
    assert np.all((g > lo) & (g < 0)) and np.all(np.diff(g) < 0)


def test_log_gate_is_identity():
    z = np.array([-3.0, -0.25, 0.0])
    assert np.array_equal(log_decay(z, "log"), z)


def test_l2normalize_examples():
    x = np.array([[3.0, 4.0], [0.0, 0.0]])
    y = l2normalize(x)
    assert y[0] == pytest.approx([3.0 / math.sqrt(25 + L2_EPS), 4.0 / math.sqrt(25 + L2_EPS)], rel=1e-15)
    assert np.array_equal(y[1], [0.0, 0.0])
    r = np.random.default_rng(0).normal(size=(5, 3, 16)) * 7.0
    assert np.linalg.norm(l2normalize(r), axis=-1) == pytest.approx(1.0, rel=1e-6)


def test_normalised_scan_ignores_q_k_scale():
    rng = np.random.default_rng(1)
    B, T, H, d = 1, 9, 2, 4
    q, k, v = (rng.normal(size=(B, T, H, d)) for _ in range(3))
    z = rng.normal(size=(B, T, H, d))
    beta = rng.uniform(0, 1, size=(B, T, H))
    base = oracle.scan(*prepare(q, k, z, gate="logsigmoid", l2norm_qk=True)[:2], v,
                       prepare(q, k, z, gate="logsigmoid")[2], beta, 0.5)
    # Scales >= 1 keep the epsilon of the norm below ~3e-7 of the sum of squares.
    s = rng.uniform(1.0, 10.0, size=(B, T, H, 1))
    q2, k2, g2 = prepare(q * s, k * s[..., ::-1, :] * 3.0, z, gate="logsigmoid", l2norm_qk=True)
    other = oracle.scan(q2, k2, v, g2, beta, 0.5)
    for a, b in zip(base, other):
        assert np.allclose(a, b, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("decay", ["scalar", "none"])
def test_scalar_and_no_decay_two_token_closed_form(decay):
    # Two tokens, orthonormal keys k1 = e1, k2 = e2, query q2 = e1 + e2:
    #   S1 = b1 k1 v1^T;  S2 = a2 S1 + b2 k2 (v2 - a2 S1^T k2)^T = a2 b1 e1 v1^T + b2 e2 v2^T
    #   o2 = s S2^T q2 = s (a2 b1 v1 + b2 v2),  o1 = s b1 (k1 . q1) v1.
    d, H, s = 4, 2, 0.7
    e = np.eye(d)
    rng = np.random.default_rng(2)
    v = rng.normal(size=(1, 2, H, d))
    beta = np.array([[[0.3, 0.9], [0.6, 0.25]]])              # [1, 2 tokens, H]
    q = np.zeros((1, 2, H, d)); k = np.zeros((1, 2, H, d))
    q[0, 0, :] = e[0] * 2.0
    q[0, 1, :] = e[0] + e[1]
    k[0, 0, :] = e[0]
    k[0, 1, :] = e[1]
    loga2 = np.array([-0.4, -2.0])                            # a different decay per head
    g = np.zeros((1, 2, H))
    g[0, 1] = loga2
    g[0, 0] = [-7.0, -1.5]                                     # decays of the first token touch nothing
    out, fin = oracle.scan(*prepare(q, k, g, decay=decay)[:2], v,
                           prepare(q, k, g, decay=decay)[2], beta, s)
    for h in range(H):
        a2 = math.exp(loga2[h]) if decay == "scalar" else 1.0
        b1, b2 = beta[0, 0, h], beta[0, 1, h]
        v1, v2 = v[0, 0, h], v[0, 1, h]
        assert out[0, 0, h] == pytest.approx(s * b1 * 2.0 * v1, rel=1e-12, abs=1e-14)
        assert out[0, 1, h] == pytest.approx(s * (a2 * b1 * v1 + b2 * v2), rel=1e-12, abs=1e-14)
        S2 = a2 * b1 * np.outer(e[0], v1) + b2 * np.outer(e[1], v2)
        assert fin[0, h] == pytest.approx(S2, rel=1e-12, abs=1e-14)


def test_prepare_shapes_and_broadcast():
    q = np.ones((2, 3, 4, 8))
    gh = np.arange(2 * 3 * 4, dtype=float).reshape(2, 3, 4) * -0.1
    _, _, gc = prepare(q, q, gh, decay="scalar")
    assert gc.shape == q.shape and np.array_equal(gc[..., 5], gh)
    _, _, g0 = prepare(q, q, None, decay="none")
    assert not g0.any()
    with pytest.raises(ValueError):
        prepare(q, q, gh, decay="channel")


def test_output_gate_rmsnorm_pins():
    from oracle.epilogue import output_gate_rmsnorm
    eps = 1e-6
    # Worked example: o = [3, 4], mean square 12.5; z = 0 halves; z -> +inf keeps.
    got = output_gate_rmsnorm(np.array([3.0, 4.0]), np.array([0.0, 60.0]), eps=eps)
    r = 1.0 / math.sqrt(12.5 + eps)
    assert got == pytest.approx([0.5 * 3.0 * r, 4.0 * r], rel=1e-12)
    # A constant row normalises to +-1 (up to eps); z -> -inf closes the gate.
    c = output_gate_rmsnorm(np.full(8, -2.5), np.full(8, 60.0), eps=eps)
    assert c == pytest.approx(-1.0, rel=1e-6)
    assert np.all(np.abs(output_gate_rmsnorm(np.ones(4), np.full(4, -60.0))) < 1e-25)
    # Linear in the weight, per channel.
    rng = np.random.default_rng(3)
    o, z, w = rng.normal(size=(5, 16)), rng.normal(size=(5, 16)), rng.normal(size=16)
    assert output_gate_rmsnorm(o, z, w) == pytest.approx(w * output_gate_rmsnorm(o, z), rel=1e-12)
    # Each row's mean square after normalisation (gate open) is 1.
    y = output_gate_rmsnorm(o * 7.0, np.full_like(o, 60.0))
    assert np.mean(y * y, axis=-1) == pytest.approx(1.0, rel=1e-6)
