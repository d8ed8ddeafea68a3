"""The input prologue of the scan and its decay families, in fp64.

TEST INFRASTRUCTURE, like everything under oracle/: only tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline leg may use it.

``prepare`` turns the options of kda_chunk_fwd_opt / kda_decode_step_opt into
the plain inputs of ``oracle.scan``: normalised q and k, and the per-channel
log-decay log a_t.

* L2 normalisation of q and k per token and head ("Kimi Delta Attention: How
  It Works, Step by Step", section 16: the key and query are normalised);
  the definition used is x / sqrt(sum_c x_c^2 + eps), eps = 1e-6 (the pages
  give no epsilon).
* Decay gates: a_t = sigmoid(z) ("Kimi Delta Attention: a half-life per
  channel", "Promote the scalar to a diagonal"), so log a_t = log sigmoid(z);
  or a log-decay bounded below through a sigmoid ("Understanding Kimi Delta
  Attention", closing remarks), read as log a_t = lower * sigmoid(z).
* Decay families: per channel (KDA), one scalar per head (Gated DeltaNet:
  "Kimi Delta Attention: How It Works, Step by Step", section 6; the scalar
  decay multiplies the whole state, i.e. every key channel alike), none
  (DeltaNet, a_t = 1).

Parity status: pinned by tests/test_oracle_pins.py (closed forms of the gates,
unit norms, scale invariance, and a two-token closed form of the scalar-decay
recurrence per head).
"""
import numpy as np

L2_EPS = 1e-6


def l2normalize(x, eps=L2_EPS):
    """x / sqrt(sum of squares over the last axis + eps), in fp64."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def log_decay(z, gate="log", lower=-5.0):
    """log a_t from the values z stored in g, in fp64.

    "log": z is log a_t.  "logsigmoid": a_t = 1 / (1 + e^-z), computed as
    min(z, 0) - log(1 + e^-|z|) so that no exponential overflows.
    "bounded": log a_t = lower / (1 + e^-z), between lower and 0.
    """
    z = np.asarray(z, dtype=np.float64)
    if gate == "log":
        return z
    if gate == "logsigmoid":
        return np.minimum(z, 0.0) - np.log1p(np.exp(-np.abs(z)))
    if gate == "bounded":
        return lower / (1.0 + np.exp(-z))
    raise ValueError("unknown gate %r" % (gate,))


def prepare(q, k, g, decay="channel", gate="log", gate_lower=-5.0, l2norm_qk=False):
    """(q, k, g_channel) for oracle.scan / oracle.decode_step.

    q, k ``[..., H, d_k]``. g: ``[..., H, d_k]`` for "channel", ``[..., H]``
    for "scalar" (broadcast to every key channel of its head), ignored for
    "none" (log a_t = 0).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if l2norm_qk:
        q = l2normalize(q)
        k = l2normalize(k)
    if decay == "channel":
        gc = log_decay(g, gate, gate_lower)
        if gc.shape != q.shape:
            raise ValueError("per-channel g must have q's shape")
    elif decay == "scalar":
        gh = log_decay(g, gate, gate_lower)
        if gh.shape != q.shape[:-1]:
            raise ValueError("per-head g must have q's shape without its last axis")
        gc = np.broadcast_to(gh[..., None], q.shape).copy()
    elif decay == "none":
        gc = np.zeros(q.shape, dtype=np.float64)
    else:
        raise ValueError("unknown decay %r" % (decay,))
    return q, k, gc
