"""Output gate and RMS normalisation of the token outputs, in fp64.

TEST INFRASTRUCTURE, like everything under oracle/.

The module around the scan gates and RMS-normalises each head's output
("Understanding Kimi Delta Attention", closing remarks: output gating and RMS
normalisation). The pages give no formula; the reading used is the usual one,
normalisation first over the d_v channels of one head, then a per-channel
weight and a sigmoid gate:

    out = w * o / sqrt(mean_c o_c^2 + eps) * sigmoid(z)

Parity status: pinned by tests/test_oracle_prologue_pins.py (a worked 3-4
example, constant rows, the gate's midpoint and limits, linearity in w).
"""
import numpy as np


def output_gate_rmsnorm(o, z, weight=None, eps=1e-6):
    o = np.asarray(o, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    w = 1.0 if weight is None else np.asarray(weight, dtype=np.float64)
    return w * o * r / (1.0 + np.exp(-z))
