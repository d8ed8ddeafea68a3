"""Shared test helpers: running the oracle on the same (rounded) inputs the GPU
sees, and the parity tolerances.

Tolerances (stated for the method's parity target): fp32 storage: max |error|
<= 1e-4 on the outputs and on the final state. bf16 storage with fp32 state:
max |error| <= 2e-2 and relative Frobenius error <= 5e-3, each checked
separately for the outputs and for the final state.
"""
import numpy as np
import torch

import oracle

F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 5e-3


def f64(t):
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_prefill(inp, heads=None, nthreads=0):
    """Oracle outputs for a make_prefill() input dict, optionally on a subset of
    heads (the heads are independent, so a subset is an exact sample)."""
    sel = slice(None) if heads is None else list(heads)

    def pick(t, axis):
        if t is None:
            return None
        a = f64(t)
        return a if heads is None else np.take(a, sel, axis=axis)

    q, k, v, g = (pick(inp[n], 2) for n in ("q", "k", "v", "g"))
    beta = pick(inp["beta"], 2)
    init = pick(inp["init_state"], 1)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].numpy().astype(np.int64)
    return oracle.scan(q, k, v, g, beta, inp["scale"], init, cu, nthreads=nthreads)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = got - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d) / nref) if nref > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_parity(got, ref, storage, what):
    max_abs, rel = errors(got, ref)
    if storage == "f32":
        assert max_abs <= F32_MAX_ABS, "%s: max|err| %.3g > %.1g" % (what, max_abs, F32_MAX_ABS)
    else:
        assert max_abs <= BF16_MAX_ABS, "%s: max|err| %.3g > %.1g" % (what, max_abs, BF16_MAX_ABS)
        assert rel <= BF16_REL_FRO, "%s: rel Frobenius %.3g > %.1g" % (what, rel, BF16_REL_FRO)
    return max_abs, rel
