"""GPU parity at the method's edges, against the fp64 oracle, on every path:
the tensor-core prefill (bf16, d = 128), the fp32 prefill (fp32 storage or
d = 64) and the decode step.

The decay may be any a in (0, 1] ("Understanding Kimi Delta Attention", box
"KDA: Retain, predict, correct"), so the inputs include per-token log-decays
down to -40 (far steeper than a factor spanning several tokens can carry in
fp32), gate logits whose log-sigmoid reaches the same range, heads with
beta = 0 (pure decay), beta = 1 with unit keys (the overwrite case of "Does
the write work?"), a = 1 (DeltaNet), and heads that mix steep and gentle
tokens; with ragged tails and packed sequences. Every output must be finite
and within the parity tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.prologue import prepare
from kimi_delta_attention_17_gb300 import build, chunk_fwd, decode_step, workspace_size
from kimi_delta_attention_17_gb300.inputs import (EDGE_KINDS, DecodeSpec, PrefillSpec,
                                                  make_decode_edge, make_prefill,
                                                  make_prefill_edge, steep_logits)
from tests.helpers import assert_parity, errors, f64

pytestmark = pytest.mark.gpu

PACKED = (0, 1, 63, 64, 65, 130, 200, 17, 300)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def gpu_prefill(inp, **opts):
    dev = "cuda"
    q, k, v, beta = (inp[n].to(dev) for n in ("q", "k", "v", "beta"))
    g = None if inp["g"] is None else inp["g"].to(dev)
    init = None if inp["init_state"] is None else inp["init_state"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    B, T, H, d = q.shape
    ws = torch.empty(max(1, workspace_size(B, T, H, d, d, len(inp["lengths"]), q.dtype)),
                     dtype=torch.uint8, device=dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], init, cu, workspace=ws, **opts)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    return f64(out), f64(fin)


def oracle_prefill(inp, **opts):
    q, k, g = prepare(f64(inp["q"]), f64(inp["k"]), f64(inp["g"]), **opts)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].numpy().astype(np.int64)
    return oracle.scan(q, k, f64(inp["v"]), g, f64(inp["beta"]), inp["scale"],
                       f64(inp["init_state"]), cu)


def check(got, ref, storage, what):
    assert np.isfinite(got).all(), "%s: non-finite values" % what
    assert_parity(got, ref, storage, what)
    # every head kind on its own, by the max-abs bound of its storage
    bound = 1e-4 if storage == "f32" else 2e-2
    H = got.shape[-3] if what.startswith("final") else got.shape[-2]
    for h in range(H):
        sel = (slice(None), h) if what.startswith("final") else (Ellipsis, h, slice(None))
        m, _ = errors(got[sel], ref[sel])
        assert m <= bound, "%s, head %d (%s): max|err| %.3g" % (
            what, h, EDGE_KINDS[h % len(EDGE_KINDS)], m)


def edge_case(d, dtype, packed=True, seed=40, H=6):
    if packed:
        return PrefillSpec("edge packed", H=H, d=d, fixed_lengths=PACKED, dtype=dtype,
                           init="normal0.1", seed=seed)
    return PrefillSpec("edge batch", H=H, d=d, B=2, T=300, dtype=dtype, init="normal0.1",
                       seed=seed)


@pytest.mark.parametrize("packed", [True, False], ids=["packed", "batch"])
@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "bf16"), (64, "f32"), (128, "f32")])
def test_prefill_edge_heads(d, dtype, packed):
    """Steep, beta = 0, beta = 1, a = 1, mixed and base heads on each prefill
    path (bf16 at d = 128 is the tensor-core path)."""
    inp = make_prefill_edge(edge_case(d, dtype, packed))
    out, fin = gpu_prefill(inp)
    ref_out, ref_fin = oracle_prefill(inp)
    check(out, ref_out, dtype, "O")
    check(fin, ref_fin, dtype, "final state")


def test_tensor_core_segments_with_steep_heads():
    """The segmented state pass (chunk-level parallel prefix) over the same
    head kinds: 8 chunks in 3 segments."""
    spec = PrefillSpec("edge segments", H=6, d=128, B=1, T=500, init="normal0.1", seed=41)
    inp = make_prefill_edge(spec)
    out, fin = gpu_prefill(inp, segments=3)
    ref_out, ref_fin = oracle_prefill(inp)
    check(out, ref_out, "bf16", "O")
    check(fin, ref_fin, "bf16", "final state")


@pytest.mark.parametrize("d,dtype,l2", [(128, "bf16", False), (128, "bf16", True),
                                        (64, "f32", False), (64, "bf16", True)])
def test_prefill_logsigmoid_steep_logits(d, dtype, l2):
    """Gate logits ~ N(-12, 8^2) through the log-sigmoid gate (log a down to
    about -40), packed sequences with tails."""
    inp = make_prefill(PrefillSpec("logits", H=4, d=d, fixed_lengths=PACKED, dtype=dtype,
                                   init="normal0.1", seed=42))
    inp["g"] = steep_logits(42, inp["g"].shape)
    opts = dict(gate="logsigmoid", l2norm_qk=l2)
    out, fin = gpu_prefill(inp, **opts)
    ref_out, ref_fin = oracle_prefill(inp, **opts)
    for got, ref, what in ((out, ref_out, "O"), (fin, ref_fin, "final state")):
        assert np.isfinite(got).all()
        assert_parity(got, ref, dtype, what)


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_prefill_scalar_decay_steep(d, dtype):
    """One decay per head (Gated DeltaNet form), log a ~ U[-40, 0] per token."""
    inp = make_prefill(PrefillSpec("scalar steep", H=3, d=d, fixed_lengths=PACKED, dtype=dtype,
                                   init="normal0.1", seed=43))
    gen = torch.Generator().manual_seed(43)
    inp["g"] = -40.0 * torch.rand(inp["beta"].shape, generator=gen)
    out, fin = gpu_prefill(inp, decay="scalar")
    ref_out, ref_fin = oracle_prefill(inp, decay="scalar")
    for got, ref, what in ((out, ref_out, "O"), (fin, ref_fin, "final state")):
        assert np.isfinite(got).all()
        assert_parity(got, ref, dtype, what)


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32"), (128, "f32")])
def test_decode_edge_heads(d, dtype):
    """The decode step over 8 successive tokens with the same head kinds."""
    spec = DecodeSpec("edge decode", N=5, H=6, d=d, steps=8, dtype=dtype, seed=44)
    inp = make_decode_edge(spec)
    state = inp["state0"].cuda().contiguous()
    ref_state = f64(inp["state0"])
    for t in range(spec.steps):
        args = [inp[n][t].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")]
        out = decode_step(*args, inp["scale"], state)
        torch.cuda.synchronize()
        ref_out, ref_state = oracle.decode_step(*(f64(inp[n][t]) for n in ("q", "k", "v", "g", "beta")),
                                                inp["scale"], ref_state)
        check(f64(out), ref_out, dtype, "decode O step %d" % t)
        check(f64(state), ref_state, dtype, "final state after step %d" % t)


def test_decode_overwrite_on_gpu():
    """beta = 1 with a unit key stores v under k exactly: after each step,
    S^T k = v ("Understanding Kimi Delta Attention", "Does the write work?"),
    on the fp32 decode path, whatever the decay before the write."""
    spec = DecodeSpec("overwrite", N=4, H=6, d=64, steps=6, dtype="f32", seed=45)
    inp = make_decode_edge(spec)
    state = inp["state0"].cuda().contiguous()
    h = EDGE_KINDS.index("beta1")
    for t in range(spec.steps):
        args = [inp[n][t].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")]
        decode_step(*args, inp["scale"], state)
        torch.cuda.synchronize()
        S = f64(state)[:, h]                 # [N, dk, dv]
        k = f64(inp["k"][t])[:, h]           # [N, dk]
        v = f64(inp["v"][t])[:, h]           # [N, dv]
        read = np.einsum("nkv,nk->nv", S, k)
        assert np.abs(read - v).max() <= 1e-4
