"""The output gate and RMS normalisation fused into the prefill
(kda_chunk_fwd_gated), against the fp64 oracle's scan followed by its
epilogue (oracle/epilogue.py), on the tensor-core path (where the four CTAs of
a head exchange row sums through distributed shared memory) and on the fp32
path; fixed-length and packed batches, ragged tails, steep decays."""
import numpy as np
import pytest
import torch

import oracle
from oracle.epilogue import output_gate_rmsnorm as oracle_gate
from kimi_delta_attention_17_gb300 import build, chunk_fwd, output_gate_rmsnorm, workspace_size
from kimi_delta_attention_17_gb300.inputs import PrefillSpec, make_prefill, make_prefill_edge
from tests.helpers import BF16_MAX_ABS, BF16_REL_FRO, F32_MAX_ABS, assert_parity, errors, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def gate_inputs(inp, seed, with_weight):
    gen = torch.Generator().manual_seed(seed)
    z = torch.randn(inp["v"].shape, generator=gen).to(inp["v"].dtype)
    w = (1.0 + 0.5 * torch.randn(inp["v"].shape[-1], generator=gen)) if with_weight else None
    return z, w


def run(inp, z, w, eps=1e-6, **opts):
    dev = "cuda"
    q, k, v, g, beta = (inp[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    init = None if inp["init_state"] is None else inp["init_state"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    B, T, H, d = q.shape
    ws = torch.empty(max(1, workspace_size(B, T, H, d, d, len(inp["lengths"]), q.dtype)),
                     dtype=torch.uint8, device=dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], init, cu, workspace=ws,
                         out_gate=z.to(dev), norm_weight=None if w is None else w.to(dev),
                         norm_eps=eps, **opts)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    return out, fin


def reference(inp, z, w, eps=1e-6):
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].numpy().astype(np.int64)
    o, fin = oracle.scan(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]),
                         f64(inp["beta"]), inp["scale"], f64(inp["init_state"]), cu)
    return oracle_gate(o, f64(z), None if w is None else f64(w), eps), fin, o


def assert_gated_parity(got, ref, ref_o, storage, what):
    """The gated output's bounds are the scan output's carried through the
    normalisation: relative Frobenius error as for O; max |error| as for O
    times the gain of the gate and normalisation, rms(gated) / rms(O) (the
    gated rows have unit RMS before w and the sigmoid, whatever O's scale)."""
    m, r = errors(got, ref)
    gain = max(1.0, float(np.sqrt(np.mean(ref ** 2)) / max(np.sqrt(np.mean(ref_o ** 2)), 1e-30)))
    print("\n%s: max|err| %.3g (bound %.3g), rel %.3g" % (
        what, m, (F32_MAX_ABS if storage == "f32" else BF16_MAX_ABS) * gain, r))
    if storage == "f32":
        assert m <= F32_MAX_ABS * gain, what
    else:
        assert m <= BF16_MAX_ABS * gain and r <= BF16_REL_FRO, what


CASES = [
    ("batch", PrefillSpec("gate batch", H=4, d=128, B=2, T=300, init="normal0.1", seed=51)),
    ("packed", PrefillSpec("gate packed", H=3, d=128, fixed_lengths=(0, 1, 63, 64, 65, 130, 200),
                           init="normal0.1", seed=52)),
    ("fp32-d64", PrefillSpec("gate fp32", H=3, d=64, B=2, T=150, dtype="f32", init="normal0.1",
                             seed=53)),
]


@pytest.mark.parametrize("with_weight", [True, False], ids=["weight", "ones"])
@pytest.mark.parametrize("name,spec", CASES, ids=[c[0] for c in CASES])
def test_fused_gate_matches_oracle(name, spec, with_weight):
    inp = make_prefill(spec)
    z, w = gate_inputs(inp, 7, with_weight)
    out, fin = run(inp, z, w)
    ref_out, ref_fin, ref_o = reference(inp, z, w)
    assert torch.isfinite(out.float()).all()
    assert_gated_parity(f64(out), ref_out, ref_o, spec.dtype, "gated O (%s)" % name)
    assert_parity(f64(fin), ref_fin, spec.dtype, "final state")


def test_fused_gate_steep_heads_and_segments_option():
    """Steep decays and the other edge-case heads; a segments request is
    ignored (the gate runs on the serial chain)."""
    inp = make_prefill_edge(PrefillSpec("gate edge", H=6, d=128, B=1, T=500, init="normal0.1",
                                        seed=54))
    z, w = gate_inputs(inp, 8, True)
    out, fin = run(inp, z, w, eps=1e-5, segments=3)
    ref_out, ref_fin, ref_o = reference(inp, z, w, eps=1e-5)
    assert torch.isfinite(out.float()).all()
    assert_gated_parity(f64(out), ref_out, ref_o, "bf16", "gated O (edge heads)")
    assert_parity(f64(fin), ref_fin, "bf16", "final state")


def test_fused_gate_close_to_separate_pass():
    """The fused gate reads o in fp32 before its one rounding; the separate
    pass reads the rounded o. Both agree within bf16 rounding."""
    spec = PrefillSpec("gate vs pass", H=4, d=128, B=1, T=1000, init="normal0.1", seed=55)
    inp = make_prefill(spec)
    z, w = gate_inputs(inp, 9, True)
    fused, _ = run(inp, z, w)
    dev = "cuda"
    o, _ = chunk_fwd(*(inp[n].to(dev) for n in ("q", "k", "v", "g", "beta")), inp["scale"],
                     inp["init_state"].to(dev), segments=1)
    sep = output_gate_rmsnorm(o, z.to(dev), w.to(dev))
    torch.cuda.synchronize()
    d = (fused.float() - sep.float()).abs()
    print("\nfused vs separate pass: max|diff| %.3g rel %.3g" % (float(d.max()),
                                                               float(d.norm() / sep.float().norm())))
    assert float(d.norm() / sep.float().norm()) <= 5e-3
