"""The fused single-launch prefill (kda_options.fused: phase 1 and the state
pass with 64-column slabs in one cooperative launch, each (chunk, head)
region handed over through a ready flag) against the fp64 oracle. The fused
launch is forced (fused=True) at sizes the oracle finishes in seconds:
several chunks with ragged tails, fixed-length batches (phase 1 then walks
the items chunk-major across the sequences), one packed sequence, initial
states, the decay / gate / normalisation variants, edge-case decays, the
gated output (the fused launch, then the gate pass), one workspace reused by
consecutive calls (the flags are cleared by every call), repeatability, the fall-back when
too many chains leave no SMs to phase 1, agreement with the two launches, and
the automatic choice on the long workload's shape at a shorter length."""
import numpy as np
import pytest
import torch

import oracle
from oracle.epilogue import output_gate_rmsnorm as oracle_gate
from oracle.prologue import prepare
from kimi_delta_attention_17_gb300 import build, chunk_fwd, workspace_size
from kimi_delta_attention_17_gb300.inputs import (OptionsSpec, PrefillSpec, make_prefill,
                                                  make_prefill_edge, make_prefill_opts)
from tests.helpers import BF16_MAX_ABS, BF16_REL_FRO, assert_parity, errors, f64, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def gpu(inp, ws=None, events=None, **opts):
    dev = "cuda"
    q, k, v, beta = (inp[n].to(dev) for n in ("q", "k", "v", "beta"))
    g = None if inp["g"] is None else inp["g"].to(dev)
    init = None if inp["init_state"] is None else inp["init_state"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    B, T, H, d = q.shape
    if ws is None:
        ws = torch.empty(max(1, workspace_size(B, T, H, d, d, len(inp["lengths"]), q.dtype)),
                         dtype=torch.uint8, device=dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], init, cu, workspace=ws,
                         phase_events=events, **opts)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "status word"
    return out, fin


def check(out, fin, ref_out, ref_fin, what):
    assert torch.isfinite(out.float()).all(), what
    assert_parity(f64(out), ref_out, "bf16", "O (%s)" % what)
    assert_parity(f64(fin), ref_fin, "bf16", "final state (%s)" % what)


CASES = [
    # one sequence: 11 chunks, a 60-token tail, 8 heads (16 state CTAs)
    ("one-seq", PrefillSpec("fused one", H=8, d=128, B=1, T=700, init="normal0.1", seed=61)),
    # three sequences: items chunk-major across them, a 2-token tail
    ("batch3", PrefillSpec("fused batch", H=4, d=128, B=3, T=450, init="normal0.1", seed=62)),
    # one packed sequence (cu_seqlens with a single sequence), no initial state
    ("packed1", PrefillSpec("fused packed", H=6, d=128, fixed_lengths=(777,), seed=63)),
    # one chunk only, ragged
    ("short", PrefillSpec("fused short", H=4, d=128, B=2, T=37, init="normal0.1", seed=64)),
]


@pytest.mark.parametrize("name,spec", CASES, ids=[c[0] for c in CASES])
def test_fused_matches_oracle(name, spec):
    inp = make_prefill(spec)
    out, fin = gpu(inp, fused=True)
    ref_out, ref_fin = oracle_prefill(inp)
    check(out, fin, ref_out, ref_fin, name)


def test_fused_agrees_with_two_launches():
    """Same inputs through the fused launch (64-column slabs) and the two
    launches (32-column slabs): the same products in fp32, up to rounding."""
    inp = make_prefill(PrefillSpec("fused vs two", H=8, d=128, B=2, T=520, init="normal0.1",
                                   seed=65))
    a, fa = gpu(inp, fused=True)
    b, fb = gpu(inp, fused=False)
    for x, y, what in ((a, b, "O"), (fa, fb, "final state")):
        m, r = errors(f64(x), f64(y))
        print("\nfused vs two launches, %s: max|diff| %.3g rel %.3g" % (what, m, r))
        assert r <= 1e-3, what


def test_workspace_reused_across_calls():
    """Two calls on one workspace with different inputs: the second call's
    ready flags start cleared, so it waits for its own regions."""
    spec = PrefillSpec("fused reuse", H=8, d=128, B=1, T=640, init="normal0.1", seed=66)
    first = make_prefill(spec)
    second = make_prefill(PrefillSpec("fused reuse 2", H=8, d=128, B=1, T=640, init="normal0.1",
                                      seed=67))
    B, T, H, d = first["q"].shape
    ws = torch.empty(workspace_size(B, T, H, d, d, B, first["q"].dtype), dtype=torch.uint8,
                     device="cuda")
    gpu(first, ws=ws, fused=True)
    out, fin = gpu(second, ws=ws, fused=True)
    ref_out, ref_fin = oracle_prefill(second)
    check(out, fin, ref_out, ref_fin, "second call")


FUSED_OPTIONS = [
    OptionsSpec("scalar", "log", False),
    OptionsSpec("none", "log", False),
    OptionsSpec("channel", "logsigmoid", True),
    OptionsSpec("channel", "bounded", False),
    OptionsSpec("scalar", "bounded", True),
]


@pytest.mark.parametrize("opts", FUSED_OPTIONS,
                         ids=lambda o: "%s-%s%s" % (o.decay, o.gate, "-l2" if o.l2norm_qk else ""))
def test_fused_options(opts):
    """Each phase-1 variant of the fused kernel (decay family, gate transform,
    in-kernel normalisation)."""
    spec = PrefillSpec("fused opt", H=4, d=128, B=2, T=300, init="normal0.1", seed=68)
    inp = make_prefill_opts(spec, opts)
    out, fin = gpu(inp, fused=True, **opts.kwargs())
    q, k, g = prepare(f64(inp["q"]), f64(inp["k"]), f64(inp["g"]), **opts.kwargs())
    ref_out, ref_fin = oracle.scan(q, k, f64(inp["v"]), g, f64(inp["beta"]), inp["scale"],
                                   f64(inp["init_state"]), None)
    check(out, fin, ref_out, ref_fin, "options")


def test_fused_edge_decays():
    """Steep decays (the exact steep form in phase 1), logsigmoid gates of
    very negative logits, beta = 0, beta = 1 with unit keys, no decay."""
    inp = make_prefill_edge(PrefillSpec("fused edge", H=6, d=128, B=1, T=500, init="normal0.1",
                                        seed=69))
    out, fin = gpu(inp, fused=True)
    ref_out, ref_fin = oracle_prefill(inp)
    check(out, fin, ref_out, ref_fin, "edge heads")


@pytest.mark.parametrize("T", [300, 64, 20], ids=["T300", "T64", "T20"])
def test_fused_then_gate_pass(T):
    """The gated prefill where the fused launch applies: plain outputs, then
    the gate and RMS normalisation as a pass over them (several chunks,
    exactly one chunk, a single ragged chunk)."""
    spec = PrefillSpec("fused gated", H=4, d=128, B=2, T=T, init="normal0.1", seed=70)
    inp = make_prefill(spec)
    gen = torch.Generator().manual_seed(71)
    z = torch.randn(inp["v"].shape, generator=gen).to(inp["v"].dtype)
    w = 1.0 + 0.5 * torch.randn(inp["v"].shape[-1], generator=gen)
    out, fin = gpu(inp, fused=True, out_gate=z.to("cuda"), norm_weight=w.to("cuda"))
    ref_o, ref_fin = oracle_prefill(inp)
    ref = oracle_gate(ref_o, f64(z), f64(w), 1e-6)
    m, r = errors(f64(out), ref)
    gain = max(1.0, float(np.sqrt(np.mean(ref ** 2)) / max(np.sqrt(np.mean(ref_o ** 2)), 1e-30)))
    print("\nfused + gate pass: max|err| %.3g (bound %.3g), rel %.3g" % (m, BF16_MAX_ABS * gain, r))
    assert m <= BF16_MAX_ABS * gain and r <= BF16_REL_FRO
    assert_parity(f64(fin), ref_fin, "bf16", "final state (gated)")


@pytest.mark.parametrize("fused,gated", [(True, False), (True, True), (False, True)],
                         ids=["fused-plain", "fused-gated", "two-launch-gated"])
def test_repeatable(fused, gated):
    """Twelve identical calls give bit-identical outputs: nothing in the
    launches depends on the order in which their CTAs, warps or copies finish
    (a race on a shared-memory slot, a TMEM tile, a ready flag or the gate
    logits' slot, refilled by a tensor-map copy, would show as a difference
    between calls). The two-launch gated case runs the in-pass gate of the
    32-column state pass."""
    spec = PrefillSpec("fused repeat", H=4, d=128, B=2, T=300, init="normal0.1", seed=74)
    inp = make_prefill(spec)
    gen = torch.Generator().manual_seed(75)
    extra = {}
    if gated:
        extra = dict(out_gate=torch.randn(inp["v"].shape, generator=gen).to(inp["v"].dtype).cuda(),
                     norm_weight=(1.0 + 0.5 * torch.randn(inp["v"].shape[-1], generator=gen)).cuda())
    first, ffin = gpu(inp, fused=fused, **extra)
    for _ in range(11):
        out, fin = gpu(inp, fused=fused, **extra)
        assert torch.equal(out, first) and torch.equal(fin, ffin)


def test_too_many_chains_fall_back():
    """80 heads: the 64-column state pass would need 160 CTAs, more than the
    SMs leave to phase 1, so even a forced request runs the two launches
    (the state-pass phase mark then follows a launch of its own)."""
    spec = PrefillSpec("fused fallback", H=80, d=128, B=1, T=130, init="normal0.1", seed=72)
    inp = make_prefill(spec)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    out, fin = gpu(inp, events=ev, fused=True)
    heads = [0, 41, 79]
    ref_out, ref_fin = oracle_prefill(inp, heads=heads)
    check(out[:, :, heads], fin[:, heads], ref_out, ref_fin, "80 heads")
    assert ev[2].elapsed_time(ev[3]) > 0.0


def test_automatic_choice_on_long_workload_shape():
    """The long workload's shape (one sequence, 32 heads) at 4096 tokens: the
    automatic choice runs the fused launch (both phase marks follow its one
    launch, so the state-pass interval is empty); sampled heads against the
    oracle."""
    spec = PrefillSpec("fused auto", H=32, d=128, B=1, T=4096, seed=73)
    inp = make_prefill(spec)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    out, fin = gpu(inp, events=ev)
    p1 = ev[1].elapsed_time(ev[2])
    p2 = ev[2].elapsed_time(ev[3])
    print("\nautomatic: first interval %.3f ms, second %.3f ms" % (p1, p2))
    assert p2 < 0.02 * p1
    heads = [0, 13, 31]
    ref_out, ref_fin = oracle_prefill(inp, heads=heads)
    check(out[:, :, heads], fin[:, heads], ref_out, ref_fin, "sampled heads")
