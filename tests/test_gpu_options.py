"""GPU parity of the options of kda_chunk_fwd_opt and kda_decode_step_opt
(decay families, gate transforms, in-kernel q/k normalisation) against the
fp64 oracle with its prologue (oracle/prologue.py), on both prefill paths
(tensor-core bf16 d=128; fp32 / d=64 path) and the decode step. Inputs span
several chunks, ragged tails and packed sequences."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle.prologue import prepare
from kimi_delta_attention_17_gb300 import _lib, build, chunk_fwd, decode_step, workspace_size
from kimi_delta_attention_17_gb300.inputs import (DecodeSpec, OptionsSpec, PrefillSpec,
                                                  make_decode_opts, make_prefill, make_prefill_opts)
from tests.helpers import assert_parity, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def oracle_opts(inp, opts):
    q, k, g = prepare(f64(inp["q"]), f64(inp["k"]), f64(inp["g"]), **opts.kwargs())
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].numpy().astype(np.int64)
    return oracle.scan(q, k, f64(inp["v"]), g, f64(inp["beta"]), inp["scale"],
                       f64(inp["init_state"]), cu)


def gpu_opts(inp, opts):
    dev = "cuda"
    q, k, v, beta = (inp[n].to(dev) for n in ("q", "k", "v", "beta"))
    g = None if inp["g"] is None else inp["g"].to(dev)
    init = None if inp["init_state"] is None else inp["init_state"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    B, T, H, d = q.shape
    ws = torch.empty(workspace_size(B, T, H, d, d, len(inp["lengths"]), q.dtype),
                     dtype=torch.uint8, device=dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], init, cu, workspace=ws, **opts.kwargs())
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    return f64(out), f64(fin)


TC_OPTIONS = [
    OptionsSpec("scalar", "log", False),
    OptionsSpec("none", "log", False),
    OptionsSpec("channel", "logsigmoid", True),
    OptionsSpec("channel", "bounded", False),
    OptionsSpec("scalar", "bounded", True),
    OptionsSpec("none", "log", True),
    OptionsSpec("scalar", "logsigmoid", False),
]


def _id(o):
    return "%s-%s%s" % (o.decay, o.gate, "-l2" if o.l2norm_qk else "")


@pytest.mark.parametrize("opts", TC_OPTIONS, ids=_id)
def test_tensor_core_prefill_options(opts):
    """bf16, d=128 (tensor-core path): two sequences of 300 tokens (five chunks,
    a 44-token tail), random initial states."""
    spec = PrefillSpec("opt", H=4, d=128, B=2, T=300, init="normal0.1", seed=11)
    inp = make_prefill_opts(spec, opts)
    out, fin = gpu_opts(inp, opts)
    ref_out, ref_fin = oracle_opts(inp, opts)
    assert_parity(out, ref_out, "bf16", "O")
    assert_parity(fin, ref_fin, "bf16", "final state")


@pytest.mark.parametrize("opts", [OptionsSpec("scalar", "logsigmoid", True),
                                  OptionsSpec("channel", "bounded", True)], ids=_id)
def test_tensor_core_prefill_options_packed(opts):
    """Packed sequences of lengths 70, 1, 0 and 200 (a zero-length and a
    one-token sequence) with options."""
    spec = PrefillSpec("opt-packed", H=3, d=128, fixed_lengths=(70, 1, 0, 200), init="normal0.1",
                       seed=12)
    inp = make_prefill_opts(spec, opts)
    out, fin = gpu_opts(inp, opts)
    ref_out, ref_fin = oracle_opts(inp, opts)
    assert_parity(out, ref_out, "bf16", "O")
    assert_parity(fin, ref_fin, "bf16", "final state")


@pytest.mark.parametrize("opts", [OptionsSpec("scalar", "logsigmoid", True),
                                  OptionsSpec("none", "log", True),
                                  OptionsSpec("channel", "bounded", False)], ids=_id)
@pytest.mark.parametrize("d,dtype", [(64, "f32"), (128, "f32"), (64, "bf16")])
def test_simt_prefill_options(opts, d, dtype):
    spec = PrefillSpec("opt-simt", H=2, d=d, B=1, T=150, dtype=dtype, init="normal0.1", seed=13)
    inp = make_prefill_opts(spec, opts)
    out, fin = gpu_opts(inp, opts)
    ref_out, ref_fin = oracle_opts(inp, opts)
    assert_parity(out, ref_out, dtype, "O")
    assert_parity(fin, ref_fin, dtype, "final state")


@pytest.mark.parametrize("opts", [OptionsSpec("scalar", "log", False),
                                  OptionsSpec("channel", "logsigmoid", True),
                                  OptionsSpec("none", "log", True),
                                  OptionsSpec("scalar", "bounded", True)], ids=_id)
@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_decode_options(opts, d, dtype):
    spec = DecodeSpec("opt-decode", N=5, H=3, d=d, steps=6, dtype=dtype, seed=14)
    inp = make_decode_opts(spec, opts)
    dev = "cuda"
    state = inp["state0"].to(dev)
    ref_state = f64(inp["state0"])
    for t in range(spec.steps):
        g = None if inp["g"] is None else inp["g"][t]
        out = decode_step(inp["q"][t].to(dev), inp["k"][t].to(dev), inp["v"][t].to(dev),
                          None if g is None else g.to(dev), inp["beta"][t].to(dev), inp["scale"],
                          state, **opts.kwargs())
        q, k, gc = prepare(f64(inp["q"][t]), f64(inp["k"][t]), f64(g), **opts.kwargs())
        ref_out, ref_state = oracle.decode_step(q, k, f64(inp["v"][t]), gc, f64(inp["beta"][t]),
                                                inp["scale"], ref_state)
        assert_parity(f64(out), ref_out, dtype, "decode O step %d" % t)
    torch.cuda.synchronize()
    assert_parity(f64(state), ref_state, dtype, "decode state")


def test_default_options_match_plain_entry_point():
    """kda_chunk_fwd_opt with {CHANNEL, LOG, 0, 0} is bit-identical to kda_chunk_fwd."""
    spec = PrefillSpec("opt-default", H=2, d=128, B=1, T=130, seed=15)
    inp = make_prefill(spec)
    dev = "cuda"
    q, k, v, g, beta = (inp[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    B, T, H, d = q.shape
    ws = torch.empty(workspace_size(B, T, H, d, d, 1, q.dtype), dtype=torch.uint8, device=dev)
    out1, fin1 = chunk_fwd(q, k, v, g, beta, inp["scale"], workspace=ws)
    out2, fin2 = torch.empty_like(out1), torch.empty_like(fin1)
    opts = _lib.Options(0, 0, 0.0, 0)
    st = _lib.lib().kda_chunk_fwd_opt(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(), inp["scale"], None,
        None, out2.data_ptr(), fin2.data_ptr(), B, T, H, d, d, 1, _lib.DTYPE_BF16,
        ctypes.byref(opts), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream, None)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(fin1, fin2)


@pytest.mark.parametrize("dv,dtype", [(128, "bf16"), (64, "bf16"), (128, "f32"), (64, "f32")])
@pytest.mark.parametrize("with_weight,in_place", [(True, False), (False, True)])
def test_output_gate_rmsnorm(dv, dtype, with_weight, in_place):
    """kda_output_gate_rmsnorm against the fp64 definition (oracle/epilogue.py),
    on the outputs of a prefill-sized tensor [B, T, H, dv] (1003 tokens)."""
    from oracle.epilogue import output_gate_rmsnorm as ref_fn
    from kimi_delta_attention_17_gb300 import output_gate_rmsnorm
    gen = torch.Generator().manual_seed(16)
    st = torch.bfloat16 if dtype == "bf16" else torch.float32
    o = (torch.randn((1, 1003, 3, dv), generator=gen) * 0.3).to(st)
    z = torch.randn((1, 1003, 3, dv), generator=gen).to(st)
    w = torch.randn((dv,), generator=gen) if with_weight else None
    ref = ref_fn(f64(o), f64(z), None if w is None else f64(w), 1e-6)
    od = o.cuda()
    got = output_gate_rmsnorm(od, z.cuda(), None if w is None else w.cuda(), 1e-6,
                              out=od if in_place else None)
    torch.cuda.synchronize()
    if in_place:
        assert got.data_ptr() == od.data_ptr()
    assert_parity(f64(got), ref, dtype, "gated RMSNorm output")
