"""CUDA-graph capture of the C-ABI calls: a prefill call and a run of decode
steps are captured once and replayed on inputs refilled in place; every
replay is bit-identical to the same calls made eagerly (the library only
launches kernels on the caller's stream, with no host synchronisation)."""
import pytest
import torch

from kimi_delta_attention_17_gb300 import DecodeGraph, build, chunk_fwd, decode_step, workspace_size
from kimi_delta_attention_17_gb300.inputs import DecodeSpec, PrefillSpec, make_decode, make_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


@pytest.mark.parametrize("d,dtype,H,T,segments", [(128, "bf16", 2, 300, 1), (128, "bf16", 2, 2100, 0),
                                                  (64, "f32", 3, 200, 0)])
def test_prefill_call_replays_bit_identical(d, dtype, H, T, segments):
    """Tensor-core path (serial and automatically segmented state pass) and
    the fp32 path."""
    dev = "cuda"
    names = ("q", "k", "v", "g", "beta", "init_state")
    first = make_prefill(PrefillSpec("graph-a", H=H, d=d, B=1, T=T, dtype=dtype, init="normal0.1", seed=41))
    second = make_prefill(PrefillSpec("graph-b", H=H, d=d, B=1, T=T, dtype=dtype, init="normal0.1", seed=42))
    buf = {n: first[n].to(dev) for n in names}
    B, T_, H_, d_ = buf["q"].shape
    ws = torch.empty(workspace_size(B, T_, H_, d_, d_, 1, buf["q"].dtype), dtype=torch.uint8, device=dev)
    out = torch.empty_like(buf["v"])
    fin = torch.empty((1, H_, d_, d_), dtype=torch.float32, device=dev)

    def call():
        chunk_fwd(buf["q"], buf["k"], buf["v"], buf["g"], buf["beta"], first["scale"], buf["init_state"],
                  out=out, final_state=fin, workspace=ws, segments=segments)

    call()  # eager, outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for inp in (first, second):
        for n in names:
            buf[n].copy_(inp[n])
        graph.replay()
        torch.cuda.synchronize()
        got_out, got_fin = out.clone(), fin.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(got_out, out) and torch.equal(got_fin, fin)


def test_decode_graph_matches_eager_steps():
    dev = "cuda"
    spec = DecodeSpec("graph-decode", N=3, H=4, d=128, steps=6, seed=43)
    inp = make_decode(spec)
    names = ("q", "k", "v", "g", "beta")
    buf = {n: inp[n].to(dev) for n in names}
    state_g = inp["state0"].to(dev)
    state_e = inp["state0"].to(dev)
    dg = DecodeGraph(buf["q"], buf["k"], buf["v"], buf["g"], buf["beta"], inp["scale"], state_g)
    torch.cuda.synchronize()
    assert torch.equal(state_g, inp["state0"].to(dev))  # capture ran no step on the state
    for rnd in range(2):
        if rnd:
            for n in names:
                buf[n].copy_(torch.flip(inp[n], dims=[0]))
        dg.replay()
        outs = [decode_step(buf["q"][t], buf["k"][t], buf["v"][t], buf["g"][t], buf["beta"][t],
                            inp["scale"], state_e) for t in range(spec.steps)]
        torch.cuda.synchronize()
        assert torch.equal(dg.out, torch.stack(outs)) and torch.equal(state_g, state_e)
