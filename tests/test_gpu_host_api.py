"""The host-buffer entry points of the C ABI (kda_chunk_fwd_host,
kda_decode_host, through their thin Python wrappers) pipeline copies with the
compute; their results are bit-identical to the device-tensor calls: windows
cut sequences only at whole 64-token chunks and the fp32 state crosses them
unchanged."""
import pytest
import torch

from kimi_delta_attention_17_gb300 import (build, chunk_fwd, chunk_fwd_host, decode_host,
                                           decode_step)
from kimi_delta_attention_17_gb300.inputs import (DecodeSpec, OptionsSpec, PrefillSpec, make_decode,
                                                  make_prefill, make_prefill_opts)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def _pin(inp, keys):
    return {n: None if inp[n] is None else inp[n].pin_memory() for n in keys}


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_chunk_fwd_host_matches_device_call(dtype, d):
    spec = PrefillSpec("host", H=3, d=d, B=2, T=300, dtype=dtype, init="normal0.1", seed=19)
    inp = make_prefill(spec)
    h = _pin(inp, ("q", "k", "v", "g", "beta", "init_state"))
    scratch = {}
    out_h, fin_h = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"],
                                  h["init_state"], window_tokens=128, scratch=scratch)
    out_h2, _ = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"],
                               h["init_state"], window_tokens=128, scratch=scratch)
    torch.cuda.synchronize()
    out_d, fin_d = chunk_fwd(*(inp[n].cuda() for n in ("q", "k", "v", "g", "beta")), inp["scale"],
                             inp["init_state"].cuda(), segments=1)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())
    assert torch.equal(out_h2, out_h)


@pytest.mark.parametrize("window", [64, 192, 16384])
@pytest.mark.parametrize("with_init", [True, False])
def test_chunk_fwd_host_packed_sequences(window, with_init):
    """Packed sequences (empty ones, ones shorter than a chunk, ones crossing
    several windows, more pieces than a window holds) through host cu_seqlens:
    bit-identical to one packed device call."""
    lengths = (0, 1, 63, 64, 65, 130, 0, 200, 17) + (5,) * 20 + (300,)
    spec = PrefillSpec("host packed", H=2, d=128, fixed_lengths=lengths, dtype="bf16",
                       init="normal0.1" if with_init else "zero", seed=23)
    inp = make_prefill(spec)
    h = _pin(inp, ("q", "k", "v", "g", "beta", "init_state"))
    cu_h = inp["cu_seqlens"].clone()
    out_h, fin_h = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"],
                                  h["init_state"], cu_h, window_tokens=window)
    torch.cuda.synchronize()
    init_d = None if inp["init_state"] is None else inp["init_state"].cuda()
    out_d, fin_d = chunk_fwd(*(inp[n].cuda() for n in ("q", "k", "v", "g", "beta")), inp["scale"],
                             init_d, inp["cu_seqlens"].cuda())
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(fin_h, fin_d.cpu())


def test_chunk_fwd_host_with_options():
    opts = OptionsSpec("scalar", "logsigmoid", True)
    inp = make_prefill_opts(PrefillSpec("host-opt", H=2, d=128, B=1, T=200, seed=20), opts)
    h = _pin(inp, ("q", "k", "v", "g", "beta"))
    out_h, fin_h = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"],
                                  window_tokens=64, **opts.kwargs())
    torch.cuda.synchronize()
    out_d, fin_d = chunk_fwd(*(inp[n].cuda() for n in ("q", "k", "v", "g", "beta")), inp["scale"],
                             segments=1, **opts.kwargs())
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())


def test_decode_host_matches_device_steps():
    spec = DecodeSpec("host-decode", N=6, H=2, d=128, steps=5, seed=21)
    inp = make_decode(spec)
    h = _pin(inp, ("q", "k", "v", "g", "beta"))
    s1 = inp["state0"].cuda()
    out_h = decode_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"], s1)
    s2 = inp["state0"].cuda()
    outs = [decode_step(*(inp[n][t].cuda() for n in ("q", "k", "v", "g", "beta")), inp["scale"], s2)
            for t in range(spec.steps)]
    torch.cuda.synchronize()
    assert torch.equal(out_h, torch.stack(outs).cpu()) and torch.equal(s1, s2)


@pytest.mark.slow
def test_chunk_fwd_host_full_size_matches_device_call():
    """The benchmark's end-to-end call at its size: the 131072-token, 32-head
    prefill through pinned host buffers in 16384-token windows equals one
    device call bit for bit."""
    from kimi_delta_attention_17_gb300.inputs import LONG_128K
    inp = make_prefill(LONG_128K)
    h = _pin(inp, ("q", "k", "v", "g", "beta"))
    out_h, fin_h = chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["scale"],
                                  window_tokens=16384)
    torch.cuda.synchronize()
    out_d, fin_d = chunk_fwd(*(h[n].cuda() for n in ("q", "k", "v", "g", "beta")), inp["scale"],
                             segments=1)
    torch.cuda.synchronize()
    assert torch.equal(fin_h, fin_d.cpu())
    assert torch.equal(out_h, out_d.cpu())
