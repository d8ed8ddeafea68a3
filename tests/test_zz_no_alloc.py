"""kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot
allocate device memory (it uses a fixed scratch array compiled into
libkda.so instead of a caller-provided workspace).

The GPU test calls it through the C ABI twice in a row, on two different
inputs, and compares each result with the regular kda_chunk_fwd on the same
inputs, within the parity tolerances. It needs nothing from other test files,
so it passes alone in a fresh process as well as after the rest of the suite
(this file is named to be collected last).
"""
import ctypes

import pytest
import torch

from kimi_delta_attention_17_gb300 import _lib, build, chunk_fwd, workspace_size
from kimi_delta_attention_17_gb300.inputs import PrefillSpec, make_prefill
from tests.helpers import assert_parity, f64

KDA_NOALLOC_SCRATCH_BYTES = 64 << 20
KDA_ERR_INVALID_ARGUMENT = 1
KDA_ERR_WORKSPACE = 3


def _noalloc(L, t, scale, B, T, H, d, N, dtype_code, stream):
    p = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    return L.kda_chunk_fwd_noalloc(p(t["q"]), p(t["k"]), p(t["v"]), p(t["g"]), p(t["beta"]),
                                   scale, p(t["init"]), p(t["cu"]), p(t["out"]), p(t["fin"]),
                                   B, T, H, d, d, N, dtype_code, stream)


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Sizes needing more scratch than the fixed array are refused with
    KDA_ERR_WORKSPACE before any CUDA call (runs without a GPU)."""
    build.build()
    L = _lib.lib()
    B, T, H, d = 1, 1 << 20, 32, 128
    assert L.kda_chunk_fwd_workspace_size(B, T, H, d, d, 1, 1) > KDA_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    st = L.kda_chunk_fwd_noalloc(fake, fake, fake, fake, fake, 0.1, None, None, fake, fake,
                                 B, T, H, d, d, 1, 1, None)
    assert st == KDA_ERR_WORKSPACE


def test_noalloc_checks_arguments_before_capacity():
    """A bad argument is reported as kda_chunk_fwd reports it, whatever the
    size: a misaligned q with a problem too large for the scratch gives
    KDA_ERR_INVALID_ARGUMENT from both entry points (runs without a GPU)."""
    build.build()
    L = _lib.lib()
    B, T, H, d = 1, 1 << 20, 32, 128
    fake, bad = 1 << 20, (1 << 20) + 4
    args = (bad, fake, fake, fake, fake, 0.1, None, None, fake, fake, B, T, H, d, d, 1, 1)
    assert L.kda_chunk_fwd_noalloc(*args, None) == KDA_ERR_INVALID_ARGUMENT
    assert L.kda_chunk_fwd(*args, fake, 1 << 40, None) == KDA_ERR_INVALID_ARGUMENT
    assert L.kda_chunk_fwd_noalloc_status(None, None) == KDA_ERR_INVALID_ARGUMENT


@pytest.mark.gpu
def test_noalloc_reports_bad_offsets_through_its_status_word():
    """Decreasing packed offsets: the call returns KDA_OK (the offsets live on
    the device), computes nothing, and the status word read through
    kda_chunk_fwd_noalloc_status says KDA_ERR_INVALID_ARGUMENT; a good call
    afterwards reads KDA_OK."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    L = _lib.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    inp = make_prefill(PrefillSpec("noalloc status", H=2, d=128, fixed_lengths=(70, 50, 30),
                                   dtype="bf16", init="normal0.1", seed=33))
    B, T, H, d = inp["q"].shape
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    t["init"] = inp["init_state"].to(dev)
    t["out"] = torch.zeros_like(t["v"])
    t["fin"] = torch.zeros_like(t["init"])
    word = ctypes.c_int(-1)
    for cu, want in (([0, 70, 60, 150], KDA_ERR_INVALID_ARGUMENT), ([0, 70, 120, 150], 0)):
        t["cu"] = torch.tensor(cu, dtype=torch.int32, device=dev)
        st = _noalloc(L, t, inp["scale"], B, T, H, d, 3, _lib.DTYPE_BF16, stream.cuda_stream)
        assert st == 0, _lib.STATUS_NAMES.get(st, st)
        assert L.kda_chunk_fwd_noalloc_status(ctypes.byref(word), stream.cuda_stream) == 0
        torch.cuda.synchronize()
        assert word.value == want
        if want:
            assert not t["out"].any() and not t["fin"].any()  # nothing written


@pytest.mark.gpu
def test_noalloc_matches_chunk_fwd_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    L = _lib.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    specs = [PrefillSpec("noalloc a", H=4, d=128, B=2, T=300, dtype="bf16", init="normal0.1",
                         seed=31),
             PrefillSpec("noalloc b", H=3, d=64, fixed_lengths=(70, 0, 129), dtype="f32",
                         init="normal0.1", gate="mixture", seed=32)]
    for spec in specs:
        inp = make_prefill(spec)
        B, T, H, d = inp["q"].shape
        N = len(inp["lengths"])
        assert workspace_size(B, T, H, d, d, N, inp["q"].dtype) <= KDA_NOALLOC_SCRATCH_BYTES
        t = {n: inp[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
        t["init"] = inp["init_state"].to(dev)
        t["cu"] = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
        ref_out, ref_fin = chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], inp["scale"],
                                     t["init"], t["cu"])
        t["out"] = torch.full_like(ref_out, float("nan"))
        t["fin"] = torch.full_like(ref_fin, float("nan"))
        code = _lib.DTYPE_BF16 if spec.dtype == "bf16" else _lib.DTYPE_F32
        st = _noalloc(L, t, inp["scale"], B, T, H, d, N, code, stream.cuda_stream)
        assert st == 0, _lib.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        assert_parity(f64(t["out"]), f64(ref_out), spec.dtype, spec.name + " O")
        assert_parity(f64(t["fin"]), f64(ref_fin), spec.dtype, spec.name + " final state")
