"""Argument checks of the host-side helpers (chunk_fwd_host, decode_host,
DecodeGraph, the options marshalling): they raise before any CUDA call, so
they run on the CPU."""
import pytest
import torch

from kimi_delta_attention_17_gb300 import DecodeGraph, chunk_fwd_host, decode_host, kda


def _host(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)  # pageable, not pinned


def test_chunk_fwd_host_rejects_bad_arguments():
    q = _host(1, 128, 2, 64)
    beta = _host(1, 128, 2, dtype=torch.float32)
    g = _host(1, 128, 2, 64, dtype=torch.float32)
    with pytest.raises(ValueError, match="multiple of 64"):
        chunk_fwd_host(q, q, q, g, beta, 0.125, window_tokens=100)
    with pytest.raises(ValueError, match="multiple of 64"):
        chunk_fwd_host(q, q, q, g, beta, 0.125, window_tokens=0)
    with pytest.raises(ValueError, match="host tensor"):
        chunk_fwd_host(q, q, q, g, beta.to("meta"), 0.125)
    with pytest.raises(ValueError, match="cu_seqlens must be torch.int32"):
        chunk_fwd_host(q, q, q, g, beta, 0.125, cu_seqlens=torch.zeros(2, dtype=torch.int64))


def test_decode_host_rejects_bad_arguments():
    q = _host(3, 2, 2, 64)
    beta = _host(3, 2, 2, dtype=torch.float32)
    state = torch.zeros(2, 2, 64, 64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        decode_host(q, q, q, None, beta, 0.125, state)  # the state lives on the device
    with pytest.raises(ValueError, match="steps, N, H, dk"):
        decode_host(_host(2, 2, 64), q, q, None, beta, 0.125, state.to("meta"))


def test_decode_graph_rejects_bad_shapes():
    state = torch.zeros(2, 2, 64, 64)
    with pytest.raises(ValueError, match="steps"):
        DecodeGraph(_host(2, 2, 64), _host(2, 2, 64), _host(2, 2, 64), None,
                    _host(2, 2, dtype=torch.float32), 0.125, state)
    with pytest.raises(ValueError, match="steps"):
        DecodeGraph(_host(0, 2, 2, 64), _host(0, 2, 2, 64), _host(0, 2, 2, 64), None,
                    _host(0, 2, 2, dtype=torch.float32), 0.125, state)


def test_options_marshalling():
    assert kda._options("channel", "log", -5.0, False, 0) is None  # the plain entry points
    o = kda._options("scalar", "bounded", -3.0, True, 4)
    assert (o.decay, o.gate, o.l2norm_qk, o.segments) == (1, 2, 1, 4)
    assert o.gate_lower == pytest.approx(-3.0)
    assert kda._options("channel", "log", -5.0, False, 1).segments == 1
    with pytest.raises(ValueError):
        kda._options("channel", "log", -5.0, False, -1)
    with pytest.raises(ValueError):
        kda._options("diagonal", "log", -5.0, False, 0)
    with pytest.raises(ValueError):
        kda._options("channel", "tanh", -5.0, False, 0)
