"""Python binding of libkda.so: the same entry points as include/kda.h, taking
torch CUDA tensors. It only marshals arguments (pointers, sizes, the current
stream) and allocates outputs and scratch with torch when the caller does not
pass them; every step of the computation runs in the library's kernels."""
import ctypes

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.DTYPE_F32, torch.bfloat16: _lib.DTYPE_BF16}


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _event_handle(ev):
    ev.record()  # materialises the event on the current device; re-recorded by the library
    return ev.cuda_event


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dimensions" % (name, ndim))


def status_string(status):
    return _lib.lib().kda_status_string(int(status)).decode()


def workspace_size(B, T, H, dk, dv, num_seqs, dtype):
    """Bytes of scratch kda_chunk_fwd needs (see include/kda.h)."""
    return int(_lib.lib().kda_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs,
                                                       _DTYPES[dtype]))


def _options(decay, gate, gate_lower, l2norm_qk):
    """kda_options for the given names, or None for the plain entry points."""
    if decay == "channel" and gate == "log" and not l2norm_qk:
        return None
    if decay not in _lib.DECAY or gate not in _lib.GATE:
        raise ValueError("decay must be one of %s and gate one of %s"
                         % (sorted(_lib.DECAY), sorted(_lib.GATE)))
    return _lib.Options(_lib.DECAY[decay], _lib.GATE[gate], float(gate_lower), int(bool(l2norm_qk)))


def _check_g(g, decay, nd):
    """g's expected form for the decay family: [..., H, dk], [..., H] or unused."""
    if decay == "none":
        if g is not None:
            _need(g, "g", torch.float32)
        return
    _need(g, "g", torch.float32, nd if decay == "channel" else nd - 1)


def chunk_fwd(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, *, out=None,
              final_state=None, workspace=None, output_final_state=True, stream=None,
              phase_events=None, decay="channel", gate="log", gate_lower=-5.0, l2norm_qk=False):
    """Chunkwise prefill. q, k [B, T, H, dk]; v [B, T, H, dv] (bf16 or fp32);
    g [B, T, H, dk] fp32; beta [B, T, H] fp32; init_state [N, H, dk, dv] fp32
    or None; cu_seqlens int32 [N+1] (device) or None (then N = B).
    Returns (out [B, T, H, dv], final_state [N, H, dk, dv] or None).
    ``phase_events``: optional list of 4 torch.cuda.Event (timing enabled)
    recorded at the start, after the chunk table, after the intra-chunk phase
    and after the state pass.
    Options (kda_chunk_fwd_opt): ``decay`` "channel" (g [B, T, H, dk]), "scalar"
    (g [B, T, H], Gated DeltaNet) or "none" (g unused, DeltaNet); ``gate`` "log"
    (g is log a), "logsigmoid" (a = sigmoid(g)) or "bounded" (log a =
    gate_lower * sigmoid(g)); ``l2norm_qk`` normalises q and k in the kernel."""
    _need(q, "q", ndim=4)
    dtype = q.dtype
    if dtype not in _DTYPES:
        raise ValueError("q/k/v must be bfloat16 or float32")
    for t, n in ((k, "k"), (v, "v")):
        _need(t, n, dtype, 4)
    _check_g(g, decay, 4)
    _need(beta, "beta", torch.float32, 3)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, 4)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dtype, device=q.device)
    else:
        _need(out, "out", dtype, 4)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    elif final_state is not None:
        _need(final_state, "final_state", torch.float32, 4)
    need = workspace_size(B, T, H, dk, dv, N, dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    else:
        _need(workspace, "workspace", torch.uint8, 1)
    opts = _options(decay, gate, gate_lower, l2norm_qk)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(init_state),
            _ptr(cu_seqlens), _ptr(out), _ptr(final_state), B, T, H, dk, dv, N, _DTYPES[dtype])
    tail = (_ptr(workspace), workspace.numel(), _stream_ptr(stream))
    handles = None
    if phase_events is not None:
        if len(phase_events) != 4:
            raise ValueError("phase_events needs 4 events")
        handles = (ctypes.c_void_p * 4)(*[None if e is None else _event_handle(e)
                                          for e in phase_events])
    if opts is not None:
        _lib.check("kda_chunk_fwd_opt",
                   _lib.lib().kda_chunk_fwd_opt(*head, ctypes.byref(opts), *tail, handles))
    elif handles is None:
        _lib.check("kda_chunk_fwd", _lib.lib().kda_chunk_fwd(*head, *tail))
    else:
        _lib.check("kda_chunk_fwd_timed", _lib.lib().kda_chunk_fwd_timed(*head, *tail, handles))
    return out, final_state


def decode_step(q, k, v, g, beta, scale, state, *, out=None, stream=None, decay="channel",
                gate="log", gate_lower=-5.0, l2norm_qk=False):
    """One decode step, state updated in place. q, k [N, H, dk]; v [N, H, dv];
    g [N, H, dk] fp32; beta [N, H] fp32; state [N, H, dk, dv] fp32.
    Returns out [N, H, dv]. Options as in chunk_fwd (with "scalar" decay g is
    [N, H]; kda_decode_step_opt)."""
    _need(q, "q", ndim=3)
    dtype = q.dtype
    if dtype not in _DTYPES:
        raise ValueError("q/k/v must be bfloat16 or float32")
    for t, n in ((k, "k"), (v, "v")):
        _need(t, n, dtype, 3)
    _check_g(g, decay, 3)
    _need(beta, "beta", torch.float32, 2)
    _need(state, "state", torch.float32, 4)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((N, H, dv), dtype=dtype, device=q.device)
    else:
        _need(out, "out", dtype, 3)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(state), _ptr(out),
            N, H, dk, dv, _DTYPES[dtype])
    opts = _options(decay, gate, gate_lower, l2norm_qk)
    if opts is None:
        _lib.check("kda_decode_step", _lib.lib().kda_decode_step(*head, _stream_ptr(stream)))
    else:
        _lib.check("kda_decode_step_opt",
                   _lib.lib().kda_decode_step_opt(*head, ctypes.byref(opts), _stream_ptr(stream)))
    return out


def output_gate_rmsnorm(o, z, weight=None, eps=1e-6, *, out=None, stream=None):
    """out = weight * o / sqrt(mean(o^2 over d_v) + eps) * sigmoid(z), per token
    and head (kda_output_gate_rmsnorm). o, z [..., H, dv] of one dtype (bf16 or
    fp32); weight [dv] fp32 or None. ``out`` may be ``o`` (in place)."""
    _need(o, "o")
    dtype = o.dtype
    if dtype not in _DTYPES:
        raise ValueError("o must be bfloat16 or float32")
    _need(z, "z", dtype)
    if z.shape != o.shape or o.dim() < 2:
        raise ValueError("z must have o's shape [..., H, dv]")
    H, dv = o.shape[-2], o.shape[-1]
    if weight is not None:
        _need(weight, "weight", torch.float32, 1)
    if out is None:
        out = torch.empty_like(o)
    else:
        _need(out, "out", dtype)
    tokens = o.numel() // (H * dv)
    _lib.check("kda_output_gate_rmsnorm",
               _lib.lib().kda_output_gate_rmsnorm(_ptr(o), _ptr(z), _ptr(weight), float(eps),
                                                  _ptr(out), tokens, H, dv, _DTYPES[dtype],
                                                  _stream_ptr(stream)))
    return out
