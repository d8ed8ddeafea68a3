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


def _options(decay, gate, gate_lower, l2norm_qk, segments=0, fused=None):
    """kda_options for the given names, or None for the plain entry points."""
    if decay == "channel" and gate == "log" and not l2norm_qk and segments == 0 and fused is None:
        return None
    if decay not in _lib.DECAY or gate not in _lib.GATE:
        raise ValueError("decay must be one of %s and gate one of %s"
                         % (sorted(_lib.DECAY), sorted(_lib.GATE)))
    if int(segments) < 0:
        raise ValueError("segments must be >= 0")
    return _lib.Options(_lib.DECAY[decay], _lib.GATE[gate], float(gate_lower), int(bool(l2norm_qk)),
                        int(segments), 0 if fused is None else (1 if fused else -1))


def _check_g(g, decay, nd):
    """g's expected form for the decay family: [..., H, dk], [..., H] or unused."""
    if decay == "none":
        if g is not None:
            _need(g, "g", torch.float32)
        return
    _need(g, "g", torch.float32, nd if decay == "channel" else nd - 1)


def chunk_fwd(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, *, out=None,
              final_state=None, workspace=None, output_final_state=True, stream=None,
              phase_events=None, decay="channel", gate="log", gate_lower=-5.0, l2norm_qk=False,
              segments=0, out_gate=None, norm_weight=None, norm_eps=1e-6, fused=None):
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
    gate_lower * sigmoid(g)); ``l2norm_qk`` normalises q and k in the kernel;
    ``segments`` how the state crosses the chunks on the tensor-core path (0
    automatic, 1 one serial chain, k up to k segments composed as affine maps;
    kda_options.segments). ``fused`` (kda_options.fused): None lets the
    library run phase 1 and the state pass as one cooperative launch where
    that is expected to be faster, True wherever it is supported, False never.
    ``out_gate`` (gate logits z, q's dtype and v's shape) makes ``out`` the
    gated, RMS-normalised output w * o / sqrt(mean(o^2) + norm_eps) *
    sigmoid(z), with ``norm_weight`` [dv] fp32 or None (kda_chunk_fwd_gated;
    on the tensor-core path applied in the state pass, or as a pass over the
    outputs of the fused launch)."""
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
    opts = _options(decay, gate, gate_lower, l2norm_qk, segments, fused)
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(init_state),
            _ptr(cu_seqlens), _ptr(out), _ptr(final_state), B, T, H, dk, dv, N, _DTYPES[dtype])
    tail = (_ptr(workspace), workspace.numel(), _stream_ptr(stream))
    handles = None
    if phase_events is not None:
        if len(phase_events) != 4:
            raise ValueError("phase_events needs 4 events")
        handles = (ctypes.c_void_p * 4)(*[None if e is None else _event_handle(e)
                                          for e in phase_events])
    if out_gate is not None:
        _need(out_gate, "out_gate", dtype, 4)
        if out_gate.shape != v.shape:
            raise ValueError("out_gate must have v's shape")
        if norm_weight is not None:
            _need(norm_weight, "norm_weight", torch.float32, 1)
        if opts is None:
            opts = _lib.Options(_lib.DECAY["channel"], _lib.GATE["log"], 0.0, 0, 0)
        _lib.check("kda_chunk_fwd_gated", _lib.lib().kda_chunk_fwd_gated(
            *head[:8], _ptr(out_gate), _ptr(norm_weight), float(norm_eps), *head[8:],
            ctypes.byref(opts), *tail, handles))
    elif opts is not None:
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


def _host(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError("%s must be a host tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))


def host_workspace_size(H, dk, dv, dtype, window_tokens=16384, decay="channel"):
    """Bytes of device workspace kda_chunk_fwd_host needs (include/kda.h)."""
    opts = _lib.Options(_lib.DECAY[decay], 0, 0.0, 0, 0)
    return int(_lib.lib().kda_chunk_fwd_host_workspace_size(H, dk, dv, _DTYPES[dtype],
                                                            ctypes.byref(opts), window_tokens))


def chunk_fwd_host(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, *, out=None,
                   final_state=None, window_tokens=16384, workspace=None, scratch=None,
                   device=None, stream=None, decay="channel", gate="log", gate_lower=-5.0,
                   l2norm_qk=False, fused=None):
    """The prefill with every tensor in host memory (kda_chunk_fwd_host): q, k,
    v [B, T, H, d], g, beta as in chunk_fwd, init_state [N, H, dk, dv] or None,
    cu_seqlens an int32 HOST tensor [N + 1] or None, all pinned for the copies
    to overlap with the compute. The library cuts the sequences into windows of
    ``window_tokens`` tokens (whole 64-token chunks of each sequence; results
    bit-identical to one chunk_fwd call with segments=1) and pipelines the
    copies. Returns host tensors (out [B, T, H, dv], final_state [N, H, dk, dv]);
    ``out`` / ``final_state`` may be given (pinned). ``workspace``: a device
    uint8 tensor of host_workspace_size(...) bytes, or None (allocated here,
    and kept in the ``scratch`` dict when one is given)."""
    if window_tokens <= 0 or window_tokens % 64:
        raise ValueError("window_tokens must be a positive multiple of 64")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        _host(t, n)
    if g is not None:
        _host(g, "g", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, d]")
    dtype = q.dtype
    if dtype not in _DTYPES:
        raise ValueError("q/k/v must be bfloat16 or float32")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        _host(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if init_state is not None:
        _host(init_state, "init_state", torch.float32)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dtype).pin_memory()
    if final_state is None:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32).pin_memory()
    opts = _options(decay, gate, gate_lower, l2norm_qk, 1, fused)
    need = int(_lib.lib().kda_chunk_fwd_host_workspace_size(H, dk, dv, _DTYPES[dtype],
                                                            ctypes.byref(opts), window_tokens))
    if workspace is None:
        sc = {} if scratch is None else scratch
        key = ("prefill", need, dev)
        if sc.get("key") != key:
            sc.clear()
            sc["key"] = key
            sc["ws"] = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        workspace = sc["ws"]
    _need(workspace, "workspace", torch.uint8, 1)
    _lib.check("kda_chunk_fwd_host", _lib.lib().kda_chunk_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(init_state),
        _ptr(cu_seqlens), _ptr(out), _ptr(final_state), B, T, H, dk, dv, N, _DTYPES[dtype],
        ctypes.byref(opts), int(window_tokens), _ptr(workspace), workspace.numel(),
        _stream_ptr(stream)))
    return out, final_state


def decode_host(q, k, v, g, beta, scale, state, *, out=None, workspace=None, scratch=None,
                stream=None, decay="channel", gate="log", gate_lower=-5.0, l2norm_qk=False):
    """``steps`` successive decode steps with the per-step tensors in host
    memory (kda_decode_host): q, k [steps, N, H, dk], v [steps, N, H, dv], g
    [steps, N, H, dk] (or per the decay option), beta [steps, N, H], pinned;
    ``state`` [N, H, dk, dv] fp32 stays on the device and is updated in place.
    Returns the host outputs [steps, N, H, dv] (``out``, pinned, may be given).
    ``workspace``: a device uint8 tensor, or None (allocated here, and kept in
    the ``scratch`` dict when one is given)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        _host(t, n)
    if g is not None:
        _host(g, "g", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [steps, N, H, dk]")
    _need(state, "state", torch.float32, 4)
    dtype = q.dtype
    if dtype not in _DTYPES:
        raise ValueError("q/k/v must be bfloat16 or float32")
    steps, N, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(tuple(v.shape), dtype=dtype).pin_memory()
    opts = _options(decay, gate, gate_lower, l2norm_qk, 0)
    optp = None if opts is None else ctypes.byref(opts)
    need = int(_lib.lib().kda_decode_host_workspace_size(N, H, dk, dv, _DTYPES[dtype], optp))
    if workspace is None:
        sc = {} if scratch is None else scratch
        key = ("decode", need, state.device)
        if sc.get("key") != key:
            sc.clear()
            sc["key"] = key
            sc["ws"] = torch.empty(max(need, 1), dtype=torch.uint8, device=state.device)
        workspace = sc["ws"]
    _need(workspace, "workspace", torch.uint8, 1)
    _lib.check("kda_decode_host", _lib.lib().kda_decode_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(state), _ptr(out),
        steps, N, H, dk, dv, _DTYPES[dtype], optp, _ptr(workspace), workspace.numel(),
        _stream_ptr(stream)))
    return out


class DecodeGraph:
    """``steps`` successive decode steps captured once as one CUDA graph and
    then replayed: the per-step host work (argument checks, the C call, the
    launch) is paid at capture only, which is what bounds small-batch decode.

    q, k [steps, N, H, dk]; v [steps, N, H, dv]; g and beta as in decode_step
    with a leading steps axis: device tensors that the caller refills in place
    between replays. ``state`` [N, H, dk, dv] fp32 is advanced in place by
    every replay (by all ``steps`` steps). ``out`` [steps, N, H, dv] (allocated
    when None) receives the outputs of every replay. ``options`` as in
    decode_step. Capturing runs no step on ``state``: one warm-up step runs on
    a copy, outside the graph."""

    def __init__(self, q, k, v, g, beta, scale, state, *, out=None, **options):
        if q.dim() != 4 or q.shape[0] < 1:
            raise ValueError("q must be [steps, N, H, dk] with steps >= 1")
        self.steps = q.shape[0]
        if out is None:
            out = torch.empty(tuple(v.shape), dtype=q.dtype, device=q.device)
        self.out = out

        def step(t, st):
            decode_step(q[t], k[t], v[t], None if g is None else g[t], beta[t], scale, st,
                        out=out[t], **options)

        warm = state.clone()
        step(0, warm)  # loads the library and checks the arguments outside the capture
        torch.cuda.current_stream().synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            for t in range(self.steps):
                step(t, state)

    def replay(self):
        """Runs the captured steps on the current stream."""
        self.graph.replay()
