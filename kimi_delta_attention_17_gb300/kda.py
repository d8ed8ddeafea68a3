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


def _options(decay, gate, gate_lower, l2norm_qk, segments=0):
    """kda_options for the given names, or None for the plain entry points."""
    if decay == "channel" and gate == "log" and not l2norm_qk and segments == 0:
        return None
    if decay not in _lib.DECAY or gate not in _lib.GATE:
        raise ValueError("decay must be one of %s and gate one of %s"
                         % (sorted(_lib.DECAY), sorted(_lib.GATE)))
    if int(segments) < 0:
        raise ValueError("segments must be >= 0")
    return _lib.Options(_lib.DECAY[decay], _lib.GATE[gate], float(gate_lower), int(bool(l2norm_qk)),
                        int(segments))


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
              segments=0):
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
    kda_options.segments)."""
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
    opts = _options(decay, gate, gate_lower, l2norm_qk, segments)
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


def chunk_fwd_host(q, k, v, g, beta, scale, init_state=None, *, out=None, final_state=None,
                   segment_tokens=16384, scratch=None, device=None, **options):
    """Prefill from pinned host tensors, for fixed-length batches (q, k, v
    [B, T, H, d], g, beta as in chunk_fwd; no cu_seqlens). Each sequence is cut
    into segments of ``segment_tokens`` tokens (a multiple of the 64-token
    chunk, so the chunking is that of one call, and with a serial state pass,
    segments=1, every result is bit-identical to one call's); segment
    i + 1 is copied to the device while segment i runs, and segment i's outputs
    are copied back while segment i + 1 runs. The state crosses segments in
    fp32 through init_state / final_state. Returns host tensors
    (out [B, T, H, dv], final_state [B, H, dk, dv]); ``out`` / ``final_state``
    may be given (pinned). ``scratch``: a dict kept between calls for the
    device buffers and streams. ``options`` as in chunk_fwd."""
    if segment_tokens <= 0 or segment_tokens % 64:
        raise ValueError("segment_tokens must be a positive multiple of 64")
    if q.dim() != 4 or q.shape[1] == 0:
        raise ValueError("q must be [B, T, H, d] with T > 0")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("%s must be a pinned host tensor" % n)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    sc = {} if scratch is None else scratch
    seg = min(segment_tokens, max(T, 1))
    key = (seg, H, dk, dv, q.dtype, None if g is None else tuple(g.shape[2:]))
    if sc.get("key") != key:
        sc.clear()
        sc["key"] = key
        sc["streams"] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))  # in, out copies
        sc["bufs"] = []
        for _ in range(2):  # double-buffered device segments
            b = {n: torch.empty((1, seg) + tuple(t.shape[2:]), dtype=t.dtype, device=dev)
                 for n, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g))
                 if t is not None}
            b["out"] = torch.empty((1, seg, H, dv), dtype=q.dtype, device=dev)
            sc["bufs"].append(b)
        sc["state"] = torch.empty((1, H, dk, dv), dtype=torch.float32, device=dev)
        sc["ws"] = torch.empty(max(1, workspace_size(1, seg, H, dk, dv, 1, q.dtype)),
                               dtype=torch.uint8, device=dev)
    s_in, s_out = sc["streams"]
    comp = torch.cuda.current_stream(dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype).pin_memory()
    if final_state is None:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()
    state = sc["state"]
    jobs = [(b, t0, min(T, t0 + seg)) for b in range(B) for t0 in range(0, max(T, 1), seg)]
    freed = [torch.cuda.Event(), torch.cuda.Event()]  # buffer i may be refilled
    drained = [torch.cuda.Event(), torch.cuda.Event()]  # buffer i's outputs copied out
    for i in range(2):
        freed[i].record(comp)
        drained[i].record(comp)
    for j, (b, t0, t1) in enumerate(jobs):
        buf = sc["bufs"][j % 2]
        n = t1 - t0
        loaded = torch.cuda.Event()
        with torch.cuda.stream(s_in):
            s_in.wait_event(freed[j % 2])
            for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
                if t is not None:
                    buf[name][:, :n].copy_(t[b:b + 1, t0:t1], non_blocking=True)
            loaded.record(s_in)
        comp.wait_event(loaded)
        comp.wait_event(drained[j % 2])
        first = t0 == 0
        if first and init_state is not None:
            state.copy_(init_state[b:b + 1], non_blocking=True)
        # [:, :n] of a (1, seg, ...) buffer is contiguous: the short last
        # segment runs in place.
        qd, kd, vd, bd = (buf[nm][:, :n] for nm in ("q", "k", "v", "beta"))
        chunk_fwd(qd, kd, vd, None if g is None else buf["g"][:, :n], bd, scale,
                  None if (first and init_state is None) else state, out=buf["out"][:, :n],
                  final_state=state, workspace=sc["ws"], **options)
        freed[j % 2].record(comp)
        done = torch.cuda.Event()
        done.record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            out[b:b + 1, t0:t1].copy_(buf["out"][:, :n], non_blocking=True)
            if t1 == T:
                final_state[b:b + 1].copy_(state, non_blocking=True)
            drained[j % 2].record(s_out)
        if t1 == T:
            # the next sequence's first segment must not overwrite this state early
            comp.wait_stream(s_out)
    comp.wait_stream(s_out)
    return out, final_state


def decode_host(q, k, v, g, beta, scale, state, *, out=None, scratch=None, **options):
    """``steps`` successive decode steps from pinned host tensors q, k [steps,
    N, H, dk], v [steps, N, H, dv], g [steps, N, H, dk] (or per the decay
    option), beta [steps, N, H]; ``state`` [N, H, dk, dv] fp32 stays on the
    device and is updated in place. Step t + 1's inputs are copied in while
    step t runs, and step t's outputs are copied back while step t + 1 runs.
    Returns the host outputs [steps, N, H, dv] (``out``, pinned, may be given).
    ``scratch``: a dict kept between calls for the device buffers and streams.
    ``options`` as in decode_step."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("%s must be a pinned host tensor" % n)
    steps = q.shape[0]
    dev = state.device
    sc = {} if scratch is None else scratch
    key = (tuple(q.shape[1:]), tuple(v.shape[1:]), q.dtype, None if g is None else tuple(g.shape[1:]))
    if sc.get("key") != key:
        sc.clear()
        sc["key"] = key
        sc["streams"] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        sc["bufs"] = [{n: torch.empty(tuple(t.shape[1:]), dtype=t.dtype, device=dev)
                       for n, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g))
                       if t is not None} for _ in range(2)]
        for b in sc["bufs"]:
            b["out"] = torch.empty(tuple(v.shape[1:]), dtype=q.dtype, device=dev)
    s_in, s_out = sc["streams"]
    comp = torch.cuda.current_stream(dev)
    if out is None:
        out = torch.empty(tuple(v.shape), dtype=q.dtype).pin_memory()
    freed = [torch.cuda.Event(), torch.cuda.Event()]
    drained = [torch.cuda.Event(), torch.cuda.Event()]
    for i in range(2):
        freed[i].record(comp)
        drained[i].record(comp)
    for t in range(steps):
        buf = sc["bufs"][t % 2]
        loaded = torch.cuda.Event()
        with torch.cuda.stream(s_in):
            s_in.wait_event(freed[t % 2])
            for name, x in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
                if x is not None:
                    buf[name].copy_(x[t], non_blocking=True)
            loaded.record(s_in)
        comp.wait_event(loaded)
        comp.wait_event(drained[t % 2])
        decode_step(buf["q"], buf["k"], buf["v"], buf.get("g"), buf["beta"], scale, state,
                    out=buf["out"], **options)
        freed[t % 2].record(comp)
        done = torch.cuda.Event()
        done.record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            out[t].copy_(buf["out"], non_blocking=True)
            drained[t % 2].record(s_out)
    comp.wait_stream(s_out)
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
