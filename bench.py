"""Benchmark of the KDA hot path on GB300: chunkwise prefill tokens/s (headline)
and recurrent decode steps/s, with roofline fractions, an end-to-end number
through host buffers, SM clocks sampled during the timed region, and the CPU
oracle timed on the host cores beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on stdout (rank 0). Under torchrun each rank runs the same
per-GPU workload on its own GPU (independent sequences and heads need no
exchange: weak scaling, no collective on the data path); the timed region is
bracketed by a barrier and device synchronisation and the time is the maximum
over ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kimi_delta_attention_17_gb300 import inputs as kin  # noqa: E402

PREFILL_WORKLOADS = {"long": kin.LONG_128K, "b2": kin.PREFILL_B2, "varlen": kin.VARLEN_8}
L2_BYTES = 129 * 10 ** 6
KIB = 1024


# ------------------------------------------------------------------ algorithmic work

def prefill_bytes(spec, tokens, num_seqs, has_init):
    """Bytes the prefill must move: q, k, v, out in the storage dtype, g fp32,
    beta fp32 per (token, head); the final state (and the initial one when
    given) per (sequence, head)."""
    e = 2 if spec.dtype == "bf16" else 4
    d = spec.d
    per_token_head = 4 * d * e + d * 4 + 4   # q, k, v, out + g + beta
    state = d * d * 4
    return tokens * spec.H * per_token_head + num_seqs * spec.H * state * (2 if has_init else 1)


def prefill_bytes_g(spec, tokens, num_seqs, has_init, g_bytes_per_token_head):
    """prefill_bytes with another size of g per (token, head): 4 d for a
    per-channel decay, 4 for one decay per head, 0 without decay."""
    d = spec.d
    return (prefill_bytes(spec, tokens, num_seqs, has_init)
            - tokens * spec.H * (d * 4 - g_bytes_per_token_head))


def prefill_flops(spec, tokens):
    """Dense-contraction flops per (token, head) of the chunk algebra with
    C = 64 full tiles: A, H, W, U, H*Z at 2*C*d each and the three state
    products (W S, Qbar S, Kbar^T Z) at 2*d*d each."""
    C, d = 64, spec.d
    return tokens * spec.H * (5 * 2 * C * d + 3 * 2 * d * d)


def decode_bytes(spec):
    e = 2 if spec.dtype == "bf16" else 4
    d = spec.d
    per = 2 * d * d * 4 + 4 * d * e + d * 4 + 4   # state in+out, q k v out, g, beta
    return spec.N * spec.H * per


# ------------------------------------------------------------------ distributed plumbing

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(backend):
    world, rank, _ = dist_info()
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)
    return world, rank


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x, device=None):
    """Maximum of a float over all ranks (the slowest rank sets the time)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def units_for_world(units_per_rank, world):
    """Whole-job units for weak scaling: every rank processes its own batch."""
    return units_per_rank * world


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            # The timed work starts once the sampler is producing samples (at most 3 s).
            t0 = time.time()
            while time.time() - t0 < 3.0 and self.proc.poll() is None:
                self.fh.flush()
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.02)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            lines = fh.readlines()
        os.remove(self.path)
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ roofline peaks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _code_only(text):
    """CUDA/C++ source without comments and blank space (comments do not reach
    the compiled kernels, so editing them keeps a capture's counters valid)."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] in "\"'":  # string or character literal, copied as is
            q, j = text[i], i + 1
            while j < n and text[j] != q:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_sources_sha256():
    """Hash of the kernel sources' code (comments and blank space ignored)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kimi_delta_attention_17_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))):
        h.update(os.path.basename(f).encode())
        h.update(_code_only(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()


def traffic_key(spec):
    """The entry of profiles/ncu_traffic.json captured on this workload, or None."""
    if spec == kin.LONG_128K:
        return "prefill_long_t131072"
    if spec == kin.VARLEN_8:
        return "prefill_varlen_8seq_h32"
    return None


def measured_traffic(key):
    """DRAM bytes per launch from the committed ncu capture (profiles/ncu_traffic.json),
    or None when the kernel sources have changed since it was taken (or key is None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if key is None or not os.path.exists(path):
        return None
    t = json.load(open(path))
    if t.get("kernel_sources_sha256") != kernel_sources_sha256() or key not in t:
        return None
    return t[key]["bytes_per_launch"]


# ------------------------------------------------------------------ the oracle on the host cores

def oracle_prefill_sample(inp, spec, target_s=10.0, max_tokens=None):
    """Times the oracle (as it stands) on the first tokens of every head of
    the workload; grows the sample until one run takes about target_s.
    Returns (tokens/s, cores, sample description)."""
    import numpy as np
    import oracle

    T = inp["q"].shape[1]
    max_tokens = min(T, max_tokens or T)

    def run(n):
        arr = {k: inp[k][:, :n].to(torch.float64).numpy() for k in ("q", "k", "v", "g", "beta")}
        # The sample treats each row of q as one sequence (for packed inputs:
        # the first n tokens as one sequence starting from the first state).
        init = None if inp["init_state"] is None else \
            inp["init_state"][: arr["q"].shape[0]].double().numpy()
        t0 = time.perf_counter()
        oracle.scan(arr["q"], arr["k"], arr["v"], arr["g"], arr["beta"], inp["scale"], init)
        return time.perf_counter() - t0

    n = min(512, max_tokens)
    dt = run(n)
    if dt < target_s and n < max_tokens:
        n = int(min(max_tokens, max(n, n * target_s / max(dt, 1e-3))))
        dt = run(n)
    B = inp["q"].shape[0]
    sample = "first %d tokens of each of the %d sequences x %d heads (fp64 scan)" % (n, B, spec.H)
    return n * B / dt, oracle.hw_threads(), sample, n


def oracle_decode_sample(inp, spec, n_seq=16, n_steps=4):
    import oracle
    t = 0.0
    state = inp["state0"][:n_seq].double().numpy()
    for s in range(n_steps):
        args = [inp[k][s][:n_seq].to(torch.float64).numpy() for k in ("q", "k", "v", "g", "beta")]
        t0 = time.perf_counter()
        _, state = oracle.decode_step(*args, inp["scale"], state)
        t += time.perf_counter() - t0
    per_step_full = t / n_steps * (spec.N / n_seq)
    sample = ("%d of %d sequences x %d heads, %d steps; steps/s scaled to all %d sequences"
              % (n_seq, spec.N, spec.H, n_steps, spec.N))
    return 1.0 / per_step_full, oracle.hw_threads(), sample


# ------------------------------------------------------------------ GPU arm

def to_dev(inp, dev, keys):
    return {k: (None if inp[k] is None else inp[k].to(dev)) for k in keys}


def prefill_workload_variant(spec, dev, K, world, peaks):
    """Device-resident and end-to-end timings of one prefill workload."""
    from kimi_delta_attention_17_gb300 import chunk_fwd, chunk_fwd_host, workspace_size
    inp = kin.make_prefill(spec)
    keys = ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens")
    d_in = to_dev(inp, dev, keys)
    B, T, H, d = inp["q"].shape
    N = len(inp["lengths"])
    out = torch.empty((B, T, H, d), dtype=inp["q"].dtype, device=dev)
    fin = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, workspace_size(B, T, H, d, d, N, inp["q"].dtype)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def run(ev=None):
        chunk_fwd(d_in["q"], d_in["k"], d_in["v"], d_in["g"], d_in["beta"], inp["scale"],
                  d_in["init_state"], d_in["cu_seqlens"], out=out, final_state=fin, workspace=ws,
                  phase_events=ev)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    phase = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    v0 = torch.cuda.Event(enable_timing=True)
    v1 = torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for s in range(K):
        run()
    v1.record(stream)
    torch.cuda.synchronize()
    barrier()
    vms = max_over_ranks(v0.elapsed_time(v1), dev) / K
    # The phase marks (four event records per call, about 4 us each on a
    # 0.16 ms call) are taken in a second, untimed loop.
    for s in range(K):
        run(phase[s])
    torch.cuda.synchronize()
    tokens = B * T
    vbytes = prefill_bytes(spec, tokens, N, inp["init_state"] is not None)
    names = ["chunk_table", "intra_chunk", "state_pass"]
    phases = {n: statistics.mean(phase[s][i].elapsed_time(phase[s][i + 1]) for s in range(K))
              for i, n in enumerate(names)}
    if phases["state_pass"] < 0.02 * sum(phases.values()):  # the fused single launch
        phases = {"chunk_table": phases["chunk_table"],
                  "phase1_and_state_pass_fused": phases["intra_chunk"] + phases["state_pass"]}
    flops = prefill_flops(spec, tokens)
    # end to end: pinned host inputs through kda_chunk_fwd_host (host cu_seqlens)
    h_in = {k: (None if inp[k] is None else inp[k].pin_memory()) for k in keys}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    scratch = {}

    def e2e():
        chunk_fwd_host(h_in["q"], h_in["k"], h_in["v"], h_in["g"], h_in["beta"], inp["scale"],
                       h_in["init_state"], h_in["cu_seqlens"], out=h_out, final_state=h_fin,
                       window_tokens=16384, scratch=scratch)
    e2e()
    torch.cuda.synchronize()
    e_steps = max(1, min(K, 3))
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        e2e()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ems = max_over_ranks(e0.elapsed_time(e1), dev) / e_steps
    h2d = sum(x.numel() * x.element_size() for n, x in h_in.items()
              if x is not None and n != "cu_seqlens")
    d2h = h_out.numel() * h_out.element_size() + h_fin.numel() * h_fin.element_size()
    res = {
        "metric": "KDA prefill tokens/s (%s)" % spec.name,
        "value": units_for_world(tokens, world) / (vms / 1e3), "unit": "tokens/s",
        "ms_per_step": vms,
        "config": {"workload": spec.name, "B": B, "T": T, "H": H, "d_k": d, "d_v": d,
                   "num_seqs": N, "lengths": inp["lengths"] if inp["cu_seqlens"] is not None else None,
                   "init_state": inp["init_state"] is not None},
        "roofline": {"bound": "hbm", "kernel": "kda_chunk_fwd (all phases)",
                     "achieved": vbytes / (vms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": vbytes / (vms / 1e3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": measured_traffic(traffic_key(spec)),
                     "algorithmic_bytes_per_launch": vbytes,
                     "phases_ms": phases,
                     "tensor_tflops": flops / (vms / 1e3) / 1e12,
                     "tensor_frac": flops / (vms / 1e3) / 1e12 / peaks["bf16_tflops"]},
        "e2e": {"value": units_for_world(tokens, world) / (ems / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "kda_chunk_fwd_host (C ABI): pinned host buffers, 16384-token windows, "
                       "copies overlapped with the compute"},
    }
    del d_in, out, fin, ws, h_in, h_out, h_fin, scratch
    torch.cuda.empty_cache()
    return res


def bench_ours(args):
    from kimi_delta_attention_17_gb300 import (build, chunk_fwd, chunk_fwd_host, decode_host,
                                               decode_step, workspace_size)

    world, rank = init_dist("nccl")
    _, _, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    peaks = measured_peaks()

    # ---------------- prefill inputs
    spec = PREFILL_WORKLOADS[args.workload]
    if args.T:
        spec = kin.with_(spec, T=args.T)
    inp = kin.make_prefill(spec)
    keys = ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens")
    d_in = to_dev(inp, dev, keys)
    B, T, H, d = inp["q"].shape
    N = len(inp["lengths"])
    tokens = B * T
    dt_storage = inp["q"].dtype
    out = torch.empty((B, T, H, d), dtype=dt_storage, device=dev)
    fin = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, workspace_size(B, T, H, d, d, N, dt_storage)), dtype=torch.uint8,
                     device=dev)

    def prefill(phase_events=None):
        chunk_fwd(d_in["q"], d_in["k"], d_in["v"], d_in["g"], d_in["beta"], inp["scale"],
                  d_in["init_state"], d_in["cu_seqlens"], out=out, final_state=fin, workspace=ws,
                  phase_events=phase_events)

    # ---------------- decode inputs
    dspec = kin.DECODE_256
    dinp = kin.make_decode(dspec)
    dd = {k: dinp[k].to(dev) for k in ("q", "k", "v", "g", "beta")}
    state = dinp["state0"].to(dev)
    dout = torch.empty((dspec.N, dspec.H, dspec.d), dtype=dd["q"].dtype, device=dev)

    def decode_iteration():
        for t in range(dspec.steps):
            decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t],
                        dinp["scale"], state, out=dout)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        prefill()
        decode_iteration()
    torch.cuda.synchronize()

    # ---------------- timed prefill (device-resident inputs)
    K = args.steps
    phase = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    with ClockSampler(gpu_index) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(K):
            prefill(phase_events=phase[s])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
        prefill_ms = t_start.elapsed_time(t_end)

        # ---------------- timed decode
        d_start = torch.cuda.Event(enable_timing=True)
        d_end = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        d_start.record(stream)
        for _ in range(K):
            decode_iteration()
        d_end.record(stream)
        torch.cuda.synchronize()
        barrier()
        decode_ms = d_start.elapsed_time(d_end)
    clocks = clk.summary()

    # ---------------- end to end through host buffers (pinned), prefill: the C entry
    # kda_chunk_fwd_host (through chunk_fwd_host), which copies each 16384-token
    # window in while the previous one runs and its outputs back while the next
    # runs. Timed before the variants allocate and free their own buffers.
    h_in = {k: (None if inp[k] is None else inp[k].pin_memory()) for k in keys}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for n, t in h_in.items()
              if t is not None and n != "cu_seqlens")
    d2h = h_out.numel() * h_out.element_size() + h_fin.numel() * h_fin.element_size()
    e2e_steps = max(1, min(K, 3))
    host_scratch = {}

    def e2e_prefill():
        chunk_fwd_host(h_in["q"], h_in["k"], h_in["v"], h_in["g"], h_in["beta"],
                       inp["scale"], h_in["init_state"], h_in["cu_seqlens"], out=h_out,
                       final_state=h_fin, window_tokens=16384, scratch=host_scratch)
    e2e_prefill()  # first call sizes the segment buffers
    barrier()
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(e2e_steps):
        e2e_prefill()
    e_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), dev)
    e2e_tok_s = units_for_world(tokens, world) * e2e_steps / (e2e_ms / 1e3)

    # ---------------- end to end, decode: the public host-buffer call (decode_host),
    # step t + 1's inputs copied in while step t runs
    hd = {k: dinp[k].pin_memory() for k in ("q", "k", "v", "g", "beta")}
    h_dout = torch.empty((dspec.steps,) + tuple(dout.shape), dtype=dout.dtype).pin_memory()
    d_h2d = sum(hd[k][0].numel() * hd[k][0].element_size() for k in hd)
    d_d2h = dout.numel() * dout.element_size()
    dec_scratch = {}
    decode_host(hd["q"], hd["k"], hd["v"], hd["g"], hd["beta"], dinp["scale"], state,
                out=h_dout, scratch=dec_scratch)
    barrier()
    torch.cuda.synchronize()
    de_start = torch.cuda.Event(enable_timing=True)
    de_end = torch.cuda.Event(enable_timing=True)
    de_start.record(stream)
    decode_host(hd["q"], hd["k"], hd["v"], hd["g"], hd["beta"], dinp["scale"], state,
                out=h_dout, scratch=dec_scratch)
    de_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    de_ms = max_over_ranks(de_start.elapsed_time(de_end), dev)
    del h_in, h_out, h_fin, hd, h_dout, host_scratch, dec_scratch

    # ---------------- variants: the options of kda_chunk_fwd_opt / kda_decode_step_opt on the
    # same resident inputs (one channel of g as the per-head decay; g as gate logits)
    g_head = d_in["g"][..., 0].contiguous()
    variant_defs = {
        "gated_deltanet": (dict(decay="scalar"), g_head, 4),
        "deltanet": (dict(decay="none"), None, 0),
        "kda_fused_prologue": (dict(gate="logsigmoid", l2norm_qk=True), d_in["g"], 4 * d),
    }
    variants = {}
    for name, (opts, gv, gbytes) in variant_defs.items():
        def run_variant():
            chunk_fwd(d_in["q"], d_in["k"], d_in["v"], gv, d_in["beta"], inp["scale"],
                      d_in["init_state"], d_in["cu_seqlens"], out=out, final_state=fin,
                      workspace=ws, **opts)
        run_variant()
        torch.cuda.synchronize()
        v0 = torch.cuda.Event(enable_timing=True)
        v1 = torch.cuda.Event(enable_timing=True)
        v0.record(stream)
        for _ in range(K):
            run_variant()
        v1.record(stream)
        torch.cuda.synchronize()
        vms = max_over_ranks(v0.elapsed_time(v1), dev) / K
        vbytes = prefill_bytes_g(spec, tokens, N, inp["init_state"] is not None, gbytes)
        variants[name] = {
            "metric": "prefill tokens/s (%s, %s)" % (spec.name, ", ".join(
                "%s=%s" % kv for kv in sorted(opts.items()))),
            "value": units_for_world(tokens, world) / (vms / 1e3), "unit": "tokens/s",
            "ms_per_step": vms,
            "roofline": {"bound": "hbm", "achieved": vbytes / (vms / 1e3) / 1e9,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": vbytes / (vms / 1e3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                         "algorithmic_bytes_per_launch": vbytes}}

    # The same prefill as two launches (phase 1 on every SM, then the state
    # pass with 32-column slabs), with the time of each phase.
    tl_phase = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]

    def two_launches(ev=None):
        chunk_fwd(d_in["q"], d_in["k"], d_in["v"], d_in["g"], d_in["beta"], inp["scale"],
                  d_in["init_state"], d_in["cu_seqlens"], out=out, final_state=fin, workspace=ws,
                  phase_events=ev, fused=False)
    two_launches()
    torch.cuda.synchronize()
    v0 = torch.cuda.Event(enable_timing=True)
    v1 = torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for s in range(K):
        two_launches()
    v1.record(stream)
    torch.cuda.synchronize()
    tl_ms = max_over_ranks(v0.elapsed_time(v1), dev) / K
    # The phase marks (four event records per call) outside the timed loop.
    for s in range(K):
        two_launches(tl_phase[s])
    torch.cuda.synchronize()
    tl_bytes = prefill_bytes(spec, tokens, N, inp["init_state"] is not None)
    variants["prefill_two_launches"] = {
        "metric": "KDA prefill tokens/s (%s, fused=False)" % spec.name,
        "value": units_for_world(tokens, world) / (tl_ms / 1e3), "unit": "tokens/s",
        "ms_per_step": tl_ms,
        "phases_ms": {n: statistics.mean(tl_phase[s][i].elapsed_time(tl_phase[s][i + 1])
                                         for s in range(K))
                      for i, n in enumerate(("chunk_table", "intra_chunk", "state_pass"))},
        "roofline": {"bound": "hbm", "achieved": tl_bytes / (tl_ms / 1e3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": tl_bytes / (tl_ms / 1e3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "algorithmic_bytes_per_launch": tl_bytes}}

    # The other prefill workloads of the metric's shape (the two-sequence
    # 4096-token batch on 16 heads and the 8 packed sequences of mixed lengths
    # on 32 heads), each timed on the device and end to end through the
    # host-buffer entry point, with per-phase times.
    if not args.no_workload_variants:
        for vname, vspec in (("prefill_b2_h16_t4096", kin.PREFILL_B2),
                             ("prefill_varlen_8seq_h32", kin.VARLEN_8)):
            variants[vname] = prefill_workload_variant(vspec, dev, K, world, peaks)

    # Few (sequence, head) chains: the first 4 heads of the same inputs (a
    # 4-head shard of the workload) with one serial state chain per head and
    # with the automatic segmented state pass (chunk-level parallel prefix).
    if inp["cu_seqlens"] is None and H >= 4:
        sub = {n: (None if d_in[n] is None else d_in[n][:, :, :4].contiguous())
               for n in ("q", "k", "v", "g", "beta")}
        sub_init = None if d_in["init_state"] is None else d_in["init_state"][:, :4].contiguous()
        sub_out = torch.empty_like(sub["v"])
        sub_fin = torch.empty((N, 4, d, d), dtype=torch.float32, device=dev)
        sub_ws = torch.empty(max(1, workspace_size(B, T, 4, d, d, N, dt_storage)),
                             dtype=torch.uint8, device=dev)
        sub_spec = kin.with_(spec, H=4)
        for name, segs in (("four_heads_serial_chain", 1), ("four_heads_parallel_prefix", 0)):
            def run_sub():
                chunk_fwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], inp["scale"],
                          sub_init, None, out=sub_out, final_state=sub_fin, workspace=sub_ws,
                          segments=segs)
            run_sub()
            torch.cuda.synchronize()
            v0 = torch.cuda.Event(enable_timing=True)
            v1 = torch.cuda.Event(enable_timing=True)
            v0.record(stream)
            for _ in range(K):
                run_sub()
            v1.record(stream)
            torch.cuda.synchronize()
            vms = max_over_ranks(v0.elapsed_time(v1), dev) / K
            vbytes = prefill_bytes(sub_spec, tokens, N, sub_init is not None)
            variants[name] = {
                "metric": "prefill tokens/s (%s restricted to 4 heads, segments=%s)" % (
                    spec.name, "auto" if segs == 0 else segs),
                "value": units_for_world(tokens, world) / (vms / 1e3), "unit": "tokens/s",
                "ms_per_step": vms,
                "roofline": {"bound": "hbm", "achieved": vbytes / (vms / 1e3) / 1e9,
                             "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": vbytes / (vms / 1e3) / 1e9 / peaks["hbm_gbs"],
                             "traffic": None, "algorithmic_bytes_per_launch": vbytes}}
        del sub, sub_out, sub_ws

    # Output gate + RMS normalisation (kda_output_gate_rmsnorm) on the prefill's
    # output, gate logits drawn on the device: o and z read, out written.
    from kimi_delta_attention_17_gb300 import output_gate_rmsnorm
    zgate = torch.randn(out.shape, device=dev, dtype=out.dtype,
                        generator=torch.Generator(device=dev).manual_seed(17))
    wnorm = torch.ones(d, device=dev)
    eout = torch.empty_like(out)
    output_gate_rmsnorm(out, zgate, wnorm, out=eout)
    torch.cuda.synchronize()
    v0 = torch.cuda.Event(enable_timing=True)
    v1 = torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for _ in range(K):
        output_gate_rmsnorm(out, zgate, wnorm, out=eout)
    v1.record(stream)
    torch.cuda.synchronize()
    ems = max_over_ranks(v0.elapsed_time(v1), dev) / K
    ebytes = 3 * out.numel() * out.element_size() + wnorm.numel() * 4
    variants["output_gate_rmsnorm"] = {
        "metric": "gated RMSNorm epilogue tokens/s (%s outputs)" % spec.name,
        "value": units_for_world(tokens, world) / (ems / 1e3), "unit": "tokens/s",
        "ms_per_step": ems,
        "roofline": {"bound": "hbm", "achieved": ebytes / (ems / 1e3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ebytes / (ems / 1e3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "algorithmic_bytes_per_launch": ebytes}}
    # The same gate fused into the prefill (kda_chunk_fwd_gated): the outputs
    # leave the state pass gated and normalised, so o is written once and
    # never re-read.
    fout = torch.empty_like(out)

    def fused_prefill():
        chunk_fwd(d_in["q"], d_in["k"], d_in["v"], d_in["g"], d_in["beta"], inp["scale"],
                  d_in["init_state"], d_in["cu_seqlens"], out=fout, final_state=fin, workspace=ws,
                  out_gate=zgate, norm_weight=wnorm)
    fused_prefill()
    torch.cuda.synchronize()
    v0 = torch.cuda.Event(enable_timing=True)
    v1 = torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for _ in range(K):
        fused_prefill()
    v1.record(stream)
    torch.cuda.synchronize()
    fms = max_over_ranks(v0.elapsed_time(v1), dev) / K
    fbytes = prefill_bytes(spec, tokens, N, inp["init_state"] is not None) + \
        out.numel() * out.element_size() + wnorm.numel() * 4   # + z read
    variants["prefill_fused_gate_rmsnorm"] = {
        "metric": "KDA prefill with fused output gate + RMSNorm, tokens/s (%s)" % spec.name,
        "value": units_for_world(tokens, world) / (fms / 1e3), "unit": "tokens/s",
        "ms_per_step": fms,
        "roofline": {"bound": "hbm", "achieved": fbytes / (fms / 1e3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": fbytes / (fms / 1e3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                     "algorithmic_bytes_per_launch": fbytes}}
    del zgate, eout, fout

    def decode_fused():
        for t in range(dspec.steps):
            decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t],
                        dinp["scale"], state, out=dout, gate="logsigmoid", l2norm_qk=True)
    decode_fused()
    torch.cuda.synchronize()
    v0 = torch.cuda.Event(enable_timing=True)
    v1 = torch.cuda.Event(enable_timing=True)
    v0.record(stream)
    for _ in range(K):
        decode_fused()
    v1.record(stream)
    torch.cuda.synchronize()
    dfms = max_over_ranks(v0.elapsed_time(v1), dev) / (K * dspec.steps)
    variants["decode_fused_prologue"] = {
        "metric": "decode steps/s (%s, gate=logsigmoid, l2norm_qk=True)" % dspec.name,
        "value": world / (dfms / 1e3), "unit": "steps/s", "ms_per_step": dfms,
        "roofline": {"bound": "hbm", "achieved": decode_bytes(dspec) / (dfms / 1e3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": decode_bytes(dspec) / (dfms / 1e3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": None, "algorithmic_bytes_per_launch": decode_bytes(dspec)}}

    # Small-batch decode (4 sequences x the same heads, 128 steps): the steps
    # are too short for per-call host work to hide, so they are timed eagerly
    # (one C call per step) and as one CUDA-graph replay of all the steps.
    from kimi_delta_attention_17_gb300 import DecodeGraph
    sspec = kin.with_(dspec, N=4, name="decode bf16 4 seqs x H=%d d=%d, %d steps" % (
        dspec.H, dspec.d, dspec.steps))
    sinp = kin.make_decode(sspec)
    sb = {n: sinp[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    sstate = sinp["state0"].to(dev)
    sout = torch.empty(tuple(sb["v"].shape[1:]), dtype=sb["v"].dtype, device=dev)

    def small_eager():
        for t in range(sspec.steps):
            decode_step(sb["q"][t], sb["k"][t], sb["v"][t], sb["g"][t], sb["beta"][t],
                        sinp["scale"], sstate, out=sout)
    small_graph = DecodeGraph(sb["q"], sb["k"], sb["v"], sb["g"], sb["beta"], sinp["scale"],
                              sstate)
    sbytes = decode_bytes(sspec)
    for name, fn in (("decode_small_batch_eager", small_eager),
                     ("decode_small_batch_graph", small_graph.replay)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        v0 = torch.cuda.Event(enable_timing=True)
        v1 = torch.cuda.Event(enable_timing=True)
        v0.record(stream)
        for _ in range(K):
            fn()
        v1.record(stream)
        torch.cuda.synchronize()
        sms = max_over_ranks(v0.elapsed_time(v1), dev) / (K * sspec.steps)
        variants[name] = {
            "metric": "decode steps/s (%s, %s)" % (
                sspec.name, "one C call per step" if name.endswith("eager") else
                "all steps replayed as one CUDA graph"),
            "value": world / (sms / 1e3), "unit": "steps/s", "ms_per_step": sms,
            "roofline": {"bound": "hbm", "achieved": sbytes / (sms / 1e3) / 1e9,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": sbytes / (sms / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "traffic": None, "algorithmic_bytes_per_launch": sbytes}}
    del small_graph

    prefill_ms = max_over_ranks(prefill_ms, dev)
    decode_ms = max_over_ranks(decode_ms, dev)
    names = ["chunk_table", "intra_chunk", "state_pass"]
    phase_ms = {n: statistics.mean(phase[s][i].elapsed_time(phase[s][i + 1]) for s in range(K))
                for i, n in enumerate(names)}
    ms_step = prefill_ms / K
    tok_per_s = units_for_world(tokens, world) * K / (prefill_ms / 1e3)
    pbytes = prefill_bytes(spec, tokens, N, inp["init_state"] is not None)
    # The fused prefill (phase 1 and the state pass in one cooperative launch)
    # records both phase marks after its one launch.
    fused_ran = phase_ms["state_pass"] < 0.02 * sum(phase_ms.values())
    if fused_ran:
        phase_ms = {"chunk_table": phase_ms["chunk_table"],
                    "phase1_and_state_pass_fused": phase_ms["intra_chunk"] + phase_ms["state_pass"]}
    dominant = max(phase_ms, key=phase_ms.get)

    steps_total = dspec.steps * K
    dec_steps_s = world * steps_total / (decode_ms / 1e3)
    dbytes = decode_bytes(dspec)
    dec_ms_launch = decode_ms / steps_total
    dec_gbs = dbytes / (dec_ms_launch / 1e3) / 1e9

    result = None
    if rank == 0:
        cpu_val, cores, sample, _ = oracle_prefill_sample(inp, spec, target_s=args.cpu_seconds)
        dcpu_val, dcores, dsample = oracle_decode_sample(dinp, dspec)
        achieved_gbs = pbytes / (ms_step / 1e3) / 1e9
        flops = prefill_flops(spec, tokens)
        result = {
            "metric": "KDA prefill tokens/s (%s)" % spec.name,
            "value": tok_per_s,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            # bf16 storage at d = 128 runs the tensor-core path (bf16 operands,
            # fp32 accumulation and state); everything else the fp32 path.
            "dtype": "bf16" if (spec.dtype == "bf16" and d == 128) else "f32",
            "data": "synthetic",
            "config": {"workload": spec.name, "B": B, "T": T, "H": H, "d_k": d, "d_v": d,
                       "chunk": 64, "storage": spec.dtype, "num_seqs": N,
                       "l2": "inputs and outputs (%.2f GB) larger than L2, no flush" % (pbytes / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm",
                         "kernel": "kda_chunk_fwd (all phases%s)" % (
                             ": tc_prefill_fused, one cooperative launch" if fused_ran else ""),
                         "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved_gbs / peaks["hbm_gbs"],
                         "traffic": measured_traffic(traffic_key(spec)),
                         "algorithmic_bytes_per_launch": pbytes,
                         "peak_source": peaks["source"],
                         "phases_ms": phase_ms, "dominant_phase": dominant,
                         "tensor_tflops": flops / (ms_step / 1e3) / 1e12,
                         "tensor_frac": flops / (ms_step / 1e3) / 1e12 / peaks["bf16_tflops"]},
            "cpu_baseline": {"value": cpu_val, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": e2e_tok_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "api": "kda_chunk_fwd_host (C ABI): pinned host buffers, 16384-token "
                           "windows, copies overlapped with the compute"},
            "gpu_launches": (2 if fused_ran else 3) * K + steps_total,
            "clocks": clocks,
            "variants": variants,
            "decode": {
                "metric": "KDA decode steps/s (%s)" % dspec.name,
                "value": dec_steps_s, "unit": "steps/s", "ms_per_step": dec_ms_launch,
                "roofline": {"bound": "hbm", "kernel": "decode_step_kernel",
                             "achieved": dec_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": dec_gbs / peaks["hbm_gbs"],
                             "traffic": measured_traffic("decode_256x32"),
                             "algorithmic_bytes_per_launch": dbytes},
                "e2e": {"value": world * dspec.steps / (de_ms / 1e3), "unit": "steps/s",
                        "h2d_bytes_per_step": d_h2d, "d2h_bytes_per_step": d_d2h,
                        "api": "kda_decode_host (C ABI): pinned host buffers, step t+1's "
                               "inputs in and step t-1's outputs out while step t runs"},
                "cpu_baseline": {"value": dcpu_val, "unit": "steps/s", "cores": dcores,
                                 "kind": "oracle", "sample": dsample},
            },
        }
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()
    return result


# ------------------------------------------------------------------ reference arm (the oracle)

def bench_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return None
    spec = PREFILL_WORKLOADS[args.workload]
    if args.T:
        spec = kin.with_(spec, T=args.T)
    inp = kin.make_prefill(spec)
    B = inp["q"].shape[0]
    # Size each step so the whole run stays within a few minutes.
    budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    _, cores, sample, n_tok = oracle_prefill_sample(inp, spec,
                                                    target_s=min(budget, args.cpu_seconds))
    times = []
    import oracle
    arr = {k: inp[k][:, :n_tok].to(torch.float64).numpy() for k in ("q", "k", "v", "g", "beta")}
    init = None if inp["init_state"] is None else inp["init_state"][:B].double().numpy()
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.scan(arr["q"], arr["k"], arr["v"], arr["g"], arr["beta"], inp["scale"], init)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    val = n_tok * B * len(times) / total
    return {
        "impl": "reference",
        "metric": "KDA prefill tokens/s (%s)" % spec.name,
        "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "B": B, "T": inp["q"].shape[1], "H": spec.H,
                   "d_k": spec.d, "d_v": spec.d, "chunk": 64, "storage": spec.dtype},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(PREFILL_WORKLOADS), default="long")
    ap.add_argument("--T", type=int, default=0, help="override the per-sequence length")
    ap.add_argument("--no-workload-variants", action="store_true",
                    help="skip the other prefill workloads (two-sequence and packed)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target duration of the oracle baseline sample")
    args = ap.parse_args(argv)
    res = bench_reference(args) if args.impl == "reference" else bench_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
