"""Seeded synthetic inputs for the KDA prefill and decode paths.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic, so both the CUDA path's tests/benchmark and the CPU oracle
can consume the very same buffers.

Recipe (one torch CPU ``Generator`` per workload, seeded with the workload's
seed; fixed draw order: sequence lengths, q, k, v, beta, g, initial state):

* q, k ~ N(0, 1), then L2-normalised over the key channels of each
  (token, head), then rounded to the storage dtype (bf16 or fp32);
* v ~ N(0, 1), rounded to the storage dtype;
* beta = sigmoid(N(0, 1)), fp32, one per (token, head);
* g = -softplus(N(0, 1) - 2), fp32, one per (token, head, key channel): the
  per-token log-decay log a_t, so a_t = exp(g) lies in (0, 1);
* the "mixture" gate: in each head, key channels [0, d_k/2) draw
  -softplus(N(0, 1) - 5) (slow, long half-lives) and [d_k/2, d_k) draw
  -softplus(N(0, 1)) (fast);
* initial states are zero or N(0, 0.1^2), fp32, [N, H, d_k, d_v];
* varlen lengths are uniform integers in [lo, hi], packed back to back and
  described by int32 ``cu_seqlens``;
* the query scale is d_k^{-1/2}, passed separately (q itself is not scaled).

Inputs of the options of kda_chunk_fwd_opt / kda_decode_step_opt
(``make_prefill_opts``, ``make_decode_opts``; same generator and draw order,
then the option-specific draws):

* with in-kernel normalisation, q and k are left raw: N(0, 1) times a
  per-(token, head) magnitude exp(N(0, 0.5^2));
* gate values by gate kind: "log" as above; "logsigmoid" logits z ~ N(2, 1)
  (log sigmoid(z) then has the base gate's distribution); "bounded" logits
  z ~ N(-4, 1) for a lower bound of -5 (mean log-decay near -0.1);
* decay layout: per channel [.., H, d_k], one per head [.., H] (Gated
  DeltaNet), or none (g is None).
"""
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class PrefillSpec:
    name: str
    H: int
    d: int
    B: int = 1
    T: int = 0                      # per-sequence length when lengths is None
    num_seqs: int = 0               # varlen: number of packed sequences
    lengths: Optional[Tuple[int, int]] = None   # varlen: uniform length range
    fixed_lengths: Optional[Tuple[int, ...]] = None  # varlen: explicit lengths
    dtype: str = "bf16"             # storage dtype of q, k, v and the output
    init: str = "zero"              # "zero" or "normal0.1"
    gate: str = "base"              # "base" or "mixture"
    seed: int = 0


@dataclass(frozen=True)
class DecodeSpec:
    name: str
    N: int
    H: int
    d: int
    steps: int
    dtype: str = "bf16"
    seed: int = 4


# The five workloads the method is exercised on. The first is small enough
# for the oracle to finish in seconds; the long prefill and the decode batch
# are the ones timed.
SMALL_FP32 = PrefillSpec("prefill fp32 B=1 H=2 T=256 d=64", H=2, d=64, B=1, T=256,
                         dtype="f32", seed=0)
PREFILL_B2 = PrefillSpec("prefill bf16 B=2 H=16 T=4096 d=128", H=16, d=128, B=2, T=4096, seed=1)
VARLEN_8 = PrefillSpec("varlen prefill bf16 8 seqs in [512,16384] H=32 d=128", H=32, d=128,
                       num_seqs=8, lengths=(512, 16384), init="normal0.1", gate="mixture", seed=2)
LONG_128K = PrefillSpec("prefill bf16 B=1 H=32 T=131072 d=128", H=32, d=128, B=1, T=131072,
                        seed=3)
DECODE_256 = DecodeSpec("decode bf16 256 seqs x H=32 d=128, 128 steps", N=256, H=32, d=128,
                        steps=128, seed=4)


def _dtype(name):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _unit(x):
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _gate(gen, shape, kind):
    d = shape[-1]
    if kind == "base":
        return -torch.nn.functional.softplus(torch.randn(shape, generator=gen) - 2.0)
    if kind == "mixture":
        z = torch.randn(shape, generator=gen)
        shift = torch.zeros(d)
        shift[: d // 2] = 5.0
        return -torch.nn.functional.softplus(z - shift)
    raise ValueError(kind)


def seq_lengths(spec: PrefillSpec):
    """Per-sequence lengths (list of ints) without drawing the tensors."""
    gen = torch.Generator().manual_seed(spec.seed)
    if spec.fixed_lengths is not None:
        return list(spec.fixed_lengths)
    if spec.lengths is not None:
        lo, hi = spec.lengths
        return [int(x) for x in torch.randint(lo, hi + 1, (spec.num_seqs,), generator=gen)]
    return [spec.T] * spec.B


def make_prefill(spec: PrefillSpec):
    """Returns a dict of CPU tensors: q, k, v [B, T, H, d] (storage dtype),
    g [B, T, H, d] fp32, beta [B, T, H] fp32, init_state [N, H, d, d] fp32 or
    None, cu_seqlens int32 [N+1] or None, scale (float), lengths (list)."""
    gen = torch.Generator().manual_seed(spec.seed)
    varlen = spec.lengths is not None or spec.fixed_lengths is not None
    if spec.fixed_lengths is not None:
        lengths = list(spec.fixed_lengths)
    elif spec.lengths is not None:
        lo, hi = spec.lengths
        lengths = [int(x) for x in torch.randint(lo, hi + 1, (spec.num_seqs,), generator=gen)]
    else:
        lengths = [spec.T] * spec.B
    if varlen:
        B, T = 1, sum(lengths)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    else:
        B, T = spec.B, spec.T
        cu = None
    H, d = spec.H, spec.d
    st = _dtype(spec.dtype)
    q = _unit(torch.randn((B, T, H, d), generator=gen)).to(st)
    k = _unit(torch.randn((B, T, H, d), generator=gen)).to(st)
    v = torch.randn((B, T, H, d), generator=gen).to(st)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=gen))
    g = _gate(gen, (B, T, H, d), spec.gate)
    N = len(lengths)
    if spec.init == "zero":
        init = None
    elif spec.init == "normal0.1":
        init = 0.1 * torch.randn((N, H, d, d), generator=gen)
    else:
        raise ValueError(spec.init)
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=init, cu_seqlens=cu,
                scale=d ** -0.5, lengths=lengths)


def make_decode(spec: DecodeSpec):
    """Returns a dict of CPU tensors for ``steps`` successive decode steps:
    q, k, v [steps, N, H, d] (storage dtype), g [steps, N, H, d] fp32,
    beta [steps, N, H] fp32, state0 [N, H, d, d] fp32 ~ N(0, 0.1^2), scale."""
    gen = torch.Generator().manual_seed(spec.seed)
    s, N, H, d = spec.steps, spec.N, spec.H, spec.d
    st = _dtype(spec.dtype)
    q = _unit(torch.randn((s, N, H, d), generator=gen)).to(st)
    k = _unit(torch.randn((s, N, H, d), generator=gen)).to(st)
    v = torch.randn((s, N, H, d), generator=gen).to(st)
    beta = torch.sigmoid(torch.randn((s, N, H), generator=gen))
    g = _gate(gen, (s, N, H, d), "base")
    state0 = 0.1 * torch.randn((N, H, d, d), generator=gen)
    return dict(q=q, k=k, v=v, g=g, beta=beta, state0=state0, scale=d ** -0.5)


def with_(spec, **kw):
    """A copy of a spec with some fields replaced (smaller parity variants)."""
    return replace(spec, **kw)


@dataclass(frozen=True)
class OptionsSpec:
    """Options of kda_chunk_fwd_opt / kda_decode_step_opt, as the binding names them."""
    decay: str = "channel"      # "channel", "scalar" or "none"
    gate: str = "log"           # "log", "logsigmoid" or "bounded"
    l2norm_qk: bool = False
    gate_lower: float = -5.0

    def kwargs(self):
        return dict(decay=self.decay, gate=self.gate, gate_lower=self.gate_lower,
                    l2norm_qk=self.l2norm_qk)


def _gate_values(gen, shape, gate):
    if gate == "log":
        return _gate(gen, shape, "base")
    if gate == "logsigmoid":
        return torch.randn(shape, generator=gen) + 2.0
    if gate == "bounded":
        return torch.randn(shape, generator=gen) - 4.0
    raise ValueError(gate)


def _opt_inputs(gen, lead, H, d, st, opts):
    """q, k, v, beta, g for the leading shape ``lead`` (tokens or steps x N)."""
    shape = lead + (H, d)
    if opts.l2norm_qk:
        q = torch.randn(shape, generator=gen)
        k = torch.randn(shape, generator=gen)
    else:
        q = _unit(torch.randn(shape, generator=gen))
        k = _unit(torch.randn(shape, generator=gen))
    v = torch.randn(shape, generator=gen).to(st)
    beta = torch.sigmoid(torch.randn(lead + (H,), generator=gen))
    if opts.decay == "channel":
        g = _gate_values(gen, shape, opts.gate)
    elif opts.decay == "scalar":
        g = _gate_values(gen, lead + (H,), opts.gate)
    elif opts.decay == "none":
        g = None
    else:
        raise ValueError(opts.decay)
    if opts.l2norm_qk:
        q = q * torch.exp(0.5 * torch.randn(lead + (H, 1), generator=gen))
        k = k * torch.exp(0.5 * torch.randn(lead + (H, 1), generator=gen))
    return q.to(st), k.to(st), v, beta, g


def make_prefill_opts(spec: PrefillSpec, opts: OptionsSpec):
    """make_prefill for the options: the same keys, with q, k raw when the
    kernel normalises them, and g shaped by the decay layout (None for "none")."""
    gen = torch.Generator().manual_seed(spec.seed)
    lengths = seq_lengths(spec)
    if spec.lengths is not None:
        torch.randint(spec.lengths[0], spec.lengths[1] + 1, (spec.num_seqs,), generator=gen)
    varlen = spec.lengths is not None or spec.fixed_lengths is not None
    if varlen:
        B, T = 1, sum(lengths)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    else:
        B, T = spec.B, spec.T
        cu = None
    H, d = spec.H, spec.d
    q, k, v, beta, g = _opt_inputs(gen, (B, T), H, d, _dtype(spec.dtype), opts)
    N = len(lengths)
    init = None if spec.init == "zero" else 0.1 * torch.randn((N, H, d, d), generator=gen)
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=init, cu_seqlens=cu,
                scale=d ** -0.5, lengths=lengths)


def make_decode_opts(spec: DecodeSpec, opts: OptionsSpec):
    """make_decode for the options (g [steps, N, H] for "scalar", None for "none")."""
    gen = torch.Generator().manual_seed(spec.seed)
    s, N, H, d = spec.steps, spec.N, spec.H, spec.d
    q, k, v, beta, g = _opt_inputs(gen, (s, N), H, d, _dtype(spec.dtype), opts)
    state0 = 0.1 * torch.randn((N, H, d, d), generator=gen)
    return dict(q=q, k=k, v=v, g=g, beta=beta, state0=state0, scale=d ** -0.5)


# ---------------------------------------------------------------- edge cases
# Heads of the edge-case inputs take, in turn (head h gets kind h mod 6):
#   0 "steep":   g ~ U[-40, 0] per channel and token (decays far beyond what a
#                factor spanning several tokens can carry in fp32)
#   1 "beta0":   beta = 0 (no write: pure decay of the initial state)
#   2 "beta1":   beta = 1 (the overwrite case: with a unit key the write
#                replaces the value stored under that key)
#   3 "nodecay": g = 0 (a = 1, DeltaNet)
#   4 "mixed":   each token, with probability 1/2, g ~ U[-40, 0] per channel,
#                else the base gate (steep and gentle blocks side by side)
#   5 "base":    the base recipe
EDGE_KINDS = ("steep", "beta0", "beta1", "nodecay", "mixed", "base")


def _edge_override(gen, beta, g):
    """Applies the per-head kinds above, in place, to beta [..., H] and g
    [..., H, d] drawn by the base recipe (draw order: steep g, mixed mask,
    mixed g)."""
    H = beta.shape[-1]
    steep = -40.0 * torch.rand(g.shape, generator=gen)
    mask = torch.rand(g.shape[:-1] + (1,), generator=gen) < 0.5
    steep2 = -40.0 * torch.rand(g.shape, generator=gen)
    for h in range(H):
        kind = EDGE_KINDS[h % len(EDGE_KINDS)]
        if kind == "steep":
            g[..., h, :] = steep[..., h, :]
        elif kind == "beta0":
            beta[..., h] = 0.0
        elif kind == "beta1":
            beta[..., h] = 1.0
        elif kind == "nodecay":
            g[..., h, :] = 0.0
        elif kind == "mixed":
            g[..., h, :] = torch.where(mask[..., h, :], steep2[..., h, :], g[..., h, :])


def make_prefill_edge(spec: PrefillSpec):
    """make_prefill, then the per-head edge-case kinds of EDGE_KINDS (the
    base draws first, in the usual order, then the overrides)."""
    inp = make_prefill(spec)
    gen = torch.Generator().manual_seed(spec.seed + 1000)
    _edge_override(gen, inp["beta"], inp["g"])
    return inp


def make_decode_edge(spec: DecodeSpec):
    """make_decode, then the per-head edge-case kinds of EDGE_KINDS."""
    inp = make_decode(spec)
    gen = torch.Generator().manual_seed(spec.seed + 1000)
    _edge_override(gen, inp["beta"], inp["g"])
    return inp


def steep_logits(spec_seed, shape):
    """Gate logits z ~ N(-12, 8^2) (seeded): through the log-sigmoid gate they
    give per-token log-decays from about -40 to 0, mostly steep."""
    gen = torch.Generator().manual_seed(spec_seed + 2000)
    return -12.0 + 8.0 * torch.randn(shape, generator=gen)
