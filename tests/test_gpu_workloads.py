"""Parity at the full sizes of the five workloads, in the launch configuration
the benchmark times. The GPU always processes the whole workload; the oracle
checks an exact sample of it: every head of the B=2, T=4096 prefill, two of the
32 heads (all tokens, all sequences) of the varlen and 131072-token prefills,
and every head of 6 of the 256 decode sequences over all 128 steps (heads and
sequences are independent, so a subset is checked element by element)."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_17_gb300 import build, chunk_fwd, decode_step
from kimi_delta_attention_17_gb300.inputs import (DECODE_256, LONG_128K, PREFILL_B2, SMALL_FP32,
                                                  VARLEN_8, make_decode, make_prefill)
from tests.helpers import assert_parity, f64, oracle_prefill

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def gpu_prefill(inp):
    dev = "cuda"
    q, k, v, g, beta = (inp[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    init = None if inp["init_state"] is None else inp["init_state"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], init, cu)
    torch.cuda.synchronize()
    return out, fin


@pytest.mark.parametrize("spec,heads", [
    (SMALL_FP32, None),
    (PREFILL_B2, None),
    (VARLEN_8, [0, 31]),
    (LONG_128K, [0, 17]),
], ids=["small-fp32", "b2-h16-t4096", "varlen-8seq-h32", "t131072-h32"])
def test_prefill_workload(spec, heads):
    inp = make_prefill(spec)
    out, fin = gpu_prefill(inp)
    sel = slice(None) if heads is None else heads
    out_s = f64(out[:, :, sel])
    fin_s = f64(fin[:, sel])
    del out, fin
    ref_out, ref_fin = oracle_prefill(inp, heads=heads)
    eo = assert_parity(out_s, ref_out, spec.dtype, "O")
    es = assert_parity(fin_s, ref_fin, spec.dtype, "final state")
    print("\n%s: O max|err| %.3g rel %.3g; final state max|err| %.3g rel %.3g"
          % (spec.name, eo[0], eo[1], es[0], es[1]))


def test_decode_workload():
    spec = DECODE_256
    inp = make_decode(spec)
    seqs = [0, 1, 77, 128, 200, 255]
    dev = "cuda"
    q, k, v, g, beta = (inp[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    state = inp["state0"].to(dev)
    ref_state = f64(inp["state0"][seqs])
    outs = []
    for t in range(spec.steps):
        out = decode_step(q[t], k[t], v[t], g[t], beta[t], inp["scale"], state)
        outs.append(out[seqs].float().cpu())
    torch.cuda.synchronize()
    for t in range(spec.steps):
        ref_out, ref_state = oracle.decode_step(*(f64(inp[n][t][seqs]) for n in ("q", "k", "v", "g", "beta")),
                                                inp["scale"], ref_state)
        assert_parity(f64(outs[t]), ref_out, spec.dtype, "decode O step %d" % t)
    es = assert_parity(f64(state[seqs]), ref_state, spec.dtype, "decode state after %d steps" % spec.steps)
    print("\n%s: state after %d steps max|err| %.3g rel %.3g" % (spec.name, spec.steps, es[0], es[1]))


def test_four_head_shard_parallel_prefix():
    """The 131072-token prefill on 4 heads, as the benchmark times its
    parallel-prefix variant (automatic: 6 segments of 342 chunks): two heads
    against the oracle over all tokens, and all four against the serial chain."""
    from kimi_delta_attention_17_gb300.inputs import with_
    spec = with_(LONG_128K, H=4, name="prefill bf16 B=1 H=4 T=131072 d=128")
    inp = make_prefill(spec)
    dev = "cuda"
    args = [inp[n].to(dev) for n in ("q", "k", "v", "g", "beta")]
    out_p, fin_p = chunk_fwd(*args, inp["scale"], segments=0)
    out_s, fin_s = chunk_fwd(*args, inp["scale"], segments=1)
    torch.cuda.synchronize()
    for a, b, what in ((out_p, out_s, "O"), (fin_p, fin_s, "final state")):
        a64, b64 = a.double(), b.double()
        rel = float(torch.linalg.norm(a64 - b64) / torch.linalg.norm(b64))
        assert rel < 2e-4, (what, rel)
    heads = [0, 3]
    out_h, fin_h = f64(out_p[:, :, heads]), f64(fin_p[:, heads])
    del out_p, fin_p, out_s, fin_s
    ref_out, ref_fin = oracle_prefill(inp, heads=heads)
    eo = assert_parity(out_h, ref_out, spec.dtype, "O")
    es = assert_parity(fin_h, ref_fin, spec.dtype, "final state")
    print("\n%s, parallel prefix: O max|err| %.3g rel %.3g; final state max|err| %.3g rel %.3g"
          % (spec.name, eo[0], eo[1], es[0], es[1]))


def test_varlen_workload_every_head():
    """The 8-sequence packed prefill (mixture gates: half the key channels with
    half-lives of hundreds of tokens; nonzero initial states), where the bf16
    error budget is tightest: all 32 heads against the oracle, and each head on
    its own within the bounds. Prints the worst head's errors."""
    spec = VARLEN_8
    inp = make_prefill(spec)
    out, fin = gpu_prefill(inp)
    out64, fin64 = f64(out), f64(fin)
    del out, fin
    ref_out, ref_fin = oracle_prefill(inp)
    assert_parity(out64, ref_out, spec.dtype, "O")
    assert_parity(fin64, ref_fin, spec.dtype, "final state")
    worst = {}
    for h in range(spec.H):
        for what, got, ref in (("O", out64[:, :, h], ref_out[:, :, h]),
                               ("final state", fin64[:, h], ref_fin[:, h])):
            m, r = assert_parity(got, ref, spec.dtype, "%s, head %d" % (what, h))
            if r > worst.get(what, (0, 0.0, 0.0))[2]:
                worst[what] = (h, m, r)
    for what, (h, m, r) in worst.items():
        print("\n%s, every head: worst %s is head %d: max|err| %.3g rel %.3g"
              % (spec.name, what, h, m, r))
