"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle, on
small seeded inputs that span several chunks, ragged tails and the edge cases
(empty sequences, sequences shorter than a chunk, NULL initial/final states,
in-place state carry, both head sizes, both storage dtypes)."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_17_gb300 import build, chunk_fwd, decode_step, workspace_size
from kimi_delta_attention_17_gb300.inputs import (SMALL_FP32, DecodeSpec, PrefillSpec, make_decode,
                                                  make_prefill)
from tests.helpers import assert_parity, f64, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def run_prefill(inp, alias=False, want_final=True):
    dev = "cuda"
    q, k, v, g, beta = (inp[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    init = None if inp["init_state"] is None else inp["init_state"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    final = init if alias else None
    B, T, H, d = q.shape
    ws = torch.empty(workspace_size(B, T, H, d, d, len(inp["lengths"]), q.dtype),
                     dtype=torch.uint8, device=dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], init, cu, final_state=final,
                         output_final_state=want_final, workspace=ws)
    torch.cuda.synchronize()
    # The device status word (first int of the workspace) stays 0 unless a
    # bounded device-side wait gave up.
    assert int(ws[:4].view(torch.int32).item()) == 0
    return f64(out), (None if fin is None else f64(fin))


def check_prefill(spec, **kw):
    inp = make_prefill(spec)
    out, fin = run_prefill(inp, **kw)
    ref_out, ref_fin = oracle_prefill(inp)
    assert_parity(out, ref_out, spec.dtype, "O")
    if fin is not None:
        assert_parity(fin, ref_fin, spec.dtype, "final state")
    return inp


def test_small_fp32_workload():
    """The fp32 workload B=1, H=2, T=256, d=64 (zero initial state, seed 0)."""
    check_prefill(SMALL_FP32)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_batches(d, dtype):
    spec = PrefillSpec("ragged", H=3, d=d, B=2, T=300, dtype=dtype, init="normal0.1", seed=11)
    check_prefill(spec)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_varlen_with_empty_and_short_sequences(dtype):
    spec = PrefillSpec("varlen edge", H=2, d=128, fixed_lengths=(0, 1, 63, 64, 65, 130, 0, 200),
                       dtype=dtype, init="normal0.1", gate="mixture", seed=12)
    inp = check_prefill(spec)
    # Zero-length sequences hand back their initial state exactly.
    _, fin = run_prefill(inp)
    for n in (0, 6):
        assert np.array_equal(fin[n], f64(inp["init_state"][n]))


def test_shorter_than_one_chunk():
    check_prefill(PrefillSpec("short", H=4, d=128, B=3, T=17, dtype="bf16", seed=13))


def test_null_initial_and_final_state():
    spec = PrefillSpec("nulls", H=2, d=128, B=1, T=150, dtype="bf16", init="zero", seed=14)
    inp = make_prefill(spec)
    out, fin = run_prefill(inp, want_final=False)
    assert fin is None
    ref_out, _ = oracle_prefill(inp)
    assert_parity(out, ref_out, "bf16", "O")


def test_in_place_state_carry():
    spec = PrefillSpec("alias", H=2, d=64, B=2, T=130, dtype="f32", init="normal0.1", seed=15)
    inp = make_prefill(spec)
    ref_out, ref_fin = oracle_prefill(inp)
    out, fin = run_prefill(inp, alias=True)
    assert_parity(out, ref_out, "f32", "O")
    assert_parity(fin, ref_fin, "f32", "final state")


def test_all_sequences_empty():
    spec = PrefillSpec("empty", H=2, d=128, fixed_lengths=(0, 0, 0), dtype="bf16",
                       init="normal0.1", seed=16)
    inp = make_prefill(spec)
    _, fin = run_prefill(inp)
    assert np.array_equal(fin, f64(inp["init_state"]))


def test_resume_matches_single_call():
    """Splitting a sequence and carrying final -> initial state reproduces one call."""
    spec = PrefillSpec("resume", H=2, d=128, B=1, T=256, dtype="f32", init="normal0.1", seed=17)
    inp = make_prefill(spec)
    out_all, fin_all = run_prefill(inp)
    first = dict(inp, **{n: inp[n][:, :128] for n in ("q", "k", "v", "g", "beta")})
    out_a, fin_a = run_prefill(first)
    second = dict(inp, **{n: inp[n][:, 128:].contiguous() for n in ("q", "k", "v", "g", "beta")})
    second["init_state"] = torch.from_numpy(fin_a).float()
    out_b, fin_b = run_prefill(second)
    assert np.abs(np.concatenate([out_a, out_b], 1) - out_all).max() <= 1e-5
    assert np.abs(fin_b - fin_all).max() <= 1e-5


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32"), (128, "f32")])
def test_decode_steps(d, dtype):
    spec = DecodeSpec("decode small", N=5, H=3, d=d, steps=6, dtype=dtype, seed=21)
    inp = make_decode(spec)
    state = inp["state0"].cuda().contiguous()
    ref_state = f64(inp["state0"])
    for t in range(spec.steps):
        args = [inp[n][t].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")]
        out = decode_step(*args, inp["scale"], state)
        torch.cuda.synchronize()
        ref_out, ref_state = oracle.decode_step(*(f64(inp[n][t]) for n in ("q", "k", "v", "g", "beta")),
                                                inp["scale"], ref_state)
        assert_parity(f64(out), ref_out, dtype, "decode O step %d" % t)
        assert_parity(f64(state), ref_state, dtype, "decode state step %d" % t)


def test_decode_equals_prefill():
    """T decode steps on the GPU reproduce a T-token GPU prefill."""
    spec = PrefillSpec("dp", H=2, d=128, B=3, T=70, dtype="f32", init="normal0.1", seed=22)
    inp = make_prefill(spec)
    out_p, fin_p = run_prefill(inp)
    state = inp["init_state"].cuda().clone()
    for t in range(spec.T):
        args = [inp[n][:, t].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")]
        out = decode_step(*args, inp["scale"], state)
        assert np.abs(f64(out) - out_p[:, t]).max() <= 1e-4
    torch.cuda.synchronize()
    assert np.abs(f64(state) - fin_p).max() <= 1e-4


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_more_sequences_than_table_threads(d, dtype):
    """1100 packed sequences of 0-70 tokens (some empty, some past one chunk):
    more sequences than the chunk table kernel has threads, and more than it
    ranks longest-first (their order is then the identity)."""
    rng = np.random.default_rng(13)
    lengths = tuple(int(x) for x in rng.integers(0, 71, size=1100))
    spec = PrefillSpec("many sequences", H=1, d=d, fixed_lengths=lengths, dtype=dtype,
                       init="normal0.1", seed=14)
    check_prefill(spec)
