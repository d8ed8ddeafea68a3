"""GPU parity of the segmented state pass (kda_options.segments; a chunk-level
parallel prefix over the affine chunk maps, tensor-core path) against the
fp64 oracle, and its agreement with the serial chain. Inputs span many chunks
with a ragged tail and nonzero initial states; segment counts cover the
automatic choice, two segments (no composition step), and counts that leave a
short last segment."""
import pytest
import torch

from kimi_delta_attention_17_gb300 import build, chunk_fwd, workspace_size
from kimi_delta_attention_17_gb300.inputs import PrefillSpec, make_prefill
from tests.helpers import assert_parity, f64, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def run(inp, segments, **kw):
    dev = "cuda"
    q, k, v, g, beta = (inp[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    init = None if inp["init_state"] is None else inp["init_state"].to(dev)
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    B, T, H, d = q.shape
    ws = torch.empty(workspace_size(B, T, H, d, d, len(inp["lengths"]), q.dtype),
                     dtype=torch.uint8, device=dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], init, cu, workspace=ws,
                         segments=segments, **kw)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    return out, fin


@pytest.mark.parametrize("segments", [0, 2, 3, 5, 12])
def test_segmented_prefill_parity(segments):
    """B=1, H=2, T=2000 (32 chunks, a 16-token tail): automatic (4 segments of
    8 chunks), and forced counts, against the oracle."""
    spec = PrefillSpec("seg", H=2, d=128, B=1, T=2000, init="normal0.1", seed=31)
    inp = make_prefill(spec)
    out, fin = run(inp, segments)
    ref_out, ref_fin = oracle_prefill(inp)
    assert_parity(f64(out), ref_out, "bf16", "O")
    assert_parity(f64(fin), ref_fin, "bf16", "final state")


@pytest.mark.parametrize("segments", [4, 7])
def test_segmented_batch_of_sequences(segments):
    """B=3 sequences of 700 tokens (11 chunks), one head: every sequence is
    segmented; a zero initial state."""
    spec = PrefillSpec("seg-b3", H=1, d=128, B=3, T=700, seed=32)
    inp = make_prefill(spec)
    out, fin = run(inp, segments)
    ref_out, ref_fin = oracle_prefill(inp)
    assert_parity(f64(out), ref_out, "bf16", "O")
    assert_parity(f64(fin), ref_fin, "bf16", "final state")


def test_segmented_matches_serial_chain():
    """The same inputs through the serial chain and through 6 segments: the
    two differ only by fp32 rounding of the state."""
    spec = PrefillSpec("seg-vs-serial", H=4, d=128, B=1, T=4096, init="normal0.1", seed=33)
    inp = make_prefill(spec)
    out1, fin1 = run(inp, 1)
    out6, fin6 = run(inp, 6)
    for a, b, name in ((out6, out1, "O"), (fin6, fin1, "final state")):
        a, b = a.double(), b.double()
        rel = float(torch.linalg.norm(a - b) / torch.linalg.norm(b))
        assert rel < 2e-4, (name, rel)
    ref_out, ref_fin = oracle_prefill(inp, heads=[0, 3])
    assert_parity(f64(out6)[:, :, [0, 3]], ref_out, "bf16", "O")
    assert_parity(f64(fin6)[:, [0, 3]], ref_fin, "bf16", "final state")


def test_segments_with_options_and_in_place_state():
    """Segments with a fused prologue (log-sigmoid gate, q/k normalisation) and
    final_state aliasing init_state."""
    from oracle.prologue import prepare
    import oracle
    from kimi_delta_attention_17_gb300.inputs import OptionsSpec, make_prefill_opts
    opts = OptionsSpec("channel", "logsigmoid", True)
    spec = PrefillSpec("seg-opt", H=2, d=128, B=1, T=1500, init="normal0.1", seed=34)
    inp = make_prefill_opts(spec, opts)
    dev = "cuda"
    q, k, v, g, beta = (inp[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    state = inp["init_state"].to(dev)
    out, fin = chunk_fwd(q, k, v, g, beta, inp["scale"], state, final_state=state, segments=4,
                         **opts.kwargs())
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    qo, ko, go = prepare(f64(inp["q"]), f64(inp["k"]), f64(inp["g"]), **opts.kwargs())
    ref_out, ref_fin = oracle.scan(qo, ko, f64(inp["v"]), go, f64(inp["beta"]), inp["scale"],
                                   f64(inp["init_state"]))
    assert_parity(f64(out), ref_out, "bf16", "O")
    assert_parity(f64(fin), ref_fin, "bf16", "final state")


def test_packed_sequences_ignore_segments():
    """Packed batches keep the serial chain whatever the option says."""
    spec = PrefillSpec("seg-packed", H=2, d=128, fixed_lengths=(900, 300, 1), init="normal0.1",
                       seed=35)
    inp = make_prefill(spec)
    out1, fin1 = run(inp, 1)
    out5, fin5 = run(inp, 5)
    assert torch.equal(out1, out5) and torch.equal(fin1, fin5)
