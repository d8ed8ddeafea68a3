"""Failure detection on the GPU without a fault: a bounded device wait that
nothing completes gives up, reports KDA_ERR_TIMEOUT through a status word the
host reads (the same wait helper and reporting path as the prefill kernels'
workspace status word), and the context stays usable for the next call."""
import pytest
import torch

from kimi_delta_attention_17_gb300 import _lib, build, chunk_fwd
from kimi_delta_attention_17_gb300.inputs import PrefillSpec, make_prefill
from tests.helpers import assert_parity, f64, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = _lib.lib().kda_selftest_wait_timeout(status.data_ptr(), 20000,
                                             torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 5  # KDA_ERR_TIMEOUT
    # The context is intact: a prefill right after it still meets parity.
    inp = make_prefill(PrefillSpec("after timeout", H=2, d=128, B=1, T=100, seed=18))
    out, fin = chunk_fwd(*(inp[n].cuda() for n in ("q", "k", "v", "g", "beta")), inp["scale"])
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_prefill(inp)
    assert_parity(f64(out), ref_out, "bf16", "O after a timeout")
    assert_parity(f64(fin), ref_fin, "bf16", "final state after a timeout")
