"""The chunk table's device check of cu_seqlens: offsets that do not start
at 0, decrease, or do not end at T make the call compute nothing and report
KDA_ERR_INVALID_ARGUMENT in the workspace status word (both prefill paths);
outputs and final states stay as they were."""
import pytest
import torch

from kimi_delta_attention_17_gb300 import _lib, build, chunk_fwd, workspace_size

pytestmark = pytest.mark.gpu

INVALID = 1  # KDA_ERR_INVALID_ARGUMENT


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
@pytest.mark.parametrize("offsets,ok", [((0, 100, 300), True),
                                        ((0, 200, 100, 300), False),   # a decrease
                                        ((4, 100, 300), False),        # does not start at 0
                                        ((0, 100, 299), False)])       # does not end at T
def test_cu_seqlens_device_check(d, dtype, offsets, ok):
    dev = "cuda"
    T, H = 300, 2
    gen = torch.Generator(device="cpu").manual_seed(51)
    q = torch.nn.functional.normalize(torch.randn(1, T, H, d, generator=gen), dim=-1).to(dtype).to(dev)
    k = torch.nn.functional.normalize(torch.randn(1, T, H, d, generator=gen), dim=-1).to(dtype).to(dev)
    v = torch.randn(1, T, H, d, generator=gen).to(dtype).to(dev)
    g = (-torch.rand(1, T, H, d, generator=gen) * 0.1).to(dev)
    beta = torch.rand(1, T, H, generator=gen).to(dev)
    cu = torch.tensor(offsets, dtype=torch.int32, device=dev)
    N = len(offsets) - 1
    ws = torch.empty(workspace_size(1, T, H, d, d, N, dtype), dtype=torch.uint8, device=dev)
    out = torch.full((1, T, H, d), 7.0, dtype=dtype, device=dev)
    fin = torch.full((N, H, d, d), 7.0, dtype=torch.float32, device=dev)
    chunk_fwd(q, k, v, g, beta, d ** -0.5, None, cu, out=out, final_state=fin, workspace=ws)
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).item())
    if ok:
        assert status == 0
        assert not torch.equal(fin, torch.full_like(fin, 7.0))
    else:
        assert status == INVALID
        assert _lib.lib().kda_status_string(status).decode() == "KDA_ERR_INVALID_ARGUMENT"
        assert bool((out == 7.0).all()) and bool((fin == 7.0).all())
