"""CPU-only checks of the C ABI: the library builds and loads, exports every
function include/kda.h declares, and its host-side validation rejects bad
arguments before any CUDA call (so these run without a GPU)."""
import ctypes

import pytest

from kimi_delta_attention_17_gb300 import _lib, build

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    names = _lib.declared_symbols()
    assert set(names) >= {"kda_chunk_fwd", "kda_decode_step", "kda_chunk_fwd_workspace_size",
                          "kda_status_string"}
    for n in names:
        assert hasattr(L, n), "libkda.so does not export %s" % n


def test_status_strings(L):
    for code, name in _lib.STATUS_NAMES.items():
        assert L.kda_status_string(code).decode() == name
    assert L.kda_status_string(99).decode() == "KDA_ERR_UNKNOWN"


def test_workspace_size_rules(L):
    ws = L.kda_chunk_fwd_workspace_size
    assert ws(2, 4096, 16, 128, 128, 2, 1) > 0
    assert ws(1, 100, 2, 64, 64, 1, 0) > 0
    # Unsupported head sizes and invalid shapes report 0.
    assert ws(1, 64, 1, 96, 96, 1, 1) == 0
    assert ws(1, 64, 1, 128, 64, 1, 1) == 0
    assert ws(2, 64, 1, 128, 128, 3, 1) == 0      # packed needs B == 1
    assert ws(1, 64, 0, 128, 128, 1, 1) == 0
    # Monotone in T and H; packed bound covers one extra chunk per sequence.
    assert ws(1, 128, 4, 64, 64, 1, 1) < ws(1, 129, 4, 64, 64, 1, 1)
    assert ws(1, 1000, 4, 64, 64, 1, 1) < ws(1, 1000, 8, 64, 64, 1, 1)
    assert ws(1, 1000, 4, 64, 64, 1, 1) < ws(1, 1000, 4, 64, 64, 5, 1)
    # Zero tokens with sequences to carry is valid.
    assert ws(1, 0, 4, 64, 64, 3, 1) > 0


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced on these paths


def fwd(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=0.1, init=None, cu=None, out=FAKE,
             fin=FAKE, B=1, T=64, H=1, dk=64, dv=64, N=1, dt=1, ws=FAKE, wsb=1 << 40, stream=None)
    a.update(kw)
    return L.kda_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["init"],
                           a["cu"], a["out"], a["fin"], a["B"], a["T"], a["H"], a["dk"], a["dv"],
                           a["N"], a["dt"], a["ws"], a["wsb"], a["stream"])


def test_chunk_fwd_rejects_bad_arguments(L):
    assert fwd(L, q=None) == INVALID
    assert fwd(L, out=None) == INVALID
    assert fwd(L, beta=None) == INVALID
    assert fwd(L, H=0) == INVALID
    assert fwd(L, T=-1) == INVALID
    assert fwd(L, dt=7) == INVALID
    assert fwd(L, scale=float("nan")) == INVALID
    assert fwd(L, N=2) == INVALID                 # N must equal B without cu_seqlens
    assert fwd(L, cu=FAKE, B=2, N=2) == INVALID   # packed needs B == 1
    assert fwd(L, q=FAKE + 4) == INVALID          # misaligned
    assert fwd(L, beta=FAKE + 2) == INVALID
    assert fwd(L, dk=96, dv=96) == UNSUPPORTED
    assert fwd(L, dk=128, dv=64) == UNSUPPORTED
    assert fwd(L, ws=None) == WORKSPACE
    assert fwd(L, wsb=16) == WORKSPACE
    assert fwd(L, ws=FAKE + 16) == WORKSPACE      # workspace must be 256-byte aligned


def test_decode_rejects_bad_arguments(L):
    def dec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=0.1, S=FAKE, out=FAKE, N=4, H=2,
                 dk=128, dv=128, dt=1, stream=None)
        a.update(kw)
        return L.kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["S"],
                                 a["out"], a["N"], a["H"], a["dk"], a["dv"], a["dt"], a["stream"])
    assert dec(S=None) == INVALID
    assert dec(N=-1) == INVALID
    assert dec(H=0) == INVALID
    assert dec(S=FAKE + 8) == INVALID
    assert dec(dk=32, dv=32) == UNSUPPORTED
    assert dec(dt=3) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def fwd_opt(L, decay=0, gate=0, lower=0.0, l2=0, g=FAKE, opts=True, wsb=16, segments=0):
    o = _lib.Options(decay, gate, lower, l2, segments)
    return L.kda_chunk_fwd_opt(FAKE, FAKE, FAKE, g, FAKE, 0.1, None, None, FAKE, FAKE, 1, 64, 1,
                               128, 128, 1, 1, ctypes.byref(o) if opts else None, FAKE, wsb, None,
                               None)


def test_options_validation(L):
    # Accepted options reach the workspace check (an undersized workspace here).
    assert fwd_opt(L) == WORKSPACE
    assert fwd_opt(L, opts=False) == WORKSPACE
    assert fwd_opt(L, decay=1, gate=1, l2=1) == WORKSPACE
    assert fwd_opt(L, decay=2, g=None) == WORKSPACE          # no decay: g unused, may be NULL
    assert fwd_opt(L, decay=1, g=FAKE + 4) == WORKSPACE      # per-head g: 4-byte alignment
    assert fwd_opt(L, gate=2, lower=-5.0) == WORKSPACE
    # Rejected before any CUDA call.
    assert fwd_opt(L, decay=3) == INVALID
    assert fwd_opt(L, gate=7) == INVALID
    assert fwd_opt(L, decay=0, g=None) == INVALID            # per-channel decay needs g
    assert fwd_opt(L, decay=0, g=FAKE + 4) == INVALID        # per-channel g: 16-byte alignment
    assert fwd_opt(L, gate=2, lower=0.0) == INVALID          # bound must be negative
    assert fwd_opt(L, gate=2, lower=-11.0) == INVALID
    assert fwd_opt(L, gate=2, lower=float("nan")) == INVALID
    # Segments of the state pass: any count >= 0 (clamped later), never negative.
    assert fwd_opt(L, segments=1) == WORKSPACE
    assert fwd_opt(L, segments=1000) == WORKSPACE
    assert fwd_opt(L, segments=-1) == INVALID


def test_workspace_reserves_segment_buffers(L):
    # Fixed-length bf16 d=128 batches with few (sequence, head) chains reserve
    # [E | M] and the entering state (3 d^2 fp32) per chain and segment, with
    # chains x segments <= 32; packed batches and the fp32 path reserve none.
    ws = L.kda_chunk_fwd_workspace_size
    per = 3 * 128 * 128 * 4
    few = ws(1, 4096, 4, 128, 128, 1, 1)
    many = ws(1, 4096, 32, 128, 128, 1, 1)
    assert few - many // 8 >= 4 * 8 * per - 4096
    assert ws(1, 4096, 4, 128, 128, 1, 1) > ws(1, 4096, 4, 128, 128, 1, 0) // 2


def test_decode_options_validation(L):
    def dec(decay=0, gate=0, lower=0.0, g=FAKE, N=4):
        o = _lib.Options(decay, gate, lower, 0)
        return L.kda_decode_step_opt(FAKE, FAKE, FAKE, g, FAKE, 0.1, FAKE, FAKE, N, 2, 96, 96, 1,
                                     ctypes.byref(o), None)
    # d = 96 is unsupported: accepted options reach that check.
    assert dec() == UNSUPPORTED
    assert dec(decay=2, g=None) == UNSUPPORTED
    assert dec(decay=1, g=FAKE + 4) == UNSUPPORTED
    assert dec(decay=5) == INVALID
    assert dec(decay=0, g=None) == INVALID
    assert dec(gate=2, lower=1.0) == INVALID


def test_output_gate_rmsnorm_validation(L):
    f = L.kda_output_gate_rmsnorm
    assert f(FAKE, FAKE, None, 1e-6, FAKE, 0, 2, 128, 1, None) == 0        # no tokens: nothing to do
    assert f(FAKE, FAKE, None, 1e-6, FAKE, 10, 2, 96, 1, None) == UNSUPPORTED
    assert f(FAKE, FAKE, None, 0.0, FAKE, 10, 2, 128, 1, None) == INVALID   # eps must be > 0
    assert f(FAKE, FAKE, None, float("inf"), FAKE, 10, 2, 128, 1, None) == INVALID
    assert f(None, FAKE, None, 1e-6, FAKE, 10, 2, 128, 1, None) == INVALID
    assert f(FAKE + 8, FAKE, None, 1e-6, FAKE, 10, 2, 128, 1, None) == INVALID
    assert f(FAKE, FAKE, FAKE + 2, 1e-6, FAKE, 10, 2, 128, 1, None) == INVALID
    assert f(FAKE, FAKE, None, 1e-6, FAKE, -1, 2, 128, 1, None) == INVALID
    assert f(FAKE, FAKE, None, 1e-6, FAKE, 10, 2, 128, 5, None) == INVALID


def test_selftest_validation(L):
    f = L.kda_selftest_wait_timeout
    assert f(None, 100, None) == INVALID
    assert f(FAKE + 2, 100, None) == INVALID
    assert f(FAKE, 0, None) == INVALID
    assert f(FAKE, (1 << 22) + 1, None) == INVALID


def test_host_entry_points_check_arguments_before_any_cuda_call(L):
    """kda_chunk_fwd_host / kda_decode_host validate on the host: window size,
    workspace, host cu_seqlens (read here), sizes (runs without a GPU)."""
    from kimi_delta_attention_17_gb300 import _lib as lib_mod
    vp = ctypes.c_void_p
    opts = lib_mod.Options(0, 0, 0.0, 0, 0)
    hsz = L.kda_chunk_fwd_host_workspace_size
    assert hsz(2, 128, 128, 1, None, 16384) > 0
    assert hsz(2, 128, 128, 1, ctypes.byref(opts), 100) == 0     # window not a multiple of 64
    assert hsz(2, 96, 96, 1, None, 64) == 0                       # unsupported head size
    need = hsz(2, 64, 64, 1, None, 128)

    def host(cu=None, N=1, B=1, T=64, window=128, wsb=None, dk=64):
        return L.kda_chunk_fwd_host(FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, None, cu, FAKE, FAKE, B, T, 2,
                                    dk, dk, N, 1, None, window, FAKE,
                                    need if wsb is None else wsb, None)
    assert host(window=100) == INVALID
    assert host(wsb=need - 1) == WORKSPACE
    assert host(dk=96) == UNSUPPORTED
    bad = (ctypes.c_int32 * 3)(0, 40, 30)                          # decreasing offsets
    assert host(cu=bad, N=2, T=30) == INVALID
    short = (ctypes.c_int32 * 3)(0, 20, 50)                        # ends before T
    assert host(cu=short, N=2, T=64) == INVALID
    assert host(cu=short, N=2, B=2, T=25) == INVALID               # packed needs B == 1
    dsz = L.kda_decode_host_workspace_size
    assert dsz(4, 2, 128, 128, 1, None) > 0 and dsz(0, 2, 128, 128, 1, None) == 0
    dneed = dsz(4, 2, 64, 64, 1, None)

    def dec(steps=3, N=4, wsb=None, g=FAKE):
        return L.kda_decode_host(FAKE, FAKE, FAKE, g, FAKE, 0.1, FAKE, FAKE, steps, N, 2, 64, 64, 1,
                                 None, FAKE, dneed if wsb is None else wsb, None)
    assert dec(steps=-1) == INVALID
    assert dec(steps=0) == 0                                       # nothing to do
    assert dec(wsb=dneed - 1) == WORKSPACE
    assert dec(g=None) == INVALID
