"""Loads libkda.so (built in-tree by kimi_delta_attention_17_gb300.build) and
declares the C signatures of include/kda.h. There is no fallback: if the
library is missing, every call raises."""
import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkda.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "kda.h")

KDA_OK = 0
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARGUMENT", 2: "KDA_ERR_UNSUPPORTED",
                3: "KDA_ERR_WORKSPACE", 4: "KDA_ERR_CUDA", 5: "KDA_ERR_TIMEOUT"}
DTYPE_F32 = 0
DTYPE_BF16 = 1
DECAY = {"channel": 0, "scalar": 1, "none": 2}           # kda_decay
GATE = {"log": 0, "logsigmoid": 1, "bounded": 2}          # kda_gate


class Options(ctypes.Structure):
    """kda_options of include/kda.h."""
    _fields_ = [("decay", ctypes.c_int), ("gate", ctypes.c_int), ("gate_lower", ctypes.c_float),
                ("l2norm_qk", ctypes.c_int), ("segments", ctypes.c_int), ("fused", ctypes.c_int)]


_vp = ctypes.c_void_p
_SIGNATURES = {
    "kda_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "kda_chunk_fwd_workspace_size": ([ctypes.c_int] * 6 + [ctypes.c_int], ctypes.c_size_t),
    "kda_chunk_fwd": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
                      + [ctypes.c_int] * 7 + [_vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "kda_chunk_fwd_timed": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
                            + [ctypes.c_int] * 7 + [_vp, ctypes.c_size_t, _vp, _vp], ctypes.c_int),
    "kda_chunk_fwd_noalloc": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
                              + [ctypes.c_int] * 7 + [_vp], ctypes.c_int),
    "kda_chunk_fwd_noalloc_status": ([_vp, _vp], ctypes.c_int),
    "kda_chunk_fwd_gated": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp,
                             ctypes.c_float, _vp, _vp] + [ctypes.c_int] * 7
                            + [_vp, _vp, ctypes.c_size_t, _vp, _vp], ctypes.c_int),
    "kda_chunk_fwd_host_workspace_size": ([ctypes.c_int] * 4 + [_vp, ctypes.c_int], ctypes.c_size_t),
    "kda_chunk_fwd_host": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
                           + [ctypes.c_int] * 7 + [_vp, ctypes.c_int, _vp, ctypes.c_size_t, _vp],
                           ctypes.c_int),
    "kda_decode_host_workspace_size": ([ctypes.c_int] * 5 + [_vp], ctypes.c_size_t),
    "kda_decode_host": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]
                        + [ctypes.c_int] * 6 + [_vp, _vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "kda_decode_step": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]
                        + [ctypes.c_int] * 5 + [_vp], ctypes.c_int),
    "kda_chunk_fwd_opt": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
                          + [ctypes.c_int] * 7 + [_vp, _vp, ctypes.c_size_t, _vp, _vp], ctypes.c_int),
    "kda_decode_step_opt": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]
                            + [ctypes.c_int] * 5 + [_vp, _vp], ctypes.c_int),
    "kda_selftest_wait_timeout": ([_vp, ctypes.c_uint, _vp], ctypes.c_int),
    "kda_output_gate_rmsnorm": ([_vp, _vp, _vp, ctypes.c_float, _vp, ctypes.c_longlong,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp], ctypes.c_int),
}

_lib = None


class KdaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s returned %s" % (fn, STATUS_NAMES.get(status, status)))


def declared_symbols():
    """Function names declared in include/kda.h (what the library must export)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libkda.so is not built (expected at %s); run "
                "`python -m kimi_delta_attention_17_gb300.build` first" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def check(fn, status):
    if status != KDA_OK:
        raise KdaError(fn, status)
