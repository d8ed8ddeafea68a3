"""Kimi Delta Attention gated delta-rule scan for GB300 (sm_103a).

The compute lives in libkda.so (C ABI: include/kda.h); this package is its thin
Python binding plus the seeded synthetic-input generator. Importing the package
does not load the library; the first call does, and raises if it is missing.
"""
from .kda import (DecodeGraph, chunk_fwd, chunk_fwd_host, decode_host,  # noqa: F401
                  decode_step, host_workspace_size, output_gate_rmsnorm, status_string,
                  workspace_size)

__all__ = ["DecodeGraph", "chunk_fwd", "chunk_fwd_host", "decode_host", "decode_step",
           "host_workspace_size", "output_gate_rmsnorm", "status_string", "workspace_size"]
