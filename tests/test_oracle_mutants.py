"""Plants one plausible mistake at a time into a temporary copy of the oracle's
C scan, rebuilds it, and checks that the pins in test_oracle_pins.py catch
every one of them (at least one pin fails per mutant). The oracle's own source
is never modified. CPU only.
"""
import ctypes
import inspect
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_scan.c")

# name -> list of (original text, replacement) applied to kda_scan.c
MUTANTS = {
    "additive write (linear attention)": [
        ("e[j] = bt * (vt[j] - vhat[j]);", "e[j] = bt * vt[j];")],
    "no decay": [
        ("const double a = exp(gt[c]);", "const double a = 1.0;")],
    "decay with the wrong sign": [
        ("const double a = exp(gt[c]);", "const double a = exp(-gt[c]);")],
    "decay applied after the write": [
        ("for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;", ""),
        ("for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += kt[c] * e[j];",
         "for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] = exp(gt[c]) * "
         "(S[(size_t)c * dv + j] + kt[c] * e[j]);")],
    "decay scales value columns": [
        ("for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;",
         "for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= exp(gt[j % dk]);")],
    "beta applied twice": [
        ("e[j] = bt * (vt[j] - vhat[j]);", "e[j] = bt * bt * (vt[j] - vhat[j]);")],
    "query scale dropped": [
        ("acc += S[(size_t)c * dv + j] * (J->scale * qt[c]);",
         "acc += S[(size_t)c * dv + j] * qt[c];")],
    "key scaled like the query": [
        ("vhat[j] += S[(size_t)c * dv + j] * kt[c];",
         "vhat[j] += S[(size_t)c * dv + j] * kt[c] * J->scale;")],
    "read before the write": [
        ("/* S = S~ + k_t e^T. */",
         "for (int j = 0; j < dv; ++j) { double acc = 0.0; for (int c = 0; c < dk; ++c) "
         "acc += S[(size_t)c * dv + j] * (J->scale * qt[c]); "
         "J->out[((size_t)t * H + h) * dv + j] = acc; }"),
        ("ot[j] = acc;", "(void)acc; (void)ot;")],
    "initial state ignored": [
        ("if (J->init_state)", "if (0)")],
}


def _build_mutant(edits, workdir):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, "mutation anchor vanished: %r" % old
        src = src.replace(old, new)
    path = os.path.join(workdir, "mutant.c")
    open(path, "w").write(src)
    lib = os.path.join(workdir, "libmutant.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-D_GNU_SOURCE", path, "-o",
                    lib, "-lm", "-lpthread"], check=True)
    return lib


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        if "C" in inspect.signature(fn).parameters:
            out.append((name, lambda fn=fn: fn(64)))
        elif not inspect.signature(fn).parameters:
            out.append((name, fn))
    return out


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_mutant(mutant, monkeypatch):
    oracle._load()  # make sure the genuine library's argtypes are known
    with tempfile.TemporaryDirectory() as d:
        lib = ctypes.CDLL(_build_mutant(MUTANTS[mutant], d))
        lib.kda_oracle_scan.argtypes = oracle._lib.kda_oracle_scan.argtypes
        lib.kda_oracle_scan.restype = ctypes.c_int
        lib.kda_oracle_hw_threads.restype = ctypes.c_int
        monkeypatch.setattr(oracle, "_lib", lib)
        caught = []
        for name, fn in _pin_functions():
            try:
                fn()
            except Exception:  # a failed assertion or a pin that cannot even run
                caught.append(name)
        assert caught, "no pin caught the mutant %r" % mutant
