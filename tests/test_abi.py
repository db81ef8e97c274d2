"""The C-ABI library builds, loads and exports every entry point include/pi.h
declares; host-only helpers agree with the oracle.  No GPU needed."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
from activation_sparse_decode_sigmoid_gb300 import build as B
from activation_sparse_decode_sigmoid_gb300 import pi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols() -> list[str]:
    src = open(os.path.join(ROOT, "include", "pi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pi_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pi.load_library()


def test_header_declares_the_boundary():
    syms = header_symbols()
    for name in ("pi_create", "pi_load_layer", "pi_predict", "pi_sparse_ffn", "pi_decode_step"):
        assert name in syms
    assert set(syms) == set(pi.EXPORTS), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(B.LIB)
    for name in header_symbols():
        assert hasattr(raw, name), name


def test_perm_from_counts_matches_oracle(lib):
    rng = np.random.default_rng(0)
    for n in (1, 17, 4096, 28672):
        c = rng.integers(0, 50, n).astype(np.int32)
        assert np.array_equal(pi.pi_perm_from_counts(c), O.perm_from_counts(c))


def test_null_and_range_arguments_fail_on_host(lib):
    out = ctypes.c_void_p()
    assert lib.pi_create(None, 0, None, 1, 1) == pi.PI_ERR_ARG
    assert lib.pi_create(ctypes.byref(out), 0, None, 0, 1) == pi.PI_ERR_ARG
    assert lib.pi_create(ctypes.byref(out), 0, None, 1, 65) == pi.PI_ERR_ARG
    assert lib.pi_destroy(None) == pi.PI_ERR_ARG
    assert lib.pi_perm_from_counts(None, 3, None) == pi.PI_ERR_ARG
    assert lib.pi_last_error(None) == b"null context"


def test_no_device_is_an_error_not_a_crash(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    out = ctypes.c_void_p()
    assert lib.pi_create(ctypes.byref(out), 0, None, 1, 1) == pi.PI_ERR_CUDA
    assert out.value is None
