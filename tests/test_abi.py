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


def test_hot_prefix_crossover_hand_computed(lib):
    """The prefix runs while (1 - c/T)^B < P/F (a neuron the union would
    miss that rarely costs less computed than predicted); the cases below use
    powers that are exact in binary floating point."""
    f = pi.pi_hot_prefix_crossover
    c = np.array([4, 3, 2, 2, 1, 0], np.int32)
    # P/F = 1/4: B = 2 -> (0, 1/16, 1/4 ...): the third is not below 1/4
    assert f(c, 4, 2, 1.0, 4.0) == 2
    assert f(c, 4, 1, 1.0, 4.0) == 1          # (0, 3/4 ...)
    assert f(c, 4, 3, 1.0, 4.0) == 4          # (0, 1/64, 1/8, 1/8, 27/64 ...)
    assert f(c, 4, 3, 1.0, 2.0) == 5          # 27/64 < 1/2; a neuron never selected stays predicted
    # a longer batch never shortens the prefix
    rng = np.random.default_rng(3)
    counts = np.sort(rng.integers(0, 257, 5000))[::-1].astype(np.int32)
    hs = [f(counts, 256, b, 2050.0, 28674.0) for b in (1, 2, 4, 8, 16, 64)]
    assert hs == sorted(hs) and hs[0] < hs[-1]
    # the prefix stops at the first neuron that fails, whatever follows
    assert f(np.array([4, 0, 4], np.int32), 4, 1, 1.0, 4.0) == 1
    # every neuron always selected -> all hot; predicting dearer than computing -> all hot
    assert f(np.full(7, 9, np.int32), 9, 1, 1.0, 100.0) == 7
    assert f(np.zeros(7, np.int32), 9, 1, 3.0, 2.0) == 7
    assert f(np.zeros(7, np.int32), 9, 1, 1.0, 2.0) == 0


def test_hot_prefix_arguments_fail_on_host(lib):
    hot = np.zeros(1, np.int32)
    ok = np.array([1, 2], np.int32)
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    assert lib.pi_hot_prefix_crossover(P(ok), 2, 2, 1, 1.0, 4.0, P(hot)) == pi.PI_OK
    for args in ((None, 2, 2, 1, 1.0, 4.0, P(hot)), (P(ok), 0, 2, 1, 1.0, 4.0, P(hot)),
                 (P(ok), 2, 0, 1, 1.0, 4.0, P(hot)), (P(ok), 2, 2, 0, 1.0, 4.0, P(hot)),
                 (P(ok), 2, 2, 1, 0.0, 4.0, P(hot)), (P(ok), 2, 2, 1, 1.0, -1.0, P(hot)),
                 (P(ok), 2, 1, 1, 1.0, 4.0, P(hot)),  # a count above T
                 (P(np.array([-1, 0], np.int32)), 2, 2, 1, 1.0, 4.0, P(hot)),
                 (P(ok), 2, 2, 1, 1.0, 4.0, None)):
        assert lib.pi_hot_prefix_crossover(*args) == pi.PI_ERR_ARG
    assert lib.pi_set_hot_prefix(None, 0, 0) == pi.PI_ERR_ARG
    assert lib.pi_choose_hot_prefix(None, 0, None, 1, 1, None) == pi.PI_ERR_ARG


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
