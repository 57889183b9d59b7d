"""Host-side checks of the CUDA library that need no GPU: the shared library
loads, exports every symbol include/tq.h declares, and its host logic (the
Lloyd-Max codebook, the seeded constants, page sizes, argument checks) agrees
with the oracle and with the documented behaviour."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq():
    from online_kv_cache_encode_gb300 import build
    build.build()
    from online_kv_cache_encode_gb300 import tq as T
    return T


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    return sorted(set(re.findall(r"TQ_API\s+[\w\s\*]+?\b(tq_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(tq):
    names = _declared_symbols()
    assert len(names) >= 14
    L = tq.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(tq.SIGNATURES), "binding and header disagree"
    nm = subprocess.run(["nm", "-D", "--defined-only", tq.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (tq_\w+)", nm))
    assert exported == set(names), exported ^ set(names)


@pytest.mark.parametrize("d,b", [(128, 1), (128, 2), (128, 3), (128, 4), (64, 4), (16, 2), (256, 3)])
def test_host_codebook_matches_oracle(tq, oracle, d, b):
    cb = tq.Codebook(d, b)
    c, t, _ = oracle.lloyd_max(d, b)
    np.testing.assert_allclose(cb.centroids, c, rtol=0, atol=1e-12)
    np.testing.assert_allclose(cb.boundaries, t, rtol=0, atol=1e-12)
    assert cb.passes < 10000
    np.testing.assert_array_equal(cb.boundaries, 0.5 * (cb.centroids[:-1] + cb.centroids[1:]))


def test_host_codebook_matches_scipy(tq):
    from tests.test_oracle_pins import _scipy_lloyd
    for b in (2, 4):
        np.testing.assert_allclose(tq.Codebook(128, b).centroids, _scipy_lloyd(128, b), rtol=0, atol=1e-12)


@pytest.mark.parametrize("b", [5, 6, 7, 8])
def test_wide_key_boundaries_fit_the_encode_grid(tq, b):
    """The tensor-core encode decides keys wider than 4 bits on a grid of
    64 cells per unit of z = |u| / gamma, each cell holding at most one
    positive boundary sqrt(d) t_b: the boundaries (and the first one from 0)
    must lie more than a cell apart, as they do for every d = 128 codebook."""
    cb = tq.Codebook(128, b)
    half = 1 << (b - 1)
    pos = np.sqrt(128.0) * cb.boundaries[half:]
    assert cb.boundaries[half - 1] == 0.0
    assert np.diff(np.concatenate([[0.0], pos])).min() > 1.0 / 64
    assert pos[-1] < 16.0  # inside the grid's range


@pytest.mark.parametrize("seed", [0, 1, 42, 2**63 + 17])
def test_seeded_constants_match_oracle_bit_for_bit(tq, oracle, seed):
    s, S = tq.method_constants(128, 128, seed)
    np.testing.assert_array_equal(s.astype(np.float64), oracle.signs(seed, 128))
    np.testing.assert_array_equal(S, oracle.gaussian(seed, 128, 128))


def test_page_bytes(tq, oracle):
    for kb in range(1, 9):
        for vb in range(1, 9):
            for m in (0, 64, 128):
                assert tq.page_bytes(128, kb, vb, m, 16) == oracle.page_bytes(128, kb, vb, m, 16)
    assert tq.page_bytes(128, 4, 4, 0, 16) == 2144
    assert tq.page_bytes(128, 3, 3, 0, 16) == 1632
    assert tq.page_bytes(128, 2, 2, 128, 16) == 1408
    assert tq.page_bytes(128, 9, 4, 0, 16) == -1
    assert tq.page_bytes(100, 4, 4, 0, 16) == -1


def test_argument_checks_need_no_gpu(tq):
    L = tq.lib()
    h = ctypes.c_void_p()
    assert L.tq_cache_create(None, 4, 16, 1, 128, 4, 4, 0, 0, ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_cache_create(ctypes.c_void_p(0x1008), 4, 16, 1, 128, 4, 4, 0, 0,
                             ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG  # not 16-byte aligned
    fake = ctypes.c_void_p(0x100000)
    assert L.tq_cache_create(fake, 4, 16, 1, 64, 4, 4, 0, 0, ctypes.byref(h)) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_cache_create(fake, 4, 8, 1, 128, 4, 4, 0, 0, ctypes.byref(h)) == tq.TQ_ERR_UNSUPPORTED
    # widths 1 .. 8 are built; the QJL sketch only for 2- to 4-bit keys and values
    assert L.tq_cache_create(fake, 4, 16, 1, 128, 5, 4, 128, 0, ctypes.byref(h)) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_cache_create(fake, 4, 16, 1, 128, 4, 1, 128, 0, ctypes.byref(h)) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_cache_create(fake, 4, 16, 1, 128, 9, 4, 0, 0, ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_cache_create(fake, 4, 16, 1, 128, 4, 4, 64, 0, ctypes.byref(h)) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_cache_create(fake, 0, 16, 1, 128, 4, 4, 0, 0, ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_encode_kv(None, None, None, 0, 1, None, None, None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_decode_attention(None, None, 0, 1, 1, None, 1, None, 0.1, None, None, 0, None,
                                 None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_decode_workspace_bytes(None, 1, 1, 1) == 0
    assert L.tq_codebook_init(7, 4, ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_codebook_init(128, 9, ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_method_constants(0, 0, 0, None, None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_device_accessible(fake, None) == tq.TQ_ERR_INVALID_ARG
    acc = ctypes.c_int(7)
    assert L.tq_device_accessible(None, ctypes.byref(acc)) == tq.TQ_OK and acc.value == 0  # NULL: never
    import torch
    assert not tq.device_accessible(torch.empty(4))  # pageable host memory: no runtime call needed
    assert b"invalid" in L.tq_status_string(tq.TQ_ERR_INVALID_ARG)
    assert L.tq_last_error()  # the last failure left a message


def test_binding_refuses_without_library(tq, monkeypatch):
    monkeypatch.setattr(tq, "_lib", None)
    monkeypatch.setattr(tq, "LIB_PATH", "/nonexistent/libtq.so")
    with pytest.raises(RuntimeError, match="missing"):
        tq.lib()


def test_octopus_codebooks_match_the_oracle(tq, oracle):
    """The library computes its OCTOPUS codebooks on the host by a different
    method (cumulative Simpson tables) than the oracle (Gauss-Legendre cells);
    both must reach the same Lloyd-Max levels."""
    for kind, bits in ((0, 3), (0, 5), (1, 1), (1, 3)):
        lib = tq.octopus_codebook(128, bits, kind)
        ref = oracle.oct_codebook(kind, 128, bits)[0]
        assert abs(lib - ref).max() < 1e-9, (kind, bits)
    assert tq.lib().tq_octopus_page_bytes(128, 4, 4, 16) == 16 * 72 + 16 * 64 + 96
    assert tq.lib().tq_octopus_page_bytes(128, 5, 4, 16) == -1
