"""Oracle for online KV-cache compression -- TEST INFRASTRUCTURE ONLY.

A plain float64 CPU restatement (``tq_oracle.c``) of what the CUDA library
computes: norm/direction split, sign-flipped Walsh-Hadamard rotation, Lloyd-Max
key codes, min-max value codes, optional QJL sign sketch, bit-packed paged
cache, and softmax attention over the reconstructed cache.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this package.  It shares no code with the
library under ``online_kv_cache_encode_gb300/``.

This module is argument marshalling over ctypes plus the build step
(``build()`` compiles the C file with gcc; OpenMP if the compiler has it).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB = os.path.join(_HERE, "libtq_oracle.so")
_lock = threading.Lock()
_lib = None

FLAG_OVERFLOW = 1
FLAG_BAD_SLOT = 2
FLAG_NONFINITE = 4


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libtq_oracle.so`` (gcc, -O2)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:5] + ["-fopenmp"] + base[5:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, u64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        sig = {
            "orc_set_threads": (i32, [i32]),
            "orc_stream_at": (u64, [u64, u64, u64]),
            "orc_stream": (None, [u64, u64, u64, i64, P]),
            "orc_signs": (None, [u64, i32, P]),
            "orc_gaussian": (None, [u64, i32, i32, P]),
            "orc_hadamard": (None, [i32, P]),
            "orc_rotate": (None, [i32, P, P, P]),
            "orc_rotate_inverse": (None, [i32, P, P, P]),
            "orc_density": (f64, [i32, f64]),
            "orc_cell_mass": (f64, [i32, f64, f64]),
            "orc_cell_moment": (f64, [i32, f64, f64]),
            "orc_lloyd_max": (i32, [i32, i32, f64, i32, P, P]),
            "orc_fp16_round": (f64, [f64]),
            "orc_fp16_bits": (ctypes.c_uint16, [f64]),
            "orc_fp16_value": (f64, [ctypes.c_uint16]),
            "orc_page_bytes": (i64, [i32, i32, i32, i32, i32]),
            "orc_encode_key_vector": (None, [i32, i32, P, P, P, i32, P, P, P, P, P, P]),
            "orc_encode_value_vector": (None, [i32, i32, P, P, P, P, P]),
            "orc_encode": (i32, [i32, i32, i32, i32, i32, i32, i64, P, P, P, P, P, P, i64, P, P]),
            "orc_unpack_slot": (None, [i32, i32, i32, i32, i32, P, i32, P, P, P, P, P, P, P]),
            "orc_decode": (i32, [i32, i32, i32, i32, i32, i32, i64, P, P, P, P, P, i32, i32, P, i32, P, f64, P]),
            "orc_oct_map": (None, [P, P, P]),
            "orc_oct_inverse": (None, [f64, f64, P]),
            "orc_oct_density": (f64, [f64, f64]),
            "orc_oct_marginal": (f64, [f64]),
            "orc_rho_density": (f64, [i32, f64]),
            "orc_oct_cell_mass": (f64, [i32, i32, f64, f64]),
            "orc_lloyd_density": (i32, [i32, i32, i32, f64, i32, P, P]),
            "orc_oct_encode_triplet": (f64, [P, P, P, i32, P, P, i32, P, P, P]),
            "orc_oct_page_bytes": (i64, [i32, i32, i32, i32]),
            "orc_oct_encode_key_vector": (None, [i32, P, P, i32, P, P, i32, P, P, P, P, P, P]),
            "orc_oct_encode": (i32, [i32, i32, i32, i32, i32, i64, P, P, P, P, P, P, P, i64, P, P]),
            "orc_oct_unpack_slot": (None, [i32, i32, i32, i32, P, i32, P, P, P, P, P, P, P]),
            "orc_oct_decode": (i32, [i32, i32, i32, i32, i32, i64, P, P, P, P, P, i32, i32, P, i32, P, f64, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def set_threads(n: int) -> int:
    """Set the OpenMP thread count (0 keeps it); returns the count in effect."""
    return _load().orc_set_threads(int(n))


# --- generator --------------------------------------------------------------

def stream(seed: int, tag: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().orc_stream(seed, tag, start, n, _p(out))
    return out


def signs(seed: int, d: int) -> np.ndarray:
    out = np.empty(d, dtype=np.float64)
    _load().orc_signs(seed, d, _p(out))
    return out


def gaussian(seed: int, m: int, d: int) -> np.ndarray:
    out = np.empty((m, d), dtype=np.float64)
    _load().orc_gaussian(seed, m, d, _p(out))
    return out


# --- rotation ---------------------------------------------------------------

def hadamard(d: int) -> np.ndarray:
    out = np.empty((d, d), dtype=np.float64)
    _load().orc_hadamard(d, _p(out))
    return out


def rotate(s: np.ndarray, x: np.ndarray) -> np.ndarray:
    s, x = _f64(s), _f64(x)
    y = np.empty_like(x)
    _load().orc_rotate(x.shape[-1], _p(s), _p(x), _p(y))
    return y


def rotate_inverse(s: np.ndarray, y: np.ndarray) -> np.ndarray:
    s, y = _f64(s), _f64(y)
    x = np.empty_like(y)
    _load().orc_rotate_inverse(y.shape[-1], _p(s), _p(y), _p(x))
    return x


# --- codebook ---------------------------------------------------------------

def density(d: int, x: float) -> float:
    return _load().orc_density(d, x)


def cell_mass(d: int, a: float, b: float) -> float:
    return _load().orc_cell_mass(d, a, b)


def cell_moment(d: int, a: float, b: float) -> float:
    return _load().orc_cell_moment(d, a, b)


_cb_cache: dict = {}


def lloyd_max(d: int, bits: int, tol: float = 1e-14, max_iter: int = 10000):
    """(centroids[2^bits], boundaries[2^bits - 1], passes)."""
    key = (d, bits, tol, max_iter)
    if key not in _cb_cache:
        c = np.empty(1 << bits, dtype=np.float64)
        t = np.empty((1 << bits) - 1, dtype=np.float64)
        it = _load().orc_lloyd_max(d, bits, tol, max_iter, _p(c), _p(t))
        _cb_cache[key] = (c, t, it)
    c, t, it = _cb_cache[key]
    return c.copy(), t.copy(), it


# --- fp16 -------------------------------------------------------------------

def fp16_round(x: float) -> float:
    return _load().orc_fp16_round(float(x))


def fp16_bits(x: float) -> int:
    return int(_load().orc_fp16_bits(float(x)))


def fp16_value(h: int) -> float:
    return _load().orc_fp16_value(int(h) & 0xFFFF)


# --- layout / encode / decode ---------------------------------------------------

def page_bytes(d: int, kb: int, vb: int, m: int, bs: int) -> int:
    return int(_load().orc_page_bytes(d, kb, vb, m, bs))


class Cache:
    """Geometry + method constants of one compressed cache (oracle side)."""

    def __init__(self, d: int, key_bits: int, value_bits: int, qjl_m: int, block_size: int,
                 num_kv_heads: int, num_blocks: int, seed: int):
        self.d, self.kb, self.vb, self.m = d, key_bits, value_bits, qjl_m
        self.bs, self.hkv, self.num_blocks, self.seed = block_size, num_kv_heads, num_blocks, seed
        self.C, self.T, _ = lloyd_max(d, key_bits)
        self.s = signs(seed, d)
        self.S = gaussian(seed, qjl_m, d) if qjl_m > 0 else np.zeros((1, d))
        self.page_bytes = page_bytes(d, key_bits, value_bits, qjl_m, block_size)
        self.pool_bytes = self.page_bytes * num_kv_heads * num_blocks

    def new_pool(self) -> np.ndarray:
        return np.zeros(self.pool_bytes, dtype=np.uint8)

    def encode_key_vector(self, k: np.ndarray):
        k = _f64(k)
        idx = np.empty(self.d, dtype=np.int32)
        sig = np.empty(max(self.m, 1), dtype=np.int32)
        g, rho = ctypes.c_double(), ctypes.c_double()
        _load().orc_encode_key_vector(self.d, self.kb, _p(self.C), _p(self.T), _p(self.s), self.m,
                                      _p(_f64(self.S)), _p(k), ctypes.byref(g), _p(idx),
                                      ctypes.byref(rho), _p(sig))
        return g.value, idx, rho.value, sig[: self.m]

    def encode_value_vector(self, v: np.ndarray):
        v = _f64(v)
        q = np.empty(self.d, dtype=np.int32)
        sc, zr = ctypes.c_double(), ctypes.c_double()
        _load().orc_encode_value_vector(self.d, self.vb, _p(self.s), _p(v), ctypes.byref(sc),
                                        ctypes.byref(zr), _p(q))
        return sc.value, zr.value, q

    def encode(self, K: np.ndarray, V: np.ndarray, slot_mapping: np.ndarray, pool: np.ndarray) -> int:
        """Encode K, V [T, hkv, d] (any float dtype, widened exactly) into pool in place."""
        K, V = _f64(K), _f64(V)
        T = K.shape[0]
        assert K.shape == (T, self.hkv, self.d) and V.shape == K.shape
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert pool.dtype == np.uint8 and pool.flags.c_contiguous and pool.size == self.pool_bytes
        return _load().orc_encode(self.d, self.kb, self.vb, self.m, self.bs, self.hkv,
                                  self.num_blocks, _p(self.C), _p(self.T), _p(self.s),
                                  _p(_f64(self.S)), _p(K), _p(V), T, _p(sm), _p(pool))

    def unpack_slot(self, pool: np.ndarray, block: int, head: int, off: int):
        page = pool[(block * self.hkv + head) * self.page_bytes:][: self.page_bytes]
        page = np.ascontiguousarray(page)
        kidx = np.empty(self.d, dtype=np.int32)
        vq = np.empty(self.d, dtype=np.int32)
        sig = np.empty(max(self.m, 1), dtype=np.int32)
        g, sc, zr, rho = (ctypes.c_double() for _ in range(4))
        _load().orc_unpack_slot(self.d, self.kb, self.vb, self.m, self.bs, _p(page), off,
                                _p(kidx), _p(vq), ctypes.byref(g), ctypes.byref(sc),
                                ctypes.byref(zr), ctypes.byref(rho), _p(sig))
        return dict(kidx=kidx, vq=vq, gamma=g.value, scale=sc.value, zero=zr.value,
                    rho=rho.value, sig=sig[: self.m])

    def decode(self, pool: np.ndarray, q: np.ndarray, block_table: np.ndarray, lens: np.ndarray,
               sm_scale: float):
        """q [B, Hq, d] -> (out [B, Hq, d] float64, status bits)."""
        q = _f64(q)
        B, hq, d = q.shape
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        ln = np.ascontiguousarray(lens, dtype=np.int32)
        assert bt.shape[0] == B and ln.shape == (B,)
        out = np.empty_like(q)
        st = _load().orc_decode(self.d, self.kb, self.vb, self.m, self.bs, self.hkv,
                                self.num_blocks, _p(self.C), _p(self.s), _p(_f64(self.S)),
                                _p(pool), _p(q), B, hq, _p(bt), bt.shape[1], _p(ln),
                                float(sm_scale), _p(out))
        return out, st


# --- OCTOPUS triplet codec ------------------------------------------------------

def oct_map(n) -> tuple:
    n = _f64(n)
    xi, eta = ctypes.c_double(), ctypes.c_double()
    _load().orc_oct_map(_p(n), ctypes.byref(xi), ctypes.byref(eta))
    return xi.value, eta.value


def oct_inverse(xi: float, eta: float) -> np.ndarray:
    n = np.empty(3)
    _load().orc_oct_inverse(float(xi), float(eta), _p(n))
    return n


def oct_density(xi: float, eta: float) -> float:
    return _load().orc_oct_density(float(xi), float(eta))


def oct_marginal(xi: float) -> float:
    return _load().orc_oct_marginal(float(xi))


def rho_density(d: int, rho: float) -> float:
    return _load().orc_rho_density(d, float(rho))


def oct_cell_mass(kind: int, d: int, a: float, b: float) -> float:
    return _load().orc_oct_cell_mass(kind, d, float(a), float(b))


_oct_cb = {}


def oct_codebook(kind: int, d: int, bits: int, tol: float = 1e-13, max_iter: int = 20000):
    """Lloyd-Max codebook of the xi marginal (kind 0) or the triplet norm (kind 1):
    (centroids, boundaries, passes); cached per (kind, d, bits)."""
    key = (kind, d if kind == 1 else 0, bits)
    if key not in _oct_cb:
        n = 1 << bits
        c, t = np.empty(n), np.empty(max(n - 1, 1))
        it = _load().orc_lloyd_density(kind, d, bits, tol, max_iter, _p(c), _p(t))
        _oct_cb[key] = (c, t[: n - 1], it)
    return _oct_cb[key]


def oct_page_bytes(d: int, b: int, vb: int, bs: int) -> int:
    return int(_load().orc_oct_page_bytes(d, b, vb, bs))


class OctCache:
    """An OCTOPUS cache (triplet keys, min-max values), oracle side."""

    def __init__(self, d: int, bits: int, value_bits: int, block_size: int, num_kv_heads: int,
                 num_blocks: int, seed: int):
        assert bits >= 2
        self.d, self.b, self.vb, self.bs, self.hkv = d, bits, value_bits, block_size, num_kv_heads
        self.num_blocks, self.seed = num_blocks, seed
        self.ntri = (d + 2) // 3
        self.Cxi, self.Txi, _ = oct_codebook(0, d, bits + 1)
        self.Crho, self.Trho, _ = oct_codebook(1, d, bits - 1)
        self.s = signs(seed, d)
        self.page_bytes = oct_page_bytes(d, bits, value_bits, block_size)
        self.pool_bytes = self.page_bytes * num_kv_heads * num_blocks

    def new_pool(self) -> np.ndarray:
        return np.zeros(self.pool_bytes, dtype=np.uint8)

    def encode_triplet(self, t):
        t = _f64(t)
        a, b, r = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        sc = _load().orc_oct_encode_triplet(_p(t), _p(self.Cxi), _p(self.Txi), len(self.Cxi), _p(self.Crho),
                                            _p(self.Trho), len(self.Crho), ctypes.byref(a), ctypes.byref(b),
                                            ctypes.byref(r))
        return a.value, b.value, r.value, sc

    def encode_key_vector(self, k):
        k = _f64(k)
        ixi, ieta, irho = (np.empty(self.ntri, dtype=np.int32) for _ in range(3))
        g = ctypes.c_double()
        _load().orc_oct_encode_key_vector(self.d, _p(self.Cxi), _p(self.Txi), len(self.Cxi), _p(self.Crho),
                                          _p(self.Trho), len(self.Crho), _p(self.s), _p(k), ctypes.byref(g),
                                          _p(ixi), _p(ieta), _p(irho))
        return g.value, ixi, ieta, irho

    def direction(self, ixi, ieta, irho) -> np.ndarray:
        """The rotated unit key the codes stand for (rebuilt from the triplets)."""
        u = np.zeros(3 * self.ntri)
        for i in range(self.ntri):
            u[3 * i: 3 * i + 3] = self.Crho[irho[i]] * oct_inverse(self.Cxi[ixi[i]], self.Cxi[ieta[i]])
        return u[: self.d]

    def encode(self, K, V, slot_mapping, pool: np.ndarray) -> int:
        K, V = _f64(K), _f64(V)
        T = K.shape[0]
        assert K.shape == (T, self.hkv, self.d) and V.shape == K.shape
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert pool.dtype == np.uint8 and pool.flags.c_contiguous and pool.size == self.pool_bytes
        return _load().orc_oct_encode(self.d, self.b, self.vb, self.bs, self.hkv, self.num_blocks,
                                      _p(self.Cxi), _p(self.Txi), _p(self.Crho), _p(self.Trho), _p(self.s),
                                      _p(K), _p(V), T, _p(sm), _p(pool))

    def unpack_slot(self, pool: np.ndarray, block: int, head: int, off: int):
        page = np.ascontiguousarray(pool[(block * self.hkv + head) * self.page_bytes:][: self.page_bytes])
        ixi, ieta, irho = (np.empty(self.ntri, dtype=np.int32) for _ in range(3))
        vq = np.empty(self.d, dtype=np.int32)
        g, sc, zr = (ctypes.c_double() for _ in range(3))
        _load().orc_oct_unpack_slot(self.d, self.b, self.vb, self.bs, _p(page), off, _p(ixi), _p(ieta), _p(irho),
                                    _p(vq), ctypes.byref(g), ctypes.byref(sc), ctypes.byref(zr))
        return dict(ixi=ixi, ieta=ieta, irho=irho, vq=vq, gamma=g.value, scale=sc.value, zero=zr.value)

    def decode(self, pool: np.ndarray, q, block_table, lens, sm_scale: float):
        q = _f64(q)
        B, hq, d = q.shape
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        ln = np.ascontiguousarray(lens, dtype=np.int32)
        out = np.empty_like(q)
        st = _load().orc_oct_decode(self.d, self.b, self.vb, self.bs, self.hkv, self.num_blocks, _p(self.Cxi),
                                    _p(self.Crho), _p(self.s), _p(pool), _p(q), B, hq, _p(bt), bt.shape[1],
                                    _p(ln), float(sm_scale), _p(out))
        return out, st
