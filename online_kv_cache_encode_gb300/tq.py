"""Python binding of the C ABI in ``include/tq.h`` (ctypes, argument marshalling only).

PyTorch supplies device memory and the current CUDA stream; every step of
encode and decode runs in the library's CUDA kernels.  The binding refuses to
work without ``libtq.so``: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_WORKSPACE = range(5)
FLAG_OVERFLOW, FLAG_BAD_SLOT, FLAG_NONFINITE, FLAG_TIMEOUT, FLAG_INTERNAL = 1, 2, 4, 8, 16
TQ_F32, TQ_BF16, TQ_F16 = 0, 1, 2
NOALLOC_WORKSPACE_BYTES = 4 << 20  # TQ_NOALLOC_WORKSPACE_BYTES

# every exported symbol of include/tq.h: (restype, argtypes)
_P, _I, _I64, _U64, _F, _SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                               ctypes.c_float, ctypes.c_size_t)
SIGNATURES = {
    "tq_codebook_init": (_I, [_I, _I, ctypes.POINTER(_P)]),
    "tq_codebook_get": (_I, [_P, _P, _P, _P]),
    "tq_codebook_free": (None, [_P]),
    "tq_page_bytes": (_I64, [_I, _I, _I, _I, _I]),
    "tq_cache_create": (_I, [_P, _I64, _I, _I, _I, _I, _I, _I, _U64, ctypes.POINTER(_P)]),
    "tq_cache_free": (None, [_P]),
    "tq_method_constants": (_I, [_I, _I, _U64, _P, _P]),
    "tq_cache_signs": (_I, [_P, _P]),
    "tq_cache_gaussian": (_I, [_P, _P]),
    "tq_encode_kv": (_I, [_P, _P, _P, _I, _I64, _P, _P, _P]),
    "tq_decode_workspace_bytes": (_SZ, [_P, _I, _I, _I]),
    "tq_decode_attention": (_I, [_P, _P, _I, _I, _I, _P, _I, _P, _F, _P, _P, _SZ, _P, _P]),
    "tq_decode_attention_noalloc": (_I, [_P, _P, _I, _I, _I, _P, _I, _P, _F, _P, _P, _P]),
    "tq_decode_attention_append": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _P, _I, _P, _F, _P, _P, _SZ, _P, _P]),
    "tq_decode_attention_ring_append": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _P, _I, _P, _I, _F, _P, _P, _SZ, _P,
                                             _P]),
    "tq_cache_create_octopus": (_I, [_P, ctypes.c_int64, _I, _I, _I, _I, _I, ctypes.c_uint64, ctypes.POINTER(_P)]),
    "tq_octopus_page_bytes": (ctypes.c_int64, [_I, _I, _I, _I]),
    "tq_octopus_codebook": (_I, [_I, _I, _I, _P]),
    "tq_prefill_workspace_bytes": (_SZ, [_P, _I, _I, _I]),
    "tq_prefill_attention": (_I, [_P, _P, _I, _I, _I, _P, _I, _I, _F, _P, _P, _SZ, _P, _P]),
    "tq_device_accessible": (_I, [_P, ctypes.POINTER(_I)]),
    "tq_test_stall_waits": (None, [_I64]),
    "tq_selftest_tcgen05": (_I, [_P, _P, _P, _P, _P]),
    "tq_status_string": (ctypes.c_char_p, [_I]),
    "tq_last_error": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class TQError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"tq status {status}: {detail}")
        self.status = status


def lib():
    """Load libtq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _check(st: int):
    if st != TQ_OK:
        raise TQError(st, lib().tq_last_error().decode())


_DTYPE_CODES = {torch.float32: TQ_F32, torch.bfloat16: TQ_BF16, torch.float16: TQ_F16}


def _dtype_code(t: torch.Tensor) -> int:
    return _DTYPE_CODES[t.dtype]


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    # a plain int: the c_void_p argtypes convert it
    return None if t is None else t.data_ptr()


def device_accessible(t: torch.Tensor) -> bool:
    """Whether the decode kernels can read / write tensor t in place: a CUDA
    tensor, or a pinned host tensor mapped into the device's address space
    (the kernel then reaches it over the host link, with no copy launch)."""
    if t.is_cuda:
        return True
    if not t.is_pinned():
        return False
    a = ctypes.c_int(0)
    _check(lib().tq_device_accessible(_ptr(t), ctypes.byref(a)))
    return a.value == 1


def set_test_stall(cycles: int) -> None:
    """Test hook of the device-side timeout path (tq_test_stall_waits): with
    cycles > 0 every later decode launch lets warp 0 of each odd split give up
    a bounded wait; 0 turns it off."""
    lib().tq_test_stall_waits(int(cycles))


def selftest_tcgen05(A: torch.Tensor, B: torch.Tensor, status: torch.Tensor | None = None) -> torch.Tensor:
    """tq_selftest_tcgen05: A [128, 256] and B [256, 16] fp16 (CUDA) -> out [6, 128, 16] fp32."""
    assert A.is_cuda and A.dtype == torch.float16 and A.shape == (128, 256) and A.is_contiguous()
    assert B.is_cuda and B.dtype == torch.float16 and B.shape == (256, 16) and B.is_contiguous()
    out = torch.full((6, 128, 16), float("nan"), dtype=torch.float32, device=A.device)
    _check(lib().tq_selftest_tcgen05(_ptr(A), _ptr(B), _ptr(out), _ptr(status), _stream()))
    return out


def ring_slots(block_row, positions, window: int, block_size: int = 16):
    """Slots of token positions in a sequence's ring of `window` slots (its
    block-table row block_row): position t lives in slot t % window."""
    r = positions % window
    return block_row[r // block_size] * block_size + r % block_size


def page_bytes(d: int, key_bits: int, value_bits: int, qjl_m: int = 0, block_size: int = 16) -> int:
    return int(lib().tq_page_bytes(d, key_bits, value_bits, qjl_m, block_size))


class Codebook:
    """Host Lloyd-Max codebook (centroids, boundaries, passes)."""

    def __init__(self, d: int, bits: int):
        h = ctypes.c_void_p()
        _check(lib().tq_codebook_init(d, bits, ctypes.byref(h)))
        try:
            n = 1 << bits
            self.centroids = np.empty(n, dtype=np.float64)
            self.boundaries = np.empty(n - 1, dtype=np.float64)
            passes = ctypes.c_int()
            _check(lib().tq_codebook_get(h, self.centroids.ctypes.data_as(_P),
                                         self.boundaries.ctypes.data_as(_P), ctypes.byref(passes)))
            self.passes = passes.value
        finally:
            lib().tq_codebook_free(h)


def method_constants(d: int, m: int, seed: int):
    """(signs[d] int8, S[m, d] float64) that a seed defines (host, no GPU)."""
    s = np.empty(d, dtype=np.int8)
    S = np.empty((m, d), dtype=np.float64)
    _check(lib().tq_method_constants(d, m, seed, s.ctypes.data_as(_P), S.ctypes.data_as(_P) if m else None))
    return s, S


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


class Cache:
    """A compressed paged KV cache on the current CUDA device.

    pool: uint8 [num_blocks * num_kv_heads * page_bytes], allocated here unless given.
    """

    def __init__(self, num_blocks: int, num_kv_heads: int, key_bits: int = 4, value_bits: int = 4,
                 qjl_m: int = 0, seed: int = 0, block_size: int = 16, d: int = 128,
                 pool: torch.Tensor | None = None, device="cuda"):
        self.num_blocks, self.hkv, self.kb, self.vb = num_blocks, num_kv_heads, key_bits, value_bits
        self.m, self.seed, self.bs, self.d = qjl_m, seed, block_size, d
        self.page_bytes = page_bytes(d, key_bits, value_bits, qjl_m, block_size)
        if self.page_bytes < 0:
            raise TQError(TQ_ERR_INVALID_ARG, "invalid geometry")
        nbytes = self.page_bytes * num_kv_heads * num_blocks
        if pool is None:
            pool = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        assert pool.dtype == torch.uint8 and pool.numel() >= nbytes and pool.is_contiguous()
        self.pool = pool
        self._h = ctypes.c_void_p()
        _check(lib().tq_cache_create(_ptr(pool), num_blocks, block_size, num_kv_heads, d, key_bits,
                                     value_bits, qjl_m, seed, ctypes.byref(self._h)))
        self._ws = None

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.tq_cache_free(h)
            self._h = None

    # ---- derived constants (host copies) ----
    def signs(self) -> np.ndarray:
        s = np.empty(self.d, dtype=np.int8)
        _check(lib().tq_cache_signs(self._h, s.ctypes.data_as(_P)))
        return s

    def gaussian(self) -> np.ndarray:
        S = np.empty((self.m, self.d), dtype=np.float64)
        _check(lib().tq_cache_gaussian(self._h, S.ctypes.data_as(_P)))
        return S

    # ---- encode ----
    def encode(self, K: torch.Tensor, V: torch.Tensor, slot_mapping: torch.Tensor,
               status: torch.Tensor | None = None):
        """K, V: [T, num_kv_heads, d] (f32/bf16/f16, CUDA); slot_mapping: int64 [T]."""
        assert K.is_cuda and K.shape == V.shape and K.dtype == V.dtype
        assert K.dim() == 3 and K.shape[1] == self.hkv and K.shape[2] == self.d
        assert K.is_contiguous() and V.is_contiguous()
        assert slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous()
        assert slot_mapping.numel() == K.shape[0]
        _check(lib().tq_encode_kv(self._h, _ptr(K), _ptr(V), _dtype_code(K), K.shape[0],
                                  _ptr(slot_mapping), _ptr(status), _stream()))

    # ---- decode ----
    def workspace_bytes(self, batch: int, num_q_heads: int, max_blocks_per_seq: int) -> int:
        return int(lib().tq_decode_workspace_bytes(self._h, batch, num_q_heads, max_blocks_per_seq))

    def new_workspace(self, batch: int, num_q_heads: int, max_blocks_per_seq: int) -> torch.Tensor:
        n = self.workspace_bytes(batch, num_q_heads, max_blocks_per_seq)
        return torch.zeros(max(n, 256), dtype=torch.uint8, device=self.pool.device)

    def decode(self, q: torch.Tensor, block_table: torch.Tensor, lens: torch.Tensor,
               sm_scale: float | None = None, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, status: torch.Tensor | None = None) -> torch.Tensor:
        """q: [B, Hq, d]; block_table: int32 [B, max_blocks]; lens: int32 [B] -> out fp32 [B, Hq, d].
        q and out may be pinned host tensors (see device_accessible)."""
        assert device_accessible(q) and q.dim() == 3 and q.shape[2] == self.d and q.is_contiguous()
        B, hq, _ = q.shape
        assert block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.shape[0] == B
        assert block_table.is_contiguous() and lens.dtype == torch.int32 and lens.numel() == B
        mb = block_table.shape[1]
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.d)
        if out is None:
            out = torch.empty((B, hq, self.d), dtype=torch.float32, device=self.pool.device)
        assert device_accessible(out)
        if workspace is None:
            key = (B, hq, mb)
            if self._ws is None or self._ws[0] != key:
                self._ws = (key, self.new_workspace(B, hq, mb))
            workspace = self._ws[1]
        _check(lib().tq_decode_attention(self._h, _ptr(q), _dtype_code(q), B, hq, _ptr(block_table), mb,
                                         _ptr(lens), float(sm_scale), _ptr(out), _ptr(workspace),
                                         workspace.numel(), _ptr(status), _stream()))
        return out

    def decode_append(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor, block_table: torch.Tensor,
                      lens: torch.Tensor, sm_scale: float | None = None, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                      window: int | None = None) -> torch.Tensor:
        """One decode step: append the new token of every sequence (k_new, v_new:
        [B, num_kv_heads, d], position lens[b] - 1) and attend over lens[b] tokens.
        With `window`, each sequence's blocks form a ring of `window` slots: the
        token goes to slot (lens[b] - 1) % window and the query attends over the
        min(lens[b], window) tokens the ring holds."""
        assert device_accessible(k_new) and device_accessible(v_new)
        assert k_new.shape == v_new.shape and k_new.dtype == v_new.dtype
        assert k_new.dim() == 3 and k_new.shape[1] == self.hkv and k_new.shape[2] == self.d
        assert k_new.is_contiguous() and v_new.is_contiguous()
        assert device_accessible(q) and q.dim() == 3 and q.shape[2] == self.d and q.is_contiguous()
        B, hq, _ = q.shape
        assert k_new.shape[0] == B
        assert block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.shape[0] == B
        assert block_table.is_contiguous() and lens.dtype == torch.int32 and lens.numel() == B
        mb = block_table.shape[1]
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.d)
        if out is None:
            out = torch.empty((B, hq, self.d), dtype=torch.float32, device=self.pool.device)
        assert device_accessible(out)
        if workspace is None:
            key = (B, hq, mb)
            if self._ws is None or self._ws[0] != key:
                self._ws = (key, self.new_workspace(B, hq, mb))
            workspace = self._ws[1]
        if window is None:
            _check(lib().tq_decode_attention_append(self._h, _ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(q),
                                                    _dtype_code(q), B, hq, _ptr(block_table), mb, _ptr(lens),
                                                    float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                                    _ptr(status), _stream()))
        else:
            _check(lib().tq_decode_attention_ring_append(self._h, _ptr(k_new), _ptr(v_new), _dtype_code(k_new),
                                                         _ptr(q), _dtype_code(q), B, hq, _ptr(block_table), mb,
                                                         _ptr(lens), int(window), float(sm_scale), _ptr(out),
                                                         _ptr(workspace), workspace.numel(), _ptr(status),
                                                         _stream()))
        return out

    def prefill(self, q: torch.Tensor, block_row: torch.Tensor, first_position: int, sm_scale: float | None = None,
                out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                status: torch.Tensor | None = None) -> torch.Tensor:
        """Causal attention of the query positions first_position .. first_position + C - 1
        (q: [C, Hq, d]) of one sequence over its cached tokens (the chunk's own
        keys and values already encoded); block_row: int32 [max_blocks]."""
        assert q.is_cuda and q.dim() == 3 and q.shape[2] == self.d and q.is_contiguous()
        assert block_row.dtype == torch.int32 and block_row.dim() == 1 and block_row.is_contiguous()
        C, hq, _ = q.shape
        mb = block_row.shape[0]
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.d)
        if out is None:
            out = torch.empty((C, hq, self.d), dtype=torch.float32, device=q.device)
        if workspace is None:
            n = int(lib().tq_prefill_workspace_bytes(self._h, C, hq, mb))
            workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
        _check(lib().tq_prefill_attention(self._h, _ptr(q), _dtype_code(q), C, hq, _ptr(block_row), mb,
                                          int(first_position), float(sm_scale), _ptr(out), _ptr(workspace),
                                          workspace.numel(), _ptr(status), _stream()))
        return out

    def decode_noalloc(self, q: torch.Tensor, block_table: torch.Tensor, lens: torch.Tensor,
                       sm_scale: float | None = None, out: torch.Tensor = None,
                       status: torch.Tensor | None = None) -> torch.Tensor:
        """decode() through tq_decode_attention_noalloc: the library's fixed
        workspace instead of a caller one (for callers that must not allocate).
        `out` must be given: this call allocates nothing, here or in the library."""
        assert out is not None and out.dtype == torch.float32 and out.is_contiguous()
        assert q.is_cuda and q.dim() == 3 and q.shape[2] == self.d and q.is_contiguous()
        B, hq, _ = q.shape
        assert out.shape == (B, hq, self.d)
        assert block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous()
        assert lens.dtype == torch.int32 and lens.numel() == B
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.d)
        _check(lib().tq_decode_attention_noalloc(self._h, _ptr(q), _dtype_code(q), B, hq, _ptr(block_table),
                                                 block_table.shape[1], _ptr(lens), float(sm_scale), _ptr(out),
                                                 _ptr(status), _stream()))
        return out


class OctopusCache(Cache):
    """A cache whose keys use the OCTOPUS triplet codec (bits 2..4 per
    coordinate on average: (bits + 1)-bit direction codes, (bits - 1)-bit norm
    codes per triplet); values keep min-max codes.  encode / decode as Cache."""

    def __init__(self, num_blocks: int, num_kv_heads: int, bits: int = 4, value_bits: int = 4, seed: int = 0,
                 block_size: int = 16, d: int = 128, pool: torch.Tensor | None = None, device="cuda"):
        self.num_blocks, self.hkv, self.kb, self.vb = num_blocks, num_kv_heads, bits, value_bits
        self.m, self.seed, self.bs, self.d = 0, seed, block_size, d
        self.page_bytes = int(lib().tq_octopus_page_bytes(d, bits, value_bits, block_size))
        if self.page_bytes < 0:
            raise TQError(TQ_ERR_INVALID_ARG, "invalid geometry")
        nbytes = self.page_bytes * num_kv_heads * num_blocks
        if pool is None:
            pool = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        assert pool.dtype == torch.uint8 and pool.numel() >= nbytes and pool.is_contiguous()
        self.pool = pool
        self._h = ctypes.c_void_p()
        _check(lib().tq_cache_create_octopus(_ptr(pool), num_blocks, block_size, num_kv_heads, d, bits, value_bits,
                                             seed, ctypes.byref(self._h)))
        self._ws = None


def octopus_codebook(d: int, bits: int, kind: int) -> np.ndarray:
    """The library's host-computed OCTOPUS levels (kind 0: xi / eta, kind 1: triplet norm)."""
    out = np.empty(1 << bits, dtype=np.float64)
    _check(lib().tq_octopus_codebook(d, bits, kind, out.ctypes.data_as(ctypes.c_void_p)))
    return out
