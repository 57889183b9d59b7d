"""Seeded synthetic workloads: shapes, data and block tables.

Inputs only -- this module holds none of the method's arithmetic.  Both the
CUDA path and the oracle are fed from here.

Data recipe (numpy PCG64, data seed 1234, independent of the method seed):
  - keys/values are i.i.d. N(0, 1) float32, generated in chunks of 256 tokens
    from a generator keyed by (workload, tensor, sequence, chunk), so any token
    range can be regenerated on its own;
  - "outlier channels": 4 distinct channels per (layer, KV head) scaled x20,
    drawn independently for K and V (the tiny workload instead fixes key
    channels {7, 33, 90, 121} and gives values none);
  - "per-token lognormal(0, 0.25)": one factor exp(N(0, 0.25^2)) per token
    position, shared by all heads of that token, drawn separately for K and V;
  - bf16 and f16 workloads round the float32 values to that type (nearest,
    ties to even);
  - queries are N(0, 1) in the workload dtype;
  - block tables hand each sequence blocks from a seeded random permutation of
    the pool (the tiny workload uses blocks in order).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

DATA_SEED = 1234
CHUNK = 256


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int
    hq: int
    hkv: int
    d: int
    key_bits: int
    value_bits: int
    qjl_m: int
    block_size: int
    lens: tuple          # tokens per sequence before the decode steps
    dtype: str           # "f32", "bf16" or "f16"
    seed: int            # method seed (rotation signs, QJL matrix)
    prefill_chunk: int   # tokens per encode call during prefill
    decode_steps: int    # decode steps after prefill, each appending `append` tokens per sequence
    append: int
    layers_as_batch: bool = False
    fixed_key_channels: tuple | None = None
    value_outliers: bool = True
    lognormal: bool = True
    permute_blocks: bool = True
    description: str = ""

    @property
    def batch(self) -> int:
        return len(self.lens)

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    def max_len(self) -> int:
        return max(self.lens) + self.decode_steps * self.append

    def max_blocks(self) -> int:
        return -(-self.max_len() // self.block_size)

    def num_blocks(self) -> int:
        return self.batch * self.max_blocks()

    def bytes_per_token_head(self) -> int:
        """Compressed bytes one (token, KV head) occupies."""
        d = self.d
        n = d * self.key_bits // 8 + d * self.value_bits // 8 + 6
        if self.qjl_m:
            n += 2 + self.qjl_m // 8
        return n


def _lens_qjl() -> tuple:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([DATA_SEED, 5, 99])))
    return tuple(int(x) for x in rng.integers(1024, 16384 + 1, size=64))


WORKLOADS = {
    "tiny": Workload(
        "tiny", 1, hq=1, hkv=1, d=128, key_bits=4, value_bits=4, qjl_m=0, block_size=16,
        lens=(1024,), dtype="f32", seed=0, prefill_chunk=1024, decode_steps=0, append=0,
        fixed_key_channels=(7, 33, 90, 121), value_outliers=False, lognormal=False,
        permute_blocks=False,
        description="1 KV head, 1 query head, d=128, 1024 tokens, fp32, 4-bit keys/values"),
    "swa8x4096": Workload(
        "swa8x4096", 2, hq=20, hkv=20, d=128, key_bits=4, value_bits=4, qjl_m=0, block_size=16,
        lens=(4096,) * 8, dtype="bf16", seed=0, prefill_chunk=4096, decode_steps=0, append=0,
        layers_as_batch=True,
        description="8 layers (as 8 independent sequences) x 20 heads (MHA), window 4096, bf16, 4/4"),
    "gqa32k": Workload(
        "gqa32k", 3, hq=64, hkv=8, d=128, key_bits=4, value_bits=4, qjl_m=0, block_size=16,
        lens=(32768,), dtype="bf16", seed=0, prefill_chunk=4096, decode_steps=0, append=0,
        description="Llama-3.1-70B-shaped layer: 64 q / 8 KV heads, 32K context, batch 1, bf16, 4/4"),
    "long128k3": Workload(
        "long128k3", 4, hq=64, hkv=8, d=128, key_bits=3, value_bits=3, qjl_m=0, block_size=16,
        lens=(131072,) * 4, dtype="bf16", seed=0, prefill_chunk=4096, decode_steps=64, append=1,
        description="64 q / 8 KV heads, 128K tokens x batch 4, bf16, 3/3, 4K-chunk prefill + 64 steps"),
    "qjl64": Workload(
        "qjl64", 5, hq=32, hkv=8, d=128, key_bits=2, value_bits=2, qjl_m=128, block_size=16,
        lens=_lens_qjl(), dtype="bf16", seed=0, prefill_chunk=4096, decode_steps=128, append=1,
        description="64 sequences, lengths U[1K,16K], 32 q / 8 KV heads, 2-bit keys + QJL m=128, 2-bit values"),
}


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _gen(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([DATA_SEED, *key])))


def outlier_channels(w: Workload, tensor: int, layer: int) -> np.ndarray:
    """[hkv, 4] channel indices scaled x20 for tensor 0 (K) / 1 (V) of a layer (empty if none)."""
    if tensor == 0 and w.fixed_key_channels is not None:
        return np.tile(np.array(w.fixed_key_channels), (w.hkv, 1))
    if tensor == 1 and not w.value_outliers:
        return np.zeros((w.hkv, 0), dtype=np.int64)
    rng = _gen(w.wid, 10 + tensor, layer)
    return np.stack([rng.choice(w.d, size=4, replace=False) for _ in range(w.hkv)])


def kv_tokens(w: Workload, tensor: int, seq: int, t0: int, t1: int) -> np.ndarray:
    """K (tensor 0) or V (tensor 1) for tokens [t0, t1) of a sequence: float32 [t1-t0, hkv, d]."""
    layer = seq if w.layers_as_batch else 0
    ch = outlier_channels(w, tensor, layer)
    out = np.empty((t1 - t0, w.hkv, w.d), dtype=np.float32)
    c0, c1 = t0 // CHUNK, (t1 - 1) // CHUNK if t1 > t0 else t0 // CHUNK - 1
    for c in range(c0, c1 + 1):
        rng = _gen(w.wid, tensor, seq, c)
        x = rng.standard_normal((CHUNK, w.hkv, w.d), dtype=np.float32)
        if ch.shape[1]:
            for h in range(w.hkv):
                x[:, h, ch[h]] *= 20.0
        if w.lognormal:
            x *= np.exp(rng.normal(0.0, 0.25, size=(CHUNK, 1, 1))).astype(np.float32)
        lo, hi = max(t0, c * CHUNK), min(t1, (c + 1) * CHUNK)
        out[lo - t0:hi - t0] = x[lo - c * CHUNK:hi - c * CHUNK]
    return to_dtype(w, out)


def to_dtype(w: Workload, x: np.ndarray) -> np.ndarray:
    """The float32 values a workload of dtype w.dtype carries (bf16 or fp16
    rounded to nearest even, f32 unchanged)."""
    if w.dtype == "bf16":
        return bf16_round(x)
    if w.dtype == "f16":
        return x.astype(np.float16).astype(np.float32)
    return x


def kv_step(w: Workload, tensor: int, t0: int, t1: int) -> np.ndarray:
    """Tokens [t0, t1) of every sequence at once: float32 [batch, t1-t0, hkv, d]."""
    return np.stack([kv_tokens(w, tensor, b, t0, t1) for b in range(w.batch)])


def queries(w: Workload, step: int) -> np.ndarray:
    """Decode query of step `step` for every sequence: float32 [batch, hq, d]."""
    rng = _gen(w.wid, 2, step)
    q = rng.standard_normal((w.batch, w.hq, w.d), dtype=np.float32)
    return to_dtype(w, q)


def block_table(w: Workload) -> np.ndarray:
    """int32 [batch, max_blocks]: disjoint physical blocks per sequence."""
    mb, nb = w.max_blocks(), w.num_blocks()
    if w.permute_blocks:
        perm = _gen(w.wid, 3).permutation(nb)
    else:
        perm = np.arange(nb)
    return perm.reshape(w.batch, mb).astype(np.int32)


def slots(w: Workload, bt: np.ndarray, seq: int, t0: int, t1: int) -> np.ndarray:
    """Physical slots (block * block_size + offset) of tokens [t0, t1) of a sequence."""
    t = np.arange(t0, t1)
    return bt[seq, t // w.block_size].astype(np.int64) * w.block_size + t % w.block_size


def ring_slots(w: Workload, bt: np.ndarray, seq: int, t0: int, t1: int, window: int) -> np.ndarray:
    """Physical slots of tokens [t0, t1) of a sequence kept in a ring of `window`
    slots (the first window / block_size blocks of its block-table row): token t
    lives in slot t mod window."""
    r = np.arange(t0, t1) % window
    return bt[seq, r // w.block_size].astype(np.int64) * w.block_size + r % w.block_size


def scaled(w: Workload, **changes) -> Workload:
    """The same workload with some fields changed (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def sm_scale(w: Workload) -> float:
    return 1.0 / math.sqrt(w.d)
