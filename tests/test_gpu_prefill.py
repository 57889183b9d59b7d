"""Chunked prefill attention over the compressed cache: each query position of
the chunk attends causally over the sequence's tokens up to itself, both sides
reading the oracle's cache."""
import os

import numpy as np
import pytest

from online_kv_cache_encode_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq(oracle):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_kv_cache_encode_gb300 import build
    build.build()
    from online_kv_cache_encode_gb300 import tq as T
    oracle.set_threads(os.cpu_count() or 1)
    return T


def _prefill_case(tq, oracle, first, C, kb=4, vb=4, G=8, octopus=False, dtype="bf16", bad_block=None):
    import torch

    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(first + C,), hkv=2, hq=2 * G, key_bits=kb, value_bits=vb,
                 dtype=dtype)
    bt = W.block_table(w)
    nb = w.num_blocks()
    K = W.kv_tokens(w, 0, 0, 0, first + C)
    V = W.kv_tokens(w, 1, 0, 0, first + C)
    sl = W.slots(w, bt, 0, 0, first + C)
    if octopus:
        oc = oracle.OctCache(w.d, kb, vb, w.block_size, w.hkv, nb, w.seed)
    else:
        oc = oracle.Cache(w.d, kb, vb, 0, w.block_size, w.hkv, nb, w.seed)
    pool = oc.new_pool()
    assert oc.encode(K, V, sl, pool) == 0
    q = W.to_dtype(w, np.random.default_rng(first * 7 + C).standard_normal((C, w.hq, w.d)).astype(np.float32))
    sm = W.sm_scale(w)
    lens = np.arange(first + 1, first + C + 1, dtype=np.int32)
    if bad_block is not None:
        bt = bt.copy()
        bt[0, bad_block] = nb + 3   # a block id past the pool: that page is skipped and flagged
    out_o, st = oc.decode(pool, q.astype(np.float64), np.repeat(bt, C, axis=0), lens, sm)
    assert st == (0 if bad_block is None else oracle.FLAG_BAD_SLOT)
    dev = torch.device("cuda")
    pt = torch.from_numpy(pool).to(dev)
    gc = (tq.OctopusCache(nb, w.hkv, kb, vb, w.seed, pool=pt) if octopus
          else tq.Cache(nb, w.hkv, kb, vb, 0, w.seed, pool=pt))
    status = tq.new_status()
    tdt = {"f32": torch.float32, "f16": torch.float16}.get(dtype, torch.bfloat16)
    out = gc.prefill(torch.from_numpy(q).to(dev, tdt), torch.from_numpy(bt[0]).to(dev), first, sm,
                     status=status).cpu().numpy().astype(np.float64)
    assert int(status.item()) == (0 if bad_block is None else tq.FLAG_BAD_SLOT)
    assert np.all(np.isfinite(out))
    return parity.rel_err(out, out_o)


@pytest.mark.parametrize("first,C", [(1000, 48), (0, 40), (31, 1), (4000, 64)])
def test_prefill_matches_causal_attention(tq, oracle, first, C):
    assert _prefill_case(tq, oracle, first, C) <= parity.DECODE_RTOL


def test_prefill_three_bit_and_single_query_group(tq, oracle):
    assert _prefill_case(tq, oracle, 700, 33, kb=3, vb=3, G=1) <= parity.DECODE_RTOL


def test_prefill_octopus_cache(tq, oracle):
    assert _prefill_case(tq, oracle, 500, 24, kb=4, vb=4, octopus=True) <= parity.DECODE_RTOL


@pytest.mark.parametrize("G,vb,C", [(1, 4, 70), (4, 2, 33), (8, 3, 200), (2, 1, 5)])
def test_prefill_tensor_core_shapes(tq, oracle, G, vb, C):
    """4-bit keys (the tensor-core prefill): query groups 1..8, value widths 1..4,
    chunks whose rows fill several 128-row blocks or only part of one."""
    assert _prefill_case(tq, oracle, 900, C, vb=vb, G=G) <= parity.DECODE_RTOL


def test_prefill_fp32_queries_and_start_of_sequence(tq, oracle):
    assert _prefill_case(tq, oracle, 0, 130, dtype="f32") <= parity.DECODE_RTOL


def test_prefill_bad_block_is_skipped_and_flagged(tq, oracle):
    assert _prefill_case(tq, oracle, 600, 40, bad_block=7) <= parity.DECODE_RTOL
