"""Sliding-window attention kept as a ring buffer of `window` slots per
sequence: the one-launch ring step (append into slot (len - 1) mod window,
attend over the tokens the ring holds) against the oracle over a stream of
steps that crosses the wrap."""
import os

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


def _check(results):
    assert results
    for r in results:
        parity.assert_encode_parity(r)
        d = r["dec"]
        assert d["status_gpu"] == d["status_oracle"] == 0, (r["step"], d["status_gpu"])
        assert d["rel_err"] <= parity.DECODE_RTOL, (r["step"], d["rel_err"])
        assert d["same_as_plain_decode"], r["step"]


@pytest.mark.parametrize("kb,vb", [(4, 4), (3, 3), (8, 8), (1, 5)])
def test_ring_stream_crosses_the_wrap(tq, oracle, kb, vb):
    """Three sequences in rings of 256 slots: one far from full, one that wraps
    after 6 steps, one full from the start; 120 steps."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(256, 256, 256), hkv=2, hq=16, key_bits=kb, value_bits=vb)
    _check(parity.run_ring_stream(w, oracle, tq, 256, (100, 250, 256), 120, {0, 5, 6, 7, 60, 119}))


def test_ring_small_window_many_wraps(tq, oracle):
    """A 32-slot ring (two blocks) wrapped several times, G = 1 and G = 8 groups."""
    for G in (1, 8):
        w = W.scaled(W.WORKLOADS["gqa32k"], lens=(32, 32), hkv=2, hq=2 * G)
        _check(parity.run_ring_stream(w, oracle, tq, 32, (5, 31), 100, {0, 26, 27, 28, 57, 99}))


def test_ring_swa_full_size(tq, oracle):
    """The sliding-window workload streaming past its window: 8 layers x 20 heads,
    W = 4096, every ring full, three steps that overwrite the oldest tokens."""
    w = W.WORKLOADS["swa8x4096"]
    _check(parity.run_ring_stream(w, oracle, tq, 4096, (4096,) * w.batch, 3, {0, 2}))
