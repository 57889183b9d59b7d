"""A seeded sweep of random configurations through encode and decode against
the oracle: key and value widths, query-group sizes, KV heads, batch sizes,
ragged lengths (empty sequences, single tokens, page boundaries), the
three input dtypes and, for widths 2..4, the QJL sketch."""
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


def _config(seed):
    rng = np.random.default_rng(1000 + seed)
    kb, vb = (int(x) for x in rng.integers(1, 9, size=2))
    G = int(rng.integers(1, 9))
    hkv = int(rng.integers(1, 4))
    batch = int(rng.integers(1, 5))
    pool = [0, 1, 15, 16, 17, 31, 32, 33, 100, 257, 999, 1500]
    lens = tuple(int(x) for x in rng.choice(pool, size=batch))
    if max(lens) == 0:
        lens = (lens[0] + 5,) + lens[1:]
    dtype = ["bf16", "f16", "f32"][int(rng.integers(0, 3))]
    qjl_m = 0
    if rng.random() < 0.25:
        # the sketch is defined for key and value widths 2..4
        qjl_m, kb, vb = 128, int(rng.integers(2, 5)), int(rng.integers(2, 5))
    return dict(key_bits=kb, value_bits=vb, qjl_m=qjl_m, hq=hkv * G, hkv=hkv, lens=lens, dtype=dtype)


@pytest.mark.parametrize("seed", range(32))
def test_random_configuration(tq, oracle, seed):
    cfg = _config(seed)
    w = W.scaled(W.WORKLOADS["gqa32k"], **cfg)
    res = parity.run_case(w, oracle, tq, q_step=seed)
    parity.assert_encode_parity(res)
    parity.assert_decode_parity(res)


@pytest.mark.parametrize("seed", range(12))
def test_random_append_step(tq, oracle, seed):
    """The one-launch decode step (append, then attend) on random configurations
    without the sketch; every sequence holds at least the token it appends."""
    cfg = _config(100 + seed)
    cfg["qjl_m"] = 0
    cfg["lens"] = tuple(max(n, 1) for n in cfg["lens"])
    w = W.scaled(W.WORKLOADS["gqa32k"], **cfg)
    res = parity.run_append_case(w, oracle, tq, q_step=seed)
    parity.assert_encode_parity(res)
    d = res["dec"]
    assert d["status_gpu"] == d["status_oracle"] == 0, d
    assert d["rel_err"] <= parity.DECODE_RTOL, d["rel_err"]
    assert d["same_as_plain_decode"]
    assert d["same_as_encode_call"]


@pytest.mark.parametrize("seed", range(8))
def test_random_octopus(tq, oracle, seed):
    """OCTOPUS keys (b in 2..4) with min-max values of any width on random
    configurations."""
    cfg = _config(200 + seed)
    rng = np.random.default_rng(2000 + seed)
    cfg["qjl_m"] = 0
    cfg["key_bits"] = int(rng.integers(2, 5))
    w = W.scaled(W.WORKLOADS["gqa32k"], **cfg)
    parity.assert_octopus_parity(parity.run_octopus_case(w, oracle, tq, q_step=seed))
