"""Codes of every width 1 .. 8 for keys and for values, chosen per cache (per
layer): the GPU path against the oracle, the one-launch append step at the new
widths, and the 8-bit pin (the output approaches exact attention as the value
width grows)."""
import math
import os

import numpy as np
import pytest

from online_kv_cache_encode_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

# every width appears at least once for keys and for values, and together
# with narrow and wide partners
PAIRS = [(1, 1), (1, 8), (5, 5), (5, 2), (6, 6), (6, 3), (7, 7), (7, 4), (8, 8), (8, 1), (2, 5), (3, 6), (4, 7)]


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


@pytest.mark.parametrize("G", [1, 8])
@pytest.mark.parametrize("kb,vb", PAIRS)
def test_widths_parity(tq, oracle, kb, vb, G):
    """Encode and decode at (key bits, value bits); ragged lengths, several splits."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(1333, 40, 1), hkv=2, hq=2 * G, key_bits=kb, value_bits=vb)
    res = parity.run_case(w, oracle, tq)
    parity.assert_encode_parity(res)
    parity.assert_decode_parity(res)


@pytest.mark.parametrize("kb,vb", [(8, 8), (5, 7), (1, 1), (6, 2)])
def test_widths_append(tq, oracle, kb, vb):
    """The one-launch decode step at the new widths: cache bytes equal a one-token
    encode, output equals the plain decode of that cache and matches the oracle."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(3000, 1201, 16, 1), hkv=2, hq=16, key_bits=kb, value_bits=vb)
    res = parity.run_append_case(w, oracle, tq)
    parity.assert_encode_parity(res)
    d = res["dec"]
    assert d["status_gpu"] == d["status_oracle"] == 0, d
    assert d["rel_err"] <= parity.DECODE_RTOL, d["rel_err"]
    assert d["same_as_plain_decode"]
    assert d["same_as_encode_call"]


def test_eight_bit_gqa32k_full_size(tq, oracle):
    """The 32768-token GQA workload with 8-bit keys and values."""
    w = W.scaled(W.WORKLOADS["gqa32k"], key_bits=8, value_bits=8)
    res = parity.run_case(w, oracle, tq, decode_gpu_pool=False)
    parity.assert_encode_parity(res)
    parity.assert_decode_parity(res)


def test_output_approaches_exact_attention_with_width(tq):
    """With logits near zero the keys hardly matter and the output error against
    exact attention on the unquantised inputs is the value quantisation error:
    at most sqrt(d) * scale / 2 per coordinate (a rotated-frame error of at most
    scale / 2 per coordinate, rotated back), shrinking as the width grows."""
    import torch

    d, T, hkv = 128, 40, 1
    rng = np.random.default_rng(4)
    K = rng.standard_normal((T, hkv, d)).astype(np.float32)
    V = rng.standard_normal((T, hkv, d)).astype(np.float32)
    q = (rng.standard_normal((1, 1, d)) * 1e-9).astype(np.float32)
    exact = V[:, 0].astype(np.float64).mean(axis=0)
    errs = {}
    for vb in (2, 4, 6, 8):
        c = tq.Cache(4, hkv, 8, vb, 0, 3)
        slots = torch.arange(T, dtype=torch.int64, device="cuda")
        c.encode(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda(), slots)
        bt = torch.arange(4, dtype=torch.int32, device="cuda").reshape(1, 4)
        lens = torch.tensor([T], dtype=torch.int32, device="cuda")
        out = c.decode(torch.from_numpy(q).cuda(), bt, lens, 1 / math.sqrt(d)).cpu().numpy().astype(np.float64)
        L = parity.Layout(d, 8, vb, 0, 16, hkv, c.page_bytes)
        f = parity.unpack(c.pool.cpu().numpy(), L, np.arange(T), np.zeros(T, dtype=np.int64))
        scale = f["scale"].view(np.float16).astype(np.float64).max()
        errs[vb] = np.abs(out[0, 0] - exact).max()
        assert errs[vb] <= math.sqrt(d) * scale / 2 * 1.01 + 1e-3, (vb, errs[vb], scale)
    assert errs[8] < errs[6] < errs[4] < errs[2], errs
    assert errs[8] < 0.01, errs
