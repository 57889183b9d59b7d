"""tq_decode_attention_append: one launch that appends each sequence's new token
and attends over it, against the oracle (which encodes all tokens, then decodes)
and against the plain decode of the same cache."""
import pytest

from online_kv_cache_encode_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_kv_cache_encode_gb300 import build
    build.build()
    from online_kv_cache_encode_gb300 import tq as T
    return T


def _check(res):
    parity.assert_encode_parity(res)
    d = res["dec"]
    assert d["status_gpu"] == d["status_oracle"] == 0, d
    assert d["rel_err"] <= parity.DECODE_RTOL, d["rel_err"]
    assert d["same_as_plain_decode"]
    assert d["same_as_encode_call"]


@pytest.mark.parametrize("kb,vb", [(4, 4), (3, 3), (2, 4), (4, 2)])
def test_append_ragged(tq, oracle, kb, vb):
    """Several splits, a sequence whose new token opens a fresh page (len % 16 == 1),
    one that fills a page (len % 16 == 0) and a one-token sequence."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(3000, 1201, 16, 1), hkv=2, hq=16, key_bits=kb, value_bits=vb)
    _check(parity.run_append_case(w, oracle, tq))


def test_append_gqa32k_full_size(tq, oracle):
    """The 32768-token GQA workload's decode step in one launch."""
    _check(parity.run_append_case(W.WORKLOADS["gqa32k"], oracle, tq))


@pytest.mark.parametrize("kb,vb", [(2, 2), (3, 4), (4, 3)])
def test_append_qjl(tq, oracle, kb, vb):
    """Caches with the QJL sketch (m = 128): the appended token's sign row and
    residual norm are the bytes tq_encode_kv writes, and the step matches the
    oracle and the plain decode."""
    w = W.scaled(W.WORKLOADS["qjl64"], lens=(3000, 1201, 16, 1), hkv=2, hq=8, key_bits=kb, value_bits=vb)
    _check(parity.run_append_case(w, oracle, tq))
