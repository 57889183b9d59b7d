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


def test_append_refuses_qjl(tq):
    import torch
    c = tq.Cache(8, 2, 2, 2, 128)
    z = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        c.decode_append(z, z, q, bt, lens)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
