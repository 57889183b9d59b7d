"""The OCTOPUS triplet key codec on the GPU against the oracle: pages (codes
bit-exact except near-ties in the oracle's own arithmetic, fp16 fields within
one ulp) and decode attention with both sides reading the oracle's cache."""
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


@pytest.mark.parametrize("G", [1, 8])
@pytest.mark.parametrize("b,vb", [(4, 4), (3, 3), (2, 2), (4, 8), (2, 5), (3, 1)])
def test_octopus_ragged(tq, oracle, b, vb, G):
    """Lengths 333, 40 and 1, two KV heads, several splits."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(333, 40, 1), hkv=2, hq=2 * G, key_bits=b, value_bits=vb)
    parity.assert_octopus_parity(parity.run_octopus_case(w, oracle, tq))


def test_octopus_many_splits(tq, oracle):
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(5003, 1200), hkv=2, hq=16)
    parity.assert_octopus_parity(parity.run_octopus_case(w, oracle, tq, q_step=1))


def test_octopus_tiny_workload_fp32(tq, oracle):
    """The tiny workload (fp32 keys with four x20 channels) through the OCTOPUS codec."""
    parity.assert_octopus_parity(parity.run_octopus_case(W.WORKLOADS["tiny"], oracle, tq))
