"""The bulk encode on the tensor cores (16-bit inputs without the QJL sketch,
at least one 128-row tile per SM): parity with the oracle with a ragged last
tile, bf16 and fp16 inputs and key / value widths 1..8; the status flags of
its rows (non-finite input, fp16 overflow, a slot past the pool, a skipped
slot)."""
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


def _bulk_tokens(hkv: int, tiles_per_sm: int = 2) -> int:
    """Tokens whose (token, KV head) items fill `tiles_per_sm` 128-row tiles per
    SM, plus a ragged last tile."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (tiles_per_sm * sms * 128 + hkv - 1) // hkv + 37


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("kb,vb", [(4, 4), (3, 3), (2, 4), (1, 1), (5, 6), (8, 8), (6, 2), (7, 5)])
def test_bulk_encode_parity(tq, oracle, dtype, kb, vb):
    n = _bulk_tokens(8)
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n,), hkv=8, hq=16, key_bits=kb, value_bits=vb, dtype=dtype)
    res = parity.run_case(w, oracle, tq, decode=False)
    assert (n * 8) % 128 != 0
    parity.assert_encode_parity(res)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_one_tile_per_sm(tq, oracle, dtype):
    """The smallest encode the tensor cores take: one tile per SM and a few
    more, so most CTAs code a single tile and some slots none."""
    n = _bulk_tokens(8, tiles_per_sm=1)
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n,), hkv=8, hq=16, dtype=dtype)
    parity.assert_encode_parity(parity.run_case(w, oracle, tq, decode=False))


def test_bulk_encode_two_sequences_and_decode(tq, oracle):
    """Two sequences in one call (the second starting mid-tile) and a decode
    of the GPU's own cache against the oracle end to end."""
    n = _bulk_tokens(4)
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n // 2 + 3, n // 2 + 61), hkv=4, hq=16)
    res = parity.run_case(w, oracle, tq)
    parity.assert_encode_parity(res)
    parity.assert_decode_parity(res)
    assert res["dec"]["rel_err_end_to_end"] < 2e-2


def test_bulk_encode_flags(tq, oracle):
    import torch
    dev = "cuda"
    n = _bulk_tokens(8)
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n,), hkv=8, hq=16)
    nb = w.num_blocks()
    bt = W.block_table(w)
    K = W.kv_tokens(w, 0, 0, 0, n)
    V = W.kv_tokens(w, 1, 0, 0, n)
    slots = W.slots(w, bt, 0, 0, n)
    c = tq.Cache(nb, 8)
    st = tq.new_status()

    def run(K, V, slots):
        st.zero_()
        c.encode(torch.from_numpy(K).to(dev, torch.bfloat16), torch.from_numpy(V).to(dev, torch.bfloat16),
                 torch.from_numpy(slots).to(dev), st)
        torch.cuda.synchronize()
        return int(st.item())

    assert run(K, V, slots) == 0
    Kn = K.copy()
    Kn[n - 5, 3, 17] = np.nan
    assert run(Kn, V, slots) == tq.FLAG_NONFINITE
    Vn = V.copy()
    Vn[1000, 0, 0] = np.inf
    assert run(K, Vn, slots) == tq.FLAG_NONFINITE
    Kb = K.copy()
    Kb[7] *= 1e5  # gamma above the fp16 range
    assert run(Kb, V, slots) == tq.FLAG_OVERFLOW
    sb = slots.copy()
    sb[n // 2] = nb * 16
    assert run(K, V, sb) == tq.FLAG_BAD_SLOT
    # a skipped token (slot -1) leaves its slot's bytes alone
    c.pool.fill_(0xAB)
    sk = slots.copy()
    sk[100] = -1
    assert run(K, V, sk) == 0
    pool = c.pool.cpu().numpy()
    oc = oracle.Cache(w.d, w.key_bits, w.value_bits, 0, w.block_size, w.hkv, nb, w.seed)
    L = parity.Layout(w.d, w.key_bits, w.value_bits, 0, w.block_size, w.hkv, oc.page_bytes)
    page = (int(slots[100]) // 16 * 8 + np.arange(8)) * L.page_bytes
    off = int(slots[100]) % 16
    for base, nbytes in [(L.k, 64), (L.v, 64), (L.g, 2), (L.s, 2), (L.z, 2)]:
        for p in page:
            assert np.all(pool[p + base + off * nbytes: p + base + (off + 1) * nbytes] == 0xAB)
