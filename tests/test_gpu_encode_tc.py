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


@pytest.mark.parametrize("kb,vb", [(4, 4), (3, 2), (6, 6), (8, 8)])
def test_bulk_encode_structured_rows(tq, oracle, kb, vb):
    """Rows the random inputs do not produce, on the tensor-core path: a zero
    key, keys with two equal coordinates (half of their rotated coordinates
    exactly 0: the sign decision at 0 must give 2^(kb-1) - 1, as x > 0 does),
    a key on one coordinate (every rotated coordinate of one magnitude), keys
    scaled by 2^-12, 2^-20 and 2^10 (other threshold scales), a zero value row
    (scale 0) and a value row of a tiny spread."""
    import torch
    dev = "cuda"
    n = _bulk_tokens(8)
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n,), hkv=8, hq=16, key_bits=kb, value_bits=vb)
    K = W.kv_tokens(w, 0, 0, 0, n).copy()
    V = W.kv_tokens(w, 1, 0, 0, n).copy()
    K[10] = 0.0
    K[12] = 0.0
    K[12, :, 5] = 1.0
    K[12, :, 77] = 1.0
    K[13] *= 2.0 ** -12
    K[14] *= 2.0 ** 10
    K[15] = 0.0
    K[15, :, 3] = -3.0
    K[16] *= 2.0 ** -20
    V[11] = 0.0
    V[17] = 0.0
    V[17, :, 9] = 2.0 ** -14
    bt = W.block_table(w)
    nb = w.num_blocks()
    slots = W.slots(w, bt, 0, 0, n)
    oc = oracle.Cache(w.d, kb, vb, 0, w.block_size, w.hkv, nb, w.seed)
    pool_o = oc.new_pool()
    st_o = oc.encode(K, V, slots, pool_o)
    gc = tq.Cache(nb, w.hkv, kb, vb, 0, w.seed, w.block_size, w.d)
    st = tq.new_status()
    gc.encode(torch.from_numpy(K).to(dev, torch.bfloat16), torch.from_numpy(V).to(dev, torch.bfloat16),
              torch.from_numpy(slots).to(dev), st)
    torch.cuda.synchronize()
    pool_g = gc.pool.cpu().numpy()
    L = parity.Layout(w.d, kb, vb, 0, w.block_size, w.hkv, oc.page_bytes)
    all_slots = np.repeat(slots, w.hkv)
    all_heads = np.tile(np.arange(w.hkv), n)
    fo = parity.unpack(pool_o, L, all_slots, all_heads)
    fg = parity.unpack(pool_g, L, all_slots, all_heads)
    half = 1 << (kb - 1)
    rows = lambda t: slice(t * w.hkv, (t + 1) * w.hkv)  # noqa: E731
    # the exactly-zero rotated coordinates of the two-coordinate keys take the
    # lower code of the tie (the upper one is for x > 0 only); the oracle's middle
    # boundary is 0 only up to its rounding (-5e-17 at 3 bits), so its code
    # there may be either, and those 512 ties stay out of the mismatch budget
    zero = np.abs(oracle.rotate(oc.s, K[12, 0].astype(np.float64))) == 0.0
    assert zero.sum() == 64
    assert np.all(fg["k"][rows(12)][:, zero] == half - 1)
    ties = np.ix_(np.arange(12 * w.hkv, 13 * w.hkv), np.where(zero)[0])
    fo["k"][ties] = fg["k"][ties]
    enc = parity.compare_encode(fo, fg, K.reshape(-1, w.d).astype(np.float64), V.reshape(-1, w.d).astype(np.float64),
                                oc, oracle)
    enc["status_oracle"], enc["status_gpu"] = st_o, int(st.item())
    enc["other_bytes_equal"] = True
    parity.assert_encode_parity(dict(enc=enc))
    assert np.all(fg["k"][rows(10)] == half - 1) and np.all(fo["k"][rows(10)] == half - 1)
    assert np.all(fg["v"][rows(11)] == 0) and np.all(fo["v"][rows(11)] == 0)
    # rows with no coordinate near a boundary agree with the oracle code for code
    for t in (10, 11, 17):
        np.testing.assert_array_equal(fg["k"][rows(t)], fo["k"][rows(t)], err_msg=f"token {t}")
        np.testing.assert_array_equal(fg["v"][rows(t)], fo["v"][rows(t)], err_msg=f"token {t}")
    assert set(np.unique(fg["v"][rows(17)])) <= {0, (1 << vb) - 1}
    # one coordinate: every rotated coordinate has one magnitude, so one code per sign
    assert all(len(np.unique(r)) <= 2 for r in fg["k"][rows(15)])


@pytest.mark.parametrize("kb,vb", [(5, 7), (6, 6), (8, 8), (3, 1)])
def test_bulk_encode_leaves_other_bytes(tq, oracle, kb, vb):
    """Every width's code stores (direct, 32-byte, or staged rows written by
    one bulk copy each) write exactly the slots they encode: a pool of 0xAB
    keeps every byte outside them, skipped tokens (slot -1) included, and the
    written rows match the oracle's."""
    import torch
    dev = "cuda"
    n = _bulk_tokens(8)
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n,), hkv=8, hq=16, key_bits=kb, value_bits=vb)
    K = W.kv_tokens(w, 0, 0, 0, n)
    V = W.kv_tokens(w, 1, 0, 0, n)
    bt = W.block_table(w)
    nb = w.num_blocks()
    slots = W.slots(w, bt, 0, 0, n).copy()
    skipped = np.arange(5, n, 97)
    slots[skipped] = -1
    gc = tq.Cache(nb, w.hkv, kb, vb, 0, w.seed, w.block_size, w.d)
    gc.pool.fill_(0xAB)
    st = tq.new_status()
    gc.encode(torch.from_numpy(K).to(dev, torch.bfloat16), torch.from_numpy(V).to(dev, torch.bfloat16),
              torch.from_numpy(slots).to(dev), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    oc = oracle.Cache(w.d, kb, vb, 0, w.block_size, w.hkv, nb, w.seed)
    pool_o = oc.new_pool()
    pool_o[:] = 0xAB
    oc.encode(K, V, slots, pool_o)
    pool_g = gc.pool.cpu().numpy()
    L = parity.Layout(w.d, kb, vb, 0, w.block_size, w.hkv, oc.page_bytes)
    written = slots >= 0
    all_slots = np.repeat(slots[written], w.hkv)
    all_heads = np.tile(np.arange(w.hkv), int(written.sum()))
    # outside the written slots both pools hold the fill byte
    mask = np.ones(pool_g.size, dtype=bool)
    page = (all_slots // L.bs * L.hkv + all_heads) * L.page_bytes
    for base, nbytes in [(L.k, w.d * kb // 8), (L.v, w.d * vb // 8), (L.g, 2), (L.s, 2), (L.z, 2)]:
        idx = (page + base + (all_slots % L.bs) * nbytes)[:, None] + np.arange(nbytes)[None, :]
        mask[idx.ravel()] = False
    assert np.all(pool_g[mask] == 0xAB)
    assert np.all(pool_o[mask] == 0xAB)
    fo = parity.unpack(pool_o, L, all_slots, all_heads)
    fg = parity.unpack(pool_g, L, all_slots, all_heads)
    kin = K[written].reshape(-1, w.d).astype(np.float64)
    vin = V[written].reshape(-1, w.d).astype(np.float64)
    enc = parity.compare_encode(fo, fg, kin, vin, oc, oracle)
    enc["status_oracle"], enc["status_gpu"] = 0, 0
    enc["other_bytes_equal"] = True
    parity.assert_encode_parity(dict(enc=enc))


@pytest.mark.parametrize("kb,vb", [(4, 4), (8, 8), (4, 2)])
def test_bulk_encode_pool_16_byte_aligned(tq, oracle, kb, vb):
    """A pool that is 16-byte but not 32-byte aligned (the API asks for 16):
    the 4- and 8-bit rows fall back from 32-byte to 16-byte stores and the
    pool bytes come out the same as on an aligned pool."""
    import torch
    dev = "cuda"
    n = _bulk_tokens(8)
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n,), hkv=8, hq=16, key_bits=kb, value_bits=vb)
    K = torch.from_numpy(W.kv_tokens(w, 0, 0, 0, n)).to(dev, torch.bfloat16)
    V = torch.from_numpy(W.kv_tokens(w, 1, 0, 0, n)).to(dev, torch.bfloat16)
    bt = W.block_table(w)
    nb = w.num_blocks()
    slots = torch.from_numpy(W.slots(w, bt, 0, 0, n)).to(dev)
    a = tq.Cache(nb, w.hkv, kb, vb, 0, w.seed, w.block_size, w.d)
    nbytes = a.pool.numel()
    big = torch.zeros(nbytes + 64, dtype=torch.uint8, device=dev)
    assert big.data_ptr() % 32 == 0
    b = tq.Cache(nb, w.hkv, kb, vb, 0, w.seed, w.block_size, w.d, pool=big[16:16 + nbytes])
    assert b.pool.data_ptr() % 32 == 16
    st = tq.new_status()
    a.encode(K, V, slots, st)
    b.encode(K, V, slots, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(a.pool, b.pool)
    assert torch.all(big[:16] == 0) and torch.all(big[16 + nbytes:] == 0)
