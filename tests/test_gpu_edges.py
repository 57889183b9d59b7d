"""Edge cases of the later features: odd query-group sizes on both codecs,
OCTOPUS edge inputs (zero key, skipped and bad slots, non-finite input,
empty sequences), slots that were never written, decode steps on page-locked
host buffers, a one-page sliding window, and argument checks of prefill."""
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


@pytest.mark.parametrize("G", [3, 5, 7])
def test_odd_group_sizes(tq, oracle, G):
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(700, 33, 1), hkv=2, hq=2 * G)
    res = parity.run_case(w, oracle, tq)
    parity.assert_encode_parity(res)
    parity.assert_decode_parity(res)
    parity.assert_octopus_parity(parity.run_octopus_case(w, oracle, tq))


def test_octopus_edge_inputs(tq, oracle):
    import torch
    dev = "cuda"
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(40, 0, 20), hkv=1, hq=4)
    nb = w.num_blocks()
    bt = W.block_table(w)
    gc = tq.OctopusCache(nb, 1, 3, 4, 0)
    oc = oracle.OctCache(128, 3, 4, 16, 1, nb, 0)
    pool_o = oc.new_pool()
    K = W.kv_tokens(w, 0, 0, 0, 40)
    V = W.kv_tokens(w, 1, 0, 0, 40)
    K[3] = 0.0                                 # a zero key: every triplet rho = 0, n = (0, 0, 1)
    slots = W.slots(w, bt, 0, 0, 40)
    slots[5] = -1                              # a skipped token
    st = tq.new_status()
    gc.encode(torch.from_numpy(K).to(dev, torch.bfloat16), torch.from_numpy(V).to(dev, torch.bfloat16),
              torch.from_numpy(slots).to(dev), st)
    assert oc.encode(K, V, slots, pool_o) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    pg = gc.pool.cpu().numpy()
    z_g = oc.unpack_slot(pg, int(slots[3]) // 16, 0, int(slots[3]) % 16)
    z_o = oc.unpack_slot(pool_o, int(slots[3]) // 16, 0, int(slots[3]) % 16)
    for f in ("ixi", "ieta", "irho"):
        assert np.array_equal(z_g[f], z_o[f]), f
    assert z_g["gamma"] == 0.0
    skipped = oc.unpack_slot(pg, int(W.slots(w, bt, 0, 5, 6)[0]) // 16, 0, 5)
    assert skipped["gamma"] == 0.0 and not skipped["ixi"].any()
    bad = torch.tensor([nb * 16 + 3], dtype=torch.int64, device=dev)
    gc.encode(torch.ones(1, 1, 128, device=dev), torch.ones(1, 1, 128, device=dev), bad, st)
    torch.cuda.synchronize()
    assert st.item() & tq.FLAG_BAD_SLOT
    st.zero_()
    Kn = torch.ones(1, 1, 128, device=dev)
    Kn[0, 0, 7] = float("inf")
    gc.encode(Kn, torch.ones(1, 1, 128, device=dev), torch.tensor([int(slots[0])], device=dev), st)
    torch.cuda.synchronize()
    assert st.item() & tq.FLAG_NONFINITE
    # decode on the oracle's cache: the empty sequence gives zeros
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    go = tq.OctopusCache(nb, 1, 3, 4, 0, pool=torch.from_numpy(pool_o).to(dev))
    st.zero_()
    out = go.decode(q, torch.from_numpy(bt).to(dev), torch.tensor(w.lens, dtype=torch.int32, device=dev),
                    status=st).cpu().numpy()
    ref, _ = oc.decode(pool_o, q.float().cpu().numpy().astype(np.float64), bt, np.array(w.lens), W.sm_scale(w))
    assert st.item() == 0
    assert np.all(out[1] == 0)
    assert parity.rel_err(out[[0, 2]], ref[[0, 2]]) <= parity.DECODE_RTOL


@pytest.mark.parametrize("codec", ["main", "octopus"])
def test_unwritten_slots_are_not_read(tq, codec):
    """The slots past a sequence's end in its last page hold whatever the pool
    held (here 0xFF bytes: fp16 NaN for every gamma, scale and zero); the
    output must not depend on them."""
    import torch
    dev = "cuda"
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(21, 300, 5), hkv=2, hq=16)
    nb = w.num_blocks()
    bt = torch.from_numpy(W.block_table(w)).to(dev)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    outs = []
    for fill in (0x00, 0xFF):
        c = tq.OctopusCache(nb, 2, 4, 4, 0) if codec == "octopus" else tq.Cache(nb, 2)
        c.pool.fill_(fill)
        for b in range(w.batch):
            K = torch.from_numpy(W.kv_tokens(w, 0, b, 0, w.lens[b])).to(dev, torch.bfloat16)
            V = torch.from_numpy(W.kv_tokens(w, 1, b, 0, w.lens[b])).to(dev, torch.bfloat16)
            c.encode(K, V, torch.from_numpy(W.slots(w, W.block_table(w), b, 0, w.lens[b])).to(dev))
        st = tq.new_status()
        outs.append(c.decode(q, bt, lens, status=st).cpu().numpy())
        torch.cuda.synchronize()
        assert st.item() == 0
    assert np.isfinite(outs[1]).all()
    assert np.array_equal(outs[0], outs[1])


def test_decode_step_on_host_buffers(tq):
    """Where the kernel can reach page-locked host memory in place, a decode
    step whose k_new, v_new, q and out live there gives the cache bytes and the
    output of the same step on device buffers, bit for bit."""
    import torch
    dev = "cuda"
    probe = torch.empty(1).pin_memory()
    if not tq.device_accessible(probe):
        pytest.skip("page-locked host memory is not mapped into the device's address space here")
    assert not tq.device_accessible(torch.empty(1))  # pageable host memory never is
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(300, 17, 1), hkv=2, hq=16)
    nb = w.num_blocks()
    bt_np = W.block_table(w)
    bt = torch.from_numpy(bt_np).to(dev)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    q = torch.from_numpy(W.queries(w, 0)).to(torch.bfloat16)
    kn = torch.from_numpy(np.stack([W.kv_tokens(w, 0, b, w.lens[b] - 1, w.lens[b])[0] for b in range(w.batch)]))
    vn = torch.from_numpy(np.stack([W.kv_tokens(w, 1, b, w.lens[b] - 1, w.lens[b])[0] for b in range(w.batch)]))
    kn, vn = kn.to(torch.bfloat16), vn.to(torch.bfloat16)
    res = []
    for host in (False, True):
        c = tq.Cache(nb, 2)
        for b in range(w.batch):
            n = w.lens[b] - 1
            if n:
                K = torch.from_numpy(W.kv_tokens(w, 0, b, 0, n)).to(dev, torch.bfloat16)
                V = torch.from_numpy(W.kv_tokens(w, 1, b, 0, n)).to(dev, torch.bfloat16)
                c.encode(K, V, torch.from_numpy(W.slots(w, bt_np, b, 0, n)).to(dev))
        if host:
            args = [t.pin_memory() for t in (kn, vn, q)]
            out = torch.empty(w.batch, w.hq, 128).pin_memory()
        else:
            args = [t.to(dev) for t in (kn, vn, q)]
            out = torch.empty(w.batch, w.hq, 128, device=dev)
        st = tq.new_status()
        c.decode_append(*args, bt, lens, out=out, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        res.append((out.cpu().clone(), c.pool.cpu().clone()))
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])


def test_ring_one_page_window(tq, oracle):
    """A ring of 16 slots (one block), overwritten every 16 steps."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(16, 16), hkv=2, hq=16)
    results = parity.run_ring_stream(w, oracle, tq, 16, (3, 16), 40, {0, 12, 13, 29, 39})
    for r in results:
        parity.assert_encode_parity(r)
        assert r["dec"]["rel_err"] <= parity.DECODE_RTOL
        assert r["dec"]["same_as_plain_decode"]


def test_prefill_and_ring_argument_checks(tq):
    import torch
    c = tq.Cache(4, 2)
    q = torch.zeros((8, 16, 128), dtype=torch.bfloat16, device="cuda")
    row = torch.arange(4, dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        c.prefill(q, row, 60)                  # positions 60 .. 67 do not fit 4 blocks
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    z = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    for window in (0, 24, 80):                 # not a positive multiple of 16, or past the table
        with pytest.raises(tq.TQError) as e:
            c.decode_append(z, z, q[:1], bt, lens, window=window)
        assert e.value.status == tq.TQ_ERR_INVALID_ARG
