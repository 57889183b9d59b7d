"""The device-side timeout path of the decode kernels.

Every wait in the decode kernels is bounded; a wait that gives up sets
TQ_FLAG_TIMEOUT and the call returns with an incomplete output.  The test hook
tq_test_stall_waits makes warp 0 of every odd split wait on a shared-memory
barrier that nothing arrives on, with a short bound, so that this path runs
for real without faulting or hanging anything.  After such a call the same
workspace must serve the next call exactly: the timed-out CTAs still take part
in the split merge, so the split counters are back at zero.
"""
import numpy as np
import pytest

from online_kv_cache_encode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STALL_CYCLES = 200_000  # about 0.1 ms at GB300 clocks


@pytest.fixture(scope="module")
def tq():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_kv_cache_encode_gb300 import build
    build.build()
    from online_kv_cache_encode_gb300 import tq as T
    yield T
    T.set_test_stall(0)


def _filled(tq, cache_cls, w, **kw):
    import torch
    dev = "cuda"
    nb = w.num_blocks()
    bt = W.block_table(w)
    cache = cache_cls(nb, w.hkv, **kw)
    for b in range(w.batch):
        K = torch.from_numpy(W.kv_tokens(w, 0, b, 0, w.lens[b])).to(dev, torch.bfloat16)
        V = torch.from_numpy(W.kv_tokens(w, 1, b, 0, w.lens[b])).to(dev, torch.bfloat16)
        cache.encode(K, V, torch.from_numpy(W.slots(w, bt, b, 0, w.lens[b])).to(dev))
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    return cache, q, torch.from_numpy(bt).to(dev), torch.tensor(w.lens, dtype=torch.int32, device=dev)


def _counters(ws, batch, hkv, need):
    """The split counters at the end of a main-codec workspace."""
    n = batch * hkv * 4
    region = (n + 255) // 256 * 256
    return ws[need - region: need - region + n].cpu().numpy()


def test_timeout_leaves_the_workspace_usable(tq):
    import torch
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(3000, 1700), hkv=2, hq=16)
    cache, q, bt, lens = _filled(tq, tq.Cache, w)
    need = cache.workspace_bytes(w.batch, w.hq, bt.shape[1])
    ref = cache.decode(q, bt, lens, workspace=cache.new_workspace(w.batch, w.hq, bt.shape[1])).clone()
    ws = cache.new_workspace(w.batch, w.hq, bt.shape[1])
    st = tq.new_status()
    tq.set_test_stall(STALL_CYCLES)
    try:
        bad = cache.decode(q, bt, lens, workspace=ws, status=st).clone()
        torch.cuda.synchronize()
    finally:
        tq.set_test_stall(0)
    assert st.item() & tq.FLAG_TIMEOUT
    assert torch.isfinite(bad).all()
    assert not torch.equal(bad, ref)  # the odd splits' pages are missing
    assert np.all(_counters(ws, w.batch, w.hkv, need) == 0)
    st.zero_()
    again = cache.decode(q, bt, lens, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(again, ref)


def test_timeout_in_the_append_step(tq):
    """The one-launch append + decode step: a timed-out call still appends the
    token (its encoder is not stalled), and the next call on the same workspace
    gives the exact result."""
    import torch
    dev = "cuda"
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(2501,), hkv=2, hq=16)
    cache, q, bt, lens = _filled(tq, tq.Cache, W.scaled(w, lens=(2500,)))
    kn = torch.from_numpy(W.kv_tokens(w, 0, 0, 2500, 2501)).to(dev, torch.bfloat16).contiguous()
    vn = torch.from_numpy(W.kv_tokens(w, 1, 0, 2500, 2501)).to(dev, torch.bfloat16).contiguous()
    lens = torch.tensor([2501], dtype=torch.int32, device=dev)
    ref = cache.decode_append(kn, vn, q, bt, lens, workspace=cache.new_workspace(1, w.hq, bt.shape[1])).clone()
    pool_ref = cache.pool.clone()
    ws = cache.new_workspace(1, w.hq, bt.shape[1])
    st = tq.new_status()
    tq.set_test_stall(STALL_CYCLES)
    try:
        cache.decode_append(kn, vn, q, bt, lens, workspace=ws, status=st)
        torch.cuda.synchronize()
    finally:
        tq.set_test_stall(0)
    assert st.item() & tq.FLAG_TIMEOUT
    assert torch.equal(cache.pool, pool_ref)
    st.zero_()
    again = cache.decode_append(kn, vn, q, bt, lens, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(again, ref)


def test_timeout_octopus(tq):
    import torch
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(3000,), hkv=2, hq=16)
    cache, q, bt, lens = _filled(tq, tq.OctopusCache, w, bits=4, value_bits=4)
    ref = cache.decode(q, bt, lens).clone()
    st = tq.new_status()
    tq.set_test_stall(STALL_CYCLES)
    try:
        bad = cache.decode(q, bt, lens, status=st).clone()
        torch.cuda.synchronize()
    finally:
        tq.set_test_stall(0)
    assert st.item() & tq.FLAG_TIMEOUT
    assert torch.isfinite(bad).all()
    st.zero_()
    again = cache.decode(q, bt, lens, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(again, ref)


def test_timeout_prefill(tq):
    """The tensor-core prefill: CTAs of odd splits give up a bounded wait and
    contribute empty partials; the call is flagged and the next one is exact."""
    import torch
    dev = "cuda"
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(3000,), hkv=2, hq=16)
    cache, _, bt, _ = _filled(tq, tq.Cache, w)
    q = torch.from_numpy(W.bf16_round(np.random.default_rng(3).standard_normal((64, 16, 128)).astype(np.float32)))
    q = q.to(dev, torch.bfloat16)
    row = bt[0].contiguous()
    ref = cache.prefill(q, row, 3000 - 64).clone()
    st = tq.new_status()
    tq.set_test_stall(STALL_CYCLES)
    try:
        cache.prefill(q, row, 3000 - 64, status=st)
        torch.cuda.synchronize()
    finally:
        tq.set_test_stall(0)
    assert st.item() & tq.FLAG_TIMEOUT
    st.zero_()
    again = cache.prefill(q, row, 3000 - 64, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(again, ref)
