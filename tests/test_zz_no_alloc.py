"""The allocation-free decode entry point, tq_decode_attention_noalloc.

It serves callers that may not allocate device memory when they decode (an
engine that plans its memory ahead of time, code inside a pool it does not
own, a serving loop where an allocation could stall the device): instead of a
caller workspace it uses a fixed scratch area built into the library.  Here it
is called through the C ABI twice in a row and must give exactly what the
ordinary entry point gives (the same kernel with the same split plan, so bit
for bit, well inside the decode tolerance the parity tests use), for both
codecs, without changing the device's free memory; a shape that needs more
scratch than the fixed area must be refused without a launch.

This file is collected last on purpose and must pass alone or after the rest.
"""
import numpy as np
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


def test_noalloc_matches_workspace_entry_point_twice(tq):
    import torch
    dev = "cuda"
    # several splits per sequence (the counters matter), a ragged tail and a short sequence
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(3000, 1200, 17), hkv=2, hq=16)
    nb = w.num_blocks()
    bt = W.block_table(w)
    cache = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed)
    for b in range(w.batch):
        K = torch.from_numpy(W.kv_tokens(w, 0, b, 0, w.lens[b])).to(dev, torch.bfloat16)
        V = torch.from_numpy(W.kv_tokens(w, 1, b, 0, w.lens[b])).to(dev, torch.bfloat16)
        cache.encode(K, V, torch.from_numpy(W.slots(w, bt, b, 0, w.lens[b])).to(dev))
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    btt = torch.from_numpy(bt).to(dev)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    assert cache.workspace_bytes(w.batch, w.hq, bt.shape[1]) <= tq.NOALLOC_WORKSPACE_BYTES

    ref = cache.decode(q, btt, lens).cpu().numpy().astype(np.float64)
    outs = [torch.full((w.batch, w.hq, w.d), float("nan"), dtype=torch.float32, device=dev) for _ in range(3)]
    sts = [tq.new_status() for _ in range(3)]
    cache.decode_noalloc(q, btt, lens, out=outs[0], status=sts[0])  # warm-up: the module is loaded
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for i in (1, 2):
        cache.decode_noalloc(q, btt, lens, out=outs[i], status=sts[i])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "the no-allocation entry point changed the free device memory"
    for st, o in zip(sts, outs):
        assert st.item() == 0
        o = o.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(o))
        assert parity.rel_err(o, ref) <= parity.DECODE_RTOL
        assert np.array_equal(o, ref)


def test_noalloc_octopus_matches_workspace_entry_point(tq):
    import torch
    dev = "cuda"
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(2000, 33), hkv=2, hq=8)
    nb = w.num_blocks()
    bt = W.block_table(w)
    cache = tq.OctopusCache(nb, w.hkv, bits=3, value_bits=4)
    for b in range(w.batch):
        K = torch.from_numpy(W.kv_tokens(w, 0, b, 0, w.lens[b])).to(dev, torch.bfloat16)
        V = torch.from_numpy(W.kv_tokens(w, 1, b, 0, w.lens[b])).to(dev, torch.bfloat16)
        cache.encode(K, V, torch.from_numpy(W.slots(w, bt, b, 0, w.lens[b])).to(dev))
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    btt = torch.from_numpy(bt).to(dev)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    ref = cache.decode(q, btt, lens).clone()
    for _ in range(2):
        st = tq.new_status()
        out = torch.full((w.batch, w.hq, w.d), float("nan"), dtype=torch.float32, device=dev)
        cache.decode_noalloc(q, btt, lens, out=out, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert torch.equal(out, ref)


def test_noalloc_refuses_shapes_beyond_the_fixed_workspace(tq):
    import torch
    dev = "cuda"
    hkv, hq, batch = 8, 64, 2048
    cache = tq.Cache(4, hkv)
    need = cache.workspace_bytes(batch, hq, 1)
    assert need > tq.NOALLOC_WORKSPACE_BYTES
    q = torch.zeros((batch, hq, 128), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((batch, 1), dtype=torch.int32, device=dev)
    lens = torch.zeros(batch, dtype=torch.int32, device=dev)
    out = torch.empty((batch, hq, 128), dtype=torch.float32, device=dev)
    with pytest.raises(tq.TQError) as e:
        cache.decode_noalloc(q, bt, lens, out=out)
    assert e.value.status == tq.TQ_ERR_WORKSPACE
    assert "fixed workspace" in str(e.value)
