"""The allocation-free decode entry point, tq_decode_attention_noalloc.

It serves callers that may not allocate device memory when they decode (an
engine that plans its memory ahead of time, code inside a pool it does not
own, a serving loop where an allocation could stall the device): instead of a
caller workspace it uses a fixed scratch area built into the library.  Here it
is called through the C ABI twice in a row and must agree with the ordinary
entry point within the decode tolerance the parity tests use; a shape that
needs more scratch than the fixed area must be refused without a launch.

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
    outs = []
    for _ in range(2):
        st = tq.new_status()
        out = torch.full((w.batch, w.hq, w.d), float("nan"), dtype=torch.float32, device=dev)
        cache.decode_noalloc(q, btt, lens, out=out, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append(out.cpu().numpy().astype(np.float64))
    for o in outs:
        assert np.all(np.isfinite(o))
        assert parity.rel_err(o, ref) <= parity.DECODE_RTOL
    assert parity.rel_err(outs[1], outs[0]) <= parity.DECODE_RTOL


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
