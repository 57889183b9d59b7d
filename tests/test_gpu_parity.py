"""GPU parity: the CUDA path through the C ABI against the oracle, element by
element, on the same seeded inputs (tolerances in tests/parity.py)."""
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


def _check(res, decode=True):
    parity.assert_encode_parity(res)
    if decode:
        parity.assert_decode_parity(res)


def test_tiny_workload(tq, oracle):
    """1 KV head, 1 query head, 1024 fp32 tokens with four x20 key channels, 4/4 bits, seed 0."""
    res = parity.run_case(W.WORKLOADS["tiny"], oracle, tq)
    _check(res)
    assert res["dec"]["rel_err_end_to_end"] < 2e-2


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_lengths_and_groups(tq, oracle, G, dtype):
    """Lengths 1, 15, 16, 17 and 300 tokens (partial pages, single-token sequences)."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(1, 15, 16, 17, 300), hkv=2, hq=2 * G, dtype=dtype)
    _check(parity.run_case(w, oracle, tq))


@pytest.mark.parametrize("n", [2000, 5003])
def test_many_splits(tq, oracle, n):
    """Long enough that each sequence is split over several CTAs; ragged tail."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(n, n // 3), hkv=2, hq=16)
    _check(parity.run_case(w, oracle, tq))


@pytest.mark.parametrize("kb,vb,m", [(3, 3, 0), (2, 2, 128), (4, 2, 0), (2, 4, 128), (3, 4, 0), (4, 3, 128),
                                     (2, 3, 0), (3, 2, 128), (4, 4, 128)])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_other_bit_widths_and_qjl(tq, oracle, kb, vb, m, G):
    """Every built (key bits, value bits, QJL) page format, ragged lengths, several group sizes."""
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(333, 40, 1), hkv=2, hq=2 * G, key_bits=kb, value_bits=vb, qjl_m=m)
    _check(parity.run_case(w, oracle, tq))


def test_long3bit_shape_reduced(tq, oracle):
    """The 128K / 3-bit workload's head layout (64 q / 8 KV heads) at 4 x 2500 tokens."""
    w = W.scaled(W.WORKLOADS["long128k3"], lens=(2500, 2501, 17, 2000))
    _check(parity.run_case(w, oracle, tq, decode_gpu_pool=False))


def test_qjl64_shape_reduced(tq, oracle):
    """The high-concurrency QJL workload's format (2-bit + QJL m=128, 2-bit values, G=4) with
    its first 8 sequence lengths divided by 8."""
    lens = tuple(max(1, x // 8) for x in W.WORKLOADS["qjl64"].lens[:8])
    w = W.scaled(W.WORKLOADS["qjl64"], lens=lens)
    _check(parity.run_case(w, oracle, tq, decode_gpu_pool=False))


def test_swa_workload_full_size(tq, oracle):
    """8 layers x 20 heads x 4096 tokens, bf16, 4/4."""
    _check(parity.run_case(W.WORKLOADS["swa8x4096"], oracle, tq, decode_gpu_pool=False))


@pytest.mark.parametrize("q_step", [1, 2, 3, 4])
def test_swa_workload_other_queries(tq, oracle, q_step):
    """The same workload with the queries of later decode steps (160 heads with one
    query each: the widest spread of per-head errors among the workloads)."""
    _check(parity.run_case(W.WORKLOADS["swa8x4096"], oracle, tq, q_step=q_step, decode_gpu_pool=False))


def test_gqa32k_workload_full_size(tq, oracle):
    """64 q / 8 KV heads, 32768 tokens, permuted 16-token blocks, bf16, 4/4."""
    _check(parity.run_case(W.WORKLOADS["gqa32k"], oracle, tq, decode_gpu_pool=False))


def test_edge_cases(tq, oracle):
    import torch
    dev = "cuda"
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(40, 0, 20), hkv=1, hq=4)
    nb = w.num_blocks()
    bt = W.block_table(w)
    gc = tq.Cache(nb, 1)
    oc = oracle.Cache(128, 4, 4, 0, 16, 1, nb, 0)
    pool_o = oc.new_pool()
    K = W.kv_tokens(w, 0, 0, 0, 40)
    V = W.kv_tokens(w, 1, 0, 0, 40)
    K[3] = 0.0                                # a zero key
    slots = W.slots(w, bt, 0, 0, 40)
    slots[5] = -1                              # a skipped token
    st = tq.new_status()
    gc.encode(torch.from_numpy(K).to(dev, torch.bfloat16), torch.from_numpy(V).to(dev, torch.bfloat16),
              torch.from_numpy(slots).to(dev), st)
    assert oc.encode(K, V, slots, pool_o) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    pg = gc.pool.cpu().numpy()
    np.testing.assert_array_equal(pg, pool_o)   # small case: every byte equal
    # a slot past the pool and non-finite input raise flags, nothing else is written
    bad = torch.tensor([nb * 16 + 3], dtype=torch.int64, device=dev)
    gc.encode(torch.ones(1, 1, 128, device=dev), torch.ones(1, 1, 128, device=dev), bad, st)
    torch.cuda.synchronize()
    assert st.item() & tq.FLAG_BAD_SLOT
    st.zero_()
    Kn = torch.ones(1, 1, 128, device=dev)
    Kn[0, 0, 7] = float("nan")
    gc.encode(Kn, torch.ones(1, 1, 128, device=dev), torch.tensor([int(slots[0])], device=dev), st)
    torch.cuda.synchronize()
    assert st.item() & tq.FLAG_NONFINITE
    # decode: a zero-length sequence gives zeros; a bad block id is skipped and flagged
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    btt = torch.from_numpy(bt).to(dev)
    gco = tq.Cache(nb, 1, pool=torch.from_numpy(pool_o).to(dev))
    st.zero_()
    out = gco.decode(q, btt, lens, status=st).cpu().numpy()
    ref, _ = oc.decode(pool_o, q.float().cpu().numpy().astype(np.float64), bt, np.array(w.lens), W.sm_scale(w))
    assert st.item() == 0
    assert np.all(out[1] == 0)
    assert parity.rel_err(out[[0, 2]], ref[[0, 2]]) < 2e-3
    bt2 = bt.copy()
    bt2[0, 1] = nb + 5
    st.zero_()
    out2 = gco.decode(q, torch.from_numpy(bt2).to(dev), lens, status=st).cpu().numpy()
    ref2, ost = oc.decode(pool_o, q.float().cpu().numpy().astype(np.float64), bt2, np.array(w.lens), W.sm_scale(w))
    assert st.item() & tq.FLAG_BAD_SLOT and ost & oracle.FLAG_BAD_SLOT
    assert parity.rel_err(out2, ref2) < 2e-3


def test_workspace_reuse_and_determinism(tq, oracle):
    import torch
    w = W.scaled(W.WORKLOADS["gqa32k"], lens=(3000,), hkv=2, hq=16)
    res = parity.run_case(w, oracle, tq, decode_gpu_pool=False)
    dev = "cuda"
    nb = w.num_blocks()
    bt = torch.from_numpy(W.block_table(w)).to(dev)
    gc = tq.Cache(nb, 2, pool=torch.zeros(nb * 2 * 2144, dtype=torch.uint8, device=dev))
    K = torch.from_numpy(W.kv_tokens(w, 0, 0, 0, 3000)).to(dev, torch.bfloat16)
    V = torch.from_numpy(W.kv_tokens(w, 1, 0, 0, 3000)).to(dev, torch.bfloat16)
    gc.encode(K, V, torch.from_numpy(W.slots(w, W.block_table(w), 0, 0, 3000)).to(dev))
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    lens = torch.tensor([3000], dtype=torch.int32, device=dev)
    ws = gc.new_workspace(1, 16, bt.shape[1])
    outs = [gc.decode(q, bt, lens, workspace=ws).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert res["dec"]["rel_err"] < 2e-3
