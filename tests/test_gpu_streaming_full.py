"""Full-size parity of the two streaming workloads, through their whole life:
prefill, then every decode step.

  long128k3  4 sequences x 131072 tokens, 64 q / 8 KV heads, 3-bit keys and
             values; prefill encoded in 4096-token chunks, then 64 steps, each
             one tq_decode_attention_append launch that appends one token per
             sequence and attends.
  qjl64      64 sequences of U[1K, 16K] tokens, 32 q / 8 KV heads, 2-bit keys
             with the QJL sketch (m = 128), 2-bit values; 128 steps, each one
             append + attend launch.

The GPU runs the whole workload at its stated size.  The oracle is too slow
to encode and decode everything, so it follows a seeded subset of (sequence,
KV head) units in full: it encodes each such unit's every token, prefill and
appended ones, from the same seeded inputs.  Checks:

  - encode, tolerance (a)/(b): the GPU pool's pages of the sampled units after
    prefill, and every unit's appended token at the checked steps, against the
    oracle's encoding of the same vectors;
  - decode, tolerance (c) on identical caches: at the checked steps a copy of
    the GPU pool gets the sampled units' pages from the oracle's own cache,
    the GPU decodes the full batch on it in the launch configuration of the
    step (same batch, heads, block table, lengths, split plan), and the
    sampled units' outputs are compared with the oracle's decode;
  - the step's own output (GPU cache) against the oracle, and against a plain
    decode of the same cache (bit for bit).

No CUDA output ever becomes an oracle input.
"""
import os

import numpy as np
import pytest

from online_kv_cache_encode_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

UNITS = 8          # (sequence, KV head) units the oracle follows in full
APPEND_QJL = True   # whether the one-launch append step takes caches with the QJL sketch
EXTRA_CHECKS = 2   # seeded checked steps besides the first, middle and last


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


def _checked_steps(n, seed):
    fixed = {0, n // 2 - 1 if n == 64 else n // 2, n - 1}
    rng = np.random.default_rng(seed)
    rest = sorted(set(range(n)) - fixed)
    return sorted(fixed | set(int(x) for x in rng.choice(rest, EXTRA_CHECKS, replace=False)))


def _run(w, oracle, tq, checks):
    import torch
    dev = "cuda"
    B, hkv, G, d = w.batch, w.hkv, w.group, w.d
    bt = W.block_table(w)
    mb = bt.shape[1]
    nb = w.num_blocks()
    rng = np.random.default_rng([w.wid, 77])
    flat = rng.choice(B * hkv, UNITS, replace=False)
    units = [(int(u) // hkv, int(u) % hkv) for u in sorted(flat)]

    # ---- GPU: prefill in chunks ----
    gc = tq.Cache(nb, hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, d)
    status = tq.new_status()
    # ---- oracle: one hkv = 1 cache holding the sampled units as sequences ----
    oc = oracle.Cache(d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, 1, UNITS * mb, w.seed)
    pool_o = oc.new_pool()
    ubt = np.arange(UNITS * mb, dtype=np.int32).reshape(UNITS, mb)   # unit u owns blocks u*mb ..
    st_o = 0
    kin = {u: [] for u in range(UNITS)}
    vin = {u: [] for u in range(UNITS)}
    for b in range(B):
        for t0 in range(0, w.lens[b], w.prefill_chunk):
            t1 = min(w.lens[b], t0 + w.prefill_chunk)
            K = W.kv_tokens(w, 0, b, t0, t1)
            V = W.kv_tokens(w, 1, b, t0, t1)
            gc.encode(torch.from_numpy(K).to(dev, torch.bfloat16), torch.from_numpy(V).to(dev, torch.bfloat16),
                      torch.from_numpy(W.slots(w, bt, b, t0, t1)).to(dev), status)
            for u, (ub, uh) in enumerate(units):
                if ub != b:
                    continue
                t = np.arange(t0, t1)
                st_o |= oc.encode(K[:, uh:uh + 1], V[:, uh:uh + 1], ubt[u, t // 16].astype(np.int64) * 16 + t % 16,
                                  pool_o)
                kin[u].append(K[:, uh])
                vin[u].append(V[:, uh])
    torch.cuda.synchronize()
    assert status.item() == 0 and st_o == 0

    Lg = parity.Layout(d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, hkv, gc.page_bytes)
    Lo = parity.Layout(d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, 1, oc.page_bytes)

    def compare_units(pool_g, lens_now, lo_tok=None):
        """Encode parity of the sampled units' tokens [lo_tok or 0, lens_now[b])."""
        res = []
        for u, (ub, uh) in enumerate(units):
            t = np.arange(0 if lo_tok is None else lo_tok[ub], lens_now[ub])
            gs = W.slots(w, bt, ub, int(t[0]), int(t[-1]) + 1)
            os_ = ubt[u, t // 16].astype(np.int64) * 16 + t % 16
            fg = parity.unpack(pool_g, Lg, gs, np.full(len(t), uh))
            fo = parity.unpack(pool_o, Lo, os_, np.zeros(len(t), dtype=np.int64))
            k = np.concatenate(kin[u])[t].astype(np.float64)
            v = np.concatenate(vin[u])[t].astype(np.float64)
            res.append(parity.compare_encode(fo, fg, k, v, oc, oracle))
        return res

    def assert_enc(rs):
        for e in rs:
            e = dict(e, status_gpu=0, status_oracle=0, other_bytes_equal=True)
            parity.assert_encode_parity(dict(enc=e))

    assert_enc(compare_units(gc.pool.cpu().numpy(), w.lens))

    # ---- decode steps ----
    steps = w.decode_steps
    newK = [W.kv_tokens(w, 0, b, w.lens[b], w.lens[b] + steps) for b in range(B)]
    newV = [W.kv_tokens(w, 1, b, w.lens[b], w.lens[b] + steps) for b in range(B)]
    btt = torch.from_numpy(bt).to(dev)
    smv = W.sm_scale(w)
    ws = gc.new_workspace(B, w.hq, mb)
    lens0 = np.array(w.lens, dtype=np.int64)
    report = []
    for i in range(steps):
        lens = (lens0 + i + 1).astype(np.int32)
        kn = np.stack([newK[b][i] for b in range(B)])
        vn = np.stack([newV[b][i] for b in range(B)])
        q = W.queries(w, i)
        qt = torch.from_numpy(q).to(dev, torch.bfloat16)
        lt = torch.from_numpy(lens).to(dev)
        knt = torch.from_numpy(kn).to(dev, torch.bfloat16).contiguous()
        vnt = torch.from_numpy(vn).to(dev, torch.bfloat16).contiguous()
        if w.qjl_m and not APPEND_QJL:
            # caches with the QJL sketch: the step is an encode launch, then a decode launch
            new_slots = np.array([W.slots(w, bt, b, int(lens[b]) - 1, int(lens[b]))[0] for b in range(B)])
            gc.encode(knt, vnt, torch.from_numpy(new_slots).to(dev), status)
            out_step = gc.decode(qt, btt, lt, smv, workspace=ws, status=status)
        else:
            out_step = gc.decode_append(knt, vnt, qt, btt, lt, smv, workspace=ws, status=status)
        for u, (ub, uh) in enumerate(units):
            t = int(lens[ub]) - 1
            st_o |= oc.encode(kn[ub:ub + 1, uh:uh + 1], vn[ub:ub + 1, uh:uh + 1],
                              np.array([ubt[u, t // 16] * 16 + t % 16], dtype=np.int64), pool_o)
            kin[u].append(kn[ub:ub + 1, uh])
            vin[u].append(vn[ub:ub + 1, uh])
        if i not in checks:
            continue
        torch.cuda.synchronize()
        assert status.item() == 0 and st_o == 0, (i, status.item(), st_o)
        pool_g = gc.pool.cpu().numpy()
        # the appended token of every unit against the oracle's encoding of it
        oa = oracle.Cache(d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, hkv, B, w.seed)
        pool_a = oa.new_pool()
        assert oa.encode(kn, vn, np.arange(B, dtype=np.int64) * 16, pool_a) == 0
        sl = np.repeat(lens.astype(np.int64) - 1, hkv)
        gsl = np.array([W.slots(w, bt, s // hkv, int(sl[s]), int(sl[s]) + 1)[0] for s in range(B * hkv)])
        hh = np.tile(np.arange(hkv), B)
        fg = parity.unpack(pool_g, Lg, gsl, hh)
        fa = parity.unpack(pool_a, parity.Layout(d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, hkv,
                                                 oa.page_bytes), np.repeat(np.arange(B, dtype=np.int64) * 16, hkv), hh)
        e_new = parity.compare_encode(fa, fg, kn.reshape(-1, d).astype(np.float64),
                                      vn.reshape(-1, d).astype(np.float64), oa, oracle)
        assert_enc([e_new])
        # decode on identical caches: the sampled units' pages from the oracle's cache
        patched = gc.pool.clone()
        pg = patched.view(-1, gc.page_bytes)
        po = torch.from_numpy(pool_o).to(dev).view(-1, oc.page_bytes)
        for u, (ub, uh) in enumerate(units):
            nblk = -(-int(lens[ub]) // 16)
            dst = torch.from_numpy(bt[ub, :nblk].astype(np.int64) * hkv + uh).to(dev)
            pg[dst] = po[u * mb: u * mb + nblk]
        gp = tq.Cache(nb, hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, d, pool=patched)
        dst_ = tq.new_status()
        out_p = gp.decode(qt, btt, lt, smv, workspace=ws, status=dst_).cpu().numpy().astype(np.float64)
        out_plain = gc.decode(qt, btt, lt, smv, workspace=ws).cpu().numpy().astype(np.float64)
        torch.cuda.synchronize()
        assert dst_.item() == 0
        qo = np.stack([q[ub, uh * G:(uh + 1) * G] for ub, uh in units]).astype(np.float64)
        out_o, dst_o = oc.decode(pool_o, qo, ubt, np.array([lens[ub] for ub, _ in units], dtype=np.int32), smv)
        assert dst_o == 0
        got = np.stack([out_p[ub, uh * G:(uh + 1) * G] for ub, uh in units])
        own = np.stack([out_step.cpu().numpy().astype(np.float64)[ub, uh * G:(uh + 1) * G] for ub, uh in units])
        r = dict(step=i, rel_err=parity.rel_err(got, out_o), rel_err_own_cache=parity.rel_err(own, out_o),
                 same_as_plain=bool(np.array_equal(out_step.cpu().numpy().astype(np.float64), out_plain)))
        report.append(r)
        assert np.all(np.isfinite(got))
        assert r["rel_err"] <= parity.DECODE_RTOL, r
        assert r["rel_err_own_cache"] <= 2e-2, r
        assert r["same_as_plain"], r
    assert status.item() == 0
    return report


def test_long128k3_full_size_stream(tq, oracle):
    """4 x 131072 tokens of 3/3, 4096-token prefill chunks, 64 append + attend steps."""
    w = W.WORKLOADS["long128k3"]
    rep = _run(w, oracle, tq, _checked_steps(w.decode_steps, 4))
    assert [r["step"] for r in rep][:1] == [0] and rep[-1]["step"] == 63
    assert any(r["step"] == 31 for r in rep)


def test_qjl64_full_size_stream(tq, oracle):
    """64 sequences of U[1K, 16K] tokens, 2-bit keys + QJL (m = 128), 2-bit values, 128 steps."""
    w = W.WORKLOADS["qjl64"]
    rep = _run(w, oracle, tq, _checked_steps(w.decode_steps, 5))
    assert rep[0]["step"] == 0 and rep[-1]["step"] == 127
    assert any(r["step"] == 64 for r in rep)
