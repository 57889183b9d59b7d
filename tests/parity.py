"""Parity harness: run a workload through the CUDA library and through the
oracle on the same seeded inputs, and compare at the stated tolerances.

  (a) codes bit-exact, except coordinates within 1e-5 of a decision boundary
      (rotated-direction units for keys, code steps for values, |(S r)_i| /
      (||S_i|| rho) for QJL bits); such mismatches stay under 1e-5 of all
      coordinates;
  (b) fp16 norm, scale, zero and rho within 1 fp16 ulp;
  (c) decode output: max over query heads of ||gpu - oracle||_inf /
      ||oracle||_inf <= 2e-3, both sides reading the identical compressed cache
      (the oracle's own encoding of the inputs).

Tolerance (a) is stated for 2- to 4-bit codes.  Wider codes have 2^(b-4)
times denser decision boundaries, so the same fp32 rounding of the decision
variable meets a boundary 2^(b-4) times as often: the mismatch budget scales
by that factor for b > 4.  For values the decision variable (v - min) / scale
also grows to 2^b - 1, and its fp32 rounding with it: the near-boundary
distance for value codes is max(1e-5, 2^(b-21)) code steps (eight fp32 ulps
of 2^b).  Both reduce to (a) for b <= 4.

Pages are unpacked here with numpy from the layout the header documents, a
reader independent of both implementations.
"""
from __future__ import annotations

import math

import numpy as np

from online_kv_cache_encode_gb300 import workloads as W

BOUNDARY_TOL = 1e-5
MISMATCH_FRACTION = 1e-5
DECODE_RTOL = 2e-3


def width_factor(b: int) -> float:
    """Density of a b-bit code's decision boundaries relative to 4-bit codes (at least 1)."""
    return float(2 ** max(0, b - 4))


def value_boundary_tol(b: int) -> float:
    """Near-boundary distance, in code steps, for b-bit value codes."""
    return max(BOUNDARY_TOL, 2.0 ** (b - 21))


class Layout:
    def __init__(self, d, kb, vb, m, bs, hkv, page_bytes):
        self.d, self.kb, self.vb, self.m, self.bs, self.hkv = d, kb, vb, m, bs, hkv
        self.page_bytes = page_bytes
        off = 0
        self.k = off; off += bs * d * kb // 8
        self.v = off; off += bs * d * vb // 8
        self.g = off; off += 2 * bs
        self.s = off; off += 2 * bs
        self.z = off; off += 2 * bs
        if m:
            self.r = off; off += 2 * bs
            self.sig = off; off += bs * m // 8
        assert (off + 15) // 16 * 16 == page_bytes


def unpack(pool: np.ndarray, L: Layout, slots: np.ndarray, heads: np.ndarray) -> dict:
    """Fields of the given (slot, head) pairs: codes as int arrays, fp16 as raw uint16."""
    blk, off = slots // L.bs, slots % L.bs
    page = (blk * L.hkv + heads) * L.page_bytes

    def rows(base, nbytes):
        idx = (page + base + off * nbytes)[:, None] + np.arange(nbytes)[None, :]
        return pool[idx]

    def codes(base, b):
        bits = np.unpackbits(rows(base, L.d * b // 8), axis=1, bitorder="little")
        bits = bits.reshape(len(slots), L.d, b).astype(np.int64)
        return (bits << np.arange(b)[None, None, :]).sum(axis=2)

    def f16(base):
        idx = (page + base + 2 * off)[:, None] + np.arange(2)[None, :]
        return pool[idx].copy().view(np.uint16)[:, 0]

    out = dict(k=codes(L.k, L.kb), v=codes(L.v, L.vb), gamma=f16(L.g), scale=f16(L.s), zero=f16(L.z))
    if L.m:
        out["rho"] = f16(L.r)
        out["sig"] = np.unpackbits(rows(L.sig, L.m // 8), axis=1, bitorder="little").astype(np.int64)
    return out


def octopus_key_row_bytes(d: int, b: int) -> int:
    """Bytes of one OCTOPUS key row: ceil(d / 3) triplets of 3 b + 1 bits, in 4-byte words."""
    return 4 * -(-((d + 2) // 3 * (3 * b + 1)) // 32)


def unpack_octopus(pool: np.ndarray, d: int, b: int, vb: int, bs: int, hkv: int, page_bytes: int,
                   slots: np.ndarray, heads: np.ndarray) -> dict:
    """Fields of OCTOPUS (slot, head) pairs, read with numpy from the layout the
    header documents: bs key rows of KR bytes (triplet i's xi code, eta code and
    rho code, b + 1, b + 1 and b - 1 bits, LSB first from bit i (3 b + 1)), then
    value code rows, gamma, scale and zero as in the main layout."""
    slots = np.asarray(slots, dtype=np.int64)
    heads = np.asarray(heads, dtype=np.int64)
    ntri, KR, VR = (d + 2) // 3, octopus_key_row_bytes(d, b), d * vb // 8
    blk, off = slots // bs, slots % bs
    page = (blk * hkv + heads) * page_bytes
    vbase = bs * KR
    gam = vbase + bs * VR

    def rows(base, nbytes):
        idx = (page + base + off * nbytes)[:, None] + np.arange(nbytes)[None, :]
        return np.unpackbits(pool[idx], axis=1, bitorder="little").astype(np.int64)

    def field(bits, start, n):
        return (bits[:, start:start + n] << np.arange(n)[None, :]).sum(axis=1)

    kb = rows(0, KR)
    ixi = np.stack([field(kb, i * (3 * b + 1), b + 1) for i in range(ntri)], axis=1)
    ieta = np.stack([field(kb, i * (3 * b + 1) + b + 1, b + 1) for i in range(ntri)], axis=1)
    irho = np.stack([field(kb, i * (3 * b + 1) + 2 * b + 2, b - 1) for i in range(ntri)], axis=1)
    vbits = rows(vbase, VR).reshape(len(slots), d, vb)
    vq = (vbits << np.arange(vb)[None, None, :]).sum(axis=2)

    def f16(base):
        idx = (page + base + 2 * off)[:, None] + np.arange(2)[None, :]
        return pool[idx].copy().view(np.float16)[:, 0].astype(np.float64)

    return dict(ixi=ixi, ieta=ieta, irho=irho, vq=vq, gamma=f16(gam), scale=f16(gam + 2 * bs),
                zero=f16(gam + 4 * bs))


def _ordered(h: np.ndarray) -> np.ndarray:
    """fp16 bit patterns mapped to integers that step by one per representable value."""
    h = h.astype(np.int64)
    return np.where(h & 0x8000, -(h & 0x7FFF), h)


def _inputs(w):
    K = [W.kv_tokens(w, 0, b, 0, w.lens[b]) for b in range(w.batch)]
    V = [W.kv_tokens(w, 1, b, 0, w.lens[b]) for b in range(w.batch)]
    return K, V


def run_case(w, oracle, tq, q_step: int = 0, decode_gpu_pool: bool = True, decode: bool = True) -> dict:
    """Encode the workload's prefill on both sides, compare; decode one step on both, compare."""
    import torch

    dev = torch.device("cuda")
    tdt = {"f32": torch.float32, "f16": torch.float16}.get(w.dtype, torch.bfloat16)
    bt = W.block_table(w)
    nb = w.num_blocks()
    K, V = _inputs(w)
    slots = [W.slots(w, bt, b, 0, w.lens[b]) for b in range(w.batch)]

    # ---- oracle ----
    oc = oracle.Cache(w.d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, w.hkv, nb, w.seed)
    pool_o = oc.new_pool()
    st_o = 0
    for b in range(w.batch):
        st_o |= oc.encode(K[b], V[b], slots[b], pool_o)

    # ---- GPU encode ----
    gc = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, w.d)
    status = tq.new_status()
    Kt = torch.from_numpy(np.concatenate(K)).to(dev, tdt).contiguous()
    Vt = torch.from_numpy(np.concatenate(V)).to(dev, tdt).contiguous()
    sm = torch.from_numpy(np.concatenate(slots)).to(dev)
    gc.encode(Kt, Vt, sm, status)
    torch.cuda.synchronize()
    pool_g = gc.pool.cpu().numpy()
    st_g = int(status.item())

    L = Layout(w.d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, w.hkv, oc.page_bytes)
    all_slots = np.repeat(np.concatenate(slots), w.hkv)
    all_heads = np.tile(np.arange(w.hkv), len(all_slots) // w.hkv)
    fo = unpack(pool_o, L, all_slots, all_heads)
    fg = unpack(pool_g, L, all_slots, all_heads)
    kin = np.concatenate(K).reshape(-1, w.d).astype(np.float64)
    vin = np.concatenate(V).reshape(-1, w.d).astype(np.float64)
    enc = compare_encode(fo, fg, kin, vin, oc, oracle)
    enc["status_oracle"], enc["status_gpu"] = st_o, st_g
    # bytes outside the written slots (padding, other slots) must be equal
    mask = np.ones(pool_o.size, dtype=bool)
    for sl, hh in ((all_slots, all_heads),):
        page = (sl // L.bs * L.hkv + hh) * L.page_bytes
        for base, nbytes in [(L.k, w.d * w.key_bits // 8), (L.v, w.d * w.value_bits // 8),
                             (L.g, 2), (L.s, 2), (L.z, 2)] + ([(L.r, 2), (L.sig, w.qjl_m // 8)] if w.qjl_m else []):
            idx = (page + base + (sl % L.bs) * nbytes)[:, None] + np.arange(nbytes)[None, :]
            mask[idx.ravel()] = False
    enc["other_bytes_equal"] = bool(np.array_equal(pool_o[mask], pool_g[mask]))

    if not decode:
        return dict(enc=enc, dec=None, w=w)
    # ---- decode one step on the oracle's cache, both sides ----
    q = W.queries(w, q_step)
    lens = np.array(w.lens, dtype=np.int32)
    smv = W.sm_scale(w)
    out_o, dst_o = oc.decode(pool_o, q.astype(np.float64), bt, lens, smv)
    gc_o = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, w.d,
                    pool=torch.from_numpy(pool_o).to(dev))
    qt = torch.from_numpy(q).to(dev, tdt).contiguous()
    btt = torch.from_numpy(bt).to(dev)
    lt = torch.from_numpy(lens).to(dev)
    dstatus = tq.new_status()
    out_g = gc_o.decode(qt, btt, lt, smv, status=dstatus).cpu().numpy().astype(np.float64)
    dec = dict(rel_err=rel_err(out_g, out_o), status_gpu=int(dstatus.item()), status_oracle=dst_o,
               out_gpu=out_g, out_oracle=out_o)
    if decode_gpu_pool:
        # end to end: the GPU's own cache through the GPU decode vs the oracle end to end
        out_gg = gc.decode(qt, btt, lt, smv).cpu().numpy().astype(np.float64)
        dec["rel_err_end_to_end"] = rel_err(out_gg, out_o)
    torch.cuda.synchronize()
    return dict(enc=enc, dec=dec, w=w)


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over query heads of ||got - ref||_inf / ||ref||_inf."""
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


def compare_encode(fo, fg, kin, vin, oc, oracle) -> dict:
    n_vec, d = fo["k"].shape
    res = {}
    # keys
    kmis = np.argwhere(fo["k"] != fg["k"])
    bad_k = 0
    for vi, j in kmis:
        k = kin[vi]
        u = oracle.rotate(oc.s, k / np.linalg.norm(k))
        # a code may move only across the boundary it lies next to: by one level
        if np.min(np.abs(u[j] - oc.T)) > BOUNDARY_TOL or abs(int(fo["k"][vi, j]) - int(fg["k"][vi, j])) > 1:
            bad_k += 1
    res["key_mismatch"], res["key_mismatch_far"] = len(kmis), bad_k
    # values
    vmis = np.argwhere(fo["v"] != fg["v"])
    bad_v = 0
    for vi, j in vmis:
        vr = oracle.rotate(oc.s, vin[vi])
        sc = (vr.max() - vr.min()) / ((1 << oc.vb) - 1)
        x = (vr[j] - vr.min()) / sc
        if abs((x - math.floor(x)) - 0.5) > value_boundary_tol(oc.vb) or abs(int(fo["v"][vi, j]) - int(fg["v"][vi, j])) > 1:
            bad_v += 1
    res["val_mismatch"], res["val_mismatch_far"] = len(vmis), bad_v
    res["coords"] = 2 * n_vec * d
    # mismatch budget: (a) per coordinate, scaled for codes wider than 4 bits
    res["mismatch_budget"] = MISMATCH_FRACTION * n_vec * d * (width_factor(oc.kb) + width_factor(oc.vb))
    # fp16 fields
    for f in ("gamma", "scale", "zero") + (("rho",) if "rho" in fo else ()):
        res[f + "_max_ulp"] = int(np.abs(_ordered(fo[f]) - _ordered(fg[f])).max()) if n_vec else 0
    if "sig" in fo:
        ok_rows = np.all(fo["k"] == fg["k"], axis=1)
        smis = np.argwhere((fo["sig"] != fg["sig"]) & ok_rows[:, None])
        bad_s = 0
        for vi, i in smis:
            k = kin[vi]
            g = np.linalg.norm(k)
            u = oracle.rotate(oc.s, k / g)
            r = u - oc.C[fo["k"][vi]]
            if abs(oc.S[i] @ r) > BOUNDARY_TOL * np.linalg.norm(oc.S[i]) * np.linalg.norm(r):
                bad_s += 1
        res["sig_mismatch"], res["sig_mismatch_far"] = len(smis), bad_s
        res["sig_rows_skipped"] = int((~ok_rows).sum())
    return res


def run_append_case(w, oracle, tq, q_step: int = 0) -> dict:
    """The fused decode step: the GPU encodes each sequence's first lens[b] - 1
    tokens, then tq_decode_attention_append appends token lens[b] - 1 and
    attends.  The resulting cache is compared with the oracle's encoding of all
    lens[b] tokens, the output with the oracle's decode, and with the plain GPU
    decode of the same cache (which must agree bit for bit).  The cache must
    also equal, byte for byte, what tq_encode_kv of the new tokens makes of the
    cache as it was before the step.  Decode parity (c) is taken on identical
    caches: the GPU decodes the oracle's cache and is compared with the
    oracle's decode (a code within rounding of a boundary may legitimately
    differ between the two encodings and move a logit)."""
    import torch

    dev = torch.device("cuda")
    tdt = {"f32": torch.float32, "f16": torch.float16}.get(w.dtype, torch.bfloat16)
    bt = W.block_table(w)
    nb = w.num_blocks()
    K, V = _inputs(w)
    slots = [W.slots(w, bt, b, 0, w.lens[b]) for b in range(w.batch)]

    oc = oracle.Cache(w.d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, w.hkv, nb, w.seed)
    pool_o = oc.new_pool()
    st_o = 0
    for b in range(w.batch):
        st_o |= oc.encode(K[b], V[b], slots[b], pool_o)
    q = W.queries(w, q_step)
    lens = np.array(w.lens, dtype=np.int32)
    smv = W.sm_scale(w)
    out_o, dst_o = oc.decode(pool_o, q.astype(np.float64), bt, lens, smv)

    gc = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, w.d)
    status = tq.new_status()
    Kp = torch.from_numpy(np.concatenate([k[:-1] for k in K])).to(dev, tdt).contiguous()
    Vp = torch.from_numpy(np.concatenate([v[:-1] for v in V])).to(dev, tdt).contiguous()
    sp = torch.from_numpy(np.concatenate([sl[:-1] for sl in slots])).to(dev)
    if Kp.shape[0]:
        gc.encode(Kp, Vp, sp, status)
    kn = torch.from_numpy(np.stack([k[-1] for k in K])).to(dev, tdt).contiguous()
    vn = torch.from_numpy(np.stack([v[-1] for v in V])).to(dev, tdt).contiguous()
    qt = torch.from_numpy(q).to(dev, tdt).contiguous()
    btt = torch.from_numpy(bt).to(dev)
    lt = torch.from_numpy(lens).to(dev)
    pool_pre = gc.pool.clone()
    out_a = gc.decode_append(kn, vn, qt, btt, lt, smv, status=status).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    pool_g = gc.pool.cpu().numpy()
    ge = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, w.d, pool=pool_pre)
    ge.encode(kn, vn, torch.from_numpy(np.array([sl[-1] for sl in slots])).to(dev))
    same_as_encode = bool(np.array_equal(pool_g, pool_pre.cpu().numpy()))
    st_g = int(status.item())
    out_p = gc.decode(qt, btt, lt, smv).cpu().numpy().astype(np.float64)
    go = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, w.d,
                  pool=torch.from_numpy(pool_o).to(dev))
    out_go = go.decode(qt, btt, lt, smv).cpu().numpy().astype(np.float64)

    L = Layout(w.d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, w.hkv, oc.page_bytes)
    all_slots = np.repeat(np.concatenate(slots), w.hkv)
    all_heads = np.tile(np.arange(w.hkv), len(all_slots) // w.hkv)
    fo = unpack(pool_o, L, all_slots, all_heads)
    fg = unpack(pool_g, L, all_slots, all_heads)
    kin = np.concatenate(K).reshape(-1, w.d).astype(np.float64)
    vin = np.concatenate(V).reshape(-1, w.d).astype(np.float64)
    enc = compare_encode(fo, fg, kin, vin, oc, oracle)
    enc["status_oracle"], enc["status_gpu"] = st_o | dst_o, st_g
    enc["other_bytes_equal"] = True
    return dict(enc=enc, dec=dict(rel_err=rel_err(out_go, out_o), status_gpu=st_g, status_oracle=st_o | dst_o,
                                  out_gpu=out_go, out_oracle=out_o, rel_err_own_cache=rel_err(out_a, out_o),
                                  same_as_plain_decode=bool(np.array_equal(out_a, out_p)),
                                  same_as_encode_call=same_as_encode), w=w)


def assert_encode_parity(res: dict):
    e = res["enc"]
    assert e["status_gpu"] == e["status_oracle"], e
    assert e["key_mismatch_far"] == 0 and e["val_mismatch_far"] == 0, e
    assert e["key_mismatch"] + e["val_mismatch"] <= e["mismatch_budget"], e
    for f in ("gamma", "scale", "zero", "rho"):
        if f + "_max_ulp" in e:
            assert e[f + "_max_ulp"] <= 1, (f, e)
    if "sig_mismatch" in e:
        assert e["sig_mismatch_far"] == 0, e
    assert e["other_bytes_equal"], e


def assert_decode_parity(res: dict):
    d = res["dec"]
    assert d["status_gpu"] == d["status_oracle"] == 0, d
    assert np.all(np.isfinite(d["out_gpu"]))
    assert d["rel_err"] <= DECODE_RTOL, d["rel_err"]


def run_ring_stream(w, oracle, tq, window: int, t0s, steps: int, checks) -> list:
    """Sliding-window decode through rings of `window` slots per sequence.

    Both sides encode the last `window` of each sequence's first t0s[b] tokens
    into its ring (token t in slot t mod window).  Then, for `steps` steps, the
    GPU runs one tq_decode_attention_ring_append launch per step: it appends
    token t0s[b] + i and attends.  The oracle encodes the same token into the
    same slot and decodes over the min(len, window) slots the ring holds.  At
    the steps in `checks`, the ring contents are compared field by field
    (every slot that holds a token), and the output against the oracle and
    against a plain GPU decode of the same ring.  Decode parity (c) is taken
    on identical caches: the GPU decodes the oracle's ring and is compared
    with the oracle's decode."""
    import torch

    dev = torch.device("cuda")
    tdt = {"f32": torch.float32, "f16": torch.float16}.get(w.dtype, torch.bfloat16)
    bt = W.block_table(w)
    nb = w.num_blocks()
    B = w.batch
    t0s = np.asarray(t0s, dtype=np.int64)
    oc = oracle.Cache(w.d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, w.hkv, nb, w.seed)
    pool_o = oc.new_pool()
    gc = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, w.d)
    status = tq.new_status()
    st_o = 0
    for b in range(B):
        lo = max(0, int(t0s[b]) - window)
        if lo == t0s[b]:
            continue
        K = W.kv_tokens(w, 0, b, lo, int(t0s[b]))
        V = W.kv_tokens(w, 1, b, lo, int(t0s[b]))
        sl = W.ring_slots(w, bt, b, lo, int(t0s[b]), window)
        st_o |= oc.encode(K, V, sl, pool_o)
        gc.encode(torch.from_numpy(K).to(dev, tdt).contiguous(), torch.from_numpy(V).to(dev, tdt).contiguous(),
                  torch.from_numpy(sl).to(dev), status)
    btt = torch.from_numpy(bt).to(dev)
    smv = W.sm_scale(w)
    L = Layout(w.d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, w.hkv, oc.page_bytes)
    results = []
    for i in range(steps):
        lens = (t0s + i + 1).astype(np.int32)
        kn = np.stack([W.kv_tokens(w, 0, b, int(lens[b]) - 1, int(lens[b]))[0] for b in range(B)])
        vn = np.stack([W.kv_tokens(w, 1, b, int(lens[b]) - 1, int(lens[b]))[0] for b in range(B)])
        q = W.queries(w, i)
        for b in range(B):
            st_o |= oc.encode(kn[b:b + 1], vn[b:b + 1],
                              W.ring_slots(w, bt, b, int(lens[b]) - 1, int(lens[b]), window), pool_o)
        qt = torch.from_numpy(q).to(dev, tdt).contiguous()
        lt = torch.from_numpy(lens).to(dev)
        out_g = gc.decode_append(torch.from_numpy(kn).to(dev, tdt).contiguous(),
                                 torch.from_numpy(vn).to(dev, tdt).contiguous(), qt, btt, lt, smv,
                                 status=status, window=window)
        if i not in checks:
            continue
        held = np.minimum(lens, window).astype(np.int32)
        out_a = out_g.cpu().numpy().astype(np.float64)
        out_p = gc.decode(qt, btt, torch.from_numpy(held).to(dev), smv).cpu().numpy().astype(np.float64)
        torch.cuda.synchronize()
        st_g = int(status.item())
        out_o, dst_o = oc.decode(pool_o, q.astype(np.float64), bt, held, smv)
        go = tq.Cache(nb, w.hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed, w.block_size, w.d,
                      pool=torch.from_numpy(pool_o).to(dev))
        out_go = go.decode(qt, btt, torch.from_numpy(held).to(dev), smv).cpu().numpy().astype(np.float64)
        pool_g = gc.pool.cpu().numpy()
        sl, kin, vin = [], [], []
        for b in range(B):
            lo = int(lens[b]) - int(held[b])
            sl.append(W.ring_slots(w, bt, b, lo, int(lens[b]), window))
            kin.append(W.kv_tokens(w, 0, b, lo, int(lens[b])))
            vin.append(W.kv_tokens(w, 1, b, lo, int(lens[b])))
        all_slots = np.repeat(np.concatenate(sl), w.hkv)
        all_heads = np.tile(np.arange(w.hkv), len(all_slots) // w.hkv)
        fo = unpack(pool_o, L, all_slots, all_heads)
        fg = unpack(pool_g, L, all_slots, all_heads)
        kin = np.concatenate(kin).reshape(-1, w.d).astype(np.float64)
        vin = np.concatenate(vin).reshape(-1, w.d).astype(np.float64)
        enc = compare_encode(fo, fg, kin, vin, oc, oracle)
        enc["status_oracle"], enc["status_gpu"] = st_o | dst_o, st_g
        enc["other_bytes_equal"] = True
        results.append(dict(step=i, enc=enc,
                            dec=dict(rel_err=rel_err(out_go, out_o), status_gpu=st_g, status_oracle=st_o | dst_o,
                                     out_gpu=out_go, out_oracle=out_o, rel_err_own_cache=rel_err(out_a, out_o),
                                     same_as_plain_decode=bool(np.array_equal(out_a, out_p)))))
    return results


def run_octopus_case(w, oracle, tq, q_step: int = 0) -> dict:
    """OCTOPUS keys (w.key_bits is the codec's b), min-max values: encode the
    workload on both sides and compare the pages; decode one step with the GPU
    reading the oracle's cache and compare with the oracle's decode.

    A key triplet's codes may differ only where the decision is within 1e-5 of
    a tie in the oracle's own arithmetic: the GPU's direction pair scores
    within 1e-5 of the oracle's pair (<n, n^>), or xi, eta or rho lies within
    1e-5 of a boundary of its codebook.  Such triplets stay under the (a)
    budget, 1e-5 of all triplets scaled by the direction width factor."""
    import torch

    dev = torch.device("cuda")
    tdt = {"f32": torch.float32, "f16": torch.float16}.get(w.dtype, torch.bfloat16)
    bt = W.block_table(w)
    nb = w.num_blocks()
    K, V = _inputs(w)
    slots = [W.slots(w, bt, b, 0, w.lens[b]) for b in range(w.batch)]
    oc = oracle.OctCache(w.d, w.key_bits, w.value_bits, w.block_size, w.hkv, nb, w.seed)
    pool_o = oc.new_pool()
    st_o = 0
    for b in range(w.batch):
        st_o |= oc.encode(K[b], V[b], slots[b], pool_o)
    gc = tq.OctopusCache(nb, w.hkv, w.key_bits, w.value_bits, w.seed)
    assert gc.page_bytes == oc.page_bytes
    status = tq.new_status()
    for b in range(w.batch):
        if w.lens[b]:
            gc.encode(torch.from_numpy(K[b]).to(dev, tdt).contiguous(), torch.from_numpy(V[b]).to(dev, tdt).contiguous(),
                      torch.from_numpy(slots[b]).to(dev), status)
    torch.cuda.synchronize()
    pool_g = gc.pool.cpu().numpy()
    st_g = int(status.item())
    # ---- keys ----
    kin = np.concatenate(K).reshape(-1, w.hkv, w.d).astype(np.float64)
    vin = np.concatenate(V).reshape(-1, w.hkv, w.d).astype(np.float64)
    all_slots = np.concatenate(slots)
    mism = far = 0
    vmis = vfar = 0
    ulp = {"gamma": 0, "scale": 0, "zero": 0}
    n_tri = 0
    sl_all = np.repeat(all_slots, w.hkv)
    hd_all = np.tile(np.arange(w.hkv), len(all_slots))
    fo = unpack_octopus(pool_o, w.d, w.key_bits, w.value_bits, w.block_size, w.hkv, oc.page_bytes, sl_all, hd_all)
    fg = unpack_octopus(pool_g, w.d, w.key_bits, w.value_bits, w.block_size, w.hkv, oc.page_bytes, sl_all, hd_all)
    for i, sl in enumerate(all_slots):
        for h in range(w.hkv):
            r_ = i * w.hkv + h
            uo = {f: v[r_] for f, v in fo.items()}
            ug = {f: v[r_] for f, v in fg.items()}
            n_tri += oc.ntri
            for f in ulp:
                a16 = np.array([uo[f]], dtype=np.float16).view(np.int16).astype(np.int64)[0]
                b16 = np.array([ug[f]], dtype=np.float16).view(np.int16).astype(np.int64)[0]
                ulp[f] = max(ulp[f], int(abs(_ordered(np.array([a16 & 0xFFFF], dtype=np.uint16))[0] -
                                             _ordered(np.array([b16 & 0xFFFF], dtype=np.uint16))[0])))
            bad = np.nonzero((uo["ixi"] != ug["ixi"]) | (uo["ieta"] != ug["ieta"]) | (uo["irho"] != ug["irho"]))[0]
            if len(bad):
                k = kin[i, h]
                u = oracle.rotate(oc.s, k / np.linalg.norm(k))
                u = np.concatenate([u, np.zeros(3 * oc.ntri - w.d)])
                for j in bad:
                    mism += 1
                    t = u[3 * j: 3 * j + 3]
                    rho = np.linalg.norm(t)
                    n = t / rho if rho > 0 else np.array([0.0, 0.0, 1.0])
                    xi, eta = oracle.oct_map(n)
                    near = False
                    if uo["irho"][j] != ug["irho"][j]:
                        near = np.min(np.abs(oc.Trho - rho)) <= BOUNDARY_TOL
                    else:
                        near = True
                    if (uo["ixi"][j], uo["ieta"][j]) != (ug["ixi"][j], ug["ieta"][j]):
                        so = n @ oracle.oct_inverse(oc.Cxi[uo["ixi"][j]], oc.Cxi[uo["ieta"][j]])
                        sg = n @ oracle.oct_inverse(oc.Cxi[ug["ixi"][j]], oc.Cxi[ug["ieta"][j]])
                        tie = abs(so - sg) <= BOUNDARY_TOL
                        edge = min(np.min(np.abs(oc.Txi - xi)), np.min(np.abs(oc.Txi - eta))) <= BOUNDARY_TOL
                        near = near and (tie or edge)
                    far += 0 if near else 1
            vb_ = np.nonzero(uo["vq"] != ug["vq"])[0]
            if len(vb_):
                vr = oracle.rotate(oc.s, vin[i, h])
                sc = (vr.max() - vr.min()) / ((1 << w.value_bits) - 1)
                for j in vb_:
                    vmis += 1
                    x = (vr[j] - vr.min()) / sc
                    if abs((x - math.floor(x)) - 0.5) > value_boundary_tol(w.value_bits) or abs(int(uo["vq"][j]) - int(ug["vq"][j])) > 1:
                        vfar += 1
    enc = dict(triplet_mismatch=mism, triplet_mismatch_far=far, val_mismatch=vmis, val_mismatch_far=vfar,
               triplets=n_tri, coords=len(all_slots) * w.hkv * w.d,
               budget=MISMATCH_FRACTION * (n_tri * width_factor(w.key_bits + 1) + len(all_slots) * w.hkv * w.d *
                                           width_factor(w.value_bits)),
               status_oracle=st_o, status_gpu=st_g, **{f + "_max_ulp": v for f, v in ulp.items()})
    # ---- decode on identical caches ----
    q = W.queries(w, q_step)
    lens = np.array(w.lens, dtype=np.int32)
    smv = W.sm_scale(w)
    out_o, dst_o = oc.decode(pool_o, q.astype(np.float64), bt, lens, smv)
    go = tq.OctopusCache(nb, w.hkv, w.key_bits, w.value_bits, w.seed, pool=torch.from_numpy(pool_o).to(dev))
    dstat = tq.new_status()
    out_g = go.decode(torch.from_numpy(q).to(dev, tdt).contiguous(), torch.from_numpy(bt).to(dev),
                      torch.from_numpy(lens).to(dev), smv, status=dstat).cpu().numpy().astype(np.float64)
    dec = dict(rel_err=rel_err(out_g, out_o), status_gpu=int(dstat.item()), status_oracle=dst_o,
               out_gpu=out_g, out_oracle=out_o)
    return dict(enc=enc, dec=dec, w=w)


def assert_octopus_parity(res: dict):
    e = res["enc"]
    assert e["status_gpu"] == e["status_oracle"], e
    assert e["triplet_mismatch_far"] == 0 and e["val_mismatch_far"] == 0, e
    assert e["triplet_mismatch"] + e["val_mismatch"] <= e["budget"], e
    for f in ("gamma", "scale", "zero"):
        assert e[f + "_max_ulp"] <= 1, (f, e)
    assert_decode_parity(res)
