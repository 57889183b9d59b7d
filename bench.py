"""Benchmark: one decode step of the 32K-context GQA workload on the compressed cache.

A step is the whole online path for one new token: encode (append) the new
key/value of all 8 KV heads into the paged 4-bit cache, then decode attention
for the 64 query heads over the 32768 cached tokens.  The metric is GB/s of
compressed KV the decode reads (32768 tokens x 8 KV heads x 134 B = 35.13 MB per
step) over the step time.  Prefill encode throughput (Mtokens/s) is reported
beside it.

Inputs are synthetic and seeded; caches are rotated among 16 distinct copies
(562 MB in total, above the 129 MB L2) so that every step reads from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (under torch.distributed.run) each rank runs its own replica of the
workload (independent sequences, no data-path collective: weak scaling); the
reported value is the bytes all ranks read over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from online_kv_cache_encode_gb300 import workloads as W  # noqa: E402

WORKLOAD = "gqa32k"
METRIC = "compressed-KV decode-attention GB/s (% of HBM peak); KV encode Mtokens/s"
N_COPIES = 16
# other key / value widths measured on the same workload shape (the widths a
# cache may choose per layer); each row: encode and decode-only throughput
WIDTHS = [(1, 1), (3, 3), (5, 5), (6, 6), (8, 8)]
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("tq_decode_impl.cuh", "tq_device.cuh", "tq_internal.h"):
        with open(os.path.join(ROOT, "online_kv_cache_encode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_gqa32k.md")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash()
    for line in open(p):
        if line.startswith("traffic_bytes_per_launch:"):
            parts = line.split()
            if len(parts) >= 4 and parts[2] == "source" and parts[3] == want:
                return float(parts[1])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"tq_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def count(self) -> int:
        if self.proc is None:
            return 0
        self.fh.flush()
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import torch
    from online_kv_cache_encode_gb300 import tq

    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[WORKLOAD]
    T = w.lens[0]
    hkv, hq, d = w.hkv, w.hq, w.d
    nb = w.num_blocks()
    bt_np = W.block_table(w)
    bt = torch.from_numpy(bt_np).to(dev)
    lens = torch.tensor([T], dtype=torch.int32, device=dev)
    bpth = w.bytes_per_token_head()
    decode_bytes = T * hkv * bpth

    # ---- prefill: encode the context once (timed: encode throughput), then copy to the replicas ----
    K = torch.from_numpy(W.kv_tokens(w, 0, 0, 0, T)).to(dev, torch.bfloat16)
    V = torch.from_numpy(W.kv_tokens(w, 1, 0, 0, T)).to(dev, torch.bfloat16)
    slots = torch.from_numpy(W.slots(w, bt_np, 0, 0, T)).to(dev)
    status = tq.new_status(dev)
    base = tq.Cache(nb, hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        base.encode(K, V, slots, status)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_enc = 10
    e0.record(stream)
    for _ in range(n_enc):
        base.encode(K, V, slots, status)
    e1.record(stream)
    torch.cuda.synchronize()
    enc_ms = e0.elapsed_time(e1) / n_enc
    copies = [base] + [tq.Cache(nb, hkv, w.key_bits, w.value_bits, w.qjl_m, w.seed,
                                pool=base.pool.clone()) for _ in range(N_COPIES - 1)]
    q_w = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    if args.profile_octopus:
        # an OCTOPUS 4/4 cache of the same context, then six decode launches
        # (ncu -k regex:oct_decode -s 1 -c 1)
        oc = tq.OctopusCache(nb, hkv, 4, 4, w.seed)
        oc.encode(K, V, slots, status)
        ows = oc.new_workspace(1, hq, bt.shape[1])
        oout = torch.empty((1, hq, d), dtype=torch.float32, device=dev)
        for _ in range(6):
            oc.decode(q_w, bt, lens, out=oout, workspace=ows, status=status)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "gqa32k OCTOPUS 4/4 decode", "device_status": int(status.item())}), flush=True)
        return
    if args.profile_prefill:
        # the 64-position chunked prefill at the end of the context, four launches
        # (ncu -k regex:prefill_tc_kernel -s 1 -c 1)
        C = 64
        qp = torch.from_numpy(W.bf16_round(np.random.default_rng(5).standard_normal((C, hq, d)).astype(np.float32)))
        qp = qp.to(dev, torch.bfloat16)
        row = bt[0].contiguous()
        pout = torch.empty((C, hq, d), dtype=torch.float32, device=dev)
        nbytes = int(tq.lib().tq_prefill_workspace_bytes(base._h, C, hq, row.shape[0]))
        pws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        for _ in range(4):
            base.prefill(qp, row, T - C, out=pout, workspace=pws, status=status)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "gqa32k 64-position prefill", "device_status": int(status.item())}), flush=True)
        return
    widths = [] if args.profile or args.no_widths else width_sweep(tq, w, K, V, slots, bt, q_w, measured_peaks()[0])
    ring = {} if args.profile or args.no_widths else ring_stream(tq, dev, measured_peaks()[0])
    octopus = [] if args.profile or args.no_widths else octopus_sweep(tq, w, K, V, slots, bt, q_w, measured_peaks()[0])
    prefill = {} if args.profile or args.no_widths else prefill_chunk(tq, w, base, bt)
    configs = {} if args.profile or args.no_widths else config_rows(tq, dev, measured_peaks()[0])
    del K, V

    # ---- per-step inputs: the new token (position T-1) and the query ----
    newK = torch.from_numpy(W.kv_tokens(w, 0, 0, T - 1, T)).to(dev, torch.bfloat16)
    newV = torch.from_numpy(W.kv_tokens(w, 1, 0, T - 1, T)).to(dev, torch.bfloat16)
    new_slot = torch.from_numpy(W.slots(w, bt_np, 0, T - 1, T)).to(dev)
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    out = torch.empty((1, hq, d), dtype=torch.float32, device=dev)
    wss = [c.new_workspace(1, hq, bt.shape[1]) for c in copies]

    if args.profile:
        # three warm-up decode launches, then three to capture (ncu -k regex:decode_kernel -s 3 -c 3)
        for i in range(6):
            copies[i % N_COPIES].decode(q, bt, lens, out=out, workspace=wss[i % N_COPIES], status=status)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "gqa32k decode", "device_status": int(status.item())}), flush=True)
        return

    def step(i):
        # the decode step in one launch: append the new token, then attend
        c = copies[i % N_COPIES]
        c.decode_append(newK, newV, q, bt, lens, out=out, workspace=wss[i % N_COPIES], status=status)

    def capture(fn, n):
        """CUDA graph of n calls of fn(i) (the library launches on torch's current stream)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                fn(i)
        return g

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    steps_graph = capture(step, args.steps)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # the sampler sees the GPU under this same load before and after the timed region
        steps_graph.replay()
        torch.cuda.synchronize()
        deadline = time.time() + 3.0
        while clk.count() < 3 and time.time() < deadline:
            steps_graph.replay()
            torch.cuda.synchronize()
        barrier(dist)
        torch.cuda.synchronize()
        t0.record(stream)
        steps_graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        n_before = clk.count()
        deadline = time.time() + 1.0
        while clk.count() <= n_before and time.time() < deadline:
            steps_graph.replay()
            torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    step_ms = t0.elapsed_time(t1) / args.steps
    launches = args.steps
    del steps_graph

    # ---- the decode kernel alone (roofline): a graph of back-to-back decode launches ----
    def dec(i):
        copies[i % N_COPIES].decode(q, bt, lens, out=out, workspace=wss[i % N_COPIES])

    nd = max(args.steps, 20)
    dec_graph = capture(dec, nd)
    dec_graph.replay()
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    dec_graph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    dec_ms = d0.elapsed_time(d1) / nd
    del dec_graph

    # ---- end to end through the public API with host buffers ----
    # the step's inputs (new K, new V, q) staged in one pinned host buffer and
    # copied with one host-to-device transfer per step; the output comes back
    # with one device-to-host copy.  (The API also lets the kernel read and
    # write pinned host memory in place; inputs in place measured slower, and
    # the output in place no better: 27.1 / 30.2 / 32.9 us per step in three
    # runs against 30.7 / 31.4 us.)
    nk, nv, nq = newK.numel(), newV.numel(), q.numel()
    hin = torch.cat([newK.reshape(-1), newV.reshape(-1), q.reshape(-1)]).cpu().pin_memory()
    hout = torch.empty_like(out, device="cpu").pin_memory()
    din = torch.empty_like(hin, device=dev)
    dK = din[:nk].view(newK.shape)
    dV = din[nk:nk + nv].view(newV.shape)
    dq = din[nk + nv:].view(q.shape)

    def e2e_step(i):
        din.copy_(hin, non_blocking=True)
        c = copies[i % N_COPIES]
        c.decode_append(dK, dV, dq, bt, lens, out=out, workspace=wss[i % N_COPIES], status=status)
        hout.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(args.steps + i)
    torch.cuda.synchronize()
    barrier(dist)
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = x0.elapsed_time(x1) / args.steps
    st = int(status.item())
    # the last step's host-resident output against the same step through device buffers
    i_last = args.steps - 1
    c = copies[i_last % N_COPIES]
    ref_out = c.decode(q, bt, lens, workspace=wss[i_last % N_COPIES]).cpu()
    e2e_same = bool(torch.equal(hout, ref_out))

    step_ms = max_over_ranks(step_ms, dist)
    e2e_ms = max_over_ranks(e2e_ms, dist)
    dec_ms = max_over_ranks(dec_ms, dist)
    enc_ms = max_over_ranks(enc_ms, dist)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    value = world * decode_bytes / (step_ms * 1e-3) / 1e9
    achieved = decode_bytes / (dec_ms * 1e-3) / 1e9
    enc_tokens = T  # tokens (positions) per prefill encode call, all 8 KV heads each
    enc_bytes = T * hkv * (2 * d * 2 + bpth)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "operands": "4-bit key centroids as two-level fp16 (integer part + remainder) x fp16 hi+lo queries; value "
                    "codes as exact fp16 subnormals x fp16 weights; mma.sync, fp32 accumulate",
        "data": "synthetic (seeded N(0,1) bf16 K/V with 4 x20 outlier channels per KV head and per-token lognormal(0,0.25); N(0,1) bf16 q)",
        "config": {
            "workload": "gqa32k: 64 query / 8 KV heads, head_dim 128, 32768-token context, batch 1, "
                        "4-bit keys and values, 16-token pages in a permuted block table",
            "step": "append 1 new token (8 KV heads) + decode attention for 64 query heads over 32768 tokens, one launch (tq_decode_attention_append)",
            "decode_bytes_per_step": decode_bytes,
            "l2": f"inputs larger than L2: {N_COPIES} distinct caches rotated ({N_COPIES * decode_bytes / 1e6:.0f} MB)",
            "timing": "the K steps captured in one CUDA graph, replayed once between CUDA events; "
                      "e2e is eager per-call through the Python binding",
            "parallelism": f"replica per GPU x{world}",
        },
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "roofline": {
            "kernel": "decode_kernel<4,4,0>",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(),
            "algorithmic_bytes_per_launch": decode_bytes,
            "decode_ms": round(dec_ms, 5),
        },
        "encode": {
            "metric": "KV encode Mtokens/s (prefill, 1 token = 8 KV heads of one position)",
            "value": round(enc_tokens / (enc_ms * 1e-3) / 1e6, 2),
            "tokens_per_call": enc_tokens,
            "ms_per_call": round(enc_ms, 5),
            "achieved_GBps": round(enc_bytes / (enc_ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(enc_bytes / (enc_ms * 1e-3) / 1e9 / peak, 4),
        },
        "e2e": {
            "value": round(world * decode_bytes / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 5),
            "h2d_bytes_per_step": int(newK.numel() * 2 + newV.numel() * 2 + q.numel() * 2),
            "d2h_bytes_per_step": int(out.numel() * 4),
            "path": "one host-to-device copy, the decode launch, one device-to-host copy per step",
            "output_equals_device_path": e2e_same,
        },
        "widths": widths,
        "ring": ring,
        "octopus": octopus,
        "prefill": prefill,
        "configs": configs,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "device_status": st,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


def width_sweep(tq, w, K, V, slots, bt, q, peak):
    """Encode and decode-only throughput of the workload at the other widths in
    WIDTHS: the same seeded K/V encoded at each width, decodes timed as one CUDA
    graph over enough distinct cache copies to exceed L2 (about 512 MB)."""
    import torch

    T, hkv, hq, d = w.lens[0], w.hkv, w.hq, w.d
    nb = w.num_blocks()
    lens = torch.tensor([T], dtype=torch.int32, device=K.device)
    out = torch.empty((1, hq, d), dtype=torch.float32, device=K.device)
    rows = []
    for kb, vb in WIDTHS:
        base = tq.Cache(nb, hkv, kb, vb, 0, w.seed)
        for _ in range(3):
            base.encode(K, V, slots)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            base.encode(K, V, slots)
        e1.record()
        torch.cuda.synchronize()
        enc_ms = e0.elapsed_time(e1) / 10
        bpth = tq.page_bytes(d, kb, vb, 0, w.block_size) // w.block_size
        dec_bytes = T * hkv * bpth
        n = max(2, -(-512_000_000 // dec_bytes))
        caches = [base] + [tq.Cache(nb, hkv, kb, vb, 0, w.seed, pool=base.pool.clone()) for _ in range(n - 1)]
        wss = [c.new_workspace(1, hq, bt.shape[1]) for c in caches]
        reps = max(20, n)
        for i in range(3):
            caches[i % n].decode(q, bt, lens, out=out, workspace=wss[i % n])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                caches[i % n].decode(q, bt, lens, out=out, workspace=wss[i % n])
        g.replay()
        torch.cuda.synchronize()
        best = 1e9
        for _ in range(3):
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / reps)
        gbps = dec_bytes / (best * 1e-3) / 1e9
        enc_gbps = T * hkv * (2 * d * 2 + bpth) / (enc_ms * 1e-3) / 1e9
        rows.append({"key_bits": kb, "value_bits": vb, "bytes_per_token_head": bpth,
                     "decode_GBps": round(gbps, 1), "decode_frac": round(gbps / peak, 4),
                     "decode_us": round(best * 1e3, 2), "decode_copies": n,
                     "encode_Mtok_s": round(T / (enc_ms * 1e-3) / 1e6, 1), "encode_frac": round(enc_gbps / peak, 4)})
        del g, caches, wss, base
        torch.cuda.empty_cache()
    return rows


def octopus_sweep(tq, w, K, V, slots, bt, q, peak):
    """The OCTOPUS triplet key codec on the same workload and inputs: encode
    Mtokens/s and decode GB/s of compressed bytes read (one decode launch plus
    its merge launch, timed as a CUDA graph over caches larger than L2)."""
    import torch

    T, hkv, hq, d = w.lens[0], w.hkv, w.hq, w.d
    nb = w.num_blocks()
    lens = torch.tensor([T], dtype=torch.int32, device=K.device)
    out = torch.empty((1, hq, d), dtype=torch.float32, device=K.device)
    rows = []
    for b, vb in ((4, 4), (2, 2)):
        base = tq.OctopusCache(nb, hkv, b, vb, w.seed)
        for _ in range(3):
            base.encode(K, V, slots)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            base.encode(K, V, slots)
        e1.record()
        torch.cuda.synchronize()
        enc_ms = e0.elapsed_time(e1) / 10
        pb = base.page_bytes
        dec_bytes = (T // w.block_size) * hkv * pb
        n = max(2, -(-512_000_000 // dec_bytes))
        caches = [base] + [tq.OctopusCache(nb, hkv, b, vb, w.seed, pool=base.pool.clone()) for _ in range(n - 1)]
        wss = [c.new_workspace(1, hq, bt.shape[1]) for c in caches]
        reps = max(20, n)
        for i in range(3):
            caches[i % n].decode(q, bt, lens, out=out, workspace=wss[i % n])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                caches[i % n].decode(q, bt, lens, out=out, workspace=wss[i % n])
        g.replay()
        torch.cuda.synchronize()
        best = 1e9
        for _ in range(3):
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / reps)
        gbps = dec_bytes / (best * 1e-3) / 1e9
        rows.append({"bits": b, "value_bits": vb, "page_bytes": pb, "decode_us": round(best * 1e3, 2),
                     "decode_GBps": round(gbps, 1), "decode_frac": round(gbps / peak, 4),
                     "encode_Mtok_s": round(T / (enc_ms * 1e-3) / 1e6, 1), "launches_per_decode": 2})
        del g, caches, wss, base
        torch.cuda.empty_cache()
    return rows


def prefill_chunk(tq, w, base, bt, C=64):
    """Chunked prefill attention on the same cache: the last C positions of the
    32768-token sequence (their keys and values already in the cache) attend
    causally over the cache; timed as a CUDA graph over 4 cache copies."""
    import torch

    hq, d = w.hq, w.d
    T = w.lens[0]
    n = 4
    caches = [base] + [tq.Cache(base.num_blocks, base.hkv, base.kb, base.vb, 0, base.seed, pool=base.pool.clone())
                       for _ in range(n - 1)]
    q = torch.from_numpy(W.bf16_round(np.random.default_rng(5).standard_normal((C, hq, d)).astype(np.float32)))
    q = q.to(base.pool.device, torch.bfloat16)
    row = bt[0].contiguous()
    out = torch.empty((C, hq, d), dtype=torch.float32, device=q.device)
    nbytes = int(tq.lib().tq_prefill_workspace_bytes(base._h, C, hq, row.shape[0]))
    wss = [torch.zeros(nbytes, dtype=torch.uint8, device=q.device) for _ in range(n)]
    for i in range(3):
        caches[i % n].prefill(q, row, T - C, out=out, workspace=wss[i % n])
    torch.cuda.synchronize()
    reps = 8
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            caches[i % n].prefill(q, row, T - C, out=out, workspace=wss[i % n])
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e9
    for _ in range(3):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / reps)
    del g, caches, wss
    torch.cuda.empty_cache()
    flops = 2 * 2 * C * hq * T * d  # scores and PV, 2 FLOP per multiply-add (causal: < 0.2 % fewer)
    return {"workload": f"gqa32k: the last {C} positions of the 32768-token sequence, causal, 4/4",
            "us_per_chunk": round(best * 1e3, 2), "positions_per_s": round(C / (best * 1e-3), 1),
            "tflops": round(flops / (best * 1e-3) / 1e12, 1),
            "kernel": "prefill_tc_kernel (tcgen05: 128 query rows per CTA, each page unpacked once per row block) "
                      "+ prefill_merge_kernel"}


def ring_stream(tq, dev, peak):
    """The sliding-window workload streaming past its window: 8 layers x 20 KV
    heads (G = 1), window 4096 kept as a ring per layer, every ring full.  One
    step = one tq_decode_attention_ring_append launch per layer (append the
    layer's new token into slot (len - 1) mod 4096, attend over the 4096 tokens
    the ring holds).  Steps are timed as one CUDA graph over enough copies of
    the 8 layers to exceed L2; lens stays fixed across replays, so every replay
    rewrites the same slot, which does not change the work."""
    import torch

    w = W.WORKLOADS["swa8x4096"]
    win, layers, hkv = 4096, w.batch, w.hkv
    nb = win // w.block_size
    bt = torch.from_numpy(np.random.default_rng(7).permutation(nb).astype(np.int32)[None, :]).to(dev)
    slots = bt[0].repeat_interleave(w.block_size).to(torch.int64) * w.block_size + \
        torch.arange(win, device=dev).remainder(w.block_size)
    base = []
    for l in range(layers):
        c = tq.Cache(nb, hkv, w.key_bits, w.value_bits, 0, w.seed)
        K = torch.from_numpy(W.kv_tokens(w, 0, l, 0, win)).to(dev, torch.bfloat16)
        V = torch.from_numpy(W.kv_tokens(w, 1, l, 0, win)).to(dev, torch.bfloat16)
        c.encode(K, V, slots)
        base.append(c)
    step_bytes = layers * win * hkv * w.bytes_per_token_head()
    nsets = max(2, -(-512_000_000 // step_bytes))
    sets = [base] + [[tq.Cache(nb, hkv, w.key_bits, w.value_bits, 0, w.seed, pool=c.pool.clone()) for c in base]
                     for _ in range(nsets - 1)]
    kn = [torch.from_numpy(W.kv_tokens(w, 0, l, win, win + 1)).to(dev, torch.bfloat16) for l in range(layers)]
    vn = [torch.from_numpy(W.kv_tokens(w, 1, l, win, win + 1)).to(dev, torch.bfloat16) for l in range(layers)]
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    qs = [q[l:l + 1].contiguous() for l in range(layers)]
    lens = torch.tensor([win + 1], dtype=torch.int32, device=dev)
    out = torch.empty((1, w.hq, w.d), dtype=torch.float32, device=dev)
    wss = [[c.new_workspace(1, w.hq, nb) for c in cs] for cs in sets]

    def step(i):
        k = i % nsets
        for l in range(layers):
            sets[k][l].decode_append(kn[l], vn[l], qs[l], bt, lens, out=out, workspace=wss[k][l], window=win)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    reps = max(10, nsets)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            step(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e9
    for _ in range(3):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / reps)
    gbps = step_bytes / (best * 1e-3) / 1e9
    del g, sets, wss, base
    torch.cuda.empty_cache()
    return {"workload": "swa8x4096 streaming: 8 layers x 20 KV heads (G = 1), window 4096 ring per layer, full",
            "launches_per_step": layers, "us_per_step": round(best * 1e3, 2),
            "bytes_per_step": step_bytes, "GBps": round(gbps, 1), "frac": round(gbps / peak, 4),
            "copies": nsets}


def device_kv(dev, T, hkv, d, seed, dtype=None):
    """Synthetic K or V [T, hkv, d] made on the device with the workloads' recipe
    (N(0,1), 4 channels per KV head scaled x20, one lognormal(0, 0.25) factor per
    token), for throughput rows whose full-size inputs would take long to draw
    on the host; the parity tests use the host generator."""
    import torch
    g = torch.Generator(device=dev).manual_seed(seed)
    x = torch.randn((T, hkv, d), generator=g, device=dev)
    ch = torch.stack([torch.randperm(d, generator=g, device=dev)[:4] for _ in range(hkv)])
    scale = torch.ones((hkv, d), device=dev)
    scale.scatter_(1, ch, 20.0)
    x = x * scale[None] * torch.exp(0.25 * torch.randn((T, 1, 1), generator=g, device=dev))
    return x.to(dtype or torch.bfloat16)


def _time_graph(fn, reps, warm=3, rounds=3):
    """Best per-call milliseconds of fn(i) captured reps times in one CUDA graph."""
    import torch
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e9
    for _ in range(rounds):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / reps)
    del g
    return best


def config_rows(tq, dev, peak):
    """Throughput of every workload at its stated size: encode Mtokens/s (one
    token = one position of one sequence, all its KV heads) and the decode step
    in GB/s of compressed cache read and as a fraction of HBM.  Caches that fit
    in L2 are rotated among copies until the working set exceeds 512 MB."""
    import torch
    rows = {}

    def rotated(make, nbytes):
        n = max(1, -(-512_000_000 // max(nbytes, 1)))
        return [make(i) for i in range(n)], n

    # --- tiny: 1 KV head, 1024 fp32 tokens, 4/4 ---
    w = W.WORKLOADS["tiny"]
    T = w.lens[0]
    K = torch.from_numpy(W.kv_tokens(w, 0, 0, 0, T)).to(dev)
    V = torch.from_numpy(W.kv_tokens(w, 1, 0, 0, T)).to(dev)
    bt = torch.from_numpy(W.block_table(w)).to(dev)
    sl = torch.from_numpy(W.slots(w, W.block_table(w), 0, 0, T)).to(dev)
    base = tq.Cache(w.num_blocks(), 1, 4, 4, 0, w.seed)
    enc_ms = _time_graph(lambda i: base.encode(K, V, sl), 20)
    nbytes = T * w.bytes_per_token_head()
    caches, n = rotated(lambda i: base if i == 0 else tq.Cache(w.num_blocks(), 1, 4, 4, 0, w.seed,
                                                              pool=base.pool.clone()), nbytes)
    q = torch.from_numpy(W.queries(w, 0)).to(dev)
    lens = torch.tensor([T], dtype=torch.int32, device=dev)
    out = torch.empty((1, 1, w.d), dtype=torch.float32, device=dev)
    wss = [c.new_workspace(1, 1, bt.shape[1]) for c in caches]
    dec_ms = _time_graph(lambda i: caches[i % n].decode(q, bt, lens, out=out, workspace=wss[i % n]), max(20, n))
    rows["tiny"] = {"encode_Mtok_s": round(T / (enc_ms * 1e-3) / 1e6, 2), "encode_us": round(enc_ms * 1e3, 2),
                    "decode_us": round(dec_ms * 1e3, 2), "decode_GBps": round(nbytes / (dec_ms * 1e-3) / 1e9, 1),
                    "decode_frac": round(nbytes / (dec_ms * 1e-3) / 1e9 / peak, 4), "decode_copies": n,
                    "note": "137 KB of cache per step: latency-bound by size"}
    del caches, wss, base
    # --- swa8x4096: 8 layers (as 8 sequences) x 20 heads, window 4096, 4/4 ---
    w = W.WORKLOADS["swa8x4096"]
    T, B = w.lens[0], w.batch
    btn = W.block_table(w)
    bt = torch.from_numpy(btn).to(dev)
    K = torch.cat([torch.from_numpy(W.kv_tokens(w, 0, b, 0, T)) for b in range(B)]).to(dev, torch.bfloat16)
    V = torch.cat([torch.from_numpy(W.kv_tokens(w, 1, b, 0, T)) for b in range(B)]).to(dev, torch.bfloat16)
    sl = torch.from_numpy(np.concatenate([W.slots(w, btn, b, 0, T) for b in range(B)])).to(dev)
    base = tq.Cache(w.num_blocks(), w.hkv, 4, 4, 0, w.seed)
    enc_ms = _time_graph(lambda i: base.encode(K, V, sl), 10)
    nbytes = B * T * w.hkv * w.bytes_per_token_head()
    caches, n = rotated(lambda i: base if i == 0 else tq.Cache(w.num_blocks(), w.hkv, 4, 4, 0, w.seed,
                                                              pool=base.pool.clone()), nbytes)
    q = torch.from_numpy(W.queries(w, 0)).to(dev, torch.bfloat16)
    lens = torch.tensor(w.lens, dtype=torch.int32, device=dev)
    out = torch.empty((B, w.hq, w.d), dtype=torch.float32, device=dev)
    wss = [c.new_workspace(B, w.hq, bt.shape[1]) for c in caches]
    dec_ms = _time_graph(lambda i: caches[i % n].decode(q, bt, lens, out=out, workspace=wss[i % n]), max(20, n))
    rows["swa8x4096"] = {"encode_Mtok_s": round(B * T / (enc_ms * 1e-3) / 1e6, 2), "encode_us": round(enc_ms * 1e3, 2),
                         "decode_us": round(dec_ms * 1e3, 2),
                         "decode_GBps": round(nbytes / (dec_ms * 1e-3) / 1e9, 1),
                         "decode_frac": round(nbytes / (dec_ms * 1e-3) / 1e9 / peak, 4), "decode_copies": n,
                         "step": "the 8 layers' windows in one decode launch (batch 8)"}
    del caches, wss, base, K, V
    torch.cuda.empty_cache()
    # --- long128k3: 4 x 131072 tokens, 3/3; prefill in 4096-token chunks, then the append + attend step ---
    w = W.WORKLOADS["long128k3"]
    T, B, C = w.lens[0], w.batch, w.prefill_chunk
    btn = W.block_table(w)
    bt = torch.from_numpy(btn).to(dev)
    cache = tq.Cache(w.num_blocks(), w.hkv, 3, 3, 0, w.seed)
    chunks = [(device_kv(dev, C, w.hkv, w.d, 10 + k), device_kv(dev, C, w.hkv, w.d, 20 + k)) for k in range(4)]
    slot_chunks = [torch.from_numpy(W.slots(w, btn, b, t0, t0 + C)).to(dev) for b in range(B) for t0 in range(0, T, C)]
    nch = len(slot_chunks)
    enc_ms = _time_graph(lambda i: cache.encode(chunks[i % 4][0], chunks[i % 4][1], slot_chunks[i % nch]), nch)
    kn = device_kv(dev, B, w.hkv, w.d, 30)
    vn = device_kv(dev, B, w.hkv, w.d, 31)
    q = device_kv(dev, B, w.hq, w.d, 32)
    lens = torch.full((B,), T + 1, dtype=torch.int32, device=dev)
    out = torch.empty((B, w.hq, w.d), dtype=torch.float32, device=dev)
    ws = cache.new_workspace(B, w.hq, bt.shape[1])
    nbytes = B * (T + 1) * w.hkv * w.bytes_per_token_head()
    step_ms = _time_graph(lambda i: cache.decode_append(kn, vn, q, bt, lens, out=out, workspace=ws), 20)
    dec_ms = _time_graph(lambda i: cache.decode(q, bt, lens, out=out, workspace=ws), 20)
    rows["long128k3"] = {"prefill_encode_Mtok_s": round(C / (enc_ms * 1e-3) / 1e6, 2),
                         "prefill_chunk_us": round(enc_ms * 1e3, 2),
                         "step_us": round(step_ms * 1e3, 2), "step_GBps": round(nbytes / (step_ms * 1e-3) / 1e9, 1),
                         "step_frac": round(nbytes / (step_ms * 1e-3) / 1e9 / peak, 4),
                         "decode_us": round(dec_ms * 1e3, 2),
                         "decode_GBps": round(nbytes / (dec_ms * 1e-3) / 1e9, 1),
                         "decode_frac": round(nbytes / (dec_ms * 1e-3) / 1e9 / peak, 4),
                         "cache_MB": round(nbytes / 1e6, 1),
                         "step": "append 1 token per sequence + attend 64 query heads over 131073 tokens, one launch",
                         "data": "K/V/q drawn on the device with the workloads' recipe"}
    del cache, chunks, slot_chunks, ws
    torch.cuda.empty_cache()
    # --- qjl64: 64 sequences of U[1K, 16K] tokens, 2-bit keys + QJL (m = 128), 2-bit values ---
    w = W.WORKLOADS["qjl64"]
    B = w.batch
    btn = W.block_table(w)
    bt = torch.from_numpy(btn).to(dev)
    cache = tq.Cache(w.num_blocks(), w.hkv, 2, 2, 128, w.seed)
    tot = sum(w.lens)
    Kall = device_kv(dev, tot, w.hkv, w.d, 40)
    Vall = device_kv(dev, tot, w.hkv, w.d, 41)
    sl = torch.from_numpy(np.concatenate([W.slots(w, btn, b, 0, w.lens[b]) for b in range(B)])).to(dev)
    enc_ms = _time_graph(lambda i: cache.encode(Kall, Vall, sl), 5)
    kn = device_kv(dev, B, w.hkv, w.d, 42)
    vn = device_kv(dev, B, w.hkv, w.d, 43)
    q = device_kv(dev, B, w.hq, w.d, 44)
    lens_np = np.array(w.lens, dtype=np.int64) + 1
    lens = torch.from_numpy(lens_np.astype(np.int32)).to(dev)
    out = torch.empty((B, w.hq, w.d), dtype=torch.float32, device=dev)
    ws = cache.new_workspace(B, w.hq, bt.shape[1])
    nbytes = int(lens_np.sum()) * w.hkv * w.bytes_per_token_head()

    step_ms = _time_graph(lambda i: cache.decode_append(kn, vn, q, bt, lens, out=out, workspace=ws), 20)
    dec_ms = _time_graph(lambda i: cache.decode(q, bt, lens, out=out, workspace=ws), 20)
    rows["qjl64"] = {"prefill_encode_Mtok_s": round(tot / (enc_ms * 1e-3) / 1e6, 2),
                     "step_us": round(step_ms * 1e3, 2), "step_GBps": round(nbytes / (step_ms * 1e-3) / 1e9, 1),
                     "step_frac": round(nbytes / (step_ms * 1e-3) / 1e9 / peak, 4),
                     "decode_us": round(dec_ms * 1e3, 2),
                     "decode_GBps": round(nbytes / (dec_ms * 1e-3) / 1e9, 1),
                     "decode_frac": round(nbytes / (dec_ms * 1e-3) / 1e9 / peak, 4),
                     "cache_MB": round(nbytes / 1e6, 1), "launches_per_step": 1,
                     "step": "append 1 token per sequence (codes, QJL sign row) + attend 32 query heads, one launch",
                     "data": "K/V/q drawn on the device with the workloads' recipe"}
    del cache, Kall, Vall, ws
    torch.cuda.empty_cache()
    return rows


# --------------------------------------------------------------------------- oracle (CPU)
CPU_SAMPLE_TOKENS = 32768  # cpu_baseline: steps over the whole 32768-token context
CPU_SAMPLE_SECONDS = 8.0   # ... repeated until about this much CPU time has been measured
REF_SAMPLE_TOKENS = 1024   # reference arm: each step over a 1024-token window (a fraction of a second)


def _oracle_sample(w, n_tokens):
    """Oracle cache holding the first n_tokens of the workload's context, built
    outside any timed region."""
    import oracle
    threads = oracle.set_threads(len(os.sched_getaffinity(0)))
    bt = W.block_table(w)
    oc = oracle.Cache(w.d, w.key_bits, w.value_bits, w.qjl_m, w.block_size, w.hkv, w.num_blocks(), w.seed)
    pool = oc.new_pool()
    oc.encode(W.kv_tokens(w, 0, 0, 0, n_tokens), W.kv_tokens(w, 1, 0, 0, n_tokens),
              W.slots(w, bt, 0, 0, n_tokens), pool)
    return oc, pool, bt, threads


def _oracle_step(w, oc, pool, bt, n_tokens):
    """The step on the oracle: append token n_tokens-1, attend all 64 query heads over n_tokens."""
    t = n_tokens
    oc.encode(W.kv_tokens(w, 0, 0, t - 1, t), W.kv_tokens(w, 1, 0, t - 1, t), W.slots(w, bt, 0, t - 1, t), pool)
    q = W.queries(w, 0).astype(np.float64)
    out, _ = oc.decode(pool, q, bt, np.array([t], dtype=np.int32), W.sm_scale(w))
    return out


def cpu_baseline(w):
    n = CPU_SAMPLE_TOKENS
    oc, pool, bt, threads = _oracle_sample(w, n)
    steps = 0
    t = time.perf_counter()
    while True:
        _oracle_step(w, oc, pool, bt, n)
        steps += 1
        dt = time.perf_counter() - t
        if dt >= CPU_SAMPLE_SECONDS or steps >= 16:
            break
    nbytes = steps * n * w.hkv * w.bytes_per_token_head()
    return {"value": round(nbytes / dt / 1e9, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} steps (append 1 token, attend 64 query heads over all {n} context tokens), "
                      "float64 oracle; its cache pre-encoded by the oracle outside the timing",
            "seconds": round(dt, 3)}


def run_reference(args, rank, world):
    if rank != 0:
        return  # the oracle arm runs on rank 0 only
    w = W.WORKLOADS[WORKLOAD]
    n = REF_SAMPLE_TOKENS
    oc, pool, bt, threads = _oracle_sample(w, n)
    for _ in range(args.warmup):
        _oracle_step(w, oc, pool, bt, n)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(w, oc, pool, bt, n)
    dt = (time.perf_counter() - t) / args.steps
    nbytes = n * w.hkv * w.bytes_per_token_head()
    v = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": "gqa32k: 64 query / 8 KV heads, head_dim 128, 32768-token context, batch 1, "
                               "4-bit keys and values, 16-token pages in a permuted block table",
                   "step": f"oracle: encode 1 new token + decode attention for 64 query heads over a "
                           f"{n}-token window of the context (bytes counted for that window)"},
        "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: append + decode over the first {n} context tokens, float64 oracle"},
        "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-widths", action="store_true", help="skip the other-widths measurements")
    ap.add_argument("--profile", action="store_true",
                    help="only build the caches and launch the decode kernel 6 times (for ncu)")
    ap.add_argument("--profile-prefill", action="store_true",
                    help="only build the cache and launch the 64-position chunked prefill 4 times (for ncu)")
    ap.add_argument("--profile-octopus", action="store_true",
                    help="only build an OCTOPUS 4/4 cache and launch its decode 6 times (for ncu)")
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
