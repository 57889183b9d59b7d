// Decode attention with the score contraction on the Blackwell tensor cores
// (tcgen05), for 4-bit keys without the QJL sketch and value codes of 1..4
// bits.
//
// Grid (split, KV head, sequence), one CTA per SM, two warpgroups of four
// warps.  A warpgroup takes tiles of 8 pages (128 tokens) of its split,
// tiles wg, wg + 2, ...; warp q of it owns pages 2q and 2q + 1 of a tile and
// streams them into its own ring of shared-memory slots with bulk async copies.
// Per tile:
//  scores  Each lane unpacks the 4-bit key codes of its part of the warp's two
//          pages through the lane-private table into the two-level centroid
//          operand C[c] = delta (N[c] + rem2[c] / delta) -- N[c] an integer of
//          magnitude <= 2047 and |rem2 / delta| <= 1/2, both exact enough in
//          fp16 -- and writes it to tensor memory (the warpgroup's 128 lanes =
//          the tile's 128 tokens, 64 columns for N and 64 for rem2 / delta).
//          One thread then issues the contraction with the query operand in
//          shared memory, x = sm_scale log2(e) delta q_rot / qscale split into
//          fp16 hi (rows 0..7) and lo (rows 8..15): 16 kind::f16 MMAs of
//          M = 128, N = 16, K = 16 into a 16-column fp32 accumulator, whose
//          completion is signalled on an mbarrier.  The scores come back with
//          the 16-lane x 256-bit load, which leaves them in the accumulator
//          layout of mma.sync m16n8 (token rows, query columns).
//  softmax and values as the mma.sync decode kernel: lazy running max,
//          O^T += Vcode^T (p * scale)^T on mma.sync, value codes as exact fp16
//          subnormals.
// The MMA of tile t + 1 runs while the warps do the softmax and values of
// tile t.  Warps merge in shared memory and the splits of a sequence are
// merged by the last CTA to finish, as in the mma.sync kernel.
// Logits and values stay in the rotated frame; keys are never reconstructed
// ["OCTOPUS ..." -- TL;DR / step 7; deep dive -- [RHT effect]]; attention is
// softmax(q K^T / sqrt(d_h)) V [Bit-Axon -- attention under quantized KV].
#pragma once
#include <cuda_runtime.h>

#include "tq_decode_impl.cuh"
#include "tq_tcgen05.cuh"

namespace tq {

constexpr int kTcWarps = 8;               // two warpgroups of four warps
constexpr int kTcGroups = kTcWarps / 4;
constexpr int kTcMaxSlots = 8;            // ring slots per warp: up to four tiles of two pages
constexpr int kTcTmemCols = 512;          // per warpgroup: key operand (128) + scores (16), 256 apart
constexpr int kTcBq = 16 * kHeadDim * 2;  // query operand: 16 rows x 128 dims in fp16
constexpr uint32_t kTcLbo = 128;          // core matrices adjacent along K
constexpr uint32_t kTcSbo = kHeadDim / 8 * 128;  // the next 8 rows of the query operand

// Column c (0..63) of the key operand holds code byte tc_byte(c) of each token's
// key row (dims 2 tc_byte(c), 2 tc_byte(c) + 1): the order in which the
// 16-lane x 256-bit stores leave the 16 code bytes 16 qd .. 16 qd + 15 a lane
// with quad index qd unpacks.  Columns 64 + c hold the remainders of the same
// dims; the query operand uses the same order along K.
__host__ __device__ constexpr int tc_byte(int c) { return 16 * ((c & 7) >> 1) + 2 * (c >> 3) + (c & 1); }

struct TcLayout {
    int bq, qrot, qscale, tab, stage, bars, mbar, ok, taddr, ringA, nwA, spw, total;
};

// Shared memory: small fixed region, then ring slots of the first nwA warps
// below the lane-private table at kLutAddr and of the others above it; as many
// slots per warp (at most kTcMaxSlots) as fit.
template <int VB>
__host__ __device__ constexpr TcLayout tc_layout() {
    TcLayout L{};
    int off = 0;
    L.bq = off; off += kTcBq;
    L.qrot = off; off += 8 * kQStride * 4;
    L.qscale = off; off += 8 * 4;
    L.tab = off; off += 2 * 16 * 2;                // N and rem2 / delta in binary16
    L.stage = off; off += kStageBytes;             // appended token (see kStage*)
    L.bars = off; off += 8 * kTcWarps * kTcMaxSlots;
    L.mbar = off; off += 8 * kTcGroups;
    L.ok = off; off += 4 * kTcWarps * kTcMaxSlots;
    L.taddr = off; off += 16;
    L.ringA = (off + 127) / 128 * 128;
    const int capA = (int)kLutAddr - kMaxSmemBase - L.ringA;
    for (int spw = kTcMaxSlots; spw >= 1; --spw) {
        const int per = spw * PageFmt<4, VB, 0>::stride;
        const int nA = capA / per < kTcWarps ? capA / per : kTcWarps;
        const int total = (int)kLutAddr + kLutBytes + (kTcWarps - nA) * per;
        const int merge_end = (int)kLutAddr + 2048 + kTcWarps * 8 * kHeadDim * 4;
        const int need = total > merge_end ? total : merge_end;
        if (need <= kSmemLimit) {
            L.spw = spw;
            L.nwA = nA;
            L.total = need;
            return L;
        }
    }
    return L;  // spw == 0: does not fit
}

// Whether the tensor-core decode is built for this page format.
__host__ __device__ constexpr bool tc_decode_fits(int kb, int vb, int m) {
    return kb == 4 && m == 0 && vb >= 1 && vb <= 4;
}

template <int VB>
__global__ void __launch_bounds__(kTcWarps * 32, 1) decode_tc_kernel(const DecodeArgs a) {
    using F = PageFmt<4, VB, 0>;
    constexpr int NW = kTcWarps, NT = NW * 32, D = kHeadDim, KROW = D * 4 / 8;
    constexpr TcLayout LY = tc_layout<VB>();
    constexpr int SPW = LY.spw;
    static_assert(SPW >= 6, "the tensor-core decode needs two tiles in use and one ahead per warp");
    static_assert(LY.bq % 16 == 0, "the query operand must be 16-byte aligned");
    extern __shared__ __align__(128) uint8_t sm[];
    const Geometry& g = a.g;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wg = warp >> 2, wq = warp & 3;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = a.group;

    // The layout assumes dynamic shared memory starts below kMaxSmemBase (the
    // same start for every CTA: all return here or none does).
    const uint32_t sbase = smem_u32(sm);
    if (sbase > (uint32_t)kMaxSmemBase) {
        grid_dependency_wait();
        if (tid == 0) flag(a.status, TQ_FLAG_INTERNAL);
        return;
    }
    const int lut_off = (int)kLutAddr - (int)sbase;
    const uint32_t ring_w = (warp < LY.nwA) ? sbase + LY.ringA + warp * SPW * F::stride
                                           : kLutAddr + kLutBytes + (warp - LY.nwA) * SPW * F::stride;
    const uint32_t bar_w = sbase + LY.bars + 8 * warp * kTcMaxSlots;
    const uint32_t mbar = sbase + LY.mbar + 8 * wg;
    const uint32_t stage_bar = sbase + LY.stage + kStageBar;
    const uint32_t never_bar = sbase + LY.stage + kStageNever;
    int* slot_ok = reinterpret_cast<int*>(sm + LY.ok) + warp * kTcMaxSlots;
    float* qrot = reinterpret_cast<float*>(sm + LY.qrot);
    float* qscale = reinterpret_cast<float*>(sm + LY.qscale);
    const int p0 = split * a.pages_per_split;
    const float ksc = a.sm_scale_log2;

    // ---- shared-memory-only setup: barriers, tensor memory, lane-private table ----
    if (lane == 0) {
        for (int k = 0; k < SPW; ++k) mbar_init(bar_w + 8 * k, 1);
        if (warp == 0) {
            mbar_init(stage_bar, 1);
            mbar_init(never_bar, 1);
            for (int k = 0; k < kTcGroups; ++k) mbar_init(sbase + LY.mbar + 8 * k, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc<kTcTmemCols>(sbase + LY.taddr);
    uint16_t* tab = reinterpret_cast<uint16_t*>(sm + LY.tab);
    if (tid < 16) tab[tid] = a.c.cint_f16[tid];
    else if (tid < 32) tab[tid] = a.c.cremd_f16[tid - 16];
    __syncthreads();
    {
        // byte e (codes e & 15, e >> 4) -> (N[e & 15], N[e >> 4]), (rem2/delta[e & 15], rem2/delta[e >> 4]),
        // 8 bytes for each lane at entry * 256 + lane * 8
        uint8_t* lut = sm + lut_off;
        for (int i = tid; i < 256 * 16; i += NT) {
            const int e = i >> 4, k = i & 15;
            const uint32_t xx = (uint32_t)tab[e & 15] | ((uint32_t)tab[e >> 4] << 16);
            const uint32_t yy = (uint32_t)tab[16 + (e & 15)] | ((uint32_t)tab[16 + (e >> 4)] << 16);
            *reinterpret_cast<uint4*>(lut + e * 256 + 16 * k) = make_uint4(xx, yy, xx, yy);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + LY.taddr);
    const uint32_t tA = tmem + (uint32_t)(wg * 256);  // this warpgroup's key operand (128 columns)
    const uint32_t tD = tA + 128;                     // its scores (16 columns)
    const uint32_t tl = (uint32_t)(wq * 32) << 16;    // this warp's 32 lanes
    // Launched as a programmatic dependent of the previous kernel in the stream:
    // nothing in global memory is touched before that grid has completed.
    grid_dependency_wait();
    grid_launch_dependents();

    // ---- sequence range of this split ----
    int len = __ldg(a.lens + b);
    if (len < 0) len = 0;
    int pos_new = len - 1;  // slot of the appended token
    if (a.window > 0) {
        if (len > 0) pos_new = (len - 1) % a.window;
        if (len > a.window) len = a.window;
    }
    if (len > a.max_blocks * g.bs) {
        if (tid == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
        len = a.max_blocks * g.bs;
    }
    int npages = (len + kBlockSize - 1) / kBlockSize - p0;
    if (npages > a.pages_per_split) npages = a.pages_per_split;
    if (npages < 0) npages = 0;
    const int ntiles = (npages + 7) >> 3;
    const int nt = ntiles > wg ? (ntiles - wg + kTcGroups - 1) / kTcGroups : 0;  // this warpgroup's tiles
    const int njw = 2 * nt;  // warp-local pages j = 2 t + e of tile t
    // split-local page of warp-local page j; pages at or past npages are not loaded
    auto page_of = [&](int j) { return 8 * (wg + kTcGroups * (j >> 1)) + 2 * wq + (j & 1); };
    auto valid = [&](int j) { return page_of(j) < npages; };
    const int32_t* btr = a.block_table + (int64_t)b * a.bt_stride + p0;
    // lane l: block id of warp-local page l of the current batch of 32 and of the next
    int bid_cur = (lane < njw && valid(lane)) ? __ldg(btr + page_of(lane)) : -1;
    int bid_nxt = (32 + lane < njw && valid(32 + lane)) ? __ldg(btr + page_of(32 + lane)) : -1;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < G) load4(a.q, a.dtype, ((int64_t)b * a.hq + (int64_t)h * G + warp) * D + 4 * lane, x);

    auto issue = [&](int j, int blk) {
        const int slot = j % SPW;
        const bool ok = blk >= 0 && blk < g.num_blocks;
        const uint32_t bar = bar_w + 8 * slot;
        slot_ok[slot] = ok;
        if (ok) {
            mbar_arrive_tx(bar, (uint32_t)F::bytes);
            bulk_g2s(ring_w + slot * F::stride, a.pool + ((int64_t)blk * g.hkv + h) * F::bytes, (uint32_t)F::bytes,
                     bar);
        } else {
            flag(a.status, TQ_FLAG_BAD_SLOT);
            mbar_arrive(bar);
        }
    };
    // The appended token lies in page pos_new / 16 of the sequence; the warp that
    // owns that page encodes it (after the query is prepared; its inputs are
    // requested now and waited on only when used), writes it to the pool and
    // patches its own shared-memory copy of the page before unpacking it.
    int jnew = -1;
    int blknew = -1;
    const int offnew = pos_new & (kBlockSize - 1);
    uint32_t kraw[4] = {0u, 0u, 0u, 0u}, vraw[4] = {0u, 0u, 0u, 0u};
    if (a.knew != nullptr && len > 0) {
        const int pi = pos_new / kBlockSize - p0;
        if (pi >= 0 && pi < npages) {
            const int T = pi >> 3;
            if (warp == 4 * (T % kTcGroups) + ((pi & 7) >> 1)) {
                jnew = 2 * (T / kTcGroups) + (pi & 1);
                const int64_t e = ((int64_t)b * g.hkv + h) * D + 4 * lane;
                raw4(a.knew, a.kv_dtype, e, kraw);
                raw4(a.vnew, a.kv_dtype, e, vraw);
                blknew = __ldg(btr + pi);
            }
        }
    }
    // the first tile's two pages now, the rest of the ring once the query is prepared
    if (lane < 2 && lane < njw && valid(lane)) issue(lane, bid_cur);

    bool timed_out = false;
    float m0 = kMinusBig, m1 = kMinusBig, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    // ---- q_rot = R q for query (warp) of this group; qscale = power of two putting
    //      max |ksc delta q_rot| / qscale in (256, 512] ----
    {
        if (warp < G) {
            apply_signs(x, lane_signs(a.c, lane));
            fwht128(x, lane);
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] *= 0.08838834764831845f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) qrot[warp * kQStride + 4 * lane + i] = x[i];
        const float mx = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
        const float big = fabsf(a.c.delta) * ksc * mx;
        const float scl = (big > 0.f) ? exp2f(ceilf(log2f(big / 512.f))) : 1.f;
        if (lane == 0) qscale[warp] = scl;
    }
    __syncthreads();
    // ---- the query operand, written once: row n (< 8 the fp16 hi part, >= 8 the lo
    //      part of x = ksc delta q_rot / qscale of query n % 8), K index 2c, 2c + 1 =
    //      dims 2 tc_byte(c), 2 tc_byte(c) + 1, in the K-major core-matrix layout ----
    for (int i = tid; i < 16 * 64; i += NT) {
        const int n = i >> 6, c = i & 63, gq = n & 7, byte = tc_byte(c);
        const float e = ksc * a.c.delta / qscale[gq];
        const float x0 = e * qrot[gq * kQStride + 2 * byte], x1 = e * qrot[gq * kQStride + 2 * byte + 1];
        uint32_t v = pack_h2(x0, x1);
        if (n >= 8) {
            const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&v));
            v = pack_h2(x0 - hf.x, x1 - hf.y);
        }
        *reinterpret_cast<uint32_t*>(sm + LY.bq + (n >> 3) * kTcSbo + (c >> 2) * kTcLbo + (n & 7) * 16 + (c & 3) * 4) = v;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
    __syncthreads();
    if (lane >= 2 && lane < SPW && lane < njw && valid(lane)) issue(lane, bid_cur);
    if (jnew >= 0) {
        // a bad block id leaves the pool alone; this warp's copy of that page is
        // flagged and skipped, so what it patches in is never used
        if (blknew >= 0 && blknew < g.num_blocks) {
            uint8_t* page = const_cast<uint8_t*>(a.pool) + ((int64_t)blknew * g.hkv + h) * F::bytes;
            append_token<4, VB, 0>(a, page, offnew, sm + LY.stage, lane, kraw, vraw);
        }
        if (lane == 0) mbar_arrive(stage_bar);
    }

    const int r = lane >> 2, qd = lane & 3;
    // score row r of a page holds slot tr (and row r + 8 slot tr + 8), so that the
    // value loads of the mma.sync contraction avoid bank conflicts
    const int tr = r ^ ((r >> 1) & 1);
    const int ta = (2 * qd) ^ (qd & 1), tb = (2 * qd + 1) ^ (qd & 1);
    const uint32_t lw = kLutAddr | ((uint32_t)lane << 3);
    const float qs0 = qscale[2 * qd], qs1 = qscale[2 * qd + 1];
    constexpr uint32_t idesc = tc::idesc_f16_f32(128, 16);

    int issued = njw < SPW ? njw : SPW;  // warp-local pages whose copies may have started: j < issued
    int jfail = njw;                      // first page not waited for after a wait gave up
    if (a.stall_cycles > 0 && (split & 1) && warp == 0) {
        // test hook: a bounded wait on a barrier that nothing arrives on runs out
        if (!mbar_wait_for(never_bar, 0, a.stall_cycles)) {
            timed_out = true;
            jfail = 0;
        }
    }
    auto wait_page = [&](int j) {
        if (timed_out || !valid(j)) return;
        if (!mbar_wait(bar_w + 8 * (j % SPW), (uint32_t)((j / SPW) & 1))) {
            timed_out = true;
            jfail = j;
        }
    };
    // keys of warp-local page j into lanes 16 e .. 16 e + 15 of this warp's block
    auto unpack = [&](int j, int e) {
        const uint32_t pg = ring_w + (j % SPW) * F::stride;
        if (j == jnew && !timed_out) {
            if (!mbar_wait(stage_bar, 0)) {
                timed_out = true;
                if (jfail > j) jfail = j;
            } else {
                patch_page<4, VB, 0>(sm + (pg - sbase), offnew, sm + LY.stage, lane);
                // the slot is refilled later by a bulk copy: order these generic
                // writes before that async-proxy write
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
        }
        const uint32_t ka = pg + F::kcode + tr * KROW + qd * 16;
        const uint4 va = lds128(ka), vb = lds128(ka + 8 * KROW);
        const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
        uint32_t NR[32], RR[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint2 a0 = key_lut4(wa, lw, 2 * k), a1 = key_lut4(wa, lw, 2 * k + 1);
            const uint2 b0 = key_lut4(wb, lw, 2 * k), b1 = key_lut4(wb, lw, 2 * k + 1);
            NR[4 * k] = a0.x; NR[4 * k + 1] = a1.x; NR[4 * k + 2] = b0.x; NR[4 * k + 3] = b1.x;
            RR[4 * k] = a0.y; RR[4 * k + 1] = a1.y; RR[4 * k + 2] = b0.y; RR[4 * k + 3] = b1.y;
        }
        const uint32_t dst = tA + tl + ((uint32_t)(16 * e) << 16);
        tc::st_16x256b_x8(dst, NR);
        tc::st_16x256b_x8(dst + 64, RR);
    };
    // all four warps' keys are in tensor memory: one thread issues the tile's MMAs
    auto mma_tile = [&]() {
        tc::wait_st();
        tc::fence_before_sync();
        asm volatile("bar.sync %0, 128;" ::"r"(1 + wg) : "memory");
        if (wq == 0 && lane == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma_f16_ts(tD, tA + 8 * s, tc::smem_desc(sbase + LY.bq + 256 * s, kTcLbo, kTcSbo), idesc,
                               s > 0 ? 1u : 0u);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                tc::mma_f16_ts(tD, tA + 64 + 8 * s, tc::smem_desc(sbase + LY.bq + 256 * s, kTcLbo, kTcSbo), idesc, 1u);
            tc::commit(mbar);
        }
    };
    float S[2][8];
    auto load_scores = [&](int t) {
        if (!mbar_wait(mbar, (uint32_t)(t & 1))) {
            if (!timed_out) jfail = 2 * t;
            timed_out = true;
        }
        tc::fence_after_sync();
        uint32_t f0[8], f1[8];
        tc::ld_16x256b_x2(tD + tl, f0);
        tc::ld_16x256b_x2(tD + tl + (16u << 16), f1);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            S[0][i] = __uint_as_float(f0[i]);
            S[1][i] = __uint_as_float(f1[i]);
        }
    };

    if (nt > 0) {
        wait_page(0);
        wait_page(1);
        unpack(0, 0);
        unpack(1, 1);
        mma_tile();
        load_scores(0);
    }
    for (int t = 0; t < nt; ++t) {
        const bool more = t + 1 < nt;
        if (more) {
            const int j0 = 2 * t + 2;
            wait_page(j0);
            wait_page(j0 + 1);
            unpack(j0, 0);
            unpack(j0 + 1, 1);
            mma_tile();
        }
        // softmax and values of pages 2t, 2t + 1 while the next tile's MMAs run
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 2 * t + e;
            if (valid(j) && !timed_out) {
                const float t0 = qs0 * (S[e][0] + S[e][4]), t1 = qs1 * (S[e][1] + S[e][5]);
                const float t2 = qs0 * (S[e][2] + S[e][6]), t3 = qs1 * (S[e][3] + S[e][7]);
                softmax_pv_page<4, VB, 0>(ring_w + (j % SPW) * F::stride, slot_ok[j % SPW] != 0,
                                          (p0 + page_of(j)) * kBlockSize, len, t0, t1, t2, t3, r, tr, ta, tb, m0,
                                          m1, l0, l1, z0, z1, acc);
            }
        }
        __syncwarp();  // every lane has read both slots: refill them with the pages SPW ahead
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int jn = 2 * t + e + SPW;
            if (jn < njw) {
                if ((jn & 31) == 0) {  // next batch of block ids; prefetch the one after it
                    bid_cur = bid_nxt;
                    const int jj = jn + 32 + lane;
                    bid_nxt = (jj < njw && valid(jj)) ? __ldg(btr + page_of(jj)) : -1;
                }
                if (valid(jn) && !timed_out) {
                    if (lane == (jn & 31)) issue(jn, bid_cur);
                    issued = jn + 1;
                }
            }
        }
        if (more) load_scores(t + 1);
    }
    if (timed_out) {
        // copies this warp started must land before its shared memory goes away;
        // one shared deadline for all of them
        const long long c0 = clock64();
        for (int jj = jfail; jj < issued; ++jj) {
            if (!valid(jj)) continue;
            const uint32_t bar = bar_w + 8 * (jj % SPW);
            while (!mbar_try(bar, (uint32_t)((jj / SPW) & 1)) && clock64() - c0 < kWaitCycles) {
            }
        }
    }
    decode_epilogue<NW, VB, kTcTmemCols>(a, sm, lut_off, timed_out, split, h, b, m0, m1, l0, l1, z0, z1, acc, tmem);
}

template <int VB>
static int launch_decode_tc_t(const DecodeArgs& a, cudaStream_t s) {
    using F = PageFmt<4, VB, 0>;
    const Geometry& g = a.g;
    if (g.page_bytes != F::bytes || g.vcode_off != F::vcode || g.gam_off != F::gam || g.scl_off != F::scl ||
        g.zer_off != F::zer || g.bs != kBlockSize || g.d != kHeadDim || g.m != 0)
        return (int)cudaErrorInvalidValue;  // the cache's geometry is not the format this kernel was built for
    constexpr TcLayout L = tc_layout<VB>();
    auto kern = decode_tc_kernel<VB>;
    static int done[64] = {};
    cudaError_t e = ensure_smem_limit(kern, L.total, done);
    if (e != cudaSuccess) return (int)e;
    return (int)launch_programmatic(kern, dim3((unsigned)a.num_splits, (unsigned)g.hkv, (unsigned)a.batch),
                                    dim3(kTcWarps * 32), (size_t)L.total, s, a);
}

}  // namespace tq
