// Chunked-prefill attention on the tcgen05 tensor cores: C consecutive query
// positions of one sequence attend causally over its compressed cache, for
// 4-bit keys without the QJL sketch and value codes of 1..4 bits.
//
// A chunk gives every KV head C x G query rows; they are far more than the
// decode's 8, so scores and values are dense contractions and each page is
// unpacked once for all of them.  Grid (split, row block, KV head): a CTA
// takes 128 query rows (row r = position index * G + query in group) and the
// 128-token tiles of its split of the token range (tiles past the block's last
// position are skipped).  Its 15 warps:
//   warps 0-7  softmax, two warps per query row: thread = (column half, query
//              row = tensor-memory lane).  Before the tiles the pair rotates
//              its query (q_rot = R q: each half takes 64 dimensions through
//              the butterflies that stay inside them, the last stage through
//              shared memory) and stores x = sm_scale log2(e) delta q_rot /
//              qscale in fp16 hi and lo parts as the tensor-memory A operand.
//              Per tile each half reads its 64 score columns, applies the key
//              norms, the causal mask and a lazy running max (the two halves'
//              tile maxima are exchanged; the max is raised only when a score
//              beats it by more than 8 in log2 units, so p <= 2^8; a tile with
//              a value scale above 255 takes the exact max; a raise rescales
//              the half's 64 output columns), and writes the weights
//              p * scale in fp16 hi and lo parts over its scores as the A
//              operand of PV.  The two halves' sums meet at the end.
//   warps 8-11 key producers: thread = token of the tile.  They unpack the
//              key codes through a 256-entry table into the two-level centroid
//              operand C[c] / delta = N[c] + rem2[c] / delta (N an integer of
//              magnitude <= 2047, |rem2 / delta| <= 1/2, both exact enough in
//              fp16).
//   warps 13-14 value producers: thread = two tokens of the tile.  They unpack
//              the value codes into exact fp16 subnormals, and the norms,
//              scales, zero points and masks into shared memory.
//   warp 12    lane 0 loads the pages (bulk async copies into a four-tile
//              ring) and issues the MMAs: scores S [128 rows x 128 tokens] =
//              q_hi . N + q_lo . N + q_hi . rem2/delta (24 kind::f16 MMAs,
//              K = 16), and O [128 rows x 128 dims] += w_hi . V + w_lo . V (16
//              MMAs) in fp32 tensor memory, each group committed to an
//              mbarrier.  Right after the softmax of tile u it issues PV of
//              tile u, starts the copies of tile u + 4 and the scores of tile
//              u + 2.
// Scores and weights of a tile share tensor-memory columns (the weights
// overwrite the scores the softmax has read), two tiles deep, and the value
// operand is double-buffered: the scores of tile u + 1 run on the tensor cores
// while the softmax works on tile u, and the values of tile u + 1 are unpacked
// before PV of tile u has read its operand.
// Logits and values stay in the rotated frame; keys are never reconstructed
// ["OCTOPUS ..." -- TL;DR / step 7; deep dive -- [RHT effect]].  Each split
// writes its rows' partial (max, sum, unnormalised rotated accumulator with
// the zero-point term) and a second kernel merges the splits and applies the
// one inverse rotation R^T = diag(s) H / sqrt(d) per output.  The chunk's own
// keys and values are in the cache before attention reads it [TurboQuant deep
// dive -- attention forward with kv_cache.update].
#include <cuda_runtime.h>

#include "tq_decode_impl.cuh"
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

constexpr int kPfRows = 128;                    // query rows per CTA (tensor-memory lanes)
constexpr int kPfTile = 128;                    // tokens per tile
constexpr int kPfPages = kPfTile / kBlockSize;  // pages per tile
constexpr int kPfWarps = 15;                    // softmax 0-7 (two per row), key producers 8-11, issuer 12, value producers 13-14
constexpr int kPfSoftmax = 256;                 // softmax threads (named barrier 1)
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPartRow = 4 + kHeadDim;          // partial record: max, sum, 2 pad, acc[128]
// tensor-memory columns: query operand (hi 0..63, lo 64..127); scores of tile
// u at kTs + 128 (u & 1), overwritten first by its logits and then by its
// weights (for the 16 tokens of K-step s: hi parts at +16 s .. +16 s + 7, lo
// parts at +16 s + 8 .. +16 s + 15); output accumulator
constexpr uint32_t kTq = 0, kTs = 128, kTo = 384;
constexpr int kTmemCols = 512;
constexpr int kRing = 4;                        // tiles of pages in flight
// key operand [N = 128 tokens x K = 128 dims], K-major core matrices
constexpr uint32_t kKLbo = 128, kKSbo = 2048;
// value operand [K = 128 tokens x N = 128 dims], MN-major core matrices (8
// tokens x 8 dims, dims contiguous): 8-token groups 128 bytes apart, 8-dim
// groups 2048 apart.  The descriptor's leading byte offset is the step along K
// and its stride byte offset the step along N, as in the K-major layout (the
// self-test checks this reading).
constexpr uint32_t kVLbo = 128, kVSbo = 2048;
// barriers: page slots [kRing][8], then key operand full, value operand full
// [2], scores full [2], weights full [2], values multiplied [2] (all four by
// tile parity), query operand stored, and one that nothing arrives on (the
// wait-timeout test hook waits on it)
constexpr int kBarBk = kRing * kPfPages, kBarBv = kBarBk + 1, kBarS = kBarBv + 2, kBarP = kBarS + 2,
              kBarO = kBarP + 2, kBarQ = kBarO + 2, kBarNever = kBarQ + 1, kNumBars = kBarNever + 1;
// The output takes 2^24 back: the value codes are held as fp16 subnormals.
constexpr float kOutScale = 16777216.f;

template <int VB>
struct PfLayout {
    static constexpr int bn = 0;                        // key operand, integer parts
    static constexpr int br = bn + kPfTile * kHeadDim * 2;   // key operand, remainders / delta
    static constexpr int bv = br + kPfTile * kHeadDim * 2;   // value operand [2] (by tile parity)
    static constexpr int bv_size = kPfTile * kHeadDim * 2;
    static constexpr int ring = bv + 2 * bv_size;
    static constexpr int stride = PageFmt<4, VB, 0>::stride;
    // per token of a tile: gamma and the mask (0, or -inf for a token that is
    // not there) four tiles deep (by u & 3: the scores of tile u + 1 may finish
    // while the softmax still reads tile u - 1's), scale and zero two deep
    static constexpr int gam = ring + kRing * kPfPages * stride;
    static constexpr int msk = gam + 4 * kPfTile * 4;
    static constexpr int scl = msk + 4 * kPfTile * 4;
    static constexpr int zer = scl + 2 * kPfTile * 4;
    static constexpr int big = zer + 2 * kPfTile * 4;   // per tile parity and value producer warp: a scale > kBigScale
    static constexpr int inv = big + 2 * 4 * 4;         // per tile (u & 3) and value producer warp: a token not there
    static constexpr int xch = inv + 4 * 4 * 4;         // softmax pair exchange: [2][2][128] floats x 2
    static constexpr int lut = xch + 4 * 2 * kPfRows * 4;   // 256 entries x (N pair, rem2/delta pair)
    static constexpr int bars = lut + 256 * 8;
    static constexpr int ok = bars + 8 * kNumBars;      // page copy issued and its block id valid [kRing][8]
    static constexpr int taddr = ok + 4 * kRing * kPfPages;
    static constexpr int total = taddr + 16;
};

// element (token t, dims 8 dg .. 8 dg + 7) chunk of the key operand
__device__ __forceinline__ uint32_t key_chunk(int t, int dg) {
    return (uint32_t)((t >> 3) * kKSbo + dg * kKLbo + (t & 7) * 16);
}
// element (token t, dims 8 dg .. 8 dg + 7) chunk of the value operand
__device__ __forceinline__ uint32_t val_chunk(int t, int dg) {
    return (uint32_t)(dg * kVSbo + (t >> 3) * kVLbo + (t & 7) * 16);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Bounded wait that gives up at once after an earlier one of this thread gave up.
__device__ __forceinline__ void pf_wait(uint32_t bar, uint32_t parity, bool& bad) {
    if (!bad && !mbar_wait(bar, parity)) bad = true;
}

template <int VB>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_tc_kernel(const PrefillArgs a) {
    using F = PageFmt<4, VB, 0>;
    using L = PfLayout<VB>;
    constexpr int D = kHeadDim;
    static_assert(L::total <= kSmemLimit, "prefill does not fit in shared memory");
    extern __shared__ __align__(128) uint8_t sm[];
    const Geometry& g = a.g;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, rb = blockIdx.y, h = blockIdx.z;
    const int G = a.group;
    const int R = a.C * G;                            // query rows of this KV head
    const int r0 = rb * kPfRows;                      // first row of the block
    const int rows = min(kPfRows, R - r0);
    const int p_hi = a.first + (r0 + rows - 1) / G;   // last position of the block
    const int nt_rb = p_hi / kPfTile + 1;             // tiles the block needs
    const int t_first = split * a.tiles_per_split;
    const int U = min(a.tiles_per_split, nt_rb - t_first);  // this CTA's tiles
    float* part = a.partials + (((int64_t)h * a.nrb + rb) * a.splits + split) * kPfRows * kPartRow;

    grid_dependency_wait();
    grid_launch_dependents();
    if (U <= 0) {
        // no tile of this split reaches the block's positions: empty partials
        for (int i = tid; i < kPfRows; i += kPfThreads) {
            part[i * kPartRow] = kMinusBig;
            part[i * kPartRow + 1] = 0.f;
        }
        for (int i = tid; i < kPfRows * D; i += kPfThreads) part[(i / D) * kPartRow + 4 + (i % D)] = 0.f;
        return;
    }

    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar0 = sbase + L::bars;
    auto bar = [&](int i) { return bar0 + 8 * i; };
    int* page_ok = reinterpret_cast<int*>(sm + L::ok);
    float* gam_s = reinterpret_cast<float*>(sm + L::gam);
    float* scl_s = reinterpret_cast<float*>(sm + L::scl);
    float* zer_s = reinterpret_cast<float*>(sm + L::zer);
    float* msk_s = reinterpret_cast<float*>(sm + L::msk);
    int* big_s = reinterpret_cast<int*>(sm + L::big);
    int* inv_s = reinterpret_cast<int*>(sm + L::inv);
    if (tid == 0) {
        for (int i = 0; i < kRing * kPfPages; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(kBarBk), 4);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(kBarBv + b), 2);
            mbar_init(bar(kBarS + b), 1);
            mbar_init(bar(kBarP + b), 8);
            mbar_init(bar(kBarO + b), 1);
        }
        mbar_init(bar(kBarQ), 8);
        mbar_init(bar(kBarNever), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc<kTmemCols>(sbase + L::taddr);
    // the flags: two of the four entries per tile are written (two value producer warps)
    for (int i = tid; i < 2 * 4 + 4 * 4; i += kPfThreads) big_s[i] = 0;  // big and inv are adjacent
    {
        // byte e (codes e & 15, e >> 4) -> (N[e & 15], N[e >> 4]), (rem2/delta[e & 15], rem2/delta[e >> 4])
        uint32_t* lut = reinterpret_cast<uint32_t*>(sm + L::lut);
        for (int e = tid; e < 256; e += kPfThreads) {
            lut[2 * e] = (uint32_t)a.c.cint_f16[e & 15] | ((uint32_t)a.c.cint_f16[e >> 4] << 16);
            lut[2 * e + 1] = (uint32_t)a.c.cremd_f16[e & 15] | ((uint32_t)a.c.cremd_f16[e >> 4] << 16);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + L::taddr);
    bool bad = false;  // a bounded wait of this thread gave up
    bool stalled = false;
    if (a.stall_cycles > 0 && (split & 1)) {
        // test hook: every thread of the CTA waits on a barrier that nothing
        // arrives on; the wait runs out and the CTA skips its tiles
        stalled = !mbar_wait_for(bar(kBarNever), 0, a.stall_cycles);
    }

    // ---- loader / MMA issuer (lane 0 of warp 8) ----
    const int npg = (p_hi + kBlockSize) / kBlockSize;  // pages the block needs
    // the block ids of tile u's pages (fetched a tile ahead of their use)
    auto fetch_ids = [&](int u, int (&blks)[kPfPages]) {
#pragma unroll
        for (int j = 0; j < kPfPages; ++j) {
            const int pgi = (t_first + u) * kPfPages + j;
            blks[j] = (u < U && pgi < npg) ? __ldg(a.block_row + pgi) : 0;
        }
    };
    auto load_tile = [&](int u, const int (&blks)[kPfPages]) {
        const int slot = u & (kRing - 1);
#pragma unroll
        for (int j = 0; j < kPfPages; ++j) {
            const int pgi = (t_first + u) * kPfPages + j;
            const int si = slot * kPfPages + j;
            const uint32_t b = bar(si);
            if (pgi < npg) {
                const int blk = blks[j];
                if (blk >= 0 && blk < g.num_blocks) {
                    page_ok[si] = 1;
                    mbar_arrive_tx(b, (uint32_t)F::bytes);
                    bulk_g2s(sbase + L::ring + si * L::stride, a.pool + ((int64_t)blk * g.hkv + h) * F::bytes,
                             (uint32_t)F::bytes, b);
                } else {
                    flag(a.status, TQ_FLAG_BAD_SLOT);
                    page_ok[si] = 0;
                    mbar_arrive(b);
                }
            } else {
                page_ok[si] = -1;  // past the block's last position: not loaded
                mbar_arrive(b);
            }
        }
    };
    constexpr uint32_t idesc_s = tc::idesc_f16_f32(kPfRows, kPfTile);
    constexpr uint32_t idesc_v = tc::idesc_f16_f32_bmn(kPfRows, kHeadDim);
    // scores of tile u into its columns: needs its key operand (written once
    // the scores of tile u - 1 had read the previous one); issued after PV of
    // tile u - 2, which read the weights these columns held
    auto issue_scores = [&](int u) {
        pf_wait(bar(kBarBk), u & 1, bad);
        tc::fence_after_sync();
        const uint32_t ts = tmem + kTs + 128 * (u & 1);
#pragma unroll
        for (int s = 0; s < 8; ++s)
            tc::mma_f16_ts(ts, tmem + kTq + 8 * s, tc::smem_desc(sbase + L::bn + 256 * s, kKLbo, kKSbo), idesc_s,
                           s > 0 ? 1u : 0u);
#pragma unroll
        for (int s = 0; s < 8; ++s)
            tc::mma_f16_ts(ts, tmem + kTq + 64 + 8 * s, tc::smem_desc(sbase + L::bn + 256 * s, kKLbo, kKSbo), idesc_s,
                           1u);
#pragma unroll
        for (int s = 0; s < 8; ++s)
            tc::mma_f16_ts(ts, tmem + kTq + 8 * s, tc::smem_desc(sbase + L::br + 256 * s, kKLbo, kKSbo), idesc_s, 1u);
        tc::commit(bar(kBarS + (u & 1)));
    };
    // values of tile u: needs its value operand and all weights
    auto issue_values = [&](int u) {
        pf_wait(bar(kBarBv + (u & 1)), (u >> 1) & 1, bad);
        pf_wait(bar(kBarP + (u & 1)), (u >> 1) & 1, bad);
        tc::fence_after_sync();
        const uint32_t tp = tmem + kTs + 128 * (u & 1);
        const uint32_t bv = sbase + L::bv + (u & 1) * L::bv_size;
        // K-step s: hi parts at columns 16 s .., lo parts at 16 s + 8 ..
#pragma unroll
        for (int s = 0; s < 8; ++s)
            tc::mma_f16_ts(tmem + kTo, tp + 16 * s, tc::smem_desc(bv + 256 * s, kVLbo, kVSbo), idesc_v,
                           (u > 0 || s > 0) ? 1u : 0u);
#pragma unroll
        for (int s = 0; s < 8; ++s)
            tc::mma_f16_ts(tmem + kTo, tp + 16 * s + 8, tc::smem_desc(bv + 256 * s, kVLbo, kVSbo), idesc_v, 1u);
        tc::commit(bar(kBarO + (u & 1)));
    };

    if (stalled) {
        for (int i = tid; i < kPfRows; i += kPfThreads) {
            part[i * kPartRow] = kMinusBig;
            part[i * kPartRow + 1] = 0.f;
        }
        for (int i = tid; i < kPfRows * D; i += kPfThreads) part[(i / D) * kPartRow + 4 + (i % D)] = 0.f;
        bad = true;
    } else if (warp == 12) {
        // ================= loader and MMA issuer =================
        // Issuing an MMA waits while the tensor pipe's queue is full, so this
        // warp does nothing else: its waits never hold up the softmax.
        if (lane == 0) {
            int ids[kPfPages];
            for (int u = 0; u < kRing && u < U; ++u) {
                fetch_ids(u, ids);
                load_tile(u, ids);
            }
            fetch_ids(kRing, ids);
            pf_wait(bar(kBarQ), 0, bad);
            issue_scores(0);
            if (U > 1) issue_scores(1);
            for (int u = 0; u < U; ++u) {
                issue_values(u);
                // the ring slot of tile u is free: its values are unpacked
                if (u + kRing < U) {
                    load_tile(u + kRing, ids);
                    fetch_ids(u + kRing + 1, ids);
                }
                // into the columns whose weights PV of tile u has just been queued to read
                if (u + 2 < U) issue_scores(u + 2);
            }
        }
        __syncwarp();
    } else if (warp >= 8 && warp < 12) {
        // ================= key producers: thread = token of the tile =================
        const int t = tid - 256;          // token of the tile
        const int j = t >> 4, slot = t & 15;
        const uint32_t* lut = reinterpret_cast<const uint32_t*>(sm + L::lut);
        for (int u = 0; u < U; ++u) {
            const int si = (u & (kRing - 1)) * kPfPages + j;
            pf_wait(bar(si), (u / kRing) & 1, bad);
            const int pok = page_ok[si];
            const int tok = (t_first + u) * kPfTile + t;
            const bool valid = pok == 1 && tok <= p_hi && !bad;
            const uint32_t pg = sbase + L::ring + si * L::stride;
            // ---- keys: the previous tile's scores MMA has read the operand ----
            if (u > 0) pf_wait(bar(kBarS + ((u - 1) & 1)), ((u - 1) >> 1) & 1, bad);
            // the softmax warps use the key operand's space for the query rotation
            else pf_wait(bar(kBarQ), 0, bad);
            // 16 code bytes (32 dims) at a time; the loop is not unrolled (the
            // warps of four roles share the instruction cache)
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                const uint4 v4 = valid ? lds128(pg + F::kcode + slot * 64 + 16 * c) : make_uint4(0, 0, 0, 0);
                const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // dims 8 dg .. 8 dg + 7 = code bytes 4 dg .. 4 dg + 3 = word q
                    const int dg = 4 * c + q;
                    uint32_t nn[4], rr[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t e = (w4[q] >> (8 * k)) & 0xFFu;
                        const uint2 v = valid ? *reinterpret_cast<const uint2*>(lut + 2 * e) : make_uint2(0u, 0u);
                        nn[k] = v.x;
                        rr[k] = v.y;
                    }
                    sts128(sbase + L::bn + key_chunk(t, dg), nn[0], nn[1], nn[2], nn[3]);
                    sts128(sbase + L::br + key_chunk(t, dg), rr[0], rr[1], rr[2], rr[3]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarBk));
        }
    } else if (warp >= 13) {
        // ================= value producers: thread = two tokens of the tile =================
        // Tokens v and v + 64 of the tile: their value operand rows, scales, zero
        // points, norms and masks, and the tile's flags (a token not there, a
        // scale above kBigScale), all written before the arrival on the value
        // barrier the softmax waits on.
        const int vw = warp - 13;
        const int v = tid - 13 * 32;      // 0 .. 63
        for (int u = 0; u < U; ++u) {
            const int half = u & 1;
            // ---- values: PV of tile u - 2 has read this value buffer ----
            if (u > 1) pf_wait(bar(kBarO + half), ((u - 2) >> 1) & 1, bad);
            bool any_inv = false, bg = false;
#pragma unroll 1
            for (int i = 0; i < 2; ++i) {
                const int t = v + 64 * i;
                const int j = t >> 4, slot = t & 15;
                const int si = (u & (kRing - 1)) * kPfPages + j;
                pf_wait(bar(si), (u / kRing) & 1, bad);
                const int pok = page_ok[si];
                const int tok = (t_first + u) * kPfTile + t;
                const bool valid = pok == 1 && tok <= p_hi && !bad;
                const uint32_t pg = sbase + L::ring + si * L::stride;
                constexpr int VROW = D * VB / 8;
                const uint32_t bvb = sbase + L::bv + half * L::bv_size;
                if constexpr (VB == 3) {
                    uint32_t w[VB * 4];
#pragma unroll
                    for (int c = 0; c < VB; ++c) {
                        const uint4 v4 = valid ? lds128(pg + F::vcode + slot * VROW + 16 * c) : make_uint4(0, 0, 0, 0);
                        w[4 * c] = v4.x; w[4 * c + 1] = v4.y; w[4 * c + 2] = v4.z; w[4 * c + 3] = v4.w;
                    }
#pragma unroll
                    for (int dg = 0; dg < 16; ++dg) {
                        uint32_t pr[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            // codes of dims 8 dg + 2k, 8 dg + 2k + 1 as fp16 subnormals c * 2^-24
                            const uint32_t c0 = bits_at<VB * 4>(w, VB * (8 * dg + 2 * k), VB);
                            const uint32_t c1 = bits_at<VB * 4>(w, VB * (8 * dg + 2 * k + 1), VB);
                            pr[k] = c0 | (c1 << 16);
                        }
                        sts128(bvb + val_chunk(t, dg), pr[0], pr[1], pr[2], pr[3]);
                    }
                } else {
                    // 16 code bytes at a time: 16 / VB groups of 8 dims
                    constexpr int DGC = 16 / VB;
#pragma unroll 1
                    for (int c = 0; c < VB; ++c) {
                        const uint4 v4 = valid ? lds128(pg + F::vcode + slot * VROW + 16 * c) : make_uint4(0, 0, 0, 0);
                        const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                        for (int q = 0; q < DGC; ++q) {
                            uint32_t pr[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                // codes of dims 8 dg + 2k, 8 dg + 2k + 1 as fp16 subnormals c * 2^-24
                                const uint32_t c0 = bits_at<4>(w4, VB * (8 * q + 2 * k), VB);
                                const uint32_t c1 = bits_at<4>(w4, VB * (8 * q + 2 * k + 1), VB);
                                pr[k] = c0 | (c1 << 16);
                            }
                            sts128(bvb + val_chunk(t, DGC * c + q), pr[0], pr[1], pr[2], pr[3]);
                        }
                    }
                }
                float sc = 0.f, zr = 0.f, gm = 0.f;
                if (valid) {
                    sc = lds_h2f(pg + F::scl + 2 * slot);
                    zr = lds_h2f(pg + F::zer + 2 * slot);
                    gm = lds_h2f(pg + F::gam + 2 * slot);
                }
                scl_s[half * kPfTile + t] = sc;
                zer_s[half * kPfTile + t] = zr;
                gam_s[(u & 3) * kPfTile + t] = gm;
                msk_s[(u & 3) * kPfTile + t] = valid ? 0.f : -INFINITY;
                any_inv = any_inv || !valid;
                // a scale above kBigScale makes this tile take the exact max, so
                // that p * scale (p <= 1 then) stays inside the fp16 range
                bg = bg || sc > kBigScale;
            }
            any_inv = __any_sync(0xffffffffu, any_inv);
            bg = __any_sync(0xffffffffu, bg);
            if (lane == 0) {
                inv_s[(u & 3) * 4 + vw] = any_inv ? 1 : 0;
                big_s[half * 4 + vw] = bg ? 1 : 0;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarBv + half));
        }
    } else {
        // ================= softmax: two threads per query row =================
        // Warps w and w + 4 share tensor-memory lanes 32 (w % 4) ..: thread
        // (row r, half hf) works on columns 64 hf .. 64 hf + 63 of the row's
        // scores and weights and on dims 64 hf .. 64 hf + 63 of its query and
        // output.  The halves exchange the row's maxima and sums in shared
        // memory (named barrier 1 over the 256 softmax threads).
        const int r = tid & 127, hf = warp >> 2;
        const int rg = r0 + r;
        const bool row_ok = r < rows;
        const int pos = row_ok ? a.first + rg / G : -1;  // the row's position (-1: padding row)
        const uint32_t tl = (uint32_t)((warp & 3) * 32) << 16;
        const float ksc = a.sm_scale_log2;
        float* xch = reinterpret_cast<float*>(sm + L::xch);  // [4][2][128]: two rounds x halves x rows
        auto pair_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(kPfSoftmax) : "memory"); };
        float qs = 1.f;
        {
            // q_rot = R q: the half of the row in registers (signs, butterflies of
            // strides 1 .. 32), the last stage (stride 64) through shared memory
            // (the key operand's space, which the producers leave alone until the
            // query operand is stored)
            float x[64];
            if (row_ok) {
                const int64_t qrow = ((int64_t)(rg / G) * a.hq + (int64_t)h * G + rg % G) * D + 64 * hf;
#pragma unroll
                for (int i = 0; i < 64; i += 4) load4(a.q, a.dtype, qrow + i, x + i);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) x[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int d = 64 * hf + i;
                if ((a.c.sign_bits[d >> 5] >> (d & 31)) & 1u) x[i] = -x[i];
            }
#pragma unroll
            for (int hh = 1; hh < 64; hh <<= 1)
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if ((i & hh) == 0) {
                        const float p = x[i], q2 = x[i + hh];
                        x[i] = p + q2;
                        x[i + hh] = p - q2;
                    }
            float* xs = reinterpret_cast<float*>(sm + L::bn);  // [half][64][128 rows]
#pragma unroll
            for (int i = 0; i < 64; ++i) xs[(hf * 64 + i) * kPfRows + r] = x[i];
            pair_sync();
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const float o = xs[((1 - hf) * 64 + i) * kPfRows + r];
                // dims i and i + 64: (first half) + (second half), (first half) - (second half)
                x[i] = (hf == 0 ? x[i] + o : o - x[i]) * 0.08838834764831845f;
                mx = fmaxf(mx, fabsf(x[i]));
            }
            xch[hf * kPfRows + r] = mx;
            pair_sync();
            mx = fmaxf(xch[r], xch[kPfRows + r]);
            const float big = fabsf(a.c.delta) * ksc * mx;
            qs = (big > 0.f) ? exp2f(ceilf(log2f(big / 512.f))) : 1.f;
            const float e = ksc * a.c.delta / qs;
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float x0 = e * x[2 * k], x1 = e * x[2 * k + 1];
                hi[k] = pack_h2(x0, x1);
                const float2 hf2 = __half22float2(*reinterpret_cast<const __half2*>(&hi[k]));
                lo[k] = pack_h2(x0 - hf2.x, x1 - hf2.y);
            }
            tc::st_32x32b_x32(tmem + tl + kTq + 32 * hf, hi);
            tc::st_32x32b_x32(tmem + tl + kTq + 64 + 32 * hf, lo);
            tc::wait_st();
        }
        // the query operand of this warp's 32 rows, half hf, is in tensor memory
        tc::fence_before_sync();
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(bar(kBarQ));

        float m = kMinusBig;
        uint64_t l2 = 0ull, z2acc = 0ull;  // this half's running sum and zero-point sum, two lanes each
        const int p_lo = a.first + r0 / G;  // the block's first position
        for (int u = 0; u < U; ++u) {
            const int base = (t_first + u) * kPfTile;
            // scores of tile u, then its per-token norms, masks, scales and zero
            // points: the producers write them all before arriving on the value
            // barrier of the tile's parity (whose next phase needs these warps'
            // weights, so a wait on it never falls a whole phase behind)
            pf_wait(bar(kBarS + (u & 1)), (u >> 1) & 1, bad);
            pf_wait(bar(kBarBv + (u & 1)), (u >> 1) & 1, bad);
            tc::fence_after_sync();
            const uint32_t tsp = tmem + tl + kTs + 128 * (u & 1);
            // logit (log2 units) = S * qscale * gamma of this half's 64 tokens;
            // tokens that are not there and, causally, tokens after the row's
            // position get -inf
            const int kmax = pos - base;  // the last token of the tile the row sees
            // a tile wholly before the block's first position needs no causal mask
            // (uniform over the CTA)
            const bool diag = base + kPfTile - 1 > p_lo;
            const int4 iv4 = *reinterpret_cast<const int4*>(inv_s + 4 * (u & 3));
            const bool plain = !diag && (iv4.x | iv4.y | iv4.z | iv4.w) == 0;
            const float2* g2 = reinterpret_cast<const float2*>(gam_s + (u & 3) * kPfTile);
            const float2* m2 = reinterpret_cast<const float2*>(msk_s + (u & 3) * kPfTile);
            const uint64_t QS2 = f2_pack(qs, qs);
            float x[64];
            float mt0 = kMinusBig, mt1 = kMinusBig;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col = 64 * hf + 32 * c;
                uint32_t v[32];
                tc::ld_32x32b_x32(tsp + col, v);
                tc::wait_ld();
                tc::reg_fence(v);
#pragma unroll
                for (int k2 = 0; k2 < 16; ++k2) {
                    const float2 gg = g2[col / 2 + k2];
                    const uint64_t s2 = f2_mul(f2_pack(__uint_as_float(v[2 * k2]), __uint_as_float(v[2 * k2 + 1])), QS2);
                    float* xx = x + 32 * c + 2 * k2;
                    if (plain) {
                        f2_unpack(f2_mul(s2, f2_pack(gg.x, gg.y)), xx[0], xx[1]);
                    } else {
                        const float2 mm = m2[col / 2 + k2];
                        f2_unpack(f2_fma(s2, f2_pack(gg.x, gg.y), f2_pack(mm.x, mm.y)), xx[0], xx[1]);
                        const int k = col + 2 * k2;
                        if (k > kmax) xx[0] = -INFINITY;
                        if (k + 1 > kmax) xx[1] = -INFINITY;
                    }
                    mt0 = fmaxf(mt0, xx[0]);
                    mt1 = fmaxf(mt1, xx[1]);
                }
            }
            // the row's tile max from both halves (exchange buffer by tile parity)
            float* mxx = xch + 2 * kPfRows * (2 + (u & 1));
            mxx[hf * kPfRows + r] = fmaxf(mt0, mt1);
            pair_sync();
            const float mt = fmaxf(mxx[r], mxx[kPfRows + r]);
            // The tensor-memory loads and stores are warp-wide (.sync.aligned), so
            // the rescale is decided for the whole warp (both halves decide alike):
            // a row that keeps its max takes the factor 1.
            const int4 bg4 = *reinterpret_cast<const int4*>(big_s + 4 * (u & 1));
            const bool exact = (bg4.x | bg4.y | bg4.z | bg4.w) != 0;
            const bool raise = mt > m + kLazy || (exact && mt > m);
            if (__any_sync(0xffffffffu, raise)) {
                const float mn = raise ? mt : m;
                const float f = ex2(m - mn);
                const uint64_t F2 = f2_pack(f, f);
                l2 = f2_mul(l2, F2);
                z2acc = f2_mul(z2acc, F2);
                if (u > 0) {
                    // the output accumulator holds every PV up to tile u - 1
                    pf_wait(bar(kBarO + ((u - 1) & 1)), ((u - 1) >> 1) & 1, bad);
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t ov[32];
                        tc::ld_32x32b_x32(tmem + tl + kTo + 64 * hf + 32 * c, ov);
                        tc::wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * f);
                        tc::st_32x32b_x32(tmem + tl + kTo + 64 * hf + 32 * c, ov);
                    }
                }
                m = mn;
            }
            // the weights over the scores: the 16 tokens of K-step s take columns
            // 16 s .. 16 s + 7 (hi parts, pairs) and 16 s + 8 .. 16 s + 15 (lo parts)
            const float2* z2 = reinterpret_cast<const float2*>(zer_s + (u & 1) * kPfTile);
            const float2* c2 = reinterpret_cast<const float2*>(scl_s + (u & 1) * kPfTile);
            const uint64_t M2 = f2_pack(m, m);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col = 64 * hf + 32 * c;
                uint32_t v[32];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float d0, d1;
                    f2_unpack(f2_sub(f2_pack(x[32 * c + 2 * k], x[32 * c + 2 * k + 1]), M2), d0, d1);
                    const uint64_t P2 = f2_pack(ex2(d0), ex2(d1));
                    const float2 zz = z2[col / 2 + k], cc = c2[col / 2 + k];
                    l2 = f2_add(l2, P2);
                    z2acc = f2_fma(P2, f2_pack(zz.x, zz.y), z2acc);
                    const uint64_t W2 = f2_mul(P2, f2_pack(cc.x, cc.y));
                    float w0, w1;
                    f2_unpack(W2, w0, w1);
                    const uint32_t hi = pack_h2(w0, w1);
                    const float2 hf2 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                    float lo0, lo1;
                    f2_unpack(f2_sub(W2, f2_pack(hf2.x, hf2.y)), lo0, lo1);
                    v[16 * (k >> 3) + (k & 7)] = hi;
                    v[16 * (k >> 3) + 8 + (k & 7)] = pack_h2(lo0, lo1);
                }
                tc::st_32x32b_x32(tsp + col, v);
            }
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(bar(kBarP + (u & 1)));
        }
        // ---- this split's partial for the row: max, sum, rotated accumulator + zero term ----
        float l, z, l_b, z_b;
        f2_unpack(l2, l, l_b);
        f2_unpack(z2acc, z, z_b);
        l += l_b;
        z += z_b;
        xch[hf * kPfRows + r] = l;
        xch[2 * kPfRows + hf * kPfRows + r] = z;
        pair_sync();
        l = xch[r] + xch[kPfRows + r];
        z = xch[2 * kPfRows + r] + xch[3 * kPfRows + r];
        pf_wait(bar(kBarO + ((U - 1) & 1)), ((U - 1) >> 1) & 1, bad);
        tc::fence_after_sync();
        float* pr = part + r * kPartRow;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            tc::ld_32x32b_x32(tmem + tl + kTo + 64 * hf + 32 * c, v);
            tc::wait_ld();
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(pr + 4 + 64 * hf + 32 * c + k) =
                    make_float4(fmaf(__uint_as_float(v[k]), kOutScale, z), fmaf(__uint_as_float(v[k + 1]), kOutScale, z),
                                fmaf(__uint_as_float(v[k + 2]), kOutScale, z), fmaf(__uint_as_float(v[k + 3]), kOutScale, z));
        }
        if (hf == 0) {
            pr[0] = m;
            pr[1] = l;
        }
    }
    // every tensor-core operation of the CTA is complete (the softmax warps
    // waited for the last PV commit): release tensor memory
    bad = __syncthreads_or(bad);
    if (bad && tid == 0) flag(a.status, TQ_FLAG_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc<kTmemCols>(tmem);
    }
}

// One warp per output row (position, query head): merge the splits' partials
// of its row and rotate back, out = R^T (acc / sum) = diag(s) H (acc / sum) / sqrt(d).
__global__ void __launch_bounds__(128) prefill_merge_kernel(const PrefillArgs a) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);  // i * hq + query head
    if (row >= (int64_t)a.C * a.hq) return;
    const int i = (int)(row / a.hq), qh = (int)(row % a.hq);
    const int G = a.group, h = qh / G, g = qh % G;
    const int rg = i * G + g, rb = rg / kPfRows, r = rg % kPfRows;
    const float* base = a.partials + (((int64_t)h * a.nrb + rb) * a.splits) * kPfRows * kPartRow + r * kPartRow;
    const int64_t sstride = (int64_t)kPfRows * kPartRow;
    float M = kMinusBig;
    for (int s = 0; s < a.splits; ++s) M = fmaxf(M, base[s * sstride]);
    float Ls = 0.f, x[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < a.splits; ++s) {
        const float* p = base + s * sstride;
        const float f = exp2f(p[0] - M);
        Ls = fmaf(f, p[1], Ls);
        const float4 v = *reinterpret_cast<const float4*>(p + 4 + 4 * lane);
        x[0] = fmaf(f, v.x, x[0]); x[1] = fmaf(f, v.y, x[1]); x[2] = fmaf(f, v.z, x[2]); x[3] = fmaf(f, v.w, x[3]);
    }
    const float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] *= inv;
    fwht128(x, lane);
    const uint32_t sg = (a.c.sign_bits[lane >> 3] >> (4 * (lane & 7))) & 0xFu;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[k] *= 0.08838834764831845f;
        if ((sg >> k) & 1u) x[k] = -x[k];
    }
    *reinterpret_cast<float4*>(a.out + row * kHeadDim + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
}

template <int VB>
int launch_prefill_tc_t(const PrefillArgs& a, cudaStream_t s) {
    using F = PageFmt<4, VB, 0>;
    const Geometry& g = a.g;
    if (g.page_bytes != F::bytes || g.vcode_off != F::vcode || g.gam_off != F::gam || g.scl_off != F::scl ||
        g.zer_off != F::zer || g.bs != kBlockSize || g.d != kHeadDim || g.m != 0 || g.kb != 4)
        return (int)cudaErrorInvalidValue;
    auto kern = prefill_tc_kernel<VB>;
    static int done[64] = {};
    cudaError_t e = ensure_smem_limit(kern, PfLayout<VB>::total, done);
    if (e != cudaSuccess) return (int)e;
    e = launch_programmatic(kern, dim3((unsigned)a.splits, (unsigned)a.nrb, (unsigned)g.hkv), dim3(kPfThreads),
                            (size_t)PfLayout<VB>::total, s, a);
    if (e != cudaSuccess) return (int)e;
    const int64_t rows = (int64_t)a.C * a.hq;
    return (int)launch_programmatic(prefill_merge_kernel, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, s, a);
}

}  // namespace

bool prefill_tc_supported(const Geometry& g) { return g.kb == 4 && g.m == 0 && g.vb >= 1 && g.vb <= 4; }

size_t prefill_tc_partials_bytes(const Geometry& g, int C, int hq, int splits) {
    const int G = hq / g.hkv;
    const int64_t nrb = ((int64_t)C * G + kPfRows - 1) / kPfRows;
    return (size_t)g.hkv * nrb * splits * kPfRows * kPartRow * sizeof(float);
}

int prefill_tc_rows_per_block() { return kPfRows; }
int prefill_tc_tile_tokens() { return kPfTile; }

int launch_prefill_tc(const PrefillArgs& a, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (a.g.vb) {
        case 1: return launch_prefill_tc_t<1>(a, s);
        case 2: return launch_prefill_tc_t<2>(a, s);
        case 3: return launch_prefill_tc_t<3>(a, s);
        case 4: return launch_prefill_tc_t<4>(a, s);
        default: return (int)cudaErrorNotSupported;
    }
}

}  // namespace tq
