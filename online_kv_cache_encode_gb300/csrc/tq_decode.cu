// Decode attention over the compressed paged cache (split-K flash decode).
//
// Grid (split, KV head, sequence); one CTA per SM (shared memory bound).
//  - Producer warp: reads block ids, streams whole pages (one page = 16
//    tokens of one KV head, contiguous) into a shared-memory ring with 1-D
//    bulk async copies (cp.async.bulk) completing on mbarriers.
//  - 8 consumer warps: each takes whole pages and keeps its own online-softmax
//    state for the G <= 8 query heads of the group.  Per page:
//      scores  S[16 tok x 8 q] = A[16 tok x 128] . B[128 x 8 q]  (mma.sync m16n8k16,
//              tokens as rows) where the key centroid is split as
//              C[c] = alpha (c - mid) + rem[c]: the integer code c is exact in
//              fp16 and multiplies alpha*q_rot split into fp16 hi + lo; rem[c]
//              comes from a lane-private shared-memory table and multiplies
//              q_rot's hi part.  logit = gamma_t * sm_scale * (S - alpha*mid*sum q_rot)
//      softmax running max / sum per query (exp2 domain)
//      values  O^T[128 x 8 q] += Vcode^T[128 x 16 tok] . (p * scale)^T[16 tok x 8 q],
//              value codes exact in fp16, p*scale split into hi + lo; the
//              zero-point term sum_t p_t zero_t is accumulated in fp32.
//    Keys are never reconstructed; everything stays in the rotated frame
//    ["OCTOPUS ..." -- TL;DR / step 7; deep dive -- [RHT effect]: inner
//    products are preserved by the rotation].
//  - Warps merge in shared memory; a sequence split over several CTAs writes
//    partials (max, sum, acc) and the last CTA to finish (atomic counter)
//    merges them and applies the one inverse rotation R^T = diag(s) H / sqrt(d).
// Attention itself: softmax(q K^T / sqrt(d_h)) V [Bit-Axon -- attention under
// quantized KV].
#include <cuda_runtime.h>

#include <cuda_fp8.h>

#include "tq_device.cuh"

namespace tq {

constexpr int kNCW = 8;                       // warps per CTA, each consumes (and fetches) its own pages
constexpr int kThreads = kNCW * 32;
constexpr int kSlotsPerWarp = 8;              // ring slots per warp: pages a warp keeps in flight
constexpr int kLutBytes = 256 * 256;          // 256 entries x 256 B (lanes use 128 B)
constexpr long long kWaitCycles = 3000000000ll;  // bound on any wait: ~1.5 s at 2 GHz
// split partial record: max, sum, 2 pad, acc[128] (keeps the acc 16-byte aligned)
constexpr int kPartStride = 4 + kHeadDim;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of the given parity.  Spins on try_wait and looks at the
// SM cycle counter only every 256 tries; gives up after kWaitCycles (about a
// second or two at GB300 clocks).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try(bar, parity)) return true;
        if (clock64() - t0 > kWaitCycles) return false;
    }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds_h2f(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t m, uint32_t o) {
    return (a & m) | o;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t movtrans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D += A . B with A 16x32, B 32x8 of e4m3, fp32 accumulate (exact products, fp32 sums)
__device__ __forceinline__ void mma_e4m3(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t f2e4m3(float x) {
    return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_2f(uint32_t b) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3)));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_h2(uint32_t v) {
    return __half22float2(*reinterpret_cast<__half2*>(&v));
}
// x ~= hi + lo, both binary16
__device__ __forceinline__ void split_h2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_h2(x0, x1);
    float2 h = unpack_h2(hi);
    lo = pack_h2(x0 - h.x, x1 - h.y);
}
__device__ __forceinline__ float h2f(uint16_t b) {
    return __half2float(*reinterpret_cast<__half*>(&b));
}

// Four fp16x2 registers from one word of eight 4-bit codes n0..n7 (n_i at
// bits 4i): reg i holds (n_i, n_{i+4}) as exact small integers.
__device__ __forceinline__ void nib8_to_h2(uint32_t w, uint32_t f[4]) {
    const uint32_t magic = 0x64006400u;           // fp16 1024.0 in both halves
    const uint32_t k1024 = 0x64006400u;
    const uint32_t k16 = 0x2C002C00u;             // 1/16
    const uint32_t km64 = 0xD400D400u;            // -64
    const uint32_t w8 = w >> 8;
    f[0] = hsub2(lop_and_or(w, 0x000F000Fu, magic), k1024);
    f[1] = hfma2(lop_and_or(w, 0x00F000F0u, magic), k16, km64);
    f[2] = hsub2(lop_and_or(w8, 0x000F000Fu, magic), k1024);
    f[3] = hfma2(lop_and_or(w8, 0x00F000F0u, magic), k16, km64);
}

// ---------------------------------------------------------------------------
// shared memory map (dynamic)
// ---------------------------------------------------------------------------
struct SmemMap {
    int lut, rem, qrot, qoff, qscale, sq, bars, ok, ring;
    int stages, stride, total;
};

__host__ __device__ inline SmemMap smem_map(int page_bytes) {
    SmemMap m;
    int off = 0;
    m.lut = off; off += kLutBytes;
    m.rem = off; off += 16 * 2;
    m.qrot = off; off += 8 * kHeadDim * 4;
    m.qoff = off; off += 8 * 4;
    m.qscale = off; off += 8 * 4;
    m.sq = off; off += 8 * kHeadDim * 4;
    m.stride = (page_bytes + 127) / 128 * 128;
    m.stages = kNCW * kSlotsPerWarp;
    m.bars = (off + 7) / 8 * 8; off = m.bars + 8 * m.stages;
    m.ok = off; off += 4 * m.stages;
    m.ring = (off + 127) / 128 * 128; off = m.ring + m.stride * m.stages;
    m.total = off;
    return m;
}

int decode_smem_bytes(const Geometry& g) { return smem_map((int)g.page_bytes).total; }

// ---------------------------------------------------------------------------
// code unpacking: every key / value code becomes an exact small integer in
// fp16 (the 0x6400 "1024 + x" bit pattern, then the 1024 removed exactly)
// ---------------------------------------------------------------------------
// sixteen 2-bit codes c0..c15 of w (c_i at bits 2i) -> eight fp16x2 (c_i, c_{i+8})
__device__ __forceinline__ void crumb16_to_h2(uint32_t w, uint32_t f[8]) {
    const uint32_t magic = 0x64006400u;
    const uint32_t scale[4] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u};  // 1, 1/4, 1/16, 1/64
    const uint32_t bias[4] = {0xE400E400u, 0xDC00DC00u, 0xD400D400u, 0xCC00CC00u};   // -1024, -256, -64, -16
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t x = (i < 4) ? w : (w >> 8);
        const int k = i & 3;
        f[i] = hfma2(lop_and_or(x, 0x00030003u << (2 * k), magic), scale[k], bias[k]);
    }
}

// bits [pos, pos + n) of a little-endian multi-word bit string (pos, n compile-time after unrolling)
template <int NW>
__device__ __forceinline__ uint32_t bits_at(const uint32_t (&w)[NW], int pos, int n) {
    const int wi = pos >> 5, sh = pos & 31;
    uint32_t x = (sh + n <= 32 || wi + 1 >= NW) ? (w[wi] >> sh) : __funnelshift_r(w[wi], w[wi + 1], sh);
    return x & ((1u << n) - 1u);
}

__device__ __forceinline__ uint32_t int_pair_h2(uint32_t c0, uint32_t c1) {
    return hsub2((c0 | (c1 << 16)) | 0x64006400u, 0x64006400u);
}

// Key chunk of one token: the 32 codes of dims 32qd .. 32qd+31 (4*KB bytes).
template <int KB>
__device__ __forceinline__ void key_words(uint32_t row, int qd, uint32_t (&w)[KB]) {
    if constexpr (KB == 4) {
        const uint4 v = lds128(row + qd * 16);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (KB == 2) {
        const uint2 v = lds64(row + qd * 8);
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = lds32(row + qd * 12); w[1] = lds32(row + qd * 12 + 4); w[2] = lds32(row + qd * 12 + 8);
    }
}

// The integer codes as e4m3 operand bytes.  A code byte n < 16 read as e4m3 is
// exactly n * 2^-9 (exponent field 0 is the subnormal n * 2^-9, field 1 is
// (8 + m) * 2^-9), so the codes need only be spread into bytes.
// E[e] byte i holds the code of chunk dim key_fp8_dim<KB>(e, i).
template <int KB>
__host__ __device__ constexpr int key_fp8_dim(int e, int i) {
    return KB == 4 ? 8 * (e >> 1) + 2 * i + (e & 1)
         : KB == 2 ? 16 * (e >> 2) + 4 * i + (e & 3)
                   : 4 * e + i;
}

__device__ __forceinline__ uint32_t spread3x4(uint32_t t) {  // four 3-bit fields -> four bytes
    return (t & 0x7u) | ((t & 0x38u) << 5) | ((t & 0x1C0u) << 10) | ((t & 0xE00u) << 15);
}

template <int KB>
__device__ __forceinline__ void key_bytes(const uint32_t (&w)[KB], uint32_t E[8]) {
    if constexpr (KB == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            E[2 * i] = w[i] & 0x0F0F0F0Fu;
            E[2 * i + 1] = (w[i] >> 4) & 0x0F0F0F0Fu;
        }
    } else if constexpr (KB == 2) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int sh = 0; sh < 4; ++sh) E[4 * i + sh] = (w[i] >> (2 * sh)) & 0x03030303u;
    } else {
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
            const uint32_t x = bits_at<3>(w, 24 * gi, 24);
            E[2 * gi] = spread3x4(x & 0xFFFu);
            E[2 * gi + 1] = spread3x4(x >> 12);
        }
    }
}

// Remainder operands: R[n] = (rem[c_{2n}], rem[c_{2n+1}]) from the lane-private table.
template <int KB>
__device__ __forceinline__ void key_rem(const uint32_t (&w)[KB], uint32_t lut, uint32_t lane, uint32_t R[16]) {
    if constexpr (KB == 4) {
        const uint32_t lw = lane << 2;
#pragma unroll
        for (int n = 0; n < 16; ++n) R[n] = lds32(lut + prmt(w[n >> 2], lw, 0x5504u | ((uint32_t)(n & 3) << 4)));
    } else if constexpr (KB == 2) {
        const uint32_t lw = lane << 3;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint2 v = lds64(lut + prmt(w[j >> 2], lw, 0x5504u | ((uint32_t)(j & 3) << 4)));
            R[2 * j] = v.x;
            R[2 * j + 1] = v.y;
        }
    } else {
        const uint32_t lw = lane << 2;
#pragma unroll
        for (int n = 0; n < 16; ++n) R[n] = lds32(lut + (bits_at<3>(w, 6 * n, 6) << 7) + lw);
    }
}

// Value codes of dims 16r .. 16r+15 for a token pair (ta, tb): P[i] = (code_ta, code_tb)
// of dim 16r + i as exact fp16 integers.
template <int VB>
__device__ __forceinline__ void value_pair(uint32_t vbase, int r, int ta, int tb, uint32_t P[16]) {
    constexpr int ROW = kHeadDim * VB / 8;
    if constexpr (VB == 4) {
        const uint2 va = lds64(vbase + ta * ROW + r * 8);
        const uint2 vb = lds64(vbase + tb * ROW + r * 8);
        nib8_to_h2(prmt(va.x, vb.x, 0x5410u), &P[0]);
        nib8_to_h2(prmt(va.x, vb.x, 0x7632u), &P[4]);
        nib8_to_h2(prmt(va.y, vb.y, 0x5410u), &P[8]);
        nib8_to_h2(prmt(va.y, vb.y, 0x7632u), &P[12]);
    } else if constexpr (VB == 2) {
        const uint32_t wa = lds32(vbase + ta * ROW + r * 4);
        const uint32_t wb = lds32(vbase + tb * ROW + r * 4);
        crumb16_to_h2(prmt(wa, wb, 0x5410u), &P[0]);
        crumb16_to_h2(prmt(wa, wb, 0x7632u), &P[8]);
    } else {
        const int base = (6 * r) & ~3, sh = ((6 * r) & 3) * 8;
        const uint32_t a0 = lds32(vbase + ta * ROW + base), a1 = lds32(vbase + ta * ROW + base + 4);
        const uint32_t b0 = lds32(vbase + tb * ROW + base), b1 = lds32(vbase + tb * ROW + base + 4);
        const uint32_t xa[2] = {__funnelshift_r(a0, a1, sh), a1 >> sh};
        const uint32_t xb[2] = {__funnelshift_r(b0, b1, sh), b1 >> sh};
#pragma unroll
        for (int i = 0; i < 16; ++i) P[i] = int_pair_h2(bits_at<2>(xa, 3 * i, 3), bits_at<2>(xb, 3 * i, 3));
    }
}

// QJL sign bits of one token (bits 32qd .. 32qd+31 of its sigma row):
// Z[n] = (+-1 for bit n, +-1 for bit n+16) in fp16.
__device__ __forceinline__ void sign_chunk(uint32_t w, uint32_t Z[16]) {
#pragma unroll
    for (int n = 0; n < 16; ++n) Z[n] = ((w << (15 - n)) & 0x80008000u) ^ 0xBC00BC00u;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int KB, int VB, int M>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeArgs a) {
    static_assert(KB >= 2 && KB <= 4 && VB >= 2 && VB <= 4 && (M == 0 || M == 128), "unsupported page format");
    extern __shared__ __align__(128) uint8_t sm[];
    const Geometry& g = a.g;
    constexpr int D = kHeadDim;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = a.group;
    const SmemMap mp = smem_map((int)g.page_bytes);
    constexpr int SPW = kSlotsPerWarp;

    float* qrot = reinterpret_cast<float*>(sm + mp.qrot);
    float* qoff = reinterpret_cast<float*>(sm + mp.qoff);
    float* qscale = reinterpret_cast<float*>(sm + mp.qscale);
    int* slot_ok = reinterpret_cast<int*>(sm + mp.ok);
    const uint32_t bar_full = smem_u32(sm + mp.bars);
    const uint32_t lut_base = smem_u32(sm + mp.lut);
    const uint32_t ring_base = smem_u32(sm + mp.ring);
    uint8_t* ring = sm + mp.ring;
    const int p0 = split * a.pages_per_split;

    // ---- independent global loads first: length, this warp's block ids, the query ----
    // Warp w handles pages w, w + 8, w + 16, ... of the split (its j-th page is
    // w + 8 j) in its own ring slots w*SPW .. w*SPW + SPW - 1.  Lane l holds the
    // block id of the warp's page l of the current batch of 32 (bid_cur) and of
    // the next batch (bid_nxt).
    int len = __ldg(a.lens + b);
    const int32_t* btw = a.block_table + (int64_t)b * a.max_blocks + p0 + warp;
    const int reach = min(a.pages_per_split, a.max_blocks - p0) - warp;  // pages of the split at or after this warp's first
    int bid_cur = (8 * lane < reach) ? __ldg(btw + 8 * lane) : -1;
    int bid_nxt = (8 * (32 + lane) < reach) ? __ldg(btw + 8 * (32 + lane)) : -1;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < G) load4(a.q, a.dtype, ((int64_t)b * a.hq + (int64_t)h * G + warp) * D + 4 * lane, x);
    if (lane == 0) {
        for (int k = 0; k < SPW; ++k) mbar_init(bar_full + 8 * (warp * SPW + k), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    // ---- sequence range of this split ----
    if (len > a.max_blocks * g.bs) {
        if (tid == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
        len = a.max_blocks * g.bs;
    }
    if (len < 0) len = 0;
    const int seq_pages = (len + g.bs - 1) / g.bs;
    int npages = seq_pages - p0;
    if (npages > a.pages_per_split) npages = a.pages_per_split;
    if (npages < 0) npages = 0;
    const int nmine = npages > warp ? (npages - warp + kNCW - 1) / kNCW : 0;  // this warp's pages

    // Start a page copy into the warp's ring slot; a bad block id arrives on the
    // barrier without data and the page is skipped.
    auto issue = [&](int j, int blk) {
        const int sl = warp * SPW + (j % SPW);
        const bool ok = blk >= 0 && blk < g.num_blocks;
        slot_ok[sl] = ok;
        if (ok) {
            mbar_arrive_tx(bar_full + 8 * sl, (uint32_t)g.page_bytes);
            bulk_g2s(ring_base + sl * mp.stride, a.pool + ((int64_t)blk * g.hkv + h) * g.page_bytes,
                     (uint32_t)g.page_bytes, bar_full + 8 * sl);
        } else {
            flag(a.status, TQ_FLAG_BAD_SLOT);
            mbar_arrive(bar_full + 8 * sl);
        }
    };
    if (lane < SPW && lane < nmine) issue(lane, bid_cur);  // the first SPW pages, one lane each

    bool timed_out = false;
    {
        // Lane-private remainder table (copy for lane l at entry*stride + l*width):
        //   4-bit keys: byte e (2 codes) -> (rem[e&15], rem[e>>4])              stride 256, 4 B
        //   2-bit keys: byte e (4 codes) -> (rem[c0], rem[c1]), (rem[c2], rem[c3]) stride 256, 8 B
        //   3-bit keys: 6 bits e (2 codes) -> (rem[e&7], rem[e>>3])              stride 128, 4 B
        uint16_t* rem = reinterpret_cast<uint16_t*>(sm + mp.rem);
        if (tid < 16) rem[tid] = a.c.rem_f16[tid];
        __syncthreads();
        {
            if constexpr (KB == 4) {
                for (int i = tid; i < 256 * 32; i += kNCW * 32) {
                    const int e = i >> 5, l = i & 31;
                    *reinterpret_cast<uint32_t*>(sm + mp.lut + e * 256 + 4 * l) =
                        (uint32_t)rem[e & 15] | ((uint32_t)rem[e >> 4] << 16);
                }
            } else if constexpr (KB == 2) {
                for (int i = tid; i < 256 * 32; i += kNCW * 32) {
                    const int e = i >> 5, l = i & 31;
                    uint2 v;
                    v.x = (uint32_t)rem[e & 3] | ((uint32_t)rem[(e >> 2) & 3] << 16);
                    v.y = (uint32_t)rem[(e >> 4) & 3] | ((uint32_t)rem[e >> 6] << 16);
                    *reinterpret_cast<uint2*>(sm + mp.lut + e * 256 + 8 * l) = v;
                }
            } else {
                for (int i = tid; i < 64 * 32; i += kNCW * 32) {
                    const int e = i >> 5, l = i & 31;
                    *reinterpret_cast<uint32_t*>(sm + mp.lut + e * 128 + 4 * l) =
                        (uint32_t)rem[e & 7] | ((uint32_t)rem[e >> 3] << 16);
                }
            }
        }
        // q_rot = R q for query (warp) of this group, and alpha * mid * sum(q_rot)
        {
            if (warp < G) {
                apply_signs(x, lane_signs(a.c, lane));
                fwht128(x, lane);
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] *= 0.08838834764831845f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) qrot[warp * D + 4 * lane + i] = x[i];
            const float sq = warp_sum(x[0] + x[1] + x[2] + x[3]);
            // power-of-two scale putting max |alpha q_rot 2^9| / scale in (112, 224]: e4m3 range
            const float mx = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
            const float big = fabsf(a.c.alpha) * 512.f * mx;
            const float scl = (big > 0.f) ? exp2f(ceilf(log2f(big / 224.f))) : 1.f;
            if (lane == 0) {
                qoff[warp] = a.c.alpha * (float)((1 << KB) - 1) * 0.5f * sq;
                qscale[warp] = scl;
            }
        }
        __syncthreads();
        float* sqv = reinterpret_cast<float*>(sm + mp.sq);  // [8][128]: S q_rot per query
        if constexpr (M > 0) {
            // (S q_rot)_i for every query of the group: thread -> row i, queries g0, g0+2, ...
            const int i = tid & (M - 1), g0 = tid / M;
            const float4* srow = reinterpret_cast<const float4*>(a.S + (int64_t)i * D);
            float acc4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int j4 = 0; j4 < D / 4; ++j4) {
                const float4 sv = __ldg(srow + j4);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int gq = g0 + (kNCW * 32 / M) * k;
                    if (gq < 8) {
                        const float4 qv = *reinterpret_cast<const float4*>(qrot + gq * D + 4 * j4);
                        acc4[k] = fmaf(sv.x, qv.x, fmaf(sv.y, qv.y, fmaf(sv.z, qv.z, fmaf(sv.w, qv.w, acc4[k]))));
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int gq = g0 + (kNCW * 32 / M) * k;
                if (gq < 8) sqv[gq * D + i] = acc4[k];
            }
            __syncthreads();
        }

        const int r = lane >> 2, qd = lane & 3;   // r: token row / query column; qd: quad index
        // ---- B fragments (queries as columns): k-step ks, slot s uses pair n = 2ks + s ----
        //   QT:      alpha*q_rot*2^9/scale at the code dims, as four e4m3 terms t_k, the
        //            k-th carrying 16^k x the residual left by the earlier ones (~16 bits)
        //   QB:      q_rot hi at the remainder dims (2n, 2n+1)
        //   QSh/QSl: S q_rot at sign dims (n, n+16), hi + lo (QJL)
        uint32_t QT[4][4][2], QB[8][2];
        uint32_t QSh[M > 0 ? 8 : 1][2], QSl[M > 0 ? 8 : 1][2];
        {
            const float* qr = qrot + r * D + 32 * qd;
            const float al = a.c.alpha * 512.f / qscale[r];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    uint32_t tb[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float res = al * qr[key_fp8_dim<KB>(2 * ks + sl, i)];
                        float mul = 1.f;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t t = f2e4m3(res * mul);
                            res -= e4m3_2f(t) / mul;
                            mul *= 16.f;
                            tb[k] |= t << (8 * i);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) QT[k][ks][sl] = tb[k];
                }
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int n = 2 * ks + sl;
                    QB[ks][sl] = pack_h2(qr[2 * n], qr[2 * n + 1]);
                    if constexpr (M > 0) {
                        const float* sr = sqv + r * D + 32 * qd;
                        split_h2(sr[n], sr[n + 16], QSh[ks][sl], QSl[ks][sl]);
                    }
                }
            }
        }
        const float off0 = qoff[2 * qd], off1 = qoff[2 * qd + 1];
        const float qs0 = qscale[2 * qd], qs1 = qscale[2 * qd + 1];
        const float ksc = a.sm_scale_log2;
        const float cq = 1.2533141373155003f / (float)(M > 0 ? M : 1);  // sqrt(pi/2) / m
        constexpr int KROW = D * KB / 8;

        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
        float acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

        int jdone = 0;  // pages of this warp consumed
        for (int j = 0; j < nmine; ++j) {
            const int pi = warp + kNCW * j;
            const int s = warp * SPW + (j % SPW);
            if (!mbar_wait(bar_full + 8 * s, (j / SPW) & 1)) {
                timed_out = true;
                break;
            }
            const uint32_t pg = ring_base + s * mp.stride;  // shared-space address of the page
            const bool pok = slot_ok[s] != 0;

            // ---------- scores: tokens r (rows 0-7) and r+8 (rows 8-15) ----------
            float sI[4][4], sC[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 4; ++k) sI[k][0] = sI[k][1] = sI[k][2] = sI[k][3] = 0.f;
            {
                uint32_t wa[KB], wb[KB];
                key_words<KB>(pg + g.kcode_off + r * KROW, qd, wa);
                key_words<KB>(pg + g.kcode_off + (r + 8) * KROW, qd, wb);
                uint32_t Ea[8], Eb[8];
                key_bytes<KB>(wa, Ea);
                key_bytes<KB>(wb, Eb);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_e4m3(sI[k], Ea[2 * ks], Eb[2 * ks], Ea[2 * ks + 1], Eb[2 * ks + 1], QT[k][ks][0], QT[k][ks][1]);
                uint32_t Ra[16], Rb[16];
                key_rem<KB>(wa, lut_base, (uint32_t)lane, Ra);
                key_rem<KB>(wb, lut_base, (uint32_t)lane, Rb);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int n = 2 * ks;
                    mma16816(sC, Ra[n], Rb[n], Ra[n + 1], Rb[n + 1], QB[ks][0], QB[ks][1]);
                }
            }
            float iv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                iv[c] = sI[0][c] + 0.0625f * sI[1][c] + 0.00390625f * sI[2][c] + 0.000244140625f * sI[3][c];
            float t0 = fmaf(qs0, iv[0], sC[0] - off0), t1 = fmaf(qs1, iv[1], sC[1] - off1);
            float t2 = fmaf(qs0, iv[2], sC[2] - off0), t3 = fmaf(qs1, iv[3], sC[3] - off1);
            if constexpr (M > 0) {
                float sQ[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t Za[16], Zb[16];
                sign_chunk(lds32(pg + g.sig_off + r * (M / 8) + 4 * qd), Za);
                sign_chunk(lds32(pg + g.sig_off + (r + 8) * (M / 8) + 4 * qd), Zb);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int n = 2 * ks;
                    mma16816(sQ, Za[n], Zb[n], Za[n + 1], Zb[n + 1], QSh[ks][0], QSh[ks][1]);
                    mma16816(sQ, Za[n], Zb[n], Za[n + 1], Zb[n + 1], QSl[ks][0], QSl[ks][1]);
                }
                const float rr = cq * lds_h2f(pg + g.rho_off + 2 * r), rr8 = cq * lds_h2f(pg + g.rho_off + 2 * (r + 8));
                t0 = fmaf(rr, sQ[0], t0); t1 = fmaf(rr, sQ[1], t1);
                t2 = fmaf(rr8, sQ[2], t2); t3 = fmaf(rr8, sQ[3], t3);
            }
            const float gr = lds_h2f(pg + g.gam_off + 2 * r) * ksc, gr8 = lds_h2f(pg + g.gam_off + 2 * (r + 8)) * ksc;
            const int tok = (p0 + pi) * g.bs;
            const bool v_r = pok && (tok + r < len), v_r8 = pok && (tok + r + 8 < len);
            const float s0 = v_r ? t0 * gr : -INFINITY;
            const float s1 = v_r ? t1 * gr : -INFINITY;
            const float s2 = v_r8 ? t2 * gr8 : -INFINITY;
            const float s3 = v_r8 ? t3 * gr8 : -INFINITY;

            // ---------- online softmax ----------
            float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            if (__any_sync(0xffffffffu, n0 > m0 || n1 > m1)) {
                const float f0 = (n0 > m0) ? exp2f(m0 - n0) : 1.f;
                const float f1 = (n1 > m1) ? exp2f(m1 - n1) : 1.f;
                l0 *= f0; z0 *= f0; l1 *= f1; z1 *= f1;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[i][0] *= f0; acc[i][2] *= f0;
                    acc[i][1] *= f1; acc[i][3] *= f1;
                }
                m0 = n0;
                m1 = n1;
            }
            const float b0 = (m0 == -INFINITY) ? 0.f : m0, b1 = (m1 == -INFINITY) ? 0.f : m1;
            const float p0v = exp2f(s0 - b0), p1v = exp2f(s1 - b1), p2v = exp2f(s2 - b0), p3v = exp2f(s3 - b1);
            const float sr = lds_h2f(pg + g.scl_off + 2 * r), sr8 = lds_h2f(pg + g.scl_off + 2 * (r + 8));
            const float zr = lds_h2f(pg + g.zer_off + 2 * r), zr8 = lds_h2f(pg + g.zer_off + 2 * (r + 8));
            l0 += p0v + p2v;
            l1 += p1v + p3v;
            z0 = fmaf(p0v, zr, fmaf(p2v, zr8, z0));
            z1 = fmaf(p1v, zr, fmaf(p3v, zr8, z1));
            // the weights p * scale go in as single fp16 (their rounding costs ~1e-4 of output)
            const uint32_t h01 = pack_h2(p0v * sr, p1v * sr), h23 = pack_h2(p2v * sr8, p3v * sr8);
            const uint32_t bh0 = movtrans(h01), bh1 = movtrans(h23);

            // ---------- values: lane (r, qd) holds dims 16r..16r+15 of tokens 2qd, 2qd+1, 2qd+8, 2qd+9 ----------
            {
                uint32_t Pab[16], Pcd[16];
                value_pair<VB>(pg + g.vcode_off, r, 2 * qd, 2 * qd + 1, Pab);
                value_pair<VB>(pg + g.vcode_off, r, 2 * qd + 8, 2 * qd + 9, Pcd);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)  // rows: dim 16r + 2mt (row r), 16r + 2mt + 1 (row r + 8)
                    mma16816(acc[mt], Pab[2 * mt], Pab[2 * mt + 1], Pcd[2 * mt], Pcd[2 * mt + 1], bh0, bh1);
            }
            __syncwarp();  // every lane has read the slot: refill it with the page SPW ahead
            jdone = j + 1;
            const int jn = j + SPW;
            if (jn < nmine) {
                if ((jn & 31) == 0) {  // next batch of block ids; prefetch the one after it
                    bid_cur = bid_nxt;
                    const int k = 8 * (jn + 32 + lane);
                    bid_nxt = (k < reach) ? __ldg(btw + k) : -1;
                }
                const int bk = __shfl_sync(0xffffffffu, bid_cur, jn & 31);
                if (lane == 0) issue(jn, bk);
            }
        }
        if (timed_out) {
            // copies this warp started must land before its shared memory goes away;
            // one shared deadline for all of them
            const long long t0 = clock64();
            for (int jj = jdone; jj < min(jdone + SPW, nmine); ++jj) {
                const uint32_t bar = bar_full + 8 * (warp * SPW + (jj % SPW));
                while (!mbar_try(bar, (jj / SPW) & 1) && clock64() - t0 < kWaitCycles) {
                }
            }
        }

        // ---- reduce l, z over the 8 token rows, publish warp state ----
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            z0 += __shfl_xor_sync(0xffffffffu, z0, o);
            z1 += __shfl_xor_sync(0xffffffffu, z1, o);
        }
        __syncthreads();  // (A) ring is free: all copies landed, all pages consumed
        float* wst = reinterpret_cast<float*>(ring);                 // [kNCW][8][3]
        float* wacc = reinterpret_cast<float*>(ring) + kNCW * 8 * 3;  // [kNCW][8][128]
        if (r == 0) {
            wst[(warp * 8 + 2 * qd) * 3 + 0] = m0;
            wst[(warp * 8 + 2 * qd) * 3 + 1] = l0;
            wst[(warp * 8 + 2 * qd) * 3 + 2] = z0;
            wst[(warp * 8 + 2 * qd + 1) * 3 + 0] = m1;
            wst[(warp * 8 + 2 * qd + 1) * 3 + 1] = l1;
            wst[(warp * 8 + 2 * qd + 1) * 3 + 2] = z1;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int dim = 16 * r + 2 * mt;
            wacc[(warp * 8 + 2 * qd) * D + dim] = acc[mt][0];
            wacc[(warp * 8 + 2 * qd + 1) * D + dim] = acc[mt][1];
            wacc[(warp * 8 + 2 * qd) * D + dim + 1] = acc[mt][2];
            wacc[(warp * 8 + 2 * qd + 1) * D + dim + 1] = acc[mt][3];
        }
    }
    timed_out = __syncthreads_or(timed_out);  // (B)
    if (timed_out) {
        if (tid == 0) flag(a.status, TQ_FLAG_TIMEOUT);
        return;
    }

    // ---- merge the warps: thread (query warp, lane) owns dims 4 lane .. 4 lane + 3 ----
    const float* wst = reinterpret_cast<const float*>(ring);
    const float* wacc = reinterpret_cast<const float*>(ring) + kNCW * 8 * 3;
    const int qg = warp;  // query of this warp (consumer warps only)
    float Mx = -INFINITY, L = 0.f, O[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < kNCW) {
        for (int w = 0; w < kNCW; ++w) Mx = fmaxf(Mx, wst[(w * 8 + qg) * 3]);
        if (Mx != -INFINITY) {
            float Z = 0.f;
            for (int w = 0; w < kNCW; ++w) {
                const float mw = wst[(w * 8 + qg) * 3];
                if (mw == -INFINITY) continue;
                const float f = exp2f(mw - Mx);
                L = fmaf(f, wst[(w * 8 + qg) * 3 + 1], L);
                Z = fmaf(f, wst[(w * 8 + qg) * 3 + 2], Z);
                const float4 v = *reinterpret_cast<const float4*>(wacc + (w * 8 + qg) * D + 4 * lane);
                O[0] = fmaf(f, v.x, O[0]); O[1] = fmaf(f, v.y, O[1]);
                O[2] = fmaf(f, v.z, O[2]); O[3] = fmaf(f, v.w, O[3]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) O[i] += Z;
        }
    }

    const int64_t unit = (int64_t)b * g.hkv + h;
    bool finalize = (a.num_splits == 1);
    if (!finalize) {
        // publish this split's partial (max, sum, acc with the zero term folded in)
        float* part = a.partials + ((unit * a.num_splits + split) * G) * kPartStride;
        if (warp < G) {
            float* pp = part + qg * kPartStride;
            if (lane == 0) { pp[0] = Mx; pp[1] = L; }
            *reinterpret_cast<float4*>(pp + 4 + 4 * lane) = make_float4(O[0], O[1], O[2], O[3]);
        }
        // The CTA barrier orders every thread's partial writes before thread 0's
        // gpu-scope release (cumulativity); the acquire side pairs with the other
        // CTAs' releases before the last one reads their partials.
        __syncthreads();
        __shared__ int s_last;
        if (tid == 0) {
            unsigned old;
            asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.counters + unit) : "memory");
            s_last = (old == (unsigned)a.num_splits - 1);
        }
        __syncthreads();
        if (!s_last) return;
        finalize = true;
        if (warp < G) {
            // All loads of a chunk of up to kMergeChunk splits are issued before
            // any is used, so a chunk costs one L2 round trip; chunks merge with
            // a running max.
            constexpr int kMergeChunk = 20;
            const float* base = a.partials + (unit * a.num_splits * G) * kPartStride;
            const int ns = a.num_splits;
            float runM = -INFINITY, runL = 0.f;
            O[0] = O[1] = O[2] = O[3] = 0.f;
            for (int s0 = 0; s0 < ns; s0 += kMergeChunk) {
                const int n = min(kMergeChunk, ns - s0);
                float ms = -INFINITY, ls = 0.f;
                if (lane < n) {
                    ms = __ldcg(base + ((s0 + lane) * G + qg) * kPartStride);
                    ls = __ldcg(base + ((s0 + lane) * G + qg) * kPartStride + 1);
                }
                float4 v[kMergeChunk];
#pragma unroll
                for (int k = 0; k < kMergeChunk; ++k)
                    v[k] = (k < n) ? __ldcg(reinterpret_cast<const float4*>(base + ((s0 + k) * G + qg) * kPartStride + 4 + 4 * lane))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                const float nm = fmaxf(runM, warp_max(ms));
                if (nm == -INFINITY) continue;
                const float fr = (runM == -INFINITY) ? 0.f : exp2f(runM - nm);
                const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - nm);
                runL = fmaf(runL, fr, warp_sum(f * ls));
#pragma unroll
                for (int i = 0; i < 4; ++i) O[i] *= fr;
#pragma unroll
                for (int k = 0; k < kMergeChunk; ++k) {
                    const float fk = __shfl_sync(0xffffffffu, f, k);
                    O[0] = fmaf(fk, v[k].x, O[0]); O[1] = fmaf(fk, v[k].y, O[1]);
                    O[2] = fmaf(fk, v[k].z, O[2]); O[3] = fmaf(fk, v[k].w, O[3]);
                }
                runM = nm;
            }
            Mx = runM;
            L = runL;
        }
        if (tid == 0) a.counters[unit] = 0u;
    }
    if (finalize && warp < G) {
        // out = R^T (acc / l) = s (.) H (acc / l) / sqrt(d)
        const float inv = (L > 0.f) ? 1.f / L : 0.f;
        float x[4] = {O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv};
        fwht128(x, lane);
        const uint32_t sg = lane_signs(a.c, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] *= 0.08838834764831845f;
            if ((sg >> i) & 1u) x[i] = -x[i];
        }
        float* o = a.out + ((int64_t)b * a.hq + (int64_t)h * G + qg) * D;
        *reinterpret_cast<float4*>(o + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
    }
}

template <int KB, int VB, int M>
static int launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
    const int smem = smem_map((int)a.g.page_bytes).total;
    auto kern = decode_kernel<KB, VB, M>;
    static int done[64] = {};
    cudaError_t e = ensure_smem_limit(kern, smem, done);
    if (e != cudaSuccess) return (int)e;
    dim3 grid((unsigned)a.num_splits, (unsigned)a.g.hkv, (unsigned)a.batch);
    kern<<<grid, kThreads, smem, s>>>(a);
    return (int)cudaGetLastError();
}

int launch_decode(const DecodeArgs& a, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int kb = a.g.kb, vb = a.g.vb, m = a.g.m;
#define TQ_DEC(KB_, VB_)                                                                          \
    if (kb == KB_ && vb == VB_)                                                                   \
        return m ? launch_decode_t<KB_, VB_, 128>(a, s) : launch_decode_t<KB_, VB_, 0>(a, s);
    TQ_DEC(2, 2) TQ_DEC(2, 3) TQ_DEC(2, 4)
    TQ_DEC(3, 2) TQ_DEC(3, 3) TQ_DEC(3, 4)
    TQ_DEC(4, 2) TQ_DEC(4, 3) TQ_DEC(4, 4)
#undef TQ_DEC
    return (int)cudaErrorNotSupported;
}

}  // namespace tq

// ===========================================================================
// Decode without any device allocation by the caller or the library.
//
// Some callers cannot call cudaMalloc at the point where they decode: an
// inference engine that pre-plans all of its device memory up front, code
// running inside a memory pool it does not own, or a host that forbids
// allocations on the serving path because they can synchronise the device.
// For them this entry point uses a fixed scratch area that is part of the
// library image itself (a file-scope __device__ array), sized
// TQ_NOALLOC_WORKSPACE_BYTES.  Every device that loads the library keeps that
// memory until the process exits.
// ===========================================================================
#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_noalloc_workspace[TQ_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Host code only
// holds a stand-in for the array's name; the real address comes from the
// runtime, looked up once per device with that device current.
tq_status noalloc_workspace(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        tq::set_error("cudaGetDevice: %s", cudaGetErrorString(e));
        return TQ_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        tq::set_error("device ordinal %d is beyond the %d devices this entry point tracks", dev, kMaxDevices);
        return TQ_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess || !p) {
            tq::set_error("cudaGetSymbolAddress of the fixed decode workspace: %s", cudaGetErrorString(e));
            return TQ_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return TQ_OK;
}

}  // namespace

extern "C" TQ_API tq_status tq_decode_attention_noalloc(const tq_cache* cache, const void* q, tq_dtype dtype,
                                                        int batch, int num_q_heads, const int32_t* block_table,
                                                        int max_blocks_per_seq, const int32_t* lens, float sm_scale,
                                                        float* out, int32_t* dev_status, void* stream) {
    if (!cache) {
        tq::set_error("cache is NULL");
        return TQ_ERR_INVALID_ARG;
    }
    if (batch == 0) return TQ_OK;
    const size_t need = tq_decode_workspace_bytes(cache, batch, num_q_heads, max_blocks_per_seq);
    if (need == 0) {
        tq::set_error("bad batch / num_q_heads / max_blocks_per_seq");
        return TQ_ERR_INVALID_ARG;
    }
    if (need > (size_t)TQ_NOALLOC_WORKSPACE_BYTES) {
        tq::set_error("this batch shape needs %zu bytes of decode workspace, more than the %zu bytes of the "
                      "fixed workspace; use tq_decode_attention with a workspace of your own",
                      need, (size_t)TQ_NOALLOC_WORKSPACE_BYTES);
        return TQ_ERR_WORKSPACE;
    }
    void* ws = nullptr;
    tq_status st = noalloc_workspace(&ws);
    if (st != TQ_OK) return st;
    // The split counters sit at the end of the workspace and must start at
    // zero; the array keeps whatever the previous call left, so clear them.
    const size_t counters = (size_t)batch * cache->g.hkv * sizeof(unsigned);
    const size_t counters_region = (counters + 255) / 256 * 256;
    cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(ws) + (need - counters_region), 0, counters,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        tq::set_error("clearing the fixed workspace counters: %s", cudaGetErrorString(e));
        return TQ_ERR_CUDA;
    }
    return tq_decode_attention(cache, q, dtype, batch, num_q_heads, block_table, max_blocks_per_seq, lens, sm_scale,
                               out, ws, need, dev_status, stream);
}
