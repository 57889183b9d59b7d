// Decode attention over the compressed paged cache (split-K flash decode).
//
// Grid (split, KV head, sequence); one CTA per SM.
//  - Every warp takes every NW-th page of its split (one page = 16 tokens of
//    one KV head, contiguous) and streams it into its own shared-memory ring
//    slots with 1-D bulk async copies (cp.async.bulk) completing on mbarriers.
//  - Per page, for the G <= 8 query heads of the group (queries as the n8 side
//    of mma.sync, tokens as rows):
//      scores  the key centroid is split into an exactly representable part
//              and a small remainder, each multiplied on mma.sync m16n8k16 with
//              fp32 accumulation:
//              - 4-bit keys: C[c] = delta N[c] + rem2[c] with N[c] an integer of
//                magnitude <= 2047 (exact in fp16) and |rem2[c]| <= delta / 2;
//                both come, for the two codes of a code byte, from one 8-byte
//                load of a lane-private shared-memory table; N multiplies
//                delta*q_rot split into fp16 hi + lo, rem2 multiplies q_rot.
//              - other widths: C[c] = alpha (c - mid) + rem[c].  The integer
//                code c, masked in place inside a 16-bit lane, is the exact fp16
//                subnormal c * 2^-e; it multiplies alpha*q_rot split into fp16
//                hi + lo parts that carry the matching 2^(e-24), so all
//                products share one scale.  rem[c] comes in fp16 from the
//                lane-private table and multiplies q_rot.
//              logit = gamma_t * sm_scale * (sum_j C[c_j] q_rot[j]) [+ QJL term]
//      softmax running max / sum per query in the exp2 domain; the max is
//              raised (and the state rescaled) only when a score beats it by
//              more than 8 (log2), which after the first page is rare
//      values  O^T[128 x 8 q] += Vcode^T[128 x 16 tok] . (p * scale)^T[16 tok x 8 q]
//              (m16n8k16).  A value code masked in place inside a 16-bit lane is
//              an exact fp16 subnormal c * 2^-e; the power of two is removed once
//              at the end.  The zero-point term sum_t p_t zero_t is kept in fp32.
//    Keys are never reconstructed; everything stays in the rotated frame
//    ["OCTOPUS ..." -- TL;DR / step 7; deep dive -- [RHT effect]: inner
//    products are preserved by the rotation].
//  - Warps merge in shared memory; a sequence split over several CTAs writes
//    partials (max, sum, acc) and the last CTA to finish (atomic counter)
//    merges them and applies the one inverse rotation R^T = diag(s) H / sqrt(d).
// Attention itself: softmax(q K^T / sqrt(d_h)) V [Bit-Axon -- attention under
// quantized KV].
#pragma once
#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_tcgen05.cuh"

namespace tq {

constexpr int kMaxSlotsPerWarp = 8;            // ring slots per warp: pages a warp keeps in flight
constexpr int kFirstPages = 2;                 // pages per warp requested before the query is prepared
constexpr int kQStride = kHeadDim + 4;         // padded row of q_rot / S q_rot in shared memory (float4-aligned)
constexpr uint32_t kLutAddr = 0x10000;         // shared-window address of the remainder table
constexpr int kLutBytes = 0x10000;
constexpr int kMaxSmemBase = 4096;             // dynamic shared memory must start below this address
constexpr int kSmemLimit = 227 * 1024;         // opt-in dynamic shared memory per CTA
constexpr long long kWaitCycles = 3000000000ll;  // bound on any wait: ~1.5 s at 2 GHz
constexpr float kMinusBig = -1.0e30f;          // running max before any token (finite: no inf - inf)
// stage of the appended token in shared memory: key row, value row (up to 128 B
// each), gamma / scale / zero / rho, the barrier that hands it to the page's
// owner, a barrier nothing arrives on (the wait-timeout test hook waits on it),
// and the QJL sign row (m / 8 = 16 bytes)
constexpr int kStageValue = 128, kStageMeta = 256, kStageBar = 272, kStageNever = 280, kStageSig = 288,
              kStageBytes = 304;
// The running max is raised only when a score beats it by more than kLazy (log2
// units), so weights stay below 2^kLazy (any reference max gives the same
// softmax).  A page whose value scale exceeds kBigScale takes the exact max, so
// that p * scale stays inside the fp16 range of the PV operand.
constexpr float kLazy = 8.f;
constexpr float kBigScale = 255.f;
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
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, long long limit) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try(bar, parity)) return true;
        if (clock64() - t0 > limit) return false;
    }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, kWaitCycles);
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// Programmatic dependent launch: wait for the grid this one depends on (a
// no-op when launched without the attribute); allow the next grid to launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
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
__device__ __forceinline__ uint32_t movtrans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
// D = A . B + C, m16n8k16, fp16 operands, fp32 accumulate
__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// the same with the accumulator's starting value given separately
__device__ __forceinline__ void mma16816_c(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}
// 2^x with the hardware approximation (relative error ~2^-22; -inf gives 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// page format and shared memory map, both fixed at compile time per format
// ---------------------------------------------------------------------------
template <int KB, int VB, int M>
struct PageFmt {
    static constexpr int kcode = 0;
    static constexpr int vcode = kBlockSize * kHeadDim * KB / 8;
    static constexpr int gam = vcode + kBlockSize * kHeadDim * VB / 8;
    static constexpr int scl = gam + 2 * kBlockSize;
    static constexpr int zer = scl + 2 * kBlockSize;
    static constexpr int rho = zer + 2 * kBlockSize;
    static constexpr int sig = rho + (M ? 2 * kBlockSize : 0);
    static constexpr int bytes = (sig + kBlockSize * M / 8 + 15) / 16 * 16;
    static constexpr int stride = (bytes + 127) / 128 * 128;  // ring slot size
};

// Warps per CTA: the QJL sign term needs 32 more registers of query fragments.
template <int M>
__host__ __device__ constexpr int decode_warps() { return M ? 8 : 12; }

// Per-lane query fragments (uint4 vectors): 8 of fp16 hi/lo alpha q_rot at the
// code dims, 4 of fp16 q_rot at the remainder dims, 8 of fp16 hi/lo S q_rot for
// the QJL term.
template <int M>
__host__ __device__ constexpr int frag_vecs() { return 8 + 4 + (M ? 8 : 0); }

struct Layout {
    int frag, qrot, sq, qoff, qscale, rem, stage, bars, ok;  // small fixed region at the start
    int ringA, nwA;   // ring slots of warps 0 .. nwA-1 sit below the remainder table
    int spw;          // ring slots per warp
    int total;        // dynamic bytes to request: enough for any start address up to kMaxSmemBase
};

// The remainder table must sit at shared address kLutAddr (its entry index then
// drops straight into bits 8..15 of the lookup address).  Ring slots of the
// first warps fill the space below it, the rest follow it.
template <int KB, int VB, int M>
__host__ __device__ constexpr Layout decode_layout() {
    constexpr int NW = decode_warps<M>();
    Layout L{};
    int off = 0;
    L.frag = off; off += 32 * 16 * frag_vecs<M>();
    L.qrot = off; off += 8 * kQStride * 4;
    L.sq = off; off += M ? 8 * kQStride * 4 : 0;
    L.qoff = off; off += 8 * 4;
    L.qscale = off; off += 8 * 4;
    L.rem = off; off += 3 * 16 * 2;  // rem | N | rem2 (4-bit keys) in binary16
    L.stage = off; off += kStageBytes;  // appended token (see kStage*)
    L.bars = off; off += 8 * NW * kMaxSlotsPerWarp;
    L.ok = off; off += 4 * NW * kMaxSlotsPerWarp;
    L.ringA = (off + 127) / 128 * 128;
    const int stride = PageFmt<KB, VB, M>::stride;
    const int capA = (int)kLutAddr - kMaxSmemBase - L.ringA;
    for (int spw = kMaxSlotsPerWarp; spw >= 1; --spw) {
        const int per = spw * stride;
        const int nA = capA / per < NW ? capA / per : NW;
        const int total = (int)kLutAddr + kLutBytes + (NW - nA) * per;  // start address 0 is the worst case
        // the warp merge reuses the space from the table on: states + accumulators
        const int merge_end = (int)kLutAddr + 2048 + NW * 8 * kHeadDim * 4;
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

// ---------------------------------------------------------------------------
// code unpacking
// ---------------------------------------------------------------------------
// bits [pos, pos + n) of a little-endian multi-word bit string (pos, n compile-time after unrolling)
template <int NW>
__device__ __forceinline__ uint32_t bits_at(const uint32_t (&w)[NW], int pos, int n) {
    const int wi = pos >> 5, sh = pos & 31;
    uint32_t x = (sh + n <= 32 || wi + 1 >= NW) ? (w[wi] >> sh) : __funnelshift_r(w[wi], w[wi + 1], sh);
    return x & ((1u << n) - 1u);
}

// Key chunk of one token: the 32 codes of one 32-dim chunk (4*KB bytes).
template <int KB>
__device__ __forceinline__ void key_words(uint32_t addr, uint32_t (&w)[KB]) {
    if constexpr (KB == 4) {
        const uint4 v = lds128(addr);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (KB == 2) {
        const uint2 v = lds64(addr);
        w[0] = v.x; w[1] = v.y;
    } else if constexpr (KB == 8) {
        const uint4 v = lds128(addr), u = lds128(addr + 16);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        w[4] = u.x; w[5] = u.y; w[6] = u.z; w[7] = u.w;
    } else {
#pragma unroll
        for (int i = 0; i < KB; ++i) w[i] = lds32(addr + 4 * i);
    }
}

// The integer codes as fp16 A operands.  A code c masked in place inside a
// 16-bit half, below bit 10, is the exact subnormal c * 2^-24 shifted by its
// bit position, so only masks (and one shift per word) are needed.  X[n] holds
// two codes of the lane's 32-dim chunk: element h (0 low, 1 high) is chunk dim
// key_dim<KB>(n, h), scaled by 2^-key_exp<KB>(n).  MMA k-step ks uses X[2ks]
// (k = 2qd, 2qd+1) and X[2ks+1] (k = 8+2qd, 8+2qd+1).
//
// 4-bit keys instead take the centroid's integer part N[c] (C[c] = delta N[c]
// + rem2[c], |N| <= 2047, exact in fp16 at unit scale) from the lookup table
// together with rem2, for the code pair of one code byte: X[n] holds chunk
// dims (2n, 2n+1) (key_lut4 below).
template <int KB>
__host__ __device__ constexpr int key_dim(int n, int h) {
    return KB == 2 ? 16 * (n >> 3) + (n & 7) + 8 * h : 2 * n + h;
}
template <int KB>
__host__ __device__ constexpr int key_exp(int n) {
    return KB == 2 ? 24 - 2 * (n & 3) : 24;
}
// Scale of the integer part's MMA result: 2^24 undoes the subnormal code
// operands, 4-bit integer parts are unit-scale fp16.
template <int KB>
__host__ __device__ constexpr float key_int_scale() {
    return KB == 4 ? 1.f : 16777216.f;
}

template <int KB>
__device__ __forceinline__ void key_halves(const uint32_t (&w)[KB], uint32_t X[16]) {
    static_assert(KB != 4, "4-bit keys take their operands from key_lut4");
    if constexpr (KB == 2) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t y = w[i] >> 8;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                X[8 * i + m] = w[i] & (0x00030003u << (2 * m));
                X[8 * i + 4 + m] = y & (0x00030003u << (2 * m));
            }
        }
    } else if constexpr (KB == 8) {
        // codes 2n, 2n+1 are bytes 2(n&1), 2(n&1)+1 of word n/2: one byte permute
#pragma unroll
        for (int n = 0; n < 16; ++n) X[n] = prmt(w[n >> 1], 0u, (n & 1) ? 0x4342u : 0x4140u);
    } else {
        // any other width: the two codes as one 2 KB-bit field, split into the halves
        constexpr uint32_t mask = (1u << KB) - 1u;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const uint32_t x = bits_at<KB>(w, 2 * KB * n, 2 * KB);
            X[n] = (x & mask) | ((x >> KB) << 16);
        }
    }
}

// Remainder operands R[n] = (rem[c_{2n}], rem[c_{2n+1}]) from the lane-private
// table at kLutAddr.  lw = kLutAddr | lane offset; for 2- and 4-bit keys a code
// byte is the entry index and is dropped into bits 8..15 of the address with
// one byte permute.
template <int KB>
__device__ __forceinline__ void key_rem(const uint32_t (&w)[KB], uint32_t lw, uint32_t R[16]) {
    static_assert(KB != 4, "4-bit keys take their operands from key_lut4");
    if constexpr (KB == 2) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint2 v = lds64(prmt(w[j >> 2], lw, 0x7604u | ((uint32_t)(j & 3) << 4)));
            R[2 * j] = v.x;
            R[2 * j + 1] = v.y;
        }
    } else if constexpr (KB == 8) {
        // one code per byte, entries of 256 B holding (rem[c], rem[c]): the code
        // byte drops into bits 8..15 of the address as for 4-bit keys
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const uint32_t k0 = 2 * (n & 1);
            const uint32_t r0 = lds32(prmt(w[n >> 1], lw, 0x7604u | (k0 << 4)));
            const uint32_t r1 = lds32(prmt(w[n >> 1], lw, 0x7604u | ((k0 + 1) << 4)));
            R[n] = prmt(r0, r1, 0x5410u);
        }
    } else if constexpr (KB >= 5) {
        // one code per entry of 128 B holding (rem[c], rem[c])
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const uint32_t r0 = lds32(lw | (bits_at<KB>(w, 2 * KB * n, KB) << 7));
            const uint32_t r1 = lds32(lw | (bits_at<KB>(w, 2 * KB * n + KB, KB) << 7));
            R[n] = prmt(r0, r1, 0x5410u);
        }
    } else {
        // 1- and 3-bit keys: two codes per entry of 128 B holding (rem[c0], rem[c1])
#pragma unroll
        for (int n = 0; n < 16; ++n) R[n] = lds32(lw | (bits_at<KB>(w, 2 * KB * n, 2 * KB) << 7));
    }
}

// 4-bit keys: both operands of code byte n of the lane's chunk (codes 2n, 2n+1)
// with one 8-byte load: (N[c0], N[c1]) and (rem2[c0], rem2[c1]) in fp16.  The
// table has 256-byte entries (8 bytes per lane), so the code byte is the
// address's bits 8..15, put there with one byte permute.
__device__ __forceinline__ uint2 key_lut4(const uint32_t (&w)[4], uint32_t lw, int n) {
    return lds64(prmt(w[n >> 2], lw, 0x7604u | ((uint32_t)(n & 3) << 4)));
}

// Value codes of dims 16r .. 16r+15 for a token pair (ta, tb): P[i] holds the
// codes of dim 16r + i for ta (low half) and tb (high half) as fp16 subnormals
// code * 2^-value_exp<VB>(i), exact.
template <int VB>
__host__ __device__ constexpr int value_exp(int i) {
    return VB == 4 ? ((i & 1) ? 20 : 24) : VB == 2 ? 24 - 2 * (i & 3) : 24;
}
template <int VB>
__device__ __forceinline__ void value_codes(uint32_t vbase, int r, int ta, int tb, uint32_t P[16]) {
    constexpr int ROW = kHeadDim * VB / 8;
    if constexpr (VB == 4) {
        const uint2 va = lds64(vbase + ta * ROW + r * 8);
        const uint2 vb = lds64(vbase + tb * ROW + r * 8);
        const uint32_t x[4] = {prmt(va.x, vb.x, 0x5410u), prmt(va.x, vb.x, 0x7632u), prmt(va.y, vb.y, 0x5410u),
                               prmt(va.y, vb.y, 0x7632u)};
#pragma unroll
        for (int hq = 0; hq < 4; ++hq) {
            P[4 * hq + 0] = x[hq] & 0x000F000Fu;
            P[4 * hq + 1] = x[hq] & 0x00F000F0u;
            P[4 * hq + 2] = (x[hq] >> 8) & 0x000F000Fu;
            P[4 * hq + 3] = (x[hq] >> 8) & 0x00F000F0u;
        }
    } else if constexpr (VB == 2) {
        const uint32_t wa = lds32(vbase + ta * ROW + r * 4);
        const uint32_t wb = lds32(vbase + tb * ROW + r * 4);
        const uint32_t x[2] = {prmt(wa, wb, 0x5410u), prmt(wa, wb, 0x7632u)};
#pragma unroll
        for (int hq = 0; hq < 2; ++hq)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t y = (i < 4) ? x[hq] : (x[hq] >> 8);
                P[8 * hq + i] = y & (0x00030003u << (2 * (i & 3)));
            }
    } else {
        // any other width: the 16 codes are bytes 2 VB r .. 2 VB r + 2 VB - 1 of
        // the token's row, which starts on an even byte
        constexpr int NWV = (2 * VB + ((VB & 1) ? 2 : 0) + 3) / 4;  // 32-bit words spanning them
        const int base = (2 * VB * r) & ~3, sh = ((2 * VB * r) & 3) * 8;
        uint32_t a[NWV], bw[NWV], xa[NWV], xb[NWV];
#pragma unroll
        for (int k = 0; k < NWV; ++k) {
            a[k] = lds32(vbase + ta * ROW + base + 4 * k);
            bw[k] = lds32(vbase + tb * ROW + base + 4 * k);
        }
#pragma unroll
        for (int k = 0; k < NWV; ++k) {
            xa[k] = (k + 1 < NWV) ? __funnelshift_r(a[k], a[k + 1], sh) : (a[k] >> sh);
            xb[k] = (k + 1 < NWV) ? __funnelshift_r(bw[k], bw[k + 1], sh) : (bw[k] >> sh);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) P[i] = bits_at<NWV>(xa, VB * i, VB) | (bits_at<NWV>(xb, VB * i, VB) << 16);
    }
}

// Value widths above 4 bits give small scales, so that the PV weights
// p * scale would sit near the fp16 subnormal range; they are taken times
// 2^value_wshift (and the power removed with the code's own at the end).
template <int VB>
__host__ __device__ constexpr int value_wshift() {
    return VB > 4 ? VB - 4 : 0;
}

// QJL sign bits of one token (bits 32qd .. 32qd+31 of its sigma row):
// Z[n] = (+-1 for bit n, +-1 for bit n+16) in fp16.
__device__ __forceinline__ void sign_chunk(uint32_t w, uint32_t Z[16]) {
#pragma unroll
    for (int n = 0; n < 16; ++n) Z[n] = ((w << (15 - n)) & 0x80008000u) ^ 0xBC00BC00u;
}

// ---------------------------------------------------------------------------
// append: one warp encodes the new token of (sequence, KV head) exactly as the
// encode kernel does with one warp per token (lane l holds coordinates
// 4l .. 4l+3), writes it into its page in the pool and keeps a staged copy
// (key row, value row, gamma / scale / zero at kStage*) that the page's owner
// patches into its shared-memory copy of the page before consuming it.
// ["TurboQuant: KV Cache Vector Quantization" -- three steps; deep dive --
//  Step 1 (RHT), Step 3 (value codes); "OCTOPUS ..." -- methodology step 8]
// ---------------------------------------------------------------------------
template <int B>
__device__ __forceinline__ void store_row_both(uint8_t* g, uint8_t* st, uint32_t p, int lane) {
    if constexpr (B == 4) {
        reinterpret_cast<uint16_t*>(g)[lane] = (uint16_t)p;
        reinterpret_cast<uint16_t*>(st)[lane] = (uint16_t)p;
    } else if constexpr (B == 2) {
        g[lane] = (uint8_t)p;
        st[lane] = (uint8_t)p;
    } else if constexpr (B == 8) {
        reinterpret_cast<uint32_t*>(g)[lane] = p;
        reinterpret_cast<uint32_t*>(st)[lane] = p;
    } else {
        const uint32_t w = row_word<B>(p, lane);
        if (lane < 4 * B) {
            reinterpret_cast<uint32_t*>(g)[lane] = w;
            reinterpret_cast<uint32_t*>(st)[lane] = w;
        }
    }
}

// Raw bits of elements i .. i+3 of a row: one 8-byte load for 16-bit types,
// two for fp32.  Nothing here uses the loaded registers, so the warp does not
// wait for them until cvt4 converts them.
__device__ __forceinline__ void raw4(const void* base, int dtype, int64_t i, uint32_t r[4]) {
    const int f32 = dtype == TQ_F32;
    const char* p = reinterpret_cast<const char*>(base) + i * (f32 ? 4 : 2);
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.s32 q, %5, 0;\n"
        " ld.global.nc.v2.u32 {%0, %1}, [%4];\n"
        " @q ld.global.nc.v2.u32 {%2, %3}, [%4+8];\n}\n"
        : "=r"(r[0]), "=r"(r[1]), "+r"(r[2]), "+r"(r[3])
        : "l"(p), "r"(f32));
}
__device__ __forceinline__ void cvt4(const uint32_t r[4], int dtype, float x[4]) {
    if (dtype == TQ_F32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __uint_as_float(r[i]);
    } else if (dtype == TQ_BF16) {
        x[0] = __uint_as_float(r[0] << 16);
        x[1] = __uint_as_float(r[0] & 0xFFFF0000u);
        x[2] = __uint_as_float(r[1] << 16);
        x[3] = __uint_as_float(r[1] & 0xFFFF0000u);
    } else {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&r[0]));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&r[1]));
        x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
    }
}

// Warp sum in the order the encode kernel's one-warp layout uses (strides 1, 2,
// .. 16), so that the appended token's bytes equal what tq_encode_kv writes.
__device__ __forceinline__ float warp_sum_up(float v) {
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// kraw, vraw: raw4 bits of this lane's coordinates 4 lane .. 4 lane + 3 of the new token
template <int KB, int VB, int M>
__device__ void append_token(const DecodeArgs& a, uint8_t* page, int off, uint8_t* stage, int lane,
                             const uint32_t kraw[4], const uint32_t vraw[4]) {
    using F = PageFmt<KB, VB, M>;
    constexpr int D = kHeadDim;
    constexpr int HALF = 1 << (KB - 1), VMAX = (1 << VB) - 1;
    float k[4], v[4];
    cvt4(kraw, a.kv_dtype, k);
    cvt4(vraw, a.kv_dtype, v);
    float z = 0.f, ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        z = fmaf(k[i], 0.f, fmaf(v[i], 0.f, z));  // x * 0 is 0 for finite x, NaN for inf / NaN
        ss = fmaf(k[i], k[i], ss);
    }
    const bool finite = (warp_sum(z) == 0.f);
    if (!finite && lane == 0) flag(a.status, TQ_FLAG_NONFINITE);
    const float gamma = sqrtf(warp_sum_up(ss));
    const uint32_t sg = lane_signs(a.c, lane);
    apply_signs(k, sg);
    fwht128(k, lane);
    uint32_t kp = 0;
    float rsd[4] = {0.f, 0.f, 0.f, 0.f};  // QJL: residual r = u_rot - C[code] in the unit frame
    if constexpr (KB <= 4) {
        const KeyThresholds<KB> kt(a.c, gamma);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = (gamma > 0.f) ? kt.code(k[i]) : HALF - 1;
            kp |= (uint32_t)c << (KB * i);
            if constexpr (M > 0) {
                if (gamma > 0.f) {
                    const float u = (k[i] * 0.08838834764831845f) / gamma;
                    float cv = 0.f;
#pragma unroll
                    for (int bb = 0; bb < (1 << KB); ++bb) cv = (c == bb) ? a.c.centroid[bb] : cv;
                    rsd[i] = u - cv;
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = (gamma > 0.f) ? key_code_search<KB>(k[i], gamma, a.tab->boundary_sd_pos) : HALF - 1;
            kp |= (uint32_t)c << (KB * i);
        }
    }
    apply_signs(v, sg);
    fwht128(v, lane);
    float lo = 3.4e38f, hi = -3.4e38f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] *= 0.08838834764831845f;
        lo = fminf(lo, v[i]);
        hi = fmaxf(hi, v[i]);
    }
    const float mn = warp_min(lo), mx = warp_max(hi);
    const float scale = (mx - mn) / (float)VMAX;
    uint32_t vp = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float qv = (scale > 0.f) ? fminf(fmaxf(rintf((v[i] - mn) / scale), 0.f), (float)VMAX) : 0.f;
        vp |= (uint32_t)qv << (VB * i);
    }
    store_row_both<KB>(page + F::kcode + off * (D * KB / 8), stage, kp, lane);
    store_row_both<VB>(page + F::vcode + off * (D * VB / 8), stage + kStageValue, vp, lane);
    uint16_t hr = 0;
    if constexpr (M > 0) {
        // rho = ||r||; sigma_i = [(S r)_i >= 0] with the encode kernel's arithmetic
        // (one warp, four coordinates per lane): per chunk of 32 rows every lane
        // forms the partial dot products over its coordinates, a butterfly sums
        // them so that lane l ends with row 32 ch + l, and the bits are OR-ed
        // into words.  ["OCTOPUS ..." -- contribution "Optional 1-bit QJL
        // residual"; methodology step 8]
        float rr = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) rr = fmaf(rsd[i], rsd[i], rr);
        const float rho = sqrtf(warp_sum_up(rr));
        hr = f16_bits(rho);
        const float4* S4 = reinterpret_cast<const float4*>(a.S) + lane;  // row i: S4[32 i]
        uint32_t wb[M / 32];
#pragma unroll
        for (int ch = 0; ch < M / 32; ++ch) {
            float pr[32];
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {
                const float4 sv = __ldg(S4 + (ch * 32 + kk) * 32);
                pr[kk] = fmaf(sv.x, rsd[0], fmaf(sv.y, rsd[1], fmaf(sv.z, rsd[2], fmaf(sv.w, rsd[3], 0.f))));
            }
#pragma unroll
            for (int m = 16, half = 16; m >= 1; m >>= 1, half >>= 1) {
                const bool up = (lane & m) != 0;
#pragma unroll
                for (int kk = 0; kk < half; ++kk) {
                    const float keep = up ? pr[kk + half] : pr[kk];
                    const float give = up ? pr[kk] : pr[kk + half];
                    pr[kk] = keep + __shfl_xor_sync(0xffffffffu, give, m);
                }
            }
            wb[ch] = __ballot_sync(0xffffffffu, pr[0] >= 0.f);
        }
        if (lane < M / 32) {
            uint32_t word = wb[0];
#pragma unroll
            for (int ch = 1; ch < M / 32; ++ch) word = (lane == ch) ? wb[ch] : word;
            if (!(gamma > 0.f)) word = 0xffffffffu;
            reinterpret_cast<uint32_t*>(page + F::sig + off * (M / 8))[lane] = word;
            reinterpret_cast<uint32_t*>(stage + kStageSig)[lane] = word;
        }
    }
    if (lane == 0) {
        const uint16_t hg = f16_bits(gamma), hs = f16_bits(scale), hz = f16_bits(mn);
        reinterpret_cast<uint16_t*>(page + F::gam)[off] = hg;
        reinterpret_cast<uint16_t*>(page + F::scl)[off] = hs;
        reinterpret_cast<uint16_t*>(page + F::zer)[off] = hz;
        uint16_t* sm3 = reinterpret_cast<uint16_t*>(stage + kStageMeta);
        sm3[0] = hg; sm3[1] = hs; sm3[2] = hz;
        bool ovf = ((hg & 0x7FFF) == 0x7C00) || ((hs & 0x7FFF) == 0x7C00) || ((hz & 0x7FFF) == 0x7C00);
        if constexpr (M > 0) {
            reinterpret_cast<uint16_t*>(page + F::rho)[off] = hr;
            sm3[3] = hr;
            ovf = ovf || ((hr & 0x7FFF) == 0x7C00);
        }
        if (ovf && finite) flag(a.status, TQ_FLAG_OVERFLOW);
    }
    __syncwarp();
}

// Copy the staged token into slot `off` of the shared-memory page at `pg`.
template <int KB, int VB, int M>
__device__ __forceinline__ void patch_page(uint8_t* pg, int off, const uint8_t* stage, int lane) {
    using F = PageFmt<KB, VB, M>;
    constexpr int KROW = kHeadDim * KB / 8, VROW = kHeadDim * VB / 8;
    if (lane < KROW / 4)
        reinterpret_cast<uint32_t*>(pg + F::kcode + off * KROW)[lane] = reinterpret_cast<const uint32_t*>(stage)[lane];
    if (lane < VROW / 4)
        reinterpret_cast<uint32_t*>(pg + F::vcode + off * VROW)[lane] = reinterpret_cast<const uint32_t*>(stage + kStageValue)[lane];
    if (lane == 0) {
        const uint16_t* sm3 = reinterpret_cast<const uint16_t*>(stage + kStageMeta);
        reinterpret_cast<uint16_t*>(pg + F::gam)[off] = sm3[0];
        reinterpret_cast<uint16_t*>(pg + F::scl)[off] = sm3[1];
        reinterpret_cast<uint16_t*>(pg + F::zer)[off] = sm3[2];
        if constexpr (M > 0) reinterpret_cast<uint16_t*>(pg + F::rho)[off] = sm3[3];
    }
    if constexpr (M > 0) {
        if (lane < M / 32)
            reinterpret_cast<uint32_t*>(pg + F::sig + off * (M / 8))[lane] =
                reinterpret_cast<const uint32_t*>(stage + kStageSig)[lane];
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// One page's online softmax and PV contraction for lane (r, qd) of a warp:
// t0..t3 are the lane's logits in log2 units before the key norm (rows r and
// r + 8, i.e. slots tr and tr + 8; queries 2qd and 2qd + 1), tok the sequence
// position of the page's first slot.  Values: O^T[128 x 8 q] += Vcode^T[128 x 16
// tok] . (p * scale)^T[16 tok x 8 q] on mma.sync m16n8k16 (lane (r, qd) holds
// dims 16r..16r+15 of the tokens of rows 2qd, 2qd+1, 2qd+8, 2qd+9).
// ---------------------------------------------------------------------------
template <int KB, int VB, int M>
__device__ __forceinline__ void softmax_pv_page(uint32_t pg, bool pok, int tok, int len, float t0, float t1, float t2,
                                                float t3, int r, int tr, int ta, int tb, float& m0, float& m1,
                                                float& l0, float& l1, float& z0, float& z1, float (&acc)[8][4]) {
    using F = PageFmt<KB, VB, M>;
    const float gr = lds_h2f(pg + F::gam + 2 * tr), gr8 = lds_h2f(pg + F::gam + 2 * (tr + 8));
    float s0 = t0 * gr, s1 = t1 * gr, s2 = t2 * gr8, s3 = t3 * gr8;
    // the sequence's last page or a skipped one (warp-uniform): rows past
    // the end get no weight, and the scale and zero of their slots (never
    // written: any bytes, NaN included) are replaced by 0
    const bool tail = !pok || tok + kBlockSize > len;
    const bool v0 = pok && tok + tr < len, v8 = pok && tok + tr + 8 < len;
    if (tail) {
        if (!v0) s0 = s1 = -INFINITY;
        if (!v8) s2 = s3 = -INFINITY;
    }

    // ---------- online softmax; the max moves only when a score beats it by kLazy ----------
    float sr = lds_h2f(pg + F::scl + 2 * tr), sr8 = lds_h2f(pg + F::scl + 2 * (tr + 8));
    if (tail) {
        sr = v0 ? sr : 0.f;
        sr8 = v8 ? sr8 : 0.f;
    }
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
    constexpr float kWScale = (float)(1 << value_wshift<VB>());
    const bool exact = fmaxf(sr, sr8) > kBigScale / kWScale;
    if (__any_sync(0xffffffffu, mx0 > m0 + kLazy || mx1 > m1 + kLazy || (exact && (mx0 > m0 || mx1 > m1)))) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float f0 = ex2(m0 - n0), f1 = ex2(m1 - n1);
        l0 *= f0; z0 *= f0; l1 *= f1; z1 *= f1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc[i][0] *= f0; acc[i][2] *= f0;
            acc[i][1] *= f1; acc[i][3] *= f1;
        }
        m0 = n0;
        m1 = n1;
    }
    const float p0v = ex2(s0 - m0), p1v = ex2(s1 - m1), p2v = ex2(s2 - m0), p3v = ex2(s3 - m1);
    float zr = lds_h2f(pg + F::zer + 2 * tr), zr8 = lds_h2f(pg + F::zer + 2 * (tr + 8));
    if (tail) {
        zr = v0 ? zr : 0.f;
        zr8 = v8 ? zr8 : 0.f;
    }
    l0 += p0v + p2v;
    l1 += p1v + p3v;

    // ---------- values: lane (r, qd) holds dims 16r..16r+15 of the tokens of rows 2qd, 2qd+1, 2qd+8, 2qd+9 ----------
    // The weights w = p * scale (p <= 2^kLazy) go in as single fp16 w'.  The
    // codes are not centred, so the rounding w - w' is also added back times
    // the mid code through the fp32 zero-point sum; what is left is
    // (w - w') (c - mid), a few 1e-4 of the output at most.
    {
        const float srw = sr * kWScale, sr8w = sr8 * kWScale;
        const float w0 = p0v * srw, w1 = p1v * srw, w2 = p2v * sr8w, w3 = p3v * sr8w;
        const uint32_t h01 = pack_h2(w0, w1), h23 = pack_h2(w2, w3);
        const float2 r01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 r23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        constexpr float kMid = 0.5f * (float)((1 << VB) - 1) / kWScale;
        z0 = fmaf(p0v, zr, fmaf(p2v, zr8, fmaf(kMid, (w0 - r01.x) + (w2 - r23.x), z0)));
        z1 = fmaf(p1v, zr, fmaf(p3v, zr8, fmaf(kMid, (w1 - r01.y) + (w3 - r23.y), z1)));
        const uint32_t bh0 = movtrans(h01);
        const uint32_t bh1 = movtrans(h23);
        uint32_t Pab[16], Pcd[16];
        value_codes<VB>(pg + F::vcode, r, ta, tb, Pab);
        value_codes<VB>(pg + F::vcode, r, ta + 8, tb + 8, Pcd);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)  // rows: dim 16r + 2mt (row r), 16r + 2mt + 1 (row r + 8)
            mma16816(acc[mt], Pab[2 * mt], Pab[2 * mt + 1], Pcd[2 * mt], Pcd[2 * mt + 1], bh0, bh1);
    }
}

// ---------------------------------------------------------------------------
// Epilogue shared by the decode kernels: reduce each warp's softmax state over
// its token rows, merge the NW warps in shared memory (over the remainder
// table, free by then), rotate back, and either write the output (one split)
// or publish this split's partial and let the last CTA of the (sequence, KV
// head) merge the splits.  A CTA whose wait gave up contributes an empty
// partial.  With TMEM_COLS > 0 the CTA's tensor memory is released once every
// warp is past its pages.
// ---------------------------------------------------------------------------
template <int NW, int VB, int TMEM_COLS>
__device__ __forceinline__ void decode_epilogue(const DecodeArgs& a, uint8_t* sm, int lut_off, bool timed_out,
                                                int split, int h, int b, float m0, float m1, float l0, float l1,
                                                float z0, float z1, float (&acc)[8][4], uint32_t tmem) {
    constexpr int D = kHeadDim;
    const Geometry& g = a.g;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, qd = lane & 3;
    const int G = a.group;
    // ---- reduce l, z over the 8 token rows, publish warp state ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        z0 += __shfl_xor_sync(0xffffffffu, z0, o);
        z1 += __shfl_xor_sync(0xffffffffu, z1, o);
    }
    if constexpr (TMEM_COLS > 0) tc::fence_before_sync();
    __syncthreads();  // (A) every warp is past its pages: the remainder table is free
    if constexpr (TMEM_COLS > 0) {
        // every tensor-core operation of the CTA is complete: release tensor memory
        if (warp == 0) {
            tc::fence_after_sync();
            tc::tmem_dealloc<TMEM_COLS>(tmem);
        }
    }
    // warp states [NW][8][3] and accumulators [NW][8][128] over the table; a
    // query's dims are stored XOR-swizzled by 4 * (query / 2) so that both
    // these stores and the merge's 16-byte loads stay clear of bank conflicts
    float* wst_w = reinterpret_cast<float*>(sm + lut_off);
    float* wacc_w = reinterpret_cast<float*>(sm + lut_off + 2048);
    if (r == 0) {
        wst_w[(warp * 8 + 2 * qd) * 3 + 0] = m0;
        wst_w[(warp * 8 + 2 * qd) * 3 + 1] = l0;
        wst_w[(warp * 8 + 2 * qd) * 3 + 2] = z0;
        wst_w[(warp * 8 + 2 * qd + 1) * 3 + 0] = m1;
        wst_w[(warp * 8 + 2 * qd + 1) * 3 + 1] = l1;
        wst_w[(warp * 8 + 2 * qd + 1) * 3 + 2] = z1;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        // undo the fp16-subnormal scaling of the value codes of dims d, d + 1
        const float e0 = (float)(1u << (value_exp<VB>(2 * mt) - value_wshift<VB>()));
        const float e1 = (float)(1u << (value_exp<VB>(2 * mt + 1) - value_wshift<VB>()));
        const int d = (16 * r + 2 * mt) ^ (4 * qd);
        *reinterpret_cast<float2*>(wacc_w + (warp * 8 + 2 * qd) * D + d) = make_float2(acc[mt][0] * e0, acc[mt][2] * e1);
        *reinterpret_cast<float2*>(wacc_w + (warp * 8 + 2 * qd + 1) * D + d) =
            make_float2(acc[mt][1] * e0, acc[mt][3] * e1);
    }
    // A CTA with a wait that gave up flags it and contributes an empty partial
    // (max -inf, sum 0, acc 0), but still takes part in the split merge below:
    // every CTA bumps the counter, so the last one still merges and resets it,
    // and the workspace stays usable for the next call.
    timed_out = __syncthreads_or(timed_out);  // (B)
    if (timed_out && tid == 0) flag(a.status, TQ_FLAG_TIMEOUT);

    // ---- merge the warps: thread (query warp, lane) owns dims 4 lane .. 4 lane + 3 ----
    const float* wst = reinterpret_cast<const float*>(sm + lut_off);
    const float* wacc = reinterpret_cast<const float*>(sm + lut_off + 2048);
    const int qg = warp;  // query of this warp (warps 0..7)
    float Mx = kMinusBig, L = 0.f, O[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < 8 && !timed_out) {
        for (int w = 0; w < NW; ++w) Mx = fmaxf(Mx, wst[(w * 8 + qg) * 3]);
        float Z = 0.f;
        const int dsw = (4 * lane) ^ (4 * (qg >> 1));
        for (int w = 0; w < NW; ++w) {
            const float f = exp2f(wst[(w * 8 + qg) * 3] - Mx);
            L = fmaf(f, wst[(w * 8 + qg) * 3 + 1], L);
            Z = fmaf(f, wst[(w * 8 + qg) * 3 + 2], Z);
            const float4 v = *reinterpret_cast<const float4*>(wacc + (w * 8 + qg) * D + dsw);
            O[0] = fmaf(f, v.x, O[0]); O[1] = fmaf(f, v.y, O[1]);
            O[2] = fmaf(f, v.z, O[2]); O[3] = fmaf(f, v.w, O[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) O[i] += Z;
    }

    // Rotate this CTA's unnormalised accumulator back now, R^T O = s (.) H O / sqrt(d):
    // R^T is linear, so the split merge below is then a plain weighted sum.
    if (warp < G) {
        fwht128(O, lane);
        const uint32_t sg = lane_signs(a.c, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            O[i] *= 0.08838834764831845f;
            if ((sg >> i) & 1u) O[i] = -O[i];
        }
    }
    float* o = a.out + ((int64_t)b * a.hq + (int64_t)h * G + qg) * D;
    if (a.num_splits == 1) {
        if (warp < G) {
            const float inv = (L > 0.f) ? 1.f / L : 0.f;
            *reinterpret_cast<float4*>(o + 4 * lane) = make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
        }
        return;
    }

    // publish this split's partial (max, sum, rotated acc with the zero term folded in)
    const int64_t unit = (int64_t)b * g.hkv + h;
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
    if (warp < G) {
        // Lane k loads (max, sum) of split s0 + k and every lane its 4 dims of all
        // kChunk splits, all before any use: one L2 round trip per chunk.
        constexpr int kChunk = 20;
        const float* base = a.partials + (unit * a.num_splits * G + qg) * kPartStride;
        const int ns = a.num_splits;
        float runM = kMinusBig, runL = 0.f;
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < ns; s0 += kChunk) {
            const int n = min(kChunk, ns - s0);
            float ms = kMinusBig, ls = 0.f;
            if (lane < n) {
                ms = __ldcg(base + (int64_t)(s0 + lane) * G * kPartStride);
                ls = __ldcg(base + (int64_t)(s0 + lane) * G * kPartStride + 1);
            }
            float4 v[kChunk];
#pragma unroll
            for (int k = 0; k < kChunk; ++k)
                v[k] = (k < n) ? __ldcg(reinterpret_cast<const float4*>(base + (int64_t)(s0 + k) * G * kPartStride + 4 + 4 * lane))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            const float cm = fmaxf(runM, warp_max(ms));
            const float fr = exp2f(runM - cm);
            const float f = exp2f(ms - cm);
            runL = fmaf(runL, fr, warp_sum(f * ls));
#pragma unroll
            for (int i = 0; i < 4; ++i) acc4[i] *= fr;
#pragma unroll
            for (int k = 0; k < kChunk; ++k) {
                const float fk = __shfl_sync(0xffffffffu, f, k);
                acc4[0] = fmaf(fk, v[k].x, acc4[0]); acc4[1] = fmaf(fk, v[k].y, acc4[1]);
                acc4[2] = fmaf(fk, v[k].z, acc4[2]); acc4[3] = fmaf(fk, v[k].w, acc4[3]);
            }
            runM = cm;
        }
        const float inv = (runL > 0.f) ? 1.f / runL : 0.f;
        *reinterpret_cast<float4*>(o + 4 * lane) =
            make_float4(acc4[0] * inv, acc4[1] * inv, acc4[2] * inv, acc4[3] * inv);
    }
    if (tid == 0) a.counters[unit] = 0u;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int KB, int VB, int M>
__global__ void __launch_bounds__(decode_warps<M>() * 32, 1) decode_kernel(const DecodeArgs a) {
    static_assert(KB >= 1 && KB <= 8 && VB >= 1 && VB <= 8 && (M == 0 || (M == 128 && KB >= 2 && KB <= 4)),
                  "unsupported page format");
    using F = PageFmt<KB, VB, M>;
    constexpr int NW = decode_warps<M>();
    constexpr int NT = NW * 32;
    constexpr Layout LY = decode_layout<KB, VB, M>();
    constexpr int SPW = LY.spw;
    static_assert(SPW >= 1, "page format does not fit in shared memory");
    constexpr int D = kHeadDim;
    constexpr int KROW = D * KB / 8;
    extern __shared__ __align__(128) uint8_t sm[];
    const Geometry& g = a.g;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = a.group;

    // The layout assumes dynamic shared memory starts below kMaxSmemBase.  The
    // start address is the same for every CTA of the launch, so either all of
    // them return here (no split counter is touched) or none does.
    const uint32_t sbase = smem_u32(sm);
    if (sbase > (uint32_t)kMaxSmemBase) {
        grid_dependency_wait();
        if (tid == 0) flag(a.status, TQ_FLAG_INTERNAL);
        return;
    }
    const int lut_off = (int)kLutAddr - (int)sbase;  // byte offset of the remainder table in sm[]
    const uint32_t ring_w = (warp < LY.nwA) ? sbase + LY.ringA + warp * SPW * F::stride
                                           : kLutAddr + kLutBytes + (warp - LY.nwA) * SPW * F::stride;
    const uint32_t bar_w = sbase + LY.bars + 8 * warp * kMaxSlotsPerWarp;
    int* slot_ok = reinterpret_cast<int*>(sm + LY.ok) + warp * kMaxSlotsPerWarp;
    float* qrot = reinterpret_cast<float*>(sm + LY.qrot);
    float* qoff = reinterpret_cast<float*>(sm + LY.qoff);
    float* qscale = reinterpret_cast<float*>(sm + LY.qscale);
    const int p0 = split * a.pages_per_split;
    const float ksc = a.sm_scale_log2;

    // ---- shared-memory-only setup: it may overlap the previous kernel's tail ----
    const uint32_t stage_bar = sbase + LY.stage + kStageBar;
    if (lane == 0) {
        for (int k = 0; k < SPW; ++k) mbar_init(bar_w + 8 * k, 1);
        if (warp == 0) {
            mbar_init(stage_bar, 1);
            mbar_init(sbase + LY.stage + kStageNever, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    uint16_t* rem = reinterpret_cast<uint16_t*>(sm + LY.rem);
    if (tid < 16) rem[tid] = a.c.rem_f16[tid];
    else if (tid < 32) rem[tid] = a.c.cint_f16[tid - 16];
    else if (tid < 48) rem[tid] = a.c.crem_f16[tid - 32];
    __syncthreads();
    // Lane-private remainder table at shared address kLutAddr (copy for
    // lane l at entry*stride + l*width):
    //   4-bit keys: byte e (2 codes) -> (N[e&15], N[e>>4]), (rem2[e&15], rem2[e>>4])  stride 256, 8 B
    //   2-bit keys: byte e (4 codes) -> (rem[c0], rem[c1]), (rem[c2], rem[c3]) stride 256, 8 B
    //   3-bit keys: 6 bits e (2 codes) -> (rem[e&7], rem[e>>3])              stride 128, 4 B
    //   1-bit keys: 2 bits e (2 codes) -> (rem[e&1], rem[e>>1])              stride 128, 4 B
    //   5..7-bit keys: code e -> (rem[e], rem[e])                           stride 128, 4 B
    //   8-bit keys: code e -> (rem[e], rem[e])                              stride 256, 4 B
    // Widths above 4 bits read rem from the cache's table in global memory,
    // so their table is built after the wait below.
    auto build_lut = [&](const uint16_t* rsrc) {
        uint8_t* lut = sm + lut_off;
        if constexpr (KB == 4) {
            const uint16_t* ni = rsrc + 16;  // N, then rem2
            const uint16_t* r2 = rsrc + 32;
            for (int i = tid; i < 256 * 16; i += NT) {  // entry e, lanes 2k, 2k+1
                const int e = i >> 4, k = i & 15;
                const uint32_t xx = (uint32_t)ni[e & 15] | ((uint32_t)ni[e >> 4] << 16);
                const uint32_t yy = (uint32_t)r2[e & 15] | ((uint32_t)r2[e >> 4] << 16);
                *reinterpret_cast<uint4*>(lut + e * 256 + 16 * k) = make_uint4(xx, yy, xx, yy);
            }
        } else if constexpr (KB == 2) {
            for (int i = tid; i < 256 * 16; i += NT) {  // entry e, lanes 2k, 2k+1
                const int e = i >> 4, k = i & 15;
                const uint32_t xx = (uint32_t)rsrc[e & 3] | ((uint32_t)rsrc[(e >> 2) & 3] << 16);
                const uint32_t yy = (uint32_t)rsrc[(e >> 4) & 3] | ((uint32_t)rsrc[e >> 6] << 16);
                *reinterpret_cast<uint4*>(lut + e * 256 + 16 * k) = make_uint4(xx, yy, xx, yy);
            }
        } else if constexpr (KB == 8) {
            for (int i = tid; i < 256 * 8; i += NT) {   // entry e, lanes 4k..4k+3
                const int e = i >> 3, k = i & 7;
                const uint32_t r = __ldg(rsrc + e);
                const uint32_t v = r | (r << 16);
                *reinterpret_cast<uint4*>(lut + e * 256 + 16 * k) = make_uint4(v, v, v, v);
            }
        } else if constexpr (KB >= 5) {
            for (int i = tid; i < (1 << KB) * 8; i += NT) {
                const int e = i >> 3, k = i & 7;
                const uint32_t r = __ldg(rsrc + e);
                const uint32_t v = r | (r << 16);
                *reinterpret_cast<uint4*>(lut + e * 128 + 16 * k) = make_uint4(v, v, v, v);
            }
        } else {
            constexpr int mask = (1 << KB) - 1;
            for (int i = tid; i < (1 << (2 * KB)) * 8; i += NT) {
                const int e = i >> 3, k = i & 7;
                const uint32_t v = (uint32_t)rsrc[e & mask] | ((uint32_t)rsrc[e >> KB] << 16);
                *reinterpret_cast<uint4*>(lut + e * 128 + 16 * k) = make_uint4(v, v, v, v);
            }
        }
    };
    if constexpr (KB <= 4) build_lut(rem);
    // Launched as a programmatic dependent of the previous kernel in the stream:
    // nothing in global memory is touched before that grid has completed.
    grid_dependency_wait();
    grid_launch_dependents();
    if constexpr (KB > 4) build_lut(a.tab->rem_f16);

    // ---- global loads: length, this warp's block ids, the query ----
    // Warp w handles pages w, w + NW, w + 2 NW, ... of the split (its j-th page
    // is w + NW j) in its own SPW ring slots.  Lane l holds the block id of the
    // warp's page l of the current batch of 32 (bid_cur) and of the next batch
    // (bid_nxt).
    int len = __ldg(a.lens + b);
    const int32_t* btw = a.block_table + (int64_t)b * a.bt_stride + p0 + warp;
    const int reach = min(a.pages_per_split, a.max_blocks - p0) - warp;  // pages of the split at or after this warp's first
    int bid_cur = (NW * lane < reach) ? __ldg(btw + NW * lane) : -1;
    int bid_nxt = (NW * (32 + lane) < reach) ? __ldg(btw + NW * (32 + lane)) : -1;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp < G) load4(a.q, a.dtype, ((int64_t)b * a.hq + (int64_t)h * G + warp) * D + 4 * lane, x);

    // ---- sequence range of this split ----
    // len counts the sequence's tokens (the appended one included).  A ring of
    // `window` slots holds the last `window` of them, token t in slot t mod
    // window; attention runs over the slots that hold tokens, in any order.
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
    const int seq_pages = (len + g.bs - 1) / g.bs;
    int npages = seq_pages - p0;
    if (npages > a.pages_per_split) npages = a.pages_per_split;
    if (npages < 0) npages = 0;
    const int nmine = npages > warp ? (npages - warp + NW - 1) / NW : 0;  // this warp's pages

    // Start a page copy into ring slot `slot` of this warp; a bad block id
    // arrives on the barrier without data and the page is skipped.
    auto issue = [&](int slot, int blk) {
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
    // The appended token lies in page pos_new / 16 of the sequence (without a
    // ring: its last page, the split's last page pi = npages - 1).  The warp
    // that owns that page patches the token into its shared-memory copy when
    // it gets there.  When the owner is one of the warps with an extra page,
    // the encoding is done by warp npages % NW (one page fewer), otherwise by
    // the owner, right after the query is prepared, and handed over through
    // the stage barrier.  Its inputs are requested now, ahead of the page
    // copies, and waited on only when used.
    int jnew = -1;        // owner: its index of the page that takes the token
    bool enc = false;     // this warp encodes the token
    int blknew = -1;
    const int offnew = pos_new & (kBlockSize - 1);
    uint32_t kraw[4] = {0u, 0u, 0u, 0u}, vraw[4] = {0u, 0u, 0u, 0u};
    {
        if (a.knew != nullptr && len > 0) {
            const int pi = pos_new / kBlockSize - p0;
            if (pi >= 0 && pi < npages) {
                const int owner = pi % NW, rest = npages % NW;
                const int encoder = (rest != 0 && owner < rest) ? rest : owner;
                if (warp == owner) jnew = pi / NW;
                if (warp == encoder) {
                    enc = true;
                    const int64_t e = ((int64_t)b * g.hkv + h) * D + 4 * lane;
                    raw4(a.knew, a.kv_dtype, e, kraw);
                    raw4(a.vnew, a.kv_dtype, e, vraw);
                    blknew = __ldg(a.block_table + (int64_t)b * a.bt_stride + p0 + pi);
                }
            }
        }
    }

    // The first kFirstPages pages of every warp now, one lane each; the rest of
    // the ring once the query is prepared, so that the first pages of all warps
    // are not queued behind the whole initial burst.
    constexpr int kFirst = SPW < kFirstPages ? SPW : kFirstPages;
    if (lane < kFirst && lane < nmine) issue(lane, bid_cur);

    bool timed_out = false;
    float m0 = kMinusBig, m1 = kMinusBig, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    {
        // q_rot = R q for query (warp) of this group; its per-query constants:
        //   qoff   = sm_scale log2(e) alpha mid sum(q_rot)
        //   qscale = power of two putting max |ksc alpha q_rot| / qscale in (256, 512]
        if (warp < 8) {
            if (warp < G) {
                apply_signs(x, lane_signs(a.c, lane));
                fwht128(x, lane);
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] *= 0.08838834764831845f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) qrot[warp * kQStride + 4 * lane + i] = x[i];
            const float sq = warp_sum(x[0] + x[1] + x[2] + x[3]);
            const float mx = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
            const float slope = (KB == 4) ? a.c.delta : a.c.alpha;  // scale of the integer part
            const float big = fabsf(slope) * ksc * mx;
            const float scl = (big > 0.f) ? exp2f(ceilf(log2f(big / 512.f))) : 1.f;
            if (lane == 0) {
                qoff[warp] = (KB == 4) ? 0.f : ksc * a.c.alpha * (float)((1 << KB) - 1) * 0.5f * sq;
                qscale[warp] = scl;
            }
        }
        __syncthreads();
        float* sqv = reinterpret_cast<float*>(sm + LY.sq);  // [8][128]: sm_scale log2(e) S q_rot per query
        if constexpr (M > 0) {
            // thread -> row i of S, queries g0, g0 + NT/M, ...
            const int i = tid & (M - 1), g0 = tid / M;
            constexpr int GS = NT / M;
            const float4* srow = reinterpret_cast<const float4*>(a.S + (int64_t)i * D);
            float acc4[(8 + GS - 1) / GS];
#pragma unroll
            for (int k = 0; k < (8 + GS - 1) / GS; ++k) acc4[k] = 0.f;
            for (int j4 = 0; j4 < D / 4; ++j4) {
                const float4 sv = __ldg(srow + j4);
#pragma unroll
                for (int k = 0; k < (8 + GS - 1) / GS; ++k) {
                    const int gq = g0 + GS * k;
                    if (gq < 8) {
                        const float4 qv = *reinterpret_cast<const float4*>(qrot + gq * kQStride + 4 * j4);
                        acc4[k] = fmaf(sv.x, qv.x, fmaf(sv.y, qv.y, fmaf(sv.z, qv.z, fmaf(sv.w, qv.w, acc4[k]))));
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < (8 + GS - 1) / GS; ++k) {
                const int gq = g0 + GS * k;
                if (gq < 8) sqv[gq * kQStride + i] = ksc * acc4[k];
            }
            __syncthreads();
        }

        // ---- per-lane query fragments, written once per CTA in lane-major order ----
        // (word w of lane l at ((w / 4) * 32 + l) * 16 + (w % 4) * 4, so that a
        // warp reads each group of four words with one conflict-free 16-byte load;
        // thread (vector v, lane l) computes and stores one such group)
        //   words  0..31  QI: x = ksc alpha q_rot / qscale in fp16 hi + lo; word
        //                 4 ks + 2 part + slot holds part (0 hi, 1 lo) of x 2^(e-24)
        //                 at the dims of key register X[2 ks + slot] (e its scale)
        //   words 32..47  QB: sm_scale log2(e) q_rot in fp16 at remainder dims (2n, 2n+1)
        //   words 48..79  QSh / QSl: sqv hi + lo in fp16 at sign dims (n, n + 16)
        {
            uint4* fr = reinterpret_cast<uint4*>(sm + LY.frag);
            for (int t = tid; t < 32 * frag_vecs<M>(); t += NT) {
                const int v = t >> 5, ln = t & 31;
                const int gq = ln >> 2, ch = 32 * (ln & 3);  // query, first dim of the lane's chunk
                const float* qr = qrot + gq * kQStride + ch;
                uint32_t wv[4];
                if (v < 8) {
                    const float xs = ksc * ((KB == 4) ? a.c.delta : a.c.alpha) / qscale[gq];
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        const int n = 2 * v + sl;
                        const float e = xs * exp2f((float)(key_exp<KB>(n) - 24));
                        const float x0 = e * qr[key_dim<KB>(n, 0)], x1 = e * qr[key_dim<KB>(n, 1)];
                        const uint32_t hi = pack_h2(x0, x1);
                        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                        wv[sl] = hi;
                        wv[2 + sl] = pack_h2(x0 - hf.x, x1 - hf.y);
                    }
                } else if (v < 12) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int n = 4 * (v - 8) + i;
                        wv[i] = pack_h2(qr[2 * n] * ksc, qr[2 * n + 1] * ksc);
                    }
                } else {
                    const float* sr = sqv + gq * kQStride + ch;
                    const int lo = v >= 16;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int n = 4 * (v - (lo ? 16 : 12)) + i;
                        const uint32_t hi = pack_h2(sr[n], sr[n + 16]);
                        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                        wv[i] = lo ? pack_h2(sr[n] - hf.x, sr[n + 16] - hf.y) : hi;
                    }
                }
                fr[v * 32 + ln] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
        }
        __syncthreads();
        if (lane >= kFirst && lane < SPW && lane < nmine) issue(lane, bid_cur);
        if (enc) {
            // a bad block id leaves the pool alone; the owner's copy of that
            // page is flagged and skipped, so what it patches in is never used
            if (blknew >= 0 && blknew < g.num_blocks) {
                uint8_t* page = const_cast<uint8_t*>(a.pool) + ((int64_t)blknew * g.hkv + h) * F::bytes;
                append_token<KB, VB, M>(a, page, offnew, sm + LY.stage, lane, kraw, vraw);
            }
            if (lane == 0) mbar_arrive(stage_bar);
        }
        const int r = lane >> 2, qd = lane & 3;   // r: token row / query column; qd: quad index
        uint32_t QI[8][4], QB[16];
        uint32_t QSh[M > 0 ? 16 : 1], QSl[M > 0 ? 16 : 1];
        {
            const uint4* fv = reinterpret_cast<const uint4*>(sm + LY.frag) + lane;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint4 t = fv[v * 32];
                QI[v][0] = t.x; QI[v][1] = t.y; QI[v][2] = t.z; QI[v][3] = t.w;
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 t = fv[(8 + v) * 32];
                QB[4 * v] = t.x; QB[4 * v + 1] = t.y; QB[4 * v + 2] = t.z; QB[4 * v + 3] = t.w;
            }
            if constexpr (M > 0) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 t = fv[(12 + v) * 32], u = fv[(16 + v) * 32];
                    QSh[4 * v] = t.x; QSh[4 * v + 1] = t.y; QSh[4 * v + 2] = t.z; QSh[4 * v + 3] = t.w;
                    QSl[4 * v] = u.x; QSl[4 * v + 1] = u.y; QSl[4 * v + 2] = u.z; QSl[4 * v + 3] = u.w;
                }
            }
        }
        const float off0 = qoff[2 * qd], off1 = qoff[2 * qd + 1];
        const float qs0 = qscale[2 * qd] * key_int_scale<KB>(), qs1 = qscale[2 * qd + 1] * key_int_scale<KB>();
        const float cq = 1.2533141373155003f / (float)(M > 0 ? M : 1);  // sqrt(pi/2) / m
        const uint32_t lw = kLutAddr | ((uint32_t)lane << ((KB == 2 || KB == 4) ? 3 : 2));
        // Score row r holds token tr = r ^ ((r >> 1) & 1) (and row r + 8 token tr + 8):
        // tokens 2 and 3, 6 and 7 trade rows, so that the value loads below (tokens
        // of rows 2qd, 2qd+1 for qd = 0..3) alternate between the two halves of the
        // bank space instead of colliding four ways.
        const int tr = r ^ ((r >> 1) & 1);
        const int ta = (2 * qd) ^ (qd & 1), tb = (2 * qd + 1) ^ (qd & 1);  // tokens of rows 2qd, 2qd+1
        const int koff = F::kcode + tr * KROW + qd * 4 * KB;  // this lane's key chunk in a page


        int slot = 0;
        uint32_t phase = 0;
        int issued = min(SPW, nmine);   // pages of this warp whose copies were started
        int jfail = nmine;              // first page whose wait gave up
        if (a.stall_cycles > 0 && (split & 1) && warp == 0) {
            // test hook: a bounded wait on a barrier that nothing arrives on runs
            // out, and the warp takes the timeout path below before its first page
            if (!mbar_wait_for(sbase + LY.stage + kStageNever, 0, a.stall_cycles)) {
                timed_out = true;
                jfail = 0;
            }
        }
        for (int j = 0; j < (timed_out ? 0 : nmine); ++j) {
            if (!mbar_wait(bar_w + 8 * slot, phase)) {
                timed_out = true;
                jfail = j;
                break;
            }
            const uint32_t pg = ring_w + slot * F::stride;  // shared-space address of the page
            const bool pok = slot_ok[slot] != 0;
            if (j == jnew) {
                if (!mbar_wait(stage_bar, 0)) {
                    timed_out = true;
                    jfail = j;
                    break;
                }
                patch_page<KB, VB, M>(sm + (pg - sbase), offnew, sm + LY.stage, lane);
                // the slot is refilled later by a bulk copy: order these generic
                // writes before that async-proxy write
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }

            // ---------- scores: tokens r (rows 0-7) and r+8 (rows 8-15) ----------
            uint32_t wa[KB], wb[KB];
            key_words<KB>(pg + koff, wa);
            key_words<KB>(pg + koff + 8 * KROW, wb);
            float I0[4], I1[4], R0[4], R1[4];
            if constexpr (KB == 4) {
                // per k-step: the operands of code bytes 2ks, 2ks+1 of both tokens,
                // then the integer part (hi and lo query) and the remainder
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint2 a0 = key_lut4(wa, lw, 2 * ks), b0 = key_lut4(wb, lw, 2 * ks);
                    const uint2 a1 = key_lut4(wa, lw, 2 * ks + 1), b1 = key_lut4(wb, lw, 2 * ks + 1);
                    float* I = (ks & 1) ? I1 : I0;
                    float* Rr = (ks & 1) ? R1 : R0;
                    if (ks < 2) {
                        mma16816_c(I, a0.x, b0.x, a1.x, b1.x, QI[ks][0], QI[ks][1], 0.f, 0.f, 0.f, 0.f);
                        mma16816_c(Rr, a0.y, b0.y, a1.y, b1.y, QB[2 * ks], QB[2 * ks + 1], 0.f, 0.f, 0.f, 0.f);
                    } else {
                        mma16816(I, a0.x, b0.x, a1.x, b1.x, QI[ks][0], QI[ks][1]);
                        mma16816(Rr, a0.y, b0.y, a1.y, b1.y, QB[2 * ks], QB[2 * ks + 1]);
                    }
                    mma16816(I, a0.x, b0.x, a1.x, b1.x, QI[ks][2], QI[ks][3]);
                }
            } else {
            {
                uint32_t Xa[16], Xb[16];
                key_halves<KB>(wa, Xa);
                key_halves<KB>(wb, Xb);
                mma16816_c(I0, Xa[0], Xb[0], Xa[1], Xb[1], QI[0][0], QI[0][1], 0.f, 0.f, 0.f, 0.f);
                mma16816(I0, Xa[0], Xb[0], Xa[1], Xb[1], QI[0][2], QI[0][3]);
                mma16816_c(I1, Xa[2], Xb[2], Xa[3], Xb[3], QI[1][0], QI[1][1], 0.f, 0.f, 0.f, 0.f);
                mma16816(I1, Xa[2], Xb[2], Xa[3], Xb[3], QI[1][2], QI[1][3]);
#pragma unroll
                for (int ks = 2; ks < 8; ++ks) {
                    float* I = (ks & 1) ? I1 : I0;
                    mma16816(I, Xa[2 * ks], Xb[2 * ks], Xa[2 * ks + 1], Xb[2 * ks + 1], QI[ks][0], QI[ks][1]);
                    mma16816(I, Xa[2 * ks], Xb[2 * ks], Xa[2 * ks + 1], Xb[2 * ks + 1], QI[ks][2], QI[ks][3]);
                }
            }
            {
                uint32_t Ra[16], Rb[16];
                key_rem<KB>(wa, lw, Ra);
                key_rem<KB>(wb, lw, Rb);
                mma16816_c(R0, Ra[0], Rb[0], Ra[1], Rb[1], QB[0], QB[1], -off0, -off1, -off0, -off1);
                mma16816_c(R1, Ra[2], Rb[2], Ra[3], Rb[3], QB[2], QB[3], 0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int ks = 2; ks < 8; ++ks) {
                    const int n = 2 * ks;
                    mma16816((ks & 1) ? R1 : R0, Ra[n], Rb[n], Ra[n + 1], Rb[n + 1], QB[n], QB[n + 1]);
                }
            }
            }
            float t0 = fmaf(qs0, I0[0] + I1[0], R0[0] + R1[0]), t1 = fmaf(qs1, I0[1] + I1[1], R0[1] + R1[1]);
            float t2 = fmaf(qs0, I0[2] + I1[2], R0[2] + R1[2]), t3 = fmaf(qs1, I0[3] + I1[3], R0[3] + R1[3]);
            if constexpr (M > 0) {
                float sQ[4];
                uint32_t Za[16], Zb[16];
                sign_chunk(lds32(pg + F::sig + tr * (M / 8) + 4 * qd), Za);
                sign_chunk(lds32(pg + F::sig + (tr + 8) * (M / 8) + 4 * qd), Zb);
                mma16816_c(sQ, Za[0], Zb[0], Za[1], Zb[1], QSh[0], QSh[1], 0.f, 0.f, 0.f, 0.f);
                mma16816(sQ, Za[0], Zb[0], Za[1], Zb[1], QSl[0], QSl[1]);
#pragma unroll
                for (int ks = 1; ks < 8; ++ks) {
                    const int n = 2 * ks;
                    mma16816(sQ, Za[n], Zb[n], Za[n + 1], Zb[n + 1], QSh[n], QSh[n + 1]);
                    mma16816(sQ, Za[n], Zb[n], Za[n + 1], Zb[n + 1], QSl[n], QSl[n + 1]);
                }
                const float rr = cq * lds_h2f(pg + F::rho + 2 * tr), rr8 = cq * lds_h2f(pg + F::rho + 2 * (tr + 8));
                t0 = fmaf(rr, sQ[0], t0); t1 = fmaf(rr, sQ[1], t1);
                t2 = fmaf(rr8, sQ[2], t2); t3 = fmaf(rr8, sQ[3], t3);
            }
            softmax_pv_page<KB, VB, M>(pg, pok, (p0 + warp + NW * j) * kBlockSize, len, t0, t1, t2, t3, r, tr, ta, tb,
                                       m0, m1, l0, l1, z0, z1, acc);

            __syncwarp();  // every lane has read the slot: refill it with the page SPW ahead
            const int jn = j + SPW;
            if (jn < nmine) {
                if ((jn & 31) == 0) {  // next batch of block ids; prefetch the one after it
                    bid_cur = bid_nxt;
                    const int k = NW * (jn + 32 + lane);
                    bid_nxt = (k < reach) ? __ldg(btw + k) : -1;
                }
                if (lane == (jn & 31)) issue(slot, bid_cur);
                ++issued;
            }
            if (++slot == SPW) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (timed_out) {
            // copies this warp started must land before its shared memory goes away;
            // one shared deadline for all of them
            const long long t0 = clock64();
            for (int jj = jfail; jj < issued; ++jj) {
                const uint32_t bar = bar_w + 8 * (jj % SPW);
                while (!mbar_try(bar, (uint32_t)((jj / SPW) & 1)) && clock64() - t0 < kWaitCycles) {
                }
            }
        }

    }
    decode_epilogue<NW, VB, 0>(a, sm, lut_off, timed_out, split, h, b, m0, m1, l0, l1, z0, z1, acc, 0u);
}

template <int KB, int VB, int M>
static int launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
    using F = PageFmt<KB, VB, M>;
    const Geometry& g = a.g;
    if (g.page_bytes != F::bytes || g.vcode_off != F::vcode || g.gam_off != F::gam || g.scl_off != F::scl ||
        g.zer_off != F::zer || (M && (g.rho_off != F::rho || g.sig_off != F::sig)) || g.bs != kBlockSize ||
        g.d != kHeadDim)
        return (int)cudaErrorInvalidValue;  // the cache's geometry is not the format this kernel was built for
    constexpr Layout L = decode_layout<KB, VB, M>();
    auto kern = decode_kernel<KB, VB, M>;
    static int done[64] = {};
    cudaError_t e = ensure_smem_limit(kern, L.total, done);
    if (e != cudaSuccess) return (int)e;
    return (int)launch_programmatic(kern, dim3((unsigned)a.num_splits, (unsigned)g.hkv, (unsigned)a.batch),
                                    dim3(decode_warps<M>() * 32), (size_t)L.total, s, a);
}

template <int KB>
int decode_smem_kb(const Geometry& g) {
    if constexpr (KB >= 2 && KB <= 4) {
        if (g.m) {
            if (g.vb == 2) return decode_layout<KB, 2, 128>().total;
            if (g.vb == 3) return decode_layout<KB, 3, 128>().total;
            if (g.vb == 4) return decode_layout<KB, 4, 128>().total;
            return -1;
        }
    }
    if (g.m) return -1;
    switch (g.vb) {
        case 1: return decode_layout<KB, 1, 0>().total;
        case 2: return decode_layout<KB, 2, 0>().total;
        case 3: return decode_layout<KB, 3, 0>().total;
        case 4: return decode_layout<KB, 4, 0>().total;
        case 5: return decode_layout<KB, 5, 0>().total;
        case 6: return decode_layout<KB, 6, 0>().total;
        case 7: return decode_layout<KB, 7, 0>().total;
        case 8: return decode_layout<KB, 8, 0>().total;
        default: return -1;
    }
}

// All value widths (and the QJL sketch, for widths 2 .. 4) of one key width.
template <int KB>
int launch_decode_kb(const DecodeArgs& a, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int vb = a.g.vb, m = a.g.m;
    if constexpr (KB >= 2 && KB <= 4) {
        if (m) {
            if (vb == 2) return launch_decode_t<KB, 2, 128>(a, s);
            if (vb == 3) return launch_decode_t<KB, 3, 128>(a, s);
            if (vb == 4) return launch_decode_t<KB, 4, 128>(a, s);
            return (int)cudaErrorNotSupported;
        }
    }
    if (m) return (int)cudaErrorNotSupported;
    switch (vb) {
        case 1: return launch_decode_t<KB, 1, 0>(a, s);
        case 2: return launch_decode_t<KB, 2, 0>(a, s);
        case 3: return launch_decode_t<KB, 3, 0>(a, s);
        case 4: return launch_decode_t<KB, 4, 0>(a, s);
        case 5: return launch_decode_t<KB, 5, 0>(a, s);
        case 6: return launch_decode_t<KB, 6, 0>(a, s);
        case 7: return launch_decode_t<KB, 7, 0>(a, s);
        case 8: return launch_decode_t<KB, 8, 0>(a, s);
        default: return (int)cudaErrorNotSupported;
    }
}

}  // namespace tq
