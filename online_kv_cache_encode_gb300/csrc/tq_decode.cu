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

#include "tq_device.cuh"

namespace tq {

constexpr int kNCW = 8;                       // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;     // + producer warp
constexpr int kLutBytes = 256 * 256;          // 256 entries x 256 B (lanes use 128 B)
constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s bound on any wait
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
// Wait for the phase of the given parity; gives up after kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try(bar, parity))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
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
    int lut, qrot, qoff, bars, ok, ring;
    int stages, stride, total;
};

__host__ __device__ inline SmemMap smem_map(int page_bytes) {
    SmemMap m;
    int off = 0;
    m.lut = off; off += kLutBytes;
    m.qrot = off; off += 8 * kHeadDim * 4;
    m.qoff = off; off += 8 * 4;
    m.stride = (page_bytes + 127) / 128 * 128;
    const int budget = 227 * 1024 - 1024;
    int fixed = off + 64;
    int stages = (budget - fixed) / (m.stride + 2 * 8 + 4);
    if (stages > 64) stages = 64;
    m.stages = stages;
    m.bars = (off + 7) / 8 * 8; off = m.bars + 2 * 8 * stages;
    m.ok = off; off += 4 * stages;
    m.ring = (off + 127) / 128 * 128; off = m.ring + m.stride * stages;
    m.total = off;
    return m;
}

int decode_smem_bytes(const Geometry& g) { return smem_map((int)g.page_bytes).total; }

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int KB, int VB, int M>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeArgs a) {
    static_assert(KB == 4 && VB == 4 && M == 0, "only 4/4-bit pages are built so far");
    extern __shared__ __align__(128) uint8_t sm[];
    const Geometry& g = a.g;
    constexpr int D = kHeadDim;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = a.group;
    const SmemMap mp = smem_map((int)g.page_bytes);
    const int ST = mp.stages;

    float* qrot = reinterpret_cast<float*>(sm + mp.qrot);
    float* qoff = reinterpret_cast<float*>(sm + mp.qoff);
    int* slot_ok = reinterpret_cast<int*>(sm + mp.ok);
    const uint32_t bar_full = smem_u32(sm + mp.bars);
    const uint32_t bar_empty = bar_full + 8 * ST;
    const uint32_t lut_base = smem_u32(sm + mp.lut);
    const uint32_t ring_base = smem_u32(sm + mp.ring);
    uint8_t* ring = sm + mp.ring;

    // ---- sequence range of this split ----
    int len = a.lens[b];
    if (len > a.max_blocks * g.bs) {
        if (tid == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
        len = a.max_blocks * g.bs;
    }
    if (len < 0) len = 0;
    const int seq_pages = (len + g.bs - 1) / g.bs;
    const int p0 = split * a.pages_per_split;
    int npages = seq_pages - p0;
    if (npages > a.pages_per_split) npages = a.pages_per_split;
    if (npages < 0) npages = 0;

    // ---- barriers ----
    if (tid == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    bool timed_out = false;
    if (warp == kNCW) {
        // =================== producer ===================
        const int32_t* bt = a.block_table + (int64_t)b * a.max_blocks + p0;
        int issued = 0;
        for (int base = 0; base < npages && !timed_out; base += 32) {
            const int mine = base + lane;
            const int blk = mine < npages ? bt[mine] : -1;
            const int cnt = min(32, npages - base);
            for (int k = 0; k < cnt; ++k) {
                const int bk = __shfl_sync(0xffffffffu, blk, k);
                if (lane == 0 && !timed_out) {
                    const int pi = base + k, s = pi % ST;
                    if (pi >= ST && !mbar_wait(bar_empty + 8 * s, ((pi / ST) & 1) ^ 1)) {
                        timed_out = true;
                    } else {
                        const bool ok = bk >= 0 && bk < g.num_blocks;
                        slot_ok[s] = ok;
                        if (ok) {
                            mbar_arrive_tx(bar_full + 8 * s, (uint32_t)g.page_bytes);
                            bulk_g2s(ring_base + s * mp.stride,
                                     a.pool + ((int64_t)bk * g.hkv + h) * g.page_bytes,
                                     (uint32_t)g.page_bytes, bar_full + 8 * s);
                        } else {
                            flag(a.status, TQ_FLAG_BAD_SLOT);
                            mbar_arrive(bar_full + 8 * s);
                        }
                        ++issued;
                    }
                }
                timed_out = __shfl_sync(0xffffffffu, timed_out, 0);
                if (timed_out) break;
            }
        }
        // every copy this CTA started must land before shared memory is reused
        if (lane == 0) {
            for (int pi = issued - ST > 0 ? issued - ST : 0; pi < issued; ++pi)
                if (!mbar_wait(bar_full + 8 * (pi % ST), (pi / ST) & 1)) timed_out = true;
        }
        timed_out = __shfl_sync(0xffffffffu, timed_out, 0);
    } else {
        // =================== consumers ===================
        // lane-private remainder table: entry e (a byte holding two key codes)
        // -> (rem[e & 15], rem[e >> 4]) as fp16x2, copy for lane l at e*256 + 4l
        for (int i = tid; i < 256 * 32; i += kNCW * 32) {
            const int e = i >> 5, l = i & 31;
            const uint32_t v = (uint32_t)a.c.rem_f16[e & 15] | ((uint32_t)a.c.rem_f16[e >> 4] << 16);
            *reinterpret_cast<uint32_t*>(sm + mp.lut + e * 256 + 4 * l) = v;
        }
        // q_rot = R q for query (warp) of this group, and alpha * mid * sum(q_rot)
        {
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            if (warp < G) {
                load4(a.q, a.dtype, ((int64_t)b * a.hq + (int64_t)h * G + warp) * D + 4 * lane, x);
                apply_signs(x, lane_signs(a.c, lane));
                fwht128(x, lane);
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] *= 0.08838834764831845f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) qrot[warp * D + 4 * lane + i] = x[i];
            const float sq = warp_sum(x[0] + x[1] + x[2] + x[3]);
            if (lane == 0) qoff[warp] = a.c.alpha * (float)((1 << KB) - 1) * 0.5f * sq;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kNCW * 32) : "memory");

        const int r = lane >> 2, qd = lane & 3;   // r: token row / query column; qd: quad index
        // ---- B fragments (queries as columns) ----
        // int-code MMA: word wi of the lane's 32-dim chunk covers dims 8wi..8wi+7;
        // k-step ks uses regs 2(ks&1), 2(ks&1)+1 of word ks>>1, i.e. dim pairs
        // (8wi+i, 8wi+i+4) with i = 2(ks&1) (b0) and i+1 (b1).
        uint32_t QAh[8][2], QAl[8][2], QB[8][2];
        {
            const float* qr = qrot + r * D + 32 * qd;
            const float al = a.c.alpha;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int wi = ks >> 1, i = 2 * (ks & 1);
                const int d0 = 8 * wi + i;
                split_h2(al * qr[d0], al * qr[d0 + 4], QAh[ks][0], QAl[ks][0]);
                split_h2(al * qr[d0 + 1], al * qr[d0 + 5], QAh[ks][1], QAl[ks][1]);
                QB[ks][0] = pack_h2(qr[4 * ks], qr[4 * ks + 1]);
                QB[ks][1] = pack_h2(qr[4 * ks + 2], qr[4 * ks + 3]);
            }
        }
        const float off0 = qoff[2 * qd], off1 = qoff[2 * qd + 1];
        const float ksc = a.sm_scale_log2;
        const uint32_t lanew = (uint32_t)lane << 2;

        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
        float acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

        for (int pi = warp; pi < npages; pi += kNCW) {
            const int s = pi % ST;
            if (!mbar_wait(bar_full + 8 * s, (pi / ST) & 1)) {
                timed_out = true;
                break;
            }
            const uint8_t* pg = ring + s * mp.stride;
            const bool pok = slot_ok[s] != 0;

            // ---------- scores ----------
            const uint4 ka = *reinterpret_cast<const uint4*>(pg + g.kcode_off + r * 64 + qd * 16);
            const uint4 kb = *reinterpret_cast<const uint4*>(pg + g.kcode_off + (r + 8) * 64 + qd * 16);
            const uint32_t kaw[4] = {ka.x, ka.y, ka.z, ka.w}, kbw[4] = {kb.x, kb.y, kb.z, kb.w};
            float sA[4] = {0.f, 0.f, 0.f, 0.f}, sB[4] = {0.f, 0.f, 0.f, 0.f}, sC[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                uint32_t fa[4], fb[4];
                nib8_to_h2(kaw[wi], fa);
                nib8_to_h2(kbw[wi], fb);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int ks = 2 * wi + hh;
                    mma16816(sA, fa[2 * hh], fb[2 * hh], fa[2 * hh + 1], fb[2 * hh + 1], QAh[ks][0], QAh[ks][1]);
                    mma16816(sB, fa[2 * hh], fb[2 * hh], fa[2 * hh + 1], fb[2 * hh + 1], QAl[ks][0], QAl[ks][1]);
                }
                // remainder lookups: byte j of the chunk holds dims (2j, 2j+1)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int ks = 2 * wi + hh;  // bytes 2ks, 2ks+1 live in word wi
                    const uint32_t sel0 = 0x5504u | ((uint32_t)(2 * hh) << 4);
                    const uint32_t sel1 = 0x5504u | ((uint32_t)(2 * hh + 1) << 4);
                    uint32_t la0, la1, lb0, lb1;
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(la0) : "r"(lut_base + prmt(kaw[wi], lanew, sel0)));
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(lb0) : "r"(lut_base + prmt(kbw[wi], lanew, sel0)));
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(la1) : "r"(lut_base + prmt(kaw[wi], lanew, sel1)));
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(lb1) : "r"(lut_base + prmt(kbw[wi], lanew, sel1)));
                    mma16816(sC, la0, lb0, la1, lb1, QB[ks][0], QB[ks][1]);
                }
            }
            const uint16_t* gam = reinterpret_cast<const uint16_t*>(pg + g.gam_off);
            const uint16_t* vsc = reinterpret_cast<const uint16_t*>(pg + g.scl_off);
            const uint16_t* vze = reinterpret_cast<const uint16_t*>(pg + g.zer_off);
            const float gr = h2f(gam[r]) * ksc, gr8 = h2f(gam[r + 8]) * ksc;
            const int tok = (p0 + pi) * g.bs;
            const bool v_r = pok && (tok + r < len), v_r8 = pok && (tok + r + 8 < len);
            float s0 = v_r ? (sA[0] + sB[0] + sC[0] - off0) * gr : -INFINITY;
            float s1 = v_r ? (sA[1] + sB[1] + sC[1] - off1) * gr : -INFINITY;
            float s2 = v_r8 ? (sA[2] + sB[2] + sC[2] - off0) * gr8 : -INFINITY;
            float s3 = v_r8 ? (sA[3] + sB[3] + sC[3] - off1) * gr8 : -INFINITY;

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
            const float sr = h2f(vsc[r]), sr8 = h2f(vsc[r + 8]), zr = h2f(vze[r]), zr8 = h2f(vze[r + 8]);
            l0 += p0v + p2v;
            l1 += p1v + p3v;
            z0 = fmaf(p0v, zr, fmaf(p2v, zr8, z0));
            z1 = fmaf(p1v, zr, fmaf(p3v, zr8, z1));
            uint32_t h01, l01, h23, l23;
            split_h2(p0v * sr, p1v * sr, h01, l01);
            split_h2(p2v * sr8, p3v * sr8, h23, l23);
            const uint32_t bh0 = movtrans(h01), bh1 = movtrans(h23);
            const uint32_t bl0 = movtrans(l01), bl1 = movtrans(l23);

            // ---------- values ----------
            // lane (r, qd): dims 16r..16r+15 of tokens 2qd, 2qd+1, 2qd+8, 2qd+9
            const uint8_t* vrow = pg + g.vcode_off + r * 8;
            const uint2 va = *reinterpret_cast<const uint2*>(vrow + (2 * qd) * 64);
            const uint2 vb = *reinterpret_cast<const uint2*>(vrow + (2 * qd + 1) * 64);
            const uint2 vc = *reinterpret_cast<const uint2*>(vrow + (2 * qd + 8) * 64);
            const uint2 vd = *reinterpret_cast<const uint2*>(vrow + (2 * qd + 9) * 64);
            const uint32_t wab[4] = {prmt(va.x, vb.x, 0x5410u), prmt(va.x, vb.x, 0x7632u),
                                     prmt(va.y, vb.y, 0x5410u), prmt(va.y, vb.y, 0x7632u)};
            const uint32_t wcd[4] = {prmt(vc.x, vd.x, 0x5410u), prmt(vc.x, vd.x, 0x7632u),
                                     prmt(vc.y, vd.y, 0x5410u), prmt(vc.y, vd.y, 0x7632u)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t fab[4], fcd[4];
                nib8_to_h2(wab[j], fab);
                nib8_to_h2(wcd[j], fcd);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int mt = 2 * j + hh;  // dims 16r + 2mt (row r) and 16r + 2mt + 1 (row r+8)
                    mma16816(acc[mt], fab[2 * hh], fab[2 * hh + 1], fcd[2 * hh], fcd[2 * hh + 1], bh0, bh1);
                    mma16816(acc[mt], fab[2 * hh], fab[2 * hh + 1], fcd[2 * hh], fcd[2 * hh + 1], bl0, bl1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
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
    if (warp == kNCW) __syncthreads();  // producer's side of (A)
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
        __threadfence();
        __syncthreads();
        __shared__ int s_last;
        if (tid == 0) s_last = (atomicAdd(a.counters + unit, 1u) == (unsigned)a.num_splits - 1);
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        finalize = true;
        if (warp < G) {
            const float* base = a.partials + (unit * a.num_splits * G) * kPartStride;
            Mx = -INFINITY;
            for (int sp = 0; sp < a.num_splits; ++sp) Mx = fmaxf(Mx, __ldcg(base + (sp * G + qg) * kPartStride));
            L = 0.f;
            O[0] = O[1] = O[2] = O[3] = 0.f;
            if (Mx != -INFINITY) {
                for (int sp = 0; sp < a.num_splits; ++sp) {
                    const float* pp = base + (sp * G + qg) * kPartStride;
                    const float ms = __ldcg(pp);
                    if (ms == -INFINITY) continue;
                    const float f = exp2f(ms - Mx);
                    L = fmaf(f, __ldcg(pp + 1), L);
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(pp + 4 + 4 * lane));
                    O[0] = fmaf(f, v.x, O[0]); O[1] = fmaf(f, v.y, O[1]);
                    O[2] = fmaf(f, v.z, O[2]); O[3] = fmaf(f, v.w, O[3]);
                }
            }
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
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    dim3 grid((unsigned)a.num_splits, (unsigned)a.g.hkv, (unsigned)a.batch);
    kern<<<grid, kThreads, smem, s>>>(a);
    return (int)cudaGetLastError();
}

int launch_decode(const DecodeArgs& a, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (a.g.kb == 4 && a.g.vb == 4 && a.g.m == 0) return launch_decode_t<4, 4, 0>(a, s);
    return (int)cudaErrorNotSupported;
}

}  // namespace tq
