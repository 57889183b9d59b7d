// OCTOPUS triplet key codec: encode, and decode attention on the tensor cores.
//
// Keys: gamma = ||k||, u = R k / gamma with the same rotation as the main
// codec; u is cut into 43 triplets (the last padded with a zero), each stored
// as a norm code (b-1 bits, levels fitted to the norm of three coordinates of
// a uniform point on S^127) and two direction codes (b+1 bits each) for the
// octahedral coordinates (xi, eta) of its direction, chosen by "3x3 joint
// rounding": among the nearest levels of xi and of eta and their neighbours,
// the pair whose direction is closest to the triplet's.  Values keep their
// per-token min-max codes.
// ["OCTOPUS: Optimized KV Cache for Transformers via Octahedral
//  Parametrization ..." -- key contribution "Octahedral triplet direction
//  quantizer with norm marginals", methodology steps 1-7, bit split (b+1, b-1)]
//
// Decode never builds K^ in global memory: for token t the logit is gamma_t
// times the sum over triplets of rho^_i <q_rot[3i..3i+2], n^_i>, with n^ the
// unit direction of the stored level pair (methodology step 7; the encode
// scores candidates against a table of them, the decode derives each from
// its two levels).  Each warp rebuilds rho^ n^ of one page in shared memory
// and scores it on the tensor cores; values accumulate in the rotated frame and one inverse
// rotation is applied per output.  The warps of a CTA merge in shared memory
// and write one partial per query; a second kernel merges the partials of a
// sequence.
#include <cuda_runtime.h>

#include "tq_decode_impl.cuh"  // the main codec's MMA, value-code and page-ring helpers
#include "tq_device.cuh"

namespace tq {

namespace {

constexpr float kOctMinus = -1.0e30f;

__device__ __forceinline__ uint32_t oct_signs(const uint32_t (&sb)[kHeadDim / 32], int lane) {
    return (sb[lane >> 3] >> (4 * (lane & 7))) & 0xFu;
}

// ---------------------------------------------------------------------------
// encode: one warp per (token, KV head); lane l holds coordinates 4l .. 4l+3
// ---------------------------------------------------------------------------
template <int B, int VB>
__global__ void __launch_bounds__(kOctWarps * 32) oct_encode_kernel(const OctArgs a) {
    constexpr int NXI = 1 << (B + 1), NRHO = 1 << (B - 1), FB = 3 * B + 1;
    constexpr int D = kHeadDim, VMAX = (1 << VB) - 1;
    __shared__ float s_u[kOctWarps][D + 4];
    __shared__ uint32_t s_row[kOctWarps][24];
    __shared__ float s_bxi[NXI], s_brho[NRHO];
    __shared__ float4 s_dir[NXI * NXI];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = threadIdx.x; i < NXI * NXI; i += blockDim.x) {
        const int pa = i / NXI, pb = i % NXI;
        const float* d4 = a.tab->dir[pa * kOctMaxDir + pb];
        s_dir[i] = make_float4(d4[0], d4[1], d4[2], 0.f);
    }
    for (int i = threadIdx.x; i < NXI; i += blockDim.x) s_bxi[i] = a.tab->bxi[i];
    for (int i = threadIdx.x; i < NRHO; i += blockDim.x) s_brho[i] = a.tab->brho[i];
    __syncthreads();
    const Geometry& g = a.g;
    const int hkv = g.hkv;
    const int64_t items = a.num_tokens * hkv;
    const int64_t cap = g.num_blocks * kBlockSize;
    const uint32_t sg = oct_signs(a.sign_bits, lane);
    const float inv_sqrt_d = 0.08838834764831845f;
    for (int64_t it = (int64_t)blockIdx.x * kOctWarps + warp; it < items; it += (int64_t)gridDim.x * kOctWarps) {
        const int64_t t = it / hkv;
        const int h = (int)(it - t * hkv);
        const int64_t slot = a.slot_mapping[t];
        const bool store = slot >= 0 && slot < cap;
        if (slot >= cap && lane == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
        float k[4], v[4];
        load4(a.K, a.dtype, it * D + 4 * lane, k);
        load4(a.V, a.dtype, it * D + 4 * lane, v);
        float z = 0.f, ss = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            z = fmaf(k[i], 0.f, fmaf(v[i], 0.f, z));
            ss = fmaf(k[i], k[i], ss);
        }
        const bool finite = warp_sum(z) == 0.f;
        if (store && !finite && lane == 0) flag(a.status, TQ_FLAG_NONFINITE);
        const float gamma = sqrtf(warp_sum(ss));
        apply_signs(k, sg);
        fwht128(k, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) s_u[warp][4 * lane + i] = (gamma > 0.f) ? (k[i] * inv_sqrt_d) / gamma : 0.f;
        if (lane < 4) s_u[warp][D + lane] = 0.f;
        if (lane < 24) s_row[warp][lane] = 0u;
        __syncwarp();
        for (int i = lane; i < kOctTri; i += 32) {
            const float t0 = s_u[warp][3 * i], t1 = s_u[warp][3 * i + 1], t2 = s_u[warp][3 * i + 2];
            const float rho = sqrtf(fmaf(t0, t0, fmaf(t1, t1, t2 * t2)));
            float n0 = 0.f, n1 = 0.f, n2 = 1.f;
            if (rho > 0.f) {
                n0 = t0 / rho;
                n1 = t1 / rho;
                n2 = t2 / rho;
            }
            int ir = 0;
#pragma unroll
            for (int j = 0; j < NRHO - 1; ++j) ir += (s_brho[j] < rho) ? 1 : 0;
            // octahedral coordinates: project onto |x| + |y| + |z| = 1, fold the lower half
            const float l1 = fabsf(n0) + fabsf(n1) + fabsf(n2);
            const float px = n0 / l1, py = n1 / l1;
            float xi = px, eta = py;
            if (n2 < 0.f) {
                xi = (1.f - fabsf(py)) * (px < 0.f ? -1.f : 1.f);
                eta = (1.f - fabsf(px)) * (py < 0.f ? -1.f : 1.f);
            }
            // nearest levels: #{boundaries < x} by binary search (the same count)
            int ia = 0, ie = 0;
#pragma unroll
            for (int step = NXI / 2; step >= 1; step >>= 1) {
                if (s_bxi[ia + step - 1] < xi) ia += step;
                if (s_bxi[ie + step - 1] < eta) ie += step;
            }
            // 3 x 3 joint rounding: the neighbouring level pair closest in direction
            float best = -3.f;
            int ba = ia, bb = ie;
#pragma unroll
            for (int da = -1; da <= 1; ++da) {
                const int aa = ia + da;
                if (aa < 0 || aa >= NXI) continue;
#pragma unroll
                for (int db = -1; db <= 1; ++db) {
                    const int bq = ie + db;
                    if (bq < 0 || bq >= NXI) continue;
                    const float4 d4 = s_dir[aa * NXI + bq];
                    const float sc = fmaf(n0, d4.x, fmaf(n1, d4.y, n2 * d4.z));
                    if (sc > best) {
                        best = sc;
                        ba = aa;
                        bb = bq;
                    }
                }
            }
            const uint32_t field = (uint32_t)ba | ((uint32_t)bb << (B + 1)) | ((uint32_t)ir << (2 * (B + 1)));
            const int pos = i * FB, sh = pos & 31;
            atomicOr(&s_row[warp][pos >> 5], field << sh);
            if (sh + FB > 32) atomicOr(&s_row[warp][(pos >> 5) + 1], field >> (32 - sh));
        }
        __syncwarp();
        const int64_t blk = store ? (slot >> 4) : 0;
        const int off = (int)(slot & (kBlockSize - 1));
        uint8_t* page = a.pool + (blk * hkv + h) * g.page_bytes;
        if (store && lane < a.key_row / 4)
            reinterpret_cast<uint32_t*>(page + off * a.key_row)[lane] = s_row[warp][lane];

        // ---- value: rotate, per-token min / max, codes ----
        apply_signs(v, sg);
        fwht128(v, lane);
        float lo = 3.4e38f, hi = -3.4e38f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] *= inv_sqrt_d;
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
        uint8_t* vrow = page + g.vcode_off + off * (D * VB / 8);
        if constexpr (VB == 8) {
            if (store) reinterpret_cast<uint32_t*>(vrow)[lane] = vp;
        } else if constexpr (VB == 4) {
            if (store) reinterpret_cast<uint16_t*>(vrow)[lane] = (uint16_t)vp;
        } else if constexpr (VB == 2) {
            if (store) vrow[lane] = (uint8_t)vp;
        } else {
            const uint32_t w = row_word<VB>(vp, lane);
            if (store && lane < 4 * VB) reinterpret_cast<uint32_t*>(vrow)[lane] = w;
        }
        if (store && lane == 0) {
            const uint16_t hg = f16_bits(gamma), hs = f16_bits(scale), hz = f16_bits(mn);
            reinterpret_cast<uint16_t*>(page + g.gam_off)[off] = hg;
            reinterpret_cast<uint16_t*>(page + g.scl_off)[off] = hs;
            reinterpret_cast<uint16_t*>(page + g.zer_off)[off] = hz;
            const bool ovf = ((hg & 0x7FFF) == 0x7C00) || ((hs & 0x7FFF) == 0x7C00) || ((hz & 0x7FFF) == 0x7C00);
            if (ovf && finite) flag(a.status, TQ_FLAG_OVERFLOW);
        }
        __syncwarp();  // s_u / s_row are rewritten by the next item
    }
}

// ---------------------------------------------------------------------------
// decode: grid (split, KV head, sequence), kOctDecWarps warps, one CTA per SM.
// Warp w takes pages p0 + w, p0 + w + NW, ... of the split and streams them
// into its own ring slots with bulk async copies completing on mbarriers.  Per
// page the warp
//  - rebuilds the rotated unit keys rho^ n^ of its 16 tokens into shared
//    memory (fp32, times kOctUScale), one triplet per lane at a time; the
//    levels come from registers by shuffles and the direction is decoded
//    from them (a random lookup in a shared-memory direction table cost
//    several bank wavefronts per warp and made the rebuild
//    shared-memory-bound);
//  - scores them against the group's queries on the tensor cores
//    (mma.sync m16n8k16, tokens as rows, queries as the n8 side): the keys
//    and the queries are each split into fp16 hi + lo, and the three products
//    hi.hi + hi.lo + lo.hi are accumulated in fp32;
//  - keeps the online softmax and accumulates the min-max values exactly as
//    the main codec's decode does (value codes as exact fp16 subnormals, the
//    zero-point term and the weight rounding kept in fp32).
// The warps merge in shared memory and each CTA writes one partial per query;
// oct_combine_kernel merges the splits and rotates back.
// ---------------------------------------------------------------------------
constexpr int kOctDecWarps = 16;  // 12 warps: 8 % slower (dependency stalls in the key rebuild)
constexpr int kOctMaxSlots = 3;                 // ring slots per warp (fewer if the pages are large)
constexpr int kOctUStride = kHeadDim + 8;       // floats per rebuilt row: consecutive rows 8 banks apart
constexpr float kOctUScale = 64.f;              // |rho^ n^| <= 1: rebuilt keys are taken times 64

// Page of an OCTOPUS cache: 16 key rows of KR bytes, then the value rows,
// gamma, scale and zero, padded to 16 bytes.
template <int B, int VB>
struct OctPage {
    static constexpr int KR = 4 * ((kOctTri * (3 * B + 1) + 31) / 32);
    static constexpr int vcode = kBlockSize * KR;
    static constexpr int gam = vcode + kBlockSize * kHeadDim * VB / 8;
    static constexpr int scl = gam + 2 * kBlockSize;
    static constexpr int zer = scl + 2 * kBlockSize;
    static constexpr int bytes = (zer + 2 * kBlockSize + 15) / 16 * 16;
};

// Shared memory of the decode kernel (byte offsets).  After the page loop the
// rebuilt-key area holds the warps' states for the in-CTA merge:
// [NW][8 queries][4 + d] floats (max, sum, zero term, pad, acc).
struct OctSmem {
    int q, qsc, qf, bars, never, ok, u, pages, slot, spw, total;
};
template <int B, int VB>
__host__ __device__ constexpr OctSmem oct_dec_smem() {
    OctSmem L{};
    int off = 0;
    L.q = off; off += 8 * (kHeadDim + 4) * 4;
    L.qsc = off; off += 8 * 4;
    L.qf = off; off += 8 * 32 * 16;
    L.bars = off; off += kOctDecWarps * kOctMaxSlots * 8;
    L.never = off; off += 8;  // a barrier nothing arrives on (the wait-timeout test hook)
    L.ok = off; off += kOctDecWarps * kOctMaxSlots * 4;
    off = (off + 15) / 16 * 16;
    L.u = off; off += kOctDecWarps * kBlockSize * kOctUStride * 4;
    L.slot = OctPage<B, VB>::bytes;
    L.pages = off;
    int spw = kOctMaxSlots;
    while (spw > 1 && off + kOctDecWarps * spw * L.slot > kSmemLimit) --spw;
    L.spw = spw;
    off += kOctDecWarps * spw * L.slot;
    L.total = off;
    return L;
}
static_assert(kOctDecWarps * 8 * (4 + kHeadDim) * 4 <= kOctDecWarps * kBlockSize * kOctUStride * 4,
              "the merge states must fit over the rebuilt keys");

// fp16 hi + lo of a pair of floats: hi = rn(x), lo = rn(x - hi)
__device__ __forceinline__ void split_h2(float2 x, uint32_t& hi, uint32_t& lo) {
    hi = pack_h2(x.x, x.y);
    const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    lo = pack_h2(x.x - h.x, x.y - h.y);
}

template <int B, int VB>
__global__ void __launch_bounds__(kOctDecWarps * 32, 1) oct_decode_kernel(const OctArgs a) {
    using P = OctPage<B, VB>;
    constexpr OctSmem LY = oct_dec_smem<B, VB>();
    constexpr int NW = kOctDecWarps, SPW = LY.spw;
    constexpr int NXI = 1 << (B + 1), FB = 3 * B + 1, D = kHeadDim, QS = D + 4, US = kOctUStride;
    constexpr uint32_t kFMask = (1u << FB) - 1u;
    static_assert((kBlockSize - 1) * P::KR + ((kOctTri - 1) * FB / 32) * 4 + 8 <= P::bytes,
                  "the two words of every key field lie inside the page");
    static_assert(LY.total <= kSmemLimit, "OCTOPUS decode does not fit in shared memory");
    extern __shared__ __align__(128) uint8_t sm[];
    const Geometry& g = a.g;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = a.group;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar_w = sbase + LY.bars + 8 * warp * kOctMaxSlots;
    const uint32_t ring_w = sbase + LY.pages + warp * SPW * LY.slot;
    int* slot_ok = reinterpret_cast<int*>(sm + LY.ok) + warp * kOctMaxSlots;
    float* s_q = reinterpret_cast<float*>(sm + LY.q);
    float* s_qsc = reinterpret_cast<float*>(sm + LY.qsc);
    float* s_u = reinterpret_cast<float*>(sm + LY.u) + warp * kBlockSize * US;

    if (lane == 0) {
        for (int k = 0; k < SPW; ++k) mbar_init(bar_w + 8 * k, 1);
        if (warp == 0) mbar_init(sbase + LY.never, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dependency_wait();
    grid_launch_dependents();

    // ---- length, this warp's block ids (lane l: the warp's page l of the
    // current batch of 32, and of the next batch) ----
    int len = __ldg(a.lens + b);
    if (len < 0) len = 0;
    if (len > a.max_blocks * kBlockSize) {
        if (tid == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
        len = a.max_blocks * kBlockSize;
    }
    const int p0 = split * a.pages_per_split;
    int npages = (len + kBlockSize - 1) / kBlockSize - p0;
    if (npages > a.pages_per_split) npages = a.pages_per_split;
    if (npages < 0) npages = 0;
    const int nmine = npages > warp ? (npages - warp + NW - 1) / NW : 0;
    const int32_t* btw = a.block_table + (int64_t)b * a.bt_stride + p0 + warp;
    const int reach = min(a.pages_per_split, a.max_blocks - p0) - warp;
    int bid_cur = (NW * lane < reach) ? __ldg(btw + NW * lane) : -1;
    int bid_nxt = (NW * (32 + lane) < reach) ? __ldg(btw + NW * (32 + lane)) : -1;

    // Start a page copy into ring slot `slot`; a bad block id arrives on the
    // barrier without data and the page is skipped.
    auto issue = [&](int slot, int blk) {
        const bool ok = blk >= 0 && blk < g.num_blocks;
        const uint32_t bar = bar_w + 8 * slot;
        slot_ok[slot] = ok;
        if (ok) {
            mbar_arrive_tx(bar, (uint32_t)P::bytes);
            bulk_g2s(ring_w + slot * LY.slot, a.pool + ((int64_t)blk * g.hkv + h) * P::bytes, (uint32_t)P::bytes, bar);
        } else {
            flag(a.status, TQ_FLAG_BAD_SLOT);
            mbar_arrive(bar);
        }
    };
    __syncwarp();
    if (lane < SPW && lane < nmine) issue(lane, bid_cur);

    // ---- levels (lane l holds xi / eta level l and norm level l mod 8), and
    // the rotated queries times sm_scale log2(e) / qscale ----
    const float cx_l = a.tab->cxi[lane & (NXI - 1)];
    const float cr_l = a.tab->crho[lane & ((1 << (B - 1)) - 1)] * kOctUScale;
    if (warp < 8) {
        // qscale: a power of two putting max |x| / qscale in (256, 512]
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (warp < G) {
            load4(a.q, a.dtype, ((int64_t)b * a.hq + (int64_t)h * G + warp) * D + 4 * lane, x);
            apply_signs(x, oct_signs(a.sign_bits, lane));
            fwht128(x, lane);
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] *= 0.08838834764831845f * a.sm_scale_log2;
        }
        const float mx = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
        const float scl = (mx > 0.f) ? exp2f(ceilf(log2f(mx / 512.f))) : 1.f;
        const float inv = 1.f / scl;
#pragma unroll
        for (int i = 0; i < 4; ++i) s_q[warp * QS + 4 * lane + i] = x[i] * inv;
        if (lane == 0) s_qsc[warp] = scl / kOctUScale;
    }
    __syncthreads();

    // The B fragments of the queries, the same for every warp, once per CTA in
    // shared memory: entry (ks, lane) holds, for query lane / 4, dims
    // 16 ks + 2 (lane % 4) + {0, 1} and + {8, 9} in fp16 hi, then lo (read
    // back per k-step, which leaves the registers to the key rebuild).
    const uint32_t qf = sbase + LY.qf;
    if (tid < 8 * 32) {
        const int ks = tid >> 5, ln = tid & 31;
        const float* qr = s_q + (ln >> 2) * QS + 16 * ks + 2 * (ln & 3);
        uint32_t h0, h1, o0, o1;
        split_h2(*reinterpret_cast<const float2*>(qr), h0, o0);
        split_h2(*reinterpret_cast<const float2*>(qr + 8), h1, o1);
        *reinterpret_cast<uint4*>(sm + LY.qf + 16 * tid) = make_uint4(h0, h1, o0, o1);
    }
    __syncthreads();
    // lane (r, qd): r = token row / query of the B operand, qd = quad index
    const int r = lane >> 2, qd = lane & 3;
    const float qs0 = s_qsc[2 * qd], qs1 = s_qsc[2 * qd + 1];
    // Score row r holds token tr = r ^ ((r >> 1) & 1) (and row r + 8 token
    // tr + 8), so that the value loads (tokens of rows 2qd, 2qd+1) alternate
    // between the two halves of the bank space.
    const int tr = r ^ ((r >> 1) & 1);
    const int ta = (2 * qd) ^ (qd & 1), tb = (2 * qd + 1) ^ (qd & 1);
    const float* ua = s_u + tr * US + 2 * qd;  // A rows: token tr, then tr + 8
    const float* ub = ua + 8 * US;

    float m0 = kMinusBig, m1 = kMinusBig, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    bool timed_out = false;
    int slot = 0;
    uint32_t phase = 0;
    int issued = min(SPW, nmine);
    int jfail = nmine;
    if (a.stall_cycles > 0 && (split & 1) && warp == 0) {
        // test hook: a bounded wait on a barrier that nothing arrives on runs
        // out, and the warp takes the timeout path below before its first page
        if (!mbar_wait_for(sbase + LY.never, 0, a.stall_cycles)) {
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
        const uint32_t pg = ring_w + slot * LY.slot;
        const bool pok = slot_ok[slot] != 0;

        // ---------- rebuild u^ = rho^ n^ (times kOctUScale) of the 16 tokens ----------
        // Triplet i = lane of every token (its field sits at the same bits of
        // every key row), then the 11 x 16 triplets 32..42 spread over the lanes.
        // A field is cut from two consecutive words of its row; the second may
        // lie past the row but always inside the page.
        {
            // rho^ n^ of field f: the octahedron point (xi, eta, 1 - |xi| - |eta|),
            // folded into the lower half-space when that is negative, normalised
            // (the direction of the level pair, as the library's table has it)
            auto rebuild = [&](uint32_t f, float& x, float& y, float& z) {
                const float xi = __shfl_sync(0xffffffffu, cx_l, (int)(f & (NXI - 1)));
                const float eta = __shfl_sync(0xffffffffu, cx_l, (int)((f >> (B + 1)) & (NXI - 1)));
                const float rr = __shfl_sync(0xffffffffu, cr_l, (int)(f >> (2 * (B + 1))));
                z = 1.f - fabsf(xi) - fabsf(eta);
                const bool fold = z < 0.f;
                x = fold ? copysignf(1.f - fabsf(eta), xi) : xi;
                y = fold ? copysignf(1.f - fabsf(xi), eta) : eta;
                const float sc = rr * rsqrtf(fmaf(x, x, fmaf(y, y, z * z)));
                x *= sc;
                y *= sc;
                z *= sc;
            };
            const uint32_t kw = pg + ((lane * FB) >> 5) * 4;
            const int ksh = (lane * FB) & 31;
#pragma unroll
            for (int t = 0; t < kBlockSize; ++t) {
                const uint32_t f = __funnelshift_r(lds32(kw + t * P::KR), lds32(kw + t * P::KR + 4), ksh) & kFMask;
                float x, y, z;
                rebuild(f, x, y, z);
                float* u = s_u + t * US + 3 * lane;
                u[0] = x;
                u[1] = y;
                u[2] = z;
            }
            constexpr int kRest = kBlockSize * (kOctTri - 32);
#pragma unroll
            for (int n = 0; n < (kRest + 31) / 32; ++n) {
                const int k = lane + 32 * n;
                const bool act = k < kRest;  // every lane takes part in the shuffles
                const int t = act ? k / (kOctTri - 32) : 0, i = act ? 32 + k - (kOctTri - 32) * t : 32;
                const uint32_t w = pg + t * P::KR + ((i * FB) >> 5) * 4;
                const uint32_t f = __funnelshift_r(lds32(w), lds32(w + 4), (i * FB) & 31) & kFMask;
                float x, y, z;
                rebuild(f, x, y, z);
                if (act) {
                    float* u = s_u + t * US + 3 * i;
                    u[0] = x;
                    u[1] = y;
                    if (i < kOctTri - 1) u[2] = z;
                }
            }
        }
        __syncwarp();

        // ---------- scores: 3 products per k-step on four accumulator chains ----------
        float I0[4], I1[4], J0[4], J1[4];  // hi.hi (even / odd k-steps), hi.lo + lo.hi (even / odd)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint4 Q = lds128(qf + 16 * (32 * ks + lane));  // hi (x, y), lo (z, w)
            uint32_t h0, h1, h2, h3, o0, o1, o2, o3;
            split_h2(*reinterpret_cast<const float2*>(ua + 16 * ks), h0, o0);
            split_h2(*reinterpret_cast<const float2*>(ub + 16 * ks), h1, o1);
            split_h2(*reinterpret_cast<const float2*>(ua + 16 * ks + 8), h2, o2);
            split_h2(*reinterpret_cast<const float2*>(ub + 16 * ks + 8), h3, o3);
            float* I = (ks & 1) ? I1 : I0;
            float* J = (ks & 1) ? J1 : J0;
            if (ks < 2) {
                mma16816_c(I, h0, h1, h2, h3, Q.x, Q.y, 0.f, 0.f, 0.f, 0.f);
                mma16816_c(J, h0, h1, h2, h3, Q.z, Q.w, 0.f, 0.f, 0.f, 0.f);
            } else {
                mma16816(I, h0, h1, h2, h3, Q.x, Q.y);
                mma16816(J, h0, h1, h2, h3, Q.z, Q.w);
            }
            mma16816(J, o0, o1, o2, o3, Q.x, Q.y);
        }
        const float gr = lds_h2f(pg + P::gam + 2 * tr), gr8 = lds_h2f(pg + P::gam + 2 * (tr + 8));
        float s0 = ((I0[0] + I1[0]) + (J0[0] + J1[0])) * qs0 * gr, s1 = ((I0[1] + I1[1]) + (J0[1] + J1[1])) * qs1 * gr;
        float s2 = ((I0[2] + I1[2]) + (J0[2] + J1[2])) * qs0 * gr8, s3 = ((I0[3] + I1[3]) + (J0[3] + J1[3])) * qs1 * gr8;
        float sr, sr8, zr, zr8;
        const int tok = (p0 + warp + NW * j) * kBlockSize;
        if (pok && tok + kBlockSize <= len) {
            sr = lds_h2f(pg + P::scl + 2 * tr);
            sr8 = lds_h2f(pg + P::scl + 2 * (tr + 8));
            zr = lds_h2f(pg + P::zer + 2 * tr);
            zr8 = lds_h2f(pg + P::zer + 2 * (tr + 8));
        } else {
            // the sequence's last page or a skipped one (warp-uniform): rows
            // past the end get no weight, and their slots' bytes are not read
            const bool v0 = pok && tok + tr < len, v8 = pok && tok + tr + 8 < len;
            if (!v0) s0 = s1 = -INFINITY;
            if (!v8) s2 = s3 = -INFINITY;
            sr = v0 ? lds_h2f(pg + P::scl + 2 * tr) : 0.f;
            zr = v0 ? lds_h2f(pg + P::zer + 2 * tr) : 0.f;
            sr8 = v8 ? lds_h2f(pg + P::scl + 2 * (tr + 8)) : 0.f;
            zr8 = v8 ? lds_h2f(pg + P::zer + 2 * (tr + 8)) : 0.f;
        }

        // ---------- online softmax; the max moves only when a score beats it by kLazy ----------
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
        l0 += p0v + p2v;
        l1 += p1v + p3v;

        // ---------- values: O^T += Vcode^T . (p scale)^T, the main codec's arithmetic ----------
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
            value_codes<VB>(pg + P::vcode, r, ta, tb, Pab);
            value_codes<VB>(pg + P::vcode, r, ta + 8, tb + 8, Pcd);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)  // rows: dim 16r + 2mt (row r), 16r + 2mt + 1 (row r + 8)
                mma16816(acc[mt], Pab[2 * mt], Pab[2 * mt + 1], Pcd[2 * mt], Pcd[2 * mt + 1], bh0, bh1);
        }

        __syncwarp();  // every lane is done with the slot and with u^: refill the slot
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
        // copies this warp started must land before its shared memory goes away
        const long long t0 = clock64();
        for (int jj = jfail; jj < issued; ++jj) {
            const uint32_t bar = bar_w + 8 * (jj % SPW);
            while (!mbar_try(bar, (uint32_t)((jj / SPW) & 1)) && clock64() - t0 < kWaitCycles) {
            }
        }
    }

    // ---- reduce l, z over the 8 token rows; warp states over the rebuilt keys ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        z0 += __shfl_xor_sync(0xffffffffu, z0, o);
        z1 += __shfl_xor_sync(0xffffffffu, z1, o);
    }
    __syncthreads();  // every warp is past its pages: the rebuilt-key area is free
    float* wst = reinterpret_cast<float*>(sm + LY.u);  // [NW][8][4 + D]
    {
        float* pa = wst + (warp * 8 + 2 * qd) * (4 + D);
        float* pb = pa + (4 + D);
        if (r == 0) {
            pa[0] = m0; pa[1] = l0; pa[2] = z0;
            pb[0] = m1; pb[1] = l1; pb[2] = z1;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            // undo the fp16-subnormal scaling of the value codes of dims d, d + 1
            const float e0 = (float)(1u << (value_exp<VB>(2 * mt) - value_wshift<VB>()));
            const float e1 = (float)(1u << (value_exp<VB>(2 * mt + 1) - value_wshift<VB>()));
            const int d = 16 * r + 2 * mt;
            *reinterpret_cast<float2*>(pa + 4 + d) = make_float2(acc[mt][0] * e0, acc[mt][2] * e1);
            *reinterpret_cast<float2*>(pb + 4 + d) = make_float2(acc[mt][1] * e0, acc[mt][3] * e1);
        }
    }
    // A CTA with a wait that gave up flags it and writes an empty partial (max
    // -inf, sum 0, acc 0), so the combine kernel never reads a stale one.
    timed_out = __syncthreads_or(timed_out);
    if (timed_out && tid == 0) flag(a.status, TQ_FLAG_TIMEOUT);
    if (warp < G) {
        // query q = warp: this CTA's partial (max, sum, acc with the zero term folded in)
        const int q = warp;
        float* part = a.partials + ((((int64_t)b * g.hkv + h) * a.num_splits + split) * G + q) * (4 + D);
        if (timed_out) {
            if (lane == 0) {
                part[0] = kMinusBig;
                part[1] = 0.f;
            }
            *reinterpret_cast<float4*>(part + 4 + 4 * lane) = make_float4(0.f, 0.f, 0.f, 0.f);
            return;
        }
        float M = kMinusBig;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wst[(w * 8 + q) * (4 + D)]);
        float Ls = 0.f, Z = 0.f, x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* pq = wst + (w * 8 + q) * (4 + D);
            const float f = exp2f(pq[0] - M);
            Ls = fmaf(f, pq[1], Ls);
            Z = fmaf(f, pq[2], Z);
            const float4 v = *reinterpret_cast<const float4*>(pq + 4 + 4 * lane);
            x[0] = fmaf(f, v.x, x[0]); x[1] = fmaf(f, v.y, x[1]); x[2] = fmaf(f, v.z, x[2]); x[3] = fmaf(f, v.w, x[3]);
        }
        if (lane == 0) {
            part[0] = M;
            part[1] = Ls;
        }
        *reinterpret_cast<float4*>(part + 4 + 4 * lane) = make_float4(x[0] + Z, x[1] + Z, x[2] + Z, x[3] + Z);
    }
}

// One CTA per (sequence, query head): its warps split the partials of the
// splits, merge in shared memory, then out = R^T (acc / sum) =
// diag(s) H (acc / sum) / sqrt(d).
__global__ void __launch_bounds__(256) oct_combine_kernel(const OctArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float s_m[8], s_l[8];
    __shared__ float4 s_x[8][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = blockIdx.x;  // b * hq + query head
    const int b = (int)(row / a.hq), qh = (int)(row % a.hq);
    const int G = a.group, h = qh / G, q = qh % G;
    const int D = kHeadDim;
    const int np = a.num_splits;
    const int64_t ps = (int64_t)G * (4 + D);  // stride between the splits' partials
    const float* base = a.partials + (((int64_t)b * a.g.hkv + h) * np) * ps + q * (4 + D);
    float M = kOctMinus;
    for (int p = threadIdx.x; p < np; p += blockDim.x) M = fmaxf(M, base[p * ps]);
    M = warp_max(M);
    if (lane == 0) s_m[warp] = M;
    __syncthreads();
    M = s_m[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) M = fmaxf(M, s_m[w]);
    float Ls = 0.f, x[4] = {0.f, 0.f, 0.f, 0.f};
    for (int p = warp; p < np; p += 8) {
        const float f = exp2f(base[p * ps] - M);
        Ls = fmaf(f, base[p * ps + 1], Ls);
        const float4 v = *reinterpret_cast<const float4*>(base + p * ps + 4 + 4 * lane);
        x[0] = fmaf(f, v.x, x[0]); x[1] = fmaf(f, v.y, x[1]); x[2] = fmaf(f, v.z, x[2]); x[3] = fmaf(f, v.w, x[3]);
    }
    if (lane == 0) s_l[warp] = Ls;
    s_x[warp][lane] = make_float4(x[0], x[1], x[2], x[3]);
    __syncthreads();
    if (warp != 0) return;
    Ls = 0.f;
    x[0] = x[1] = x[2] = x[3] = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        Ls += s_l[w];
        const float4 v = s_x[w][lane];
        x[0] += v.x; x[1] += v.y; x[2] += v.z; x[3] += v.w;
    }
    const float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] *= inv;
    fwht128(x, lane);
    apply_signs(x, oct_signs(a.sign_bits, lane));
    *reinterpret_cast<float4*>(a.out + row * D + 4 * lane) =
        make_float4(x[0] * 0.08838834764831845f, x[1] * 0.08838834764831845f, x[2] * 0.08838834764831845f,
                    x[3] * 0.08838834764831845f);
}

template <int B, int VB>
int launch_oct_encode_t(const OctArgs& a, int num_sms, cudaStream_t s) {
    const int64_t items = a.num_tokens * a.g.hkv;
    int64_t blocks = (items + kOctWarps - 1) / kOctWarps;
    static int per_sm = 0;  // CTAs resident per SM: the grid is one wave
    if (per_sm == 0) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, oct_encode_kernel<B, VB>, kOctWarps * 32, 0);
        if (e != cudaSuccess) return (int)e;
        per_sm = n > 0 ? n : 1;
    }
    const int64_t cap = (int64_t)num_sms * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)launch_programmatic(oct_encode_kernel<B, VB>, dim3((unsigned)blocks), dim3(kOctWarps * 32), 0, s, a);
}

template <int B, int VB>
int launch_oct_decode_t(const OctArgs& a, cudaStream_t s) {
    using P = OctPage<B, VB>;
    const Geometry& g = a.g;
    if (g.page_bytes != P::bytes || g.kcode_off != 0 || g.vcode_off != P::vcode || g.gam_off != P::gam ||
        g.scl_off != P::scl || g.zer_off != P::zer || a.key_row != P::KR || g.bs != kBlockSize || g.d != kHeadDim)
        return (int)cudaErrorInvalidValue;  // the cache's geometry is not the format this kernel was built for
    constexpr int smem = oct_dec_smem<B, VB>().total;
    auto kern = oct_decode_kernel<B, VB>;
    static int done[64] = {};
    cudaError_t e = ensure_smem_limit(kern, smem, done);
    if (e != cudaSuccess) return (int)e;
    e = launch_programmatic(kern, dim3((unsigned)a.num_splits, (unsigned)a.g.hkv, (unsigned)a.batch),
                            dim3(kOctDecWarps * 32), (size_t)smem, s, a);
    if (e != cudaSuccess) return (int)e;
    const int64_t rows = (int64_t)a.batch * a.hq;
    return (int)launch_programmatic(oct_combine_kernel, dim3((unsigned)rows), dim3(256), 0, s, a);
}

template <int B>
int oct_encode_b(const OctArgs& a, int num_sms, cudaStream_t s) {
    switch (a.g.vb) {
        case 1: return launch_oct_encode_t<B, 1>(a, num_sms, s);
        case 2: return launch_oct_encode_t<B, 2>(a, num_sms, s);
        case 3: return launch_oct_encode_t<B, 3>(a, num_sms, s);
        case 4: return launch_oct_encode_t<B, 4>(a, num_sms, s);
        case 5: return launch_oct_encode_t<B, 5>(a, num_sms, s);
        case 6: return launch_oct_encode_t<B, 6>(a, num_sms, s);
        case 7: return launch_oct_encode_t<B, 7>(a, num_sms, s);
        case 8: return launch_oct_encode_t<B, 8>(a, num_sms, s);
        default: return (int)cudaErrorInvalidValue;
    }
}

template <int B>
int oct_decode_b(const OctArgs& a, cudaStream_t s) {
    switch (a.g.vb) {
        case 1: return launch_oct_decode_t<B, 1>(a, s);
        case 2: return launch_oct_decode_t<B, 2>(a, s);
        case 3: return launch_oct_decode_t<B, 3>(a, s);
        case 4: return launch_oct_decode_t<B, 4>(a, s);
        case 5: return launch_oct_decode_t<B, 5>(a, s);
        case 6: return launch_oct_decode_t<B, 6>(a, s);
        case 7: return launch_oct_decode_t<B, 7>(a, s);
        case 8: return launch_oct_decode_t<B, 8>(a, s);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace

int launch_oct_encode(const OctArgs& a, int num_sms, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (a.g.kb) {
        case 2: return oct_encode_b<2>(a, num_sms, s);
        case 3: return oct_encode_b<3>(a, num_sms, s);
        case 4: return oct_encode_b<4>(a, num_sms, s);
        default: return (int)cudaErrorInvalidValue;
    }
}

int launch_oct_decode(const OctArgs& a, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (a.g.kb) {
        case 2: return oct_decode_b<2>(a, s);
        case 3: return oct_decode_b<3>(a, s);
        case 4: return oct_decode_b<4>(a, s);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace tq
