// OCTOPUS triplet key codec: encode and decode attention on CUDA cores.
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
// Decode never builds K^: for token t the logit is gamma_t times the sum over
// triplets of rho^_i <q_rot[3i..3i+2], n^_i>, with n^ from a table of the
// level pairs' unit directions (methodology step 7); values accumulate in the
// rotated frame and one inverse rotation is applied per output.  Each CTA
// warp keeps an online softmax over its pages and writes its partial; a
// second kernel merges the partials of a sequence.
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {

namespace {

constexpr float kOctMinus = -1.0e30f;

__device__ __forceinline__ uint32_t oct_signs(const uint32_t (&sb)[kHeadDim / 32], int lane) {
    return (sb[lane >> 3] >> (4 * (lane & 7))) & 0xFu;
}

// bits [pos, pos + n) of a little-endian word array, 1 <= n <= 32; the next
// word is read only when the field reaches into it
__device__ __forceinline__ uint32_t oct_bits(const uint32_t* w, int pos, int n) {
    const int wi = pos >> 5, sh = pos & 31;
    uint32_t x = w[wi] >> sh;
    if (sh + n > 32) x |= w[wi + 1] << (32 - sh);
    return (n == 32) ? x : (x & ((1u << n) - 1u));
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
// decode: grid (split, KV head, sequence), kOctWarps warps; warp w takes pages
// p0 + w, p0 + w + kOctWarps, ... of the split.  Shared memory: the direction
// table, the norm levels, the rotated queries and one page per warp.
// ---------------------------------------------------------------------------
struct OctSmem {
    int dir, crho, q, pages, u, total;
};
constexpr int kOctHalf = kBlockSize / 2;  // tokens whose directions are rebuilt at a time
// a rebuilt direction row keeps each 32-dim part 4 floats apart from the next,
// so that the four parts read at once fall in different banks
constexpr int kOctURow = 4 * 36;
__host__ __device__ constexpr int oct_upos(int c) { return c + 4 * (c >> 5); }
// After the page loop the whole area holds the warps' partials for the in-CTA
// merge: [kOctWarps][8 queries][4 + d] floats.
constexpr int kOctMergeBytes = kOctWarps * 8 * (4 + kHeadDim) * 4;
__host__ __device__ inline OctSmem oct_smem(int nxi, int page_bytes) {
    OctSmem L{};
    int off = 0;
    L.dir = off; off += nxi * nxi * 16;
    L.crho = off; off += 8 * 4;
    L.q = off; off += 8 * (kHeadDim + 4) * 4;
    L.pages = off; off += kOctWarps * ((page_bytes + 15) / 16 * 16);
    L.u = off; off += kOctWarps * kOctHalf * kOctURow * 4;
    L.total = off > kOctMergeBytes ? off : kOctMergeBytes;
    return L;
}

template <int B, int VB>
__global__ void __launch_bounds__(kOctWarps * 32, 2) oct_decode_kernel(const OctArgs a) {
    constexpr int NXI = 1 << (B + 1), FB = 3 * B + 1, D = kHeadDim, QS = D + 4;
    constexpr int VROW = D * VB / 8;
    extern __shared__ __align__(16) uint8_t sm[];
    const Geometry& g = a.g;
    const OctSmem L = oct_smem(NXI, (int)g.page_bytes);
    float4* s_dir = reinterpret_cast<float4*>(sm + L.dir);
    float* s_crho = reinterpret_cast<float*>(sm + L.crho);
    float* s_q = reinterpret_cast<float*>(sm + L.q);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = a.group;
    uint8_t* s_page = sm + L.pages + warp * (int)((g.page_bytes + 15) / 16 * 16);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = threadIdx.x; i < NXI * NXI; i += blockDim.x) {
        const float* d4 = a.tab->dir[(i / NXI) * kOctMaxDir + i % NXI];
        s_dir[i] = make_float4(d4[0], d4[1], d4[2], 0.f);
    }
    if (threadIdx.x < 8) s_crho[threadIdx.x] = a.tab->crho[threadIdx.x];
    if (warp < G) {
        // rotated query, times sm_scale log2(e); coordinate 128 (the padded
        // triplet's third) is zero
        float x[4];
        load4(a.q, a.dtype, ((int64_t)b * a.hq + (int64_t)h * G + warp) * D + 4 * lane, x);
        apply_signs(x, oct_signs(a.sign_bits, lane));
        fwht128(x, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) s_q[warp * QS + 4 * lane + i] = x[i] * 0.08838834764831845f * a.sm_scale_log2;
        if (lane < 4) s_q[warp * QS + D + lane] = 0.f;
    }
    __syncthreads();

    int len = __ldg(a.lens + b);
    if (len > a.max_blocks * kBlockSize) {
        if (threadIdx.x == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
        len = a.max_blocks * kBlockSize;
    }
    if (len < 0) len = 0;
    const int p0 = split * a.pages_per_split;
    int pend = (len + kBlockSize - 1) / kBlockSize;
    if (pend > p0 + a.pages_per_split) pend = p0 + a.pages_per_split;

    // Scores: lane (query g = lane / 4, part = lane % 4) keeps dims 32 part ..
    // 32 part + 31 of its rotated query in registers and dots them with the
    // page's rebuilt rotated key directions; a query's 4 lanes then sum their
    // parts.  Softmax state per query lives in its lanes.  Values: lane l
    // accumulates dims 4l .. 4l+3 of every query.
    const int gq = lane >> 2, part = lane & 3;
    float qreg[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) qreg[c] = (gq < G) ? s_q[gq * QS + 32 * part + c] : 0.f;
    float* s_u = reinterpret_cast<float*>(sm + L.u) + warp * kOctHalf * kOctURow;
    float m_g = kOctMinus, l_g = 0.f;
    float acc[8][4];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
    for (int pi = p0 + warp; pi < pend; pi += kOctWarps) {
        const int blk = __ldg(a.block_table + (int64_t)b * a.bt_stride + pi);
        if (blk < 0 || blk >= g.num_blocks) {
            if (lane == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
            continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(a.pool + ((int64_t)blk * g.hkv + h) * g.page_bytes);
        for (int k = lane; k < (int)(g.page_bytes / 16); k += 32) reinterpret_cast<uint4*>(s_page)[k] = __ldg(src + k);
        __syncwarp();
        float sc[kBlockSize];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            // rebuild u^ = rho^ n^ of tokens 8 hf .. 8 hf + 7 (all 43 triplets)
            for (int j = lane; j < kOctHalf * kOctTri; j += 32) {
                const int t = j / kOctTri, i = j - t * kOctTri;
                const uint32_t* row = reinterpret_cast<const uint32_t*>(s_page + (kOctHalf * hf + t) * a.key_row);
                const uint32_t f = oct_bits(row, i * FB, FB);
                const int ia = f & (NXI - 1), ie = (f >> (B + 1)) & (NXI - 1), ir = f >> (2 * (B + 1));
                const float4 d4 = s_dir[ia * NXI + ie];
                const float r = s_crho[ir];
                float* u = s_u + t * kOctURow;
                u[oct_upos(3 * i)] = r * d4.x;
                u[oct_upos(3 * i + 1)] = r * d4.y;
                if (3 * i + 2 < D) u[oct_upos(3 * i + 2)] = r * d4.z;
            }
            __syncwarp();
#pragma unroll
            for (int t = 0; t < kOctHalf; ++t) {
                const float4* u4 = reinterpret_cast<const float4*>(s_u + t * kOctURow + 36 * part);
                float x = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 v = u4[c];
                    x = fmaf(v.x, qreg[4 * c], fmaf(v.y, qreg[4 * c + 1], fmaf(v.z, qreg[4 * c + 2], fmaf(v.w, qreg[4 * c + 3], x))));
                }
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                sc[kOctHalf * hf + t] = x;
            }
            __syncwarp();  // s_u is rebuilt for the second half
        }
        // ---- online softmax, query gq's state in its four lanes ----
        float mx = kOctMinus;
#pragma unroll
        for (int t = 0; t < kBlockSize; ++t) {
            const float gam = __half2float(*reinterpret_cast<const __half*>(s_page + g.gam_off + 2 * t));
            const bool valid = pi * kBlockSize + t < len;
            sc[t] = valid ? sc[t] * gam : -INFINITY;
            mx = fmaxf(mx, sc[t]);
        }
        float fct = 1.f;
        if (mx > m_g) {
            fct = exp2f(m_g - mx);
            l_g *= fct;
            m_g = mx;
        }
        // weights to shared memory (over the rebuilt directions, no longer
        // needed): p[t][query]; a query's part-0 lane writes them
#pragma unroll
        for (int t = 0; t < kBlockSize; ++t) {
            sc[t] = exp2f(sc[t] - m_g);  // -inf gives 0
            l_g += sc[t];
            if (part == 0) s_u[t * 8 + gq] = sc[t];
        }
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (q >= G) continue;
            const float f = __shfl_sync(0xffffffffu, fct, 4 * q);
            acc[q][0] *= f; acc[q][1] *= f; acc[q][2] *= f; acc[q][3] *= f;
        }
        // ---- values: lane holds dims 4 lane .. 4 lane + 3 ----
        for (int t = 0; t < kBlockSize; ++t) {
            const uint32_t* vr = reinterpret_cast<const uint32_t*>(s_page + g.vcode_off + t * VROW);
            const uint32_t cw = oct_bits(vr, 4 * lane * VB, 4 * VB);
            const float scl = __half2float(*reinterpret_cast<const __half*>(s_page + g.scl_off + 2 * t));
            const float zer = __half2float(*reinterpret_cast<const __half*>(s_page + g.zer_off + 2 * t));
            float vv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) vv[k] = fmaf(scl, (float)((cw >> (VB * k)) & ((1u << VB) - 1u)), zer);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q >= G) continue;
                const float pt = s_u[t * 8 + q];
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[q][k] = fmaf(pt, vv[k], acc[q][k]);
            }
        }
        __syncwarp();  // the page buffer is refilled next
    }
    float m[8], l[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        m[q] = __shfl_sync(0xffffffffu, m_g, 4 * q);
        l[q] = __shfl_sync(0xffffffffu, l_g, 4 * q);
    }
    // ---- merge the warps in shared memory; warp q writes the CTA's partial
    // for query q: (max, sum, 2 pad, acc[128]) ----
    __syncthreads();  // every warp is past its pages: the area is free
    float* wst = reinterpret_cast<float*>(sm);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        if (q >= G) continue;
        float* pq = wst + (warp * 8 + q) * (4 + D);
        if (lane == 0) {
            pq[0] = m[q];
            pq[1] = l[q];
        }
        *reinterpret_cast<float4*>(pq + 4 + 4 * lane) = make_float4(acc[q][0], acc[q][1], acc[q][2], acc[q][3]);
    }
    __syncthreads();
    if (warp < G) {
        const int q = warp;
        float M = kOctMinus;
#pragma unroll
        for (int w = 0; w < kOctWarps; ++w) M = fmaxf(M, wst[(w * 8 + q) * (4 + D)]);
        float Ls = 0.f, x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kOctWarps; ++w) {
            const float* pq = wst + (w * 8 + q) * (4 + D);
            const float f = exp2f(pq[0] - M);
            Ls = fmaf(f, pq[1], Ls);
            const float4 v = *reinterpret_cast<const float4*>(pq + 4 + 4 * lane);
            x[0] = fmaf(f, v.x, x[0]); x[1] = fmaf(f, v.y, x[1]); x[2] = fmaf(f, v.z, x[2]); x[3] = fmaf(f, v.w, x[3]);
        }
        float* part = a.partials + ((((int64_t)b * g.hkv + h) * a.num_splits + split) * G + q) * (4 + D);
        if (lane == 0) {
            part[0] = M;
            part[1] = Ls;
        }
        *reinterpret_cast<float4*>(part + 4 + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
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
    const int smem = oct_smem(1 << (B + 1), (int)a.g.page_bytes).total;
    auto kern = oct_decode_kernel<B, VB>;
    static int done[64] = {};
    cudaError_t e = ensure_smem_limit(kern, smem, done);
    if (e != cudaSuccess) return (int)e;
    e = launch_programmatic(kern, dim3((unsigned)a.num_splits, (unsigned)a.g.hkv, (unsigned)a.batch),
                            dim3(kOctWarps * 32), (size_t)smem, s, a);
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

int oct_decode_smem_bytes(const OctArgs& a) {
    return oct_smem(1 << (a.g.kb + 1), (int)a.g.page_bytes).total;
}

}  // namespace tq
