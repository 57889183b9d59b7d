// Encode kernel: compress new key/value vectors into the paged cache.
//
// One warp per (token, KV head).  Lane l holds coordinates 4l..4l+3 of the key
// and then of the value.
//   key:   gamma = ||k|| (warp sum of squares), u_rot = FWHT(s (.) k) / (sqrt(d) gamma),
//          code_j = #{ boundaries < u_rot[j] }; with QJL, r = u_rot - C[code],
//          rho = ||r||, sigma_i = [(S r)_i >= 0] with S staged in shared memory
//   value: v_rot = FWHT(s (.) v) / sqrt(d), per-token min/max (warp reductions),
//          code = clamp(rint((v_rot - min) / scale), 0, 2^b - 1)
// ["TurboQuant: KV Cache Vector Quantization" -- three steps; deep dive
//  (cell-devlog) -- Step 1 (RHT), Step 3 (value codes); Bit-Axon --
//  quantization function; "OCTOPUS ..." -- methodology steps 1, 2, 8]
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {

constexpr int kEncWarps = 8;
constexpr int kSPad = kHeadDim + 1;  // padded row stride of S in shared memory

// One 128-code row, lane holding the 4*B bits of codes 4 lane .. 4 lane + 3:
// 2- and 4-bit rows are plain byte / halfword stores, 3-bit rows go through
// the shuffle packer.
template <int B>
__device__ __forceinline__ void store_codes(uint8_t* row, uint32_t p, int lane) {
    if constexpr (B == 4) reinterpret_cast<uint16_t*>(row)[lane] = (uint16_t)p;
    else if constexpr (B == 2) row[lane] = (uint8_t)p;
    else store_code_row<B>(row, p, lane);
}

template <int KB, int VB, int M>
__global__ void __launch_bounds__(kEncWarps * 32) encode_kernel(const EncodeArgs a) {
    extern __shared__ float smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const Geometry& g = a.g;
    constexpr int D = kHeadDim;
    constexpr int NB = (1 << KB) - 1;
    constexpr int VMAX = (1 << VB) - 1;
    constexpr int HALF = 1 << (KB - 1);
    float* Ss = smem;                       // [M][kSPad]
    float* rbuf = smem + M * kSPad + warp * D;
    // launched as a programmatic dependent: wait for the previous grid before
    // touching global memory, and let the next one start launching
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (M > 0) {
        for (int i = threadIdx.x; i < M * D; i += blockDim.x) Ss[(i / D) * kSPad + (i % D)] = a.S[i];
        __syncthreads();
    }
    const uint32_t sm = lane_signs(a.c, lane);
    const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
    const int hkv = g.hkv;
    const int64_t items = a.num_tokens * hkv;
    const int64_t cap = g.num_blocks * kBlockSize;

    // Item it = t * hkv + h.  The grid-stride loop keeps (t, h) incrementally
    // (no 64-bit division per item) and loads the next item's K, V and slot
    // while the current one is coded.
    const int64_t stride = (int64_t)gridDim.x * kEncWarps;
    const int64_t st_t = stride / hkv;
    const int st_h = (int)(stride - st_t * hkv);
    int64_t it = (int64_t)blockIdx.x * kEncWarps + warp;
    int64_t t = it / hkv;
    int h = (int)(it - t * hkv);
    float kn[4] = {0.f, 0.f, 0.f, 0.f}, vn[4] = {0.f, 0.f, 0.f, 0.f};
    int64_t slot_n = -1;
    if (it < items) {
        load4(a.K, a.dtype, it * D + 4 * lane, kn);
        load4(a.V, a.dtype, it * D + 4 * lane, vn);
        slot_n = a.slot_mapping[t];
    }
    for (; it < items; it += stride) {
        float k[4], v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) { k[i] = kn[i]; v[i] = vn[i]; }
        const int64_t slot = slot_n;
        const int hc = h;
        // advance to the next item and start its loads
        t += st_t;
        h += st_h;
        if (h >= hkv) { h -= hkv; ++t; }
        if (it + stride < items) {
            load4(a.K, a.dtype, (it + stride) * D + 4 * lane, kn);
            load4(a.V, a.dtype, (it + stride) * D + 4 * lane, vn);
            slot_n = a.slot_mapping[t];
        }
        if (slot < 0) continue;
        if (slot >= cap) {
            if (lane == 0) flag(a.status, TQ_FLAG_BAD_SLOT);
            continue;
        }
        static_assert(kBlockSize == 16, "page index by shift");
        const int64_t blk = slot >> 4;
        const int off = (int)(slot & (kBlockSize - 1));
        uint8_t* page = a.pool + (blk * hkv + hc) * g.page_bytes;
        // x * 0 is 0 for every finite x and NaN for inf / NaN
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) z = fmaf(k[i], 0.f, fmaf(v[i], 0.f, z));
        const bool finite = (z == 0.f);
        if (!__all_sync(0xffffffffu, finite) && lane == 0) flag(a.status, TQ_FLAG_NONFINITE);

        // ---- key ----
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) ss = fmaf(k[i], k[i], ss);
        const float gamma = sqrtf(warp_sum(ss));
        apply_signs(k, sm);
        fwht128(k, lane);
        uint32_t kp = 0;
        float r[4];
        if (gamma > 0.f) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float u = (k[i] * inv_sqrt_d) / gamma;  // correctly rounded: keeps ties with the codebook rare
                // The codebook is symmetric (t_b = -t_{NB-1-b}, middle boundary 0), so
                // code = #{t_b < u} is HALF + #{positive t_b < |u|} for u > 0 and
                // HALF - 1 - #{positive t_b <= |u|} otherwise; the two differ from the
                // plain count only at a tie with a boundary.
                const float au = fabsf(u);
                int n = 0;
#pragma unroll
                for (int b = HALF; b < NB; ++b) n += (a.c.boundary[b] < au) ? 1 : 0;
                const int c = (u > 0.f) ? HALF + n : HALF - 1 - n;
                kp |= (uint32_t)c << (KB * i);
                if constexpr (M > 0) {
                    float cv = 0.f;
#pragma unroll
                    for (int b = 0; b <= NB; ++b) cv = (c == b) ? a.c.centroid[b] : cv;
                    r[i] = u - cv;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                kp |= (uint32_t)((1 << (KB - 1)) - 1) << (KB * i);
                r[i] = 0.f;
            }
        }
        store_codes<KB>(page + g.kcode_off + off * (D * KB / 8), kp, lane);

        float rho = 0.f;
        if constexpr (M > 0) {
            float rr = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                rbuf[4 * lane + i] = r[i];
                rr = fmaf(r[i], r[i], rr);
            }
            rho = sqrtf(warp_sum(rr));
            __syncwarp();
            uint32_t* sig = reinterpret_cast<uint32_t*>(page + g.sig_off + off * (M / 8));
#pragma unroll
            for (int w = 0; w < M / 32; ++w) {
                const float* srow = Ss + (w * 32 + lane) * kSPad;
                float dot = 0.f;
#pragma unroll 8
                for (int j = 0; j < D; ++j) dot = fmaf(srow[j], rbuf[j], dot);
                const uint32_t bits = __ballot_sync(0xffffffffu, dot >= 0.f);
                if (lane == w) sig[w] = (gamma > 0.f) ? bits : 0xffffffffu;
            }
            __syncwarp();
        }

        // ---- value ----
        apply_signs(v, sm);
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
        store_codes<VB>(page + g.vcode_off + off * (D * VB / 8), vp, lane);

        if (lane == 0) {
            const uint16_t hg = f16_bits(gamma), hs = f16_bits(scale), hz = f16_bits(mn);
            reinterpret_cast<uint16_t*>(page + g.gam_off)[off] = hg;
            reinterpret_cast<uint16_t*>(page + g.scl_off)[off] = hs;
            reinterpret_cast<uint16_t*>(page + g.zer_off)[off] = hz;
            bool ovf = ((hg & 0x7FFF) == 0x7C00) || ((hs & 0x7FFF) == 0x7C00) || ((hz & 0x7FFF) == 0x7C00);
            if constexpr (M > 0) {
                const uint16_t hr = f16_bits(rho);
                reinterpret_cast<uint16_t*>(page + g.rho_off)[off] = hr;
                ovf = ovf || ((hr & 0x7FFF) == 0x7C00);
            }
            if (ovf && finite) flag(a.status, TQ_FLAG_OVERFLOW);
        }
    }
}

template <int KB, int VB, int M>
static int launch_encode_t(const EncodeArgs& a, int num_sms, cudaStream_t s) {
    const size_t smem = (size_t)(M * kSPad + (M > 0 ? kEncWarps * kHeadDim : 0)) * sizeof(float);
    auto kern = encode_kernel<KB, VB, M>;
    if (smem > 48 * 1024) {
        static int done[64] = {};
        cudaError_t e = ensure_smem_limit(kern, (int)smem, done);
        if (e != cudaSuccess) return (int)e;
    }
    const int64_t items = a.num_tokens * a.g.hkv;
    int64_t blocks = (items + kEncWarps - 1) / kEncWarps;
    const int64_t cap = (int64_t)num_sms * (M > 0 ? 2 : 8);
    if (blocks > cap) blocks = cap;
    return (int)launch_programmatic(kern, dim3((unsigned)blocks), dim3(kEncWarps * 32), smem, s, a);
}

int launch_encode(const EncodeArgs& a, int num_sms, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int kb = a.g.kb, vb = a.g.vb, m = a.g.m;
#define TQ_ENC(KB_, VB_)                                                              \
    if (kb == KB_ && vb == VB_)                                                       \
        return m ? launch_encode_t<KB_, VB_, 128>(a, num_sms, s)                      \
                 : launch_encode_t<KB_, VB_, 0>(a, num_sms, s);
    TQ_ENC(2, 2) TQ_ENC(2, 3) TQ_ENC(2, 4)
    TQ_ENC(3, 2) TQ_ENC(3, 3) TQ_ENC(3, 4)
    TQ_ENC(4, 2) TQ_ENC(4, 3) TQ_ENC(4, 4)
#undef TQ_ENC
    return (int)cudaErrorInvalidValue;
}

}  // namespace tq
