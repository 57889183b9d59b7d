// Encode kernel: compress new key/value vectors into the paged cache.
//
// GRP lanes per (token, KV head) item: lane s of an item's group holds
// coordinates E s .. E s + E - 1 (E = 128 / GRP) of the key and of the value.
//  - GRP = 8 for bulk encodes: four items per warp, so the per-item work (its
//    index, the norm and min/max reductions, the fp16 metadata) is shared by
//    four items per warp instruction and the rotation needs three cross-lane
//    butterfly stages instead of five.
//  - GRP = 32 when there are too few items to fill the GPU (a decode step
//    appends one token): four coordinates per lane keep an item's latency low.
//   key:   gamma = ||k|| (group sum of squares), u_rot = FWHT(s (.) k) / (sqrt(d) gamma),
//          code_j = #{ boundaries < u_rot[j] }; with QJL, r = u_rot - C[code],
//          rho = ||r||, sigma_i = [(S r)_i >= 0] with S staged in shared memory
//   value: v_rot = FWHT(s (.) v) / sqrt(d), per-token min/max (group reductions),
//          code = clamp(rint((v_rot - min) / scale), 0, 2^b - 1)
// ["TurboQuant: KV Cache Vector Quantization" -- three steps; deep dive
//  (cell-devlog) -- Step 1 (RHT), Step 3 (value codes); Bit-Axon --
//  quantization function; "OCTOPUS ..." -- methodology steps 1, 2, 8]
#pragma once
#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {

constexpr int kEncWarps = 8;
// S in shared memory: each row's 16-coordinate segments start 20 floats apart,
// so that the 8 lanes of an item read 16-byte pieces of a row from 8
// different groups of banks
constexpr int kSSeg = 20;
constexpr int kSRow = 8 * kSSeg;
__host__ __device__ constexpr int s_pos(int c) { return kSSeg * (c >> 4) + (c & 15); }

// KeyThresholds::code by binary search over the thresholds held in registers:
// 3 comparisons instead of 7 at 4 bits, 2 instead of 3 at 3 bits.  Every
// comparison is one of the linear count's and the thresholds increase, so the
// code is the same (the fused append in the decode kernel keeps the count).
template <int KB>
__device__ __forceinline__ int key_code_bsearch(const KeyThresholds<KB>& kt, float x) {
    constexpr int HALF = 1 << (KB - 1);
    if constexpr (HALF - 1 == 7 || HALF - 1 == 3) {
        const float ax = fabsf(x);
        int n;
        if constexpr (HALF - 1 == 7) {
            const bool c4 = kt.thr[3] < ax;
            const bool c2 = (c4 ? kt.thr[5] : kt.thr[1]) < ax;
            const float t1 = c4 ? (c2 ? kt.thr[6] : kt.thr[4]) : (c2 ? kt.thr[2] : kt.thr[0]);
            n = (c4 ? 4 : 0) + (c2 ? 2 : 0) + ((t1 < ax) ? 1 : 0);
        } else {
            const bool c2 = kt.thr[1] < ax;
            n = (c2 ? 2 : 0) + (((c2 ? kt.thr[2] : kt.thr[0]) < ax) ? 1 : 0);
        }
        return (x > 0.f) ? HALF + n : HALF - 1 - n;
    } else {
        return kt.code(x);
    }
}

// E consecutive elements starting at element index i (i a multiple of E).
template <int E>
__device__ __forceinline__ void load_e(const void* base, int dtype, int64_t i, float x[E]) {
    if constexpr (E == 4) {
        load4(base, dtype, i, x);
    } else if (dtype == TQ_F32) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 v = p[k];
            x[4 * k] = v.x; x[4 * k + 1] = v.y; x[4 * k + 2] = v.z; x[4 * k + 3] = v.w;
        }
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(base) + i);
        const uint4 a = p[0], b = p[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (dtype == TQ_BF16) {
                x[2 * k] = __uint_as_float(w[k] << 16);
                x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            } else {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
                x[2 * k] = f.x;
                x[2 * k + 1] = f.y;
            }
        }
    }
}

// Unnormalised natural-order Walsh-Hadamard transform of a 128-vector over a
// GRP-lane group, lane s holding coordinates E s .. E s + E - 1: butterflies of
// stride 1 .. E/2 inside the lane, E .. 64 across lanes (lower index a+b, upper a-b).
template <int GRP, int E>
__device__ __forceinline__ void fwht128_grp(float x[E], int s) {
#pragma unroll
    for (int h = 1; h < E; h <<= 1)
#pragma unroll
        for (int i = 0; i < E; ++i)
            if ((i & h) == 0) {
                const float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
#pragma unroll
    for (int m = 1; m < GRP; m <<= 1) {
        const float sg = (s & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < E; ++i) x[i] = fmaf(sg, x[i], __shfl_xor_sync(0xffffffffu, x[i], m));
    }
}

template <int GRP>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int m = 1; m < GRP; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}
template <int GRP>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int m = 1; m < GRP; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}
template <int GRP>
__device__ __forceinline__ float group_min(float v) {
#pragma unroll
    for (int m = 1; m < GRP; m <<= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// The E codes of one lane (packed LSB-first in w) into the 128-code row of its
// item; `store` guards the memory write only, every lane of the warp takes
// part in the shuffle packer of the 4-codes-per-lane layout.
template <int B, int E>
__device__ __forceinline__ void store_lane_codes(uint8_t* row, int s, const uint32_t (&w)[(E * B + 31) / 32],
                                                 bool store) {
    if constexpr (E == 16) {
        // 2B bytes at byte 2B s of the row
        if (!store) return;
        if constexpr (B == 4) {
            *reinterpret_cast<uint2*>(row + 8 * s) = make_uint2(w[0], w[1]);
        } else if constexpr (B == 8) {
            *reinterpret_cast<uint4*>(row + 16 * s) = make_uint4(w[0], w[1], w[2], w[3]);
        } else if constexpr (B == 2) {
            *reinterpret_cast<uint32_t*>(row + 4 * s) = w[0];
        } else {
            uint16_t* p = reinterpret_cast<uint16_t*>(row + 2 * B * s);
#pragma unroll
            for (int k = 0; k < B; ++k) p[k] = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
        }
    } else {
        // 4B bits per lane
        if constexpr (B == 4) {
            if (store) reinterpret_cast<uint16_t*>(row)[s] = (uint16_t)w[0];
        } else if constexpr (B == 2) {
            if (store) row[s] = (uint8_t)w[0];
        } else if constexpr (B == 8) {
            if (store) reinterpret_cast<uint32_t*>(row)[s] = w[0];
        } else {
            const uint32_t word = row_word<B>(w[0], s);
            if (store && s < 4 * B) reinterpret_cast<uint32_t*>(row)[s] = word;
        }
    }
}

template <int KB, int VB, int M, int GRP>
__global__ void __launch_bounds__(kEncWarps * 32, M > 0 ? 2 : 3) encode_kernel(const EncodeArgs a) {
    constexpr int E = kHeadDim / GRP;   // coordinates per lane
    constexpr int IPW = 32 / GRP;       // items per warp
    extern __shared__ float smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int s = lane & (GRP - 1), grp = lane / GRP;
    const Geometry& g = a.g;
    constexpr int D = kHeadDim;
    constexpr int NB = (1 << KB) - 1;
    constexpr int VMAX = (1 << VB) - 1;
    constexpr int HALF = 1 << (KB - 1);
    float* Ss = smem;                                                  // [M][kSRow]
    // key widths above 4 bits: the positive boundaries (times sqrt(d)) for the binary search
    __shared__ float bsd_s[KB > 4 ? (1 << (KB - 1)) : 1];
    // launched as a programmatic dependent: wait for the previous grid before
    // touching global memory, and let the next one start launching
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (M > 0) {
        const float4* S4 = reinterpret_cast<const float4*>(a.S);  // four coordinates of one segment at a time
        for (int i = threadIdx.x; i < M * D / 4; i += blockDim.x) {
            const int row = (4 * i) / D, c = (4 * i) % D;
            *reinterpret_cast<float4*>(Ss + row * kSRow + s_pos(c)) = __ldg(S4 + i);
        }
        __syncthreads();
    }
    if constexpr (KB > 4) {
        for (int i = threadIdx.x; i < (1 << (KB - 1)) - 1; i += blockDim.x) bsd_s[i] = a.tab->boundary_sd_pos[i];
        __syncthreads();
    }
    // signs of coordinates E s .. E s + E - 1 (bit i set: s = -1)
    const uint32_t sgn = (a.c.sign_bits[(E * s) >> 5] >> ((E * s) & 31)) & ((1u << E) - 1u);
    const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
    const int hkv = g.hkv;
    const int64_t items = a.num_tokens * hkv;
    const int64_t cap = g.num_blocks * kBlockSize;

    // Item it = t * hkv + h; the grid-stride loop keeps (t, h) incrementally.
    const int64_t stride = (int64_t)gridDim.x * kEncWarps * IPW;
    const int64_t st_t = stride / hkv;
    const int st_h = (int)(stride - st_t * hkv);
    int64_t it = ((int64_t)blockIdx.x * kEncWarps + warp) * IPW + grp;
    int64_t t = it / hkv;
    int h = (int)(it - t * hkv);
    // The loop runs while any item of the warp is live, so that the shuffles
    // always see all 32 lanes; a finished group computes on zeros and stores nothing.
    const int64_t it_warp0 = ((int64_t)blockIdx.x * kEncWarps + warp) * IPW;
    for (int64_t base = it_warp0; base < items; base += stride, it += stride) {
        const bool live = it < items;
        float k[E], v[E];
        int64_t slot = -1;
        if (live) {
            load_e<E>(a.K, a.dtype, it * D + E * s, k);
            load_e<E>(a.V, a.dtype, it * D + E * s, v);
            slot = a.slot_mapping[t];
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) k[i] = v[i] = 0.f;
        }
        const int hc = h;
        t += st_t;
        h += st_h;
        if (h >= hkv) { h -= hkv; ++t; }
        const bool bad = live && slot >= cap;
        const bool store = live && slot >= 0 && slot < cap;
        if (bad && s == 0) flag(a.status, TQ_FLAG_BAD_SLOT);

        // ---- key ----
        float ss = 0.f, z = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            ss = fmaf(k[i], k[i], ss);
            z = fmaf(k[i], 0.f, fmaf(v[i], 0.f, z));  // x * 0 is 0 for finite x, NaN for inf / NaN
        }
        ss = group_sum<GRP>(ss);
        const bool finite = (group_sum<GRP>(z) == 0.f);
        if (store && !finite && s == 0) flag(a.status, TQ_FLAG_NONFINITE);
        const float gamma = sqrtf(ss);
#pragma unroll
        for (int i = 0; i < E; ++i)
            if ((sgn >> i) & 1u) k[i] = -k[i];
        fwht128_grp<GRP, E>(k, s);
        int kc[E];
        float r[E];
        if (gamma > 0.f) {
            const KeyThresholds<KB <= 4 ? KB : 1> kt(a.c, gamma);
#pragma unroll
            for (int i = 0; i < E; ++i) {
                if constexpr (KB <= 4) kc[i] = key_code_bsearch<KB>(kt, k[i]);
                else kc[i] = key_code_search<KB>(k[i], gamma, bsd_s);
                if constexpr (M > 0) {
                    const float u = (k[i] * inv_sqrt_d) / gamma;
                    float cv = 0.f;
#pragma unroll
                    for (int b = 0; b <= NB; ++b) cv = (kc[i] == b) ? a.c.centroid[b] : cv;
                    r[i] = u - cv;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < E; ++i) {
                kc[i] = HALF - 1;
                r[i] = 0.f;
            }
        }
        // page of the slot (kBlockSize == 16: block = slot >> 4, offset = slot & 15)
        static_assert(kBlockSize == 16, "page index by shift");
        const int64_t blk = store ? (slot >> 4) : 0;
        const int off = (int)(slot & (kBlockSize - 1));
        uint8_t* page = a.pool + (blk * hkv + hc) * g.page_bytes;
        {
            uint32_t w[(E * KB + 31) / 32];
            pack_words<KB, E>(kc, w);
            store_lane_codes<KB, E>(page + g.kcode_off + off * (D * KB / 8), s, w, store);
        }

        // ---- value ----
#pragma unroll
        for (int i = 0; i < E; ++i)
            if ((sgn >> i) & 1u) v[i] = -v[i];
        fwht128_grp<GRP, E>(v, s);
        float lo_v = 3.4e38f, hi_v = -3.4e38f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            v[i] *= inv_sqrt_d;
            lo_v = fminf(lo_v, v[i]);
            hi_v = fmaxf(hi_v, v[i]);
        }
        const float mn = group_min<GRP>(lo_v), mx = group_max<GRP>(hi_v);
        const float scale = (mx - mn) / (float)VMAX;
        int vc[E];
#pragma unroll
        for (int i = 0; i < E; ++i)
            vc[i] = (scale > 0.f) ? (int)fminf(fmaxf(rintf((v[i] - mn) / scale), 0.f), (float)VMAX) : 0;
        {
            uint32_t w[(E * VB + 31) / 32];
            pack_words<VB, E>(vc, w);
            store_lane_codes<VB, E>(page + g.vcode_off + off * (D * VB / 8), s, w, store);
        }

        float rho = 0.f;
        if constexpr (M > 0) {
            float rr = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) rr = fmaf(r[i], r[i], rr);
            rho = sqrtf(group_sum<GRP>(rr));
            // S r, CH rows at a time: every lane forms the partial dot products
            // of the CH rows over its own coordinates E s .. E s + E - 1, then
            // the item's lanes sum them, each lane ending with CH / GRP rows
            // (rows (CH/GRP) s .. of the chunk) whose sign bits it sets
            // (bit i of sigma: (S r)_i >= 0); the words are OR-ed over the group.
            constexpr int CH = (GRP == 8) ? 16 : 32;
            constexpr int RPL = CH / GRP;
            uint32_t wb[M / 32];
#pragma unroll
            for (int w = 0; w < M / 32; ++w) wb[w] = 0u;
#pragma unroll
            for (int ch = 0; ch < M / CH; ++ch) {
                float pr[CH];
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const float* srow = Ss + (ch * CH + k) * kSRow + s_pos(E * s);
                    float acc = 0.f;
#pragma unroll
                    for (int v4 = 0; v4 < E / 4; ++v4) {
                        const float4 sv = *reinterpret_cast<const float4*>(srow + 4 * v4);
                        acc = fmaf(sv.x, r[4 * v4], fmaf(sv.y, r[4 * v4 + 1], fmaf(sv.z, r[4 * v4 + 2], fmaf(sv.w, r[4 * v4 + 3], acc))));
                    }
                    pr[k] = acc;
                }
#pragma unroll
                for (int m = GRP / 2, half = CH / 2; m >= 1; m >>= 1, half >>= 1) {
                    const bool up = (s & m) != 0;
#pragma unroll
                    for (int k = 0; k < half; ++k) {
                        const float keep = up ? pr[k + half] : pr[k];
                        const float give = up ? pr[k] : pr[k + half];
                        pr[k] = keep + __shfl_xor_sync(0xffffffffu, give, m);
                    }
                }
#pragma unroll
                for (int k = 0; k < RPL; ++k)
                    if (pr[k] >= 0.f) wb[(ch * CH) >> 5] |= 1u << (((ch * CH) & 31) + RPL * s + k);
            }
            uint32_t wstore = 0u;
#pragma unroll
            for (int w = 0; w < M / 32; ++w) {
#pragma unroll
                for (int m = 1; m < GRP; m <<= 1) wb[w] |= __shfl_xor_sync(0xffffffffu, wb[w], m);
                if (s == w) wstore = wb[w];
            }
            if (store && s < M / 32) {
                uint32_t* sig = reinterpret_cast<uint32_t*>(page + g.sig_off + off * (M / 8));
                sig[s] = (gamma > 0.f) ? wstore : 0xffffffffu;
            }
        }

        if (store && s == 0) {
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

}  // namespace tq

// the tensor-core encode (uses key_code_bsearch above)
#include "tq_encode_tc.cuh"

namespace tq {

// The grid is at most one wave: the CTAs that fit on every SM at once (from
// the occupancy calculator, once per kernel) loop over the items.
template <int KB, int VB, int M, int GRP>
static int launch_encode_g(const EncodeArgs& a, int64_t items, int num_sms, cudaStream_t s) {
    constexpr int IPW = 32 / GRP;
    const size_t smem = (size_t)(M * kSRow) * sizeof(float);
    auto kern = encode_kernel<KB, VB, M, GRP>;
    if (smem > 48 * 1024) {
        static int done[64] = {};
        cudaError_t e = ensure_smem_limit(kern, (int)smem, done);
        if (e != cudaSuccess) return (int)e;
    }
    static int per_sm = 0;  // same value from any thread that computes it
    if (per_sm == 0) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kEncWarps * 32, smem);
        if (e != cudaSuccess) return (int)e;
        per_sm = n > 0 ? n : 1;
    }
    const int64_t cap = (int64_t)num_sms * per_sm;
    int64_t blocks = (items + kEncWarps * IPW - 1) / (kEncWarps * IPW);
    if (blocks > cap) blocks = cap;
    return (int)launch_programmatic(kern, dim3((unsigned)blocks), dim3(kEncWarps * 32), smem, s, a);
}

template <int KB, int VB, int M>
static int launch_encode_t(const EncodeArgs& a, int num_sms, cudaStream_t s) {
    const int64_t items = a.num_tokens * a.g.hkv;
    if constexpr (M == 0) {
        // bulk 16-bit encodes rotate on the tensor cores
        if (encode_tc_eligible(a, items, num_sms)) {
            const int r = launch_encode_tc<KB, VB>(a, items, num_sms, s);
            if (r >= 0) return r;
        }
    }
    // four items per warp once there are enough to give every warp slot of
    // the GPU four; one item per warp (lower latency) below that
    if (items >= (int64_t)num_sms * (M > 0 ? 2 : 8) * kEncWarps * 4)
        return launch_encode_g<KB, VB, M, 8>(a, items, num_sms, s);
    return launch_encode_g<KB, VB, M, 32>(a, items, num_sms, s);
}

// All value widths (and the QJL sketch, for widths 2 .. 4) of one key width.
template <int KB>
int launch_encode_kb(const EncodeArgs& a, int num_sms, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int vb = a.g.vb, m = a.g.m;
    if constexpr (KB >= 2 && KB <= 4) {
        if (m) {
            if (vb == 2) return launch_encode_t<KB, 2, 128>(a, num_sms, s);
            if (vb == 3) return launch_encode_t<KB, 3, 128>(a, num_sms, s);
            if (vb == 4) return launch_encode_t<KB, 4, 128>(a, num_sms, s);
            return (int)cudaErrorInvalidValue;
        }
    }
    if (m) return (int)cudaErrorInvalidValue;
    switch (vb) {
        case 1: return launch_encode_t<KB, 1, 0>(a, num_sms, s);
        case 2: return launch_encode_t<KB, 2, 0>(a, num_sms, s);
        case 3: return launch_encode_t<KB, 3, 0>(a, num_sms, s);
        case 4: return launch_encode_t<KB, 4, 0>(a, num_sms, s);
        case 5: return launch_encode_t<KB, 5, 0>(a, num_sms, s);
        case 6: return launch_encode_t<KB, 6, 0>(a, num_sms, s);
        case 7: return launch_encode_t<KB, 7, 0>(a, num_sms, s);
        case 8: return launch_encode_t<KB, 8, 0>(a, num_sms, s);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace tq
