// Device helpers shared by the encode and decode kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "tq_internal.h"

namespace tq {

// Raise a kernel's dynamic shared-memory limit once per device and size; the
// attribute call costs host time that would otherwise be paid on every launch.
// Concurrent first calls may both set it, which is harmless.
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kern, int bytes, int (&done)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = bytes;
    return e;
}

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel in the stream drains, and must execute griddepcontrol.wait
// before it touches global memory.
template <typename Kernel, typename... Args>
inline cudaError_t launch_programmatic(Kernel kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                       const Args&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Two fp32 lanes in one 64-bit register and the packed add / multiply / fma of
// sm_100 and later: one instruction for two coordinates.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ void flag(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

// Four consecutive elements starting at element index i of a row.
__device__ __forceinline__ void load4(const void* base, int dtype, int64_t i, float x[4]) {
    if (dtype == TQ_F32) {
        float4 v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(base) + i);
        if (dtype == TQ_BF16) {
            x[0] = __uint_as_float(v.x << 16);
            x[1] = __uint_as_float(v.x & 0xFFFF0000u);
            x[2] = __uint_as_float(v.y << 16);
            x[3] = __uint_as_float(v.y & 0xFFFF0000u);
        } else {
            __half2 a = *reinterpret_cast<__half2*>(&v.x), b = *reinterpret_cast<__half2*>(&v.y);
            float2 fa = __half22float2(a), fb = __half22float2(b);
            x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
        }
    }
}

// Key codes without a division.  With x a coordinate of H (s . k) (not yet
// divided by sqrt(d)) and gamma = ||k|| > 0, the code #{t_b < x / (sqrt(d) gamma)}
// is decided by comparing |x| with thr_b = (sqrt(d) t_b) gamma over the positive
// boundaries: the codebook is symmetric (t_b = -t_{n-2-b}, middle boundary 0),
// so the code is HALF + #{thr_b < |x|} for x > 0 and HALF - 1 - #{thr_b < |x|}
// otherwise.  This differs from dividing first only within a few fp32 roundings
// of a boundary, and from the plain count only at a tie.
template <int KB>
struct KeyThresholds {
    static constexpr int HALF = 1 << (KB - 1);
    float thr[HALF - 1 > 0 ? HALF - 1 : 1];
    __device__ __forceinline__ KeyThresholds(const Consts& c, float gamma) {
#pragma unroll
        for (int b = 0; b < HALF - 1; ++b) thr[b] = c.boundary_sd[HALF + b] * gamma;
    }
    __device__ __forceinline__ int code(float x) const {
        const float ax = fabsf(x);
        int n = 0;
#pragma unroll
        for (int b = 0; b < HALF - 1; ++b) n += (thr[b] < ax) ? 1 : 0;
        return (x > 0.f) ? HALF + n : HALF - 1 - n;
    }
};

// Key widths above 4 bits: the same decision by binary search over the
// positive boundaries (monotone, so it finds the same count as the linear
// comparison); bsd_pos[b] = sqrt(d) t_{HALF + b}.
template <int KB>
__device__ __forceinline__ int key_code_search(float x, float gamma, const float* bsd_pos) {
    constexpr int HALF = 1 << (KB - 1);
    const float ax = fabsf(x);
    int n = 0;
#pragma unroll
    for (int step = HALF / 2; step >= 1; step >>= 1)
        if (bsd_pos[n + step - 1] * gamma < ax) n += step;
    return (x > 0.f) ? HALF + n : HALF - 1 - n;
}

// E B-bit codes packed LSB-first into words (code i at bits B i ..).
template <int B, int E>
__device__ __forceinline__ void pack_words(const int c[E], uint32_t (&w)[(E * B + 31) / 32]) {
#pragma unroll
    for (int k = 0; k < (E * B + 31) / 32; ++k) w[k] = 0u;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int pos = B * i, wi = pos >> 5, sh = pos & 31;
        w[wi] |= (uint32_t)c[i] << sh;
        if (sh + B > 32) w[wi + 1] |= (uint32_t)c[i] >> (32 - sh);
    }
}

// Word `lane` of a row of 128 B-bit codes whose lane l holds the codes of
// coordinates 4l .. 4l+3 packed LSB-first in p (4B bits), gathered from the
// lanes that hold its bits.  Every lane of the warp must call it; the row has
// 4B words, so lanes from 4B on get nothing useful.
template <int B>
__device__ __forceinline__ uint32_t row_word(uint32_t p, int lane) {
    constexpr int LB = 4 * B;
    constexpr int K = 32 / LB + 2;  // lanes that can hold bits of one word
    uint32_t word = 0;
    const int src0 = (lane * 32) / LB;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int src = src0 + k;
        const uint32_t pv = __shfl_sync(0xffffffffu, p, src < 32 ? src : 31);
        const int shift = src * LB - lane * 32;
        if (src < 32) {
            if (shift >= 0 && shift < 32) word |= pv << shift;
            else if (shift < 0 && shift > -LB) word |= pv >> (-shift);
        }
    }
    return word;
}

// The 4 sign bits of coordinates 4*lane .. 4*lane+3 (bit i set: s = -1).
__device__ __forceinline__ uint32_t lane_signs(const Consts& c, int lane) {
    return (c.sign_bits[lane >> 3] >> (4 * (lane & 7))) & 0xFu;
}

__device__ __forceinline__ void apply_signs(float x[4], uint32_t sm) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if ((sm >> i) & 1u) x[i] = -x[i];
}

// Unnormalised natural-order Walsh-Hadamard transform of a 128-vector spread
// over a warp, lane holding coordinates 4*lane .. 4*lane+3: butterflies of
// stride 1 and 2 inside the lane, strides 4..64 across lanes (the lower index
// takes a+b, the upper a-b).
__device__ __forceinline__ void fwht128(float x[4], int lane) {
    float a = x[0] + x[1], b = x[0] - x[1], c = x[2] + x[3], d = x[2] - x[3];
    x[0] = a + c; x[2] = a - c; x[1] = b + d; x[3] = b - d;
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int m = 1 << k;
        const float sg = (lane & m) ? -1.f : 1.f;  // upper: y - x, lower: x + y (one exact-sign fma)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float y = __shfl_xor_sync(0xffffffffu, x[i], m);
            x[i] = fmaf(sg, x[i], y);
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

__device__ __forceinline__ uint16_t f16_bits(float x) {
    __half h = __float2half_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace tq
