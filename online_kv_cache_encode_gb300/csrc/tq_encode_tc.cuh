// Bulk encode with the rotation on the tcgen05 tensor cores (16-bit inputs,
// no QJL sketch).
//
// Rotating a tile of 128 (token, KV head) vectors is one dense contraction:
// U = X H^T, X the tile [128 rows x 128 coordinates] and
// H[n][k] = (-1)^popcount(n & k) s_k, the natural-order Walsh-Hadamard matrix
// times the random signs.  The inputs (bf16 or fp16) and H (entries +-1) are
// exact tensor-core operands; the products are exact and accumulate in fp32 in
// tensor memory, so row m of U is FWHT(s (.) x_m), unnormalised, as the CUDA-core
// encode computes it, up to the order of the fp32 additions.  H stays in shared
// memory for the whole kernel.  The rest of the encode reads one row per
// thread from tensor memory and needs no cross-lane traffic:
//   key:   gamma = ||U_k|| / sqrt(d) = ||k||; code_j = #{boundaries < u_j} with
//          u = U_k / (sqrt(d) gamma), decided as U_k against sqrt(d) t_b gamma
//          (widths up to 4) or as |U_k| / gamma against sqrt(d) t_b on a grid
//          (wider keys);
//   value: v_rot = U_v / sqrt(d); per-token min / max;
//          code = clamp(rint((v_rot - min) / scale), 0, 2^b - 1).
// ["TurboQuant: KV Cache Vector Quantization" -- three steps; deep dive
//  (cell-devlog) -- Step 1 (RHT), Step 3 (value codes); Bit-Axon --
//  quantization function; "OCTOPUS ..." -- methodology steps 1, 2]
//
// CTA: four independent warpgroups, one per tile in flight, persistent over
// the CTA's tiles (taken in turn from a shared-memory counter).  A warpgroup
// has one 32 KB input buffer in shared memory (one operand of a tile in the
// K-major core-matrix layout with the 128-byte swizzle, filled by two TMA tile
// copies of 64 coordinates x 128 rows) and 128 tensor-memory columns; each of
// its threads takes one row of the tile, so every per-row reduction stays in
// one thread.  Per tile it rotates the keys, starts the copy of the values
// into the buffer the key MMAs have just read and codes the keys while that
// copy runs, then rotates the values, starts the copy of its next tile's keys
// and codes the values: the buffer is refilled during every half of the
// epilogue, so four copies per SM are in flight most of the time.  One CTA per
// SM.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tq_decode_impl.cuh"  // mbarrier, grid-dependency and shared-address helpers
#include "tq_device.cuh"
#include "tq_tcgen05.cuh"

namespace tq {

constexpr int kEtRows = 128;                   // rows (token, KV head) per tile
constexpr int kEtGroups = 4;                   // independent warpgroups (tiles in flight)
constexpr int kEtThreads = kEtGroups * 128;
// H: K-major core matrices without swizzle, along K adjacent, 8-row groups
// 2 KB apart.  The inputs: the TMA boxes' 128-byte-swizzled K-major layout
// (row r of a box at 128 r, its 16-byte pieces permuted by r % 8; 8-row groups
// 1 KB apart; the box of coordinates 64 .. 127 16 KB after the first).
constexpr uint32_t kEtLbo = 128, kEtSbo = 2048;
constexpr uint32_t kEtXSbo = 1024, kEtXBox = 16384;
constexpr int kEtOp = kEtRows * kHeadDim * 2;  // one 128 x 128 16-bit operand: 32 KB
constexpr int kEtH = 0;                        // H [n][k]
constexpr int kEtX = kEtOp;                    // warpgroup w's buffer at kEtX + w kEtOp
// key widths above 4 bits: the decision grid over z = |u| / gamma in [0, sqrt(d)],
// 64 cells per unit (cell c: z 64 in [c - 1/2, c + 1/2]), indexed up to z = 16
constexpr int kEtCells = 1025;
constexpr int kEtGrid = kEtX + kEtGroups * kEtOp;        // [cell] (-tau 2^40 or -inf, count below)
// Code rows of 5 to 7 bits go out through shared memory: each thread stages
// its row's packed words and writes the row with one bulk copy (16 B
// multiples: a row is 16 B per code bit).  Stored directly, their chunks of
// 20, 24 or 28 bytes take 4- or 8-byte stores, each a fraction of a 32-byte
// sector from every thread; the bulk copies cost 16-41 % less time per
// encode.  Other widths store directly (16-byte stores at 4 and 8 bits): for
// them the many small bulk copies, which share the copy engine with the tile
// loads, were slower.  The staging stride is the row rounded to an odd
// multiple of 16 B, so that the threads' writes at one offset spread over the
// banks.
__host__ __device__ constexpr bool et_bulk(int B) { return B >= 5 && B <= 7; }
__host__ __device__ constexpr int et_row_stride(int B) { return et_bulk(B) ? 16 * B + ((B & 1) ? 0 : 16) : 0; }
// the rest of the layout; the grid takes space only for key widths above 4 bits
template <int KB, int VB>
struct EtLayout {
    static constexpr int rs = et_row_stride(KB) > et_row_stride(VB) ? et_row_stride(KB) : et_row_stride(VB);
    static constexpr int rows = kEtGrid + (KB > 4 ? 8 * kEtCells + 8 : 0);   // [warpgroup][row] staged code rows
    static constexpr int bars = rows + kEtGroups * kEtRows * rs;            // per warpgroup: MMAs done, copy landed
    static constexpr int next = bars + 16 * kEtGroups;   // tile counter, next tile per warpgroup
    static constexpr int taddr = next + 4 * (1 + kEtGroups);
    static constexpr int smem = taddr + 16 + 1024;       // + room to align the base to 1 KB (swizzle atoms)
    static_assert(rows % 16 == 0 && rs % 16 == 0, "bulk copies want 16-byte aligned rows");
    static_assert(smem <= 232448, "over the shared memory of one CTA");
};

// One bulk copy of `bytes` (a multiple of 16) from shared memory to global
// memory, both 16-byte aligned, in this thread's bulk group; the commit, the
// wait until the thread's copies have read their source, and the wait until
// they are complete.
__device__ __forceinline__ void et_bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void et_bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void et_bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void et_bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }


// B words to shared memory at a (4-byte aligned; 8-byte when B is even,
// 16-byte when B % 4 == 0)
template <int B>
__device__ __forceinline__ void et_sts_words(uint32_t a, const uint32_t (&w)[B]) {
    if constexpr (B % 4 == 0) {
#pragma unroll
        for (int j = 0; j < B / 4; ++j)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16 * j), "r"(w[4 * j]), "r"(w[4 * j + 1]),
                         "r"(w[4 * j + 2]), "r"(w[4 * j + 3])
                         : "memory");
    } else if constexpr (B % 2 == 0) {
#pragma unroll
        for (int j = 0; j < B / 2; ++j)
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a + 8 * j), "r"(w[2 * j]), "r"(w[2 * j + 1]) : "memory");
    } else {
#pragma unroll
        for (int j = 0; j < B; ++j) asm volatile("st.shared.u32 [%0], %1;" ::"r"(a + 4 * j), "r"(w[j]) : "memory");
    }
}

// Box (x, y) of a 2-D tensor map into shared memory, completing on `bar`.
__device__ __forceinline__ void et_tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// OR of `v` over the 128 threads of a warpgroup (named barrier `id`)
__device__ __forceinline__ bool et_any128(bool v, int id) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

// Three-input minimum and maximum of sm_100 and later: one instruction where
// two-input ones take two.
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// B words at p (4-byte aligned; 8-byte when B is even, 16-byte when B % 4 == 0)
template <int B>
__device__ __forceinline__ void et_store_words(uint8_t* p, const uint32_t (&w)[B]) {
    if constexpr (B % 4 == 0) {
#pragma unroll
        for (int j = 0; j < B / 4; ++j)
            reinterpret_cast<uint4*>(p)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    } else if constexpr (B % 2 == 0) {
#pragma unroll
        for (int j = 0; j < B / 2; ++j) reinterpret_cast<uint2*>(p)[j] = make_uint2(w[2 * j], w[2 * j + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < B; ++j) reinterpret_cast<uint32_t*>(p)[j] = w[j];
    }
}

// 32 bytes to global memory at p (32-byte aligned): one store instruction.
__device__ __forceinline__ void et_stg256(uint8_t* p, const uint32_t (&a)[4], const uint32_t (&b)[4]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a[0]), "r"(a[1]), "r"(a[2]),
                 "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3])
                 : "memory");
}
// The codes of one 32-code chunk c of a row.  An 8-bit chunk is one 32-byte
// sector: one store when the pool is 32-byte aligned (rows and chunks then are:
// pages, row offsets and chunk offsets are multiples of 32 B), 3.8 % faster
// per encode at 8/8 than two 16-byte stores.  Other widths stored chunk by
// chunk take 16, 8 or 4 bytes at a time.
template <int B>
__device__ __forceinline__ void et_store_chunk(uint8_t* row, int c, bool a32, const uint32_t (&w)[B]) {
    if constexpr (B == 8) {
        if (a32) {
            const uint32_t lo[4] = {w[0], w[1], w[2], w[3]}, hi[4] = {w[4], w[5], w[6], w[7]};
            et_stg256(row + 32 * c, lo, hi);
            return;
        }
    }
    et_store_words<B>(row + c * 4 * B, w);
}

// Rows of 1 to 4 bits are stored a group of chunks at a time: 1 bit, the whole
// 16-byte row; 2 bits, two chunks (16 bytes); 3 bits, two chunks (24 bytes, as
// three 8-byte stores); 4 bits, two chunks (one 32-byte store when the pool is
// 32-byte aligned).  Rows are 16 B per code bit on 16-byte aligned pages, so
// each group starts 16-byte (1, 2 bits), 8-byte (3 bits) or 32-byte (4 bits,
// aligned pool) aligned.  At 3/3 this took 43.8 -> 39.2 us per encode against
// one 4- or 8-byte store per word.
__host__ __device__ constexpr int et_group(int B) { return B == 1 ? 4 : 2; }
template <int B>
__device__ __forceinline__ void et_store_group(uint8_t* p, const uint32_t (&w)[et_group(B) * B], bool a32) {
    if constexpr (B == 4) {
        const uint32_t lo[4] = {w[0], w[1], w[2], w[3]}, hi[4] = {w[4], w[5], w[6], w[7]};
        if (a32) {
            et_stg256(p, lo, hi);
        } else {
            *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(p + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        }
    } else if constexpr (B == 3) {
        reinterpret_cast<uint2*>(p)[0] = make_uint2(w[0], w[1]);
        reinterpret_cast<uint2*>(p)[1] = make_uint2(w[2], w[3]);
        reinterpret_cast<uint2*>(p)[2] = make_uint2(w[4], w[5]);
    } else {
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}


// Codes are formed in the fp32 add pipe rather than with compares, selects and
// conversions: for |q| < 2^22, q + 1.5 2^23 rounds q to the nearest integer
// (ties to even) and holds it in its low mantissa bits above the constant
// 0x4B400000.  Such "biased" fields are packed by integer multiply-adds; the
// constant's share of every word is removed once (the fields do not overlap, so
// the sums are the ORs of the codes).
constexpr float kEtMagic = 12582912.f;  // 1.5 * 2^23
constexpr uint32_t kEtMagicBits = 0x4B400000u;

// The constant's share of word k when 32 B-bit biased fields are packed
// LSB-first into B words (field i at bit B i; a field that crosses a word
// boundary continues at bit 0 of the next word).
__host__ __device__ constexpr uint32_t et_pack_bias(int B, int k) {
    uint32_t sum = 0;
    for (int i = 0; i < 32; ++i) {
        const int pos = B * i, wi = pos >> 5, sh = pos & 31;
        if (wi == k) sum += kEtMagicBits << sh;
        if (sh + B > 32 && wi + 1 == k) sum += kEtMagicBits >> (32 - sh);
    }
    return 0u - sum;
}

template <int B>
__device__ __forceinline__ void et_pack_biased(const uint32_t (&f)[32], uint32_t (&w)[B]) {
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = et_pack_bias(B, k);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int pos = B * i, wi = pos >> 5, sh = pos & 31;
        w[wi] += f[i] * (1u << sh);
        if (sh + B > 32) w[wi + 1] += f[i] >> (32 - sh);
    }
}

// Key codes (widths up to 4 bits) of 32 rotated coordinates x against the
// positive thresholds scaled by F (T[b] = F sqrt(d) t_{HALF+b} gamma), with F a
// power of two such that T[0] lies in [2^24, 2^25).  Every threshold, and every
// float near one, is then an even integer, and so is |x| F once it reaches
// 2^24; the saturated difference sat(|x| F - t) is therefore exactly
// [|x| F > t] for any such t.  n = #{b : |x| > thr_b} comes from a binary
// search whose steps are these differences, two coordinates per packed
// instruction where the arithmetic allows it.  The next threshold is picked
// arithmetically, t = T[lo] + s (T[hi] - T[lo]) for a step s in {0, 1}: for
// s = 0 it is T[lo] exactly, and for s = 1 it is T[hi] up to the rounding of the
// difference (an ulp), which can move a decision only for a coordinate within
// 2^-23 (relative) of a boundary.  The sign: sg = sat(x 2^127) is [x > 0] for
// every x of magnitude 2^-127 or more, and the code HALF + n (x > 0) or
// HALF - 1 - n (otherwise) is formed as c + sg + (2 sg - 1) n with the
// rounding constant in c, so the code is an integer even for a smaller x
// (fractional sg; n is 0 there).
template <int KB>
struct EtKeySearch {
    static constexpr int HALF = 1 << (KB - 1);
    uint64_t F2;            // the scale, twice
    float t1;               // first step: T[HALF / 2 - 1]
    uint64_t lo2, d2;       // second step: T[lo] and T[hi] - T[lo] (HALF >= 4)
    uint64_t l3, d3a, d3b, d3ab;  // third step (HALF == 8): T0 + sa (T2 - T0) + sb (T4 - T0) + sa sb (T6 - T4 - T2 + T0)
    __device__ __forceinline__ EtKeySearch(const float* T, float F) {
        F2 = f2_pack(F, F);
        t1 = 0.f;
        lo2 = d2 = l3 = d3a = d3b = d3ab = 0ull;
        if constexpr (HALF == 8) {
            t1 = T[3];
            lo2 = f2_pack(T[1], T[1]);
            d2 = f2_pack(T[5] - T[1], T[5] - T[1]);
            const float a = T[2] - T[0], b = T[4] - T[0], ab = (T[6] - T[4]) - a;
            l3 = f2_pack(T[0], T[0]);
            d3a = f2_pack(a, a);
            d3b = f2_pack(b, b);
            d3ab = f2_pack(ab, ab);
        } else if constexpr (HALF == 4) {
            t1 = T[1];
            lo2 = f2_pack(T[0], T[0]);
            d2 = f2_pack(T[2] - T[0], T[2] - T[0]);
        } else if constexpr (HALF == 2) {
            t1 = T[0];
        }
    }
};

template <int KB>
__device__ __forceinline__ void et_key_codes(const float (&x)[32], const EtKeySearch<KB>& ks, uint32_t (&f)[32]) {
    constexpr int HALF = 1 << (KB - 1);
    auto c2 = [](float v) { return f2_pack(v, v); };
    const uint64_t C = c2(kEtMagic + (float)(HALF - 1));
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float X0, X1;
        f2_unpack(f2_mul(f2_pack(x[j], x[j + 1]), ks.F2), X0, X1);
        const uint64_t SG = f2_pack(__saturatef(x[j] * 0x1p127f), __saturatef(x[j + 1] * 0x1p127f));
        uint64_t N = 0ull;
        if constexpr (HALF >= 2) {
            const uint64_t S1 = f2_pack(__saturatef(fabsf(X0) - ks.t1), __saturatef(fabsf(X1) - ks.t1));
            if constexpr (HALF == 2) {
                N = S1;
            } else {
                float a0, a1;
                f2_unpack(f2_fma(S1, ks.d2, ks.lo2), a0, a1);
                const uint64_t S2 = f2_pack(__saturatef(fabsf(X0) - a0), __saturatef(fabsf(X1) - a1));
                if constexpr (HALF == 4) {
                    N = f2_fma(S1, c2(2.f), S2);
                } else {
                    // S1 picks the upper half (T4 .. T6), S2 the upper quarter of it
                    float b0, b1;
                    f2_unpack(f2_fma(S2, f2_fma(S1, ks.d3ab, ks.d3a), f2_fma(S1, ks.d3b, ks.l3)), b0, b1);
                    const uint64_t S3 = f2_pack(__saturatef(fabsf(X0) - b0), __saturatef(fabsf(X1) - b1));
                    N = f2_fma(S1, c2(4.f), f2_fma(S2, c2(2.f), S3));
                }
            }
        }
        // c + sg + (2 sg - 1) n
        const uint64_t SGN = f2_fma(SG, c2(2.f), c2(-1.f));
        float k0, k1;
        f2_unpack(f2_fma(SGN, N, f2_add(SG, C)), k0, k1);
        f[j] = __float_as_uint(k0);
        f[j + 1] = __float_as_uint(k1);
    }
}

// Key codes (widths above 4 bits) of 32 rotated coordinates x through the
// decision grid.  With z = |x| / gamma, taken as y = sat(z / 16) (a NaN or inf
// lands on an end of the grid), the cell c = rint(64 z) spans z in
// [(c - 1/2) / 64, (c + 1/2) / 64]; no two positive boundaries tau_b =
// sqrt(d) t_b lie that close, so the count n = #{b : z > tau_b} is the cell's
// count below it plus [z > tau] for the one boundary tau that may lie in the
// cell, decided as sat(2^40 z - 2^40 tau) (exact: z - tau is at least an ulp of
// tau, and 2^40 of that is at least 1).  The cell's entry is (-2^40 tau, or
// -inf for none, and the count below) at grid + 8 c; its address comes from
// the biased field of rint(64 z) by one integer multiply-add.  The sign and
// the code are formed as in et_key_codes.
template <int KB>
__device__ __forceinline__ void et_key_codes_grid(const float (&x)[32], float ig16, uint32_t grid,
                                                  uint32_t (&f)[32]) {
    constexpr int HALF = 1 << (KB - 1);
    auto c2 = [](float v) { return f2_pack(v, v); };
    const uint64_t C = c2(kEtMagic + (float)(HALF - 1)), MG = c2(kEtMagic), W = c2(1024.f);
    const uint32_t adj = grid - (kEtMagicBits << 3);  // wraps: 8 bits(rint) + adj = grid + 8 c
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float y0 = __saturatef(fabsf(x[j]) * ig16), y1 = __saturatef(fabsf(x[j + 1]) * ig16);
        float r0, r1;
        f2_unpack(f2_fma(f2_pack(y0, y1), W, MG), r0, r1);
        float nt0, n00, nt1, n01;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(nt0), "=f"(n00) : "r"(__float_as_uint(r0) * 8u + adj));
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(nt1), "=f"(n01) : "r"(__float_as_uint(r1) * 8u + adj));
        const uint64_t S = f2_pack(__saturatef(fmaf(y0, 0x1p44f, nt0)), __saturatef(fmaf(y1, 0x1p44f, nt1)));
        const uint64_t N = f2_add(f2_pack(n00, n01), S);
        const uint64_t SG = f2_pack(__saturatef(x[j] * 0x1p127f), __saturatef(x[j + 1] * 0x1p127f));
        float k0, k1;
        f2_unpack(f2_fma(f2_fma(SG, c2(2.f), c2(-1.f)), N, f2_add(SG, C)), k0, k1);
        f[j] = __float_as_uint(k0);
        f[j + 1] = __float_as_uint(k1);
    }
}

// Value codes of 32 coordinates x (rotated, unnormalised) of one row, biased:
// rint((x / sqrt(d) - mn) / scale), the quotient formed as a product with
// rs = 1 / scale.  That product is within VMAX 2^-22 of the exact quotient,
// so it rounds to the same integer unless it lies within 2^(VB - 21) of a
// half-integer; if any of the 32 does, the row's chunk is coded again with the
// division (rint of the correctly rounded quotient, as everywhere else).
template <int VB>
__device__ __forceinline__ void et_value_codes(const float (&x)[32], float mn, float scale, float rs, uint32_t (&f)[32]) {
    constexpr float VMAX = (float)((1 << VB) - 1);
    constexpr float kTie = 0.5f - (float)(1 << VB) * 4.76837158203125e-7f;  // 0.5 - 2^(VB - 21)
    const float inv_sqrt_d = 0.08838834764831845f;
    if (!(scale > 0.f)) {
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = kEtMagicBits;
        return;
    }
    float emax[2] = {0.f, 0.f};  // the largest |q - rint(q)|, two chains
    const uint64_t C2 = f2_pack(inv_sqrt_d, inv_sqrt_d), NMN2 = f2_pack(-mn, -mn), RS2 = f2_pack(rs, rs),
                   MG2 = f2_pack(kEtMagic, kEtMagic);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        // q = (x / sqrt(d) - mn) / scale as fma then product, two coordinates at a time
        const uint64_t q = f2_mul(f2_fma(f2_pack(x[j], x[j + 1]), C2, NMN2), RS2);
        const uint64_t t = f2_add(q, MG2);
        float e0, e1, t0, t1;
        f2_unpack(f2_sub(q, f2_sub(t, MG2)), e0, e1);
        f2_unpack(t, t0, t1);
        emax[(j >> 1) & 1] = fmax3(emax[(j >> 1) & 1], fabsf(e0), fabsf(e1));
        f[j] = __float_as_uint(t0);
        f[j + 1] = __float_as_uint(t1);
    }
    if (fmaxf(emax[0], emax[1]) > kTie) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            f[j] = __float_as_uint(fminf(fmaxf(rintf(fmaf(x[j], inv_sqrt_d, -mn) / scale), 0.f), VMAX) + kEtMagic);
    }
}

// This thread's row of tensor memory, 32 columns at ta.
__device__ __forceinline__ void et_load32(uint32_t ta, float (&x)[32]) {
    uint32_t r[32];
    tc::ld_32x32b_x32(ta, r);
    tc::wait_ld();
    tc::reg_fence(r);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
}

template <int KB, int VB>
__global__ void __launch_bounds__(kEtThreads, 1)
    encode_tc_kernel(const EncodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     int64_t items, int num_tiles) {
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    constexpr int D = kHeadDim;
    constexpr int HALF = 1 << (KB - 1);
    constexpr int VMAX = (1 << VB) - 1;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int wg = tid >> 7, tw = tid & 127;
    const Geometry& g = a.g;
    // the swizzled layout repeats every 1 KB and is anchored at 1 KB boundaries
    uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    using LY = EtLayout<KB, VB>;
    int* next_s = reinterpret_cast<int*>(sm + LY::next);  // [0]: tile counter; [1 + w]: warpgroup w's next tile

    // The set-up up to the H matrix reads only kernel parameters and shared
    // memory, so it runs before the wait for the previous grid (programmatic
    // dependent launch) and overlaps that grid's last CTAs.
    if (tid == 0) {
        for (int b = 0; b < 2 * kEtGroups; ++b) mbar_init(sbase + LY::bars + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        next_s[0] = kEtGroups;
    }
    if (warp == 0) tc::tmem_alloc<512>(sbase + LY::taddr);
    {
        // H[n][k] = (-1)^(popcount(n & k) + [s_k = -1]) in the input type, K-major:
        // element (n, k) at (n / 8) 2048 + (k / 8) 128 + (n % 8) 16 + (k % 8) 2
        const uint32_t one = (a.dtype == TQ_BF16) ? 0x3F80u : 0x3C00u;
        for (int c = tid; c < D * (D / 8); c += kEtThreads) {
            const int n = c >> 4, k8 = c & 15;
            uint32_t w[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t hv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 8 * k8 + 2 * p + e;
                    const uint32_t neg = ((uint32_t)__popc(n & k) + ((a.c.sign_bits[k >> 5] >> (k & 31)) & 1u)) & 1u;
                    hv[e] = one | (neg << 15);
                }
                w[p] = hv[0] | (hv[1] << 16);
            }
            *reinterpret_cast<uint4*>(sm + kEtH + (n >> 3) * kEtSbo + k8 * kEtLbo + (n & 7) * 16) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    grid_dependency_wait();  // the previous grid's writes (inputs, pool) are visible
    int grid_bad = 0;
    if constexpr (KB > 4) {
        // the decision grid: per cell the count of positive boundaries below it
        // and the one boundary inside it, if any
        const float* bp = a.tab->boundary_sd_pos;  // HALF - 1 increasing values
        float2* grid = reinterpret_cast<float2*>(sm + kEtGrid);
        for (int c = tid; c < kEtCells; c += kEtThreads) {
            const float lo = ((float)c - 0.5f) * (1.f / 64.f), hi = ((float)c + 0.5f) * (1.f / 64.f);
            int n0 = 0;  // #{b : bp[b] < lo}
#pragma unroll
            for (int step = HALF / 2; step >= 1; step >>= 1)
                if (n0 + step <= HALF - 1 && bp[n0 + step - 1] < lo) n0 += step;
            float nt = -INFINITY;
            if (n0 < HALF - 1 && bp[n0] <= hi) {
                nt = -bp[n0] * 0x1p40f;
                if (n0 + 1 < HALF - 1 && bp[n0 + 1] <= hi) grid_bad = 1;
            }
            grid[c] = make_float2(nt, (float)n0);
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // H: generic writes -> tensor-core reads
    tc::fence_before_sync();
    // a grid cell with two boundaries (none for the codebooks of d = 128) sends
    // the wide-key decisions to the search over the boundaries
    grid_bad = __syncthreads_or(grid_bad);
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + LY::taddr);
    // only now may a dependent grid start: one of its CTAs on this SM must not
    // take the tensor-memory columns this CTA waits for
    grid_launch_dependents();

    const uint32_t xb = sbase + kEtX + wg * kEtOp;                                  // this warpgroup's buffer
    const uint32_t tcol = tmem + 128u * (uint32_t)wg;                                // its columns
    const uint32_t trow = tcol + ((uint32_t)((warp & 3) * 32) << 16);                // this warp's lanes
    const uint32_t done = sbase + LY::bars + 16 * wg, full = done + 8;
    const uint32_t rowbuf = sbase + LY::rows + (uint32_t)((wg * kEtRows + tw) * LY::rs);  // this thread's staged row
    // 8-bit code rows start on 32-byte boundaries (see et_store_chunk)
    const bool a32 = ((reinterpret_cast<uintptr_t>(a.pool) | (uintptr_t)g.page_bytes | (uintptr_t)g.vcode_off) & 31u) == 0;
    const int bar_id = 1 + wg;  // named barrier of the warpgroup
    // one operand of `tile` into the buffer (thread 0 of the warpgroup): box j
    // holds coordinates 64 j .. 64 j + 63 of the 128 rows, rows past the last
    // item zero-filled
    auto load = [&](const CUtensorMap* map, int tile) {
        mbar_arrive_tx(full, (uint32_t)kEtOp);
        et_tma_2d(xb, map, 0, tile * kEtRows, full);
        et_tma_2d(xb + kEtXBox, map, 64, tile * kEtRows, full);
    };
    // 8 MMAs: U = X H^T of the operand in the buffer into the columns
    const uint32_t idesc = (a.dtype == TQ_BF16) ? tc::idesc_bf16_f32(kEtRows, D) : tc::idesc_f16_f32(kEtRows, D);
    auto rotate = [&]() {
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
            tc::mma_f16_ss(tcol, tc::smem_desc_sw128(xb + (s >> 2) * kEtXBox + 32 * (s & 3), kEtXSbo),
                           tc::smem_desc(sbase + kEtH + 256 * s, kEtLbo, kEtSbo), idesc, s > 0 ? 1u : 0u);
        tc::commit(done);
    };
    const float inv_sqrt_d = 0.08838834764831845f;  // 1/sqrt(128)
    const int hkv = g.hkv;
    const int64_t cap = g.num_blocks * kBlockSize;
    // the CTA's tiles are blockIdx.x + k gridDim.x; warpgroup w starts with k = w
    const int nk = (num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    int k = wg;
    bool bad = false;
    uint32_t ph = 0;  // phase of both barriers: each completes twice per tile
    if (tw == 0 && k < nk) load(&tmk, (int)blockIdx.x + k * (int)gridDim.x);
    while (k < nk) {
        const int tile = (int)blockIdx.x + k * (int)gridDim.x;
        // ---- keys (the barrier at the end of the previous tile ordered the
        // threads' reads of the columns before these MMAs) ----
        if (tw == 0) {
            // a copy wait that gives up issues nothing: the MMA wait below then gives up too
            if (mbar_wait(full, ph)) {
                tc::fence_after_sync();
                rotate();
            }
        }
        // this row's (token, KV head) item and its slot, loaded while the MMAs run
        const int64_t it = (int64_t)tile * kEtRows + tw;
        const bool live = it < items;
        const uint32_t itu = (uint32_t)(live ? it : 0);  // items < 2^31
        const uint32_t t = itu / (uint32_t)hkv;
        const int hc = (int)(itu - t * (uint32_t)hkv);
        const int64_t sl = live ? __ldg(a.slot_mapping + t) : -1;
        // a wait that gives up ends the warpgroup's loop for all its threads
        // together (its named barrier needs all 128)
        bad = et_any128(!mbar_wait(done, ph), bar_id);
        if (bad) break;
        tc::fence_after_sync();
        if (tw == 0) load(&tmv, tile);  // the key MMAs have read the buffer

        if (live && sl >= cap) flag(a.status, TQ_FLAG_BAD_SLOT);
        const bool store = live && sl >= 0 && sl < cap;
        static_assert(kBlockSize == 16, "page index by shift");
        const int64_t blk = store ? (sl >> 4) : 0;
        const int off = (int)(sl & (kBlockSize - 1));
        uint8_t* page = a.pool + (blk * hkv + hc) * g.page_bytes;
        float x[32];

        // gamma = ||U_k|| / sqrt(d) (||U_k||^2 = d ||k||^2, d = 128: an exact scaling)
        uint64_t ss2[2] = {0ull, 0ull};  // four partial sums of squares, two per register
        bool finite = true;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            et_load32(trow + 32 * c, x);
            // a non-finite input coordinate makes every rotated coordinate inf
            // or NaN (H has no zero entry), so one coordinate tells
            finite = finite && isfinite(x[0]);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const uint64_t p = f2_pack(x[j], x[j + 1]);
                ss2[(j >> 1) & 1] = f2_fma(p, p, ss2[(j >> 1) & 1]);
            }
        }
        float s4[4];
        f2_unpack(ss2[0], s4[0], s4[1]);
        f2_unpack(ss2[1], s4[2], s4[3]);
        const float gamma = sqrtf(((s4[0] + s4[1]) + (s4[2] + s4[3])) * (1.f / 128.f));
        {
            uint8_t* krow = page + g.kcode_off + off * (D * KB / 8);
            const KeyThresholds<KB <= 4 ? KB : 1> kt(a.c, gamma);
            // T = F thr: F = 2^(24 - e) with 2^e <= thr_0 < 2^(e + 1), so that
            // T[0] lies in [2^24, 2^25) and the search's steps are exact; |x| F
            // stays below 2^25 / t_{HALF} (|x| <= sqrt(d) gamma)
            constexpr int NT = (KB <= 4 && HALF > 1) ? HALF - 1 : 1;
            float T[NT] = {};
            float F = 1.f;
            bool fast = KB <= 4 && gamma > 0.f;
            if constexpr (KB <= 4 && HALF > 1) {
                const int e0 = (int)((__float_as_uint(kt.thr[0]) >> 23) & 0xFFu) - 127;
                fast = fast && e0 > -100 && e0 < 100;
                F = __uint_as_float((uint32_t)(127 + 24 - e0) << 23);
#pragma unroll
                for (int b = 0; b < NT; ++b) T[b] = kt.thr[b] * F;
            }
            const EtKeySearch<(KB <= 4) ? KB : 1> ks(T, F);
            // wide keys: z / 16 = |x| / (16 gamma)
            const float ig16 = (KB > 4 && gamma > 0.f) ? 0.0625f / gamma : 0.f;
            if constexpr (KB > 4) fast = !grid_bad && gamma > 1e-30f && ig16 < 3.0e38f;
            // the staged row's last bulk copy (the previous tile's values) has read it
            if constexpr (et_bulk(KB)) et_bulk_wait_read();
            // the packed key words of chunk c
            auto key_chunk = [&](int c, uint32_t (&wk)[KB]) {
                et_load32(trow + 32 * c, x);
                uint32_t fk[32];
                if (fast) {
                    if constexpr (KB <= 4) et_key_codes<KB>(x, ks, fk);
                    else et_key_codes_grid<KB>(x, ig16, sbase + kEtGrid, fk);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        int code = HALF - 1;  // a zero key (gamma = 0)
                        if (gamma > 0.f) {
                            if constexpr (KB <= 4) code = key_code_bsearch<KB>(kt, x[j]);
                            else code = key_code_search<KB>(x[j], gamma, a.tab->boundary_sd_pos);
                        }
                        fk[j] = kEtMagicBits + (uint32_t)code;
                    }
                }
                et_pack_biased<KB>(fk, wk);
            };
            if constexpr (KB <= 4) {
                // narrow rows: a group of chunks per step, stored in wider pieces
                constexpr int NG = et_group(KB);
#pragma unroll 1
                for (int c = 0; c < 4; c += NG) {
                    uint32_t wg_[NG * KB];
#pragma unroll
                    for (int h = 0; h < NG; ++h) {
                        uint32_t wk[KB];
                        key_chunk(c + h, wk);
#pragma unroll
                        for (int i = 0; i < KB; ++i) wg_[h * KB + i] = wk[i];
                    }
                    if (store) et_store_group<KB>(krow + 4 * KB * c, wg_, a32);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t wk[KB];
                    key_chunk(c, wk);
                    if constexpr (et_bulk(KB)) et_sts_words<KB>(rowbuf + c * 4 * KB, wk);
                    else if (store) et_store_chunk<KB>(krow, c, a32, wk);
                }
            }
            if constexpr (et_bulk(KB)) {
                if (store) {
                    // the row's generic shared-memory writes -> the bulk copy's reads
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    et_bulk_s2g(krow, rowbuf, 16 * KB);
                    et_bulk_commit();
                }
            }
        }

        // ---- values: the threads are done reading the key columns ----
        tc::fence_before_sync();
        asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
        if (tw == 0) {
            if (mbar_wait(full, ph ^ 1u)) {
                tc::fence_after_sync();
                rotate();
            }
        }
        bad = et_any128(!mbar_wait(done, ph ^ 1u), bar_id);
        if (bad) break;
        tc::fence_after_sync();
        if (tw == 0) {
            // the value MMAs have read the buffer: the keys of this warpgroup's next tile
            const int kn = atomicAdd(next_s, 1);
            next_s[1 + wg] = kn;
            if (kn < nk) load(&tmk, (int)blockIdx.x + kn * (int)gridDim.x);
        }
        // v_rot = U_v / sqrt(d): the scaling is monotone, so min and max commute with it
        float lo2[2] = {3.4e38f, 3.4e38f}, hi2[2] = {-3.4e38f, -3.4e38f};
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            et_load32(trow + 32 * c, x);
            finite = finite && isfinite(x[0]);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                lo2[(j >> 1) & 1] = fmin3(lo2[(j >> 1) & 1], x[j], x[j + 1]);
                hi2[(j >> 1) & 1] = fmax3(hi2[(j >> 1) & 1], x[j], x[j + 1]);
            }
        }
        const float mn = fminf(lo2[0], lo2[1]) * inv_sqrt_d;
        const float mx = fmaxf(hi2[0], hi2[1]) * inv_sqrt_d;
        const float scale = (mx - mn) / (float)VMAX;
        const float rs = 1.f / scale;
        {
            uint8_t* vrow = page + g.vcode_off + off * (D * VB / 8);
            // the staged row's key copy has read it
            if constexpr (et_bulk(VB)) et_bulk_wait_read();
            // the packed value words of chunk c
            auto value_chunk = [&](int c, uint32_t (&wv)[VB]) {
                et_load32(trow + 32 * c, x);
                uint32_t fv[32];
                et_value_codes<VB>(x, mn, scale, rs, fv);
                et_pack_biased<VB>(fv, wv);
            };
            if constexpr (VB <= 4) {
                constexpr int NG = et_group(VB);
#pragma unroll 1
                for (int c = 0; c < 4; c += NG) {
                    uint32_t wg_[NG * VB];
#pragma unroll
                    for (int h = 0; h < NG; ++h) {
                        uint32_t wv[VB];
                        value_chunk(c + h, wv);
#pragma unroll
                        for (int i = 0; i < VB; ++i) wg_[h * VB + i] = wv[i];
                    }
                    if (store) et_store_group<VB>(vrow + 4 * VB * c, wg_, a32);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t wv[VB];
                    value_chunk(c, wv);
                    if constexpr (et_bulk(VB)) et_sts_words<VB>(rowbuf + c * 4 * VB, wv);
                    else if (store) et_store_chunk<VB>(vrow, c, a32, wv);
                }
            }
            if constexpr (et_bulk(VB)) {
                if (store) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    et_bulk_s2g(vrow, rowbuf, 16 * VB);
                    et_bulk_commit();
                }
            }
        }
        if (store) {
            if (!finite) flag(a.status, TQ_FLAG_NONFINITE);
            const uint16_t hg = f16_bits(gamma), hs = f16_bits(scale), hz = f16_bits(mn);
            reinterpret_cast<uint16_t*>(page + g.gam_off)[off] = hg;
            reinterpret_cast<uint16_t*>(page + g.scl_off)[off] = hs;
            reinterpret_cast<uint16_t*>(page + g.zer_off)[off] = hz;
            const bool ovf = ((hg & 0x7FFF) == 0x7C00) || ((hs & 0x7FFF) == 0x7C00) || ((hz & 0x7FFF) == 0x7C00);
            if (ovf && finite) flag(a.status, TQ_FLAG_OVERFLOW);
        }
        // the next tile, published by thread 0 before the barrier below; every
        // thread reads it after that barrier (at the top of the keys)
        tc::fence_before_sync();
        asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
        k = next_s[1 + wg];
    }
    if (bad && tw == 0) {
        flag(a.status, TQ_FLAG_TIMEOUT);
        // a copy or MMAs this warpgroup started may still be in flight: wait (a
        // short bound each) for the current phase of both barriers, whichever
        // parity it has, before the CTA releases its memory
        for (uint32_t par = 0; par < 2; ++par) {
            mbar_wait_for(full, par, 100000000ll);
            mbar_wait_for(done, par, 100000000ll);
        }
    }
    // this thread's row copies are complete (their shared-memory source is
    // released with the CTA)
    if constexpr (et_bulk(KB) || et_bulk(VB)) et_bulk_wait_all();
    // every MMA of the CTA has completed (each warpgroup waited for its last)
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc<512>(tmem);
    }
}

// Whether the tensor-core encode takes this call: 16-bit inputs, no QJL, and
// at least one 128-row tile per SM.
inline bool encode_tc_eligible(const EncodeArgs& a, int64_t items, int num_sms) {
    return a.g.m == 0 && a.g.d == kHeadDim && (a.dtype == TQ_BF16 || a.dtype == TQ_F16) &&
           items >= (int64_t)num_sms * kEtRows && items < ((int64_t)1 << 31);
}

// The tensor map of one input: 16-bit elements, [rows][128] row-major, boxes of
// 64 coordinates x 128 rows landing in the 128-byte swizzle, out-of-range rows
// read as zero.  The encoder entry
// point comes from the driver once per process (any thread that gets there
// first stores the same pointer).
inline bool et_tensor_map(CUtensorMap* map, const void* base, int64_t rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kEtRows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches the tensor-core encode; returns -1 (nothing launched) when the
// tensor maps cannot be made, so that the caller takes the CUDA-core kernel.
template <int KB, int VB>
int launch_encode_tc(const EncodeArgs& a, int64_t items, int num_sms, cudaStream_t s) {
    CUtensorMap tmk, tmv;
    if (!et_tensor_map(&tmk, a.K, items) || !et_tensor_map(&tmv, a.V, items)) return -1;
    auto kern = encode_tc_kernel<KB, VB>;
    static int done[64] = {};
    cudaError_t e = ensure_smem_limit(kern, EtLayout<KB, VB>::smem, done);
    if (e != cudaSuccess) return (int)e;
    const int num_tiles = (int)((items + kEtRows - 1) / kEtRows);
    const int grid = num_tiles < num_sms ? num_tiles : num_sms;
    return (int)launch_programmatic(kern, dim3((unsigned)grid), dim3(kEtThreads), (size_t)EtLayout<KB, VB>::smem, s, a, tmk, tmv,
                                    items, num_tiles);
}

}  // namespace tq
