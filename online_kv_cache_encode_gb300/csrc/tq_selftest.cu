// Self-test of the tensor-core building blocks the decode kernels use (see
// tq_tcgen05.cuh): one CTA computes D = A . B for A 128 x 256 and B 256 x 16
// (fp16, fp32 accumulate) in several ways and writes every result:
//   out[0]     A from tensor memory, B from shared memory; D read back with
//              the 32-lanes x 32-bit load (thread = row);
//   out[1]     the same D read back with the 16-lanes x 256-bit load, each value
//              stored where that load's documented fragment layout puts it;
//   out[2]     A and B both from shared memory;
//   out[3]     A written to tensor memory with the 16-lanes x 256-bit store
//              (each value placed where that store's documented fragment
//              layout puts it), B from shared memory;
//   out[4], out[5]  A from tensor memory, B in the MN-major layout (element
//              (k, n) at (n / 8) 4096 + (k / 8) 128 + (k % 8) 16 + (n % 8) 2),
//              with the descriptor's leading / stride byte offsets set to
//              (128, 4096) and to (4096, 128); either setting stays inside the
//              8 KB operand, and only the first (leading = step along K) is the
//              hardware's reading.
// A test compares each with A . B computed on the host.
#include <cuda_runtime.h>

#include "tq_decode_impl.cuh"
#include "tq_tcgen05.cuh"

namespace tq {
namespace {

constexpr int kSelfM = 128, kSelfK = 256, kSelfN = 16;
constexpr int kSelfB = kSelfN * kSelfK * 2;        // B in shared memory: 8 KB
constexpr int kSelfA = kSelfM * kSelfK * 2;        // A in shared memory: 64 KB
constexpr int kSelfSmem = kSelfB + kSelfA + 16 + kSelfB;   // + barrier + TMEM address + MN-major B
constexpr uint32_t kLbo = 128;                     // core matrices along K are adjacent
constexpr uint32_t kSbo = kSelfK / 8 * 128;        // the next 8 rows: 32 core matrices on

// byte offset of element (row, k) of a K-major operand in the core-matrix layout
__host__ __device__ constexpr uint32_t kmajor_off(int row, int k) {
    return (uint32_t)((row / 8) * kSbo + (k / 8) * kLbo + (row % 8) * 16 + (k % 8) * 2);
}

__global__ void __launch_bounds__(128, 1) tc_selftest_kernel(const uint16_t* A, const uint16_t* B, float* out,
                                                             int32_t* status) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t sB = sbase, sA = sbase + kSelfB, bar = sbase + kSelfB + kSelfA;
    uint32_t* taddr_s = reinterpret_cast<uint32_t*>(sm + kSelfB + kSelfA + 8);
    if (tid == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc<512>(smem_u32(taddr_s));
    for (int i = tid; i < kSelfN * kSelfK; i += 128) {  // B[k][n] as the N x K operand
        const int k = i / kSelfN, n = i % kSelfN;
        *reinterpret_cast<uint16_t*>(sm + kmajor_off(n, k)) = B[i];
    }
    for (int i = tid; i < kSelfM * kSelfK; i += 128) {
        const int m = i / kSelfK, k = i % kSelfK;
        *reinterpret_cast<uint16_t*>(sm + kSelfB + kmajor_off(m, k)) = A[i];
    }
    uint8_t* bmn = sm + kSelfB + kSelfA + 16;  // B again, MN-major
    for (int i = tid; i < kSelfN * kSelfK; i += 128) {
        const int k = i / kSelfN, n = i % kSelfN;
        *reinterpret_cast<uint16_t*>(bmn + (n / 8) * 4096 + (k / 8) * 128 + (k % 8) * 16 + (n % 8) * 2) = B[i];
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *taddr_s;
    const uint32_t mylanes = tbase + ((uint32_t)(warp * 32) << 16);
    // A to tensor memory: thread tid holds row tid, fp16 pairs (2c, 2c + 1) in column c
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int k = 2 * (32 * c + j);
            r[j] = (uint32_t)A[tid * kSelfK + k] | ((uint32_t)A[tid * kSelfK + k + 1] << 16);
        }
        tc::st_32x32b_x32(mylanes + 32 * c, r);
    }
    tc::wait_st();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // the same A again at columns 160.., through the 16-lane stores: thread i of
    // the warp holds rows 16 e + i/4 and 16 e + i/4 + 8 of its lane block, column
    // pairs 8k + 2 (i%4), 8k + 2 (i%4) + 1 of each 8-column block k
    constexpr uint32_t kA2 = 160;
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            const int row0 = warp * 32 + 16 * e + lane / 4;
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = row0 + 8 * (q >> 1), col = 64 * half + 8 * k + 2 * (lane % 4) + (q & 1);
                    r[4 * k + q] = (uint32_t)A[row * kSelfK + 2 * col] | ((uint32_t)A[row * kSelfK + 2 * col + 1] << 16);
                }
            tc::st_16x256b_x8(tbase + ((uint32_t)(warp * 32 + 16 * e) << 16) + kA2 + 64 * half, r);
        }
    tc::wait_st();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    constexpr uint32_t kD = 128, kD2 = 144, kD3 = 288, kD4 = 304, kD5 = 320;  // TMEM columns of the results
    if (tid == 0) {
        constexpr uint32_t idesc = tc::idesc_f16_f32(kSelfM, kSelfN);
        constexpr uint32_t idesc_mn = tc::idesc_f16_f32_bmn(kSelfM, kSelfN);
        const uint32_t sBmn = sbase + kSelfB + kSelfA + 16;
#pragma unroll 1
        for (int s = 0; s < kSelfK / 16; ++s) {
            const uint64_t bd = tc::smem_desc(sB + 256 * s, kLbo, kSbo);
            tc::mma_f16_ts(tbase + kD, tbase + 8 * s, bd, idesc, s > 0);
            tc::mma_f16_ss(tbase + kD2, tc::smem_desc(sA + 256 * s, kLbo, kSbo), bd, idesc, s > 0);
            tc::mma_f16_ts(tbase + kD3, tbase + kA2 + 8 * s, bd, idesc, s > 0);
            tc::mma_f16_ts(tbase + kD4, tbase + 8 * s, tc::smem_desc(sBmn + 256 * s, 128, 4096), idesc_mn, s > 0);
            tc::mma_f16_ts(tbase + kD5, tbase + 8 * s, tc::smem_desc(sBmn + 256 * s, 4096, 128), idesc_mn, s > 0);
        }
        tc::commit(bar);
    }
    const bool ok = mbar_wait(bar, 0);
    if (!ok && tid == 0) flag(status, TQ_FLAG_TIMEOUT);
    tc::fence_after_sync();
    if (ok) {
        uint32_t r[16];
        tc::ld_32x32b_x16(mylanes + kD, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) out[tid * 16 + j] = __uint_as_float(r[j]);
        tc::ld_32x32b_x16(mylanes + kD2, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) out[2 * kSelfM * kSelfN + tid * 16 + j] = __uint_as_float(r[j]);
        tc::ld_32x32b_x16(mylanes + kD3, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) out[3 * kSelfM * kSelfN + tid * 16 + j] = __uint_as_float(r[j]);
        tc::ld_32x32b_x16(mylanes + kD4, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) out[4 * kSelfM * kSelfN + tid * 16 + j] = __uint_as_float(r[j]);
        tc::ld_32x32b_x16(mylanes + kD5, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) out[5 * kSelfM * kSelfN + tid * 16 + j] = __uint_as_float(r[j]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t f[8];
            tc::ld_16x256b_x2(tbase + ((uint32_t)(warp * 32 + 16 * h) << 16) + kD, f);
            tc::wait_ld();
            const int row0 = warp * 32 + 16 * h + lane / 4, row1 = row0 + 8, col = 2 * (lane % 4);
            float* o = out + kSelfM * kSelfN;
            o[row0 * 16 + col] = __uint_as_float(f[0]);
            o[row0 * 16 + col + 1] = __uint_as_float(f[1]);
            o[row1 * 16 + col] = __uint_as_float(f[2]);
            o[row1 * 16 + col + 1] = __uint_as_float(f[3]);
            o[row0 * 16 + 8 + col] = __uint_as_float(f[4]);
            o[row0 * 16 + 8 + col + 1] = __uint_as_float(f[5]);
            o[row1 * 16 + 8 + col] = __uint_as_float(f[6]);
            o[row1 * 16 + 8 + col + 1] = __uint_as_float(f[7]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc<512>(tbase);
    }
}

}  // namespace
}  // namespace tq

extern "C" TQ_API tq_status tq_selftest_tcgen05(const void* A, const void* B, float* out, int32_t* dev_status,
                                                void* stream) {
    if (!A || !B || !out) {
        tq::set_error("A, B and out must be non-NULL");
        return TQ_ERR_INVALID_ARG;
    }
    static int done[64] = {};
    cudaError_t e = tq::ensure_smem_limit(tq::tc_selftest_kernel, tq::kSelfSmem, done);
    if (e == cudaSuccess) {
        tq::tc_selftest_kernel<<<1, 128, tq::kSelfSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
            static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), out, dev_status);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        tq::set_error("tcgen05 self-test launch: %s", cudaGetErrorString(e));
        return TQ_ERR_CUDA;
    }
    return TQ_OK;
}
