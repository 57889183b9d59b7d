// Decode dispatch: the kernels for each key width are compiled in their own
// translation unit (tq_inst.cu, built once per width).
#include <cuda_runtime.h>

#include "tq_internal.h"

namespace tq {

int decode_smem_bytes(const Geometry& g) {
    switch (g.kb) {
        case 1: return decode_smem_kb<1>(g);
        case 2: return decode_smem_kb<2>(g);
        case 3: return decode_smem_kb<3>(g);
        case 4: return decode_smem_kb<4>(g);
        case 5: return decode_smem_kb<5>(g);
        case 6: return decode_smem_kb<6>(g);
        case 7: return decode_smem_kb<7>(g);
        case 8: return decode_smem_kb<8>(g);
        default: return -1;
    }
}

// lens[i] = first + i + 1: the causal lengths of a prefill chunk's positions
__global__ void fill_positions_kernel(int32_t* lens, int n, int first) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) lens[i] = first + i + 1;
}

int launch_fill_positions(int32_t* lens, int n, int first, void* stream) {
    if (n <= 0) return 0;
    fill_positions_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(lens, n, first);
    return (int)cudaGetLastError();
}

int launch_decode(const DecodeArgs& a, void* stream) {
    switch (a.g.kb) {
        case 1: return launch_decode_kb<1>(a, stream);
        case 2: return launch_decode_kb<2>(a, stream);
        case 3: return launch_decode_kb<3>(a, stream);
        case 4: return launch_decode_kb<4>(a, stream);
        case 5: return launch_decode_kb<5>(a, stream);
        case 6: return launch_decode_kb<6>(a, stream);
        case 7: return launch_decode_kb<7>(a, stream);
        case 8: return launch_decode_kb<8>(a, stream);
        default: return (int)cudaErrorNotSupported;
    }
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
// runtime, with that device current.  Outside stream capture the lookup (a
// host-side query) is made on every call, so a context that was reset and
// re-created since the last call gets its own address; while `stream` is
// capturing, the address found by the last uncaptured call on this device is
// used, and there must have been one.
tq_status noalloc_workspace(cudaStream_t stream, void** out) {
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
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) {
        tq::set_error("cudaStreamIsCapturing: %s", cudaGetErrorString(e));
        return TQ_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (cap != cudaStreamCaptureStatusNone) {
        if (!g_noalloc_ptr[dev]) {
            tq::set_error("the stream is capturing and this device's fixed decode workspace has not been looked up "
                          "yet: make one call outside capture first");
            return TQ_ERR_INVALID_ARG;
        }
        *out = g_noalloc_ptr[dev];
        return TQ_OK;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess || !p) {
        tq::set_error("cudaGetSymbolAddress of the fixed decode workspace: %s", cudaGetErrorString(e));
        return TQ_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
    *out = p;
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
    tq_status st = noalloc_workspace(reinterpret_cast<cudaStream_t>(stream), &ws);
    if (st != TQ_OK) return st;
    // The main codec's split counters sit at the end of its workspace and must
    // start at zero; the array keeps whatever the previous call left (another
    // shape, another cache), so clear them.  OCTOPUS caches have no counters:
    // their splits are merged by a second kernel.
    if (!cache->octopus) {
        const size_t counters = (size_t)batch * cache->g.hkv * sizeof(unsigned);
        const size_t counters_region = (counters + 255) / 256 * 256;
        cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(ws) + (need - counters_region), 0, counters,
                                        reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) {
            tq::set_error("clearing the fixed workspace counters: %s", cudaGetErrorString(e));
            return TQ_ERR_CUDA;
        }
    }
    return tq_decode_attention(cache, q, dtype, batch, num_q_heads, block_table, max_blocks_per_seq, lens, sm_scale,
                               out, ws, need, dev_status, stream);
}
