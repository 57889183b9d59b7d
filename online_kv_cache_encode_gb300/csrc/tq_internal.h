// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>

#include "tq.h"

namespace tq {

constexpr int kHeadDim = 128;   // the one head dimension the kernels are built for
constexpr int kBlockSize = 16;  // tokens per page
constexpr int kMaxCodebook = 16;   // levels held in the by-value constants (widths up to 4 bits)
constexpr int kMaxLevels = 256;    // levels of the widest codes (8 bits)

// Byte layout of one page (one block of kBlockSize slots of one KV head).
struct Geometry {
    int d, kb, vb, m, bs, hkv;
    int64_t num_blocks;
    int64_t page_bytes;
    int kcode_off, vcode_off, gam_off, scl_off, zer_off, rho_off, sig_off;
};

Geometry make_geometry(int d, int kb, int vb, int m, int bs, int hkv, int64_t num_blocks);

// Method constants the kernels take by value.
struct Consts {
    float boundary[kMaxCodebook];  // key decision boundaries (2^kb - 1 used)
    float boundary_sd[kMaxCodebook];  // sqrt(d) * boundary, rounded once from double
    float centroid[kMaxCodebook];  // key centroids (fp32), used by the QJL residual
    // Decode splits each centroid as C[c] = alpha * (c - (2^kb - 1)/2) + rem[c]:
    // the linear part goes through the tensor cores on the exact integer code,
    // rem[c] (binary16 bits) is looked up.
    float alpha;
    uint16_t rem_f16[kMaxCodebook];
    // 4-bit keys use a finer two-level split instead: C[c] = delta * N[c] +
    // rem2[c] with N[c] an integer of magnitude <= 2047 (exact in binary16)
    // and |rem2[c]| <= delta / 2, both looked up per code pair.
    float delta;
    uint16_t cint_f16[kMaxCodebook];   // N[c] in binary16
    uint16_t crem_f16[kMaxCodebook];   // rem2[c] in binary16
    uint16_t cremd_f16[kMaxCodebook];  // rem2[c] / delta in binary16 (|.| <= 1/2), for the prefill
    uint32_t sign_bits[kHeadDim / 32];  // bit j set when s_j = -1
};

// Tables for key codes of any width, in device memory written once when the
// cache is created (the by-value constants only hold widths up to 4 bits).
struct CodeTables {
    float boundary_sd_pos[kMaxLevels / 2];  // sqrt(d) t_{HALF + b}, b = 0 .. HALF - 2 (HALF = 2^(kb-1))
    uint16_t rem_f16[kMaxLevels];           // rem[c] = C[c] - alpha (c - mid) in binary16
};

struct EncodeArgs {
    Geometry g;
    Consts c;
    const CodeTables* tab;
    uint8_t* pool;
    const void* K;
    const void* V;
    int dtype;
    int64_t num_tokens;
    const int64_t* slot_mapping;
    int32_t* status;
    const float* S;  // m x d fp32, device (QJL only)
};

struct DecodeArgs {
    Geometry g;
    Consts c;
    const CodeTables* tab;
    const uint8_t* pool;
    const void* q;
    int dtype;
    int batch, hq, group;
    const int32_t* block_table;
    int max_blocks;
    int64_t bt_stride;    // elements between sequences' block-table rows (0: all share row 0)
    const int32_t* lens;
    float sm_scale_log2;  // sm_scale * log2(e)
    float* out;
    float* partials;      // [batch, hkv, splits, group, 4 + d]
    unsigned* counters;   // [batch, hkv]
    int pages_per_split;
    int num_splits;
    int32_t* status;
    const float* S;
    // append (optional): the new token of every sequence, written at position
    // lens[b] - 1 before it is attended to; null when nothing is appended
    const void* knew;     // [batch, hkv, d]
    const void* vnew;
    int kv_dtype;
    // ring of `window` slots per sequence (0: no ring): the appended token goes
    // to slot (lens[b] - 1) mod window, attention runs over min(lens[b], window) slots
    int window;
    // test hook (0: off): warp 0 of every odd split waits this many SM cycles on
    // a barrier nothing arrives on, so that the timeout path runs
    long long stall_cycles;
};

// Chunked prefill on the tensor cores (4-bit keys, no QJL, values of 1..4 bits).
struct PrefillArgs {
    Geometry g;
    Consts c;
    const uint8_t* pool;
    const void* q;        // [C, hq, d]
    int dtype;
    int C, hq, group;
    const int32_t* block_row;
    int max_blocks;
    int first;            // position of the chunk's first query
    float sm_scale_log2;
    float* out;           // [C, hq, d] fp32
    float* partials;      // [hkv, nrb, splits, 128 rows, 4 + d]
    int nrb, splits, tiles_per_split;
    int32_t* status;
    long long stall_cycles;  // test hook, as in DecodeArgs
};
bool prefill_tc_supported(const Geometry& g);
size_t prefill_tc_partials_bytes(const Geometry& g, int C, int hq, int splits);
int prefill_tc_rows_per_block();
int prefill_tc_tile_tokens();
int launch_prefill_tc(const PrefillArgs& a, void* stream);

// ---------------------------------------------------------------------------
// OCTOPUS triplet key codec (second codec of a cache; values keep min-max codes)
// ---------------------------------------------------------------------------
constexpr int kOctTri = (kHeadDim + 2) / 3;   // triplets per key (the last one padded)
constexpr int kOctMaxDir = 32;                // direction levels per axis at b = 4

// Codebooks and the direction table, in device memory written once when the
// cache is created.  dir[a * n + b] is the unit direction of level pair (a, b)
// (n = 2^(b+1) levels per axis), w unused.
struct OctTables {
    float cxi[kOctMaxDir], bxi[kOctMaxDir];   // levels and boundaries of xi and eta
    float crho[8], brho[8];                   // levels and boundaries of the triplet norm
    float dir[kOctMaxDir * kOctMaxDir][4];
};

struct OctArgs {
    Geometry g;           // kb = b (the codec's bits), vb; kcode_off = 0
    int key_row;          // bytes of one key row (4-byte multiple)
    const OctTables* tab;
    uint32_t sign_bits[kHeadDim / 32];
    uint8_t* pool;
    int32_t* status;
    // encode
    const void* K;
    const void* V;
    int dtype;
    int64_t num_tokens;
    const int64_t* slot_mapping;
    // decode
    const void* q;
    int batch, hq, group;
    const int32_t* block_table;
    int max_blocks;
    int64_t bt_stride;    // elements between sequences' block-table rows (0: all share row 0)
    const int32_t* lens;
    float sm_scale_log2;
    float* out;
    float* partials;      // [batch, hkv, splits, group, 4 + d]
    int pages_per_split, num_splits;
    long long stall_cycles;  // test hook, as in DecodeArgs
};
constexpr int kOctWarps = 8;

int launch_oct_encode(const OctArgs& a, int num_sms, void* stream);
int launch_oct_decode(const OctArgs& a, void* stream);

// Launchers (return a cudaError_t as int).  The per-key-width ones are
// explicitly instantiated, one key width per translation unit.
int launch_encode(const EncodeArgs& a, int num_sms, void* stream);
int launch_decode(const DecodeArgs& a, void* stream);
int decode_smem_bytes(const Geometry& g);
int launch_fill_positions(int32_t* lens, int n, int first, void* stream);
template <int KB>
int launch_encode_kb(const EncodeArgs& a, int num_sms, void* stream);
template <int KB>
int launch_decode_kb(const DecodeArgs& a, void* stream);
template <int KB>
int decode_smem_kb(const Geometry& g);

void set_error(const char* fmt, ...);
long long test_stall_cycles();  // the wait-timeout test hook's current setting (0: off)

}  // namespace tq

struct tq_codebook {
    int d, bits, passes;
    double centroid[256];
    double boundary[255];
};

struct tq_cache {
    void* pool;
    tq::Geometry g;
    tq::Consts c;
    uint64_t seed;
    int8_t signs[tq::kHeadDim];
    double* S_host;   // m x d
    float* S_dev;     // m x d, library-owned device memory
    tq::CodeTables* tab_dev;  // library-owned device memory
    int octopus;              // 1: OCTOPUS triplet keys (bits in g.kb)
    int oct_key_row;
    tq::OctTables* oct_dev;   // library-owned device memory (OCTOPUS)
    tq::OctTables oct_host;
    int device;
    int num_sms;
};
