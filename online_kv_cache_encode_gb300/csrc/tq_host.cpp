// Host side of the library: argument checking, the Lloyd-Max codebook, the
// seeded sign vector and Gaussian matrix, cache descriptors and the calls
// that launch the kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "tq_internal.h"

namespace tq {

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

static tq_status fail(tq_status s, const char* what) {
    set_error("%s", what);
    return s;
}

static tq_status cuda_fail(cudaError_t e, const char* what) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return TQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Counter-based SplitMix64 stream: output i of stream (seed, tag) is the
// SplitMix64 finaliser (Steele, Lea, Flood 2014) applied to
// key + (i + 1) * 0x9E3779B97F4A7C15 with key = seed ^ tag * 0xD1B54A32D192ED03.
// ---------------------------------------------------------------------------
static inline uint64_t splitmix_out(uint64_t seed, uint64_t tag, uint64_t i) {
    uint64_t z = (seed ^ (tag * 0xD1B54A32D192ED03ull)) + (i + 1) * 0x9E3779B97F4A7C15ull;
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// ---------------------------------------------------------------------------
// binary16 rounding of a double (round to nearest, ties to even), built from
// the double's bit pattern.
// ---------------------------------------------------------------------------
static uint16_t half_bits_from_double(double x) {
    uint64_t u;
    std::memcpy(&u, &x, 8);
    const uint16_t sign = (uint16_t)((u >> 48) & 0x8000);
    const int ex = (int)((u >> 52) & 0x7FF);
    uint64_t mant = u & ((1ull << 52) - 1);
    if (ex == 0x7FF) return sign | (mant ? 0x7E00 : 0x7C00);
    if (ex == 0) return sign;  // double subnormals are far below binary16's range
    const int e = ex - 1023;   // value = 1.mant * 2^e
    uint64_t sig = mant | (1ull << 52);
    int shift;                 // bits of sig to drop
    int hex;                   // binary16 exponent field
    if (e >= -14) {
        shift = 52 - 10;
        hex = e + 15;
    } else {
        shift = 52 - 10 + (-14 - e);
        hex = 0;
        if (shift > 63) return sign;
    }
    uint64_t kept = sig >> shift;
    uint64_t rem = sig & ((1ull << shift) - 1);
    uint64_t halfway = 1ull << (shift - 1);
    if (rem > halfway || (rem == halfway && (kept & 1))) ++kept;
    if (hex == 0) return sign | (uint16_t)kept;  // subnormal (may carry into the smallest normal)
    if (kept >= (1ull << 11)) {                  // mantissa overflow
        kept >>= 1;
        ++hex;
    }
    if (hex >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(hex << 10) | (uint16_t)(kept & 0x3FF);
}

// ---------------------------------------------------------------------------
// Lloyd-Max codebook for the coordinate marginal of a uniform point on
// S^{d-1}, f(x) ~ (1 - x^2)^((d-3)/2).  For even d the exponent is n/2 with
// n = d - 3 odd, and J_n(x) = int_0^x (1 - t^2)^(n/2) dt has the exact
// recurrence
//     J_{-1}(x) = asin(x),   J_n(x) = ( x (1 - x^2)^(n/2) + n J_{n-2}(x) ) / (n + 1),
// (integrate d/dx [x (1-x^2)^(n/2)] = (n+1)(1-x^2)^(n/2) - n (1-x^2)^(n/2-1)).
// A cell's mass is proportional to J(b) - J(a) and its first moment to
// ((1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)) / (d-1); the normalising constant
// cancels in the centroid.
// ---------------------------------------------------------------------------
static double sphere_J(int d, double x) {
    if (x >= 1.0 || x <= -1.0) {
        double j = (x > 0 ? 1.0 : -1.0) * (M_PI / 2.0);
        for (int n = 1; n <= d - 3; n += 2) j = (double)n * j / (double)(n + 1);
        return j;
    }
    const double w = 1.0 - x * x;
    double j = std::asin(x);
    double pw = std::sqrt(w);  // w^(n/2) for n = 1
    for (int n = 1; n <= d - 3; n += 2) {
        j = (x * pw + (double)n * j) / (double)(n + 1);
        pw *= w;
    }
    return j;
}

static double sphere_moment_term(int d, double x) {
    if (x >= 1.0 || x <= -1.0) return 0.0;
    return std::pow(1.0 - x * x, (d - 1) / 2.0) / (double)(d - 1);
}

static int lloyd_max(int d, int bits, double* c, double* t) {
    const int n = 1 << bits;
    for (int i = 0; i < n; ++i) c[i] = (2.0 * i + 1.0 - n) / n * 4.0 / std::sqrt((double)d);
    double J[257], M[257];
    int pass = 0;
    while (pass < 10000) {
        for (int i = 0; i + 1 < n; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
        J[0] = sphere_J(d, -1.0);
        M[0] = 0.0;
        for (int i = 0; i + 1 < n; ++i) {
            J[i + 1] = sphere_J(d, t[i]);
            M[i + 1] = sphere_moment_term(d, t[i]);
        }
        J[n] = sphere_J(d, 1.0);
        M[n] = 0.0;
        double delta = 0.0;
        for (int i = 0; i < n; ++i) {
            double mass = J[i + 1] - J[i];
            double cn = mass > 0 ? (M[i] - M[i + 1]) / mass : c[i];
            delta = std::fmax(delta, std::fabs(cn - c[i]));
            c[i] = cn;
        }
        ++pass;
        if (delta < 1e-14) break;
    }
    for (int i = 0; i + 1 < n; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
    return pass;
}

// ---------------------------------------------------------------------------
// geometry
// ---------------------------------------------------------------------------
Geometry make_geometry(int d, int kb, int vb, int m, int bs, int hkv, int64_t num_blocks) {
    Geometry g{};
    g.d = d; g.kb = kb; g.vb = vb; g.m = m; g.bs = bs; g.hkv = hkv;
    g.num_blocks = num_blocks;
    int off = 0;
    g.kcode_off = off; off += bs * d * kb / 8;
    g.vcode_off = off; off += bs * d * vb / 8;
    g.gam_off = off; off += 2 * bs;
    g.scl_off = off; off += 2 * bs;
    g.zer_off = off; off += 2 * bs;
    if (m > 0) {
        g.rho_off = off; off += 2 * bs;
        g.sig_off = off; off += bs * m / 8;
    } else {
        g.rho_off = g.sig_off = -1;
    }
    g.page_bytes = (off + 15) / 16 * 16;
    return g;
}

}  // namespace tq

using namespace tq;

// ===========================================================================
// C ABI
// ===========================================================================

extern "C" {

TQ_API const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported configuration";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

TQ_API const char* tq_last_error(void) { return g_last_error; }

TQ_API tq_status tq_codebook_init(int d, int bits, tq_codebook** out) {
    if (!out) return fail(TQ_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (d < 4 || d > 1024 || (d % 2) != 0) return fail(TQ_ERR_INVALID_ARG, "d must be even, 4..1024");
    if (bits < 1 || bits > 8) return fail(TQ_ERR_INVALID_ARG, "bits must be 1..8");
    tq_codebook* cb = new (std::nothrow) tq_codebook();
    if (!cb) return fail(TQ_ERR_INVALID_ARG, "out of host memory");
    cb->d = d;
    cb->bits = bits;
    cb->passes = lloyd_max(d, bits, cb->centroid, cb->boundary);
    *out = cb;
    return TQ_OK;
}

TQ_API tq_status tq_codebook_get(const tq_codebook* cb, double* centroids, double* boundaries,
                                 int* passes) {
    if (!cb) return fail(TQ_ERR_INVALID_ARG, "codebook is NULL");
    const int n = 1 << cb->bits;
    if (centroids) std::memcpy(centroids, cb->centroid, sizeof(double) * n);
    if (boundaries) std::memcpy(boundaries, cb->boundary, sizeof(double) * (n - 1));
    if (passes) *passes = cb->passes;
    return TQ_OK;
}

TQ_API void tq_codebook_free(tq_codebook* cb) { delete cb; }

TQ_API int64_t tq_page_bytes(int d, int key_bits, int value_bits, int qjl_m, int block_size) {
    if (d <= 0 || d % 8 || key_bits < 1 || key_bits > 8 || value_bits < 1 || value_bits > 8 ||
        qjl_m < 0 || qjl_m % 8 || block_size <= 0)
        return -1;
    return make_geometry(d, key_bits, value_bits, qjl_m, block_size, 1, 1).page_bytes;
}

static void derive_signs(uint64_t seed, int d, int8_t* s) {
    for (int j = 0; j < d; ++j) s[j] = (splitmix_out(seed, 0, (uint64_t)j) >> 63) ? -1 : 1;
}

static void derive_gaussian(uint64_t seed, int m, int d, double* S) {
    const double two53 = 9007199254740992.0;
    for (int64_t k = 0; k < (int64_t)m * d; ++k) {
        double u1 = ((double)(splitmix_out(seed, 1, (uint64_t)(2 * k)) >> 11) + 1.0) / two53;
        double u2 = (double)(splitmix_out(seed, 1, (uint64_t)(2 * k + 1)) >> 11) / two53;
        S[k] = std::sqrt(-2.0 * std::log(u1)) * std::cos(2.0 * M_PI * u2);
    }
}

TQ_API tq_status tq_method_constants(int d, int m, uint64_t seed, int8_t* signs, double* S) {
    if (d < 1 || d > 4096 || m < 0 || m > 4096) return fail(TQ_ERR_INVALID_ARG, "d or m out of range");
    if (signs) derive_signs(seed, d, signs);
    if (m > 0 && S) derive_gaussian(seed, m, d, S);
    return TQ_OK;
}

TQ_API tq_status tq_cache_create(void* pool, int64_t num_blocks, int block_size, int num_kv_heads,
                                 int d, int key_bits, int value_bits, int qjl_m, uint64_t seed,
                                 tq_cache** out) {
    if (!out) return fail(TQ_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!pool) return fail(TQ_ERR_INVALID_ARG, "pool is NULL");
    if ((reinterpret_cast<uintptr_t>(pool) & 15) != 0) return fail(TQ_ERR_INVALID_ARG, "pool must be 16-byte aligned");
    if (num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0 || d <= 0)
        return fail(TQ_ERR_INVALID_ARG, "sizes must be positive");
    if (tq_page_bytes(d, key_bits, value_bits, qjl_m, block_size) < 0)
        return fail(TQ_ERR_INVALID_ARG, "invalid d / bits / qjl_m combination");
    if (d != kHeadDim) return fail(TQ_ERR_UNSUPPORTED, "head dim must be 128");
    if (block_size != kBlockSize) return fail(TQ_ERR_UNSUPPORTED, "block_size must be 16");
    if (key_bits < 1 || key_bits > 8 || value_bits < 1 || value_bits > 8)
        return fail(TQ_ERR_UNSUPPORTED, "key_bits and value_bits must be 1 .. 8");
    if (qjl_m != 0 && qjl_m != 128) return fail(TQ_ERR_UNSUPPORTED, "qjl_m must be 0 or 128");
    if (qjl_m != 0 && (key_bits < 2 || key_bits > 4 || value_bits < 2 || value_bits > 4))
        return fail(TQ_ERR_UNSUPPORTED, "the QJL sketch is built for 2-, 3- and 4-bit keys and values");

    tq_cache* c = new (std::nothrow) tq_cache();
    if (!c) return fail(TQ_ERR_INVALID_ARG, "out of host memory");
    c->pool = pool;
    c->seed = seed;
    c->g = make_geometry(d, key_bits, value_bits, qjl_m, block_size, num_kv_heads, num_blocks);

    tq_codebook* cb = nullptr;
    tq_status st = tq_codebook_init(d, key_bits, &cb);
    if (st != TQ_OK) {
        delete c;
        return st;
    }
    const int n = 1 << key_bits;
    const double mid = (n - 1) / 2.0;
    double num = 0.0, den = 0.0;
    for (int i = 0; i < n; ++i) {
        num += (i - mid) * cb->centroid[i];
        den += (i - mid) * (i - mid);
    }
    const double alpha = num / den;  // least-squares slope of the centroids in the code
    std::memset(&c->c, 0, sizeof(c->c));
    c->c.alpha = (float)alpha;
    CodeTables tab;
    std::memset(&tab, 0, sizeof(tab));
    for (int i = 0; i < n; ++i) {
        // the device multiplies the code by (float)alpha; the remainder is taken
        // against exactly that product
        const uint16_t rem = half_bits_from_double(cb->centroid[i] - (double)c->c.alpha * (i - mid));
        const float bsd = (i + 1 < n) ? (float)(cb->boundary[i] * std::sqrt((double)d)) : 0.f;
        tab.rem_f16[i] = rem;
        if (i >= n / 2 && i + 1 < n) tab.boundary_sd_pos[i - n / 2] = bsd;
        if (n <= kMaxCodebook) {
            c->c.centroid[i] = (float)cb->centroid[i];
            c->c.rem_f16[i] = rem;
            if (i + 1 < n) {
                c->c.boundary[i] = (float)cb->boundary[i];
                c->c.boundary_sd[i] = bsd;
            }
        }
    }
    if (n == 16) {
        // two-level split of the 4-bit centroids: N[c] = round(C[c] / delta)
        // with delta = max|C| / 2047, the remainder taken against the fp32 delta
        double cmax = 0.0;
        for (int i = 0; i < n; ++i) cmax = std::fmax(cmax, std::fabs(cb->centroid[i]));
        const float fd = (float)(cmax / 2047.0);
        c->c.delta = fd;
        for (int i = 0; i < n; ++i) {
            double nq = std::nearbyint(cb->centroid[i] / (double)fd);
            if (nq > 2047.0) nq = 2047.0;
            if (nq < -2047.0) nq = -2047.0;
            c->c.cint_f16[i] = half_bits_from_double(nq);
            c->c.crem_f16[i] = half_bits_from_double(cb->centroid[i] - (double)fd * nq);
        }
    }
    tq_codebook_free(cb);

    derive_signs(seed, d, c->signs);
    for (int j = 0; j < d; ++j)
        if (c->signs[j] < 0) c->c.sign_bits[j / 32] |= 1u << (j % 32);

    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "cudaGetDevice");
    }
    e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "cudaDeviceGetAttribute");
    }

    e = cudaMalloc(&c->tab_dev, sizeof(CodeTables));
    if (e == cudaSuccess) e = cudaMemcpy(c->tab_dev, &tab, sizeof(CodeTables), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (c->tab_dev) cudaFree(c->tab_dev);
        delete c;
        return cuda_fail(e, "uploading the code tables");
    }

    if (qjl_m > 0) {
        const int64_t cnt = (int64_t)qjl_m * d;
        c->S_host = new (std::nothrow) double[cnt];
        float* tmp = new (std::nothrow) float[cnt];
        if (!c->S_host || !tmp) {
            delete[] tmp;
            delete[] c->S_host;
            delete c;
            return fail(TQ_ERR_INVALID_ARG, "out of host memory");
        }
        derive_gaussian(seed, qjl_m, d, c->S_host);
        for (int64_t k = 0; k < cnt; ++k) tmp[k] = (float)c->S_host[k];
        e = cudaMalloc(&c->S_dev, sizeof(float) * cnt);
        if (e == cudaSuccess) e = cudaMemcpy(c->S_dev, tmp, sizeof(float) * cnt, cudaMemcpyHostToDevice);
        delete[] tmp;
        if (e != cudaSuccess) {
            if (c->S_dev) cudaFree(c->S_dev);
            cudaFree(c->tab_dev);
            delete[] c->S_host;
            delete c;
            return cuda_fail(e, "uploading the QJL matrix");
        }
    }
    *out = c;
    return TQ_OK;
}

TQ_API void tq_cache_free(tq_cache* c) {
    if (!c) return;
    if (c->S_dev) cudaFree(c->S_dev);
    if (c->tab_dev) cudaFree(c->tab_dev);
    delete[] c->S_host;
    delete c;
}

TQ_API tq_status tq_cache_signs(const tq_cache* c, int8_t* signs) {
    if (!c || !signs) return fail(TQ_ERR_INVALID_ARG, "NULL argument");
    std::memcpy(signs, c->signs, (size_t)c->g.d);
    return TQ_OK;
}

TQ_API tq_status tq_cache_gaussian(const tq_cache* c, double* S) {
    if (!c || !S) return fail(TQ_ERR_INVALID_ARG, "NULL argument");
    if (c->g.m == 0) return fail(TQ_ERR_INVALID_ARG, "cache has no QJL matrix");
    std::memcpy(S, c->S_host, sizeof(double) * (size_t)c->g.m * c->g.d);
    return TQ_OK;
}

TQ_API tq_status tq_encode_kv(const tq_cache* c, const void* K, const void* V, tq_dtype dtype,
                              int64_t num_tokens, const int64_t* slot_mapping, int32_t* dev_status,
                              void* stream) {
    if (!c) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    if (num_tokens < 0) return fail(TQ_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return TQ_OK;
    if (!K || !V || !slot_mapping) return fail(TQ_ERR_INVALID_ARG, "K, V and slot_mapping must be non-NULL");
    if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad dtype");
    if ((reinterpret_cast<uintptr_t>(K) % 16) || (reinterpret_cast<uintptr_t>(V) % 16))
        return fail(TQ_ERR_INVALID_ARG, "K and V must be 16-byte aligned");
    EncodeArgs a{};
    a.g = c->g;
    a.c = c->c;
    a.pool = (uint8_t*)c->pool;
    a.K = K;
    a.V = V;
    a.dtype = (int)dtype;
    a.num_tokens = num_tokens;
    a.slot_mapping = slot_mapping;
    a.status = dev_status;
    a.S = c->S_dev;
    a.tab = c->tab_dev;
    int e = launch_encode(a, c->num_sms, stream);
    if (e != 0) return cuda_fail((cudaError_t)e, "encode launch");
    return TQ_OK;
}

// Splits per (sequence, KV head).  The decode kernel keeps one CTA per SM, so
// a launch runs in waves of num_sms CTAs.  The split count minimises a simple
// time model: waves x (page rounds of one CTA x 1.2 us + 6 us), a page round
// being one page per warp (12 warps, 8 with QJL).  The constants are the
// measured per-page and fixed (prologue, merge) costs on the 32K GQA
// workload: 9 rounds in ~10.9 us plus ~6 us.  At most ceil(max_blocks / 8)
// splits (8 pages or more each) and four times the count that fills the SMs.
static void decode_split_plan(const tq_cache* c, int batch, int max_blocks, int* splits, int* pps) {
    const int64_t units = (int64_t)batch * c->g.hkv;
    const int nw = c->g.m ? 8 : 12;
    const int64_t sms = c->num_sms > 0 ? c->num_sms : 1;
    int64_t lim = 4 * ((sms + units - 1) / units);
    const int64_t cap = (max_blocks + 7) / 8;
    if (lim > cap) lim = cap;
    if (lim < 1) lim = 1;
    int best_s = 1;
    double best = 1e300;
    for (int64_t s = 1; s <= lim; ++s) {
        const int64_t p = (max_blocks + s - 1) / s;
        const int64_t se = (max_blocks + p - 1) / p;
        const int64_t waves = (units * se + sms - 1) / sms;
        const double cost = (double)waves * ((double)((p + nw - 1) / nw) * 1.2 + 6.0);
        if (cost < best) {
            best = cost;
            best_s = (int)s;
        }
    }
    int p = (max_blocks + best_s - 1) / best_s;
    if (p < 1) p = 1;
    *pps = p;
    *splits = (max_blocks + p - 1) / p;
    if (*splits < 1) *splits = 1;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

TQ_API size_t tq_decode_workspace_bytes(const tq_cache* c, int batch, int num_q_heads,
                                        int max_blocks_per_seq) {
    if (!c || batch <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_q_heads % c->g.hkv) return 0;
    int splits, pps;
    decode_split_plan(c, batch, max_blocks_per_seq, &splits, &pps);
    const int group = num_q_heads / c->g.hkv;
    size_t part = (size_t)batch * c->g.hkv * splits * group * (4 + c->g.d) * sizeof(float);
    return align_up(part, 256) + align_up((size_t)batch * c->g.hkv * sizeof(unsigned), 256);
}

static tq_status decode_common(const tq_cache* c, const void* q, tq_dtype dtype, int batch, int num_q_heads,
                               const int32_t* block_table, int max_blocks_per_seq, const int32_t* lens,
                               float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream, const void* knew, const void* vnew,
                               tq_dtype kv_dtype, int window) {
    if (!c) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0)
        return fail(TQ_ERR_INVALID_ARG, "bad batch / num_q_heads / max_blocks_per_seq");
    if (batch == 0) return TQ_OK;
    if (!q || !block_table || !lens || !out || !workspace)
        return fail(TQ_ERR_INVALID_ARG, "q, block_table, lens, out and workspace must be non-NULL");
    if (num_q_heads % c->g.hkv) return fail(TQ_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
    const int group = num_q_heads / c->g.hkv;
    if (group > 8) return fail(TQ_ERR_UNSUPPORTED, "query group larger than 8");
    if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad dtype");
    if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return fail(TQ_ERR_INVALID_ARG, "sm_scale must be positive");
    const int64_t elem = dtype == TQ_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(q) % (4 * elem)) || (reinterpret_cast<uintptr_t>(out) % 16))
        return fail(TQ_ERR_INVALID_ARG, "q must be aligned to 4 elements and out to 16 bytes");
    size_t need = tq_decode_workspace_bytes(c, batch, num_q_heads, max_blocks_per_seq);
    if (workspace_bytes < need) {
        set_error("workspace has %zu bytes, needs %zu", workspace_bytes, need);
        return TQ_ERR_WORKSPACE;
    }
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(TQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    int splits, pps;
    decode_split_plan(c, batch, max_blocks_per_seq, &splits, &pps);
    DecodeArgs a{};
    a.g = c->g;
    a.c = c->c;
    a.pool = (const uint8_t*)c->pool;
    a.q = q;
    a.dtype = (int)dtype;
    a.batch = batch;
    a.hq = num_q_heads;
    a.group = group;
    a.block_table = block_table;
    a.max_blocks = max_blocks_per_seq;
    a.lens = lens;
    a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
    a.out = out;
    size_t part = (size_t)batch * c->g.hkv * splits * group * (4 + c->g.d) * sizeof(float);
    a.partials = (float*)workspace;
    a.counters = (unsigned*)((char*)workspace + align_up(part, 256));
    a.pages_per_split = pps;
    a.num_splits = splits;
    a.status = dev_status;
    a.S = c->S_dev;
    a.tab = c->tab_dev;
    a.knew = knew;
    a.vnew = vnew;
    a.kv_dtype = (int)kv_dtype;
    a.window = window;
    int e = launch_decode(a, stream);
    if (e != 0) return cuda_fail((cudaError_t)e, "decode launch");
    return TQ_OK;
}

TQ_API tq_status tq_decode_attention(const tq_cache* c, const void* q, tq_dtype dtype, int batch,
                                     int num_q_heads, const int32_t* block_table,
                                     int max_blocks_per_seq, const int32_t* lens, float sm_scale,
                                     float* out, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, void* stream) {
    return decode_common(c, q, dtype, batch, num_q_heads, block_table, max_blocks_per_seq, lens, sm_scale, out,
                         workspace, workspace_bytes, dev_status, stream, nullptr, nullptr, TQ_BF16, 0);
}

static tq_status append_common(const tq_cache* c, const void* k_new, const void* v_new, tq_dtype kv_dtype,
                               const void* q, tq_dtype dtype, int batch, int num_q_heads,
                               const int32_t* block_table, int max_blocks_per_seq, const int32_t* lens, int window,
                               float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream) {
    if (!c) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    if (c->g.m > 0)
        return fail(TQ_ERR_UNSUPPORTED, "appending inside decode is built for caches without QJL; "
                                        "use tq_encode_kv then tq_decode_attention");
    if (batch > 0 && (!k_new || !v_new)) return fail(TQ_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
    if (kv_dtype != TQ_F32 && kv_dtype != TQ_BF16 && kv_dtype != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad kv dtype");
    if ((reinterpret_cast<uintptr_t>(k_new) % 16) || (reinterpret_cast<uintptr_t>(v_new) % 16))
        return fail(TQ_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    return decode_common(c, q, dtype, batch, num_q_heads, block_table, max_blocks_per_seq, lens, sm_scale, out,
                         workspace, workspace_bytes, dev_status, stream, k_new, v_new, kv_dtype, window);
}

TQ_API tq_status tq_decode_attention_append(const tq_cache* c, const void* k_new, const void* v_new,
                                            tq_dtype kv_dtype, const void* q, tq_dtype dtype, int batch,
                                            int num_q_heads, const int32_t* block_table,
                                            int max_blocks_per_seq, const int32_t* lens, float sm_scale,
                                            float* out, void* workspace, size_t workspace_bytes,
                                            int32_t* dev_status, void* stream) {
    return append_common(c, k_new, v_new, kv_dtype, q, dtype, batch, num_q_heads, block_table, max_blocks_per_seq,
                         lens, 0, sm_scale, out, workspace, workspace_bytes, dev_status, stream);
}

TQ_API tq_status tq_decode_attention_ring_append(const tq_cache* c, const void* k_new, const void* v_new,
                                                 tq_dtype kv_dtype, const void* q, tq_dtype dtype, int batch,
                                                 int num_q_heads, const int32_t* block_table,
                                                 int max_blocks_per_seq, const int32_t* lens, int window,
                                                 float sm_scale, float* out, void* workspace,
                                                 size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (window <= 0 || window % kBlockSize)
        return fail(TQ_ERR_INVALID_ARG, "window must be a positive multiple of the block size (16)");
    if (max_blocks_per_seq <= 0 || (int64_t)window > (int64_t)max_blocks_per_seq * kBlockSize)
        return fail(TQ_ERR_INVALID_ARG, "the block table holds fewer than window slots per sequence");
    return append_common(c, k_new, v_new, kv_dtype, q, dtype, batch, num_q_heads, block_table, max_blocks_per_seq,
                         lens, window, sm_scale, out, workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"
