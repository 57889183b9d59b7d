// Host side of the library: argument checking, the Lloyd-Max codebook, the
// seeded sign vector and Gaussian matrix, cache descriptors and the calls
// that launch the kernels.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

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

// Wait-timeout test hook (tq_test_stall_waits): SM cycles the stalled warps
// wait, 0 when off.  Read once per decode launch.
static std::atomic<long long> g_stall_cycles{0};
long long test_stall_cycles() { return g_stall_cycles.load(std::memory_order_relaxed); }

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

// ---------------------------------------------------------------------------
// OCTOPUS codebooks (host).  Two densities: the xi coordinate of the
// octahedral map of a uniform direction on S^2, and the norm of three
// coordinates of a uniform point on S^{d-1}.  Lloyd-Max on each, with the cell
// integrals read from cumulative tables on a fine grid (Simpson's rule per
// grid interval, and on the partial interval up to a boundary), started from
// the equal-mass levels.
// ---------------------------------------------------------------------------
namespace {

// density of (xi, eta) on the square: 1 / (4 pi |p|^3), p the point of the
// octahedron |x| + |y| + |z| = 1 that (xi, eta) stands for (the lower half
// folded over the square's corners)
double oct_joint_density(double xi, double eta) {
    double x = xi, y = eta, z = 1.0 - std::fabs(xi) - std::fabs(eta);
    if (z < 0.0) {
        x = (1.0 - std::fabs(eta)) * (xi < 0.0 ? -1.0 : 1.0);
        y = (1.0 - std::fabs(xi)) * (eta < 0.0 ? -1.0 : 1.0);
    }
    const double r2 = x * x + y * y + z * z;
    return 1.0 / (4.0 * M_PI * r2 * std::sqrt(r2));
}

template <typename F>
double simpson(F f, double a, double b, int n) {  // n even
    const double h = (b - a) / n;
    double s = f(a) + f(b);
    for (int i = 1; i < n; ++i) s += f(a + i * h) * ((i & 1) ? 4.0 : 2.0);
    return s * h / 3.0;
}

double oct_xi_density(double xi) {
    if (xi < -1.0 || xi > 1.0) return 0.0;  // positive up to the ends (f(+-1) = f(0))
    const double e = 1.0 - std::fabs(xi);
    auto f = [xi](double eta) { return oct_joint_density(xi, eta); };
    return simpson(f, -1.0, -e, 64) + simpson(f, -e, 0.0, 64) + simpson(f, 0.0, e, 64) + simpson(f, e, 1.0, 64);
}

double oct_rho_density(int d, double r) {
    if (r <= 0.0 || r >= 1.0) return 0.0;
    const double lb = std::lgamma(1.5) + std::lgamma((d - 3) / 2.0) - std::lgamma(d / 2.0);
    return 2.0 * r * r * std::pow(1.0 - r * r, (d - 5) / 2.0) * std::exp(-lb);
}

struct CumTable {
    int kind, d, n;
    double lo, h;
    std::vector<double> F0, F1;  // mass and first moment from lo to grid point k
    double f(double x) const { return kind == 0 ? oct_xi_density(x) : oct_rho_density(d, x); }
    void build(int kind_, int d_, double lo_, double hi_, int n_) {
        kind = kind_; d = d_; n = n_; lo = lo_; h = (hi_ - lo_) / n_;
        F0.assign(n + 1, 0.0);
        F1.assign(n + 1, 0.0);
        for (int k = 0; k < n; ++k) {
            const double a = lo + k * h, m = a + 0.5 * h, b = a + h;
            const double fa = f(a), fm = f(m), fb = f(b);
            F0[k + 1] = F0[k] + h / 6.0 * (fa + 4.0 * fm + fb);
            F1[k + 1] = F1[k] + h / 6.0 * (a * fa + 4.0 * m * fm + b * fb);
        }
    }
    // integral from lo to x of f (moment 0) or x f (moment 1)
    double cum(double x, int moment) const {
        if (x <= lo) return 0.0;
        int k = (int)std::floor((x - lo) / h);
        if (k >= n) return moment ? F1[n] : F0[n];
        const double a = lo + k * h, m = 0.5 * (a + x);
        const double fa = f(a), fm = f(m), fx = f(x);
        const double part = moment ? (x - a) / 6.0 * (a * fa + 4.0 * m * fm + x * fx)
                                   : (x - a) / 6.0 * (fa + 4.0 * fm + fx);
        return (moment ? F1[k] : F0[k]) + part;
    }
};

// Lloyd-Max on a tabulated density over [lo, hi]; levels c[0..nl), boundaries
// at their midpoints
void oct_lloyd(const CumTable& T, double hi, int nl, double* c) {
    const double total = T.cum(hi, 0);
    // start: the levels that split the mass equally (bisection on the table)
    for (int i = 0; i < nl; ++i) {
        const double target = total * (i + 0.5) / nl;
        double a = T.lo, b = hi;
        for (int it = 0; it < 200; ++it) {
            const double m = 0.5 * (a + b);
            if (T.cum(m, 0) < target) a = m;
            else b = m;
        }
        c[i] = 0.5 * (a + b);
    }
    std::vector<double> t(nl > 1 ? nl - 1 : 1);
    for (int it = 0; it < 100000; ++it) {
        for (int i = 0; i + 1 < nl; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
        double delta = 0.0;
        for (int i = 0; i < nl; ++i) {
            const double a = i == 0 ? T.lo : t[i - 1], b = i == nl - 1 ? hi : t[i];
            const double mass = T.cum(b, 0) - T.cum(a, 0);
            const double cn = mass > 0.0 ? (T.cum(b, 1) - T.cum(a, 1)) / mass : 0.5 * (a + b);
            delta = std::fmax(delta, std::fabs(cn - c[i]));
            c[i] = cn;
        }
        if (delta < 1e-14) break;
    }
}

}  // namespace

// xi levels (kind 0, 2^bits of them) or triplet-norm levels (kind 1) for dimension d
void octopus_levels(int kind, int d, int bits, double* c) {
    CumTable T;
    if (kind == 0) T.build(0, d, -1.0, 1.0, 8192);
    else T.build(1, d, 0.0, 1.0, 8192);
    oct_lloyd(T, 1.0, 1 << bits, c);
}

int octopus_key_row(int d, int b) { return 4 * ((((d + 2) / 3) * (3 * b + 1) + 31) / 32); }

Geometry make_oct_geometry(int d, int b, int vb, int bs, int hkv, int64_t num_blocks) {
    Geometry g{};
    g.d = d; g.kb = b; g.vb = vb; g.m = 0; g.bs = bs; g.hkv = hkv;
    g.num_blocks = num_blocks;
    int off = 0;
    g.kcode_off = off; off += bs * octopus_key_row(d, b);
    g.vcode_off = off; off += bs * d * vb / 8;
    g.gam_off = off; off += 2 * bs;
    g.scl_off = off; off += 2 * bs;
    g.zer_off = off; off += 2 * bs;
    g.rho_off = g.sig_off = -1;
    g.page_bytes = (off + 15) / 16 * 16;
    return g;
}

}  // namespace tq

using namespace tq;

// ===========================================================================
// C ABI
// ===========================================================================

extern "C" {

TQ_API tq_status tq_device_accessible(const void* p, int* accessible) {
    if (!accessible) return fail(TQ_ERR_INVALID_ARG, "accessible is NULL");
    *accessible = 0;
    if (!p) return TQ_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaPointerAttributes at{};
    e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // memory the runtime does not know: not accessible
        return TQ_OK;
    }
    if ((at.type == cudaMemoryTypeDevice && at.device == dev) || at.type == cudaMemoryTypeManaged)
        *accessible = 1;
    else if (at.type == cudaMemoryTypeHost && at.devicePointer == p)
        *accessible = 1;
    return TQ_OK;
}

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

TQ_API void tq_test_stall_waits(int64_t cycles) {
    g_stall_cycles.store(cycles > 0 ? (long long)cycles : 0, std::memory_order_relaxed);
}

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
            c->c.cremd_f16[i] = half_bits_from_double((cb->centroid[i] - (double)fd * nq) / (double)fd);
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
    if (c->oct_dev) cudaFree(c->oct_dev);
    delete[] c->S_host;
    delete c;
}

TQ_API int64_t tq_octopus_page_bytes(int d, int bits, int value_bits, int block_size) {
    if (d <= 0 || d % 8 || bits < 2 || bits > 4 || value_bits < 1 || value_bits > 8 || block_size <= 0) return -1;
    return make_oct_geometry(d, bits, value_bits, block_size, 1, 1).page_bytes;
}

TQ_API tq_status tq_octopus_codebook(int d, int bits, int kind, double* levels) {
    if (!levels) return fail(TQ_ERR_INVALID_ARG, "levels is NULL");
    if (d < 6 || d > 1024 || kind < 0 || kind > 1 || bits < 1 || bits > 5)
        return fail(TQ_ERR_INVALID_ARG, "d 6..1024, kind 0 or 1, bits 1..5");
    octopus_levels(kind, d, bits, levels);
    return TQ_OK;
}

TQ_API tq_status tq_cache_create_octopus(void* pool, int64_t num_blocks, int block_size, int num_kv_heads, int d,
                                         int bits, int value_bits, uint64_t seed, tq_cache** out) {
    if (!out) return fail(TQ_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!pool) return fail(TQ_ERR_INVALID_ARG, "pool is NULL");
    if ((reinterpret_cast<uintptr_t>(pool) & 15) != 0) return fail(TQ_ERR_INVALID_ARG, "pool must be 16-byte aligned");
    if (num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0 || d <= 0)
        return fail(TQ_ERR_INVALID_ARG, "sizes must be positive");
    if (tq_octopus_page_bytes(d, bits, value_bits, block_size) < 0)
        return fail(TQ_ERR_INVALID_ARG, "invalid d / bits / value_bits combination (bits 2..4, value bits 1..8)");
    if (d != kHeadDim) return fail(TQ_ERR_UNSUPPORTED, "head dim must be 128");
    if (block_size != kBlockSize) return fail(TQ_ERR_UNSUPPORTED, "block_size must be 16");
    tq_cache* c = new (std::nothrow) tq_cache();
    if (!c) return fail(TQ_ERR_INVALID_ARG, "out of host memory");
    c->pool = pool;
    c->seed = seed;
    c->octopus = 1;
    c->g = make_oct_geometry(d, bits, value_bits, block_size, num_kv_heads, num_blocks);
    c->oct_key_row = octopus_key_row(d, bits);
    std::memset(&c->c, 0, sizeof(c->c));
    derive_signs(seed, d, c->signs);
    for (int j = 0; j < d; ++j)
        if (c->signs[j] < 0) c->c.sign_bits[j / 32] |= 1u << (j % 32);
    // codebooks and the direction table of the level pairs
    OctTables& T = c->oct_host;
    std::memset(&T, 0, sizeof(T));
    const int nxi = 1 << (bits + 1), nrho = 1 << (bits - 1);
    double cx[kOctMaxDir], cr[8];
    octopus_levels(0, d, bits + 1, cx);
    octopus_levels(1, d, bits - 1, cr);
    for (int i = 0; i < nxi; ++i) {
        T.cxi[i] = (float)cx[i];
        if (i + 1 < nxi) T.bxi[i] = (float)(0.5 * (cx[i] + cx[i + 1]));
    }
    for (int i = 0; i < nrho; ++i) {
        T.crho[i] = (float)cr[i];
        if (i + 1 < nrho) T.brho[i] = (float)(0.5 * (cr[i] + cr[i + 1]));
    }
    for (int a = 0; a < nxi; ++a)
        for (int b = 0; b < nxi; ++b) {
            // the unit direction of the octahedron point of (cx[a], cx[b])
            double x = cx[a], y = cx[b], z = 1.0 - std::fabs(x) - std::fabs(y);
            if (z < 0.0) {
                const double xf = (1.0 - std::fabs(cx[b])) * (cx[a] < 0.0 ? -1.0 : 1.0);
                const double yf = (1.0 - std::fabs(cx[a])) * (cx[b] < 0.0 ? -1.0 : 1.0);
                x = xf;
                y = yf;
            }
            const double r = std::sqrt(x * x + y * y + z * z);
            float* dd = T.dir[a * kOctMaxDir + b];
            dd[0] = (float)(x / r);
            dd[1] = (float)(y / r);
            dd[2] = (float)(z / r);
            dd[3] = 0.f;
        }
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e == cudaSuccess) e = cudaMalloc(&c->oct_dev, sizeof(OctTables));
    if (e == cudaSuccess) e = cudaMemcpy(c->oct_dev, &T, sizeof(OctTables), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (c->oct_dev) cudaFree(c->oct_dev);
        delete c;
        return cuda_fail(e, "creating the OCTOPUS cache");
    }
    *out = c;
    return TQ_OK;
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
    if (c->octopus) {
        OctArgs o{};
        o.g = c->g;
        o.key_row = c->oct_key_row;
        o.tab = c->oct_dev;
        std::memcpy(o.sign_bits, c->c.sign_bits, sizeof(o.sign_bits));
        o.pool = (uint8_t*)c->pool;
        o.status = dev_status;
        o.K = K;
        o.V = V;
        o.dtype = (int)dtype;
        o.num_tokens = num_tokens;
        o.slot_mapping = slot_mapping;
        int e = launch_oct_encode(o, c->num_sms, stream);
        if (e != 0) return cuda_fail((cudaError_t)e, "OCTOPUS encode launch");
        return TQ_OK;
    }
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
// being one page per warp (12 warps, 8 with QJL, 16 for OCTOPUS keys).  The
// constants are the measured per-page and fixed (prologue, merge) costs on
// the 32K GQA workload: 9 rounds in ~10.9 us plus ~6 us.  At most ceil(max_blocks / 8)
// splits (8 pages or more each) and four times the count that fills the SMs.
static void decode_split_plan(const tq_cache* c, int batch, int max_blocks, int* splits, int* pps) {
    const int64_t units = (int64_t)batch * c->g.hkv;
    const int nw = c->octopus ? 16 : c->g.m ? 8 : 12;  // warps per CTA
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
    if (c->octopus) {
        // one partial per split: (max, sum, 2 pad, acc[d]) per query
        return align_up((size_t)batch * c->g.hkv * splits * group * (4 + c->g.d) * sizeof(float), 256);
    }
    size_t part = (size_t)batch * c->g.hkv * splits * group * (4 + c->g.d) * sizeof(float);
    return align_up(part, 256) + align_up((size_t)batch * c->g.hkv * sizeof(unsigned), 256);
}

static tq_status decode_common(const tq_cache* c, const void* q, tq_dtype dtype, int batch, int num_q_heads,
                               const int32_t* block_table, int max_blocks_per_seq, const int32_t* lens,
                               float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream, const void* knew, const void* vnew,
                               tq_dtype kv_dtype, int window, int64_t bt_stride = -1) {
    if (bt_stride < 0) bt_stride = max_blocks_per_seq;
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
    if (c->octopus) {
        if (knew) return fail(TQ_ERR_UNSUPPORTED, "appending inside decode is not built for OCTOPUS caches");
        OctArgs o{};
        o.g = c->g;
        o.key_row = c->oct_key_row;
        o.tab = c->oct_dev;
        std::memcpy(o.sign_bits, c->c.sign_bits, sizeof(o.sign_bits));
        o.pool = (uint8_t*)c->pool;
        o.status = dev_status;
        o.q = q;
        o.dtype = (int)dtype;
        o.batch = batch;
        o.hq = num_q_heads;
        o.group = group;
        o.block_table = block_table;
        o.max_blocks = max_blocks_per_seq;
        o.bt_stride = bt_stride;
        o.lens = lens;
        o.sm_scale_log2 = sm_scale * 1.4426950408889634f;
        o.out = out;
        o.partials = (float*)workspace;
        o.pages_per_split = pps;
        o.num_splits = splits;
        o.stall_cycles = test_stall_cycles();
        int e = launch_oct_decode(o, stream);
        if (e != 0) return cuda_fail((cudaError_t)e, "OCTOPUS decode launch");
        return TQ_OK;
    }
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
    a.bt_stride = bt_stride;
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
    a.stall_cycles = test_stall_cycles();
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
    if (c->octopus)
        return fail(TQ_ERR_UNSUPPORTED, "appending inside decode is not built for OCTOPUS caches; "
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

// Splits of the tensor-core prefill: the (KV head, 128-row block) units spread
// over the SMs, at most one split per 128-token tile of the block table.
static int prefill_tc_splits(const tq_cache* c, int num_positions, int num_q_heads, int max_blocks) {
    const int64_t rows = (int64_t)num_positions * (num_q_heads / c->g.hkv);
    const int64_t nrb = (rows + prefill_tc_rows_per_block() - 1) / prefill_tc_rows_per_block();
    const int64_t units = (int64_t)c->g.hkv * nrb;
    const int64_t sms = c->num_sms > 0 ? c->num_sms : 1;
    int64_t s = sms / units;
    const int64_t tiles = ((int64_t)max_blocks * c->g.bs + prefill_tc_tile_tokens() - 1) / prefill_tc_tile_tokens();
    if (s > tiles) s = tiles;
    if (s < 1) s = 1;
    return (int)s;
}

static bool prefill_on_tc(const tq_cache* c) { return !c->octopus && prefill_tc_supported(c->g); }

TQ_API size_t tq_prefill_workspace_bytes(const tq_cache* c, int num_positions, int num_q_heads,
                                         int max_blocks_per_seq) {
    if (!c || num_positions <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_q_heads % c->g.hkv) return 0;
    if (prefill_on_tc(c)) {
        const int splits = prefill_tc_splits(c, num_positions, num_q_heads, max_blocks_per_seq);
        return align_up(prefill_tc_partials_bytes(c->g, num_positions, num_q_heads, splits), 256);
    }
    const size_t w = tq_decode_workspace_bytes(c, num_positions, num_q_heads, max_blocks_per_seq);
    if (w == 0) return 0;
    return w + align_up((size_t)num_positions * sizeof(int32_t), 256);
}

TQ_API tq_status tq_prefill_attention(const tq_cache* c, const void* q, tq_dtype dtype, int num_positions,
                                      int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                                      int first_position, float sm_scale, float* out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (!c) return fail(TQ_ERR_INVALID_ARG, "cache is NULL");
    if (num_positions < 0 || first_position < 0) return fail(TQ_ERR_INVALID_ARG, "negative positions");
    if (num_positions == 0) return TQ_OK;
    if (max_blocks_per_seq <= 0 ||
        (int64_t)first_position + num_positions > (int64_t)max_blocks_per_seq * c->g.bs)
        return fail(TQ_ERR_INVALID_ARG, "the block table holds fewer slots than the chunk's last position");
    const size_t need = tq_prefill_workspace_bytes(c, num_positions, num_q_heads, max_blocks_per_seq);
    if (need == 0) return fail(TQ_ERR_INVALID_ARG, "bad num_q_heads / max_blocks_per_seq");
    if (!workspace) return fail(TQ_ERR_INVALID_ARG, "workspace is NULL");
    if (workspace_bytes < need) {
        set_error("workspace has %zu bytes, needs %zu", workspace_bytes, need);
        return TQ_ERR_WORKSPACE;
    }
    if (prefill_on_tc(c)) {
        if (num_q_heads % c->g.hkv) return fail(TQ_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
        const int group = num_q_heads / c->g.hkv;
        if (group > 8) return fail(TQ_ERR_UNSUPPORTED, "query group larger than 8");
        if (!q || !block_table || !out) return fail(TQ_ERR_INVALID_ARG, "q, block_table and out must be non-NULL");
        if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad dtype");
        if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return fail(TQ_ERR_INVALID_ARG, "sm_scale must be positive");
        const int64_t elem = dtype == TQ_F32 ? 4 : 2;
        if ((reinterpret_cast<uintptr_t>(q) % (4 * elem)) || (reinterpret_cast<uintptr_t>(out) % 16) ||
            (reinterpret_cast<uintptr_t>(workspace) % 256))
            return fail(TQ_ERR_INVALID_ARG, "q must be aligned to 4 elements, out to 16 bytes, workspace to 256");
        PrefillArgs p{};
        p.g = c->g;
        p.c = c->c;
        p.pool = (const uint8_t*)c->pool;
        p.q = q;
        p.dtype = (int)dtype;
        p.C = num_positions;
        p.hq = num_q_heads;
        p.group = group;
        p.block_row = block_table;
        p.max_blocks = max_blocks_per_seq;
        p.first = first_position;
        p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
        p.out = out;
        p.partials = (float*)workspace;
        p.nrb = (num_positions * group + prefill_tc_rows_per_block() - 1) / prefill_tc_rows_per_block();
        p.splits = prefill_tc_splits(c, num_positions, num_q_heads, max_blocks_per_seq);
        const int ntile = (first_position + num_positions + prefill_tc_tile_tokens() - 1) / prefill_tc_tile_tokens();
        p.tiles_per_split = (ntile + p.splits - 1) / p.splits;
        p.status = dev_status;
        p.stall_cycles = test_stall_cycles();
        int e = launch_prefill_tc(p, stream);
        if (e != 0) return cuda_fail((cudaError_t)e, "prefill launch");
        return TQ_OK;
    }
    const size_t dec = tq_decode_workspace_bytes(c, num_positions, num_q_heads, max_blocks_per_seq);
    int32_t* lens = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + dec);
    int e = launch_fill_positions(lens, num_positions, first_position, stream);
    if (e != 0) return cuda_fail((cudaError_t)e, "prefill lengths");
    return decode_common(c, q, dtype, num_positions, num_q_heads, block_table, max_blocks_per_seq, lens, sm_scale,
                         out, workspace, dec, dev_status, stream, nullptr, nullptr, TQ_BF16, 0, 0);
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
