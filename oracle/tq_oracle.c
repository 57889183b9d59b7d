/*
 * tq_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU restatement of online KV-cache compression and of
 * attention over the compressed cache.  Only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark may load this file's library; the
 * product path never does.  It shares no source, header, table or generator
 * with the CUDA library: every step below is written out from its definition.
 *
 * Sources (web pages, cited as "page title -- section"):
 *   [P1] "TurboQuant: KV Cache Vector Quantization" (llm-engineer card)
 *   [P2] "TurboQuant: KV Cache Compression" (Bit-Axon docs)
 *   [P3] "OCTOPUS: Optimized KV Cache for Transformers via Octahedral
 *        Parametrization ..." (aitrends.kr summary)
 *   [P4] "TurboQuant deep dive" (cell-devlog blog post 199)
 *
 * What is computed, step by step:
 *   split     gamma = ||k||_2, u = k / gamma        [P1 three steps, 1. Split;
 *                                                   P3 methodology step 1]
 *   rotate    R x = H (s (.) x) / sqrt(d), H the natural-order (Sylvester)
 *             Walsh-Hadamard matrix H[i][j] = (-1)^popcount(i & j), s in {+-1}^d
 *             drawn from the seed                  [P4 Step 1: RHT; P3 step 2]
 *   codebook  per-coordinate Lloyd-Max codebook for the marginal density of one
 *             coordinate of a uniform point on S^{d-1}
 *                                                  [P3 key idea; glossary
 *                                                   "Lloyd-Max quantization"]
 *   keys      idx_j = #{ i : t_i < u_rot[j] },  t_i = (c_i + c_{i+1}) / 2,
 *             i.e. the nearest centroid, ties to the lower index
 *                                                  [P2 quantization function]
 *   values    per-token min-max b-bit codes in the rotated frame, fp16 scale
 *             and zero                             [P4 Step 3 (value path)]
 *   QJL       r = u_rot - C[idx], rho = ||r||, sigma_i = [(S r)_i >= 0], S an
 *             m x d Gaussian matrix from the seed  [P3 contribution "Optional
 *                                                   1-bit QJL residual"; step 8]
 *   attention softmax(q K^T / sqrt(d_h)) V over the reconstructed keys/values
 *             in the original frame                [P2 attention under
 *                                                   quantized KV]
 *
 * Readings where the pages are silent or inconsistent are stated at each
 * function.  Everything is float64 except the values the cache stores in fp16,
 * which are rounded to binary16 (round to nearest even) and read back widened.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* device-status bits written by encode/decode (same meaning as the library's
 * status word; restated here, not shared) */
#define ORC_FLAG_OVERFLOW 1
#define ORC_FLAG_BAD_SLOT 2
#define ORC_FLAG_NONFINITE 4

/* ------------------------------------------------------------------------ */
/* threads                                                                   */
/* ------------------------------------------------------------------------ */

ORC_API int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Counter-based SplitMix64 stream.                                          */
/* SplitMix64 (Steele, Lea, Flood, OOPSLA 2014): state advances by the Weyl  */
/* increment 0x9E3779B97F4A7C15 and each output is the state passed through  */
/* the finaliser z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;            */
/* z *= 0x94D049BB133111EB; z ^= z>>31.                                      */
/* Stream (seed, tag), output i (i = 0, 1, ...):                             */
/*     z_i = mix(key + (i + 1) * 0x9E3779B97F4A7C15),                        */
/*     key = seed XOR (tag * 0xD1B54A32D192ED03).                            */
/* Tag 0 gives the rotation signs, tag 1 the QJL Gaussian matrix.  The pages */
/* draw signs from torch's generator [P4 Step 1]; that generator is not     */
/* reproduced -- this one is defined here instead.                           */
/* ------------------------------------------------------------------------ */

static uint64_t orc_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

ORC_API uint64_t orc_stream_at(uint64_t seed, uint64_t tag, uint64_t i) {
    uint64_t key = seed ^ (tag * 0xD1B54A32D192ED03ULL);
    return orc_mix(key + (i + 1) * 0x9E3779B97F4A7C15ULL);
}

ORC_API void orc_stream(uint64_t seed, uint64_t tag, uint64_t start, int64_t n,
                        uint64_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_stream_at(seed, tag, start + (uint64_t)i);
}

/* s_j = +1 if the top bit of z_j(seed, 0) is clear, else -1. */
ORC_API void orc_signs(uint64_t seed, int d, double* s) {
    for (int j = 0; j < d; ++j) s[j] = (orc_stream_at(seed, 0, (uint64_t)j) >> 63) ? -1.0 : 1.0;
}

/* S[i][j] (row-major, n = i*d + j): Box-Muller (1958), cosine branch,
 *   u1 = ((z_{2n} >> 11) + 1) * 2^-53  in (0, 1],
 *   u2 =  (z_{2n+1} >> 11)    * 2^-53  in [0, 1),
 *   S  = sqrt(-2 ln u1) * cos(2 pi u2). */
ORC_API void orc_gaussian(uint64_t seed, int m, int d, double* S) {
    const double two53 = 9007199254740992.0;
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t n = 0; n < (int64_t)m * d; ++n) {
        uint64_t a = orc_stream_at(seed, 1, (uint64_t)(2 * n));
        uint64_t b = orc_stream_at(seed, 1, (uint64_t)(2 * n + 1));
        double u1 = ((double)(a >> 11) + 1.0) / two53;
        double u2 = (double)(b >> 11) / two53;
        S[n] = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
    }
}

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard rotation, explicit O(d^2) matrix.                          */
/* ------------------------------------------------------------------------ */

static int orc_popcount(unsigned v) {
    int c = 0;
    while (v) { c += (int)(v & 1u); v >>= 1; }
    return c;
}

/* H[i][j] = (-1)^popcount(i & j): the natural-order (Sylvester) Hadamard
 * matrix that the pages' divide-and-conquer transform applies [P4 Step 1]. */
ORC_API void orc_hadamard(int d, double* H) {
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            H[(int64_t)i * d + j] = (orc_popcount((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
}

/* y = R x = H (s (.) x) / sqrt(d): signs first, then H, then 1/sqrt(d)
 * [P4 Step 1].  The 1/sqrt(d) that [P3 step 2] omits is kept so that R is
 * orthogonal. */
ORC_API void orc_rotate(int d, const double* s, const double* x, double* y) {
    const double inv = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) {
            double h = (orc_popcount((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
            acc += h * s[j] * x[j];
        }
        y[i] = acc * inv;
    }
}

/* x = R^T y = s (.) (H y) / sqrt(d).  [P4 Step 3] says the inverse is "apply
 * the transform again"; that is not so (R R != I), the transpose is used. */
ORC_API void orc_rotate_inverse(int d, const double* s, const double* y, double* x) {
    const double inv = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) {
            double h = (orc_popcount((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
            acc += h * y[j];
        }
        x[i] = s[i] * acc * inv;
    }
}

/* ------------------------------------------------------------------------ */
/* Lloyd-Max codebook for one coordinate of a uniform point on S^{d-1}.      */
/*   f(x) = K (1 - x^2)^((d-3)/2) on [-1, 1],                                */
/*   K = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)).                             */
/* Cell mass: substitute x = -cos(theta), so f(x) dx = K sin^(d-2)(theta)    */
/* dtheta, and integrate with composite Gauss-Legendre in theta.             */
/* Cell first moment: closed form                                            */
/*   int_a^b x f(x) dx = K/(d-1) [ (1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2) ].  */
/* ------------------------------------------------------------------------ */

#define ORC_GL_N 20
static double orc_gl_x[ORC_GL_N], orc_gl_w[ORC_GL_N];
static int orc_gl_ready = 0;

/* Gauss-Legendre nodes/weights on [-1,1] by Newton's method on P_n, with
 * P_n from the recurrence (k) P_k = (2k-1) x P_{k-1} - (k-1) P_{k-2} and
 * P_n'(x) = n (x P_n - P_{n-1}) / (x^2 - 1); weight 2 / ((1-x^2) P_n'(x)^2). */
static void orc_legendre(int n, double x, double* pn, double* dpn) {
    double p0 = 1.0, p1 = x;
    for (int k = 2; k <= n; ++k) {
        double p2 = ((2.0 * k - 1.0) * x * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
    }
    *pn = p1;
    *dpn = n * (x * p1 - p0) / (x * x - 1.0);
}

static void orc_gl_init(void) {
    if (orc_gl_ready) return;
    const int n = ORC_GL_N;
    for (int i = 0; i < n; ++i) {
        double x = cos(M_PI * (i + 0.75) / (n + 0.5)), p, dp;
        for (int it = 0; it < 100; ++it) {
            orc_legendre(n, x, &p, &dp);
            double dx = p / dp;
            x -= dx;
            if (fabs(dx) < 1e-16) break;
        }
        orc_legendre(n, x, &p, &dp);
        orc_gl_x[i] = x;
        orc_gl_w[i] = 2.0 / ((1.0 - x * x) * dp * dp);
    }
    orc_gl_ready = 1;
}

/* K = r(d) / sqrt(pi) with r(d) = Gamma(d/2) / Gamma((d-1)/2), from
 * r(2) = 1/sqrt(pi), r(3) = sqrt(pi)/2 and r(n+2) = r(n) * n / (n-1)
 * (Gamma(x+1) = x Gamma(x)); exact up to one rounding per step. */
static double orc_norm_const(int d) {
    double r = (d % 2 == 0) ? 1.0 / sqrt(M_PI) : sqrt(M_PI) / 2.0;
    for (int n = (d % 2 == 0) ? 2 : 3; n < d; n += 2) r *= (double)n / (double)(n - 1);
    return r / sqrt(M_PI);
}

ORC_API double orc_density(int d, double x) {
    if (x <= -1.0 || x >= 1.0) return 0.0;
    return orc_norm_const(d) * pow(1.0 - x * x, (d - 3) / 2.0);
}

/* int_a^b f(x) dx, a <= b, both in [-1, 1] */
ORC_API double orc_cell_mass(int d, double a, double b) {
    orc_gl_init();
    if (a < -1.0) a = -1.0;
    if (b > 1.0) b = 1.0;
    if (b <= a) return 0.0;
    double ta = acos(-a), tb = acos(-b);
    int pieces = (int)ceil((tb - ta) / 0.02);
    if (pieces < 1) pieces = 1;
    double h = (tb - ta) / pieces, sum = 0.0;
    for (int p = 0; p < pieces; ++p) {
        double lo = ta + p * h, mid = lo + 0.5 * h, part = 0.0;
        for (int i = 0; i < ORC_GL_N; ++i) {
            double th = mid + 0.5 * h * orc_gl_x[i];
            part += orc_gl_w[i] * pow(sin(th), d - 2);
        }
        sum += 0.5 * h * part;
    }
    return orc_norm_const(d) * sum;
}

/* int_a^b x f(x) dx (closed form) */
ORC_API double orc_cell_moment(int d, double a, double b) {
    if (a < -1.0) a = -1.0;
    if (b > 1.0) b = 1.0;
    if (b <= a) return 0.0;
    double e = (d - 1) / 2.0;
    return orc_norm_const(d) / (d - 1) * (pow(1.0 - a * a, e) - pow(1.0 - b * b, e));
}

/* Lloyd-Max iteration [P3 glossary "Lloyd-Max quantization": centroids are
 * updated alternately with the cells so as to minimise mean squared error]:
 *   boundaries t_i = (c_i + c_{i+1}) / 2,
 *   centroids  c_i = int_cell x f / int_cell f,
 * from c_i = (2i + 1 - n)/n * 4/sqrt(d) (n = 2^bits, evenly spaced over four
 * standard deviations), until max |c_new - c_old| < tol or max_iter passes.
 * Writes n centroids and n-1 boundaries; returns the passes taken. */
ORC_API int orc_lloyd_max(int d, int bits, double tol, int max_iter,
                          double* centroids, double* boundaries) {
    const int n = 1 << bits;
    double* c = centroids;
    double* t = boundaries;
    for (int i = 0; i < n; ++i) c[i] = (2.0 * i + 1.0 - n) / n * 4.0 / sqrt((double)d);
    int it = 0;
    for (; it < max_iter; ++it) {
        for (int i = 0; i + 1 < n; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
        double delta = 0.0;
        for (int i = 0; i < n; ++i) {
            double lo = (i == 0) ? -1.0 : t[i - 1];
            double hi = (i == n - 1) ? 1.0 : t[i];
            double mass = orc_cell_mass(d, lo, hi);
            double cn = (mass > 0.0) ? orc_cell_moment(d, lo, hi) / mass : 0.5 * (lo + hi);
            double dd = fabs(cn - c[i]);
            if (dd > delta) delta = dd;
            c[i] = cn;
        }
        if (delta < tol) { ++it; break; }
    }
    for (int i = 0; i + 1 < n; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
    return it;
}

/* ------------------------------------------------------------------------ */
/* binary16 rounding (IEEE 754 round to nearest, ties to even).             */
/* ------------------------------------------------------------------------ */

/* the binary16 value nearest to x, as a double (+-inf past the largest) */
ORC_API double orc_fp16_round(double x) {
    if (isnan(x)) return x;
    double ax = fabs(x);
    if (ax >= 65520.0) return x > 0 ? INFINITY : -INFINITY;
    if (ax == 0.0) return x;
    int e;
    frexp(ax, &e);          /* ax = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
    int ue = e - 1;
    if (ue < -14) ue = -14; /* subnormal range: fixed quantum 2^-24 */
    double quantum = ldexp(1.0, ue - 10);
    double r = nearbyint(ax / quantum) * quantum; /* default mode: ties to even */
    return x < 0 ? -r : r;
}

ORC_API uint16_t orc_fp16_bits(double x) {
    double r = orc_fp16_round(x);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isnan(r)) return 0x7E00;
    if (isinf(r)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    int e;
    double f = frexp(a, &e);   /* a = f 2^e, f in [0.5,1) */
    int ue = e - 1;
    if (ue < -14) {            /* subnormal: a = mant * 2^-24 */
        return sign | (uint16_t)nearbyint(a * 16777216.0);
    }
    uint16_t mant = (uint16_t)nearbyint((f * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)((ue + 15) << 10) | mant;
}

ORC_API double orc_fp16_value(uint16_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, mant = h & 1023;
    double v;
    if (ex == 0) v = ldexp((double)mant, -24);
    else if (ex == 31) v = mant ? NAN : INFINITY;
    else v = ldexp(1024.0 + mant, ex - 25);
    return sign ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Paged cache layout.                                                       */
/* One page = one block of `bs` token slots of one KV head; page (block n,   */
/* head h) starts at byte (n * Hkv + h) * page_bytes.  Sections in order:    */
/*   key codes     bs rows of d*kb/8 bytes                                   */
/*   value codes   bs rows of d*vb/8 bytes                                   */
/*   gamma         bs binary16                                               */
/*   value scale   bs binary16                                               */
/*   value zero    bs binary16                                               */
/*   rho           bs binary16            (only if m > 0)                    */
/*   sigma         bs rows of m/8 bytes   (only if m > 0)                    */
/* then zero padding to a multiple of 16 bytes.  Inside a row, code j takes  */
/* bits [j*b, j*b + b) of the row read as a little-endian bit string (bit k  */
/* of the row is bit k%8 of byte k/8); sigma bit i is 1 iff (S r)_i >= 0.    */
/* The bit budget per key, d*b + 16, is the one [P4 "PolarQuant 압축 효율"]  */
/* counts.                                                                   */
/* ------------------------------------------------------------------------ */

typedef struct {
    int d, kb, vb, m, bs, hkv;
    int64_t kcode, vcode, gam, scl, zer, rho, sig, bytes; /* offsets, total */
} orc_layout;

static orc_layout orc_make_layout(int d, int kb, int vb, int m, int bs, int hkv) {
    orc_layout L;
    L.d = d; L.kb = kb; L.vb = vb; L.m = m; L.bs = bs; L.hkv = hkv;
    int64_t off = 0;
    L.kcode = off; off += (int64_t)bs * d * kb / 8;
    L.vcode = off; off += (int64_t)bs * d * vb / 8;
    L.gam = off; off += 2LL * bs;
    L.scl = off; off += 2LL * bs;
    L.zer = off; off += 2LL * bs;
    if (m > 0) {
        L.rho = off; off += 2LL * bs;
        L.sig = off; off += (int64_t)bs * m / 8;
    } else {
        L.rho = L.sig = -1;
    }
    L.bytes = (off + 15) / 16 * 16;
    return L;
}

ORC_API int64_t orc_page_bytes(int d, int kb, int vb, int m, int bs) {
    return orc_make_layout(d, kb, vb, m, bs, 1).bytes;
}

static void orc_put_bits(uint8_t* row, int64_t bitpos, int nbits, unsigned v) {
    for (int k = 0; k < nbits; ++k) {
        int64_t p = bitpos + k;
        uint8_t mask = (uint8_t)(1u << (p % 8));
        if ((v >> k) & 1u) row[p / 8] |= mask;
        else row[p / 8] &= (uint8_t)~mask;
    }
}

static unsigned orc_get_bits(const uint8_t* row, int64_t bitpos, int nbits) {
    unsigned v = 0;
    for (int k = 0; k < nbits; ++k) {
        int64_t p = bitpos + k;
        v |= (unsigned)((row[p / 8] >> (p % 8)) & 1u) << k;
    }
    return v;
}

static void orc_put_f16(uint8_t* p, double x) {
    uint16_t h = orc_fp16_bits(x);
    p[0] = (uint8_t)(h & 0xFF);
    p[1] = (uint8_t)(h >> 8);
}

static double orc_get_f16(const uint8_t* p) {
    return orc_fp16_value((uint16_t)(p[0] | (p[1] << 8)));
}

/* ------------------------------------------------------------------------ */
/* Encode one vector.                                                         */
/* ------------------------------------------------------------------------ */

/* Key: split, rotate, nearest centroid, QJL sketch.
 *   gamma = ||k||  [P1 1. Split; P3 step 1]; u = k/gamma; u_rot = R u.
 *   (The norm of k equals the norm of R k, so taking it before the rotation as
 *   [P3] does, or after as [P4 Step 2] does, is the same number.)
 *   idx_j = #{t_i < u_rot[j]}: the nearest centroid, exact ties to the lower
 *   index [P2 quantization function: argmin over the codebook].
 *   QJL: r = u_rot - C[idx] in the rotated unit frame, rho = ||r||,
 *   sigma_i = [(S r)_i >= 0]  [P3 "Optional 1-bit QJL residual"].
 * A zero key (gamma = 0) takes u = 0: every code is 2^(b-1) - 1 (the count of
 * negative boundaries), rho = 0, every sigma bit 1.  [P4 Step 2] adds 1e-8 to
 * the norm; that is dropped.
 * Outputs: *gamma, idx[d], *rho, sig[m] (0/1). */
ORC_API void orc_encode_key_vector(int d, int bits, const double* C, const double* T,
                                   const double* s, int m, const double* S,
                                   const double* k, double* gamma, int* idx,
                                   double* rho, int* sig) {
    const int n = 1 << bits;
    double g2 = 0.0;
    for (int j = 0; j < d; ++j) g2 += k[j] * k[j];
    double g = sqrt(g2);
    *gamma = g;
    double* u = (double*)malloc(sizeof(double) * d);
    double* ur = (double*)malloc(sizeof(double) * d);
    if (g == 0.0) {
        for (int j = 0; j < d; ++j) { idx[j] = n / 2 - 1; ur[j] = 0.0; u[j] = 0.0; }
        *rho = 0.0;
        for (int i = 0; i < m; ++i) sig[i] = 1;
        free(u); free(ur);
        return;
    }
    for (int j = 0; j < d; ++j) u[j] = k[j] / g;
    orc_rotate(d, s, u, ur);
    for (int j = 0; j < d; ++j) {
        int c = 0;
        for (int i = 0; i < n - 1; ++i) if (T[i] < ur[j]) ++c;
        idx[j] = c;
    }
    if (m > 0) {
        double r2 = 0.0;
        for (int j = 0; j < d; ++j) { u[j] = ur[j] - C[idx[j]]; r2 += u[j] * u[j]; }
        *rho = sqrt(r2);
        for (int i = 0; i < m; ++i) {
            double a = 0.0;
            for (int j = 0; j < d; ++j) a += S[(int64_t)i * d + j] * u[j];
            sig[i] = (a >= 0.0) ? 1 : 0;
        }
    } else {
        *rho = 0.0;
    }
    free(u); free(ur);
}

/* Value: rotate, then per-token asymmetric min-max codes in the rotated frame
 * [P4 Step 3]: scale = (max - min)/(2^b - 1), q = round((v - min)/scale) with
 * ties to even (torch's round), clamped to [0, 2^b - 1].  The codes use the
 * working-precision scale and min; the cache stores them as fp16.  If max ==
 * min the scale is 0 and every code is 0.  Outputs: *scale, *zero, q[d]. */
ORC_API void orc_encode_value_vector(int d, int bits, const double* s, const double* v,
                                     double* scale, double* zero, int* q) {
    const int qmax = (1 << bits) - 1;
    double* vr = (double*)malloc(sizeof(double) * d);
    orc_rotate(d, s, v, vr);
    double mn = vr[0], mx = vr[0];
    for (int j = 1; j < d; ++j) { if (vr[j] < mn) mn = vr[j]; if (vr[j] > mx) mx = vr[j]; }
    double sc = (mx - mn) / qmax;
    *scale = sc;
    *zero = mn;
    for (int j = 0; j < d; ++j) {
        if (sc == 0.0) { q[j] = 0; continue; }
        double x = nearbyint((vr[j] - mn) / sc);
        if (x < 0) x = 0;
        if (x > qmax) x = qmax;
        q[j] = (int)x;
    }
    free(vr);
}

/* ------------------------------------------------------------------------ */
/* Encode a batch of tokens into the paged cache.                            */
/* K, V: [T, hkv, d] float64 (the caller widens its input dtype exactly).    */
/* slot_mapping[t] = block * bs + offset; a negative slot skips the token;   */
/* a slot past the pool sets ORC_FLAG_BAD_SLOT and skips it.                 */
/* Returns the OR of the status bits.                                        */
/* ------------------------------------------------------------------------ */

ORC_API int orc_encode(int d, int kb, int vb, int m, int bs, int hkv, int64_t num_blocks,
                       const double* Ck, const double* Tk, const double* s, const double* S,
                       const double* K, const double* V, int64_t T, const int64_t* slot_mapping,
                       uint8_t* pool) {
    orc_layout L = orc_make_layout(d, kb, vb, m, bs, hkv);
    int status = 0;
    int64_t kr = (int64_t)d * kb / 8, vr = (int64_t)d * vb / 8, sr = m / 8;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : status)
    for (int64_t th = 0; th < T * hkv; ++th) {
        int64_t t = th / hkv;
        int h = (int)(th % hkv);
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * bs) { status |= ORC_FLAG_BAD_SLOT; continue; }
        int64_t blk = slot / bs;
        int off = (int)(slot % bs);
        uint8_t* page = pool + (blk * hkv + h) * L.bytes;
        const double* k = K + th * d;
        const double* v = V + th * d;
        int finite = 1;
        for (int j = 0; j < d; ++j) if (!isfinite(k[j]) || !isfinite(v[j])) finite = 0;
        if (!finite) { status |= ORC_FLAG_NONFINITE; }
        int* idx = (int*)malloc(sizeof(int) * d);
        int* q = (int*)malloc(sizeof(int) * d);
        int* sig = (int*)malloc(sizeof(int) * (m > 0 ? m : 1));
        double g, rho, sc, zr;
        orc_encode_key_vector(d, kb, Ck, Tk, s, m, S, k, &g, idx, &rho, sig);
        orc_encode_value_vector(d, vb, s, v, &sc, &zr, q);
        uint8_t* krow = page + L.kcode + off * kr;
        uint8_t* vrow = page + L.vcode + off * vr;
        for (int j = 0; j < d; ++j) orc_put_bits(krow, (int64_t)j * kb, kb, (unsigned)idx[j]);
        for (int j = 0; j < d; ++j) orc_put_bits(vrow, (int64_t)j * vb, vb, (unsigned)q[j]);
        orc_put_f16(page + L.gam + 2 * off, g);
        orc_put_f16(page + L.scl + 2 * off, sc);
        orc_put_f16(page + L.zer + 2 * off, zr);
        if (isinf(orc_fp16_round(g)) || isinf(orc_fp16_round(sc)) || isinf(orc_fp16_round(zr)))
            status |= ORC_FLAG_OVERFLOW;
        if (m > 0) {
            orc_put_f16(page + L.rho + 2 * off, rho);
            uint8_t* srow = page + L.sig + off * sr;
            for (int i = 0; i < m; ++i) orc_put_bits(srow, i, 1, (unsigned)sig[i]);
        }
        free(idx); free(q); free(sig);
    }
    return status;
}

/* Read back one token slot of one page: codes, fp16 fields widened. */
ORC_API void orc_unpack_slot(int d, int kb, int vb, int m, int bs, const uint8_t* page, int off,
                             int* kidx, int* vq, double* gamma, double* scale, double* zero,
                             double* rho, int* sig) {
    orc_layout L = orc_make_layout(d, kb, vb, m, bs, 1);
    int64_t kr = (int64_t)d * kb / 8, vr = (int64_t)d * vb / 8, sr = m / 8;
    const uint8_t* krow = page + L.kcode + off * kr;
    const uint8_t* vrow = page + L.vcode + off * vr;
    for (int j = 0; j < d; ++j) kidx[j] = (int)orc_get_bits(krow, (int64_t)j * kb, kb);
    for (int j = 0; j < d; ++j) vq[j] = (int)orc_get_bits(vrow, (int64_t)j * vb, vb);
    *gamma = orc_get_f16(page + L.gam + 2 * off);
    *scale = orc_get_f16(page + L.scl + 2 * off);
    *zero = orc_get_f16(page + L.zer + 2 * off);
    if (m > 0) {
        *rho = orc_get_f16(page + L.rho + 2 * off);
        const uint8_t* srow = page + L.sig + off * sr;
        for (int i = 0; i < m; ++i) sig[i] = (int)orc_get_bits(srow, i, 1);
    } else {
        *rho = 0.0;
    }
}

/* ------------------------------------------------------------------------ */
/* Decode attention over the compressed cache, plain definition.             */
/* For each sequence b and query head hq (KV head h = hq / (Hq/hkv)), over   */
/* the tokens t < lens[b] (page block_table[b][t / bs], slot t % bs):        */
/*   K^_t = gamma_t R^T C[idx_t]             (original frame)                */
/*   V^_t = R^T (scale_t * q_t + zero_t)     (original frame)                */
/*   logit_t = sm_scale * ( <q, K^_t>                                         */
/*             + gamma_t sqrt(pi/2)/m rho_t <S R q, 2 sigma_t - 1> )  [m > 0] */
/*   out = sum_t softmax(logit)_t V^_t                                        */
/* [P2 attention under quantized KV: softmax(Q K^T / sqrt(d_h)) V]; the QJL  */
/* term is the unbiased estimate of gamma <R q, r> [P3 "Optional 1-bit QJL   */
/* residual", step 8].  gamma, scale, zero, rho are the stored fp16 values.  */
/* q: [B, Hq, d]; out: [B, Hq, d]; a sequence with lens[b] == 0 gets zeros.  */
/* A block id outside [0, num_blocks) sets ORC_FLAG_BAD_SLOT and that page's */
/* tokens are left out.  Returns the OR of the status bits.                  */
/* ------------------------------------------------------------------------ */

ORC_API int orc_decode(int d, int kb, int vb, int m, int bs, int hkv, int64_t num_blocks,
                       const double* Ck, const double* s, const double* S, const uint8_t* pool,
                       const double* Q, int B, int hq, const int32_t* block_table,
                       int max_blocks, const int32_t* lens, double sm_scale, double* out) {
    orc_layout L = orc_make_layout(d, kb, vb, m, bs, hkv);
    const int G = hq / hkv;
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int bh = 0; bh < B * hkv; ++bh) {
        int b = bh / hkv, h = bh % hkv;
        int len = lens[b];
        if (len <= 0) {
            for (int g = 0; g < G; ++g) {
                double* o = out + ((int64_t)b * hq + (int64_t)h * G + g) * d;
                for (int j = 0; j < d; ++j) o[j] = 0.0;
            }
            continue;
        }
        double* Kh = (double*)calloc((size_t)len * d, sizeof(double));
        double* Vh = (double*)calloc((size_t)len * d, sizeof(double));
        double* qjl = (double*)calloc((size_t)len * (m > 0 ? m : 1), sizeof(double));
        double* gam = (double*)calloc((size_t)len, sizeof(double));
        double* rh = (double*)calloc((size_t)len, sizeof(double));
        char* valid = (char*)calloc((size_t)len, 1);
        int* kidx = (int*)malloc(sizeof(int) * d);
        int* vq = (int*)malloc(sizeof(int) * d);
        int* sig = (int*)malloc(sizeof(int) * (m > 0 ? m : 1));
        double* tmp = (double*)malloc(sizeof(double) * d);
        for (int t = 0; t < len; ++t) {
            int32_t blk = block_table[(int64_t)b * max_blocks + t / bs];
            if (blk < 0 || blk >= num_blocks) { status |= ORC_FLAG_BAD_SLOT; continue; }
            valid[t] = 1;
            const uint8_t* page = pool + ((int64_t)blk * hkv + h) * L.bytes;
            double g, sc, zr, rho;
            orc_unpack_slot(d, kb, vb, m, bs, page, t % bs, kidx, vq, &g, &sc, &zr, &rho, sig);
            for (int j = 0; j < d; ++j) tmp[j] = Ck[kidx[j]];
            orc_rotate_inverse(d, s, tmp, Kh + (int64_t)t * d);
            for (int j = 0; j < d; ++j) Kh[(int64_t)t * d + j] *= g;
            for (int j = 0; j < d; ++j) tmp[j] = sc * vq[j] + zr;
            orc_rotate_inverse(d, s, tmp, Vh + (int64_t)t * d);
            gam[t] = g;
            rh[t] = rho;
            for (int i = 0; i < m; ++i) qjl[(int64_t)t * m + i] = sig[i] ? 1.0 : -1.0;
        }
        double* logit = (double*)malloc(sizeof(double) * len);
        double* qr = (double*)malloc(sizeof(double) * d);
        double* sq = (double*)malloc(sizeof(double) * (m > 0 ? m : 1));
        for (int g = 0; g < G; ++g) {
            int64_t qh = (int64_t)b * hq + (int64_t)h * G + g;
            const double* qv = Q + qh * d;
            if (m > 0) {
                orc_rotate(d, s, qv, qr);
                for (int i = 0; i < m; ++i) {
                    double a = 0.0;
                    for (int j = 0; j < d; ++j) a += S[(int64_t)i * d + j] * qr[j];
                    sq[i] = a;
                }
            }
            double mx = -INFINITY;
            for (int t = 0; t < len; ++t) {
                if (!valid[t]) continue;
                double a = 0.0;
                for (int j = 0; j < d; ++j) a += qv[j] * Kh[(int64_t)t * d + j];
                if (m > 0) {
                    double c = 0.0;
                    for (int i = 0; i < m; ++i) c += sq[i] * qjl[(int64_t)t * m + i];
                    a += gam[t] * sqrt(M_PI / 2.0) / m * rh[t] * c;
                }
                logit[t] = sm_scale * a;
                if (logit[t] > mx) mx = logit[t];
            }
            double* o = out + qh * d;
            for (int j = 0; j < d; ++j) o[j] = 0.0;
            if (mx == -INFINITY) continue;
            double den = 0.0;
            for (int t = 0; t < len; ++t) {
                if (!valid[t]) continue;
                double p = exp(logit[t] - mx);
                den += p;
                for (int j = 0; j < d; ++j) o[j] += p * Vh[(int64_t)t * d + j];
            }
            for (int j = 0; j < d; ++j) o[j] /= den;
        }
        free(logit); free(qr); free(sq);
        free(Kh); free(Vh); free(qjl); free(gam); free(rh); free(valid);
        free(kidx); free(vq); free(sig); free(tmp);
    }
    return status;
}

/* ======================================================================== */
/* OCTOPUS: triplet key codec with an octahedral direction code             */
/* [P3 key contribution "Octahedral triplet direction quantizer with norm   */
/*  marginals"; methodology steps 1-7; bit split (b+1, b-1)].               */
/*                                                                          */
/* The rotated unit key u is cut into ntri = ceil(d/3) triplets t_i (the    */
/* last one padded with zeros).  Each triplet is its norm rho_i and its     */
/* direction n_i on S^2; the direction is mapped to the square by the       */
/* octahedral map, (xi, eta) = Oct(n_i).  xi and eta take (b+1)-bit codes   */
/* from one Lloyd-Max codebook fitted to the marginal of xi, rho takes a    */
/* (b-1)-bit code from a Lloyd-Max codebook fitted to the marginal of the   */
/* norm of three coordinates of a uniform point on S^{d-1}.  The page names */
/* the map and the "3x3 joint rounding" without formulas; the readings      */
/* taken are stated at each function.                                       */
/* ======================================================================== */

static double orc_sgn(double x) { return x < 0.0 ? -1.0 : 1.0; }

/* Octahedral map: p = n / (|n_x| + |n_y| + |n_z|); for n_z >= 0 the upper
 * half of the octahedron projects straight down, (xi, eta) = (p_x, p_y);
 * for n_z < 0 the lower half is folded out over the square's corners,
 * (xi, eta) = ((1 - |p_y|) sgn p_x, (1 - |p_x|) sgn p_y), sgn(0) = +1.
 * (The standard octahedral parametrisation of the sphere.) */
ORC_API void orc_oct_map(const double* n, double* xi, double* eta) {
    double l1 = fabs(n[0]) + fabs(n[1]) + fabs(n[2]);
    double px = n[0] / l1, py = n[1] / l1;
    if (n[2] >= 0.0) {
        *xi = px;
        *eta = py;
    } else {
        *xi = (1.0 - fabs(py)) * orc_sgn(px);
        *eta = (1.0 - fabs(px)) * orc_sgn(py);
    }
}

/* The octahedron point of (xi, eta): z = 1 - |xi| - |eta|; where z < 0 the
 * fold is undone, (x, y) = ((1 - |eta|) sgn xi, (1 - |xi|) sgn eta). */
static void orc_oct_point(double xi, double eta, double* p) {
    double z = 1.0 - fabs(xi) - fabs(eta);
    if (z >= 0.0) {
        p[0] = xi;
        p[1] = eta;
    } else {
        p[0] = (1.0 - fabs(eta)) * orc_sgn(xi);
        p[1] = (1.0 - fabs(xi)) * orc_sgn(eta);
    }
    p[2] = z;
}

/* Inverse map: the unit direction of the octahedron point. */
ORC_API void orc_oct_inverse(double xi, double eta, double* n) {
    double p[3];
    orc_oct_point(xi, eta, p);
    double r = sqrt(p[0] * p[0] + p[1] * p[1] + p[2] * p[2]);
    n[0] = p[0] / r;
    n[1] = p[1] / r;
    n[2] = p[2] / r;
}

/* Density of (xi, eta) in [-1,1]^2 for n uniform on S^2.  Radial projection
 * of an octahedron face (normal (1,1,1)/sqrt 3 in the first octant, area
 * element sqrt(3) dxi deta over the square) onto the sphere has solid angle
 * element (p . N) dA / |p|^3 = dxi deta / |p|^3, and the fold of the lower
 * half is area preserving, so f = 1 / (4 pi |p|^3) with p the octahedron
 * point of (xi, eta). */
ORC_API double orc_oct_density(double xi, double eta) {
    double p[3];
    orc_oct_point(xi, eta, p);
    double r2 = p[0] * p[0] + p[1] * p[1] + p[2] * p[2];
    return 1.0 / (4.0 * M_PI * r2 * sqrt(r2));
}

/* composite Gauss-Legendre of g over [a, b] in pieces no wider than w */
static double orc_gl_integrate(double (*g)(double, const void*), const void* ctx, double a, double b, double w) {
    orc_gl_init();
    if (b <= a) return 0.0;
    int pieces = (int)ceil((b - a) / w);
    if (pieces < 1) pieces = 1;
    double h = (b - a) / pieces, sum = 0.0;
    for (int p = 0; p < pieces; ++p) {
        double mid = a + (p + 0.5) * h, part = 0.0;
        for (int i = 0; i < ORC_GL_N; ++i) part += orc_gl_w[i] * g(mid + 0.5 * h * orc_gl_x[i], ctx);
        sum += 0.5 * h * part;
    }
    return sum;
}

static double orc_oct_density_eta(double eta, const void* ctx) {
    return orc_oct_density(*(const double*)ctx, eta);
}

/* Marginal of xi: int f(xi, eta) d eta over [-1, 1], in the four pieces on
 * which the integrand is smooth (split at eta = 0 and |eta| = 1 - |xi|). */
ORC_API double orc_oct_marginal(double xi) {
    if (xi < -1.0 || xi > 1.0) return 0.0;
    double e = 1.0 - fabs(xi);
    return orc_gl_integrate(orc_oct_density_eta, &xi, -1.0, -e, 0.05) +
           orc_gl_integrate(orc_oct_density_eta, &xi, -e, 0.0, 0.05) +
           orc_gl_integrate(orc_oct_density_eta, &xi, 0.0, e, 0.05) +
           orc_gl_integrate(orc_oct_density_eta, &xi, e, 1.0, 0.05);
}

/* Norm of three coordinates of a uniform point on S^{d-1}: rho^2 follows
 * Beta(3/2, (d-3)/2) (the squared coordinates of a uniform point are a
 * Dirichlet(1/2, ..., 1/2) vector), so
 * f(rho) = 2 rho^2 (1 - rho^2)^((d-5)/2) / B(3/2, (d-3)/2) on [0, 1]. */
ORC_API double orc_rho_density(int d, double rho) {
    if (rho <= 0.0 || rho >= 1.0) return 0.0;
    double lb = lgamma(1.5) + lgamma((d - 3) / 2.0) - lgamma(d / 2.0);
    return 2.0 * rho * rho * pow(1.0 - rho * rho, (d - 5) / 2.0) * exp(-lb);
}

typedef struct { int kind, d, moment; } orc_dens_ctx;

static double orc_dens_eval(double x, const void* vctx) {
    const orc_dens_ctx* c = (const orc_dens_ctx*)vctx;
    double f = (c->kind == 0) ? orc_oct_marginal(x) : orc_rho_density(c->d, x);
    return c->moment ? x * f : f;
}

/* mass (moment = 0) or first moment (1) of density `kind` over [a, b]; the
 * xi marginal has a kink at 0, where cells are split */
static double orc_dens_integral(int kind, int d, int moment, double a, double b) {
    orc_dens_ctx c = {kind, d, moment};
    double w = (kind == 0) ? 0.05 : 0.01;
    if (kind == 0 && a < 0.0 && b > 0.0)
        return orc_gl_integrate(orc_dens_eval, &c, a, 0.0, w) + orc_gl_integrate(orc_dens_eval, &c, 0.0, b, w);
    return orc_gl_integrate(orc_dens_eval, &c, a, b, w);
}

ORC_API double orc_oct_cell_mass(int kind, int d, double a, double b) {
    return orc_dens_integral(kind, d, 0, a, b);
}

/* Lloyd-Max on density `kind` (0: the xi marginal on [-1, 1]; 1: the triplet
 * norm on [0, 1] for dimension d), the same iteration as orc_lloyd_max:
 * boundaries at midpoints, centroids the cells' conditional means, from
 * evenly spaced starting levels (over [-1, 1] for xi, over [0, 4 sqrt(3/d)]
 * for rho), until max |change| < tol or max_iter passes.  Writes n = 2^bits
 * centroids and n - 1 boundaries; returns the passes taken. */
ORC_API int orc_lloyd_density(int kind, int d, int bits, double tol, int max_iter, double* c, double* t) {
    const int n = 1 << bits;
    const double lo = (kind == 0) ? -1.0 : 0.0, hi = 1.0;
    const double span = (kind == 0) ? 2.0 : 4.0 * sqrt(3.0 / d);
    for (int i = 0; i < n; ++i) c[i] = lo + (i + 0.5) * span / n;
    int it = 0;
    for (; it < max_iter; ++it) {
        for (int i = 0; i + 1 < n; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
        double delta = 0.0;
        for (int i = 0; i < n; ++i) {
            double a = (i == 0) ? lo : t[i - 1];
            double b = (i == n - 1) ? hi : t[i];
            double mass = orc_dens_integral(kind, d, 0, a, b);
            double cn = (mass > 0.0) ? orc_dens_integral(kind, d, 1, a, b) / mass : 0.5 * (a + b);
            double dd = fabs(cn - c[i]);
            if (dd > delta) delta = dd;
            c[i] = cn;
        }
        if (delta < tol) { ++it; break; }
    }
    for (int i = 0; i + 1 < n; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
    return it;
}

/* nearest level: #{boundaries < x}, ties to the lower index */
static int orc_nearest(const double* t, int n, double x) {
    int k = 0;
    for (int i = 0; i + 1 < n; ++i) k += (t[i] < x) ? 1 : 0;
    return k;
}

/* One triplet [P3 methodology steps 3-5].  rho = ||t||, n = t / rho
 * ((0, 0, 1) when rho = 0).  Norm code: the nearest level of C_rho.
 * Direction codes, the "3 x 3 joint rounding": with a, b the nearest levels
 * of C_xi to xi and to eta, the candidates are a' in {a-1, a, a+1} and
 * b' in {b-1, b, b+1} (inside the codebook); the pair whose direction
 * n^ = Oct^{-1}(C_xi[a'], C_xi[b']) has the largest <n, n^> is kept (for the
 * fixed rho^ this is the smallest ||t - rho^ n^||), ties to the first pair in
 * (a', b') order.  Returns <n, n^> of the pair kept. */
ORC_API double orc_oct_encode_triplet(const double* tr, const double* Cxi, const double* Txi, int nxi,
                                      const double* Crho, const double* Trho, int nrho,
                                      int* ixi, int* ieta, int* irho) {
    double rho = sqrt(tr[0] * tr[0] + tr[1] * tr[1] + tr[2] * tr[2]);
    double n[3] = {0.0, 0.0, 1.0};
    if (rho > 0.0) {
        n[0] = tr[0] / rho;
        n[1] = tr[1] / rho;
        n[2] = tr[2] / rho;
    }
    *irho = orc_nearest(Trho, nrho, rho);
    double xi, eta;
    orc_oct_map(n, &xi, &eta);
    int a = orc_nearest(Txi, nxi, xi), b = orc_nearest(Txi, nxi, eta);
    double best = -INFINITY;
    int ba = a, bb = b;
    for (int da = -1; da <= 1; ++da) {
        int aa = a + da;
        if (aa < 0 || aa >= nxi) continue;
        for (int db = -1; db <= 1; ++db) {
            int bq = b + db;
            if (bq < 0 || bq >= nxi) continue;
            double nh[3];
            orc_oct_inverse(Cxi[aa], Cxi[bq], nh);
            double sc = n[0] * nh[0] + n[1] * nh[1] + n[2] * nh[2];
            if (sc > best) {
                best = sc;
                ba = aa;
                bb = bq;
            }
        }
    }
    *ixi = ba;
    *ieta = bb;
    return best;
}

/* OCTOPUS page: per block of bs slots of one KV head,
 *   key rows   bs rows of KR bytes, KR = 4 ceil(ntri (3b + 1) / 32); triplet i's
 *              fields at bit i (3b + 1) of the row: xi code (b + 1 bits), eta
 *              code (b + 1 bits), rho code (b - 1 bits), LSB first
 *   value codes, gamma, scale, zero as in the page above (no QJL),
 * then zero padding to a multiple of 16 bytes.  The bit budget per triplet,
 * 2 (b + 1) + (b - 1), is the page's B_tri = 2 b_dir + b_nrm with
 * (b_dir, b_nrm) = (b + 1, b - 1) [P3 "MSE-optimal non-uniform bit allocation"]. */
static int64_t orc_oct_key_row(int d, int b) {
    int ntri = (d + 2) / 3;
    return 4LL * ((ntri * (3 * b + 1) + 31) / 32);
}

ORC_API int64_t orc_oct_page_bytes(int d, int b, int vb, int bs) {
    int64_t off = (int64_t)bs * orc_oct_key_row(d, b);
    off += (int64_t)bs * d * vb / 8;
    off += 6LL * bs;
    return (off + 15) / 16 * 16;
}

/* Key vector [P3 methodology steps 1-6]: gamma = ||k||, u = R (k / gamma),
 * triplets of u (zeros past d), each coded by orc_oct_encode_triplet.  A zero
 * key takes u = 0 (every triplet rho = 0, n = (0, 0, 1)). */
ORC_API void orc_oct_encode_key_vector(int d, const double* Cxi, const double* Txi, int nxi,
                                       const double* Crho, const double* Trho, int nrho, const double* s,
                                       const double* k, double* gamma, int* ixi, int* ieta, int* irho) {
    double g = 0.0;
    for (int j = 0; j < d; ++j) g += k[j] * k[j];
    g = sqrt(g);
    *gamma = g;
    double* u = (double*)calloc((size_t)d, sizeof(double));
    double* ur = (double*)calloc((size_t)d + 3, sizeof(double));
    if (g > 0.0)
        for (int j = 0; j < d; ++j) u[j] = k[j] / g;
    orc_rotate(d, s, u, ur);
    for (int i = 0; i < (d + 2) / 3; ++i) orc_oct_encode_triplet(ur + 3 * i, Cxi, Txi, nxi, Crho, Trho, nrho,
                                                                ixi + i, ieta + i, irho + i);
    free(u);
    free(ur);
}

/* Encode tokens into OCTOPUS pages: keys as above, values as orc_encode does.
 * Same slot and status conventions as orc_encode.  b: the page's b (xi codes
 * b + 1 bits, rho codes b - 1 bits; b >= 2). */
ORC_API int orc_oct_encode(int d, int b, int vb, int bs, int hkv, int64_t num_blocks,
                           const double* Cxi, const double* Txi, const double* Crho, const double* Trho,
                           const double* s, const double* K, const double* V, int64_t T,
                           const int64_t* slots, uint8_t* pool) {
    const int ntri = (d + 2) / 3, nxi = 1 << (b + 1), nrho = 1 << (b - 1);
    const int64_t KR = orc_oct_key_row(d, b), VR = (int64_t)d * vb / 8;
    const int64_t PB = orc_oct_page_bytes(d, b, vb, bs);
    const int64_t vcode = (int64_t)bs * KR, gam = vcode + (int64_t)bs * VR, scl = gam + 2 * bs, zer = scl + 2 * bs;
    int status = 0;
#pragma omp parallel for schedule(static) reduction(| : status)
    for (int64_t th = 0; th < T * hkv; ++th) {
        int64_t t = th / hkv;
        int h = (int)(th % hkv);
        int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * bs) { status |= ORC_FLAG_BAD_SLOT; continue; }
        const double* k = K + th * d;
        const double* v = V + th * d;
        int finite = 1;
        for (int j = 0; j < d; ++j) finite &= isfinite(k[j]) && isfinite(v[j]);
        if (!finite) status |= ORC_FLAG_NONFINITE;
        int64_t blk = slot / bs, off = slot % bs;
        uint8_t* page = pool + (blk * hkv + h) * PB;
        int* ixi = (int*)malloc(sizeof(int) * ntri);
        int* ieta = (int*)malloc(sizeof(int) * ntri);
        int* irho = (int*)malloc(sizeof(int) * ntri);
        int* vq = (int*)malloc(sizeof(int) * d);
        double gamma, scale, zero;
        orc_oct_encode_key_vector(d, Cxi, Txi, nxi, Crho, Trho, nrho, s, k, &gamma, ixi, ieta, irho);
        orc_encode_value_vector(d, vb, s, v, &scale, &zero, vq);
        uint8_t* krow = page + off * KR;
        memset(krow, 0, (size_t)KR);
        for (int i = 0; i < ntri; ++i) {
            int64_t p = (int64_t)i * (3 * b + 1);
            orc_put_bits(krow, p, b + 1, (unsigned)ixi[i]);
            orc_put_bits(krow, p + b + 1, b + 1, (unsigned)ieta[i]);
            orc_put_bits(krow, p + 2 * (b + 1), b - 1, (unsigned)irho[i]);
        }
        uint8_t* vrow = page + vcode + off * VR;
        for (int j = 0; j < d; ++j) orc_put_bits(vrow, (int64_t)j * vb, vb, (unsigned)vq[j]);
        orc_put_f16(page + gam + 2 * off, gamma);
        orc_put_f16(page + scl + 2 * off, scale);
        orc_put_f16(page + zer + 2 * off, zero);
        if (finite && (isinf(orc_fp16_round(gamma)) || isinf(orc_fp16_round(scale)) || isinf(orc_fp16_round(zero))))
            status |= ORC_FLAG_OVERFLOW;
        free(ixi); free(ieta); free(irho); free(vq);
    }
    return status;
}

/* Read back one OCTOPUS slot: codes and fp16 fields widened. */
ORC_API void orc_oct_unpack_slot(int d, int b, int vb, int bs, const uint8_t* page, int off, int* ixi,
                                 int* ieta, int* irho, int* vq, double* gamma, double* scale, double* zero) {
    const int ntri = (d + 2) / 3;
    const int64_t KR = orc_oct_key_row(d, b), VR = (int64_t)d * vb / 8;
    const int64_t vcode = (int64_t)bs * KR, gam = vcode + (int64_t)bs * VR, scl = gam + 2 * bs, zer = scl + 2 * bs;
    const uint8_t* krow = page + off * KR;
    for (int i = 0; i < ntri; ++i) {
        int64_t p = (int64_t)i * (3 * b + 1);
        ixi[i] = (int)orc_get_bits(krow, p, b + 1);
        ieta[i] = (int)orc_get_bits(krow, p + b + 1, b + 1);
        irho[i] = (int)orc_get_bits(krow, p + 2 * (b + 1), b - 1);
    }
    const uint8_t* vrow = page + vcode + off * VR;
    for (int j = 0; j < d; ++j) vq[j] = (int)orc_get_bits(vrow, (int64_t)j * vb, vb);
    *gamma = orc_get_f16(page + gam + 2 * off);
    *scale = orc_get_f16(page + scl + 2 * off);
    *zero = orc_get_f16(page + zer + 2 * off);
}

/* The rotated unit key of one slot [P3 methodology step 7: triplets rebuilt
 * from the codes]: u^[3i + c] = C_rho[irho_i] n^_i[c] with
 * n^_i = Oct^{-1}(C_xi[ixi_i], C_xi[ieta_i]), for 3i + c < d. */
static void orc_oct_direction(int d, const double* Cxi, const double* Crho, const int* ixi, const int* ieta,
                              const int* irho, double* u) {
    for (int i = 0; i < (d + 2) / 3; ++i) {
        double nh[3];
        orc_oct_inverse(Cxi[ixi[i]], Cxi[ieta[i]], nh);
        for (int c = 0; c < 3; ++c)
            if (3 * i + c < d) u[3 * i + c] = Crho[irho[i]] * nh[c];
    }
}

/* Decode attention over OCTOPUS pages, plain definition (as orc_decode):
 *   K^_t = gamma_t R^T u^_t, V^_t = R^T (scale_t q_t + zero_t),
 *   out = softmax_t(sm_scale <q, K^_t>) V^_t over t < lens[b]. */
ORC_API int orc_oct_decode(int d, int b, int vb, int bs, int hkv, int64_t num_blocks, const double* Cxi,
                           const double* Crho, const double* s, const uint8_t* pool, const double* Q, int B,
                           int hq, const int32_t* block_table, int max_blocks, const int32_t* lens,
                           double sm_scale, double* out) {
    const int G = hq / hkv, ntri = (d + 2) / 3;
    const int64_t PB = orc_oct_page_bytes(d, b, vb, bs);
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int bh = 0; bh < B * hkv; ++bh) {
        int bi = bh / hkv, h = bh % hkv;
        int len = lens[bi];
        for (int g = 0; g < G; ++g) {
            double* o = out + ((int64_t)bi * hq + (int64_t)h * G + g) * d;
            for (int j = 0; j < d; ++j) o[j] = 0.0;
        }
        if (len <= 0) continue;
        double* Kh = (double*)calloc((size_t)len * d, sizeof(double));
        double* Vh = (double*)calloc((size_t)len * d, sizeof(double));
        char* valid = (char*)calloc((size_t)len, 1);
        int* ixi = (int*)malloc(sizeof(int) * ntri);
        int* ieta = (int*)malloc(sizeof(int) * ntri);
        int* irho = (int*)malloc(sizeof(int) * ntri);
        int* vq = (int*)malloc(sizeof(int) * d);
        double* tmp = (double*)malloc(sizeof(double) * d);
        for (int t = 0; t < len; ++t) {
            int32_t blk = block_table[(int64_t)bi * max_blocks + t / bs];
            if (blk < 0 || blk >= num_blocks) { status |= ORC_FLAG_BAD_SLOT; continue; }
            valid[t] = 1;
            const uint8_t* page = pool + ((int64_t)blk * hkv + h) * PB;
            double g, sc, zr;
            orc_oct_unpack_slot(d, b, vb, bs, page, t % bs, ixi, ieta, irho, vq, &g, &sc, &zr);
            orc_oct_direction(d, Cxi, Crho, ixi, ieta, irho, tmp);
            orc_rotate_inverse(d, s, tmp, Kh + (int64_t)t * d);
            for (int j = 0; j < d; ++j) Kh[(int64_t)t * d + j] *= g;
            for (int j = 0; j < d; ++j) tmp[j] = sc * vq[j] + zr;
            orc_rotate_inverse(d, s, tmp, Vh + (int64_t)t * d);
        }
        double* logit = (double*)malloc(sizeof(double) * len);
        for (int g = 0; g < G; ++g) {
            int64_t qh = (int64_t)bi * hq + (int64_t)h * G + g;
            const double* qv = Q + qh * d;
            double mx = -INFINITY;
            for (int t = 0; t < len; ++t) {
                if (!valid[t]) continue;
                double a = 0.0;
                for (int j = 0; j < d; ++j) a += qv[j] * Kh[(int64_t)t * d + j];
                logit[t] = sm_scale * a;
                if (logit[t] > mx) mx = logit[t];
            }
            if (mx == -INFINITY) continue;
            double* o = out + qh * d;
            double den = 0.0;
            for (int t = 0; t < len; ++t) {
                if (!valid[t]) continue;
                double p = exp(logit[t] - mx);
                den += p;
                for (int j = 0; j < d; ++j) o[j] += p * Vh[(int64_t)t * d + j];
            }
            for (int j = 0; j < d; ++j) o[j] /= den;
        }
        free(logit);
        free(Kh); free(Vh); free(valid); free(ixi); free(ieta); free(irho); free(vq); free(tmp);
    }
    return status;
}
