/*
 * tq.h -- C ABI of the GB300 (sm_103a) online KV-cache compression library.
 *
 * The library compresses key/value vectors as they are produced during decode
 * and runs decode attention straight from the compressed, paged cache.
 *
 * Method, as the source pages state it (cited "page title -- section"):
 *  - Split each key into a norm and a direction, rotate the direction with a
 *    random sign flip followed by a Walsh-Hadamard transform, and store the
 *    index of the nearest codeword per coordinate.
 *      ["TurboQuant: KV Cache Vector Quantization" -- the three steps;
 *       "OCTOPUS ..." summary -- methodology steps 1-2]
 *  - The codebook is a per-coordinate Lloyd-Max quantizer for the marginal of
 *    the rotated direction.  ["OCTOPUS ..." -- key idea; glossary]
 *  - Values take per-token min-max codes in the rotated frame with an fp16
 *    scale and zero point.  [TurboQuant deep dive (cell-devlog) -- Step 3]
 *  - Optionally a 1-bit QJL sketch of the key residual, sign(S r), plus the
 *    residual norm, gives an unbiased correction to each logit.
 *      ["OCTOPUS ..." -- contribution "Optional 1-bit QJL residual"; step 8]
 *  - Attention is softmax(q K^T / sqrt(d_h)) V over the compressed cache
 *    ["TurboQuant: KV Cache Compression" (Bit-Axon) -- attention under
 *    quantized KV], computed in the rotated frame without reconstructing keys
 *    ["OCTOPUS ..." -- TL;DR, step 7; deep dive -- [RHT effect]: the rotation
 *    preserves inner products].
 *
 * Conventions
 *  - Every data pointer passed to an encode/decode call is a DEVICE pointer
 *    owned by the caller; the library never frees or reallocates it.  Host
 *    pointers are marked "host".  The one exception: q, k_new, v_new and out
 *    of the decode calls may also be page-locked host memory that the device
 *    reaches in place (tq_device_accessible).
 *  - Calls are asynchronous on the given CUDA stream (`stream` is a
 *    cudaStream_t; NULL is the legacy default stream).  Errors that the host
 *    can see are returned at once as a tq_status and nothing is launched.
 *  - Errors that only the device can see are OR-ed, as TQ_FLAG_* bits, into
 *    the int32 word at `dev_status` (a device pointer; may be NULL to ignore
 *    them).  Read it after synchronising.  Kernels never trap and never spin
 *    without a bound.
 *  - Tensor layouts are C-contiguous (row-major); sizes are element counts.
 *
 * Paged cache layout (bytes; d = head dim, kb/vb = key/value bits, m = QJL
 * rows, bs = block size in tokens).  One page holds one block of bs token
 * slots of one KV head; page (block n, KV head h) starts at byte
 * (n * num_kv_heads + h) * tq_page_bytes(...).  Sections, in order:
 *      key codes     bs rows of d*kb/8 bytes
 *      value codes   bs rows of d*vb/8 bytes
 *      gamma         bs binary16  (key norm)
 *      value scale   bs binary16
 *      value zero    bs binary16  (the rotated-frame minimum)
 *      rho           bs binary16  (QJL residual norm; only if m > 0)
 *      sigma         bs rows of m/8 bytes (QJL sign bits; only if m > 0)
 * then zero padding to a multiple of 16 bytes.  Inside a row, code j takes
 * bits [j*b, j*b + b) of the row read as a little-endian bit string (bit k is
 * bit k%8 of byte k/8).  Key code j is the index, in increasing order, of the
 * nearest centroid to rotated direction coordinate j (an exact tie goes to the
 * lower index).  Sigma bit i is 1 iff (S r)_i >= 0.
 * 4/4-bit keys/values take 134 bytes per token and KV head, 3/3-bit 102, and
 * 2/2-bit with m = 128 take 88.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define TQ_API
#else
#define TQ_API __attribute__((visibility("default")))
#endif

/* Host-visible result of every call. */
typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1, /* a NULL pointer, a negative size, a shape that does not fit */
    TQ_ERR_UNSUPPORTED = 2, /* valid in principle, not built (e.g. head dim != 128) */
    TQ_ERR_CUDA = 3,        /* a CUDA runtime call failed; tq_last_error() has the text */
    TQ_ERR_WORKSPACE = 4    /* the workspace passed to decode is too small */
} tq_status;

/* Device-detected conditions, OR-ed into *dev_status. */
#define TQ_FLAG_OVERFLOW 1  /* a norm, scale, zero or rho exceeded the fp16 range (stored as inf) */
#define TQ_FLAG_BAD_SLOT 2  /* a slot or block id outside the pool; that token/page was skipped */
#define TQ_FLAG_NONFINITE 4 /* a key or value held NaN or inf; its codes are unspecified */
#define TQ_FLAG_TIMEOUT 8   /* a bounded device wait gave up; the output is incomplete */
#define TQ_FLAG_INTERNAL 16 /* the kernel could not lay out its shared memory; no output was written */

/* Element type of K, V and q inputs. */
typedef enum { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;

/* ---------------------------------------------------------------------- */
/* Codebook                                                                */
/* ---------------------------------------------------------------------- */

/* Opaque, library-owned Lloyd-Max codebook for one (d, bits). */
typedef struct tq_codebook tq_codebook;

/* Fit the per-coordinate Lloyd-Max codebook for the marginal density of one
 * coordinate of a uniform point on the unit sphere S^{d-1},
 *     f(x) proportional to (1 - x^2)^((d-3)/2) on [-1, 1],
 * by Lloyd's iteration (boundaries at centroid midpoints, centroids at cell
 * conditional means) from evenly spaced starting centroids until no centroid
 * moves by 1e-14 (at most 10000 passes).  Host only; touches no GPU.
 * ["OCTOPUS ..." -- key idea: per-coordinate Lloyd-Max over the marginals;
 *  glossary "Lloyd-Max quantization"]
 * d: even, 4..1024.  bits: 1..8.  *out receives a handle the caller frees
 * with tq_codebook_free.  Returns TQ_ERR_INVALID_ARG for other d or bits. */
TQ_API tq_status tq_codebook_init(int d, int bits, tq_codebook** out);

/* Copy the codebook to host arrays: centroids[2^bits] (increasing),
 * boundaries[2^bits - 1] (midpoints), *passes = Lloyd passes run.  Any output
 * pointer may be NULL. */
TQ_API tq_status tq_codebook_get(const tq_codebook* cb, double* centroids, double* boundaries,
                                 int* passes);

TQ_API void tq_codebook_free(tq_codebook* cb);

/* ---------------------------------------------------------------------- */
/* Cache                                                                   */
/* ---------------------------------------------------------------------- */

/* Opaque view over a caller-owned page pool plus the method constants (the
 * codebook, the rotation signs s and, when qjl_m > 0, the m x d Gaussian
 * matrix S, which the library keeps in device memory it owns). */
typedef struct tq_cache tq_cache;

/* Bytes of one page (block_size token slots of one KV head), as laid out
 * above.  Returns -1 for an invalid combination. */
TQ_API int64_t tq_page_bytes(int d, int key_bits, int value_bits, int qjl_m, int block_size);

/* Describe a cache over `pool` (device, num_blocks * num_kv_heads *
 * tq_page_bytes(...) bytes, 16-byte aligned, caller-owned) and derive the
 * method constants from `seed`:
 *   s_j  = +1 if the top bit of z_j(seed, 0) is clear, else -1   (j < d)
 *   S_ij = sqrt(-2 ln u1) cos(2 pi u2), u1 = ((z_{2n}(seed,1) >> 11) + 1) 2^-53,
 *          u2 = (z_{2n+1}(seed,1) >> 11) 2^-53, n = i*d + j          (i < m)
 * where z_i(seed, tag) = mix(seed ^ tag*0xD1B54A32D192ED03 + (i+1)*0x9E3779B97F4A7C15)
 * and mix is the SplitMix64 finaliser (Steele, Lea, Flood 2014).  The pages
 * draw the signs from a seed [deep dive -- Step 1: RHT] with torch's
 * generator, which is not reproduced.
 * Supported on the GPU path: d = 128, block_size = 16, key_bits and
 * value_bits each 1..8 (chosen per cache, e.g. per layer [deep dive --
 * per-layer bit allocation]), qjl_m in {0, 128} with the QJL sketch only for
 * key and value bits 2..4; anything else returns TQ_ERR_UNSUPPORTED.  The
 * library allocates a small device table (codebook remainders and
 * boundaries) per cache.  Uses the current CUDA device. */
TQ_API tq_status tq_cache_create(void* pool, int64_t num_blocks, int block_size, int num_kv_heads,
                                 int d, int key_bits, int value_bits, int qjl_m, uint64_t seed,
                                 tq_cache** out);

TQ_API void tq_cache_free(tq_cache* cache);

/* ---------------------------------------------------------------------- */
/* OCTOPUS triplet key codec                                               */
/* ---------------------------------------------------------------------- */

/* A cache whose keys use the OCTOPUS triplet codec ["OCTOPUS: Optimized KV
 * Cache for Transformers via Octahedral Parametrization ..." -- key
 * contribution "Octahedral triplet direction quantizer with norm marginals",
 * methodology steps 1-7]; values keep their min-max codes.  For a key:
 *   gamma = ||k|| (fp16), u = R (k / gamma) as for the main codec;
 *   u is cut into ceil(d/3) triplets t_i (the last padded with zeros);
 *   rho_i = ||t_i|| takes a (bits - 1)-bit code: the nearest level of a
 *     Lloyd-Max codebook for the norm of three coordinates of a uniform point
 *     on S^{d-1} (rho^2 ~ Beta(3/2, (d-3)/2));
 *   the direction n_i = t_i / rho_i ((0, 0, 1) if rho_i = 0) goes through the
 *     octahedral map Oct(n) = (xi, eta) (p = n / |n|_1; the lower half folded
 *     over the square's corners), and xi, eta take (bits + 1)-bit codes of one
 *     Lloyd-Max codebook for the marginal of xi of a uniform direction; among
 *     the nearest levels of xi and of eta and their neighbours (3 x 3 pairs)
 *     the pair whose unit direction is closest to n_i is kept.
 * The split (bits + 1, bits - 1) is the page's (b_dir, b_nrm) = (b + 1, b - 1).
 * Page (per block of block_size slots of one KV head): block_size key rows of
 * KR = 4 ceil(ceil(d/3) (3 bits + 1) / 32) bytes (triplet i's fields at bit
 * i (3 bits + 1): xi code, eta code, rho code, LSB first), then value codes,
 * gamma, scale, zero as in the main layout, padded to 16 bytes.
 * Decode: logit_t = sm_scale gamma_t sum_i rho^_i <(R q)_{3i..3i+2}, n^_i>, with
 * n^_i the unit direction of the stored level pair; values and the inverse
 * rotation as for the main codec.
 * tq_encode_kv, tq_decode_attention and tq_decode_workspace_bytes accept such
 * a cache (its decode rebuilds each page's unit keys in shared memory and
 * scores them on the tensor cores; the warps' partials are merged inside each
 * CTA, the CTAs' by a second kernel); the one-launch append
 * entry points return TQ_ERR_UNSUPPORTED.  Supported: d = 128, block_size =
 * 16, bits 2..4, value_bits 1..8.  The library allocates its codebooks and
 * direction table in device memory. */
TQ_API tq_status tq_cache_create_octopus(void* pool, int64_t num_blocks, int block_size, int num_kv_heads,
                                         int d, int bits, int value_bits, uint64_t seed, tq_cache** out);

/* Bytes of one OCTOPUS page, or -1 for an invalid combination (bits 2..4,
 * value_bits 1..8, d a positive multiple of 8). */
TQ_API int64_t tq_octopus_page_bytes(int d, int bits, int value_bits, int block_size);

/* The OCTOPUS codebooks the library computes on the host (tests): kind 0 gives
 * the 2^bits levels for xi and eta, kind 1 the 2^bits levels for the triplet
 * norm at dimension d, each increasing.  d 6..1024, bits 1..5. */
TQ_API tq_status tq_octopus_codebook(int d, int bits, int kind, double* levels);

/* The constants a seed defines, derived on the host without a GPU (the same
 * derivation tq_cache_create performs): signs[d] as +-1 and, if m > 0 and S is
 * not NULL, S[m*d] row-major in double.  d: 1..4096, m: 0..4096. */
TQ_API tq_status tq_method_constants(int d, int m, uint64_t seed, int8_t* signs, double* S);

/* Host copies of the derived constants (tests): signs[d] as +-1, S[m*d]
 * row-major in double (the device holds it in fp32). */
TQ_API tq_status tq_cache_signs(const tq_cache* cache, int8_t* signs);
TQ_API tq_status tq_cache_gaussian(const tq_cache* cache, double* S);

/* ---------------------------------------------------------------------- */
/* Encode (append)                                                         */
/* ---------------------------------------------------------------------- */

/* Compress num_tokens new tokens into the cache.
 * K, V: device, [num_tokens, num_kv_heads, d] of `dtype`, 16-byte aligned.
 * slot_mapping: device int64 [num_tokens]; slot = block * block_size + offset.
 *   A negative slot skips the token; a slot past the pool sets
 *   TQ_FLAG_BAD_SLOT and skips it.
 * For each (token, KV head):
 *   key:   gamma = ||k|| (fp32) stored as fp16; u_rot = R k / gamma with
 *          R = H diag(s) / sqrt(d); code_j = #{boundaries < u_rot[j]};
 *          if qjl_m > 0: r = u_rot - C[code], rho = ||r|| as fp16,
 *          sigma_i = [(S r)_i >= 0].  A zero key stores codes 2^(kb-1) - 1,
 *          rho 0 and all sigma bits 1.
 *   value: v_rot = R v; mn = min, mx = max over coordinates; scale =
 *          (mx - mn)/(2^vb - 1); code = clamp(round-half-even((v_rot - mn) /
 *          scale), 0, 2^vb - 1) (all 0 if scale == 0); scale, mn as fp16.
 * Arithmetic is fp32.  Encodes of bf16 / fp16 inputs without QJL and with at
 * least one 128-row tile of (token, KV head) items per SM form R k and R v
 * on the tensor cores (exact products, fp32 accumulation: the same values as
 * the butterfly up to the order of the additions); the others use the
 * butterfly.  An input coordinate that is inf or NaN sets TQ_FLAG_NONFINITE
 * (on the tensor-core path, so does a finite input whose rotated coordinate
 * exceeds the fp32 range, above about 2.6e36); a stored fp16 field that
 * overflows sets TQ_FLAG_OVERFLOW.
 * [three steps (split/rotate/codebook); Bit-Axon -- quantization function;
 *  deep dive -- Step 1 (RHT), Step 3 (value codes); "OCTOPUS ..." -- step 8]
 * Tokens that map to the same slot race; the last writer is unspecified. */
TQ_API tq_status tq_encode_kv(const tq_cache* cache, const void* K, const void* V, tq_dtype dtype,
                              int64_t num_tokens, const int64_t* slot_mapping, int32_t* dev_status,
                              void* stream);

/* ---------------------------------------------------------------------- */
/* Decode attention                                                        */
/* ---------------------------------------------------------------------- */

/* Workspace bytes tq_decode_attention needs for this batch shape (split-K
 * partials plus one counter per sequence and KV head).  The workspace must
 * be zero-filled once before its first use; each call leaves its counters at
 * zero again on completion, also a call that reported TQ_FLAG_TIMEOUT, so a
 * workspace can be reused by later calls on the same stream without
 * clearing.  Two calls in flight at once must not share a workspace. */
TQ_API size_t tq_decode_workspace_bytes(const tq_cache* cache, int batch, int num_q_heads,
                                        int max_blocks_per_seq);

/* One query token per sequence over its cached tokens:
 *   out[b, hq] = sum_t softmax_t(l_t) V^_t,  t < lens[b],
 *   l_t = sm_scale * gamma_t * ( <R q, C[code_t]>
 *                                + sqrt(pi/2)/m * rho_t * <S R q, 2 sigma_t - 1> )  [QJL term if m > 0]
 *   V^_t = R^T (scale_t * vcode_t + zero_t),
 * with the KV head of query head hq being hq / (num_q_heads / num_kv_heads)
 * and token t in block block_table[b * max_blocks_per_seq + t / block_size],
 * slot t % block_size.  Logits and values are formed in the rotated frame;
 * keys are never reconstructed; one inverse rotation is applied per output.
 * q: device [batch, num_q_heads, d] of `dtype`, 4-element aligned.
 * block_table: device int32.  lens: device int32 [batch]; a zero length
 * yields a zero output row.  out: device fp32 [batch, num_q_heads, d],
 * 16-byte aligned.  q and out may instead be page-locked host memory that
 * tq_device_accessible accepts.  sm_scale: normally 1/sqrt(d).
 * workspace: device, at least tq_decode_workspace_bytes(...) bytes.
 * num_q_heads must be a multiple of num_kv_heads with a group size <= 8.
 * A block id outside the pool sets TQ_FLAG_BAD_SLOT and its page is skipped. */
TQ_API tq_status tq_decode_attention(const tq_cache* cache, const void* q, tq_dtype dtype, int batch,
                                     int num_q_heads, const int32_t* block_table,
                                     int max_blocks_per_seq, const int32_t* lens, float sm_scale,
                                     float* out, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, void* stream);

/* One decode step in one launch: append, then attend.  For every sequence b
 * with lens[b] >= 1 the new token (rows k_new[b], v_new[b] of
 * [batch, num_kv_heads, d], `kv_dtype`, device, 16-byte aligned) is encoded
 * exactly as tq_encode_kv encodes it into position lens[b] - 1, i.e. slot
 * block_table[b][(lens[b]-1) / block_size] * block_size + (lens[b]-1) % block_size,
 * and attended to together with the lens[b] - 1 tokens before it; all other
 * arguments and results are those of tq_decode_attention.  This is the order
 * of the pages' decode step -- the new key/value enters the compressed cache,
 * then the query reads it ["TurboQuant: KV Cache Vector Quantization" -- three
 * steps; Bit-Axon -- KV cache memory model] -- without a separate encode
 * launch between the two.  With a QJL sketch (qjl_m > 0) the appended token's
 * residual norm and sign row are computed in the same launch, with the same
 * arithmetic as tq_encode_kv ["OCTOPUS ..." -- methodology step 8].  OCTOPUS
 * caches return TQ_ERR_UNSUPPORTED. */
TQ_API tq_status tq_decode_attention_append(const tq_cache* cache, const void* k_new, const void* v_new,
                                            tq_dtype kv_dtype, const void* q, tq_dtype dtype, int batch,
                                            int num_q_heads, const int32_t* block_table,
                                            int max_blocks_per_seq, const int32_t* lens, float sm_scale,
                                            float* out, void* workspace, size_t workspace_bytes,
                                            int32_t* dev_status, void* stream);

/* The same decode step over a sliding window kept as a ring buffer: each
 * sequence owns `window` slots (window / block_size blocks of its block table,
 * window a positive multiple of block_size, at most max_blocks_per_seq *
 * block_size) and token t lives in slot t mod window, so the ring always holds
 * the last `window` tokens [Bit-Axon -- KV cache memory model: a sliding-
 * window layer keeps the K and V of W tokens].  lens[b] counts all of sequence b's tokens, the new one
 * included: the new token is encoded into slot (lens[b] - 1) mod window,
 * replacing the token that leaves the window, and the query attends over the
 * min(lens[b], window) tokens the ring holds (attention does not depend on
 * their order).  To fill a ring, encode only the last `window` tokens, each
 * at slot block_table[b][(t mod window) / block_size] * block_size + t mod
 * block_size; tokens of one tq_encode_kv call that map to one slot race.
 * A plain tq_decode_attention over a ring is the same attention with
 * lens[b] replaced by min(lens[b], window).  Returns TQ_ERR_INVALID_ARG for a
 * window that is not a positive multiple of block_size or does not fit the
 * block table; other arguments and results are those of
 * tq_decode_attention_append. */
TQ_API tq_status tq_decode_attention_ring_append(const tq_cache* cache, const void* k_new, const void* v_new,
                                                 tq_dtype kv_dtype, const void* q, tq_dtype dtype, int batch,
                                                 int num_q_heads, const int32_t* block_table,
                                                 int max_blocks_per_seq, const int32_t* lens, int window,
                                                 float sm_scale, float* out, void* workspace,
                                                 size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------- */
/* Chunked prefill attention                                               */
/* ---------------------------------------------------------------------- */

/* Workspace bytes tq_prefill_attention needs (zero-filled once before first
 * use, like a decode workspace). */
TQ_API size_t tq_prefill_workspace_bytes(const tq_cache* cache, int num_positions, int num_q_heads,
                                         int max_blocks_per_seq);

/* Attention for a chunk of num_positions consecutive query positions of one
 * sequence, first_position .. first_position + num_positions - 1, over the
 * compressed cache, causally: the query at position p attends over the
 * sequence's tokens 0 .. p.  The chunk's own keys and values must already be
 * in the cache (tq_encode_kv first), which is the order of the deep dive's
 * attention forward: the new keys and values update the compressed cache,
 * then attention reads it [TurboQuant deep dive -- attention forward with
 * kv_cache.update; llama.cpp results: prefill speed on a par with Q8_0].
 * q: device [num_positions, num_q_heads, d]; block_table: device int32, the
 * sequence's one row of max_blocks_per_seq blocks; out: device fp32
 * [num_positions, num_q_heads, d].  For 4-bit keys without the QJL sketch and
 * value codes of 1..4 bits the scores and values are dense tcgen05 tensor-core
 * contractions: each page is unpacked once for all num_positions x group
 * query rows of its KV head (128 rows at a time), and a second launch merges
 * the token splits.  Other caches run each position as one row of the decode
 * kernel, which reads the cached pages once per position. */
TQ_API tq_status tq_prefill_attention(const tq_cache* cache, const void* q, tq_dtype dtype, int num_positions,
                                      int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                                      int first_position, float sm_scale, float* out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream);

/* Bytes of the fixed decode workspace built into the library (see below). */
#define TQ_NOALLOC_WORKSPACE_BYTES (4u << 20)

/* Decode attention exactly as tq_decode_attention, but without a caller
 * workspace and without allocating anything.  (The source pages have no
 * counterpart to this call: it exists for callers that may not allocate.)
 *
 * Who needs it: callers that cannot call cudaMalloc when they decode -- an
 * engine that plans all of its device memory ahead of time, code running in a
 * memory pool it does not control, or a serving loop that forbids allocations
 * because they can synchronise the device.  Instead of a workspace argument
 * the call uses one fixed scratch area of TQ_NOALLOC_WORKSPACE_BYTES (4 MiB)
 * that is part of the library image; every GPU that loads the library holds
 * it until the process exits.
 *
 * Arguments are those of tq_decode_attention minus the workspace.  Returns
 * TQ_ERR_WORKSPACE, launching nothing, when the batch shape would need more
 * than TQ_NOALLOC_WORKSPACE_BYTES (tq_decode_workspace_bytes tells).
 * Uses the current CUDA device, which must be the cache's.  A call outside
 * stream capture looks up the scratch area's device address on that device
 * (a host-side query, so a device reset between calls does no harm); a call
 * while `stream` is capturing reuses the address the last uncaptured call on
 * the device found, and fails with TQ_ERR_INVALID_ARG if there was none: make
 * the first call before any capture.  For a main-codec cache each call clears
 * the area's split counters on `stream`; no call runs cudaMalloc, cudaFree or
 * any other allocating routine.
 * All calls on a device share the one area and it keeps the last call's
 * contents: two calls whose work overlaps on the GPU (different streams, or
 * host threads without ordering) race and corrupt each other's results. */
TQ_API tq_status tq_decode_attention_noalloc(const tq_cache* cache, const void* q, tq_dtype dtype,
                                             int batch, int num_q_heads, const int32_t* block_table,
                                             int max_blocks_per_seq, const int32_t* lens, float sm_scale,
                                             float* out, int32_t* dev_status, void* stream);

/* Whether code on the current device can read and write the memory at p:
 * memory of this device, managed memory, or page-locked host memory mapped
 * into the device's address space at the same address (under unified
 * addressing, what cudaHostAlloc and cudaMallocHost return).  Sets
 * *accessible to 1 or 0; memory the runtime does not know (pageable host
 * memory) gives 0.  The decode entry points read q, k_new and v_new and write
 * out in place wherever they are, so these may be page-locked host buffers
 * that this function accepts: the kernel then moves the step's inputs and its
 * result over the host link (NVLink-C2C on Grace systems) itself, with no
 * copy launches.  Every CTA of a split reads the query itself over the link,
 * so for long contexts (many splits) this is slower than staging the inputs
 * with one copy each way.  Returns TQ_ERR_INVALID_ARG for a NULL
 * `accessible`. */
TQ_API tq_status tq_device_accessible(const void* p, int* accessible);

/* Test hook for the device-side timeout path.  (The source pages have no
 * counterpart: it exists so that a test can make a bounded wait run out
 * without faulting or hanging anything.)  With cycles > 0, every decode
 * launched afterwards in this process makes warp 0 of each CTA with an odd
 * split index wait about `cycles` SM cycles on a shared-memory barrier that
 * nothing arrives on.  That wait gives up and the CTA takes the same path as
 * any timed-out wait: it waits (bounded) for its page copies in flight, sets
 * TQ_FLAG_TIMEOUT, contributes an empty partial to its sequence's split merge
 * and still takes part in it, so the call returns, its output is incomplete,
 * and its workspace is fit for the next call.  cycles <= 0 turns the hook
 * off (the default).  A process-wide host setting; not for production use. */
TQ_API void tq_test_stall_waits(int64_t cycles);

/* Self-test of the Blackwell tensor-core building blocks the decode kernels
 * use (the source pages have no counterpart: it checks this library's own
 * use of tensor memory and the asynchronous MMA).  One CTA computes
 * D = A . B with A [128 x 256] and B [256 x 16] fp16 (device, row-major,
 * 16-byte aligned) and fp32 accumulation, and writes out (device fp32,
 * 6 x 128 x 16): [0] A staged in tensor memory, B in shared memory, D read
 * back one row per thread; [1] the same D read back in the 16-lane fragment
 * layout and stored by that layout's documented positions; [2] A and B both
 * from shared memory; [3] A written to tensor memory with the 16-lane
 * fragment store; [4] and [5] B in the MN-major layout under the two
 * readings of the descriptor's byte offsets.  [0]..[3] equal A . B up to
 * fp32 summation order, and so does the one of [4], [5] whose reading the
 * hardware uses.
 * A bounded wait that gives up sets TQ_FLAG_TIMEOUT in *dev_status. */
TQ_API tq_status tq_selftest_tcgen05(const void* A, const void* B, float* out, int32_t* dev_status, void* stream);

/* Text for a status code, and the detail of the last failure on this thread. */
TQ_API const char* tq_status_string(tq_status s);
TQ_API const char* tq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
