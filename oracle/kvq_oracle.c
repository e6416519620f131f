/*
 * kvq_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow CPU statement of what the quantized-KV MLA path computes: the
 * KV8 and TQ4 row codecs, the K2/V4 GQA codec with its FP16 window overlay, and
 * softmax attention over the reconstructed rows in double precision, and the
 * PolarQuant codec of the TQ tier.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant with the CUDA library: every
 * constant it needs (the Lloyd-Max codebooks, the e4m3 and fp16 grids, the
 * rotation signs) is derived here from its definition.
 *
 * The pages are cited by title:
 *   [P1] "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant (KV_TQ) on CPU,
 *         CUDA, and Metal" (colibri pull request 399)
 *   [P2] "CPU: KV cache quantization -- KV8 (fp8 e4m3) + KV_TQ (rotated-int4 /
 *         PolarQuant)" (colibri pull request 553)
 *   [P3] "KV cache: FP16 sliding window + attention sinks, and an optional
 *         2-bit K / 4-bit V cache scheme (--kv q2k)" (Strata pull request 2318)
 *
 * Floating point: encoders work in IEEE binary32 exactly as the method states
 * (f32 row scale, f32 division, one rounding to e4m3); attention accumulates in
 * binary64.  Build with -ffp-contract=off and without -ffast-math so that no
 * multiply-add is fused behind our back.
 *
 * Parity status per function (the tests named here pin each one against
 * something other than this file):
 *   e4m3 value/encode ....... pinned (OCP e4m3 special values, brute-force
 *                              nearest-value search, CUDA's own conversion)
 *   fp16 value/encode ....... pinned (IEEE half special values, brute force,
 *                              numpy float16 casts)
 *   splitmix64 .............. pinned (published reference outputs)
 *   Lloyd-Max solver ........ pinned (Max 1960 table for 4 and 16 levels)
 *   FWHT .................... pinned (Sylvester Hadamard matrix, closed forms)
 *   KV8 / TQ4 codecs ........ pinned (round trip, distortion ~0.096 from [P1],
 *                              byte counts from [P1]/[P2], invariants)
 *   sign choice of TQ4 ...... parity unpinned against the pages (they do not
 *                              state how the seed becomes signs); pinned only by
 *                              determinism and orthogonality
 *   attention ............... pinned (closed forms, numpy softmax reference,
 *                              orthogonality identities of [P1]/[P2])
 *   K2/V4 codec + overlay ... pinned (byte counts and overlay footprint from
 *                              [P3], q4_0 nibble order fixture, gain property)
 *   PolarQuant codebooks .... pinned (closed-form centroid conditions for
 *                              k = 2 and 3, symmetry, Panter-Dite MSE limit,
 *                              sampled angle densities)
 *   PolarQuant codec ........ pinned (exact polar round trips, closed-form
 *                              angles of basis and constant vectors, codes =
 *                              nearest centroid by atan2 away from cell
 *                              edges, distortion = the sum of the levels'
 *                              quantizer MSE); its distortion at 4 bits does
 *                              not reproduce the pages' ~0.147 (reported)
 *   K2/V4 append ............ pinned (whole groups = the encoder, constant-
 *                              magnitude closed forms of the partial-group
 *                              rule, one call = two calls split at a group
 *                              boundary)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVQO_OK 0
#define KVQO_ERR_SHAPE 2
#define KVQO_ERR_ARG 1

/* ------------------------------------------------------------------------ */
/* Round-half-to-even of a non-negative double that holds few bits.         */
/* ------------------------------------------------------------------------ */
static double rne_nonneg(double x)
{
    double f = floor(x);
    double r = x - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* ------------------------------------------------------------------------ */
/* fp8 e4m3.  Value grid per [P1], rebase comment, item 3 "HIP portability":  */
/* normals (1+M/8)*2^(E-7), subnormals M*2^-9, and S.1111.111 reads as 0.    */
/* ------------------------------------------------------------------------ */
double kvqo_e4m3_value(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return 0.0;          /* the NaN pattern reads back as 0 */
    if (e == 0u) mag = ldexp((double)m, -9);
    else         mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* One rounding of an f32 value onto the e4m3 grid: nearest value, ties to the
 * even mantissa, magnitudes beyond the largest finite value (448) saturate to
 * it ([P1] Commits, item 1: "RNE, per-row amax/448 scale").  The NaN pattern is
 * never produced.  NaN input is outside the contract and yields +0. */
unsigned kvqo_e4m3_encode(float u)
{
    unsigned sign = signbit(u) ? 0x80u : 0u;
    double a = fabs((double)u);
    if (isnan(u)) return 0u;
    if (a >= 448.0) return sign | 0x7Eu;
    if (a < ldexp(1.0, -6)) {                      /* subnormal range, step 2^-9 */
        double m = rne_nonneg(a / ldexp(1.0, -9)); /* 0..8; 8 is the smallest normal, code 0x08 */
        return sign | (unsigned)m;
    }
    int k;
    frexp(a, &k);                                   /* a = f * 2^k, f in [0.5, 1) */
    int e = k - 1;                                  /* a in [2^e, 2^(e+1)) */
    double mant = rne_nonneg((ldexp(a, -e) - 1.0) * 8.0);
    if (mant == 8.0) { mant = 0.0; e += 1; }
    int E = e + 7;
    if (E > 15 || (E == 15 && mant == 7.0)) return sign | 0x7Eu;
    return sign | ((unsigned)E << 3) | (unsigned)mant;
}

void kvqo_e4m3_encode_array(const float* u, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)kvqo_e4m3_encode(u[i]);
}

/* ------------------------------------------------------------------------ */
/* IEEE binary16 (used by the K2/V4 scales and the FP16 overlay of [P3]).    */
/* ------------------------------------------------------------------------ */
double kvqo_f16_value(unsigned h)
{
    unsigned s = (h >> 15) & 1u, e = (h >> 10) & 31u, m = h & 1023u;
    double mag;
    if (e == 31u) mag = m ? NAN : INFINITY;
    else if (e == 0u) mag = ldexp((double)m, -24);
    else mag = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
    return s ? -mag : mag;
}

unsigned kvqo_f16_encode(float x)
{
    unsigned sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs((double)x);
    if (isnan(x)) return 0x7E00u;
    if (a >= 65520.0) return sign | 0x7C00u;      /* rounds past the largest finite value */
    if (a < ldexp(1.0, -14)) {
        double m = rne_nonneg(a / ldexp(1.0, -24));
        return sign | (unsigned)m;
    }
    int k;
    frexp(a, &k);
    int e = k - 1;
    double mant = rne_nonneg((ldexp(a, -e) - 1.0) * 1024.0);
    if (mant == 1024.0) { mant = 0.0; e += 1; }
    return sign | ((unsigned)(e + 15) << 10) | (unsigned)mant;
}

/* ------------------------------------------------------------------------ */
/* splitmix64 (Steele, Lea and Flood 2014; Vigna's public-domain statement). */
/* The TQ4 rotation is "seeded" ([P1] Commits, item 6); the pages do not say */
/* how the seed becomes signs.  Reading: words w_0, w_1, ... are successive  */
/* splitmix64 outputs from state = seed; each block takes ceil(n/64) fresh   */
/* words in block order, and sign i of a block is -1 when bit (i mod 64) of  */
/* its word (i / 64) is set.                                                 */
/* ------------------------------------------------------------------------ */
uint64_t kvqo_splitmix64_next(uint64_t* state)
{
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void kvqo_tq4_signs(uint64_t seed, int n_blocks, const int* bdims, int8_t* sigma)
{
    uint64_t state = seed;
    int off = 0;
    for (int b = 0; b < n_blocks; ++b) {
        int n = bdims[b];
        int words = (n + 63) / 64;
        for (int w = 0; w < words; ++w) {
            uint64_t word = kvqo_splitmix64_next(&state);
            for (int j = 0; j < 64 && w * 64 + j < n; ++j)
                sigma[off + w * 64 + j] = ((word >> j) & 1ull) ? (int8_t)-1 : (int8_t)1;
        }
        off += n;
    }
}

/* ------------------------------------------------------------------------ */
/* Lloyd-Max quantizer of N(0,1) ([P1] "Why rotated-int4 for the 4-bit tier": */
/* a fixed 16-level Lloyd-Max codebook, N(0,1)-optimal; [P3] "Why per-channel */
/* K and per-token V": the 4-level codebook of the 2-bit K).  Fixed point of  */
/* the two optimality conditions: each threshold is the midpoint of its two  */
/* levels, each level is the centroid (conditional mean) of its cell.        */
/* ------------------------------------------------------------------------ */
static double std_pdf(double t) { return isinf(t) ? 0.0 : exp(-0.5 * t * t) / sqrt(2.0 * M_PI); }
static double std_cdf(double t) { return 0.5 * erfc(-t / sqrt(2.0)); }

int kvqo_lloyd_max_gaussian(int levels, double* c, double* mse_out)
{
    /* N(0,1) is symmetric, so is its optimal quantizer: level L-1-k = -level k
     * and, for an even count, the middle threshold is exactly 0.  The
     * iteration is run on that symmetric form (averaging each mirrored pair
     * after every update) so that rounding cannot tilt it.  It stops when an
     * update changes no level by more than 1e-15. */
    if (levels < 2 || levels > 64) return -1;
    double t[65];
    for (int k = 0; k < levels; ++k)                       /* symmetric uniform start */
        c[k] = ((double)k - 0.5 * (levels - 1)) * (4.0 / levels);
    int it;
    for (it = 1; it <= 400000; ++it) {
        t[0] = -INFINITY;
        for (int k = 1; k < levels; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
        if (levels % 2 == 0) t[levels / 2] = 0.0;
        t[levels] = INFINITY;
        double cn[64];
        for (int k = 0; k < levels; ++k) {
            double mass = std_cdf(t[k + 1]) - std_cdf(t[k]);
            cn[k] = (std_pdf(t[k]) - std_pdf(t[k + 1])) / mass;
        }
        double delta = 0.0;
        for (int k = 0; k < levels; ++k) {
            double sym = 0.5 * (cn[k] - cn[levels - 1 - k]);
            if (2 * k + 1 == levels) sym = 0.0;
            if (fabs(sym - c[k]) > delta) delta = fabs(sym - c[k]);
            cn[k] = sym;
        }
        for (int k = 0; k < levels; ++k) c[k] = cn[k];
        if (delta <= 1e-15) break;
    }
    if (mse_out) {
        /* E[(X - Q(X))^2] = 1 - sum_k c_k^2 * P(cell k) for centroid levels;
         * written out directly as sum over cells of E[(X - c_k)^2 ; cell k]. */
        double mse = 0.0;
        t[0] = -INFINITY;
        for (int k = 1; k < levels; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
        if (levels % 2 == 0) t[levels / 2] = 0.0;
        t[levels] = INFINITY;
        for (int k = 0; k < levels; ++k) {
            double a = t[k], b = t[k + 1];
            double p = std_cdf(b) - std_cdf(a);
            double m1 = std_pdf(a) - std_pdf(b);                         /* E[X; cell] */
            double ta = isinf(a) ? 0.0 : a * std_pdf(a);
            double tb = isinf(b) ? 0.0 : b * std_pdf(b);
            double m2 = p + ta - tb;                                     /* E[X^2; cell] */
            mse += m2 - 2.0 * c[k] * m1 + c[k] * c[k] * p;
        }
        *mse_out = mse;
    }
    return it;
}

/* f32 levels and f32 decision thresholds of a solved codebook.  Reading: a
 * code is the number of thresholds strictly below u (ties go to the lower
 * level), thresholds being the f64 midpoints of adjacent levels rounded once
 * to f32. */
static void codebook_f32(int levels, float* lv, float* th)
{
    /* solved once per level count and kept (the solve is deterministic) */
    static double cache[65][64];
    static int have[65];
    if (!have[levels]) {
        kvqo_lloyd_max_gaussian(levels, cache[levels], NULL);
        have[levels] = 1;
    }
    const double* c = cache[levels];
    for (int k = 0; k < levels; ++k) lv[k] = (float)c[k];
    for (int k = 0; k + 1 < levels; ++k) th[k] = (float)(0.5 * (c[k] + c[k + 1]));
}

void kvqo_tq4_codebook(float* levels16, float* thresholds15) { codebook_f32(16, levels16, thresholds15); }
void kvqo_k2_codebook(float* levels4, float* thresholds3)    { codebook_f32(4, levels4, thresholds3); }

static unsigned code_of(float u, const float* th, int n_th)
{
    unsigned k = 0;
    for (int j = 0; j < n_th; ++j)
        if (th[j] < u) ++k;
    return k;
}

/* ------------------------------------------------------------------------ */
/* Fast Walsh-Hadamard transform, radix 2, unnormalized, in place.  Stage    */
/* order h = 1, 2, 4, ..., n/2; each butterfly maps (a, b) to (a+b, a-b).   */
/* [P1] Commits, item 6 and [P2] "What's in it": randomized-Hadamard        */
/* rotation through a radix-2 FWHT.                                          */
/* ------------------------------------------------------------------------ */
void kvqo_fwht_f32(float* v, int n)
{
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
}

void kvqo_fwht_f64(double* v, int n)
{
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
}

static int is_pow2_ge2(int n) { return n >= 2 && (n & (n - 1)) == 0; }

/* Sum of squares in a fixed order: 32 interleaved partial sums (partial j
 * takes elements j, j+32, j+64, ... in ascending order with one fused
 * multiply-add each), then pairwise halving: for off = 16, 8, 4, 2, 1,
 * partial j += partial j+off for j < off.  The pages leave the order open;
 * this is the reading used for the TQ4 radius and the K2 channel scale. */
static float sumsq_r32(const float* x, int n, int stride)
{
    float p[32];
    for (int j = 0; j < 32; ++j) p[j] = 0.0f;
    for (int i = 0; i < n; ++i) p[i % 32] = fmaf(x[(int64_t)i * stride], x[(int64_t)i * stride], p[i % 32]);
    for (int off = 16; off >= 1; off /= 2)
        for (int j = 0; j < off; ++j) p[j] = p[j] + p[j + off];
    return p[0];
}

/* ------------------------------------------------------------------------ */
/* KV8 row codec.  [P1] Commits, item 1 and [P2] "What's in it": fp8 e4m3    */
/* per element, one f32 scale amax/448, RNE.  Reading of the scale           */
/* granularity: one scale per scale block (latent 512 + rope 64 gives 2 f32  */
/* per row, 584 B per 576-dim row, the "~3.9x" of [P1] Summary).             */
/* ------------------------------------------------------------------------ */
static int row_dim(int n_blocks, const int* bdims)
{
    int d = 0;
    for (int b = 0; b < n_blocks; ++b) d += bdims[b];
    return d;
}

int kvqo_kv8_encode(const float* x, int64_t n_rows, int n_blocks, const int* bdims,
                    uint8_t* codes, float* scales)
{
    if (n_blocks < 1 || n_blocks > 8) return KVQO_ERR_ARG;
    int D = row_dim(n_blocks, bdims);
    for (int64_t t = 0; t < n_rows; ++t) {
        const float* xr = x + t * D;
        uint8_t* cr = codes + t * D;
        int off = 0;
        for (int b = 0; b < n_blocks; ++b) {
            int n = bdims[b];
            float amax = 0.0f;
            for (int i = 0; i < n; ++i) {
                float a = fabsf(xr[off + i]);
                if (a > amax) amax = a;
            }
            float s = amax / 448.0f;
            scales[t * n_blocks + b] = s;
            for (int i = 0; i < n; ++i) {
                if (s == 0.0f) { cr[off + i] = 0; continue; }   /* inert block: codes 0, scale 0 */
                float u = xr[off + i] / s;
                cr[off + i] = (uint8_t)kvqo_e4m3_encode(u);
            }
            off += n;
        }
    }
    return KVQO_OK;
}

/* Reconstruction x_hat = s * value(code), exact in binary64. */
void kvqo_kv8_decode(const uint8_t* codes, const float* scales, int64_t n_rows,
                     int n_blocks, const int* bdims, double* xhat)
{
    int D = row_dim(n_blocks, bdims);
    for (int64_t t = 0; t < n_rows; ++t) {
        int off = 0;
        for (int b = 0; b < n_blocks; ++b) {
            double s = (double)scales[t * n_blocks + b];
            for (int i = 0; i < bdims[b]; ++i)
                xhat[t * D + off + i] = s * kvqo_e4m3_value(codes[t * D + off + i]);
            off += bdims[b];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* TQ4 (rotated-int4) row codec.  [P1] "Why rotated-int4 for the 4-bit      */
/* tier": randomized-Hadamard rotation, fixed 16-level Lloyd-Max N(0,1)      */
/* codebook scaled by radius/sqrt(n), the radius riding the per-row scale;   */
/* [P2] "What's in it": nibble-packed.  Per block of n (a power of two):     */
/*   y = (1/sqrt n) * H_n * (sigma . x)          (f32 FWHT, then one multiply) */
/*   r = ||x||  (the rotation keeps the radius),  s = r / sqrt(n)            */
/*   code_i = number of thresholds below y_i / s                             */
/*   byte j = code_2j | code_(2j+1) << 4                                     */
/* A width that is not a power of two >= 2 is refused ([P1] rebase comment   */
/* and [P2] review-pass item 1: such rows would all become inert).           */
/* ------------------------------------------------------------------------ */
int kvqo_tq4_encode(const float* x, int64_t n_rows, int n_blocks, const int* bdims, uint64_t seed,
                    uint8_t* packed, float* scales)
{
    if (n_blocks < 1 || n_blocks > 8) return KVQO_ERR_ARG;
    for (int b = 0; b < n_blocks; ++b)
        if (!is_pow2_ge2(bdims[b])) return KVQO_ERR_SHAPE;
    int D = row_dim(n_blocks, bdims);
    int8_t* sigma = (int8_t*)malloc((size_t)D);
    float* v = (float*)malloc(sizeof(float) * (size_t)D);
    float lv[16], th[15];
    kvqo_tq4_codebook(lv, th);
    kvqo_tq4_signs(seed, n_blocks, bdims, sigma);
    for (int64_t t = 0; t < n_rows; ++t) {
        const float* xr = x + t * D;
        uint8_t* pr = packed + t * (D / 2);
        int off = 0;
        for (int b = 0; b < n_blocks; ++b) {
            int n = bdims[b];
            for (int i = 0; i < n; ++i) v[i] = sigma[off + i] < 0 ? -xr[off + i] : xr[off + i];
            kvqo_fwht_f32(v, n);
            float kn = (float)(1.0 / sqrt((double)n));
            float ss = sumsq_r32(xr + off, n, 1);
            float r = sqrtf(ss);
            float s = r / sqrtf((float)n);
            scales[t * n_blocks + b] = s;
            for (int i = 0; i < n; i += 2) {
                unsigned c0 = 0, c1 = 0;
                if (s != 0.0f) {                          /* inert block: codes 0, scale 0 */
                    float y0 = v[i] * kn, y1 = v[i + 1] * kn;
                    c0 = code_of(y0 / s, th, 15);
                    c1 = code_of(y1 / s, th, 15);
                }
                pr[(off + i) / 2] = (uint8_t)(c0 | (c1 << 4));
            }
            off += n;
        }
    }
    free(v);
    free(sigma);
    return KVQO_OK;
}

/* Rotation of whole vectors in binary64: forward y = k_n H (sigma . x), and
 * its transpose (the unrotation) x = sigma . (k_n H y), per block. */
int kvqo_tq4_rotate(const double* in, double* out, int64_t n_vecs, int n_blocks, const int* bdims,
                    uint64_t seed, int inverse)
{
    for (int b = 0; b < n_blocks; ++b)
        if (!is_pow2_ge2(bdims[b])) return KVQO_ERR_SHAPE;
    int D = row_dim(n_blocks, bdims);
    int8_t* sigma = (int8_t*)malloc((size_t)D);
    double* v = (double*)malloc(sizeof(double) * (size_t)D);
    kvqo_tq4_signs(seed, n_blocks, bdims, sigma);
    for (int64_t t = 0; t < n_vecs; ++t) {
        int off = 0;
        for (int b = 0; b < n_blocks; ++b) {
            int n = bdims[b];
            double kn = 1.0 / sqrt((double)n);
            for (int i = 0; i < n; ++i)
                v[i] = inverse ? in[t * D + off + i] : sigma[off + i] * in[t * D + off + i];
            kvqo_fwht_f64(v, n);
            for (int i = 0; i < n; ++i)
                out[t * D + off + i] = inverse ? sigma[off + i] * kn * v[i] : kn * v[i];
            off += n;
        }
    }
    free(v);
    free(sigma);
    return KVQO_OK;
}

/* Reconstruction: c_hat = s * level(code), then x_hat = unrotate(c_hat). */
int kvqo_tq4_decode(const uint8_t* packed, const float* scales, int64_t n_rows, int n_blocks,
                    const int* bdims, uint64_t seed, double* xhat)
{
    for (int b = 0; b < n_blocks; ++b)
        if (!is_pow2_ge2(bdims[b])) return KVQO_ERR_SHAPE;
    int D = row_dim(n_blocks, bdims);
    float lv[16], th[15];
    kvqo_tq4_codebook(lv, th);
    double* chat = (double*)malloc(sizeof(double) * (size_t)D);
    for (int64_t t = 0; t < n_rows; ++t) {
        int off = 0;
        for (int b = 0; b < n_blocks; ++b) {
            double s = (double)scales[t * n_blocks + b];
            for (int i = 0; i < bdims[b]; ++i) {
                unsigned byte = packed[t * (D / 2) + (off + i) / 2];
                unsigned code = ((off + i) & 1) ? (byte >> 4) : (byte & 15u);
                chat[off + i] = s * (double)lv[code];
            }
            off += bdims[b];
        }
        kvqo_tq4_rotate(chat, xhat + t * D, 1, n_blocks, bdims, seed, 1);
    }
    free(chat);
    return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* PolarQuant row codec (codec 0 of the TQ tier).  [P1] Summary names it    */
/* ("PolarQuant, arXiv 2502.02617, variable 2-6 bit"), [P1] Commits item 6   */
/* gives its shape ("randomized-Hadamard rotation + recursive polar") and    */
/* [P2] "What's in it" its bit widths (KV_TQ = 2|3|5|6, or 4 with            */
/* KV_TQ_POLAR = 1).  The steps follow the published method (Han et al.,     */
/* "PolarQuant: Quantizing KV Caches with Polar Transformation", 2025):      */
/*                                                                           */
/*   1. rotate the block as TQ4 does: y = (1/sqrt n) H_n (sigma . x), f32;   */
/*   2. level 1: each pair (y_2j, y_2j+1) becomes a radius and an angle in   */
/*      [0, 2 pi); level l >= 2: each pair of level-(l-1) radii (lo, hi)     */
/*      becomes sqrt(lo^2 + hi^2) and the angle atan2(hi, lo) in [0, pi/2];  */
/*      log2(n) levels leave one radius R, stored as the block's f32 scale;  */
/*   3. every angle is quantized to b bits with the level's own codebook:    */
/*      level 1 is uniform on the circle (its angle is uniform after the     */
/*      rotation), level l >= 2 is the Lloyd-Max quantizer of the angle's    */
/*      density, proportional to sin(2 psi)^(k-1) with k = 2^(l-1) (the      */
/*      angle between two independent k-dimensional Gaussian halves);        */
/*   4. reconstruction runs the tree back down from R with the cells'        */
/*      centroids, then unrotates.                                            */
/* Readings where the pages are silent (each also in the design notes):      */
/*   * one width b for every angle of every level, the recursion run to a   */
/*     single radius: the pages' "variable 2-6 bit" names one width per     */
/*     tier, and at b = 4 the row is then 296 bytes like TQ4's (the paper's  */
/*     own 4-level, 4/2/2/2-bit split with fp16 radii is another reading);   */
/*   * pairing of consecutive elements, angles stored level by level (level */
/*     1 first, in pair order), b bits each, least significant bit first,   */
/*     ceil(n b / 8) bytes per block;                                        */
/*   * level-1 cells [2 pi j / 2^b, 2 pi (j+1) / 2^b), reconstructed at     */
/*     their centres;                                                        */
/*   * the quantizer decisions are taken in f32 without computing an angle: */
/*     psi > t  <=>  hi * (float)cos t > lo * (float)sin t (products rounded */
/*     once each), after turning a level-1 pair into its quadrant by exact  */
/*     sign swaps; a tie goes to the lower cell and a zero pair to code 0;  */
/*   * radii as sqrtf(lo*lo + hi*hi), each operation rounded in f32.        */
/* The pages' distortion figure for 4 bits (~0.147 rel-L2, [P1] "Why        */
/* rotated-int4") is not reproduced by this reading (0.120 on Gaussian rows):*/
/* it is reported, not pinned.  Pins: closed forms of the k = 2 and k = 3   */
/* codebooks, the angle densities against sampled Gaussian vectors, exact   */
/* round trips of the polar transform, and invariants of the codec.         */
/* ------------------------------------------------------------------------ */

#define PQ_MAX_LEVEL 10   /* blocks up to 1024 */
#define PQ_MAX_BITS 8

/* Gauss-Legendre nodes and weights on [-1, 1]: Newton's method on P_n from
 * the usual cosine starting points, P_n and P_n' by the three-term recurrence. */
#define GL_N 10
static double gl_x[GL_N], gl_w[GL_N];
static int gl_ready = 0;
static void gl_init(void)
{
    if (gl_ready) return;
    for (int i = 0; i < GL_N; ++i) {
        double x = cos(M_PI * (i + 0.75) / (GL_N + 0.5)), dp = 1.0;
        for (int it = 0; it < 100; ++it) {
            double p0 = 1.0, p1 = x;
            for (int j = 2; j <= GL_N; ++j) {
                double p2 = ((2.0 * j - 1.0) * x * p1 - (j - 1.0) * p0) / j;
                p0 = p1;
                p1 = p2;
            }
            dp = GL_N * (x * p1 - p0) / (x * x - 1.0);
            double dx = p1 / dp;
            x -= dx;
            if (fabs(dx) < 1e-16) break;
        }
        gl_x[i] = x;
        gl_w[i] = 2.0 / ((1.0 - x * x) * dp * dp);
    }
    gl_ready = 1;
}

/* density of a level-l angle (l >= 2), unnormalized: sin(2 psi)^(k-1) */
static double pq_density(double psi, int k)
{
    double s = sin(2.0 * psi);
    return s > 0.0 ? pow(s, (double)(k - 1)) : 0.0;
}

/* integrals of f and psi*f over [a, b] by one Gauss-Legendre rule */
static void gl_cell(double a, double b, int k, double* F, double* M)
{
    double h = 0.5 * (b - a), m = 0.5 * (a + b), f = 0.0, g = 0.0;
    for (int i = 0; i < GL_N; ++i) {
        double t = m + h * gl_x[i], d = pq_density(t, k) * gl_w[i];
        f += d;
        g += t * d;
    }
    *F = h * f;
    *M = h * g;
}

/* Integrals of f and psi*f over each of G equal panels of [0, pi/2]; the
 * integral over a cell [a, b] adds the panels inside it and one rule over
 * each part-panel at its ends (no differences of large cumulative sums, so
 * the far-tail cells keep their relative accuracy). */
#define PQ_GRID 16384
typedef struct { int k; double pf[PQ_GRID], pm[PQ_GRID]; } pq_panels;

static void pq_panels_build(pq_panels* c, int k)
{
    const double h = (M_PI / 2) / PQ_GRID;
    c->k = k;
    for (int i = 0; i < PQ_GRID; ++i) gl_cell(i * h, (i + 1) * h, k, &c->pf[i], &c->pm[i]);
}

static void pq_cell(const pq_panels* c, double a, double b, double* F, double* M)
{
    const double h = (M_PI / 2) / PQ_GRID;
    int ia = (int)(a / h), ib = (int)(b / h);
    if (ia > PQ_GRID - 1) ia = PQ_GRID - 1;
    if (ib > PQ_GRID) ib = PQ_GRID;
    if (ia >= ib) { gl_cell(a, b, c->k, F, M); return; }
    double f, m, sf, sm;
    gl_cell(a, (ia + 1) * h, c->k, &sf, &sm);
    for (int i = ia + 1; i < ib; ++i) { sf += c->pf[i]; sm += c->pm[i]; }
    if (ib < PQ_GRID && b > ib * h) {
        gl_cell(ib * h, b, c->k, &f, &m);
        sf += f;
        sm += m;
    }
    *F = sf;
    *M = sm;
}

/* Lloyd-Max quantizer with L levels for the level-l angle density (k =
 * 2^(l-1)): a fixed point of the two optimality conditions (thresholds at
 * the midpoints of adjacent levels, each level the centroid of its cell).
 * Lloyd's alternation from the quantiles of f^(1/3) brings the levels within
 * 1e-9 rad; Newton's method on the same conditions (a tridiagonal system:
 * centroid q moves with thresholds q-1 and q, d mu/d b = f(b)(b - mu)/mass)
 * then settles them.  Returns 0, or -1 if the residual stays above 1e-13. */
static int pq_lloyd(int k, int L, double* lv, double* th, double* mse_out)
{
    gl_init();
    pq_panels* c = (pq_panels*)malloc(sizeof(pq_panels));
    pq_panels_build(c, k);
    /* start: quantiles of f^(1/3), by the trapezoid rule on a fine grid */
    {
        const int G = 200000;
        double* cw = (double*)malloc(sizeof(double) * (G + 1));
        cw[0] = 0.0;
        double prev = 0.0;
        for (int i = 1; i <= G; ++i) {
            double t = (M_PI / 2) * i / G, w = cbrt(pq_density(t, k));
            cw[i] = cw[i - 1] + 0.5 * (prev + w);
            prev = w;
        }
        int j = 0;
        for (int q = 0; q < L; ++q) {
            double target = cw[G] * (q + 0.5) / L;
            while (j < G && cw[j + 1] < target) ++j;
            double frac = (target - cw[j]) / (cw[j + 1] - cw[j]);
            lv[q] = (M_PI / 2) * (j + frac) / G;
        }
        free(cw);
    }
    double* mass = (double*)malloc(sizeof(double) * (size_t)L);
    double* mu = (double*)malloc(sizeof(double) * (size_t)L);
    double* dl = (double*)malloc(sizeof(double) * (size_t)L);
    double* dd = (double*)malloc(sizeof(double) * (size_t)L);
    double* du = (double*)malloc(sizeof(double) * (size_t)L);
    double* rhs = (double*)malloc(sizeof(double) * (size_t)L);
    int ok = 0;
    for (int it = 0; it < 200000; ++it) {           /* Lloyd */
        double move = 0.0;
        for (int q = 0; q + 1 < L; ++q) th[q] = 0.5 * (lv[q] + lv[q + 1]);
        for (int q = 0; q < L; ++q) {
            double F, M;
            pq_cell(c, q ? th[q - 1] : 0.0, q + 1 < L ? th[q] : M_PI / 2, &F, &M);
            double nv = M / F;
            if (fabs(nv - lv[q]) > move) move = fabs(nv - lv[q]);
            lv[q] = nv;
        }
        if (move <= 1e-9) break;
    }
    for (int it = 0; it < 60; ++it) {               /* Newton */
        for (int q = 0; q + 1 < L; ++q) th[q] = 0.5 * (lv[q] + lv[q + 1]);
        double resid = 0.0;
        for (int q = 0; q < L; ++q) {
            double F, M;
            pq_cell(c, q ? th[q - 1] : 0.0, q + 1 < L ? th[q] : M_PI / 2, &F, &M);
            mass[q] = F;
            mu[q] = M / F;
            rhs[q] = -(mu[q] - lv[q]);
            if (fabs(rhs[q]) > resid) resid = fabs(rhs[q]);
        }
        if (resid <= 1e-15) { ok = 1; break; }
        for (int q = 0; q < L; ++q) {
            double da = 0.0, db = 0.0;   /* d mu_q / d (lower, upper edge) */
            if (q > 0) da = pq_density(th[q - 1], k) * (mu[q] - th[q - 1]) / mass[q];
            if (q + 1 < L) db = pq_density(th[q], k) * (th[q] - mu[q]) / mass[q];
            dl[q] = 0.5 * da;
            du[q] = 0.5 * db;
            dd[q] = 0.5 * (da + db) - 1.0;
        }
        /* Thomas algorithm on (dl, dd, du) x = rhs */
        for (int q = 1; q < L; ++q) {
            double w = dl[q] / dd[q - 1];
            dd[q] -= w * du[q - 1];
            rhs[q] -= w * rhs[q - 1];
        }
        rhs[L - 1] /= dd[L - 1];
        for (int q = L - 2; q >= 0; --q) rhs[q] = (rhs[q] - du[q] * rhs[q + 1]) / dd[q];
        for (int q = 0; q < L; ++q) lv[q] += rhs[q];
        if (it == 59 && resid <= 1e-13) ok = 1;
    }
    for (int q = 0; q + 1 < L; ++q) th[q] = 0.5 * (lv[q] + lv[q + 1]);
    free(rhs); free(du); free(dd); free(dl); free(mu); free(mass);
    if (mse_out) {
        /* E[(psi - level)^2] over the normalized density, cell by cell */
        double tot = 0.0, z = 0.0;
        for (int i = 0; i < PQ_GRID; ++i) z += c->pf[i];
        for (int q = 0; q < L; ++q) {
            double a = q ? th[q - 1] : 0.0, b = q + 1 < L ? th[q] : M_PI / 2;
            const int S = 64;
            for (int s = 0; s < S; ++s) {
                double lo = a + (b - a) * s / S, hi = a + (b - a) * (s + 1) / S, hh = 0.5 * (hi - lo),
                       mm = 0.5 * (hi + lo), acc = 0.0;
                for (int i = 0; i < GL_N; ++i) {
                    double t = mm + hh * gl_x[i];
                    acc += gl_w[i] * pq_density(t, k) * (t - lv[q]) * (t - lv[q]);
                }
                tot += hh * acc;
            }
        }
        *mse_out = tot / z;
    }
    free(c);
    return ok ? 0 : -1;
}

/* The codebook of one level and width, memoized: centroids (2^b) and
 * thresholds (2^b - 1) in radians.  Level 1: uniform cells of the circle. */
static double pq_books_lv[PQ_MAX_LEVEL + 1][PQ_MAX_BITS + 1][1 << PQ_MAX_BITS];
static double pq_books_th[PQ_MAX_LEVEL + 1][PQ_MAX_BITS + 1][1 << PQ_MAX_BITS];
static double pq_books_mse[PQ_MAX_LEVEL + 1][PQ_MAX_BITS + 1];
static int pq_books_have[PQ_MAX_LEVEL + 1][PQ_MAX_BITS + 1];

int kvqo_pq_codebook(int level, int bits, double* centroids, double* thresholds, double* mse)
{
    if (level < 1 || level > PQ_MAX_LEVEL || bits < 1 || bits > PQ_MAX_BITS) return KVQO_ERR_ARG;
    const int L = 1 << bits;
    if (!pq_books_have[level][bits]) {
        double* lv = pq_books_lv[level][bits];
        double* th = pq_books_th[level][bits];
        if (level == 1) {
            const double step = 2.0 * M_PI / L;
            for (int q = 0; q < L; ++q) lv[q] = (q + 0.5) * step;
            for (int q = 1; q < L; ++q) th[q - 1] = q * step;
            pq_books_mse[level][bits] = step * step / 12.0;
        } else if (pq_lloyd(1 << (level - 1), L, lv, th, &pq_books_mse[level][bits]) < 0) {
            return KVQO_ERR_ARG;
        }
        pq_books_have[level][bits] = 1;
    }
    if (centroids) memcpy(centroids, pq_books_lv[level][bits], sizeof(double) * (size_t)L);
    if (thresholds) memcpy(thresholds, pq_books_th[level][bits], sizeof(double) * (size_t)(L - 1));
    if (mse) *mse = pq_books_mse[level][bits];
    return KVQO_OK;
}

static int ilog2(int n) { int l = 0; while ((1 << l) < n) ++l; return l; }

/* Bytes of one block's angle stream and of a whole row. */
int64_t kvqo_pq_block_bytes(int n, int bits) { return ((int64_t)n * bits + 7) / 8; }
int64_t kvqo_pq_row_bytes(int n_blocks, const int* bdims, int bits)
{
    int64_t s = 0;
    for (int b = 0; b < n_blocks; ++b) s += kvqo_pq_block_bytes(bdims[b], bits);
    return s;
}

/* The f32 decision tables: for level 1 the 2^(b-2) - 1 in-quadrant
 * thresholds j pi / 2^(b-1) (j >= 1), for level l >= 2 the codebook's
 * thresholds; each as the f32 roundings of its cosine and sine. */
static int pq_decision_table(int level, int bits, float* ct, float* st)
{
    if (level == 1) {
        const int nq = (1 << bits) / 4;
        for (int j = 1; j < nq; ++j) {
            double t = j * M_PI / (1 << (bits - 1));
            ct[j - 1] = (float)cos(t);
            st[j - 1] = (float)sin(t);
        }
        return nq - 1;
    }
    double th[1 << PQ_MAX_BITS];
    if (kvqo_pq_codebook(level, bits, NULL, th, NULL) != KVQO_OK) return -1;
    for (int j = 0; j + 1 < (1 << bits); ++j) {
        ct[j] = (float)cos(th[j]);
        st[j] = (float)sin(th[j]);
    }
    return (1 << bits) - 1;
}

int kvqo_pq_decision_table(int level, int bits, float* ct, float* st)
{
    return pq_decision_table(level, bits, ct, st);
}

/* number of thresholds t with psi > t, psi the angle of (lo, hi) in [0, pi/2] */
static unsigned pq_count(float lo, float hi, const float* ct, const float* st, int n_th)
{
    unsigned c = 0;
    for (int j = 0; j < n_th; ++j)
        if (hi * ct[j] > lo * st[j]) ++c;
    return c;
}

/* code of a level-1 pair (a, c): quadrant by exact sign swaps, then the
 * in-quadrant cells */
static unsigned pq_code1(float a, float c, int bits, const float* ct, const float* st, int n_th)
{
    unsigned q;
    float u, w;
    if (a > 0.0f && c >= 0.0f)      { q = 0; u = a;  w = c;  }
    else if (a <= 0.0f && c > 0.0f) { q = 1; u = c;  w = -a; }
    else if (a < 0.0f && c <= 0.0f) { q = 2; u = -a; w = -c; }
    else if (a >= 0.0f && c < 0.0f) { q = 3; u = -c; w = a;  }
    else return 0;                                   /* a zero pair */
    return q * (unsigned)(1 << (bits - 2)) + pq_count(u, w, ct, st, n_th);
}

static void put_bits(uint8_t* s, int64_t pos, unsigned v, int bits)
{
    for (int i = 0; i < bits; ++i)
        if ((v >> i) & 1u) s[(pos + i) >> 3] |= (uint8_t)(1u << ((pos + i) & 7));
}

static unsigned get_bits(const uint8_t* s, int64_t pos, int bits)
{
    unsigned v = 0;
    for (int i = 0; i < bits; ++i) v |= (unsigned)((s[(pos + i) >> 3] >> ((pos + i) & 7)) & 1u) << i;
    return v;
}

/* Encode.  codes [n_rows][row_bytes], radii [n_rows][n_blocks] f32.  A block
 * whose radius is not finite (a NaN or infinite input, or squares past the
 * f32 range) makes the call return KVQO_NONFINITE; its codes are then
 * whatever the steps gave, and the other rows are encoded as usual. */
#define KVQO_NONFINITE 3
int kvqo_pq_encode(const float* x, int64_t n_rows, int n_blocks, const int* bdims, uint64_t seed, int bits,
                   uint8_t* codes, float* radii)
{
    if (n_blocks < 1 || n_blocks > 8 || bits < 2 || bits > 6) return KVQO_ERR_ARG;
    for (int b = 0; b < n_blocks; ++b)
        if (!is_pow2_ge2(bdims[b]) || bdims[b] > (1 << PQ_MAX_LEVEL)) return KVQO_ERR_SHAPE;
    const int D = row_dim(n_blocks, bdims);
    const int64_t RB = kvqo_pq_row_bytes(n_blocks, bdims, bits);
    int8_t* sigma = (int8_t*)malloc((size_t)D);
    float* v = (float*)malloc(sizeof(float) * (size_t)D);
    float* rad = (float*)malloc(sizeof(float) * (size_t)D);
    float ct[PQ_MAX_LEVEL + 1][1 << 6], st[PQ_MAX_LEVEL + 1][1 << 6];
    int nth[PQ_MAX_LEVEL + 1];
    int maxl = 0;
    for (int b = 0; b < n_blocks; ++b) if (ilog2(bdims[b]) > maxl) maxl = ilog2(bdims[b]);
    for (int l = 1; l <= maxl; ++l) {
        nth[l] = pq_decision_table(l, bits, ct[l], st[l]);
        if (nth[l] < 0) { free(rad); free(v); free(sigma); return KVQO_ERR_ARG; }
    }
    kvqo_tq4_signs(seed, n_blocks, bdims, sigma);
    int status = KVQO_OK;
    memset(codes, 0, (size_t)(RB * n_rows));
    for (int64_t t = 0; t < n_rows; ++t) {
        const float* xr = x + t * D;
        uint8_t* cr = codes + t * RB;
        int off = 0;
        int64_t boff = 0;
        for (int b = 0; b < n_blocks; ++b) {
            const int n = bdims[b], L = ilog2(n);
            const float kn = (float)(1.0 / sqrt((double)n));
            for (int i = 0; i < n; ++i) v[i] = sigma[off + i] < 0 ? -xr[off + i] : xr[off + i];
            kvqo_fwht_f32(v, n);
            for (int i = 0; i < n; ++i) v[i] = v[i] * kn;
            uint8_t* s = cr + boff;
            int64_t pos = 0;
            /* level 1 */
            for (int j = 0; j < n / 2; ++j) {
                const float a = v[2 * j], c = v[2 * j + 1];
                put_bits(s, pos, pq_code1(a, c, bits, ct[1], st[1], nth[1]), bits);
                pos += bits;
                rad[j] = sqrtf(a * a + c * c);
            }
            /* levels 2 .. L */
            for (int l = 2, m = n / 4; l <= L; ++l, m /= 2) {
                for (int j = 0; j < m; ++j) {
                    const float lo = rad[2 * j], hi = rad[2 * j + 1];
                    put_bits(s, pos, pq_count(lo, hi, ct[l], st[l], nth[l]), bits);
                    pos += bits;
                    rad[j] = sqrtf(lo * lo + hi * hi);
                }
            }
            radii[t * n_blocks + b] = rad[0];
            if (!isfinite(rad[0])) status = KVQO_NONFINITE;
            off += n;
            boff += kvqo_pq_block_bytes(n, bits);
        }
    }
    free(rad);
    free(v);
    free(sigma);
    return status;
}

/* Reconstruction in binary64 from the centroids: y_hat by the tree from R
 * down, then (unless rotated != 0) x_hat = unrotate(y_hat). */
int kvqo_pq_decode(const uint8_t* codes, const float* radii, int64_t n_rows, int n_blocks, const int* bdims,
                   uint64_t seed, int bits, int rotated, double* xhat)
{
    if (n_blocks < 1 || n_blocks > 8 || bits < 2 || bits > 6) return KVQO_ERR_ARG;
    for (int b = 0; b < n_blocks; ++b)
        if (!is_pow2_ge2(bdims[b]) || bdims[b] > (1 << PQ_MAX_LEVEL)) return KVQO_ERR_SHAPE;
    const int D = row_dim(n_blocks, bdims);
    const int64_t RB = kvqo_pq_row_bytes(n_blocks, bdims, bits);
    double* y = (double*)malloc(sizeof(double) * (size_t)D);
    double* r = (double*)malloc(sizeof(double) * (size_t)D);
    double* nx = (double*)malloc(sizeof(double) * (size_t)D);
    double lv[PQ_MAX_LEVEL + 1][1 << 6];
    int maxl = 0;
    for (int b = 0; b < n_blocks; ++b) if (ilog2(bdims[b]) > maxl) maxl = ilog2(bdims[b]);
    for (int l = 1; l <= maxl; ++l)
        if (kvqo_pq_codebook(l, bits, lv[l], NULL, NULL) != KVQO_OK) { free(nx); free(r); free(y); return KVQO_ERR_ARG; }
    for (int64_t t = 0; t < n_rows; ++t) {
        const uint8_t* cr = codes + t * RB;
        int off = 0;
        int64_t boff = 0;
        for (int b = 0; b < n_blocks; ++b) {
            const int n = bdims[b], L = ilog2(n);
            const uint8_t* s = cr + boff;
            /* stream offset (in angles) of each level's first angle */
            int64_t first[PQ_MAX_LEVEL + 2];
            first[1] = 0;
            for (int l = 2; l <= L; ++l) first[l] = first[l - 1] + (n >> (l - 1));
            r[0] = (double)radii[t * n_blocks + b];
            for (int l = L, m = 1; l >= 2; --l, m *= 2) {
                for (int j = 0; j < m; ++j) {
                    const double psi = lv[l][get_bits(s, (first[l] + j) * bits, bits)];
                    nx[2 * j] = r[j] * cos(psi);
                    nx[2 * j + 1] = r[j] * sin(psi);
                }
                memcpy(r, nx, sizeof(double) * (size_t)(2 * m));
            }
            for (int j = 0; j < n / 2; ++j) {
                const double psi = lv[1][get_bits(s, j * bits, bits)];
                y[off + 2 * j] = r[j] * cos(psi);
                y[off + 2 * j + 1] = r[j] * sin(psi);
            }
            off += n;
            boff += kvqo_pq_block_bytes(n, bits);
        }
        if (rotated) memcpy(xhat + t * D, y, sizeof(double) * (size_t)D);
        else kvqo_tq4_rotate(y, xhat + t * D, 1, n_blocks, bdims, seed, 1);
    }
    free(nx);
    free(r);
    free(y);
    return KVQO_OK;
}

/* The polar transform itself in binary64, without quantization: angles
 * (level 1 first, n - 1 of them, level-1 angles in [0, 2 pi)) and the radius
 * of each block of v, and its inverse.  Test support for the round trips. */
int kvqo_polar_forward(const double* v, int n, double* angles, double* radius)
{
    if (!is_pow2_ge2(n) || n > (1 << PQ_MAX_LEVEL)) return KVQO_ERR_SHAPE;
    double* r = (double*)malloc(sizeof(double) * (size_t)n);
    int64_t pos = 0;
    for (int j = 0; j < n / 2; ++j) {
        double a = atan2(v[2 * j + 1], v[2 * j]);
        angles[pos++] = a < 0.0 ? a + 2.0 * M_PI : a;
        r[j] = sqrt(v[2 * j] * v[2 * j] + v[2 * j + 1] * v[2 * j + 1]);
    }
    for (int m = n / 4; m >= 1; m /= 2) {
        for (int j = 0; j < m; ++j) {
            angles[pos++] = atan2(r[2 * j + 1], r[2 * j]);
            r[j] = sqrt(r[2 * j] * r[2 * j] + r[2 * j + 1] * r[2 * j + 1]);
        }
    }
    *radius = r[0];
    free(r);
    return KVQO_OK;
}

int kvqo_polar_inverse(const double* angles, double radius, int n, double* v)
{
    if (!is_pow2_ge2(n) || n > (1 << PQ_MAX_LEVEL)) return KVQO_ERR_SHAPE;
    double* r = (double*)malloc(sizeof(double) * (size_t)n);
    double* nx = (double*)malloc(sizeof(double) * (size_t)n);
    int L = ilog2(n);
    int64_t first[PQ_MAX_LEVEL + 2];
    first[1] = 0;
    for (int l = 2; l <= L; ++l) first[l] = first[l - 1] + (n >> (l - 1));
    r[0] = radius;
    for (int l = L, m = 1; l >= 2; --l, m *= 2) {
        for (int j = 0; j < m; ++j) {
            nx[2 * j] = r[j] * cos(angles[first[l] + j]);
            nx[2 * j + 1] = r[j] * sin(angles[first[l] + j]);
        }
        memcpy(r, nx, sizeof(double) * (size_t)(2 * m));
    }
    for (int j = 0; j < n / 2; ++j) {
        v[2 * j] = r[j] * cos(angles[j]);
        v[2 * j + 1] = r[j] * sin(angles[j]);
    }
    free(nx);
    free(r);
    return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* Softmax attention over reconstructed rows, the plain definition:          */
/*   z_t = sm_scale * sum_i q_i K_t,i;  p_t = exp(z_t - max z);              */
/*   o_d = sum_t p_t V_t,d / sum_t p_t                                       */
/* in binary64.  For the MLA latent cache K and V are the same rows: K uses  */
/* all 576 dims (latent + rope), V the leading 512 ([P1] "Why rotated-int4": */
/* MLA's latent is both key and value).  An empty row range gives zeros.     */
/* ------------------------------------------------------------------------ */
int kvqo_attn_dense(const double* K, int64_t ldk, int dk, const double* V, int64_t ldv, int dv,
                    int64_t n_rows, const float* q, int n_q, double sm_scale, double* out)
{
    double* z = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    for (int j = 0; j < n_q; ++j) {
        const float* qj = q + (int64_t)j * dk;
        double* oj = out + (int64_t)j * dv;
        for (int d = 0; d < dv; ++d) oj[d] = 0.0;
        if (n_rows == 0) continue;
        double m = -INFINITY;
        for (int64_t t = 0; t < n_rows; ++t) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += (double)qj[i] * K[t * ldk + i];
            z[t] = sm_scale * acc;
            if (z[t] > m) m = z[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < n_rows; ++t) {
            double p = exp(z[t] - m);
            l += p;
            for (int d = 0; d < dv; ++d) oj[d] += p * V[t * ldv + d];
        }
        for (int d = 0; d < dv; ++d) oj[d] /= l;
    }
    free(z);
    return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* The consumers' own arithmetic, for the identity checks only.  [P2]       */
/* "What's in it": KV8 decodes codes inline and factors the row scale out of */
/* the score and context sums; TQ4 rotates the query once, dots it with the  */
/* scaled codebook levels, accumulates the context in the rotated domain and */
/* unrotates it once ([P1] "Ready for review" comment, finding 2:            */
/* q.x_hat == rotate(q).c and sum w x_hat == unrotate(sum w c)).             */
/* fmt: 1 = KV8, 2 = TQ4.                                                    */
/* ------------------------------------------------------------------------ */
int kvqo_attn_method(int fmt, int n_blocks, const int* bdims, uint64_t seed, int v_dim,
                     const uint8_t* codes, const float* scales, int64_t n_rows,
                     const float* q, int n_q, double sm_scale, double* out)
{
    int D = row_dim(n_blocks, bdims);
    int row_bytes = fmt == 1 ? D : D / 2;
    float lv[16], th[15];
    if (v_dim > bdims[0]) return KVQO_ERR_ARG;              /* context lives in the first block */
    if (fmt == 2) {
        for (int b = 0; b < n_blocks; ++b)
            if (!is_pow2_ge2(bdims[b])) return KVQO_ERR_SHAPE;
        kvqo_tq4_codebook(lv, th);
    }
    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    double* qr = (double*)malloc(sizeof(double) * (size_t)D);
    double* z = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    double* unit = (double*)malloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < n_q; ++j) {
        double* oj = out + (int64_t)j * v_dim;
        for (int i = 0; i < D; ++i) qd[i] = (double)q[(int64_t)j * D + i];
        if (fmt == 2) kvqo_tq4_rotate(qd, qr, 1, n_blocks, bdims, seed, 0);
        else memcpy(qr, qd, sizeof(double) * (size_t)D);
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        if (n_rows == 0) { for (int d = 0; d < v_dim; ++d) oj[d] = 0.0; continue; }
        double m = -INFINITY;
        for (int64_t t = 0; t < n_rows; ++t) {
            const uint8_t* cr = codes + t * row_bytes;
            double zt = 0.0;
            int off = 0;
            for (int b = 0; b < n_blocks; ++b) {
                double part = 0.0;
                for (int i = off; i < off + bdims[b]; ++i) {
                    double v = fmt == 1 ? kvqo_e4m3_value(cr[i])
                                        : (double)lv[(i & 1) ? (cr[i / 2] >> 4) : (cr[i / 2] & 15u)];
                    part += qr[i] * v;
                }
                zt += (double)scales[t * n_blocks + b] * part;
                off += bdims[b];
            }
            z[t] = sm_scale * zt;
            if (z[t] > m) m = z[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < n_rows; ++t) {
            const uint8_t* cr = codes + t * row_bytes;
            double p = exp(z[t] - m);
            double w = p * (double)scales[t * n_blocks + 0];
            l += p;
            for (int d = 0; d < v_dim; ++d) {
                double v = fmt == 1 ? kvqo_e4m3_value(cr[d])
                                    : (double)lv[(d & 1) ? (cr[d / 2] >> 4) : (cr[d / 2] & 15u)];
                acc[d] += w * v;
            }
        }
        if (fmt == 2) {
            for (int d = 0; d < D; ++d) unit[d] = d < v_dim ? acc[d] / l : 0.0;
            kvqo_tq4_rotate(unit, acc, 1, n_blocks, bdims, seed, 1);
            for (int d = 0; d < v_dim; ++d) oj[d] = acc[d];
        } else {
            for (int d = 0; d < v_dim; ++d) oj[d] = acc[d] / l;
        }
    }
    free(unit);
    free(acc);
    free(z);
    free(qr);
    free(qd);
    return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* K2/V4 GQA codec with the FP16 window + sink overlay of [P3].              */
/*   K: 2 bits per element, one scale per (kv head, dim, 32-cell group):     */
/*      s_rule = sqrt(sum of squares over the 32 cells / 32) (fixed order as */
/*      sumsq_r32), code = number of 4-level thresholds below x / s_rule,    */
/*      stored scale = fp16(k_gain * s_rule) with the f32 product first      */
/*      ([P3] Summary item 3 and "Measurements - Gate": stored scale = B x   */
/*      the rule, codes chosen against the un-gained scale).                 */
/*      Packing (pages silent): dim d of a cell is bits 2(d%4) of byte d/4.  */
/*   V: q4_0 per token, blocks of 32 dims: 2-byte fp16 d then 16 bytes;      */
/*      value = (code - 8) * d; element j < 16 is the low nibble of byte j,  */
/*      element j >= 16 the high nibble of byte j-16 (the parity listing of  */
/*      [P3]).  Encoder (pages show only the decode): m = the first element  */
/*      of largest magnitude, d = m / -8 in f32, code = min(15, trunc(x/d +  */
/*      8.5)); an all-zero block stores d = 0 and codes 8.                   */
/*   Overlay: fp16 copies of K and V for cells < n_sink and >= T - n_window. */
/*      Slot of a cell: c < n_sink -> c; window -> n_sink + c mod (n_window + */
/*      n_slack); else none.  ([P3] Summary item 1: window + sinks + 16      */
/*      slack slots.)                                                        */
/* Layouts (per sequence; the caller offsets by sequence):                   */
/*   k_codes [Hkv][cap][D/4]   k_scales [Hkv][cap/32][D] (fp16 bits)         */
/*   v_blocks [Hkv][cap][D/32][18]   k_win, v_win [Hkv][slots][D] (fp16)     */
/* ------------------------------------------------------------------------ */
typedef struct {
    int32_t n_kv_heads, head_dim, group;
    float k_gain;
    int32_t n_sink, n_window, n_slack;
} kvqo_k2v4_layout;

int64_t kvqo_k2v4_slot(int64_t cell, int64_t T, const kvqo_k2v4_layout* L)
{
    if (cell < L->n_sink) return cell;
    if (cell >= T - L->n_window) return L->n_sink + cell % (L->n_window + L->n_slack);
    return -1;
}

/* One q4_0 block of 32 values -> 18 bytes (fp16 d, then 16 bytes of nibbles). */
static void v4_encode_block(const float* xb, uint8_t* out)
{
    float m = 0.0f;
    for (int j = 0; j < 32; ++j)
        if (fabsf(xb[j]) > fabsf(m)) m = xb[j];
    float d = m / -8.0f;
    unsigned dh = kvqo_f16_encode(d);
    out[0] = (uint8_t)(dh & 255u);
    out[1] = (uint8_t)(dh >> 8);
    for (int j = 0; j < 16; ++j) out[2 + j] = 0;
    for (int j = 0; j < 32; ++j) {
        unsigned code = 8;
        if (d != 0.0f) {
            int c = (int)(xb[j] / d + 8.5f);
            code = (unsigned)(c > 15 ? 15 : c);
        }
        if (j < 16) out[2 + j] = (uint8_t)(out[2 + j] | code);
        else        out[2 + j - 16] = (uint8_t)(out[2 + j - 16] | (code << 4));
    }
}

int kvqo_k2v4_encode(const float* k, const float* v, int64_t T, int64_t cap, const kvqo_k2v4_layout* L,
                     uint8_t* k_codes, uint16_t* k_scales, uint8_t* v_blocks, uint16_t* k_win, uint16_t* v_win)
{
    const int H = L->n_kv_heads, D = L->head_dim, G = L->group;
    if (G != 32 || D % 32 != 0 || T % G != 0 || cap < T || cap % G != 0) return KVQO_ERR_SHAPE;
    float lv[4], th[3];
    kvqo_k2_codebook(lv, th);
    const int slots = L->n_sink + L->n_window + L->n_slack;
    for (int h = 0; h < H; ++h) {
        const float* kh = k + (int64_t)h * T * D;
        const float* vh = v + (int64_t)h * T * D;
        for (int64_t g = 0; g < T / G; ++g) {
            for (int d = 0; d < D; ++d) {
                const float* col = kh + g * G * D + d;          /* 32 cells of one channel */
                float ss = sumsq_r32(col, G, D);
                float mean = ss / 32.0f;
                float s_rule = sqrtf(mean);
                float gained = L->k_gain * s_rule;
                k_scales[((int64_t)h * (cap / G) + g) * D + d] = (uint16_t)kvqo_f16_encode(gained);
                for (int j = 0; j < G; ++j) {
                    int64_t cell = g * G + j;
                    unsigned code = 0;
                    if (s_rule != 0.0f) code = code_of(col[(int64_t)j * D] / s_rule, th, 3);
                    uint8_t* byte = k_codes + ((int64_t)h * cap + cell) * (D / 4) + d / 4;
                    if (d % 4 == 0) *byte = 0;
                    *byte = (uint8_t)(*byte | (code << (2 * (d % 4))));
                }
            }
        }
        for (int64_t cell = 0; cell < T; ++cell) {
            const float* vr = vh + cell * D;
            for (int blk = 0; blk < D / 32; ++blk)
                v4_encode_block(vr + blk * 32, v_blocks + (((int64_t)h * cap + cell) * (D / 32) + blk) * 18);
            int64_t slot = kvqo_k2v4_slot(cell, T, L);
            if (slot >= 0) {
                for (int d = 0; d < D; ++d) {
                    k_win[((int64_t)h * slots + slot) * D + d] = (uint16_t)kvqo_f16_encode(kh[cell * D + d]);
                    v_win[((int64_t)h * slots + slot) * D + d] = (uint16_t)kvqo_f16_encode(vr[d]);
                }
            }
        }
    }
    return KVQO_OK;
}

/* Append of n_new cells at positions T_old .. T_old + n_new - 1 of one
 * sequence (k_new, v_new are [Hkv][n_new][D]); the engine's append patterns of
 * [P3] ("Attention error under the engine's append patterns": decode appends,
 * speculative-verify windows, prefill chunks that fall mid-group) and its
 * "Review fixes" item "Fresh partial-group scale".  The K scale of a group:
 *   - first written by this append (fresh) with all 32 cells present: the
 *     encoder's rule, sqrt(ss / 32);
 *   - fresh with n < 32 cells present: sqrt((ss + (32 - n) * prev^2) / 32):
 *     ss the sum of squares of the n cells (the encoder's fixed order, absent
 *     cells as zero), prev the previous group's rule scale recovered from its
 *     stored fp16 value as f16(stored) / k_gain, the same whether that group
 *     was stored by an earlier call or in this one (reading: the pages have
 *     prev recomputed in the same launch or read from storage, bit-exact
 *     either way, and standing in for the previous group's mean square, i.e.
 *     in the rule's un-gained units); f32 evaluation left to right:
 *     prev * prev, times (32 - n), plus ss, over 32, square root;
 *   - fresh with n < 32 cells and no previous group (group 0): sqrt(ss / n),
 *     the RMS of the cells present (reading: the /n rule the pages state
 *     before the shrink toward prev);
 *   - a group that already holds cells from an earlier call: its stored scale
 *     is kept, the new cells are coded against f16(stored) / k_gain (reading:
 *     the pages define the rule for a group first written by a partial batch).
 * V blocks and the fp16 overlay of each new cell as in the encoder, with the
 * window taken at T = T_old + n_new. */
int kvqo_k2v4_append(const float* k_new, const float* v_new, int64_t T_old, int64_t n_new, int64_t cap,
                     const kvqo_k2v4_layout* L, uint8_t* k_codes, uint16_t* k_scales, uint8_t* v_blocks,
                     uint16_t* k_win, uint16_t* v_win)
{
    const int H = L->n_kv_heads, D = L->head_dim, G = L->group;
    if (G != 32 || D % 32 != 0 || cap % G != 0) return KVQO_ERR_SHAPE;
    if (T_old < 0 || n_new < 0 || T_old + n_new > cap) return KVQO_ERR_ARG;
    const int64_t T_new = T_old + n_new;
    float lv[4], th[3];
    kvqo_k2_codebook(lv, th);
    const int slots = L->n_sink + L->n_window + L->n_slack;
    for (int h = 0; h < H; ++h) {
        const float* kh = k_new + (int64_t)h * n_new * D;
        const float* vh = v_new + (int64_t)h * n_new * D;
        for (int64_t g = T_old / G; n_new > 0 && g <= (T_new - 1) / G; ++g) {
            const int64_t g0 = g * G;
            const int fresh = g0 >= T_old;
            const int64_t c0 = g0 > T_old ? g0 : T_old;                /* first new cell of the group */
            const int64_t c1 = g0 + G < T_new ? g0 + G : T_new;        /* one past the last */
            for (int d = 0; d < D; ++d) {
                uint16_t* sc = k_scales + ((int64_t)h * (cap / G) + g) * D + d;
                float s_rule;
                if (fresh) {
                    const int n = (int)(c1 - c0);
                    const float ss = sumsq_r32(kh + (c0 - T_old) * D + d, n, D);
                    if (n == G) {
                        s_rule = sqrtf(ss / 32.0f);
                    } else if (g == 0) {
                        s_rule = sqrtf(ss / (float)n);
                    } else {
                        const float prev = (float)kvqo_f16_value(sc[-D]) / L->k_gain;
                        const float prev2 = prev * prev;
                        const float add = (float)(G - n) * prev2;
                        const float num = ss + add;
                        s_rule = sqrtf(num / 32.0f);
                    }
                    *sc = (uint16_t)kvqo_f16_encode(L->k_gain * s_rule);
                } else {
                    s_rule = (float)kvqo_f16_value(*sc) / L->k_gain;
                }
                for (int64_t cell = c0; cell < c1; ++cell) {
                    unsigned code = 0;
                    if (s_rule != 0.0f) code = code_of(kh[(cell - T_old) * D + d] / s_rule, th, 3);
                    uint8_t* byte = k_codes + ((int64_t)h * cap + cell) * (D / 4) + d / 4;
                    if (d % 4 == 0) *byte = 0;
                    *byte = (uint8_t)(*byte | (code << (2 * (d % 4))));
                }
            }
        }
        for (int64_t cell = T_old; cell < T_new; ++cell) {
            const float* vr = vh + (cell - T_old) * D;
            for (int blk = 0; blk < D / 32; ++blk)
                v4_encode_block(vr + blk * 32, v_blocks + (((int64_t)h * cap + cell) * (D / 32) + blk) * 18);
            int64_t slot = kvqo_k2v4_slot(cell, T_new, L);
            if (slot >= 0) {
                for (int d = 0; d < D; ++d) {
                    k_win[((int64_t)h * slots + slot) * D + d] = (uint16_t)kvqo_f16_encode(kh[(cell - T_old) * D + d]);
                    v_win[((int64_t)h * slots + slot) * D + d] = (uint16_t)kvqo_f16_encode(vr[d]);
                }
            }
        }
    }
    return KVQO_OK;
}

/* What a reader sees for every cell: the overlay's fp16 value for sink and
 * window cells, the bulk's dequantization otherwise.  K_hat, V_hat are
 * [Hkv][T][D] in binary64.  use_overlay = 0 gives the bulk alone. */
int kvqo_k2v4_reconstruct(const uint8_t* k_codes, const uint16_t* k_scales, const uint8_t* v_blocks,
                          const uint16_t* k_win, const uint16_t* v_win, int64_t T, int64_t cap,
                          const kvqo_k2v4_layout* L, int use_overlay, double* K_hat, double* V_hat)
{
    const int H = L->n_kv_heads, D = L->head_dim, G = L->group;
    if (G != 32 || D % 32 != 0 || cap < T || cap % G != 0) return KVQO_ERR_SHAPE;
    float lv[4], th[3];
    kvqo_k2_codebook(lv, th);
    const int slots = L->n_sink + L->n_window + L->n_slack;
    for (int h = 0; h < H; ++h)
        for (int64_t cell = 0; cell < T; ++cell) {
            int64_t slot = use_overlay ? kvqo_k2v4_slot(cell, T, L) : -1;
            double* kr = K_hat + ((int64_t)h * T + cell) * D;
            double* vr = V_hat + ((int64_t)h * T + cell) * D;
            for (int d = 0; d < D; ++d) {
                if (slot >= 0) {
                    kr[d] = kvqo_f16_value(k_win[((int64_t)h * slots + slot) * D + d]);
                    vr[d] = kvqo_f16_value(v_win[((int64_t)h * slots + slot) * D + d]);
                    continue;
                }
                unsigned byte = k_codes[((int64_t)h * cap + cell) * (D / 4) + d / 4];
                unsigned code = (byte >> (2 * (d % 4))) & 3u;
                double sc = kvqo_f16_value(k_scales[((int64_t)h * (cap / G) + cell / G) * D + d]);
                kr[d] = (double)lv[code] * sc;
                const uint8_t* blk = v_blocks + (((int64_t)h * cap + cell) * (D / 32) + d / 32) * 18;
                double dd = kvqo_f16_value((unsigned)blk[0] | ((unsigned)blk[1] << 8));
                int j = d % 32;
                unsigned vc = j < 16 ? (blk[2 + j] & 15u) : (blk[2 + j - 16] >> 4);
                vr[d] = ((double)vc - 8.0) * dd;
            }
        }
    return KVQO_OK;
}
