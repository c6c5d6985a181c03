/*
 * CPU oracle for the MACaQ W4A4 (MXFP4) linear layer -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this library.  The product path (the CUDA library) never does,
 * and the two share no code, table or constant.
 *
 * What it states, step by step, in plain loops:
 *
 *   balance scales   MACaQ page "What is MACaQ quantization", section "How
 *                    MACaQ works", step "Channel balancing": one scale per
 *                    input channel evens out channel magnitudes.  The rule
 *                    s_j = sqrt(max|Xc[:,j]| / max|W[:,j]|), clamped to
 *                    [1e-2, 1e2], is the plainest reading; activations are
 *                    divided by s, weights multiplied by s.
 *   block Hadamard   same section, step "A small Hadamard transform": a block
 *                    Hadamard rotation over 32 channels, with the inverse
 *                    folded into the weights so the output is unchanged
 *                    before rounding.  Normalised Sylvester order 32, applied
 *                    as butterflies at strides 1, 2, 4, 8, 16 and one multiply
 *                    by fp32(1/sqrt 32).
 *   64-wide variant  (page "Huawei MACaQ Is an Open-Source Model Quantizer",
 *                    section on the llama.cpp recipe: a Hadamard block of 32 or
 *                    64 channels.)  Sylvester order 64 as butterflies at strides
 *                    1 .. 32, then one multiply by 1/8; the MX blocks stay 32
 *                    wide, so one Hadamard block spans two of them.
 *   MXFP4 encode     same page, FAQ "What is W4A4 quantization": 4-bit floats
 *                    in blocks of 32 sharing one scale.  Scale exponent
 *                    floor(log2 amax) - 2 (E8M0), element grid E2M1
 *                    {0, 0.5, 1, 1.5, 2, 3, 4, 6}, round to nearest with ties
 *                    to the even code, saturating at 6.
 *   GEMM reference   Y = deq(A) . deq(W)^T accumulated in fp64.
 *
 *   SwiGLU input     (extension: the down projection of a gated MLP reads
 *                    h = SiLU(g) * u of the gate and up outputs g, u.)  Its
 *                    definition: the real value g * u / (1 + e^-g), rounded
 *                    once to bf16 (the value an unfused layer would store).
 *                    Evaluated here in fp64 with the C library's exp, then
 *                    rounded to bf16 directly (no intermediate fp32).  Next to
 *                    each result the oracle reports the other bf16 neighbour
 *                    wherever the exact value lies within 2^-20 (relative) of a
 *                    rounding boundary: an fp32 evaluation, whose error is below
 *                    2^-21 relative, may land on either side there.
 *
 *   MoE combine      (extension: the expert outputs of a token's top-k rows,
 *                    weighted by their routing probabilities, summed into the
 *                    token's output.)  Stated in fp32: a fused multiply-add
 *                    chain over the token's choices in order, from +0, then
 *                    one rounding to bf16.
 *
 *   Flip Refinement  (page "What is MACaQ quantization", section "How MACaQ
 *                    works", step "Flip Refinement": instead of plain round to
 *                    nearest, a Hessian-aware coordinate descent moves single
 *                    4-bit weight codes to an adjacent value when that lowers
 *                    the layer's error on calibration data.)  Stated in the
 *                    rotated space, where the layer output is A . Wt^T (A the
 *                    calibration rows through the activation transform, Wt the
 *                    weight rows through the weight transform, both fp32):
 *                    H = A^T A (+ damp on the diagonal), and for one weight row
 *                    the error E(q) = (Wt - q)^T H (Wt - q) of its dequantised
 *                    codes q.  With r = Wt - q and g = H r, moving q_k by D
 *                    changes E by D (D H_kk - 2 g_k); coordinates are visited
 *                    in order k = 0 .. K-1, `sweeps` times; the adjacent grid
 *                    value (one step down or up the signed E2M1 grid, scale
 *                    unchanged) with the larger strict decrease is taken (ties
 *                    to the lower one) and g absorbs the move, g -= D H[k, :].
 *                    All of it in fp32 with explicit fused multiply-adds in
 *                    the sums (sequential order) and single roundings
 *                    elsewhere: the codes depend on every bit of g.
 *
 * Precision: the transform is stated in fp32 (IEEE, round to nearest, no
 * contraction: build with -ffp-contract=off, no fast-math), because the
 * quantised codes depend on its exact bits.  The fp64 variant exists for the
 * fold identity (output unchanged before rounding).
 *
 * Parity pins live in tests/test_oracle_*.py: closed forms (Sylvester
 * entries, scipy's Hadamard, the fold identity), a brute-force argmin for the
 * rounding, E8M0 boundary cases and an independent numpy restatement.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- balance */

/* Per-channel balance scale from a calibration batch Xc [mc, k] and the
 * weight W [n, k] (both bf16 bits, row-major).  Column maxima are exact in
 * fp64; the ratio and square root are taken in fp64 and rounded once to fp32
 * after clamping.  A channel with zero weight gets the upper clamp (1e2), a
 * channel zero on both sides gets 1.  inv_s = 1/s in fp32. */
void oracle_balance_scales(const uint16_t *xc, int64_t mc, const uint16_t *w, int64_t n,
                           int64_t k, float *s, float *inv_s)
{
    for (int64_t j = 0; j < k; ++j) {
        double cx = 0.0, cw = 0.0;
        for (int64_t m = 0; m < mc; ++m) {
            double a = fabs((double)bf16_bits_to_f32(xc[m * k + j]));
            if (a > cx) cx = a;
        }
        for (int64_t r = 0; r < n; ++r) {
            double a = fabs((double)bf16_bits_to_f32(w[r * k + j]));
            if (a > cw) cw = a;
        }
        double r;
        if (cw == 0.0) {
            r = (cx == 0.0) ? 1.0 : 1e2;
        } else {
            r = sqrt(cx / cw);
            if (r < 1e-2) r = 1e-2;
            if (r > 1e2) r = 1e2;
        }
        s[j] = (float)r;
        inv_s[j] = 1.0f / s[j];
    }
}

/* ------------------------------------------------------- block Hadamard */

/* One 32-channel block: v <- H32 . v with H32 the Sylvester matrix, as five
 * butterfly stages (stride h = 1, 2, 4, 8, 16; pair (i, i+h) for bit h of i
 * clear becomes (a + b, a - b)), then the 1/sqrt(32) normalisation. */
static void fwht32_f32(float v[32])
{
    for (int h = 1; h < 32; h <<= 1) {
        for (int i = 0; i < 32; ++i) {
            if (i & h) continue;
            float a = v[i];
            float b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
    const float c = (float)(1.0 / sqrt(32.0));
    for (int i = 0; i < 32; ++i) v[i] = v[i] * c;
}

static void fwht32_f64(double v[32])
{
    for (int h = 1; h < 32; h <<= 1) {
        for (int i = 0; i < 32; ++i) {
            if (i & h) continue;
            double a = v[i];
            double b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
    const double c = 1.0 / sqrt(32.0);
    for (int i = 0; i < 32; ++i) v[i] = v[i] * c;
}

/* One 64-channel block: butterflies at strides 1, 2, 4, 8, 16, 32, then the
 * 1/sqrt(64) = 1/8 normalisation (an exact power of two). */
static void fwht64_f32(float v[64])
{
    for (int h = 1; h < 64; h <<= 1) {
        for (int i = 0; i < 64; ++i) {
            if (i & h) continue;
            float a = v[i];
            float b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
    for (int i = 0; i < 64; ++i) v[i] = v[i] * 0.125f;
}

static void fwht64_f64(double v[64])
{
    for (int h = 1; h < 64; h <<= 1) {
        for (int i = 0; i < 64; ++i) {
            if (i & h) continue;
            double a = v[i];
            double b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
    for (int i = 0; i < 64; ++i) v[i] = v[i] * 0.125;
}

/* The transform with a 64-channel Hadamard block (k % 64 == 0). */
void oracle_transform64_f32(const uint16_t *x, int64_t rows, int64_t k, const float *f, float *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 64; ++b) {
            float v[64];
            for (int i = 0; i < 64; ++i) {
                int64_t j = 64 * b + i;
                v[i] = bf16_bits_to_f32(x[r * k + j]) * f[j];
            }
            fwht64_f32(v);
            for (int i = 0; i < 64; ++i) y[r * k + 64 * b + i] = v[i];
        }
    }
}

void oracle_transform64_f64(const double *x, int64_t rows, int64_t k, const double *f, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 64; ++b) {
            double v[64];
            for (int i = 0; i < 64; ++i) {
                int64_t j = 64 * b + i;
                v[i] = x[r * k + j] * f[j];
            }
            fwht64_f64(v);
            for (int i = 0; i < 64; ++i) y[r * k + 64 * b + i] = v[i];
        }
    }
}

/* y = (x . diag(f)) . (I_{k/32} kron H32), fp32.  x: bf16 bits [rows, k];
 * f: [k] fp32 (1/s for activations, s for weights); y: [rows, k] fp32. */
void oracle_transform_f32(const uint16_t *x, int64_t rows, int64_t k, const float *f, float *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 32; ++b) {
            float v[32];
            for (int i = 0; i < 32; ++i) {
                int64_t j = 32 * b + i;
                v[i] = bf16_bits_to_f32(x[r * k + j]) * f[j];
            }
            fwht32_f32(v);
            for (int i = 0; i < 32; ++i) y[r * k + 32 * b + i] = v[i];
        }
    }
}

/* The same transform in fp64 on fp64 input (no rounding to fp32). */
void oracle_transform_f64(const double *x, int64_t rows, int64_t k, const double *f, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 32; ++b) {
            double v[32];
            for (int i = 0; i < 32; ++i) {
                int64_t j = 32 * b + i;
                v[i] = x[r * k + j] * f[j];
            }
            fwht32_f64(v);
            for (int i = 0; i < 32; ++i) y[r * k + 32 * b + i] = v[i];
        }
    }
}

/* ------------------------------------------------------------ MXFP4 */

/* floor(log2 |a|) for a finite, non-zero fp32, read from its bits (normal:
 * biased exponent - 127; subnormal: position of the top mantissa bit - 149). */
static int floor_log2_f32(float a)
{
    uint32_t u = f32_bits(a) & 0x7fffffffu;
    uint32_t e = u >> 23;
    if (e != 0) return (int)e - 127;
    int p = 31;
    while (!((u >> p) & 1u)) --p;
    return p - 149;
}

/* Shared scale exponent of one block from its absolute maximum:
 * se = clamp(floor(log2 amax) - 2, -127, 127); amax = 0 gives -127. */
int oracle_scale_exponent(float amax)
{
    if (amax == 0.0f) return -127;
    int se = floor_log2_f32(amax) - 2;
    if (se < -127) se = -127;
    if (se > 127) se = 127;
    return se;
}

/* E2M1 encode of one fp32 value: round |t| to the format's spacing at its
 * binade (0.5 below 1, one mantissa bit above), ties to even, saturate at 6.
 * Returns the 4-bit code sign|exp(2)|man(1); the sign of t is kept, also for
 * results that round to zero. */
uint8_t oracle_e2m1_encode(float t)
{
    uint8_t sign = (f32_bits(t) >> 31) ? 0x8 : 0x0;
    double a = fabs((double)t);
    int ex;
    double quantum = 0.5;
    if (a >= 1.0) {
        frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1) */
        quantum = ldexp(1.0, ex - 2);  /* 2^(floor(log2 a) - 1) */
    }
    double q = nearbyint(a / quantum) * quantum; /* default mode: ties to even */
    if (q > 6.0) q = 6.0;
    uint8_t mag;
    if (q < 1.0) {
        mag = (uint8_t)(q * 2.0); /* 0 -> 0, 0.5 -> 1 (exp field 0) */
    } else {
        double f = frexp(q, &ex);      /* q = 2^(ex-1) * (2f), 2f in [1, 2) */
        int man = (2.0 * f > 1.0) ? 1 : 0;
        mag = (uint8_t)((ex << 1) | man);  /* exp field = floor(log2 q) + 1 */
    }
    return (uint8_t)(sign | mag);
}

/* Value of a 4-bit E2M1 code: exp field 0 is subnormal (0.5 * man), else
 * 2^(exp-1) * (1 + man/2). */
double oracle_e2m1_value(uint8_t code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Quantise y [rows, k] fp32 into MXFP4: codes [rows, k/2] (element 2i in the
 * low nibble of byte i) and one E8M0 byte (se + 127) per 32-block, row-major
 * scales [rows, k/32]. */
void oracle_quantize_mx(const float *y, int64_t rows, int64_t k, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 32; ++b) {
            const float *blk = y + r * k + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(blk[i]);
                if (a > amax) amax = a;
            }
            int se = oracle_scale_exponent(amax);
            scales[r * (k / 32) + b] = (uint8_t)(se + 127);
            for (int i = 0; i < 32; i += 2) {
                float t0 = ldexpf(blk[i], -se);
                float t1 = ldexpf(blk[i + 1], -se);
                uint8_t c0 = oracle_e2m1_encode(t0);
                uint8_t c1 = oracle_e2m1_encode(t1);
                codes[r * (k / 2) + 16 * b + i / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
}

/* Whole activation (or weight) transform: balance, block Hadamard, MXFP4. */
void oracle_quant(const uint16_t *x, int64_t rows, int64_t k, const float *f, uint8_t *codes,
                  uint8_t *scales, float *work /* [rows, k] */)
{
    oracle_transform_f32(x, rows, k, f, work);
    oracle_quantize_mx(work, rows, k, codes, scales);
}

/* deq[r, j] = value(code) * 2^(scale - 127), exactly, in fp64. */
void oracle_dequant(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t k,
                    double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < k; ++j) {
            uint8_t byte = codes[r * (k / 2) + j / 2];
            uint8_t code = (j & 1) ? (byte >> 4) : (byte & 0xf);
            int se = (int)scales[r * (k / 32) + j / 32] - 127;
            out[r * k + j] = ldexp(oracle_e2m1_value(code), se);
        }
    }
}

/* Y[m, n] = sum_k A[m, k] * B[n, k] in fp64, plain triple loop (small sizes;
 * the Python wrapper uses a library matmul for large ones). */
void oracle_gemm_f64(const double *a, const double *b, int64_t m, int64_t n, int64_t k, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int64_t p = 0; p < k; ++p) acc += a[i * k + p] * b[j * k + p];
            y[i * n + j] = acc;
        }
    }
}

/* ------------------------------------------------ scale-factor tiling */

/* Rearrange row-major E8M0 scales [rows, nkb] into the library's tiled
 * layout.  Rows pad to a multiple of 128, scale columns to a multiple of 8;
 * padding bytes are 0.  Tile (rb, ka) covers rows 128*rb.. and scale columns
 * 4*ka..4*ka+3 and holds 512 bytes at ((rb * nka) + ka) * 512; inside it row
 * r = 32*q + p, column c sits at byte 16*p + 4*q + c. */
int64_t oracle_tiled_scale_bytes(int64_t rows, int64_t nkb)
{
    int64_t rp = (rows + 127) / 128 * 128;
    int64_t kp = (nkb + 7) / 8 * 8;
    return rp * kp;
}

void oracle_tile_scales(const uint8_t *src, int64_t rows, int64_t nkb, uint8_t *dst)
{
    int64_t rp = (rows + 127) / 128 * 128;
    int64_t kp = (nkb + 7) / 8 * 8;
    int64_t nka = kp / 4;
    for (int64_t r = 0; r < rp; ++r) {
        for (int64_t c = 0; c < kp; ++c) {
            uint8_t v = (r < rows && c < nkb) ? src[r * nkb + c] : 0;
            int64_t tile = (r / 128) * nka + c / 4;
            int64_t p = r % 32, q = (r % 128) / 32;
            dst[tile * 512 + 16 * p + 4 * q + (c % 4)] = v;
        }
    }
}

/* ------------------------------------------------ batch helpers (tests) */

void oracle_e2m1_encode_many(const float *t, int64_t n, uint8_t *codes)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) codes[i] = oracle_e2m1_encode(t[i]);
}

void oracle_scale_exponent_many(const float *amax, int64_t n, int32_t *se)
{
    for (int64_t i = 0; i < n; ++i) se[i] = oracle_scale_exponent(amax[i]);
}

/* ------------------------------------------------------------------ SwiGLU */

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
static uint16_t f32_to_bf16_rne(float f)
{
    const uint32_t u = f32_bits(f);
    const uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

/* Round a finite double to the nearest bf16 (ties to even), directly: the
 * quantum is 2^(e - 8) for |v| in [2^(e-1), 2^e) (8 significant bits), and
 * 2^-133 below the smallest normal 2^-126 (bf16 subnormals); rint() rounds to
 * nearest even in the default rounding mode and the division by the quantum
 * is exact.  Results above the largest bf16 become infinities. */
static uint16_t f64_to_bf16_rne(double v)
{
    if (v == 0.0) return signbit(v) ? 0x8000u : 0x0000u;
    int e;
    (void)frexp(v, &e);
    const int qexp = (e - 8 > -133) ? e - 8 : -133;
    const double r = ldexp(rint(ldexp(v, -qexp)), qexp);
    const float f = (float)r;   /* exact: r has at most 8 significant bits */
    uint32_t u = f32_bits(f);
    if (isinf(f) || fabs(r) > 0x1.fep+127) u = signbit(v) ? 0xff800000u : 0x7f800000u;
    if (r == 0.0) u = signbit(v) ? 0x80000000u : 0u;
    return (uint16_t)(u >> 16);
}

/* The exact value of SiLU(g) * u = g * u / (1 + e^-g), in fp64. */
static double silu_mul_f64(double g, double u)
{
    const double e = exp(-g);               /* +inf for very negative g: -> -0 */
    return g / (1.0 + e) * u;
}

/* Half-width of the window (relative, plus an absolute floor far below any
 * bf16 normal) around a rounding boundary inside which an fp32 evaluation
 * may round either way. */
#define SILU_WINDOW_REL 0x1.0p-20
#define SILU_WINDOW_ABS 0x1.0p-140

/* h = bf16_rn( SiLU(g) * u ) of one element; *alt = the other bf16
 * neighbour when the exact value lies within the window of a rounding
 * boundary, else h. */
static uint16_t silu_mul_bf16(uint16_t g_bits, uint16_t u_bits, uint16_t *alt)
{
    const double g = (double)bf16_bits_to_f32(g_bits);
    const double u = (double)bf16_bits_to_f32(u_bits);
    const double v = silu_mul_f64(g, u);
    const uint16_t h = f64_to_bf16_rne(v);
    const double w = SILU_WINDOW_REL * fabs(v) + SILU_WINDOW_ABS;
    const uint16_t lo = f64_to_bf16_rne(v - w), hi = f64_to_bf16_rne(v + w);
    *alt = (lo != h) ? lo : hi;
    return h;
}

/* gu: [rows, 2F] bf16 (gate in columns 0..F-1, up in F..2F-1) -> h [rows, F]
 * and, if h_alt is not NULL, the other admissible neighbour [rows, F]. */
void oracle_silu_mul(const uint16_t *gu, int64_t rows, int64_t F, uint16_t *h, uint16_t *h_alt)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < F; ++j) {
            uint16_t alt;
            h[r * F + j] = silu_mul_bf16(gu[r * 2 * F + j], gu[r * 2 * F + F + j], &alt);
            if (h_alt) h_alt[r * F + j] = alt;
        }
}

/* The fp64 -> bf16 rounding on its own (for the pins). */
void oracle_f64_to_bf16_many(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f64_to_bf16_rne(x[i]);
}

/* ------------------------------------------------------ Flip Refinement */

/* H = A^T A for calibration rows A [m, k] (fp32), each entry a sequential
 * fused multiply-add over the rows r = 0 .. m-1 starting from +0; `damp` is
 * then added (one fp32 add) to every diagonal entry. */
void oracle_flip_hessian(const float *a, int64_t m, int64_t k, float damp, float *h)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < k; ++i) {
        for (int64_t j = 0; j < k; ++j) {
            float acc = 0.0f;
            for (int64_t r = 0; r < m; ++r) acc = fmaf(a[r * k + i], a[r * k + j], acc);
            if (i == j) acc = acc + damp;
            h[i * k + j] = acc;
        }
    }
}

/* Magnitudes of the E2M1 grid, by magnitude code 0 .. 7. */
static float e2m1_magnitude(int mag)
{
    return (float)oracle_e2m1_value((uint8_t)mag);
}

/* Signed grid position of a code: -7 .. 7, both zeros at 0. */
static int e2m1_position(uint8_t code)
{
    int mag = code & 7;
    return (code & 8) ? -mag : mag;
}

/* Code of a signed grid position; position 0 gets the sign of the value the
 * move came from (from_negative), so a zero keeps the side it was reached from. */
static uint8_t e2m1_code_at(int pos, int from_negative)
{
    if (pos > 0) return (uint8_t)pos;
    if (pos < 0) return (uint8_t)(8 | -pos);
    return from_negative ? 0x8 : 0x0;
}

static float e2m1_position_value(int pos)
{
    return pos < 0 ? -e2m1_magnitude(-pos) : e2m1_magnitude(pos);
}

/* Flip Refinement of weight rows wt [n, k] (the fp32 weight transform) whose
 * round-to-nearest codes [n, k/2] (in/out) and row-major scales [n, k/32] the
 * MXFP4 step produced, against the Hessian h [k, k] (symmetric).  flips[row]
 * (if not NULL) receives the number of moves taken. */
void oracle_flip_refine(const float *wt, const float *h, int64_t n, int64_t k, int32_t sweeps,
                        uint8_t *codes, const uint8_t *scales, int32_t *flips)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t row = 0; row < n; ++row) {
        uint8_t *c = codes + row * (k / 2);
        const uint8_t *sc = scales + row * (k / 32);
        float *r = (float *)malloc(sizeof(float) * (size_t)k);
        float *g = (float *)malloc(sizeof(float) * (size_t)k);
        /* residual of the round-to-nearest codes */
        for (int64_t j = 0; j < k; ++j) {
            uint8_t code = (j & 1) ? (c[j / 2] >> 4) : (c[j / 2] & 0xf);
            float q = ldexpf(e2m1_position_value(e2m1_position(code)), (int)sc[j / 32] - 127);
            r[j] = wt[row * k + j] - q;
        }
        /* g = H r, each entry a sequential fused multiply-add over l */
        for (int64_t j = 0; j < k; ++j) {
            float acc = 0.0f;
            for (int64_t l = 0; l < k; ++l) acc = fmaf(h[j * k + l], r[l], acc);
            g[j] = acc;
        }
        int32_t moves = 0;
        for (int32_t sw = 0; sw < sweeps; ++sw) {
            for (int64_t j = 0; j < k; ++j) {
                uint8_t code = (j & 1) ? (c[j / 2] >> 4) : (c[j / 2] & 0xf);
                int pos = e2m1_position(code);
                int se = (int)sc[j / 32] - 127;
                float t = e2m1_position_value(pos);
                float hjj = h[j * k + j];
                float two_g = 2.0f * g[j];
                int best = 0;          /* 0: stay, -1: down, +1: up */
                float best_de = 0.0f;
                float best_d = 0.0f;
                for (int dir = -1; dir <= 1; dir += 2) {
                    int np = pos + dir;
                    if (np < -7 || np > 7) continue;
                    float d = ldexpf(e2m1_position_value(np) - t, se);
                    float de = d * (d * hjj - two_g);
                    if (de < 0.0f && (best == 0 || de < best_de)) {
                        best = dir;
                        best_de = de;
                        best_d = d;
                    }
                }
                if (best == 0) continue;
                uint8_t nc = e2m1_code_at(pos + best, pos < 0);
                if (j & 1)
                    c[j / 2] = (uint8_t)((c[j / 2] & 0x0f) | (nc << 4));
                else
                    c[j / 2] = (uint8_t)((c[j / 2] & 0xf0) | nc);
                for (int64_t l = 0; l < k; ++l) g[l] = fmaf(-best_d, h[j * k + l], g[l]);
                ++moves;
            }
        }
        if (flips) flips[row] = moves;
        free(r);
        free(g);
    }
}

/* ---------------------------------------------------------- MoE combine */

/* out[t, n] = bf16( fma-chain over k = 0 .. topk-1 of w[t, k] * y[rows[t, k], n]
 * from +0 ), y bf16 bits [*, n_cols] row pitch ldy, out bf16 bits [t, n_cols]. */
void oracle_moe_combine(const uint16_t *y, int64_t ldy, const int32_t *rows, const float *w,
                        int64_t t_count, int64_t topk, int64_t n_cols, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < t_count; ++t) {
        for (int64_t n = 0; n < n_cols; ++n) {
            float acc = 0.0f;
            for (int64_t k = 0; k < topk; ++k)
                acc = fmaf(w[t * topk + k], bf16_bits_to_f32(y[(int64_t)rows[t * topk + k] * ldy + n]), acc);
            out[t * n_cols + n] = f32_to_bf16_rne(acc);
        }
    }
}
