/*
 * fp4q oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar CPU restatement of the micro-scaled FP4 hot path:
 * MXFP4 quantize / dequantize, direct FP8->MXFP4, scaled MXFP4->FP8,
 * the 16-point random Hadamard transform, NVFP4 quantize with round-to-
 * nearest-even or Philox stochastic rounding.  (The GEMM and MoE oracles are
 * float64 NumPy in oracle/__init__.py.)
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline may load this file.  It shares no code, header, table or
 * constant generator with the CUDA library and includes nothing from it.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (no FMA contraction: every float operation below is one IEEE-754
 * round-to-nearest-even operation, as written).
 *
 * Sources (web pages; every step cites the passage it restates):
 *  [MXN]  "Pretraining large language models with MXFP4 on Native FP4
 *         Hardware" (news article), section "Qu'est-ce que le MXFP4 ?"
 *  [HOP]  "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"
 *         (French and Spanish technical summaries), section 2 (methodology)
 *  [NVF]  "Pretraining Large Language Models with NVFP4" (technical
 *         summary), section 2.A (the NVFP4 format) and 2.B (recipe)
 *  [OCP]  the OCP Microscaling (MX) and OCP 8-bit floating point formats,
 *         which [MXN] names in its conclusion but does not reproduce.
 *  [PHX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *         1, 2, 3", SC'11 -- the Philox4x32-10 generator.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Bit helpers (plain C, no intrinsics)                                */
/* ------------------------------------------------------------------ */
static float u32_as_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_as_u32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* BF16 -> FP32 is exact: the 16 BF16 bits are the top half of an FP32. */
static float bf16_to_f32(uint16_t h) { return u32_as_f32(((uint32_t)h) << 16); }

/* FP32 -> BF16, round to nearest, ties to even (IEEE-754).  Finite
 * inputs that round past the largest BF16 become +-inf. */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = f32_as_u32(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) /* NaN */
        return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/NaN.     */
/* [OCP]; [MXN] (4-bit float element), [HOP] section 1 (E2M1).          */
/* ------------------------------------------------------------------ */

/* Value of a 4-bit E2M1 code, from its fields. */
double or_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* Round-to-nearest of a real value onto the E2M1 grid: the magnitude is
 * the representable magnitude nearest to |v|, ties going to the code
 * whose mantissa bit is 0 ("even"); anything beyond the largest value is
 * held at the largest value (saturation).  [MXN]: Q_FP4 rounds to the
 * nearest 4-bit float.  The sign bit is copied from v, also when the
 * magnitude rounds to 0 (a reading: the pages do not say). */
int or_e2m1_rne_d(double v) {
    int sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    if (a >= 6.0) return sign | 7;          /* saturation at the largest value */
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double err = fabs(a - or_e2m1_value(c));
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sign | best;
}

int or_e2m1_rne(float v) { return or_e2m1_rne_d((double)v); }

/* ------------------------------------------------------------------ */
/* E4M3 (the "FN" variant): bias 7, no inf, S.1111.111 is NaN, max 448. */
/* [OCP]; [HOP] section 1 (Hopper FP8 pipeline is E4M3), [NVF] 2.A      */
/* (block scales are E4M3).                                             */
/* ------------------------------------------------------------------ */
double or_e4m3_value(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest finite E4M3 value to v, ties to the even code, saturating at
 * +-448 (values beyond the largest finite value take the largest). */
uint8_t or_e4m3_rn_satfinite_d(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);   /* saturation at 448 */
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        double err = fabs(a - or_e4m3_value((uint8_t)c));
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

uint8_t or_e4m3_rn_satfinite(float v) { return or_e4m3_rn_satfinite_d((double)v); }

/* ------------------------------------------------------------------ */
/* MXFP4 quantize (a1).                                                 */
/* [MXN]: the tensor is cut into blocks of 32 elements that share one   */
/* E8M0 exponent; each element is stored as a 4-bit float and the value */
/* is rebuilt as 2^E_shared * Q_FP4(X / 2^E_shared), E_shared taken     */
/* from the largest exponent in the block.  The shared exponent is      */
/* floor(log2(block amax)) minus the largest E2M1 exponent (2), as in   */
/* [OCP]; an all-zero block takes E = -127 (byte 0; a reading).  E is   */
/* clamped to the E8M0 range [-127, 127].                               */
/* ------------------------------------------------------------------ */
#define OR_MX_BLOCK 32

/* Shared exponent of a block, from the exact binary exponent of amax. */
int or_mx_shared_exponent(double amax) {
    if (amax == 0.0) return -127;
    int ex;
    frexp(amax, &ex);          /* amax = f * 2^ex, f in [0.5, 1): exact */
    int e = (ex - 1) - 2;      /* floor(log2 amax) - emax(E2M1) */
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

static void put_nibble(uint8_t* row, int64_t i, int code) {
    /* element i of a row: low nibble of byte i/2 when i is even, high
     * nibble when odd (the OCP packing order; a reading). */
    if (i & 1) row[i >> 1] = (uint8_t)((row[i >> 1] & 0x0f) | (code << 4));
    else       row[i >> 1] = (uint8_t)((row[i >> 1] & 0xf0) | (code & 0x0f));
}

static int get_nibble(const uint8_t* row, int64_t i) {
    return (i & 1) ? (row[i >> 1] >> 4) : (row[i >> 1] & 0x0f);
}

/* x: FP32 values [rows, cols] (row stride ld_x), cols % 32 == 0.
 * q: [rows, cols/2] packed codes.  s: [rows, cols/32] E8M0 bytes. */
void or_mx_quantize_f32(const float* x, int64_t rows, int64_t cols, int64_t ld_x,
                        uint8_t* q, uint8_t* s) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ld_x;
        uint8_t* qr = q + r * (cols / 2);
        for (int64_t b = 0; b < cols / OR_MX_BLOCK; ++b) {
            const float* xb = xr + b * OR_MX_BLOCK;
            double amax = 0.0;
            for (int j = 0; j < OR_MX_BLOCK; ++j)
                if (fabs((double)xb[j]) > amax) amax = fabs((double)xb[j]);
            int e = or_mx_shared_exponent(amax);
            s[r * (cols / OR_MX_BLOCK) + b] = (uint8_t)(e + 127);
            for (int j = 0; j < OR_MX_BLOCK; ++j) {
                double v = (double)xb[j] * ldexp(1.0, -e);   /* X / 2^E, exact */
                put_nibble(qr, b * OR_MX_BLOCK + j, or_e2m1_rne_d(v));
            }
        }
    }
}

/* BF16 source: the same, on the exact FP32 widening of each element. */
void or_mx_quantize_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                         uint8_t* q, uint8_t* s) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float tmp[OR_MX_BLOCK];
        const uint16_t* xr = x + r * ld_x;
        for (int64_t b = 0; b < cols / OR_MX_BLOCK; ++b) {
            for (int j = 0; j < OR_MX_BLOCK; ++j) tmp[j] = bf16_to_f32(xr[b * OR_MX_BLOCK + j]);
            /* one block at a time through the FP32 path */
            uint8_t qb[OR_MX_BLOCK / 2];
            uint8_t sb;
            or_mx_quantize_f32(tmp, 1, OR_MX_BLOCK, OR_MX_BLOCK, qb, &sb);
            memcpy(q + r * (cols / 2) + b * (OR_MX_BLOCK / 2), qb, OR_MX_BLOCK / 2);
            s[r * (cols / OR_MX_BLOCK) + b] = sb;
        }
    }
}

/* Value of an E8M0 byte as a power-of-two exponent (byte 255 is NaN in
 * [OCP]; it is never produced and is treated as exponent 128 here). */
static int e8m0_exponent(uint8_t b) { return (int)b - 127; }

/* MXFP4 dequantize (a2): y = 2^E * value(q), exact in double, rounded to
 * FP32 (overflow -> inf).  y_bf16 (if non-NULL) gets its BF16 rounding. */
void or_mx_dequantize(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols,
                      float* y_f32, uint16_t* y_bf16) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < cols; ++i) {
            int e = e8m0_exponent(s[r * (cols / OR_MX_BLOCK) + i / OR_MX_BLOCK]);
            double v = or_e2m1_value(get_nibble(q + r * (cols / 2), i)) * ldexp(1.0, e);
            float f = (float)v;
            if (y_f32) y_f32[r * cols + i] = f;
            if (y_bf16) y_bf16[r * cols + i] = f32_to_bf16_rne(f);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Direct FP8 -> MXFP4 (a3).                                            */
/* [HOP] (abstract and section 1): activations go from FP8 straight to  */
/* FP4 with no BF16 intermediate.  The source is E4M3 with one FP32     */
/* scale per 1x128 tile of a row ([HOP] section 1: Hopper's FP8 path    */
/* scales 128-element blocks).  Each element's real value is the FP32  */
/* product decode(e4m3) * tile_scale (one IEEE multiply); the MXFP4     */
/* quantizer then runs on those products.                               */
/* ------------------------------------------------------------------ */
#define OR_FP8_TILE 128

void or_fp8_to_mx(const uint8_t* x, const float* tile_scale, int64_t rows, int64_t cols,
                  int64_t ld_x, uint8_t* q, uint8_t* s) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float tmp[OR_MX_BLOCK];
        for (int64_t b = 0; b < cols / OR_MX_BLOCK; ++b) {
            for (int j = 0; j < OR_MX_BLOCK; ++j) {
                int64_t c = b * OR_MX_BLOCK + j;
                float sc = tile_scale[r * (cols / OR_FP8_TILE) + c / OR_FP8_TILE];
                float dec = (float)or_e4m3_value(x[r * ld_x + c]);   /* exact */
                tmp[j] = dec * sc;                                   /* one RN multiply */
            }
            uint8_t qb[OR_MX_BLOCK / 2];
            uint8_t sb;
            or_mx_quantize_f32(tmp, 1, OR_MX_BLOCK, OR_MX_BLOCK, qb, &sb);
            memcpy(q + r * (cols / 2) + b * (OR_MX_BLOCK / 2), qb, OR_MX_BLOCK / 2);
            s[r * (cols / OR_MX_BLOCK) + b] = sb;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Scaled MXFP4 -> FP8 (a4).                                            */
/* [HOP] section 2.B: the four 32-element FP4 block scales inside one   */
/* 128-element FP8 tile are aligned to their maximum, which becomes the */
/* FP8 tile scale; each element is re-expressed relative to it, so the  */
/* represented value is unchanged ("hierarchical scale alignment").     */
/* [HOP, Spanish summary] section 2: subnormal results keep their value */
/* (the implicit bit is materialised).                                  */
/* The plain reading implemented here: tile scale = 2^Emax (FP32), and  */
/* element = E4M3 nearest (ties to even, saturating) to value(q) *      */
/* 2^(E_i - Emax); magnitudes below the smallest E4M3 subnormal (2^-9)  */
/* are flushed to a signed zero.                                        */
/* ------------------------------------------------------------------ */
uint8_t or_fp8_from_e2m1_shifted(int code, int d) {
    double w = or_e2m1_value(code) * ldexp(1.0, d);
    if (fabs(w) < ldexp(1.0, -9)) return (code & 8) ? 0x80 : 0x00;
    return or_e4m3_rn_satfinite_d(w);
}

void or_mx_to_fp8(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols,
                  uint8_t* y, float* tile_scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t t = 0; t < cols / OR_FP8_TILE; ++t) {
            int emax = -1000;
            for (int k = 0; k < OR_FP8_TILE / OR_MX_BLOCK; ++k) {
                int e = e8m0_exponent(s[r * (cols / OR_MX_BLOCK) + t * 4 + k]);
                if (e > emax) emax = e;
            }
            tile_scale[r * (cols / OR_FP8_TILE) + t] = (float)ldexp(1.0, emax);
            for (int j = 0; j < OR_FP8_TILE; ++j) {
                int64_t c = t * OR_FP8_TILE + j;
                int e = e8m0_exponent(s[r * (cols / OR_MX_BLOCK) + c / OR_MX_BLOCK]);
                y[r * cols + c] = or_fp8_from_e2m1_shifted(get_nibble(q + r * (cols / 2), c), e - emax);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 [PHX].                                                 */
/* Round: multiply counter words 0 and 2 by the two round multipliers,  */
/* form the new counter from the high/low product halves xored with the */
/* other two words and the key; the key is bumped by the two Weyl       */
/* constants between rounds.                                            */
/* ------------------------------------------------------------------ */
void or_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit random word of logical element i under a 64-bit seed: the
 * i-th word of the Philox stream keyed by the seed (counter = i / 4 as a
 * 128-bit integer, word = i mod 4).  A reading: the pages only say the
 * stream is keyed by the seed and the element's linear index. */
uint32_t or_sr_word(uint64_t seed, uint64_t i) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint64_t blk = i >> 2;
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u};
    uint32_t out[4];
    or_philox4x32_10(ctr, key, out);
    return out[i & 3];
}

/* ------------------------------------------------------------------ */
/* 16-point random Hadamard transform (a5).                             */
/* [NVF] 2.B (random Hadamard transforms on the weight-gradient inputs) */
/* and [MXN] (Hadamard rotation with random sign flips spreads outliers */
/* before quantization).  y = (1/4) * H16 * (D x) on each 16-element    */
/* tile along the block axis; H16 is the Sylvester Hadamard matrix and  */
/* D = diag(d) a +-1 vector.  d_j = -1 iff bit j of word 0 of           */
/* Philox4x32-10(key = seed, counter = 0) is set (a reading).           */
/* Fixed FP32 evaluation order (so results are reproducible bit for     */
/* bit): widen to FP32, apply the signs, radix-2 butterflies with       */
/* strides 1, 2, 4, 8 mapping (a, b) -> (a + b, a - b), then * 0.25.    */
/* ------------------------------------------------------------------ */
void or_rht16_signs(uint64_t seed, float d[16]) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {0, 0, 0, 0}, out[4];
    or_philox4x32_10(ctr, key, out);
    for (int j = 0; j < 16; ++j) d[j] = ((out[0] >> j) & 1u) ? -1.0f : 1.0f;
}

void or_rht16(const float x[16], const float d[16], float y[16]) {
    float t[16];
    for (int j = 0; j < 16; ++j) t[j] = d[j] * x[j];
    for (int h = 1; h < 16; h <<= 1) {
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            float a = t[i], b = t[i + h];
            t[i] = a + b;
            t[i + h] = a - b;
        }
    }
    for (int j = 0; j < 16; ++j) y[j] = t[j] * 0.25f;
}

/* ------------------------------------------------------------------ */
/* Stochastic rounding onto the E2M1 grid.                              */
/* [NVF] 2.B and [MXN]: the value goes to one of the two neighbouring   */
/* representable values, with probabilities that make the expected      */
/* rounding error zero.  Round up iff the element's random word r       */
/* satisfies r < frac * 2^32, frac = (|v| - lo) / (hi - lo) (exact      */
/* real comparison); |v| >= 6 saturates to 6; the sign is copied.       */
/* ------------------------------------------------------------------ */
int or_e2m1_sr_d(double v, uint32_t r) {
    int sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    if (a >= 6.0) return sign | 7;
    int lo = 0;
    for (int c = 0; c < 8; ++c)
        if (or_e2m1_value(c) <= a) lo = c;       /* largest grid value <= |v| */
    double vlo = or_e2m1_value(lo), vhi = or_e2m1_value(lo + 1);
    double frac = (a - vlo) / (vhi - vlo);
    int up = (double)r < frac * 4294967296.0;
    return sign | (up ? lo + 1 : lo);
}

/* ------------------------------------------------------------------ */
/* NVFP4 quantize (a5 + a6).                                            */
/* [NVF] 2.A: 16-element blocks of E2M1, one E4M3 scale per block and   */
/* one FP32 scale per tensor (two-level scaling).  With the tensor      */
/* amax of the (optionally rotated) values y:                          */
/*   s_t   = amax / (6 * 448)                      (FP32, one division) */
/*   s_b   = E4M3_RN_satfinite(blockamax / (6 * s_t))   (FP32 ops)      */
/*   sf    = float(s_b) * s_t;  rcp = 1 / sf;  v = y * rcp  (FP32 ops)  */
/*   q     = RNE_E2M1(v) or SR_E2M1(v, word of linear element index)    */
/* amax == 0, or s_b == 0, gives signed-zero codes (a reading).          */
/* ------------------------------------------------------------------ */
#define OR_NV_BLOCK 16

/* Signs of the rotation for rht mode: 0 none, 1 random signs from the seed
 * ([NVF] 2.B), 2 the deterministic H16 with D = I ("Pretraining Large
 * Language Models with MXFP4 on Native FP4 Hardware", Wgrad section: the same
 * Hadamard rotation at every step; the plain reading of "deterministic" is
 * no sign flips). */
static void nv_signs(int rht, uint64_t seed, float d[16]) {
    if (rht == 1) {
        or_rht16_signs(seed, d);
    } else {
        for (int j = 0; j < 16; ++j) d[j] = 1.0f;
    }
}

static void nv_rotated_row(const uint16_t* xr, int64_t cols, int rht, const float d[16], float* yr) {
    for (int64_t t = 0; t < cols / 16; ++t) {
        float xin[16], yo[16];
        for (int j = 0; j < 16; ++j) xin[j] = bf16_to_f32(xr[t * 16 + j]);
        if (rht) or_rht16(xin, d, yo);
        else memcpy(yo, xin, sizeof yo);
        memcpy(yr + t * 16, yo, sizeof yo);
    }
}

/* Tensor amax of the (optionally rotated) BF16 input. */
float or_nv_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, int rht, uint64_t rht_seed) {
    float d[16];
    nv_signs(rht, rht_seed, d);
    float amax = 0.0f;
#pragma omp parallel for schedule(static) reduction(max : amax)
    for (int64_t r = 0; r < rows; ++r) {
        float yr[16];
        for (int64_t t = 0; t < cols / 16; ++t) {
            nv_rotated_row(x + r * ld_x + t * 16, 16, rht, d, yr);
            for (int j = 0; j < 16; ++j)
                if (fabsf(yr[j]) > amax) amax = fabsf(yr[j]);
        }
    }
    return amax;
}

/* rounding: 0 = RNE, 1 = SR.  amax_in: if non-NULL, used as the tensor
 * amax instead of computing it.  row_offset: index of x's first row in the
 * full tensor (the SR stream is indexed by the full tensor's linear element
 * index (row_offset + r) * cols + c).  Outputs: q [rows, cols/2], s_e4m3
 * [rows, cols/16], *s_t_out (the FP32 tensor scale), *amax_out. */
void or_nv_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x,
                    int rht, uint64_t rht_seed, int rounding, uint64_t sr_seed,
                    const float* amax_in, float* amax_out, float* s_t_out,
                    uint8_t* q, uint8_t* s_e4m3, int64_t row_offset) {
    float d[16];
    nv_signs(rht, rht_seed, d);
    float amax = amax_in ? *amax_in : or_nv_amax(x, rows, cols, ld_x, rht, rht_seed);
    float s_t = amax / 2688.0f;            /* 2688 = 6 * 448 */
    if (amax_out) *amax_out = amax;
    if (s_t_out) *s_t_out = s_t;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float y[16];
        for (int64_t b = 0; b < cols / OR_NV_BLOCK; ++b) {
            nv_rotated_row(x + r * ld_x + b * 16, 16, rht, d, y);
            float ab = 0.0f;
            for (int j = 0; j < 16; ++j)
                if (fabsf(y[j]) > ab) ab = fabsf(y[j]);
            uint8_t sb = 0;
            float rcp = 0.0f;
            int zero_block = 1;
            if (s_t > 0.0f) {
                float denom = 6.0f * s_t;
                float ratio = ab / denom;
                sb = or_e4m3_rn_satfinite(ratio);
                if ((sb & 0x7f) != 0) {
                    float sf = (float)or_e4m3_value(sb) * s_t;
                    rcp = 1.0f / sf;
                    zero_block = 0;
                }
            }
            s_e4m3[r * (cols / OR_NV_BLOCK) + b] = sb;
            for (int j = 0; j < 16; ++j) {
                int64_t c = b * 16 + j;
                int code;
                if (zero_block) {
                    code = signbit(y[j]) ? 8 : 0;
                } else {
                    float v = y[j] * rcp;
                    if (rounding == 1)
                        code = or_e2m1_sr_d((double)v, or_sr_word(sr_seed, (uint64_t)((row_offset + r) * cols + c)));
                    else
                        code = or_e2m1_rne_d((double)v);
                }
                put_nibble(q + r * (cols / 2), c, code);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* NVFP4 with 2D (16 x 16) block scaling, for weights.                  */
/* [NVF] 2.B ("Mise a l'echelle bidimensionnelle"): weight blocks are   */
/* 16 x 16, so the forward pass and the backward pass (which reads the  */
/* weight transposed) quantize it identically.  Plain reading: one E4M3 */
/* scale per 16 x 16 tile from that tile's amax, with the 1D rules of   */
/* or_nv_quantize otherwise (tensor scale, scale rounding, rcp, RNE or  */
/* SR by linear element index, signed zeros for a zero scale).  No RHT  */
/* (the pages apply the RHT to Wgrad inputs, not to weights).  The      */
/* scale is stored for every row of its tile ([rows, cols/16] layout,   */
/* 16 equal rows per tile), so the 1D consumers read it unchanged.      */
/* rows % 16 == 0.                                                       */
/* ------------------------------------------------------------------ */
void or_nv_quantize_2d(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld_x, int rounding,
                       uint64_t sr_seed, const float* amax_in, float* amax_out, float* s_t_out,
                       uint8_t* q, uint8_t* s_e4m3) {
    float amax = amax_in ? *amax_in : or_nv_amax(x, rows, cols, ld_x, 0, 0);
    float s_t = amax / 2688.0f;
    if (amax_out) *amax_out = amax;
    if (s_t_out) *s_t_out = s_t;
#pragma omp parallel for schedule(static)
    for (int64_t tr = 0; tr < rows / 16; ++tr) {
        for (int64_t b = 0; b < cols / OR_NV_BLOCK; ++b) {
            float ab = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    float v = fabsf(bf16_to_f32(x[(tr * 16 + i) * ld_x + b * 16 + j]));
                    if (v > ab) ab = v;
                }
            uint8_t sb = 0;
            float rcp = 0.0f;
            int zero_block = 1;
            if (s_t > 0.0f) {
                float denom = 6.0f * s_t;
                sb = or_e4m3_rn_satfinite(ab / denom);
                if ((sb & 0x7f) != 0) {
                    float sf = (float)or_e4m3_value(sb) * s_t;
                    rcp = 1.0f / sf;
                    zero_block = 0;
                }
            }
            for (int i = 0; i < 16; ++i) {
                int64_t r = tr * 16 + i;
                s_e4m3[r * (cols / OR_NV_BLOCK) + b] = sb;
                for (int j = 0; j < 16; ++j) {
                    int64_t c = b * 16 + j;
                    float y = bf16_to_f32(x[r * ld_x + c]);
                    int code;
                    if (zero_block) {
                        code = signbit(y) ? 8 : 0;
                    } else {
                        float v = y * rcp;
                        if (rounding == 1)
                            code = or_e2m1_sr_d((double)v, or_sr_word(sr_seed, (uint64_t)(r * cols + c)));
                        else
                            code = or_e2m1_rne_d((double)v);
                    }
                    put_nibble(q + r * (cols / 2), c, code);
                }
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* FP4RowToFP8Col: row-wise MXFP4 [rows, cols] -> FP8 of the transpose. */
/* [HOP] Spanish summary, section 2 (kernels BF16ToFP4Row,              */
/* FP4RowToFP8Row, FP4RowToFP8Col) and French summary section 2.C: one  */
/* kernel dequantizes, transposes and re-quantizes (the weight-gradient */
/* operand).  Plain reading: output y = E4M3 [cols, rows] with FP32     */
/* scales per 1 x 128 tile along the output rows ([cols, rows/128]); a  */
/* tile covers input rows r0 .. r0+127 of one input column c, its scale */
/* is 2^Emax with Emax the largest block exponent among those 128       */
/* elements, and each element is or_fp8_from_e2m1_shifted(code,         */
/* E_element - Emax) -- the same rule as or_mx_to_fp8, so the tensor is */
/* carried over exactly except for the flush below 2^-9 of its tile.    */
/* rows % 128 == 0.                                                      */
/* ------------------------------------------------------------------ */
void or_mx_to_fp8_col(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols,
                      uint8_t* y, float* tile_scale) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t t = 0; t < rows / OR_FP8_TILE; ++t) {
            int emax = -1000;
            for (int j = 0; j < OR_FP8_TILE; ++j) {
                int e = e8m0_exponent(s[(t * OR_FP8_TILE + j) * (cols / OR_MX_BLOCK) + c / OR_MX_BLOCK]);
                if (e > emax) emax = e;
            }
            tile_scale[c * (rows / OR_FP8_TILE) + t] = (float)ldexp(1.0, emax);
            for (int j = 0; j < OR_FP8_TILE; ++j) {
                int64_t r = t * OR_FP8_TILE + j;
                int e = e8m0_exponent(s[r * (cols / OR_MX_BLOCK) + c / OR_MX_BLOCK]);
                y[c * rows + r] = or_fp8_from_e2m1_shifted(get_nibble(q + r * (cols / 2), c), e - emax);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* NVFP4 dequantize: value(q) * float(s_b) * s_t, exact in double.       */
/* ------------------------------------------------------------------ */
void or_nv_dequantize(const uint8_t* q, const uint8_t* s_e4m3, float s_t, int64_t rows,
                      int64_t cols, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < cols; ++i) {
            double sb = or_e4m3_value(s_e4m3[r * (cols / OR_NV_BLOCK) + i / OR_NV_BLOCK]);
            y[r * cols + i] = or_e2m1_value(get_nibble(q + r * (cols / 2), i)) * sb * (double)s_t;
        }
}

/* MXFP4 dequantize to float64 (for the GEMM oracle). */
void or_mx_dequantize_f64(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < cols; ++i) {
            int e = e8m0_exponent(s[r * (cols / OR_MX_BLOCK) + i / OR_MX_BLOCK]);
            y[r * cols + i] = or_e2m1_value(get_nibble(q + r * (cols / 2), i)) * ldexp(1.0, e);
        }
}

/* Elementwise helpers exposed for the tests' brute-force sweeps. */
void or_e2m1_rne_array(const float* v, int64_t n, uint8_t* codes) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)or_e2m1_rne(v[i]);
}

void or_e4m3_rn_satfinite_array(const float* v, int64_t n, uint8_t* codes) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) codes[i] = or_e4m3_rn_satfinite(v[i]);
}

void or_e2m1_sr_array(const float* v, const uint32_t* r, int64_t n, uint8_t* codes) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)or_e2m1_sr_d((double)v[i], r[i]);
}

void or_sr_words(uint64_t seed, uint64_t first, int64_t n, uint32_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = or_sr_word(seed, first + (uint64_t)i);
}

void or_rht16_rows(const float* x, int64_t ntiles, uint64_t seed, float* y) {
    float d[16];
    or_rht16_signs(seed, d);
    for (int64_t t = 0; t < ntiles; ++t) or_rht16(x + t * 16, d, y + t * 16);
}
