/*
 * qmd_oracle.c -- plain, slow CPU statement of the Q4_K / Q6_K x q8_K decode mat-vec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may call, link or load
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no code, header, table or constant generator with the CUDA path.
 *
 * Build: portable C99, `-O2 -ffp-contract=off` so that every f32 operation below is rounded
 * on its own (no fused multiply-add), identically on x86-64 and aarch64.
 *
 * What is computed, and from which passage
 * ----------------------------------------
 * "Language models on the device: the cajeta-llm kernels" (cajeta.dev/xpu/kernels-llm):
 *   §1  weights are GGUF K-quants, 256 values a block with per-sub-block scales; activations
 *       are quantised on the device to q8_K (256 values a block, one scale, eight sub-block
 *       sums) so that an integer dot product does the arithmetic, and the per-sub-block
 *       scales fold into a rank-one epilogue; a Q6_K weight may be split at bind into a
 *       scale prefix plus 208-byte bodies.
 *   §2.1 one output row is finished by a reduction over the row's blocks.
 * "Kernel SPI and the selection algorithm" (SKaiNET), "The descriptor: KernelKey":
 *   canonical GGUF order is blocks laid out along rows (row r's blocks are contiguous);
 *   "Why a kernel declines": a K-quant tensor whose last dimension is not a multiple of 256
 *   is rejected.
 *
 * The same page, §2.3: a Q5_K kernel differs from the Q4_K one only in how it stages the
 * codes: the fifth-bit plane is OR-ed into bit four of each 4-bit code.
 *
 * The pages do not print the bit layout of a Q4_K, Q5_K or Q6_K block, the q8_K rounding
 * rule, or the epilogue's order of operations.  The readings taken here:
 *   - block layouts: the public GGUF format definition (byte offsets in the decoders below);
 *   - q8_K: symmetric absmax scale, d = amax/127, codes round(x * 127/amax) to nearest-even
 *     in f32, clamped to [-127, 127]; an all-zero block has d = 0 and zero codes; the eight
 *     sums are over 32-value sub-blocks (the pages say eight);
 *   - epilogue per 256-value block, each f32 operation rounded separately:
 *       Q4_K, Q5_K: term = dx * ( f32(d) * (float)S  -  f32(dmin) * (float)M ),
 *             S = sum_j sc_j * dot_j,  M = sum_j m_j * bsum_j   (exact int32, j = 0..7)
 *       Q6_K: term = dx * ( f32(d) * (float)S ),  S = sum_s sc_s * dot_s   (s = 0..15)
 *   - row sum over blocks in f32, in one of two declared orders (see oracle_qmatvec).
 * Non-finite activations are outside the contract.
 *
 * RMSNorm with a residual add before the pack (oracle_rmsnorm): see its comment for the
 * reading of the formula and the declared order of the sum of squares.
 *
 * Parity pins (tests/test_oracle_pins.py): f16 decode against numpy's float16 over all 65536
 * bit patterns; Q4_K/Q6_K code maps are bijections onto the block's bits; q8_K invariants;
 * brute force in f64; closed-form special cases (unit scales, zero nibbles, q == 32).
 * Conformance of the two block layouts with GGUF files written by other software is
 * "parity unpinned": no such file is available to compare against.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 256
#define Q4K_BYTES 144
#define Q5K_BYTES 176
#define Q6K_BYTES 210
#define FMT_Q4_K 12 /* GGUF type id */
#define FMT_Q5_K 13 /* GGUF type id */
#define FMT_Q6_K 14 /* GGUF type id */

/* ---- IEEE 754 binary16 -> value, from the format's definition (exact). ----------------- */
static double half_value(uint16_t h)
{
    int sign = h >> 15;
    int expo = (h >> 10) & 31;
    int mant = h & 1023;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25); /* (1 + mant/1024) * 2^(expo-15) */
    return sign ? -v : v;
}

float oracle_f16_to_f32(uint16_t h) { return (float)half_value(h); }

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---- Q4_K block (144 bytes): [0,2) d f16, [2,4) dmin f16, [4,16) 12 bytes holding eight
 *      6-bit scales and eight 6-bit mins, [16,144) 128 bytes of 4-bit codes. ------------- */
static void q4k_scale_min(const uint8_t *s12, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s12[j] & 63;
        *m = s12[j + 4] & 63;
    } else {
        *sc = (s12[j + 4] & 15) | ((s12[j - 4] >> 6) << 4);
        *m = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

/* 4-bit code of element e (0..255) and its sub-block: each 32-byte chunk c of the code
 * bytes holds elements 64c..64c+31 in its low nibbles and 64c+32..64c+63 in its high ones. */
static int q4k_code(const uint8_t *qs, int e)
{
    int c = e / 64, t = e % 64;
    return t < 32 ? (qs[32 * c + t] & 15) : (qs[32 * c + t - 32] >> 4);
}

void oracle_q4k_fields(const uint8_t *blk, float *d, float *dmin, int32_t *sc, int32_t *m,
                       int32_t *q)
{
    *d = oracle_f16_to_f32(le16(blk));
    *dmin = oracle_f16_to_f32(le16(blk + 2));
    for (int j = 0; j < 8; ++j) {
        int a, b;
        q4k_scale_min(blk + 4, j, &a, &b);
        sc[j] = a;
        m[j] = b;
    }
    for (int e = 0; e < QK; ++e)
        q[e] = q4k_code(blk + 16, e);
}

/* weight value w_e = d * sc_j * q_e - dmin * m_j, evaluated exactly in f64 */
void oracle_q4k_dequant(const uint8_t *blk, double *w)
{
    float d, dmin;
    int32_t sc[8], m[8], q[QK];
    oracle_q4k_fields(blk, &d, &dmin, sc, m, q);
    for (int e = 0; e < QK; ++e) {
        int j = e / 32;
        w[e] = (double)d * sc[j] * q[e] - (double)dmin * m[j];
    }
}

/* ---- Q5_K block (176 bytes): [0,2) d f16, [2,4) dmin f16, [4,16) the twelve scale/min
 *      bytes packed as in Q4_K, [16,48) qh: the fifth bits, [48,176) 128 bytes of low 4-bit
 *      codes laid out as in Q4_K.  Element e = 64c + t (c = 0..3): the low four bits are
 *      q4k_code's; the fifth bit is bit 2c of qh[t] for t < 32 and bit 2c+1 of qh[t - 32]
 *      for t >= 32, so a code is in 0..31.  Sub-block j = e / 32 as in Q4_K. ------------ */
static int q5k_code(const uint8_t *blk, int e)
{
    const int c = e / 64, t = e % 64;
    const uint8_t *qh = blk + 16;
    const int high = t < 32 ? (qh[t] >> (2 * c)) & 1 : (qh[t - 32] >> (2 * c + 1)) & 1;
    return q4k_code(blk + 48, e) | (high << 4);
}

void oracle_q5k_fields(const uint8_t *blk, float *d, float *dmin, int32_t *sc, int32_t *m,
                       int32_t *q)
{
    *d = oracle_f16_to_f32(le16(blk));
    *dmin = oracle_f16_to_f32(le16(blk + 2));
    for (int j = 0; j < 8; ++j) {
        int a, b;
        q4k_scale_min(blk + 4, j, &a, &b);
        sc[j] = a;
        m[j] = b;
    }
    for (int e = 0; e < QK; ++e)
        q[e] = q5k_code(blk, e);
}

/* weight value w_e = d * sc_j * q_e - dmin * m_j, evaluated exactly in f64 */
void oracle_q5k_dequant(const uint8_t *blk, double *w)
{
    float d, dmin;
    int32_t sc[8], m[8], q[QK];
    oracle_q5k_fields(blk, &d, &dmin, sc, m, q);
    for (int e = 0; e < QK; ++e) {
        int j = e / 32;
        w[e] = (double)d * sc[j] * q[e] - (double)dmin * m[j];
    }
}

/* ---- Q6_K block (210 bytes): [0,128) ql low nibbles, [128,192) qh 2-bit highs,
 *      [192,208) sixteen int8 scales (one per 16 values), [208,210) d f16. ------------- */
static int q6k_code(const uint8_t *ql, const uint8_t *qh, int e)
{
    int h = e / 128, w = e % 128, t = w / 32, l = w % 32;
    int low4 = (ql[64 * h + 32 * (t & 1) + l] >> (4 * (t >> 1))) & 15;
    int high2 = (qh[32 * h + l] >> (2 * t)) & 3;
    return low4 | (high2 << 4); /* 0..63, stored with an offset of 32 */
}

void oracle_q6k_fields(const uint8_t *blk, float *d, int32_t *sc, int32_t *q)
{
    *d = oracle_f16_to_f32(le16(blk + 208));
    for (int s = 0; s < 16; ++s)
        sc[s] = (int8_t)blk[192 + s];
    for (int e = 0; e < QK; ++e)
        q[e] = q6k_code(blk, blk + 128, e);
}

/* weight value w_e = d * sc_{e/16} * (q_e - 32), exact in f64 */
void oracle_q6k_dequant(const uint8_t *blk, double *w)
{
    float d;
    int32_t sc[16], q[QK];
    oracle_q6k_fields(blk, &d, sc, q);
    for (int e = 0; e < QK; ++e)
        w[e] = (double)d * sc[e / 16] * (q[e] - 32);
}

/* ---- q8_K pack of one f32 vector of length K (K % 256 == 0). ----------------------------
 * Per 256-value block: amax = max |x|; if amax == 0 everything is 0; otherwise
 * iscale = 127/amax (f32 division), q = clamp(rint(x * iscale), -127, 127) with the product
 * rounded to f32 first and rint to nearest-even, d = amax / 127 (f32 division), and
 * bsums[j] = sum of the 32 codes of sub-block j.  A product that is NaN (x = 0 in a block so
 * small that 127/amax overflows to infinity) gives code 0. */
void oracle_q8k_pack(const float *x, int64_t K, int8_t *qs, float *d, int16_t *bsums)
{
    for (int64_t b = 0; b < K / QK; ++b) {
        const float *xb = x + b * QK;
        int8_t *qb = qs + b * QK;
        float amax = 0.0f;
        for (int i = 0; i < QK; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax)
                amax = a;
        }
        if (amax == 0.0f) {
            d[b] = 0.0f;
            memset(qb, 0, QK);
            for (int j = 0; j < 8; ++j)
                bsums[b * 8 + j] = 0;
            continue;
        }
        float iscale = 127.0f / amax;
        for (int i = 0; i < QK; ++i) {
            float v = xb[i] * iscale;
            /* 127/amax overflows to +inf when amax < 127/FLT_MAX; then 0 * inf is NaN: code 0 */
            float r = isnan(v) ? 0.0f : nearbyintf(v); /* nearest, ties to even */
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            qb[i] = (int8_t)r;
        }
        d[b] = amax / 127.0f;
        for (int j = 0; j < 8; ++j) {
            int s = 0;
            for (int i = 0; i < 32; ++i)
                s += qb[32 * j + i];
            bsums[b * 8 + j] = (int16_t)s;
        }
    }
}

/* ---- integer sub-block dots of one row against one packed vector. ----------------------
 * Q4_K: dots[b*8 + j]  = sum over the 32 elements of sub-block j of q_e * x8_e
 * Q6_K: dots[b*16 + s] = sum over the 16 elements of group s of (q_e - 32) * x8_e          */
void oracle_q4k_subdots(const uint8_t *row, const int8_t *qs, int64_t K, int32_t *dots)
{
    for (int64_t b = 0; b < K / QK; ++b) {
        float d, dmin;
        int32_t sc[8], m[8], q[QK];
        oracle_q4k_fields(row + b * Q4K_BYTES, &d, &dmin, sc, m, q);
        for (int j = 0; j < 8; ++j) {
            int32_t s = 0;
            for (int i = 0; i < 32; ++i)
                s += q[32 * j + i] * qs[b * QK + 32 * j + i];
            dots[b * 8 + j] = s;
        }
    }
}

void oracle_q5k_subdots(const uint8_t *row, const int8_t *qs, int64_t K, int32_t *dots)
{
    for (int64_t b = 0; b < K / QK; ++b) {
        float d, dmin;
        int32_t sc[8], m[8], q[QK];
        oracle_q5k_fields(row + b * Q5K_BYTES, &d, &dmin, sc, m, q);
        for (int j = 0; j < 8; ++j) {
            int32_t s = 0;
            for (int i = 0; i < 32; ++i)
                s += q[32 * j + i] * qs[b * QK + 32 * j + i];
            dots[b * 8 + j] = s;
        }
    }
}

void oracle_q6k_subdots(const uint8_t *row, const int8_t *qs, int64_t K, int32_t *dots)
{
    for (int64_t b = 0; b < K / QK; ++b) {
        float d;
        int32_t sc[16], q[QK];
        oracle_q6k_fields(row + b * Q6K_BYTES, &d, sc, q);
        for (int s = 0; s < 16; ++s) {
            int32_t acc = 0;
            for (int i = 0; i < 16; ++i)
                acc += (q[16 * s + i] - 32) * qs[b * QK + 16 * s + i];
            dots[b * 16 + s] = acc;
        }
    }
}

/* ---- the rank-one epilogue: one f32 term per 256-value block. --------------------------*/
void oracle_block_terms(int fmt, const uint8_t *row, const int8_t *qs, const float *xd,
                        const int16_t *bsums, int64_t K, float *terms)
{
    int64_t nb = K / QK;
    for (int64_t b = 0; b < nb; ++b) {
        if (fmt == FMT_Q4_K || fmt == FMT_Q5_K) {
            float d, dmin;
            int32_t sc[8], m[8], q[QK], dots[8];
            if (fmt == FMT_Q4_K) {
                const uint8_t *blk = row + b * Q4K_BYTES;
                oracle_q4k_fields(blk, &d, &dmin, sc, m, q);
                oracle_q4k_subdots(blk, qs + b * QK, QK, dots);
            } else {
                const uint8_t *blk = row + b * Q5K_BYTES;
                oracle_q5k_fields(blk, &d, &dmin, sc, m, q);
                oracle_q5k_subdots(blk, qs + b * QK, QK, dots);
            }
            int32_t S = 0, M = 0;
            for (int j = 0; j < 8; ++j) {
                S += sc[j] * dots[j];
                M += m[j] * bsums[b * 8 + j];
            }
            float fS = (float)S, fM = (float)M;
            float a = d * fS;
            float c = dmin * fM;
            float inner = a - c;
            terms[b] = xd[b] * inner;
        } else {
            const uint8_t *blk = row + b * Q6K_BYTES;
            float d;
            int32_t sc[16], q[QK], dots[16];
            oracle_q6k_fields(blk, &d, sc, q);
            oracle_q6k_subdots(blk, qs + b * QK, QK, dots);
            int32_t S = 0;
            for (int s = 0; s < 16; ++s)
                S += sc[s] * dots[s];
            float fS = (float)S;
            float inner = d * fS;
            terms[b] = xd[b] * inner;
        }
    }
}

/* ---- y[v][r] = sum over blocks of the block terms, in f32. ------------------------------
 * order 0: ascending blocks, left to right:  ((t0 + t1) + t2) + ...
 * order 1: blocks in groups of four, each group summed as (t0 + t1) + (t2 + t3) with an
 *          absent block (past the row's end) counted as +0.0f, then the group sums added
 *          left to right: ((G0 + G1) + G2) + ...
 * order 2: as order 1 within runs of four groups (16 blocks): each run's group sums added
 *          left to right, ((G0 + G1) + G2) + G3, absent groups past the row's end counted as
 *          +0.0f; then the run sums added left to right: ((R0 + R1) + R2) + ...
 *          This is the order the GPU path declares for its reduction (for rows of at most 16
 *          blocks it equals order 1); the oracle states it independently.
 * W is canonical GGUF blocks [rows][K/256][144, 176 or 210]; the packed vectors are batch-major:
 * qs [batch][K], xd [batch][K/256], bsums [batch][K/256][8]; y is [batch][rows].
 * Returns 0, or non-zero (and writes nothing) for a shape it is not defined on or when the
 * per-row scratch cannot be allocated; any row length is accepted.                          */
int oracle_qmatvec(int fmt, const uint8_t *W, const int8_t *qs, const float *xd,
                   const int16_t *bsums, int64_t rows, int64_t K, int batch, int order,
                   float *y)
{
    int64_t nb = K / QK;
    int64_t bb = fmt == FMT_Q4_K ? Q4K_BYTES : fmt == FMT_Q5_K ? Q5K_BYTES : Q6K_BYTES;
    if (nb < 1 || K % QK != 0 || rows < 0 || batch < 1)
        return 1; /* not a shape the mat-vec is defined on: nothing written */
    float *terms = (float *)malloc((size_t)nb * sizeof(float));
    if (!terms)
        return 2; /* out of memory: nothing written */
    for (int v = 0; v < batch; ++v) {
        for (int64_t r = 0; r < rows; ++r) {
            oracle_block_terms(fmt, W + r * nb * bb, qs + v * K, xd + v * nb,
                               bsums + v * nb * 8, K, terms);
            float acc;
            if (order == 0) {
                acc = terms[0];
                for (int64_t b = 1; b < nb; ++b)
                    acc = acc + terms[b];
            } else if (order == 1) {
                acc = 0.0f;
                for (int64_t g = 0; g < (nb + 3) / 4; ++g) {
                    float t[4];
                    for (int i = 0; i < 4; ++i)
                        t[i] = (4 * g + i < nb) ? terms[4 * g + i] : 0.0f;
                    float G = (t[0] + t[1]) + (t[2] + t[3]);
                    acc = (g == 0) ? G : acc + G;
                }
            } else {
                acc = 0.0f;
                for (int64_t run = 0; run < (nb + 15) / 16; ++run) {
                    float Rs = 0.0f;
                    for (int64_t gi = 0; gi < 4; ++gi) {
                        const int64_t g = 4 * run + gi;
                        float t[4];
                        for (int i = 0; i < 4; ++i)
                            t[i] = (4 * g + i < nb) ? terms[4 * g + i] : 0.0f;
                        float G = (t[0] + t[1]) + (t[2] + t[3]);
                        Rs = (gi == 0) ? G : Rs + G;
                    }
                    acc = (run == 0) ? Rs : acc + Rs;
                }
            }
            y[v * rows + r] = acc;
        }
    }
    free(terms);
    return 0;
}

/* ---- brute force: dequantise W and x_hat = dx * q8 to f64 and sum in f64. ------------- */
void oracle_qmatvec_f64(int fmt, const uint8_t *W, const int8_t *qs, const float *xd,
                        int64_t rows, int64_t K, int batch, double *y)
{
    int64_t nb = K / QK;
    int64_t bb = fmt == FMT_Q4_K ? Q4K_BYTES : fmt == FMT_Q5_K ? Q5K_BYTES : Q6K_BYTES;
    double w[QK];
    for (int v = 0; v < batch; ++v) {
        for (int64_t r = 0; r < rows; ++r) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = W + (r * nb + b) * bb;
                if (fmt == FMT_Q4_K)
                    oracle_q4k_dequant(blk, w);
                else if (fmt == FMT_Q5_K)
                    oracle_q5k_dequant(blk, w);
                else
                    oracle_q6k_dequant(blk, w);
                for (int i = 0; i < QK; ++i)
                    acc += w[i] * ((double)xd[v * nb + b] * qs[v * K + b * QK + i]);
            }
            y[v * rows + r] = acc;
        }
    }
}

/* ---- bind-time Q6_K split: each 210-byte block becomes a 208-byte body (ql, qh, scales,
 * unchanged) and its f16 super-scale d goes to a prefix array of row stride prefix_stride
 * (entries); padding entries of a prefix row are zero.                                    */
void oracle_q6k_split(const uint8_t *gguf, int64_t rows, int64_t K, uint8_t *body,
                      uint16_t *prefix, int64_t prefix_stride)
{
    int64_t nb = K / QK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < prefix_stride; ++i)
            prefix[r * prefix_stride + i] = 0;
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *src = gguf + (r * nb + b) * Q6K_BYTES;
            memcpy(body + (r * nb + b) * 208, src, 208);
            prefix[r * prefix_stride + b] = le16(src + 208);
        }
    }
}

/* ---- RMSNorm with an optional residual add, the step before the q8_K pack. -----------------
 * "Language models on the device: the cajeta-llm kernels", §2.6 lists the normalisation and
 * residual kernels (rmsnorm*, add*) beside the device q8_K quantiser; in a decode step they
 * produce the activation that the quantiser packs.  The pages print no formula.  The reading
 * taken here is the usual root-mean-square norm with a learned per-element gain g:
 *     h_i = x_i + r_i               (r absent: h = x; h is the new residual stream)
 *     ms  = (sum_i h_i * h_i) / K
 *     n_i = (h_i * (1 / sqrt(ms + eps))) * g_i
 * every f32 operation rounded on its own; sqrt and the two divisions are IEEE-correctly
 * rounded.  The packed codes depend on the bits of n, so the order of the sum of squares is
 * declared (the GPU path declares the same one):
 *     lane t in [0, 256) adds the squares h_{t+256j}^2 for j = 0, 1, 2, ... left to right;
 *     each group of 32 lanes (32w .. 32w+31) is added as a pairwise tree, v[l] = v[l] + v[l+s]
 *     for s = 16, 8, 4, 2, 1 and l < s, leaving the group total in v[0];
 *     the eight group totals are added left to right.
 * x, r, h, n: f32 [K]; g: f32 [K]; K % 256 == 0.                                             */
void oracle_rmsnorm(const float *x, const float *r, const float *g, float eps, int64_t K, float *h, float *n)
{
    float lane[256];
    for (int t = 0; t < 256; ++t)
        lane[t] = 0.0f;
    for (int64_t i = 0; i < K; ++i) {
        h[i] = r ? x[i] + r[i] : x[i];
        const float sq = h[i] * h[i];
        lane[i % 256] = lane[i % 256] + sq;
    }
    float total = 0.0f;
    for (int w = 0; w < 8; ++w) {
        float *v = lane + 32 * w;
        for (int s = 16; s >= 1; s /= 2)
            for (int l = 0; l < s; ++l)
                v[l] = v[l] + v[l + s];
        total = (w == 0) ? v[0] : total + v[0];
    }
    const float ms = total / (float)K;
    const float inv = 1.0f / sqrtf(ms + eps);
    for (int64_t i = 0; i < K; ++i) {
        const float hn = h[i] * inv;
        n[i] = hn * g[i];
    }
}

/* RMSNorm (above) of one vector, then its q8_K pack (oracle_q8k_pack). */
void oracle_rmsnorm_q8k_pack(const float *x, const float *r, const float *g, float eps, int64_t K, float *h,
                             float *n, int8_t *qs, float *d, int16_t *bsums)
{
    oracle_rmsnorm(x, r, g, eps, K, h, n);
    oracle_q8k_pack(n, K, qs, d, bsums);
}
