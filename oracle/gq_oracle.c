/*
 * gq_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar CPU restatement of what the low-bit matvec/matmul path computes, written
 * from the pages' definitions.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it; the product library never does, and the two share no code.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (no contraction of a*b+c into an fma,
 * which GCC does by default on aarch64).  Every floating-point step below is a single IEEE
 * binary32 operation in round-to-nearest-even; fmaf() is the C99 correctly rounded fused
 * multiply-add.
 *
 * Sources (page title, section):
 *  [P1] browseml-gpu.js (browseML / bankML), header comment and Q1_DOT_WGSL / Q1_MM_WGSL /
 *       Q1_MM4_WGSL, fn f16, fn fma_exact.
 *  [P2] kopitiam-gpu block_q8_matmul_nt.wgsl, header ("PACKING", "ACCUMULATION ORDER") and
 *       fn quant_at / fn main.
 *  [P3] "BonsaiのWebGPUカーネルを読み解く", the ternary P/N bitplane identity and the
 *       decode/prefill kernel figure (q1_bits, q1_scales).
 *  [P4] web-xpu-ops README, the op table (matvecQ8, matvecQ4G128, matmulQ8, matmulQ4G128) and
 *       "The q4 format (W4A32, group-128)".
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - Q8_0 activation quantizer (not on the pages): amax over 32, d = amax/127 (RN), stored as
 *    f16 rounded to nearest even, q = clamp(round-half-up(x/d), -127, 127), amax = 0 -> d = 0,
 *    q = 0.  Round half up follows web-xpu-ops' Math.round convention.
 *  - Bonsai prefill with Q8_0 activations: integer block sum S per 32 weights (bit 1 -> +q,
 *    bit 0 -> -q with the int8 wrapping negate), p = d_x * S (exact), acc = fma(w_s, p, acc),
 *    blocks in ascending order from +0.
 *  - block_q8_matmul_nt: products and sums are separate RN operations, as written in the WGSL.
 *  - Bonsai decode GEMV over f32 activations: the page leaves the float order open, so the
 *    oracle is the f64 definition and the GPU result is checked within a stated bound.
 *  - W8A32 / W4A32 group-128 matvec and matmul: the page states the packing and where the scale
 *    applies (per row after the dot product; per 128-column group) but no float order, so the
 *    oracle is the f64 definition.  The matmul's weight is the right-hand operand with the
 *    matvec's [rows, K] layout: out[t][n] = the matvec of weight row n with activation row t.
 *
 * Parity status: every function here is pinned by tests against closed forms, brute force or
 * library routines (see tests/test_oracle_*.py).  Bit-level agreement with bankML's own
 * vec_dot_ref binary, which the pages do not reproduce, is not claimed.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define QK1_0 128
#define QK8_0 32
#define Q1_0_BYTES 18
#define Q8_0_BYTES 34

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static int32_t sext8(uint32_t b) { b &= 0xffu; return b >= 128u ? (int32_t)b - 256 : (int32_t)b; }
/* int8 negate that wraps as the reference's i8 arithmetic does: -(-128) stays -128 [P1 kernel]. */
static int32_t neg_i8_wrap(int32_t q) { return q == -128 ? -128 : -q; }
static uint32_t le16(const uint8_t* p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }

/* [P1] fn f16: half-precision bits to f32 with integer operations only.  Zero exponent: the
 * value m * 2^-24 (exact, covers subnormals); exponent 31: Inf/NaN by bit assembly (payload
 * kept); otherwise rebias the exponent by 112 and widen the mantissa. */
float gqo_f16_to_f32(uint16_t h) {
    uint32_t sgn = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = ((uint32_t)h >> 10) & 0x1fu;
    uint32_t m = (uint32_t)h & 0x3ffu;
    if (e == 0u) {
        float v = (float)m * 5.9604644775390625e-8f; /* 2^-24 */
        return sgn ? -v : v;
    }
    if (e == 31u) return bits_to_f32(sgn | 0x7f800000u | (m << 13));
    return bits_to_f32(sgn | ((e + 112u) << 23) | (m << 13));
}

/* f32 -> f16, round to nearest, ties to even (IEEE 754 convertFormat).  Our own integer
 * routine, used only by the activation quantizer reading. */
uint16_t gqo_f32_to_f16_rne(float f) {
    uint32_t x = f32_to_bits(f);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) {                       /* Inf or NaN */
        if (ax == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | 0x7e00u | ((ax >> 13) & 0x3ffu));   /* quiet NaN */
    }
    int32_t e = (int32_t)(ax >> 23) - 127;       /* unbiased exponent */
    uint32_t man = ax & 0x7fffffu;
    if (e >= 16) return (uint16_t)(sign | 0x7c00u);   /* >= 2^16: overflow */
    if (e >= -14) {                                 /* normal f16 range */
        uint32_t h = ((uint32_t)(e + 15) << 10) | (man >> 13);
        uint32_t rem = man & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;   /* may carry to Inf */
        return (uint16_t)(sign | h);
    }
    /* subnormal f16: value / 2^-24 = M / 2^s with M the 24-bit significand */
    uint32_t M = man | 0x800000u;
    int32_t s = -e - 1;
    if (e == -127) return (uint16_t)sign;           /* f32 zero or subnormal: far below 2^-25 */
    if (s > 24) return (uint16_t)sign;
    uint32_t q = M >> s;
    uint32_t rem = M & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
}

/* [P1] fn fma_exact restated from its mathematics: b split into a 12-bit head and an exact
 * tail, Knuth's TwoSum for the exact sum and error, then Boldo-Melquiond round-to-odd of the
 * correction before the final add.  a must carry at most 12 significant bits (an f16 does).
 * Kept only to pin the reading that the page's fma is correctly rounded (== fmaf). */
static void two_sum(float a, float b, float* s, float* e) {
    volatile float vs = a + b;
    volatile float bb = vs - a;
    volatile float sb = vs - bb;
    *s = vs;
    *e = (a - sb) + (b - bb);
}
float gqo_fma_emulated(float a, float b, float c) {
    float bhi = bits_to_f32(f32_to_bits(b) & 0xfffff000u);
    float blo = b - bhi;
    float ux, uy, tx, ty, vx, vy;
    two_sum(a * bhi, a * blo, &ux, &uy);
    two_sum(c, ux, &tx, &ty);
    two_sum(ty, uy, &vx, &vy);
    uint32_t vb = f32_to_bits(vx);
    if ((vb & 1u) == 0u && vy != 0.0f) vb = ((vx > 0.0f) == (vy > 0.0f)) ? vb + 1u : vb - 1u;
    return tx + bits_to_f32(vb);
}

/* [P1] Q1_DOT_WGSL, one row: per 128 weights (block i) the f16 d0 and 128 sign bits; per 32
 * activations (sub-block k = 0..3 of block i, i.e. Q8_0 block 4i+k) the f16 d1 and 32 int8.
 * Weight e of sub-block k sits in byte 2 + 4k + e/8, bit e%8 of the Q1_0 block; bit 1 selects
 * +q, bit 0 the wrapping negate.  Eight lanes l sum four weights each (e = 4l..4l+3):
 *   prod = d1 * f32(s)           (exact)
 *   ab[l] = prod (k = 0), ab[l] = prod + ab[l] (k = 1..3)
 *   acc[l] = fma(d0, ab[l], acc[l])  (correctly rounded), acc from +0
 * and the row result is ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)).  `lanes`, when not NULL,
 * receives the eight accumulators before the final reduction. */
float gqo_q1_q8_row(const uint8_t* wrow, const uint8_t* act, int n, float* lanes) {
    int nb = n / QK1_0;
    float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    for (int i = 0; i < nb; i++) {
        const uint8_t* wb = wrow + (size_t)i * Q1_0_BYTES;
        float d0 = gqo_f16_to_f32((uint16_t)le16(wb));
        float ab[8];
        for (int k = 0; k < 4; k++) {
            const uint8_t* ab8 = act + (size_t)(4 * i + k) * Q8_0_BYTES;
            float d1 = gqo_f16_to_f32((uint16_t)le16(ab8));
            for (int l = 0; l < 8; l++) {
                int32_t s = 0;
                for (int e = 4 * l; e < 4 * l + 4; e++) {
                    int32_t q = sext8(ab8[2 + e]);
                    uint32_t bit = ((uint32_t)wb[2 + 4 * k + e / 8] >> (e % 8)) & 1u;
                    s += bit ? q : neg_i8_wrap(q);
                }
                float prod = d1 * (float)s;
                if (k == 0) {
                    ab[l] = prod;
                } else {
                    float t = prod + ab[l];
                    ab[l] = t;
                }
            }
        }
        for (int l = 0; l < 8; l++) acc[l] = fmaf(d0, ab[l], acc[l]);
    }
    if (lanes) for (int l = 0; l < 8; l++) lanes[l] = acc[l];
    float s04 = acc[0] + acc[4], s26 = acc[2] + acc[6];
    float s15 = acc[1] + acc[5], s37 = acc[3] + acc[7];
    float lo = s04 + s26, hi = s15 + s37;
    return lo + hi;
}

/* [P1] Q1_DOT_WGSL over all rows: y[r] for weights w (rows x n/128 blocks of 18 bytes) and one
 * Q8_0 vector a (n/32 blocks of 34 bytes). */
void gqo_q1_q8_gemv(const uint8_t* w, const uint8_t* a, float* y, int rows, int n) {
    size_t row_bytes = (size_t)(n / QK1_0) * Q1_0_BYTES;
    for (int r = 0; r < rows; r++) y[r] = gqo_q1_q8_row(w + (size_t)r * row_bytes, a, n, 0);
}

/* [P1] Q1_MM_WGSL / Q1_MM4_WGSL: `cols` activation vectors; every (row, column) is the
 * Q1_DOT_WGSL chain, stored at O[c * rows + r]. */
void gqo_q1_q8_gemm(const uint8_t* w, const uint8_t* a, float* y, int rows, int n, int cols) {
    size_t row_bytes = (size_t)(n / QK1_0) * Q1_0_BYTES;
    size_t act_bytes = (size_t)(n / QK8_0) * Q8_0_BYTES;
    for (int c = 0; c < cols; c++)
        for (int r = 0; r < rows; r++)
            y[(size_t)c * rows + r] = gqo_q1_q8_row(w + (size_t)r * row_bytes, a + (size_t)c * act_bytes, n, 0);
}

/* [P2] quant_at: element `index` of the packed quants is byte index%4 of word index/4,
 * sign-extended from 8 bits. */
static float quant_at(const uint32_t* quants, size_t index) {
    uint32_t word = quants[index / 4];
    uint32_t byte = (word >> ((index % 4) * 8)) & 0xffu;
    return (float)sext8(byte);
}

/* [P2] block_q8_matmul_nt: y[row, col] = sum over blocks b of scale[col, b] * block_sum_b with
 * block_sum_b = sum_{t<32} x[row, 32b+t] * quant[col, 32b+t]; every product and every sum is a
 * separate RN operation, t and b ascending, sums from +0. */
void gqo_block_q8_matmul_nt(const float* x, const uint32_t* quants, const float* scales, float* y,
                            int m, int k, int n) {
    int nbk = k / QK8_0;
    for (int row = 0; row < m; row++) {
        for (int col = 0; col < n; col++) {
            float acc = 0.0f;
            for (int b = 0; b < nbk; b++) {
                float block_sum = 0.0f;
                for (int t = 0; t < QK8_0; t++) {
                    float xv = x[(size_t)row * k + (size_t)b * QK8_0 + t];
                    float qv = quant_at(quants, (size_t)col * k + (size_t)b * QK8_0 + t);
                    float prod = xv * qv;
                    block_sum = block_sum + prod;
                }
                float sp = scales[(size_t)col * nbk + b] * block_sum;
                acc = acc + sp;
            }
            y[(size_t)row * n + col] = acc;
        }
    }
}

static int32_t popcount32(uint32_t v) {
    int32_t c = 0;
    while (v) { c += (int32_t)(v & 1u); v >>= 1; }
    return c;
}

/* [P3] ternary weights as bitplanes: w = P - N per element; X bit 1 -> +1, bit 0 -> -1.
 * Direct form: sum over elements of w * x. */
void gqo_ternary_direct(const uint32_t* P, const uint32_t* N, const uint32_t* X, int32_t* y,
                        int rows, int k, int batch) {
    int nw = k / 32;
    for (int b = 0; b < batch; b++)
        for (int r = 0; r < rows; r++) {
            int32_t acc = 0;
            for (int j = 0; j < k; j++) {
                int32_t pw = (int32_t)((P[(size_t)r * nw + j / 32] >> (j % 32)) & 1u);
                int32_t nw_ = (int32_t)((N[(size_t)r * nw + j / 32] >> (j % 32)) & 1u);
                int32_t xv = ((X[(size_t)b * nw + j / 32] >> (j % 32)) & 1u) ? 1 : -1;
                acc += (pw - nw_) * xv;
            }
            y[(size_t)b * rows + r] = acc;
        }
}

/* [P3] the popcount identity, word by word:
 *   dot = 2 * (popc(P & X) - popc(N & X)) - popc(P) + popc(N). */
void gqo_ternary_identity(const uint32_t* P, const uint32_t* N, const uint32_t* X, int32_t* y,
                          int rows, int k, int batch) {
    int nw = k / 32;
    for (int b = 0; b < batch; b++)
        for (int r = 0; r < rows; r++) {
            int32_t pa = 0, na = 0, pp = 0, nn = 0;
            for (int w = 0; w < nw; w++) {
                uint32_t p = P[(size_t)r * nw + w], q = N[(size_t)r * nw + w], x = X[(size_t)b * nw + w];
                pa += popcount32(p & x);
                na += popcount32(q & x);
                pp += popcount32(p);
                nn += popcount32(q);
            }
            y[(size_t)b * rows + r] = 2 * (pa - na) - pp + nn;
        }
}

/* Q8_0 activation quantizer (reading; not on the pages): per 32-block, amax = max |x|,
 * d = amax / 127 (RN), stored f16 = RN-even(d); q = clamp(round-half-up(x / d), -127, 127)
 * with the division by the f32 d; amax == 0 gives d = 0 and q = 0.
 * Round half up: floor(v) + (v - floor(v) >= 0.5). */
void gqo_quantize_q8_0(const float* x, int m, int k, uint16_t* d_out, int8_t* q_out) {
    int nbk = k / QK8_0;
    for (int row = 0; row < m; row++)
        for (int b = 0; b < nbk; b++) {
            const float* xb = x + (size_t)row * k + (size_t)b * QK8_0;
            float amax = 0.0f;
            for (int t = 0; t < QK8_0; t++) {
                float v = fabsf(xb[t]);
                if (v > amax) amax = v;
            }
            float d = amax / 127.0f;
            d_out[(size_t)row * nbk + b] = gqo_f32_to_f16_rne(d);
            for (int t = 0; t < QK8_0; t++) {
                int32_t qi = 0;
                if (amax != 0.0f) {
                    float v = xb[t] / d;
                    float fl = floorf(v);
                    float frac = v - fl;
                    qi = (int32_t)fl + (frac >= 0.5f ? 1 : 0);
                    if (qi > 127) qi = 127;
                    if (qi < -127) qi = -127;
                }
                q_out[(size_t)row * k + (size_t)b * QK8_0 + t] = (int8_t)qi;
            }
        }
}

/* [P3] Bonsai 1-bit weights (one u32 = 32 sign bits, one f32 scale per 32 weights) against
 * Q8_0 activations (reading): per (m, n) and block b ascending,
 *   S = sum_t (bit ? q : neg_i8_wrap(q)),  p = d_x[m,b] * f32(S) (exact),
 *   acc = fma(w_s[n,b], p, acc) from +0;  y[m * N + n] = acc. */
void gqo_prefill_q1s32(const uint32_t* signs, const float* ws, const uint16_t* xd, const int8_t* xq,
                       float* y, int M, int N, int K) {
    int nbk = K / QK8_0;
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
            float acc = 0.0f;
            for (int b = 0; b < nbk; b++) {
                uint32_t word = signs[(size_t)n * nbk + b];
                int32_t S = 0;
                for (int t = 0; t < QK8_0; t++) {
                    int32_t q = (int32_t)xq[(size_t)m * K + (size_t)b * QK8_0 + t];
                    S += ((word >> t) & 1u) ? q : neg_i8_wrap(q);
                }
                float p = gqo_f16_to_f32(xd[(size_t)m * nbk + b]) * (float)S;
                acc = fmaf(ws[(size_t)n * nbk + b], p, acc);
            }
            y[(size_t)m * N + n] = acc;
        }
}

/* [P3] Bonsai decode GEMV over f32 activations (llama-decode-q1-proj.wgsl in the decode/prefill
 * figure): each weight is +1.0 (bit 1) or -1.0 (bit 0), a 32-weight block carries one f32 scale,
 * and the page accumulates dot(x4, s4) per four weights into acc with the block's scale.  The
 * page does not fix the order of the float operations, so this is the plain definition in f64:
 *   y[m * N + n] = sum_b ws[n, b] * sum_t s(n, 32 b + t) * x[m, 32 b + t],
 * every product and sum in binary64, blocks and weights in ascending order. */
void gqo_q1s32_f32_gemv_f64(const uint32_t* signs, const float* ws, const float* x, double* y, int M, int N,
                            int K) {
    int nbk = K / QK8_0;
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (int b = 0; b < nbk; b++) {
                uint32_t word = signs[(size_t)n * nbk + b];
                double d = 0.0;
                for (int t = 0; t < QK8_0; t++) {
                    double xv = (double)x[(size_t)m * K + (size_t)b * QK8_0 + t];
                    d += ((word >> t) & 1u) ? xv : -xv;
                }
                acc += (double)ws[(size_t)n * nbk + b] * d;
            }
            y[(size_t)m * N + n] = acc;
        }
}

/* W8A32 ([P4] matvecQ8 / matmulQ8): code k of weight row n is byte (k % 4) of word
 * w[n * ceil(K/4) + k / 4], least-significant byte first, read as a signed (two's complement)
 * byte; scale[n] multiplies the row's dot product once:
 *   y[t * N + n] = scale[n] * sum_k q(n, k) * x[t * K + k]   (binary64, k ascending). */
void gqo_w8a32_f64(const uint32_t* w, const float* scale, const float* x, double* y, int T, int N, int K) {
    size_t wpr = ((size_t)K + 3) / 4;
    for (int t = 0; t < T; t++)
        for (int n = 0; n < N; n++) {
            double dot = 0.0;
            for (int k = 0; k < K; k++) {
                uint32_t word = w[(size_t)n * wpr + (size_t)k / 4];
                int8_t q = (int8_t)(uint8_t)(word >> (8 * (k % 4)));
                dot += (double)q * (double)x[(size_t)t * K + k];
            }
            y[(size_t)t * N + n] = (double)scale[n] * dot;
        }
}

/* W4A32 group-128 ([P4] matvecQ4G128 / matmulQ4G128, "The q4 format"): code k of weight row n
 * is nibble (k % 8) of word w[n * ceil(K/8) + k / 8], least-significant nibble first, read as a
 * 4-bit two's complement value (the quantizer emits [-7, 7]); scale[n * ceil(K/128) + g]
 * multiplies the dot product of the row's columns 128 g .. 128 g + 127:
 *   y[t * N + n] = sum_g scale[n, g] * sum_{k in g} q(n, k) * x[t * K + k]   (binary64). */
void gqo_w4a32g128_f64(const uint32_t* w, const float* scale, const float* x, double* y, int T, int N, int K) {
    size_t wpr = ((size_t)K + 7) / 8, gpr = ((size_t)K + 127) / 128;
    for (int t = 0; t < T; t++)
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (size_t g = 0; g < gpr; g++) {
                double dot = 0.0;
                for (int k = (int)(128 * g); k < K && k < (int)(128 * g + 128); k++) {
                    uint32_t nib = (w[(size_t)n * wpr + (size_t)k / 8] >> (4 * (k % 8))) & 0xFu;
                    int q = (int)(nib ^ 8u) - 8;
                    dot += (double)q * (double)x[(size_t)t * K + k];
                }
                acc += (double)scale[(size_t)n * gpr + g] * dot;
            }
            y[(size_t)t * N + n] = acc;
        }
}

/* Array helpers for exhaustive checks. */
void gqo_f16_to_f32_array(const uint16_t* h, float* out, size_t count) {
    for (size_t i = 0; i < count; i++) out[i] = gqo_f16_to_f32(h[i]);
}
void gqo_f32_to_f16_array(const float* f, uint16_t* out, size_t count) {
    for (size_t i = 0; i < count; i++) out[i] = gqo_f32_to_f16_rne(f[i]);
}
void gqo_fma_emulated_array(const float* a, const float* b, const float* c, float* out, size_t count) {
    for (size_t i = 0; i < count; i++) out[i] = gqo_fma_emulated(a[i], b[i], c[i]);
}
