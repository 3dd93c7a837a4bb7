/*
 * Oracle for the fused dequantize-and-multiply y = x @ W over GGUF/ggml-packed
 * weights. TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and
 * the bench's CPU-baseline leg may call it; the product path never does.
 *
 * Plain, slow, obviously correct C. It shares no code, header, table or
 * constant with the CUDA library: every format is decoded here from its byte
 * layout, one element at a time, and every sum is accumulated in double.
 *
 * What it follows:
 *  - rullama 0.5.0, src/backend/matmul.rs, module doc and `cpu_matmul_f32`:
 *    W is n rows of k weights (row j holds output column j), y[j] = sum_i
 *    w[j][i] * x[i]; the batched tests stack tokens as X[N x k] -> Y[N x n].
 *  - same page, `matmul_bf16` doc and `f32_to_bf16_bytes`: a bf16 value is
 *    the upper 16 bits of an f32.
 *  - same page, `matmul_f16`: IEEE binary16 weights.
 *  - same page, `matmul_q4_0` / `matmul_q4_k` / `matmul_q6_k`: block sizes
 *    (32 elements in 18 B; 256 in 144 B; 256 in 210 B).
 *  - rullama src/backend/dispatch/mod.rs, backward-input parity tests: the
 *    f16 d sits at bytes 0..2 of a Q4_0 block, Q4_K keeps d at 0..2 and
 *    dmin at 2..4, Q6_K keeps d at bytes 208..210.
 *  - rullama src/backend/dispatch/mod.rs, the expert-matmul tests (Q8_0 and Q5_0
 *    stacked experts): a Q8_0 block is an f16 d then 32 bytes of codes; a
 *    Q5_0 block is an f16 d, a 4-byte little-endian word of high bits, then
 *    16 bytes of nibbles (22 bytes per 32 elements); experts are stacked as
 *    whole [n rows x row bytes] slices, and position p, slot s uses the
 *    expert ids[p * top_k + s].
 *  - the remaining field layout inside the blocks (nibble order, 6-bit
 *    scale packing, Q6_K ql/qh/scales, which high bit of Q5_0 belongs to
 *    which element, Q8_0 codes as signed bytes) is the standard ggml block
 *    layout, which the pages name but do not print; it is written out below.
 *
 *  - rullama src/backend/dispatch/mod.rs, `MatmulBackInputParams` and the
 *    `matmul_q*_backward_input` dispatchers and parity tests: the gradient
 *    with respect to the input, dx[i] = sum_j w[j][i] * dy[j] for the rows
 *    j in [j_start, j_end) (the sum axis is tiled), written on the first
 *    tile and added on the others; dy has n entries, dx has k.
 *
 *  - moeflux tests/graph_diff_oracle.rs, the `EmbedGatherNTokens` test and
 *    the `MatvecNTokens (4-bit + 8-bit)` op it names: MLX-style affine
 *    weights, three arrays per matrix: codes packed into little-endian
 *    32-bit words ([n][k/8] words at 4 bits, 8 codes per word), a bf16
 *    scale and a bf16 bias per group of 64 consecutive weights of a row
 *    ([n][k/64] each), value = code * scale + bias; k a multiple of 64.
 *    Where the page leaves it open (the code order inside a word, the 8-bit
 *    packing) the plain reading is taken: code i of a word sits at bits
 *    bits*i .. bits*i + bits - 1 (lowest first), 32/bits codes per word;
 *    the value is rounded once to f32 (the page's GPU kernel contracts
 *    code * scale + bias into one fused multiply-add).
 *
 *  - gated FFN activations: rullama src/backend/dispatch/mod.rs, `silu_chained`
 *    (silu(x) = x * sigmoid(x)) and `geglu_chained` / the GeGLU backward
 *    tests (the GELU there is the tanh form, whose saturation the tests
 *    exercise); moeflux tests/graph_diff_oracle.rs, `SwigluFusedBatched`:
 *    out = act(gate) * up elementwise, gate = x Wg and up = x Wu two
 *    products of the same x. The tanh-form constants (sqrt(2/pi), 0.044715)
 *    are the published tanh approximation of GELU, which the pages name but
 *    do not print.
 *
 * Parity pins live in tests/test_oracle_pins.py (hand-packed blocks with
 * known values, closed-form sizes, exhaustive f16 decode against numpy,
 * identity / one-hot products, brute-force tiny products);
 * tests/test_oracle_mutations.py plants plausible mistakes in private copies
 * of this file and requires every one of them to fail a pin.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Format codes of this oracle (the Python wrapper maps names to them). */
enum { OR_BF16 = 0, OR_F16 = 1, OR_Q4_0 = 2, OR_Q4_K = 3, OR_Q6_K = 4, OR_Q8_0 = 5, OR_Q5_0 = 6 };

static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* IEEE binary16 -> exact value, decoded field by field. */
double oracle_f16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int mant = h & 1023;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* zero or subnormal */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25);  /* 1.mant * 2^(e-15) */
    return sign ? -v : v;
}

/* bf16 -> f32: the 16 bits become the upper half of an f32 word. */
float oracle_bf16_value(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Bytes of one packed row of k weights, or 0 if k does not fit the format. */
int64_t oracle_row_bytes(int fmt, int64_t k)
{
    if (k < 0) return 0;
    switch (fmt) {
    case OR_BF16:
    case OR_F16: return (k % 2 == 0) ? 2 * k : 0;
    case OR_Q4_0: return (k % 32 == 0) ? (k / 32) * 18 : 0;
    case OR_Q4_K: return (k % 256 == 0) ? (k / 256) * 144 : 0;
    case OR_Q6_K: return (k % 256 == 0) ? (k / 256) * 210 : 0;
    case OR_Q8_0: return (k % 32 == 0) ? (k / 32) * 34 : 0;
    case OR_Q5_0: return (k % 32 == 0) ? (k / 32) * 22 : 0;
    default: return 0;
    }
}

/* Q4_0 block: f16 d, then 16 bytes; element i (< 16) is the low nibble of
 * byte i, element i + 16 its high nibble; value = (q - 8) * d. */
static void dequant_q4_0_block(const uint8_t *blk, float *out)
{
    double d = oracle_f16_value(rd_u16(blk));
    const uint8_t *qs = blk + 2;
    for (int i = 0; i < 16; ++i) {
        int q_lo = qs[i] & 0x0F;
        int q_hi = qs[i] >> 4;
        out[i] = (float)((q_lo - 8) * d);
        out[i + 16] = (float)((q_hi - 8) * d);
    }
}

/* 6-bit scale and min of sub-block s of a Q4_K super-block (12 packed bytes):
 * s < 4 keeps them in the low 6 bits of bytes s and s+4; s >= 4 keeps the low
 * 4 bits in byte s+4 (scale low nibble, min high nibble) and the top 2 bits in
 * the top bits of bytes s-4 (scale) and s (min). */
static void q4_k_scale_min(const uint8_t *scales, int s, int *sc, int *m)
{
    if (s < 4) {
        *sc = scales[s] & 63;
        *m = scales[s + 4] & 63;
    } else {
        *sc = (scales[s + 4] & 0x0F) | ((scales[s - 4] >> 6) << 4);
        *m = (scales[s + 4] >> 4) | ((scales[s] >> 6) << 4);
    }
}

/* Q4_K super-block: d, dmin, 12 scale bytes, 128 quant bytes. Eight
 * sub-blocks of 32; the 64 elements 64c .. 64c+63 take the low nibbles of
 * qs[32c .. 32c+31] (sub-block 2c) then their high nibbles (sub-block 2c+1);
 * value = d*sc*q - dmin*m, exact in double, rounded once to f32. */
static void dequant_q4_k_block(const uint8_t *blk, float *out)
{
    double d = oracle_f16_value(rd_u16(blk));
    double dmin = oracle_f16_value(rd_u16(blk + 2));
    const uint8_t *scales = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        int sc0, m0, sc1, m1;
        q4_k_scale_min(scales, 2 * c, &sc0, &m0);
        q4_k_scale_min(scales, 2 * c + 1, &sc1, &m1);
        for (int l = 0; l < 32; ++l) {
            int q_lo = qs[32 * c + l] & 0x0F;
            int q_hi = qs[32 * c + l] >> 4;
            out[64 * c + l] = (float)(d * sc0 * q_lo - dmin * m0);
            out[64 * c + 32 + l] = (float)(d * sc1 * q_hi - dmin * m1);
        }
    }
}

/* Q6_K super-block: ql[128], qh[64], int8 scales[16], f16 d at 208. Each half
 * h of 128 elements uses ql[64h ..], qh[32h ..]; for l < 32 the four elements
 * 128h + l + 32r (r = 0..3) are:
 *   r=0: low nibble of ql[64h+l]    | bits 0-1 of qh[32h+l] << 4
 *   r=1: low nibble of ql[64h+32+l] | bits 2-3 of qh[32h+l] << 4
 *   r=2: high nibble of ql[64h+l]   | bits 4-5 of qh[32h+l] << 4
 *   r=3: high nibble of ql[64h+32+l]| bits 6-7 of qh[32h+l] << 4
 * value = d * scales[e/16] * (q - 32). */
static void dequant_q6_k_block(const uint8_t *blk, float *out)
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *scales = (const int8_t *)(blk + 192);
    double d = oracle_f16_value(rd_u16(blk + 208));
    for (int h = 0; h < 2; ++h) {
        const uint8_t *L = ql + 64 * h;
        const uint8_t *H = qh + 32 * h;
        for (int l = 0; l < 32; ++l) {
            int q[4];
            q[0] = (L[l] & 0x0F) | (((H[l] >> 0) & 3) << 4);
            q[1] = (L[l + 32] & 0x0F) | (((H[l] >> 2) & 3) << 4);
            q[2] = (L[l] >> 4) | (((H[l] >> 4) & 3) << 4);
            q[3] = (L[l + 32] >> 4) | (((H[l] >> 6) & 3) << 4);
            for (int r = 0; r < 4; ++r) {
                int e = 128 * h + l + 32 * r;
                out[e] = (float)(d * scales[e / 16] * (q[r] - 32));
            }
        }
    }
}

/* Q8_0 block: f16 d, then 32 signed bytes; value = q * d. */
static void dequant_q8_0_block(const uint8_t *blk, float *out)
{
    double d = oracle_f16_value(rd_u16(blk));
    for (int i = 0; i < 32; ++i) {
        int q = (int)(int8_t)blk[2 + i];
        out[i] = (float)(q * d);
    }
}

/* Q5_0 block: f16 d, a little-endian 32-bit word qh, 16 bytes qs; element
 * i (< 16) is the low nibble of qs[i] with bit i of qh as its fifth bit,
 * element i + 16 the high nibble of qs[i] with bit i + 16 of qh;
 * value = (q - 16) * d. */
static void dequant_q5_0_block(const uint8_t *blk, float *out)
{
    double d = oracle_f16_value(rd_u16(blk));
    uint32_t qh = (uint32_t)blk[2] | ((uint32_t)blk[3] << 8) | ((uint32_t)blk[4] << 16) |
                  ((uint32_t)blk[5] << 24);
    const uint8_t *qs = blk + 6;
    for (int i = 0; i < 16; ++i) {
        int q_lo = (qs[i] & 0x0F) | ((int)((qh >> i) & 1u) << 4);
        int q_hi = (qs[i] >> 4) | ((int)((qh >> (i + 16)) & 1u) << 4);
        out[i] = (float)((q_lo - 16) * d);
        out[i + 16] = (float)((q_hi - 16) * d);
    }
}

/* Dequantize one row of k weights into out[k]. Returns 0, or -1 on bad args. */
int oracle_dequant_row(int fmt, const uint8_t *row, int64_t k, float *out)
{
    if (oracle_row_bytes(fmt, k) == 0 && k != 0) return -1;
    switch (fmt) {
    case OR_BF16:
        for (int64_t i = 0; i < k; ++i) out[i] = oracle_bf16_value(rd_u16(row + 2 * i));
        return 0;
    case OR_F16:
        for (int64_t i = 0; i < k; ++i) out[i] = (float)oracle_f16_value(rd_u16(row + 2 * i));
        return 0;
    case OR_Q4_0:
        for (int64_t b = 0; b < k / 32; ++b) dequant_q4_0_block(row + 18 * b, out + 32 * b);
        return 0;
    case OR_Q4_K:
        for (int64_t b = 0; b < k / 256; ++b) dequant_q4_k_block(row + 144 * b, out + 256 * b);
        return 0;
    case OR_Q6_K:
        for (int64_t b = 0; b < k / 256; ++b) dequant_q6_k_block(row + 210 * b, out + 256 * b);
        return 0;
    case OR_Q8_0:
        for (int64_t b = 0; b < k / 32; ++b) dequant_q8_0_block(row + 34 * b, out + 32 * b);
        return 0;
    case OR_Q5_0:
        for (int64_t b = 0; b < k / 32; ++b) dequant_q5_0_block(row + 22 * b, out + 32 * b);
        return 0;
    default:
        return -1;
    }
}

/* Dequantize all n rows into out[n][k]. */
int oracle_dequant(int fmt, const uint8_t *w, int64_t k, int64_t n, float *out)
{
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    for (int64_t j = 0; j < n; ++j)
        if (oracle_dequant_row(fmt, w + j * rb, k, out + j * k)) return -1;
    return 0;
}

/* y[t][j] = sum_i x[t][i] * w[j][i] and s[t][j] = sum_i |x[t][i] * w[j][i]|,
 * both accumulated in double over the f32 weights and activations.
 * wrow_scratch holds k floats. */
int oracle_matmul(int fmt, const uint8_t *w, const float *x, int64_t k, int64_t n,
                  int64_t n_tokens, double *y, double *s, float *wrow_scratch)
{
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    for (int64_t j = 0; j < n; ++j) {
        if (oracle_dequant_row(fmt, w + j * rb, k, wrow_scratch)) return -1;
        for (int64_t t = 0; t < n_tokens; ++t) {
            const float *xt = x + t * k;
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < k; ++i) {
                double p = (double)xt[i] * (double)wrow_scratch[i];
                acc += p;
                mag += fabs(p);
            }
            y[t * n + j] = acc;
            s[t * n + j] = mag;
        }
    }
    return 0;
}

/* The same product for `count` chosen outputs (t_idx[c], j_idx[c]) only. */
int oracle_matmul_sampled(int fmt, const uint8_t *w, const float *x, int64_t k, int64_t n,
                          int64_t n_tokens, int64_t count, const int64_t *t_idx,
                          const int64_t *j_idx, double *y, double *s, float *wrow_scratch)
{
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    for (int64_t c = 0; c < count; ++c) {
        int64_t t = t_idx[c], j = j_idx[c];
        if (t < 0 || t >= n_tokens || j < 0 || j >= n) return -1;
        if (oracle_dequant_row(fmt, w + j * rb, k, wrow_scratch)) return -1;
        const float *xt = x + t * k;
        double acc = 0.0, mag = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            double p = (double)xt[i] * (double)wrow_scratch[i];
            acc += p;
            mag += fabs(p);
        }
        y[c] = acc;
        s[c] = mag;
    }
    return 0;
}

/* Backward with respect to the input (transposed product over a row range):
 * dx[i] = sum_{j in [j0, j1)} dy[j] * w[j][i] and s[i] = sum |dy[j] * w[j][i]|,
 * both accumulated in double; dy has n entries, dx and s have k.
 * wrow_scratch holds k floats. */
int oracle_matmul_back_input(int fmt, const uint8_t *w, const float *dy, int64_t k, int64_t n,
                             int64_t j0, int64_t j1, double *dx, double *s,
                             float *wrow_scratch)
{
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    if (j0 < 0 || j1 < j0 || j1 > n) return -1;
    for (int64_t i = 0; i < k; ++i) {
        dx[i] = 0.0;
        s[i] = 0.0;
    }
    for (int64_t j = j0; j < j1; ++j) {
        if (oracle_dequant_row(fmt, w + j * rb, k, wrow_scratch)) return -1;
        for (int64_t i = 0; i < k; ++i) {
            double p = (double)dy[j] * (double)wrow_scratch[i];
            dx[i] += p;
            s[i] += fabs(p);
        }
    }
    return 0;
}

/* Expert-indexed product: W holds n_experts slices of n rows; position p of
 * x [n_pos x k] and slot s (< top_k) use slice e = ids[p * top_k + s]:
 * y[(p * top_k + s) * n + j] = sum_i x[p][i] * w_e[j][i], and s likewise with
 * |x w|; double sums. Returns -1 on an id outside [0, n_experts). */
int oracle_matmul_experts(int fmt, const uint8_t *w, const float *x, int64_t k, int64_t n,
                          int64_t n_experts, int64_t n_pos, int64_t top_k, const int32_t *ids,
                          double *y, double *s, float *wrow_scratch)
{
    int64_t rb = oracle_row_bytes(fmt, k);
    if (rb == 0 && k != 0) return -1;
    for (int64_t p = 0; p < n_pos; ++p) {
        for (int64_t sl = 0; sl < top_k; ++sl) {
            int64_t e = ids[p * top_k + sl];
            if (e < 0 || e >= n_experts) return -1;
            const uint8_t *we = w + e * rb * n;
            for (int64_t j = 0; j < n; ++j) {
                if (oracle_dequant_row(fmt, we + j * rb, k, wrow_scratch)) return -1;
                double acc = 0.0, mag = 0.0;
                for (int64_t i = 0; i < k; ++i) {
                    double v = (double)x[p * k + i] * (double)wrow_scratch[i];
                    acc += v;
                    mag += fabs(v);
                }
                y[(p * top_k + sl) * n + j] = acc;
                s[(p * top_k + sl) * n + j] = mag;
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * MLX-style affine rows (4 or 8 bits per code, group size 64).
 * wrow: k*bits/8 bytes of little-endian 32-bit words; srow, brow: k/64 bf16
 * values each (2 bytes, little-endian). */

static uint32_t rd_u32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

int64_t oracle_affine_row_bytes(int bits, int64_t k)
{
    if ((bits != 4 && bits != 8) || k < 0 || k % 64) return -1;
    return k * bits / 8;
}

int oracle_dequant_affine_row(int bits, const uint8_t *wrow, const uint8_t *srow,
                              const uint8_t *brow, int64_t k, float *out)
{
    if (oracle_affine_row_bytes(bits, k) < 0) return -1;
    const int per_word = 32 / bits;
    const uint32_t mask = (1u << bits) - 1u;
    for (int64_t i = 0; i < k; ++i) {
        uint32_t word = rd_u32(wrow + 4 * (i / per_word));
        uint32_t q = (word >> (bits * (i % per_word))) & mask;
        double scale = (double)oracle_bf16_value(rd_u16(srow + 2 * (i / 64)));
        double bias = (double)oracle_bf16_value(rd_u16(brow + 2 * (i / 64)));
        /* q * scale is exact in double (at most 8 + 8 significant bits); the
         * sum is exact too unless bias lies far below half an f32 ulp of it,
         * so the cast is the one rounding of the exact value */
        out[i] = (float)((double)q * scale + bias);
    }
    return 0;
}

/* All n rows into out[n][k]; scales and biases are [n][k/64]. */
int oracle_dequant_affine(int bits, const uint8_t *w, const uint8_t *sc, const uint8_t *bi,
                          int64_t k, int64_t n, float *out)
{
    int64_t rb = oracle_affine_row_bytes(bits, k);
    if (rb < 0) return -1;
    for (int64_t j = 0; j < n; ++j)
        if (oracle_dequant_affine_row(bits, w + j * rb, sc + j * (k / 32), bi + j * (k / 32), k,
                                      out + j * k))
            return -1;
    return 0;
}

/* y[t][j] = sum_i x[t][i] * w[j][i], s[t][j] = sum_i |x w|, double sums. */
int oracle_matmul_affine(int bits, const uint8_t *w, const uint8_t *sc, const uint8_t *bi,
                         const float *x, int64_t k, int64_t n, int64_t n_tokens, double *y,
                         double *s, float *wrow_scratch)
{
    int64_t rb = oracle_affine_row_bytes(bits, k);
    if (rb < 0) return -1;
    for (int64_t j = 0; j < n; ++j) {
        if (oracle_dequant_affine_row(bits, w + j * rb, sc + j * (k / 32), bi + j * (k / 32), k,
                                      wrow_scratch))
            return -1;
        for (int64_t t = 0; t < n_tokens; ++t) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < k; ++i) {
                double v = (double)x[t * k + i] * (double)wrow_scratch[i];
                acc += v;
                mag += fabs(v);
            }
            y[t * n + j] = acc;
            s[t * n + j] = mag;
        }
    }
    return 0;
}

/* The same product for `count` chosen outputs (t_idx[c], j_idx[c]). */
int oracle_matmul_affine_sampled(int bits, const uint8_t *w, const uint8_t *sc,
                                 const uint8_t *bi, const float *x, int64_t k, int64_t n,
                                 int64_t n_tokens, int64_t count, const int64_t *t_idx,
                                 const int64_t *j_idx, double *y, double *s, float *wrow_scratch)
{
    int64_t rb = oracle_affine_row_bytes(bits, k);
    if (rb < 0) return -1;
    for (int64_t c = 0; c < count; ++c) {
        int64_t t = t_idx[c], j = j_idx[c];
        if (t < 0 || t >= n_tokens || j < 0 || j >= n) return -1;
        if (oracle_dequant_affine_row(bits, w + j * rb, sc + j * (k / 32), bi + j * (k / 32), k,
                                      wrow_scratch))
            return -1;
        double acc = 0.0, mag = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            double v = (double)x[t * k + i] * (double)wrow_scratch[i];
            acc += v;
            mag += fabs(v);
        }
        y[c] = acc;
        s[c] = mag;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Gated products: y = act(x Wg) * (x Wu). act 0: silu(g) = g / (1 + e^-g);
 * act 1: GELU, tanh form, 0.5 g (1 + tanh(z)) with z = sqrt(2/pi) (g +
 * 0.044715 g^3). Since 0.5 (1 + tanh z) = 1 / (1 + e^(-2z)) exactly, the
 * second form is evaluated: the first cancels to nothing in double once
 * z < -19, the second keeps its relative precision. */

double oracle_act(int act, double g)
{
    if (act == 0) return g / (1.0 + exp(-g));
    const double c = sqrt(2.0 / 3.14159265358979323846);
    const double z = c * (g + 0.044715 * g * g * g);
    return g / (1.0 + exp(-2.0 * z));
}

/* d act / d g, for the error bar of the gated product. */
double oracle_act_deriv(int act, double g)
{
    if (act == 0) {
        const double sg = 1.0 / (1.0 + exp(-g));
        return sg * (1.0 + g * (1.0 - sg));
    }
    /* d/dg [g s(2z)] = s(2z) + g s(2z) (1 - s(2z)) 2 z', s the logistic function */
    const double c = sqrt(2.0 / 3.14159265358979323846);
    const double z = c * (g + 0.044715 * g * g * g);
    const double sg = 1.0 / (1.0 + exp(-2.0 * z));
    return sg + g * sg * (1.0 - sg) * 2.0 * c * (1.0 + 3.0 * 0.044715 * g * g);
}

/* y[t][j] = act(gate) * up with gate = sum_i x w_g, up = sum_i x w_u (double
 * sums), and the error scale s[t][j] = |act'(gate)| |up| Sg + |act(gate)| Su
 * (Sg, Su the sums of |x w|): a product bar e * S on gate and up propagates to
 * at most e * s on y, to first order. */
int oracle_matmul_glu(int act, int fmt, const uint8_t *wg, const uint8_t *wu, const float *x,
                      int64_t k, int64_t n, int64_t n_tokens, double *y, double *s,
                      float *wrow_scratch)
{
    int64_t rb = oracle_row_bytes(fmt, k);
    if ((rb == 0 && k != 0) || (act != 0 && act != 1)) return -1;
    for (int64_t j = 0; j < n; ++j) {
        for (int64_t t = 0; t < n_tokens; ++t) {
            double gu[2], su[2];
            for (int m = 0; m < 2; ++m) {
                if (oracle_dequant_row(fmt, (m ? wu : wg) + j * rb, k, wrow_scratch)) return -1;
                double acc = 0.0, mag = 0.0;
                for (int64_t i = 0; i < k; ++i) {
                    double v = (double)x[t * k + i] * (double)wrow_scratch[i];
                    acc += v;
                    mag += fabs(v);
                }
                gu[m] = acc;
                su[m] = mag;
            }
            const double a = oracle_act(act, gu[0]);
            y[t * n + j] = a * gu[1];
            s[t * n + j] = fabs(oracle_act_deriv(act, gu[0])) * fabs(gu[1]) * su[0] + fabs(a) * su[1];
        }
    }
    return 0;
}
