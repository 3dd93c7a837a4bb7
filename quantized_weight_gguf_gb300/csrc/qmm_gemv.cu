// qmm_gemv.cu -- one-token fused dequantize + dot (GEMV), y[j] = sum_i w[j][i] x[i].
//
// Design (GB300, HBM-bound): each CTA owns a contiguous range of rows of W,
// i.e. a contiguous byte range of the packed weight stream. One producer lane
// streams it into a ring of shared-memory stages with 1-D bulk copies (TMA,
// 16-byte aligned windows, so unaligned block formats need no special care on
// the global side); 256 consumer threads decode from shared memory. Each
// consumer owns a fixed "unit" of k (32 or 64 weights) for the whole kernel,
// so its slice of x lives in registers and is read from global memory once.
// Per stage, every consumer writes one partial sum per (row, unit) to shared
// memory and one warp per row reduces them in a fixed order (deterministic).
//
// Decoding keeps the integer codes exact and out of the fp pipe as far as
// possible. Codes with no zero point (Q4_K, affine 4-bit) ride the float
// 0.5 + q/256 that a byte permute builds from q < 128 (q lands in mantissa
// bits 16..22), so the dot over a sub-block is
// sum q x = 256 * (sum (0.5 + q/256) x - 0.5 * sum x), where sum x is summed
// once per thread in exactly the order and pairing of the carrier's fmas:
// with every code 0 the carrier sum is then exactly half of it and the unit
// gives exactly 0. Codes with a zero point z (Q4_0, Q5_0, Q6_K, Q8_0) become
// q - z exactly (2^23 + q - (2^23 + z)), so a block whose codes all sit at
// the zero point gives exactly 0 as well.
//
// Kernel variants (template VAR): the plain GEMV; expert-indexed (grid.y runs
// one GEMV per (position, slot) on the selected expert slice); gated pairs
// (stages alternate gate and up rows, the flush writes act(gate) * up).
// Affine formats stage their scale and bias rows beside the codes.
#include "qmm_device.cuh"
#include "qmm_internal.h"

#include <algorithm>
#include <mutex>
#include <type_traits>

namespace qmm {

constexpr int kConsWarps = 8;
constexpr int kCons = kConsWarps * 32;
constexpr int kGemvThreads = kCons + 32;

struct GemvParams {
    const uint8_t *w;
    const float *x;
    float *y;
    int64_t k, row_bytes, w_total;
    int64_t j0;
    int64_t rows_base;
    int rows_rem;
    int accumulate;
    int x_ready;  // 1: x may be read before the preceding kernel completes; 2: nothing may (W included)
    int U;    // units per row
    int G;    // row groups per stage (one unit per thread), else 1
    int PU;   // partial slots per row
    int SEG;  // lanes that share a row and pre-reduce by shuffles (0: one partial per thread)
    int RPF;  // rows whose partials are buffered before a block-wide reduction (multiple of SR)
    int SR;   // rows per stage
    int SB;   // bytes per stage buffer (multiple of 128)
    int NS;   // stage buffers
    unsigned int *err;
};

// Expert-indexed calls: blockIdx.y = position * top_k + slot selects the
// expert slice ids[blockIdx.y] of W, x row `position` and y row blockIdx.y.
// A separate parameter type, so that the plain GEMV's kernel parameters (and
// its code) stay as they are.
struct GemvExpParams : GemvParams {
    const int32_t *ids;
    int64_t slice_bytes;
    int n_experts, top_k;
    int64_t n;  // row stride of y
};
// Affine formats: the bf16 scale and bias arrays ([n][k/64] each, aux_row_bytes
// per row, aux_total bytes each) are staged beside the codes of every stage:
// scales at byte aux_off of the stage buffer, biases aux_sb bytes further.
struct GemvAffFields {
    const uint8_t *sc, *bi;
    int64_t aux_row_bytes, aux_total;
    int aux_off, aux_sb;
};
struct GemvAffParams : GemvParams, GemvAffFields {};
// expert-indexed affine matrices: the scale and bias arrays are stacked like
// the codes ([n_experts][n][k/64] each)
struct GemvAffExpParams : GemvExpParams, GemvAffFields {};
// Gated pairs: w is the gate matrix, w2 the up matrix (same format and
// shape); y = act(x Wg) * (x Wu). A CTA's stages alternate between a block
// of rows of Wg and the same rows of Wu; each window of rows keeps two sets
// of partial sums, and its flush writes act(gate) * up.
struct GemvGluParams : GemvParams {
    const uint8_t *w2;
};
// everything the host fills in; each kernel instance takes only its own part
struct GemvHostParams : GemvExpParams, GemvAffFields {
    const uint8_t *w2;
    int glu;  // 0 none, 1 SwiGLU, 2 GeGLU
};

// Kernel variants: plain, expert-indexed, gated pair with SwiGLU or GeGLU.
enum GemvVar : int { kVarPlain = 0, kVarExperts = 1, kVarSwiglu = 2, kVarGeglu = 3 };

template <int FMT, int VAR>
using GemvParamsOf = typename std::conditional<
    is_affine(FMT),
    typename std::conditional<VAR == kVarExperts, GemvAffExpParams, GemvAffParams>::type,
    typename std::conditional<
        VAR == kVarExperts, GemvExpParams,
        typename std::conditional<(VAR >= kVarSwiglu), GemvGluParams, GemvParams>::type>::type>::type;

template <int FMT, int VAR>
__host__ GemvParamsOf<FMT, VAR> params_of(const GemvHostParams &h) {
    if constexpr (is_affine(FMT) && VAR == kVarExperts) {
        GemvAffExpParams a;
        static_cast<GemvExpParams &>(a) = static_cast<const GemvExpParams &>(h);
        static_cast<GemvAffFields &>(a) = static_cast<const GemvAffFields &>(h);
        return a;
    } else if constexpr (is_affine(FMT)) {
        GemvAffParams a;
        static_cast<GemvParams &>(a) = static_cast<const GemvParams &>(h);
        static_cast<GemvAffFields &>(a) = static_cast<const GemvAffFields &>(h);
        return a;
    } else if constexpr (VAR == kVarExperts) {
        return static_cast<const GemvExpParams &>(h);
    } else if constexpr (VAR >= kVarSwiglu) {
        GemvGluParams gp;
        static_cast<GemvParams &>(gp) = static_cast<const GemvParams &>(h);
        gp.w2 = h.w2;
        return gp;
    } else {
        return static_cast<const GemvParams &>(h);
    }
}



// Weights per unit: a 16-byte chunk for 16-bit formats (lane-contiguous in
// shared memory), a 32-weight block for Q4_0, Q8_0 and Q5_0, a 32-weight
// sub-block for Q4_K and a 32-weight quarter-half for Q6_K.
template <int FMT>
struct UnitK {
    static constexpr int value = (FMT == F_BF16 || FMT == F_F16) ? 8 : 32;
};

__device__ __forceinline__ int32_t bfe_s(uint32_t a, uint32_t pos) {
    int32_t d;
    asm("bfe.s32 %0, %1, %2, 8;" : "=r"(d) : "r"(a), "r"(pos));
    return d;
}

// x is staged in shared memory "unit-transposed": element e of unit u lives at
// e * (U + 1) + u, so the 32 lanes of a warp (consecutive units) read 32
// consecutive words. x_slot maps a k index to that slot.
template <int FMT>
__device__ __forceinline__ int x_slot(int k, int U) {
    int u, e;
    if (FMT == F_Q6_K) {
        // k = 256 b + 128 h + 32 r + 8 gq + i  ->  unit 8 b + 4 h + gq, element 8 r + i
        u = ((k >> 8) << 3) + (((k >> 7) & 1) << 2) + ((k >> 3) & 3);
        e = (((k >> 5) & 3) << 3) + (k & 7);
    } else {
        constexpr int UK = UnitK<FMT>::value;
        u = k / UK;
        e = k % UK;
    }
    return e * (U + 1) + u;
}

// Per-thread constants of one unit (x slice and what is derived from it).
template <int FMT>
struct UnitState {
    // the unit's x as pairs (elements 2i, 2i + 1) in 64-bit registers, the
    // operand form of the packed fmas (no register moves per use)
    uint64_t xp[UnitK<FMT>::value / 2];
    float c0;                  // sum of the unit's x (carrier and affine formats)
    uint32_t p0, p1, p2, p3;   // format-specific bit positions / byte selectors
    uint32_t lowgrp;
};

// sum of the unit's 32 x values in the order and pairing of a carrier dot:
// the packed fmas accumulate elements 4m, 4m+1, 4m+2, 4m+3 (m = 0..7) in four
// chains that are then added as (c0 + c1) + (c2 + c3). A carrier dot whose
// codes are all 0 (every carrier 0.5) then equals exactly half of this sum.
template <int N>
__device__ __forceinline__ float carrier_order_sum(const float (&xr)[N], int off = 0) {
    float c[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        c[r] = xr[off + r];
#pragma unroll
        for (int m = 1; m < 8; ++m) c[r] += xr[off + 4 * m + r];
    }
    return (c[0] + c[1]) + (c[2] + c[3]);
}

template <int FMT>
__device__ __forceinline__ void unit_init(UnitState<FMT> &st, const float *xs, int U, int u,
                                          bool valid) {
    constexpr int UK = UnitK<FMT>::value;
    // element e of unit u sits at xs[e * (U + 1) + u]
    float xr[UK];
#pragma unroll
    for (int e = 0; e < UK; ++e) xr[e] = valid ? xs[e * (U + 1) + u] : 0.0f;
#pragma unroll
    for (int i = 0; i < UK / 2; ++i) st.xp[i] = pack_f2(xr[2 * i], xr[2 * i + 1]);
    if constexpr (FMT == F_Q6_K) {
        const int gq = u & 3;
        // scale byte of quarter r sits at byte 2r + (gq >> 1) of scales[8h .. 8h+7]
        st.p0 = 8 * (0 + (gq >> 1)); st.p1 = 8 * (2 + (gq >> 1));
        st.p2 = st.p0; st.p3 = st.p1;
    } else if constexpr (FMT == F_AFF8) {
        float sx = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) sx += xr[i];
        st.c0 = sx;
    } else if constexpr (FMT == F_AFF4) {
        st.c0 = carrier_order_sum(xr);
    } else if constexpr (FMT == F_Q4_K) {
        st.c0 = carrier_order_sum(xr);
        // 6-bit scale and min of sub-block s gathered into bytes 0, 1 of a
        // word from the header words y (scales[0..3]), z (scales[4..7]) and
        // w (scales[8..11]):
        //   s < 4:  sc = y byte s & 63, m = z byte s & 63;
        //   s >= 4 (t = s - 4): sc = w byte t & 15 | (y byte t >> 6) << 4,
        //                       m = w byte t >> 4 | (z byte t >> 6) << 4.
        const int sb = u & 7;  // sub-block within the super-block
        st.lowgrp = sb < 4;
        const uint32_t t = st.lowgrp ? (uint32_t)sb : (uint32_t)sb - 4u;
        st.p0 = t | ((t + 4u) << 4);                  // byte selector (field A, top bits)
        st.p1 = st.lowgrp ? 0x3F3Fu : 0x0F0Fu;       // mask of field A
        st.p2 = st.lowgrp ? 0u : 0x3030u;            // mask of the top bits
        st.p3 = (sb & 1) ? 4u : 0u;                  // nibble of the quant bytes
    }
}

// 16-bit formats: the unit's 8 x values straight from global memory (two
// 16-byte loads when aligned; the units of a warp are consecutive).
template <int FMT>
__device__ __forceinline__ void unit_init_direct(UnitState<FMT> &st, const float *x, int u,
                                                 bool valid) {
    static_assert(UnitK<FMT>::value == 8, "16-bit formats only");
    const float *xu = x + 8 * u;
    float xr[8];
    if (!valid) {
#pragma unroll
        for (int e = 0; e < 8; ++e) xr[e] = 0.0f;
    } else if ((reinterpret_cast<uintptr_t>(xu) & 15u) == 0) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(xu));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(xu) + 1);
        xr[0] = a.x; xr[1] = a.y; xr[2] = a.z; xr[3] = a.w;
        xr[4] = b.x; xr[5] = b.y; xr[6] = b.z; xr[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) xr[e] = __ldg(xu + e);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) st.xp[i] = pack_f2(xr[2 * i], xr[2 * i + 1]);
}

// Partial dot of one unit of one row; `rowa` is the row's shared address.
template <int FMT>
__device__ __forceinline__ float unit_dot(uint32_t rowa, int u, const UnitState<FMT> &st) {
    if (FMT == F_BF16 || FMT == F_F16) {
        const uint4 v = lds128(rowa + 16u * u);
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
        float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 wf;
            if (FMT == F_BF16) {
                wf.x = __uint_as_float(wd[i] << 16);
                wf.y = __uint_as_float(wd[i] & 0xFFFF0000u);
            } else {
                wf = __half22float2(*reinterpret_cast<const __half2 *>(&wd[i]));
            }
            const uint64_t xv = st.xp[i];
            if (i & 1) a1 = ffma2(wf, xv, a1); else a0 = ffma2(wf, xv, a0);
        }
        return (a0.x + a0.y) + (a1.x + a1.y);
    } else if (FMT == F_Q4_0) {
        const uint32_t base = rowa + 18u * u;
        const float d = f16_bits_to_f32(lds16(base));
        uint32_t qw[4];
        lds_words_a2<4>(base + 2, qw);
        const float2 zp = make_float2(-8388616.0f, -8388616.0f);  // -(2^23 + 8)
        float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = qw[i] & 0x0F0F0F0Fu, hi = (qw[i] >> 4) & 0x0F0F0F0Fu;
            float2 f;
            f = fadd2(make_float2(byte_magic23<0>(lo), byte_magic23<1>(lo)), zp);
            a0 = ffma2(f, st.xp[2 * i], a0);
            f = fadd2(make_float2(byte_magic23<2>(lo), byte_magic23<3>(lo)), zp);
            a1 = ffma2(f, st.xp[2 * i + 1], a1);
            f = fadd2(make_float2(byte_magic23<0>(hi), byte_magic23<1>(hi)), zp);
            a0 = ffma2(f, st.xp[8 + 2 * i], a0);
            f = fadd2(make_float2(byte_magic23<2>(hi), byte_magic23<3>(hi)), zp);
            a1 = ffma2(f, st.xp[8 + 2 * i + 1], a1);
        }
        return d * ((a0.x + a0.y) + (a1.x + a1.y));
    } else if (FMT == F_Q4_K) {
        const int b = u >> 3, c = (u >> 1) & 3;
        const uint32_t sb = rowa + 144u * b;
        const uint4 hdr = lds128(sb);
        const uint4 q0 = lds128(sb + 16u + 32u * c);
        const uint4 q1 = lds128(sb + 32u + 32u * c);
        // [sc, m] in bytes 0 and 1 (see unit_init)
        const uint32_t fa = prmt(st.lowgrp ? hdr.y : hdr.w, st.lowgrp ? hdr.z : hdr.w >> 4, st.p0);
        const uint32_t fb = prmt(hdr.y, hdr.z, st.p0) >> 2;
        const uint32_t scm = (fa & st.p1) | (fb & st.p2);
        // v as the float 2^23 + v, then (2^23 + v) s - 2^23 s = v s exactly
        // (at most 17 significant bits): (256 d sc, dmin m) in one packed fma
        const float2 sd = make_float2(256.0f * f16_bits_to_f32(hdr.x & 0xFFFFu),
                                      f16_bits_to_f32(hdr.x >> 16));
        const float2 dsm = ffma2(make_float2(byte_magic23<0>(scm), byte_magic23<1>(scm)), sd,
                                 make_float2(-8388608.0f * sd.x, -8388608.0f * sd.y));
        const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t nib = (wd[i] >> st.p3) & 0x0F0F0F0Fu;
            a0 = ffma2(make_float2(byte_half_plus<0>(nib), byte_half_plus<1>(nib)),
                       st.xp[2 * i], a0);
            a1 = ffma2(make_float2(byte_half_plus<2>(nib), byte_half_plus<3>(nib)),
                       st.xp[2 * i + 1], a1);
        }
        const float a = (a0.x + a0.y) + (a1.x + a1.y);
        // d sc * sum q x - dmin m * sum x, with sum q x = 256 * (a - sum x / 2);
        // a - sum x / 2 is exactly 0 when every code is 0
        const float t = fmaf(-0.5f, st.c0, a);
        return fmaf(dsm.x, t, -dsm.y * st.c0);
    } else if (FMT == F_Q8_0) {
        // codes are signed bytes: flipping the top bit gives q + 128 unsigned,
        // 2^23 + (q + 128) - (2^23 + 128) = q exactly
        const uint32_t base = rowa + 34u * u;
        const float d = f16_bits_to_f32(lds16(base));
        uint32_t qw[8];
        lds_words_a2<8>(base + 2, qw);
        const float2 zp = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
        float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t v = qw[i] ^ 0x80808080u;
            float2 f = fadd2(make_float2(byte_magic23<0>(v), byte_magic23<1>(v)), zp);
            a0 = ffma2(f, st.xp[2 * i], a0);
            f = fadd2(make_float2(byte_magic23<2>(v), byte_magic23<3>(v)), zp);
            a1 = ffma2(f, st.xp[2 * i + 1], a1);
        }
        return d * ((a0.x + a0.y) + (a1.x + a1.y));
    } else if (FMT == F_Q5_0) {
        // 5-bit codes: nibble | fifth bit spread to bit 4 of each byte, then
        // q - 16 exactly as 2^23 + q - (2^23 + 16)
        const uint32_t base = rowa + 22u * u;
        const float d = f16_bits_to_f32(lds16(base));
        uint32_t qh[1], qw[4];
        lds_words_a2<1>(base + 2, qh);
        lds_words_a2<4>(base + 6, qw);
        const float2 zp = make_float2(-8388624.0f, -8388624.0f);  // -(2^23 + 16)
        float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bits j of a 4-bit field -> bit 4 of byte j
            const uint32_t hl = (((qh[0] >> (4 * i)) & 15u) * 0x02040810u) & 0x10101010u;
            const uint32_t hh = (((qh[0] >> (16 + 4 * i)) & 15u) * 0x02040810u) & 0x10101010u;
            const uint32_t lo = (qw[i] & 0x0F0F0F0Fu) | hl, hi = ((qw[i] >> 4) & 0x0F0F0F0Fu) | hh;
            float2 f;
            f = fadd2(make_float2(byte_magic23<0>(lo), byte_magic23<1>(lo)), zp);
            a0 = ffma2(f, st.xp[2 * i], a0);
            f = fadd2(make_float2(byte_magic23<2>(lo), byte_magic23<3>(lo)), zp);
            a1 = ffma2(f, st.xp[2 * i + 1], a1);
            f = fadd2(make_float2(byte_magic23<0>(hi), byte_magic23<1>(hi)), zp);
            a0 = ffma2(f, st.xp[8 + 2 * i], a0);
            f = fadd2(make_float2(byte_magic23<2>(hi), byte_magic23<3>(hi)), zp);
            a1 = ffma2(f, st.xp[8 + 2 * i + 1], a1);
        }
        return d * ((a0.x + a0.y) + (a1.x + a1.y));
    } else {  // F_Q6_K
        const int b = u >> 3, h = (u >> 2) & 1, gq = u & 3;
        const uint32_t sb = rowa + 210u * b;
        uint32_t A[2], B[2], H[2], S[2];
        lds_words_a2<2>(sb + 64u * h + 8u * gq, A);
        lds_words_a2<2>(sb + 64u * h + 32u + 8u * gq, B);
        lds_words_a2<2>(sb + 128u + 32u * h + 8u * gq, H);
        lds_words_a2<2>(sb + 192u + 8u * h, S);
        const float d = f16_bits_to_f32(lds16(sb + 208u));
        // codes q - 32 exactly as 2^23 + q - (2^23 + 32)
        const float2 zp = make_float2(-8388640.0f, -8388640.0f);
        float2 acc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
            const uint32_t q[4] = {
                (A[wi] & 0x0F0F0F0Fu) | ((H[wi] << 4) & 0x30303030u),
                (B[wi] & 0x0F0F0F0Fu) | ((H[wi] << 2) & 0x30303030u),
                ((A[wi] >> 4) & 0x0F0F0F0Fu) | (H[wi] & 0x30303030u),
                ((B[wi] >> 4) & 0x0F0F0F0Fu) | ((H[wi] >> 2) & 0x30303030u)};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 f0 = fadd2(make_float2(byte_magic23<0>(q[r]), byte_magic23<1>(q[r])), zp);
                const float2 f1 = fadd2(make_float2(byte_magic23<2>(q[r]), byte_magic23<3>(q[r])), zp);
                acc[r] = ffma2(f0, st.xp[4 * r + 2 * wi], acc[r]);
                acc[r] = ffma2(f1, st.xp[4 * r + 2 * wi + 1], acc[r]);
            }
        }
        const uint32_t pr[4] = {st.p0, st.p1, st.p2, st.p3};
        float sum = 0.0f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float a = acc[r].x + acc[r].y;
            const float sc = (float)bfe_s(S[r >> 1], pr[r]);
            sum = fmaf(sc, a, sum);
        }
        return d * sum;
    }
}

// Partial dot of one 32-weight unit (half a group) of an affine row: codes at
// `rowa`, the row's scales at `auxa`, its biases aux_sb bytes further.
//   sum_i (q_i s + b) x_i = s * sum q x + b * sum x
template <int FMT>
__device__ __forceinline__ float unit_dot_aff(uint32_t rowa, uint32_t auxa, uint32_t aux_sb, int u,
                                              const UnitState<FMT> &st) {
    const uint32_t ga = auxa + 2u * (uint32_t)(u >> 1);
    const float sc = __uint_as_float(lds16(ga) << 16);
    const float bi = __uint_as_float(lds16(ga + aux_sb) << 16);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
    if (FMT == F_AFF4) {
        // word i holds elements 8i .. 8i+7, lowest nibble first: byte j of the
        // low-nibble mask is element 8i + 2j, of the high-nibble mask 8i + 2j + 1;
        // codes ride the exact carrier 0.5 + q/256 (element 4m + r lands in
        // chain r, as in carrier_order_sum) and
        // sum q x = 256 * (sum (0.5 + q/256) x - sum x / 2)
        const uint4 v = lds128(rowa + 16u * u);
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = wd[i] & 0x0F0F0F0Fu, hi = (wd[i] >> 4) & 0x0F0F0F0Fu;
            a0 = ffma2(make_float2(byte_half_plus<0>(lo), byte_half_plus<0>(hi)),
                       st.xp[4 * i], a0);
            a1 = ffma2(make_float2(byte_half_plus<1>(lo), byte_half_plus<1>(hi)),
                       st.xp[4 * i + 1], a1);
            a0 = ffma2(make_float2(byte_half_plus<2>(lo), byte_half_plus<2>(hi)),
                       st.xp[4 * i + 2], a0);
            a1 = ffma2(make_float2(byte_half_plus<3>(lo), byte_half_plus<3>(hi)),
                       st.xp[4 * i + 3], a1);
        }
        const float a = (a0.x + a0.y) + (a1.x + a1.y);
        // exactly 0 for a group of zero codes with a zero bias
        const float t = fmaf(-0.5f, st.c0, a);
        return fmaf(256.0f * sc, t, bi * st.c0);
    } else {
        // 8-bit codes: element 4i + j is byte j of word i; 2^23 + q - 2^23 = q exactly
        const uint4 v0 = lds128(rowa + 32u * u), v1 = lds128(rowa + 32u * u + 16u);
        const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        const float2 zp = make_float2(-8388608.0f, -8388608.0f);  // -2^23
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float2 f = fadd2(make_float2(byte_magic23<0>(wd[i]), byte_magic23<1>(wd[i])), zp);
            a0 = ffma2(f, st.xp[2 * i], a0);
            f = fadd2(make_float2(byte_magic23<2>(wd[i]), byte_magic23<3>(wd[i])), zp);
            a1 = ffma2(f, st.xp[2 * i + 1], a1);
        }
        const float a = (a0.x + a0.y) + (a1.x + a1.y);
        return fmaf(sc, a, bi * st.c0);
    }
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// Where a CTA's weight slice, x row and y row start: the call's own for a
// plain GEMV (read from the parameters where used), the selected expert's
// slice and the pair's rows for an expert-indexed one.
template <bool EXP>
struct SliceSel {
    __device__ __forceinline__ const float *x(const GemvParams &p) const { return p.x; }
    __device__ __forceinline__ float *y(const GemvParams &p) const { return p.y; }
    __device__ __forceinline__ int64_t w_off() const { return 0; }
    __device__ __forceinline__ int64_t a_off() const { return 0; }
};
template <>
struct SliceSel<true> {
    const float *xg;
    float *yg;
    int64_t off;
    int64_t aoff = 0;  // affine formats: the slice's offset in the scale and bias arrays
    __device__ __forceinline__ const float *x(const GemvParams &) const { return xg; }
    __device__ __forceinline__ float *y(const GemvParams &) const { return yg; }
    __device__ __forceinline__ int64_t w_off() const { return off; }
    __device__ __forceinline__ int64_t a_off() const { return aoff; }
};

template <int FMT, int UPT, int VAR>
__global__ void __maxnreg__(96) gemv_kernel(const GemvParamsOf<FMT, VAR> p) {
    constexpr bool kChunked = (FMT == F_BF16 || FMT == F_F16);  // warp-reduced 16-byte chunks
    constexpr bool EXP = VAR == kVarExperts, GLU = VAR >= kVarSwiglu;
    extern __shared__ __align__(128) uint8_t smem[];
    const int NS = p.NS, SR = p.SR, SB = p.SB, PU = p.PU;
    const uint32_t bar0 = smem_addr(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 16 * NS);
    float *part = reinterpret_cast<float *>(smem + 16 * NS + 16);
    const int part_bytes = 4 * p.RPF * PU;
    // gated pairs: a second set of partials (the up rows) after the first
    float *part_up = part + p.RPF * PU;
    const int xs_off = (16 * NS + 16 + (GLU ? 2 : 1) * part_bytes + 127) & ~127;
    float *xs = reinterpret_cast<float *>(smem + xs_off);
    // 16-bit formats read their x slices straight from global memory (each
    // thread's units are contiguous 32-byte runs): no staging area
    const int xs_bytes = kChunked ? 0 : 4 * (int)(p.k + UnitK<FMT>::value);
    const uint32_t stage_off = (uint32_t)((xs_off + xs_bytes + 127) & ~127);
    uint8_t *stages = smem + stage_off;
    const uint32_t stage0 = bar0 + stage_off;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (NS + s); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    // byte offset of this call's weight slice, and its x and y rows
    SliceSel<EXP> sel;
    if constexpr (EXP) {
        // the ids count as input: produced by the preceding kernel unless the
        // caller vouched otherwise
        if (p.x_ready != 1) pdl_wait_prev();
        const int pair = blockIdx.y;
        const int e = p.x_ready == 1 ? __ldg(p.ids + pair) : p.ids[pair];
        if (e < 0 || e >= p.n_experts) {  // nothing read or written for a bad id
            if (threadIdx.x == 0) record_error(p.err, DERR_BAD_ID);
            return;
        }
        sel.off = (int64_t)e * p.slice_bytes;
        sel.xg = p.x + (int64_t)(pair / p.top_k) * p.k;
        sel.yg = p.y + (int64_t)pair * p.n;
        if constexpr (is_affine(FMT)) sel.aoff = (int64_t)e * p.n * p.aux_row_bytes;
    }
    const int64_t r0 = p.j0 + (int64_t)cta * p.rows_base + (cta < p.rows_rem ? cta : p.rows_rem);
    const int64_t nrows = p.rows_base + (cta < p.rows_rem ? 1 : 0);
    // gated pairs: stage 2i streams row block i of the gate matrix, stage
    // 2i + 1 the same rows of the up matrix
    const int nst_half = (int)((nrows + SR - 1) / SR);
    const int nst = GLU ? 2 * nst_half : nst_half;
    const int64_t R = p.row_bytes;
    auto stage_rows = [&](int s, int64_t &ra, int64_t &rb) {
        const int sl = GLU ? s >> 1 : s;
        ra = r0 + (int64_t)sl * SR;
        rb = min(ra + SR, r0 + nrows);
    };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kConsWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // The next kernel in the stream may begin launching once every CTA of this
    // one is running; it waits for this grid's completion before using its y.
    pdl_launch_dependents();

    if (warp == kConsWarps) {
        // ---------------- producer: one lane streams the weight bytes ----------------
        if (lane != 0) return;
        if (p.x_ready == 2) pdl_wait_prev();  // stream order: W may come from the preceding kernel
        const int64_t lim = p.w_total & ~(int64_t)15;
        int issued = 0;
        for (int s = 0; s < nst; ++s) {
            const int slot = s % NS;
            if (s >= NS && !wait_or_abort(empty(slot), ((s / NS) + 1) & 1, abort_flag)) {
                record_error(p.err, DERR_GEMV_EMPTY);
                *abort_flag = 1;
                break;
            }
            int64_t ra, rb;
            stage_rows(s, ra, rb);
            const uint8_t *wsrc = p.w;
            if constexpr (GLU) {
                if (s & 1) wsrc = p.w2;
            }
            const int64_t A = sel.w_off() + ra * R, B = sel.w_off() + rb * R;
            const int64_t a16 = A & ~(int64_t)15, b16 = (B + 15) & ~(int64_t)15;
            const int64_t tend = min(b16, lim);
            if (B > lim) {  // bytes after the last whole 16-byte chunk of W
                for (int64_t q = max(a16, lim); q < B; ++q)
                    stages[(int64_t)slot * SB + (q - a16)] = wsrc[q];
            }
            const uint32_t tx = tend > a16 ? (uint32_t)(tend - a16) : 0u;
            if constexpr (is_affine(FMT)) {
                // the stage's rows of the scale and bias arrays, the same way
                const int64_t AR = p.aux_row_bytes, alim = p.aux_total & ~(int64_t)15;
                const int64_t SA = sel.a_off() + ra * AR, SE = sel.a_off() + rb * AR;
                const int64_t s16 = SA & ~(int64_t)15;
                const int64_t send = min((SE + 15) & ~(int64_t)15, alim);
                const int64_t sdst = (int64_t)slot * SB + p.aux_off;
                if (SE > alim) {
                    for (int64_t q = max(s16, alim); q < SE; ++q) {
                        stages[sdst + (q - s16)] = p.sc[q];
                        stages[sdst + p.aux_sb + (q - s16)] = p.bi[q];
                    }
                }
                const uint32_t atx = send > s16 ? (uint32_t)(send - s16) : 0u;
                mbar_arrive_expect_tx(full(slot), tx + 2u * atx);
                if (tx) bulk_g2s(stage0 + (uint32_t)slot * SB, wsrc + a16, tx, full(slot));
                if (atx) {
                    bulk_g2s(stage0 + (uint32_t)sdst, p.sc + s16, atx, full(slot));
                    bulk_g2s(stage0 + (uint32_t)(sdst + p.aux_sb), p.bi + s16, atx, full(slot));
                }
            } else {
                mbar_arrive_expect_tx(full(slot), tx);
                if (tx) bulk_g2s(stage0 + (uint32_t)slot * SB, wsrc + a16, tx, full(slot));
            }
            ++issued;
        }
        // no copy may land after this CTA exits
        for (int s = max(0, issued - NS); s < issued; ++s)
            if (!mbar_wait(full(s % NS), (s / NS) & 1)) record_error(p.err, DERR_TEARDOWN);
        return;
    }

    // ---------------- consumers ----------------
    // x -> shared memory (unit-transposed) with coalesced global loads. Unless
    // the caller vouched that the preceding kernel does not write x, wait for
    // that kernel first (it may be producing x); y is never touched before
    // the wait.
    if (p.x_ready != 1) pdl_wait_prev();
    if (!kChunked) {
        const int k = (int)p.k;
        const int U = p.U;
        if ((reinterpret_cast<uintptr_t>(sel.x(p)) & 15u) == 0 && (k & 3) == 0) {
            const float4 *x4 = reinterpret_cast<const float4 *>(sel.x(p));
            for (int i = tid; i < k / 4; i += kCons) {
                const float4 v = __ldg(x4 + i);
                xs[x_slot<FMT>(4 * i, U)] = v.x;
                xs[x_slot<FMT>(4 * i + 1, U)] = v.y;
                xs[x_slot<FMT>(4 * i + 2, U)] = v.z;
                xs[x_slot<FMT>(4 * i + 3, U)] = v.w;
            }
        } else {
            for (int i = tid; i < k; i += kCons) xs[x_slot<FMT>(i, U)] = __ldg(sel.x(p) + i);
        }
        named_barrier(1, kCons);
    }
    const int t = tid;
    int g, u0;
    bool active;
    if (UPT == 1 && !kChunked) {
        g = t / p.U;
        u0 = t - g * p.U;
        active = g < p.G;
    } else {
        g = 0;
        u0 = t;
        active = true;
    }
    UnitState<FMT> st[UPT];
#pragma unroll
    for (int q = 0; q < UPT; ++q) {
        const int u = u0 + q * kCons;
        if constexpr (kChunked)
            unit_init_direct<FMT>(st[q], sel.x(p), u, u < p.U);
        else
            unit_init<FMT>(st[q], xs, p.U, active && u < p.U ? u : 0, active && u < p.U);
    }
    const int G = p.G;
    const int SEG = p.SEG;
    // slot of this thread's partial within a row: one per thread, or one per
    // SEG-lane segment (written by the segment's first lane)
    const int pslot = SEG == 0 ? u0 : (SEG == 32 ? (kChunked || UPT > 1 ? warp : (u0 >> 5)) : 0);
    const bool writer = SEG == 0 || (lane & (SEG - 1)) == 0;
    bool failed = false;
    int64_t fbase = r0;  // first row of the buffered window
    for (int s = 0; s < nst; ++s) {
        const int slot = s % NS;
        if (!failed && !wait_or_abort(full(slot), (s / NS) & 1, abort_flag)) {
            failed = true;
            *abort_flag = 1;
            record_error(p.err, DERR_GEMV_FULL);
        }
        int64_t ra, rb;
        stage_rows(s, ra, rb);
        const int rows_in = (int)(rb - ra);
        const int64_t a16 = (sel.w_off() + ra * R) & ~(int64_t)15;
        const uint32_t sbase = stage0 + (uint32_t)slot * SB;
        float *pb = ((GLU && (s & 1)) ? part_up : part) + (ra - fbase) * PU;
        if (!failed && active) {
            // this thread's rows g, g + G, ... of the stage: shared addresses of
            // the row (and of its affine scales) and its partial slot advance
            // by fixed 32-bit steps
            const uint32_t Rb = (uint32_t)R;
            uint32_t rowa = sbase + (uint32_t)(sel.w_off() + ra * R - a16) + (uint32_t)g * Rb;
            const uint32_t rstep = (uint32_t)G * Rb;
            uint32_t auxa = 0, astep = 0;
            if constexpr (is_affine(FMT)) {
                const int64_t AR = p.aux_row_bytes;
                const int64_t a0 = sel.a_off() + ra * AR;
                auxa = sbase + (uint32_t)p.aux_off + (uint32_t)(a0 - (a0 & ~(int64_t)15)) +
                       (uint32_t)g * (uint32_t)AR;
                astep = (uint32_t)G * (uint32_t)AR;
            }
            float *pp = pb + g * PU + pslot;
            const int pstep = G * PU;
            auto row_dot = [&](uint32_t ra_, uint32_t aa_) {
                float acc = 0.0f;
#pragma unroll
                for (int q = 0; q < UPT; ++q) {
                    const int u = u0 + q * kCons;
                    if constexpr (is_affine(FMT)) {
                        if (UPT == 1 || u < p.U)
                            acc += unit_dot_aff<FMT>(ra_, aa_, (uint32_t)p.aux_sb, u, st[q]);
                    } else {
                        if ((UPT == 1 && !kChunked) || u < p.U) acc += unit_dot<FMT>(ra_, u, st[q]);
                    }
                }
                return acc;
            };
            if (SEG == 0) {
                // one partial per thread and row: no cross-lane traffic, each
                // thread runs its own trip count
                for (int rr = g; rr < rows_in; rr += G) {
                    *pp = row_dot(rowa, auxa);
                    rowa += rstep;
                    auxa += astep;
                    pp += pstep;
                }
            } else {
                // same trip count for every lane of a warp (segments of one warp
                // may belong to different row groups), so the shuffles stay
                // convergent
                for (int base = 0; base < rows_in; base += G) {
                    const bool has = base + g < rows_in;
                    float acc = has ? row_dot(rowa, auxa) : 0.0f;
                    for (int o = SEG >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
                    if (writer && has) *pp = acc;
                    rowa += rstep;
                    auxa += astep;
                    pp += pstep;
                }
            }
        }
        // the stage is refilled by a bulk copy (the async proxy) once every
        // consumer warp has arrived: order this thread's reads of it first
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(slot));
        __syncwarp();
        // block-wide reduction once the window is full, and at the end
        if ((!GLU || (s & 1)) && (rb - fbase >= p.RPF || s == nst - 1)) {
            if (p.x_ready == 1) pdl_wait_prev();  // y may still be in use by the preceding kernel
            named_barrier(1, kCons);
            if (!failed) {
                const int wrows = (int)(rb - fbase);
                for (int rr = warp; rr < wrows; rr += kConsWarps) {
                    float v = 0.0f, vu = 0.0f;
                    for (int i = lane; i < PU; i += 32) {
                        v += part[rr * PU + i];
                        if (GLU) vu += part_up[rr * PU + i];
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                        if (GLU) vu += __shfl_xor_sync(0xFFFFFFFFu, vu, o);
                    }
                    if (lane == 0) {
                        if (GLU) v = glu_act<VAR - kVarSwiglu + 1>(v) * vu;
                        float *yp = sel.y(p) + fbase + rr;
                        *yp = p.accumulate ? *yp + v : v;
                    }
                }
            }
            named_barrier(1, kCons);
            fbase = rb;
        }
    }
}

// ------------------------------------------------------------------ host ----

static int unit_k(int fmt) { return (fmt == F_BF16 || fmt == F_F16) ? 8 : 32; }
static int max_upt(int fmt) { return (fmt == F_BF16 || fmt == F_F16) ? 8 : 2; }

bool gemv_supports(int fmt, int64_t k) {
    if (fmt < F_BF16 || (fmt > kLastFmt && !is_affine(fmt)) || k <= 0) return false;
    if (is_affine(fmt) && k % 64) return false;
    const int uk = unit_k(fmt);
    if (k % uk) return false;
    const int64_t U = k / uk;
    return U <= (int64_t)kCons * max_upt(fmt);
}

template <int FMT, int UPT, int VAR>
static cudaError_t launch_e(const GemvHostParams &h, dim3 grid, size_t smem, cudaStream_t s,
                            bool overlap) {
    const GemvParamsOf<FMT, VAR> p = params_of<FMT, VAR>(h);
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gemv_kernel<FMT, UPT, VAR>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // Every launch is a programmatic dependent of the preceding kernel, so its
    // CTAs are resident by the time that kernel ends. Without `overlap` the
    // kernel waits for it before reading W (x_ready == 2): stream order holds,
    // only the launch latency is hidden (BF16 k=n=4096 back to back: 11.6 us
    // per call instead of 12.3).
    (void)overlap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, UPT, VAR>, p);
}

// the expert-indexed kernels are separate instances: the plain GEMV carries
// no id lookup or slice offset
template <int FMT, int UPT>
static cudaError_t launch_t(const GemvHostParams &p, dim3 grid, size_t smem, cudaStream_t s,
                            bool overlap) {
    if constexpr (is_affine(FMT)) {
        if (p.glu) return cudaErrorNotSupported;  // no gated affine pairs
        return p.ids ? launch_e<FMT, UPT, kVarExperts>(p, grid, smem, s, overlap)
                     : launch_e<FMT, UPT, kVarPlain>(p, grid, smem, s, overlap);
    } else {
        if (p.ids) return launch_e<FMT, UPT, kVarExperts>(p, grid, smem, s, overlap);
        if (p.glu == 1) return launch_e<FMT, UPT, kVarSwiglu>(p, grid, smem, s, overlap);
        if (p.glu == 2) return launch_e<FMT, UPT, kVarGeglu>(p, grid, smem, s, overlap);
        return launch_e<FMT, UPT, kVarPlain>(p, grid, smem, s, overlap);
    }
}

template <int FMT>
static cudaError_t launch_chunked(const GemvHostParams &p, int upt, dim3 grid, size_t smem,
                                  cudaStream_t s, bool ov) {
    switch (upt) {
    case 1: return launch_t<FMT, 1>(p, grid, smem, s, ov);
    case 2: return launch_t<FMT, 2>(p, grid, smem, s, ov);
    case 4: return launch_t<FMT, 4>(p, grid, smem, s, ov);
    default: return launch_t<FMT, 8>(p, grid, smem, s, ov);
    }
}

cudaError_t launch_gemv(const GemvLaunch &g, const DeviceInfo &dev, cudaStream_t s) {
    if (!gemv_supports(g.fmt, g.k)) return cudaErrorNotSupported;
    const int64_t M = g.j1 - g.j0;
    if (M <= 0) return cudaSuccess;
    const bool chunked = g.fmt == F_BF16 || g.fmt == F_F16;
    const int uk = unit_k(g.fmt);
    const int U = (int)(g.k / uk);
    int upt = (U + kCons - 1) / kCons;
    if (chunked) {
        int p2 = 1;
        while (p2 < upt) p2 <<= 1;
        upt = p2;
    }
    const int G = (!chunked && upt == 1) ? kCons / U : 1;
    // per-row pre-reduction: whole warps of one row (16-bit chunks, several units
    // per thread, or U a multiple of 32), power-of-two segments (U < 32), else none
    int SEG, PU;
    // (quantized formats are ALU-bound: one shared-memory partial per thread is
    // cheaper than shuffles; 16-bit formats have 8-weight units and headroom)
    if (chunked || upt > 1) {
        SEG = 32; PU = kConsWarps;
    } else if (U < 32 && (32 % U) == 0) {
        SEG = U; PU = 1;
    } else {
        SEG = 0; PU = U;
    }
    const int64_t R = g.row_bytes;
    // expert-indexed calls run `pairs` independent GEMVs side by side (grid.y).
    // Two CTAs per SM; one for 16-bit formats launched to overlap the
    // preceding kernel: their CTAs are sized so that three fit on an SM, so
    // the whole next grid is resident, streaming, while this one finishes
    // (BF16 k=n=4096 back to back: 5.37 us per call against 6.19 with two
    // CTAs per SM; the ALU-bound quantized formats measured slower with fewer
    // CTAs: Q4_K 11.8 us against 10.7).
    const int pairs = g.ids ? g.pairs : 1;
    const int ctas_per_sm = (chunked && g.overlap_prev) ? 1 : 2;
    const int ctas_target = std::max(1, ctas_per_sm * dev.sm_count / pairs);
    const int64_t per_cta = (M + ctas_target - 1) / ctas_target;
    const size_t xs_bytes = chunked ? 0 : (size_t)4 * (g.k + uk);
    // affine formats: scale and bias rows of the stage beside its codes
    const bool aff = is_affine(g.fmt);
    const int64_t AR = aff ? (g.k / 64) * 2 : 0;
    auto code_bytes = [&](int64_t sr) { return ((sr * R + 32) + 127) & ~(int64_t)127; };
    auto aux_bytes = [&](int64_t sr) { return aff ? ((sr * AR + 32) + 127) & ~(int64_t)127 : 0; };
    auto stage_bytes = [&](int64_t sr) { return code_bytes(sr) + 2 * aux_bytes(sr); };
    // gated pairs keep a second set of partials
    auto smem_for = [&](int ns, int64_t sr, int64_t rpf) {
        const size_t part_bytes = (size_t)4 * rpf * PU * (g.glu ? 2 : 1);
        const size_t sb = (size_t)stage_bytes(sr);
        return (size_t)((((16 * ns + 16 + part_bytes + 127) & ~(size_t)127) + xs_bytes + 127) &
                        ~(size_t)127) +
               (size_t)ns * sb;
    };
    // For 16-bit formats each CTA is kept small enough that three fit on an
    // SM (3 x (smem + 1 KB reserved per block) within 228 KB): under
    // programmatic dependent launch the next GEMVs' CTAs then start streaming
    // on an SM while this kernel's still run, which hides the kernel
    // boundary. Quantized formats need their x slices staged and more ring,
    // so they keep two CTAs' worth of room.
    const size_t two_cta_limit = chunked ? 228 * 1024 / 3 - 1024 : 228 * 1024 / 2 - 1024;
    int64_t SR, RPF;
    int NS;
    const int64_t half = G * (((per_cta + 1) / 2 + G - 1) / G);
    const int ns_whole = g.glu ? 4 : 2;  // gated pairs: both matrices' rows
    if (smem_for(ns_whole, half, 2 * half) <= two_cta_limit) {
        // the CTA's whole share fits in two stages (per matrix): all of it is
        // requested at once, one memory round trip per CTA
        SR = half;
        NS = ns_whole;
        RPF = 2 * half;
    } else {
        // rows per stage: ~32 KB of weights, a multiple of the row groups, and
        // small enough that every SM gets work on small problems
        const int64_t rb = std::max<int64_t>(1, 32768 / (G * R));
        SR = G * rb;
        if (per_cta < SR) SR = std::max<int64_t>(G, ((per_cta + G - 1) / G) * G);
        // partial-sum window: ~24 KB, whole stages, no more than a CTA's rows
        RPF = std::max<int64_t>(SR, (6144 / PU) / SR * SR);
        RPF = std::min<int64_t>(RPF, std::max<int64_t>(SR, (per_cta + SR - 1) / SR * SR));
        // gated pairs: two sets of partials; the window is as many stages as
        // fit beside a two-stage ring with two CTAs per SM (fewer flushes)
        if (g.glu) {
            const int64_t cap = std::max<int64_t>(SR, (per_cta + SR - 1) / SR * SR);
            RPF = SR;
            while (RPF + SR <= cap && smem_for(2, SR, RPF + SR) <= two_cta_limit) RPF += SR;
        }
        NS = 8;
        while (NS > 2 && smem_for(NS, SR, RPF) > two_cta_limit) --NS;
        if (smem_for(NS, SR, RPF) > two_cta_limit) {  // one CTA per SM, up to 8 stages
            NS = 8;
            while (NS > 2 && smem_for(NS, SR, RPF) > 200 * 1024) --NS;
        }
    }
    const int SB = (int)stage_bytes(SR);
    const int64_t nstage_total = (M + SR - 1) / SR;
    const int gx = (int)std::max<int64_t>(1, std::min<int64_t>(nstage_total, ctas_target));
    const dim3 grid((unsigned)gx, (unsigned)pairs);
    const size_t smem = smem_for(NS, SR, RPF);
    if (smem > 200 * 1024) return cudaErrorNotSupported;

    GemvHostParams p;
    p.w = g.w; p.x = g.x; p.y = g.y;
    p.sc = g.sc;
    p.bi = g.bi;
    p.aux_row_bytes = AR;
    p.aux_total = AR * g.n * (g.ids ? g.n_experts : 1);
    p.aux_off = (int)code_bytes(SR);
    p.aux_sb = (int)aux_bytes(SR);
    p.w2 = g.w2;
    p.glu = g.glu;
    p.k = g.k; p.row_bytes = R;
    p.w_total = R * g.n * (g.ids ? g.n_experts : 1);
    p.ids = g.ids;
    p.slice_bytes = R * g.n;
    p.n_experts = g.n_experts;
    p.top_k = g.top_k;
    p.n = g.n;
    p.j0 = g.j0;
    p.rows_base = M / gx;
    p.rows_rem = (int)(M % gx);
    p.accumulate = g.accumulate;
    p.x_ready = g.overlap_prev ? (g.x_ready ? 1 : 0) : 2;
    p.U = U; p.G = G; p.PU = PU; p.SEG = SEG; p.RPF = (int)RPF; p.SR = (int)SR; p.SB = SB; p.NS = NS;
    p.err = dev.err;
    const bool ov = g.overlap_prev;
    switch (g.fmt) {
    case F_BF16: return launch_chunked<F_BF16>(p, upt, grid, smem, s, ov);
    case F_F16: return launch_chunked<F_F16>(p, upt, grid, smem, s, ov);
    case F_Q4_0: return upt == 1 ? launch_t<F_Q4_0, 1>(p, grid, smem, s, ov) : launch_t<F_Q4_0, 2>(p, grid, smem, s, ov);
    case F_Q4_K: return upt == 1 ? launch_t<F_Q4_K, 1>(p, grid, smem, s, ov) : launch_t<F_Q4_K, 2>(p, grid, smem, s, ov);
    case F_Q6_K: return upt == 1 ? launch_t<F_Q6_K, 1>(p, grid, smem, s, ov) : launch_t<F_Q6_K, 2>(p, grid, smem, s, ov);
    case F_Q8_0: return upt == 1 ? launch_t<F_Q8_0, 1>(p, grid, smem, s, ov) : launch_t<F_Q8_0, 2>(p, grid, smem, s, ov);
    case F_Q5_0: return upt == 1 ? launch_t<F_Q5_0, 1>(p, grid, smem, s, ov) : launch_t<F_Q5_0, 2>(p, grid, smem, s, ov);
    case F_AFF4: return upt == 1 ? launch_t<F_AFF4, 1>(p, grid, smem, s, ov) : launch_t<F_AFF4, 2>(p, grid, smem, s, ov);
    case F_AFF8: return upt == 1 ? launch_t<F_AFF8, 1>(p, grid, smem, s, ov) : launch_t<F_AFF8, 2>(p, grid, smem, s, ov);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
