// qmm_back_input.cu -- backward of y = x @ W with respect to the input, one
// vector: dx[i] (+)= sum_{j in [j0, j1)} dy[j] * w[j][i] (the transposed
// product; the row range tiles the sum axis).
//
// Same weight stream as the GEMV: each CTA owns a contiguous range of rows,
// i.e. a contiguous byte range of W, which one producer lane streams through a
// ring of shared-memory stages with 1-D bulk copies. Each of the 256 consumer
// threads owns a fixed unit of k (8 weights for 16-bit formats, one 32-weight
// block / sub-block / quarter-half otherwise) and keeps that unit's dx partial
// sums in registers; for every row it decodes the unit and adds dy[j] times
// the weights. Codes stay exact. Formats with a zero point z (Q4_0, Q5_0,
// Q6_K, Q8_0) turn each code into q - z exactly (2^23 + q - (2^23 + z)) and
// accumulate sum_j a_j (q - z) with a_j = dy[j] * scale, so rows whose codes
// sit at the zero point add exactly 0. Q4_K codes ride the float 0.5 + q/256
// that a byte permute builds, and the per-unit sums of a_j (accumulated in
// the same order) remove the carrier and the min:
// dx = 256 acc - (128 sum a + sum dy dmin m), exactly 0 for zero codes and
// zero mins.
// At the end the row groups of a CTA are summed in shared memory and the CTA
// writes its partial dx; a second small kernel adds the partials of all CTAs in
// a fixed order (deterministic) into dx.
#include "qmm_device.cuh"
#include "qmm_internal.h"

#include <algorithm>
#include <mutex>

namespace qmm {

namespace {

constexpr int kBwWarps = 8;
constexpr int kBwCons = kBwWarps * 32;
constexpr int kBwThreads = kBwCons + 32;

struct BackParams {
    const uint8_t *w;
    const float *dy;
    float *part;     // [grid][k] partial dx of each CTA
    int64_t k, row_bytes, w_total;
    int64_t j0;
    int64_t rows_base;
    int rows_rem;
    int U;    // units per row
    int G;    // row groups (each thread takes rows g, g + G, ...)
    int SR;   // rows per stage
    int SB;   // bytes per stage buffer (multiple of 128)
    int NS;   // stage buffers
    int dy_cap;  // rows of dy staged (>= rows per CTA)
    int x_ready; // dy may be read before the preceding kernel completes
    unsigned int *err;
};

template <int FMT>
struct BUnitK {
    static constexpr int value = (FMT == F_BF16 || FMT == F_F16) ? 8 : 32;
};

template <int FMT>
struct BAcc {
    float a[BUnitK<FMT>::value];
    float s0, s1;  // Q4_K: sum of dy * d * sc (the carrier's offset) and of dy * dmin * m
    // Q4_K: the unit's 6-bit scale and min gathered from the header by byte
    // permutes (selectors fixed per thread, as its unit is): p0 byte
    // selector, p1 / p2 masks of the low field and of the top bits, sh the
    // nibble of the quant bytes, lowgrp sub-blocks 0..3
    uint32_t p0, p1, p2, sh, lowgrp;
};


// acc += dyj * (unit u of the row at shared address rowa)
template <int FMT>
__device__ __forceinline__ void unit_axpy(uint32_t rowa, int u, float dyj, BAcc<FMT> &st) {
    if (FMT == F_BF16 || FMT == F_F16) {
        const uint4 v = lds128(rowa + 16u * u);
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
        const float2 dd = make_float2(dyj, dyj);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 wf;
            if (FMT == F_BF16) {
                wf.x = __uint_as_float(wd[i] << 16);
                wf.y = __uint_as_float(wd[i] & 0xFFFF0000u);
            } else {
                wf = __half22float2(*reinterpret_cast<const __half2 *>(&wd[i]));
            }
            const float2 r = ffma2(wf, dd, make_float2(st.a[2 * i], st.a[2 * i + 1]));
            st.a[2 * i] = r.x;
            st.a[2 * i + 1] = r.y;
        }
    } else if (FMT == F_Q4_0) {
        const uint32_t base = rowa + 18u * u;
        const float a = dyj * f16_bits_to_f32(lds16(base));
        uint32_t qw[4];
        lds_words_a2<4>(base + 2, qw);
        const float2 aa = make_float2(a, a);
        const float2 zp = make_float2(-8388616.0f, -8388616.0f);  // -(2^23 + 8)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = qw[i] & 0x0F0F0F0Fu, hi = (qw[i] >> 4) & 0x0F0F0F0Fu;
            // element 4i + b: low nibble of byte 4i + b; element 16 + 4i + b: its high nibble
            float2 r, f;
            f = fadd2(make_float2(byte_magic23<0>(lo), byte_magic23<1>(lo)), zp);
            r = ffma2(f, aa, make_float2(st.a[4 * i], st.a[4 * i + 1]));
            st.a[4 * i] = r.x; st.a[4 * i + 1] = r.y;
            f = fadd2(make_float2(byte_magic23<2>(lo), byte_magic23<3>(lo)), zp);
            r = ffma2(f, aa, make_float2(st.a[4 * i + 2], st.a[4 * i + 3]));
            st.a[4 * i + 2] = r.x; st.a[4 * i + 3] = r.y;
            f = fadd2(make_float2(byte_magic23<0>(hi), byte_magic23<1>(hi)), zp);
            r = ffma2(f, aa, make_float2(st.a[16 + 4 * i], st.a[16 + 4 * i + 1]));
            st.a[16 + 4 * i] = r.x; st.a[16 + 4 * i + 1] = r.y;
            f = fadd2(make_float2(byte_magic23<2>(hi), byte_magic23<3>(hi)), zp);
            r = ffma2(f, aa, make_float2(st.a[16 + 4 * i + 2], st.a[16 + 4 * i + 3]));
            st.a[16 + 4 * i + 2] = r.x; st.a[16 + 4 * i + 3] = r.y;
        }
    } else if (FMT == F_Q4_K) {
        // unit u = sub-block s of super-block b; its 32 codes are the low
        // (s even) or high (s odd) nibbles of quant bytes 32 (s / 2) ..
        const int b = u >> 3, c = (u & 7) >> 1;
        const uint32_t sb = rowa + 144u * b;
        const uint4 hdr = lds128(sb);
        const uint4 q0 = lds128(sb + 16u + 32u * c);
        const uint4 q1 = lds128(sb + 32u + 32u * c);
        // [sc, m] in bytes 0 and 1: s < 4: sc = y byte s & 63, m = z byte s & 63;
        // s = 4 + t: sc = w byte t & 15 | (y byte t >> 6) << 4,
        //            m = w byte t >> 4 | (z byte t >> 6) << 4
        const uint32_t fa = prmt(st.lowgrp ? hdr.y : hdr.w, st.lowgrp ? hdr.z : hdr.w >> 4, st.p0);
        const uint32_t fb = prmt(hdr.y, hdr.z, st.p0) >> 2;
        const uint32_t scm = (fa & st.p1) | (fb & st.p2);
        // (d sc, dmin m) exactly: (2^23 + v) s - 2^23 s, one packed fma
        const float2 sd = make_float2(f16_bits_to_f32(hdr.x & 0xFFFFu), f16_bits_to_f32(hdr.x >> 16));
        const float2 dsm = ffma2(make_float2(byte_magic23<0>(scm), byte_magic23<1>(scm)), sd,
                                 make_float2(-8388608.0f * sd.x, -8388608.0f * sd.y));
        const float a = dyj * dsm.x;
        const float bm = dyj * dsm.y;
        const uint32_t sh = st.sh;
        const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const float2 aa = make_float2(a, a);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t nib = (wd[i] >> sh) & 0x0F0F0F0Fu;
            float2 r;
            r = ffma2(make_float2(byte_half_plus<0>(nib), byte_half_plus<1>(nib)), aa,
                      make_float2(st.a[4 * i], st.a[4 * i + 1]));
            st.a[4 * i] = r.x; st.a[4 * i + 1] = r.y;
            r = ffma2(make_float2(byte_half_plus<2>(nib), byte_half_plus<3>(nib)), aa,
                      make_float2(st.a[4 * i + 2], st.a[4 * i + 3]));
            st.a[4 * i + 2] = r.x; st.a[4 * i + 3] = r.y;
        }
        st.s0 += a;
        st.s1 += bm;
    } else if (FMT == F_Q8_0) {
        // signed codes exactly: 2^23 + (q + 128) - (2^23 + 128)
        const uint32_t base = rowa + 34u * u;
        const float a = dyj * f16_bits_to_f32(lds16(base));
        uint32_t qw[8];
        lds_words_a2<8>(base + 2, qw);
        const float2 aa = make_float2(a, a);
        const float2 zp = make_float2(-8388736.0f, -8388736.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t v = qw[i] ^ 0x80808080u;
            float2 f = fadd2(make_float2(byte_magic23<0>(v), byte_magic23<1>(v)), zp);
            float2 r = ffma2(f, aa, make_float2(st.a[4 * i], st.a[4 * i + 1]));
            st.a[4 * i] = r.x; st.a[4 * i + 1] = r.y;
            f = fadd2(make_float2(byte_magic23<2>(v), byte_magic23<3>(v)), zp);
            r = ffma2(f, aa, make_float2(st.a[4 * i + 2], st.a[4 * i + 3]));
            st.a[4 * i + 2] = r.x; st.a[4 * i + 3] = r.y;
        }
    } else if (FMT == F_Q5_0) {
        const uint32_t base = rowa + 22u * u;
        const float a = dyj * f16_bits_to_f32(lds16(base));
        uint32_t qh[1], qw[4];
        lds_words_a2<1>(base + 2, qh);
        lds_words_a2<4>(base + 6, qw);
        const float2 aa = make_float2(a, a);
        const float2 zp = make_float2(-8388624.0f, -8388624.0f);  // -(2^23 + 16)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bits j of a 4-bit field of qh -> bit 4 of byte j
            const uint32_t hl = (((qh[0] >> (4 * i)) & 15u) * 0x02040810u) & 0x10101010u;
            const uint32_t hh = (((qh[0] >> (16 + 4 * i)) & 15u) * 0x02040810u) & 0x10101010u;
            const uint32_t lo = (qw[i] & 0x0F0F0F0Fu) | hl, hi = ((qw[i] >> 4) & 0x0F0F0F0Fu) | hh;
            float2 r, f;
            f = fadd2(make_float2(byte_magic23<0>(lo), byte_magic23<1>(lo)), zp);
            r = ffma2(f, aa, make_float2(st.a[4 * i], st.a[4 * i + 1]));
            st.a[4 * i] = r.x; st.a[4 * i + 1] = r.y;
            f = fadd2(make_float2(byte_magic23<2>(lo), byte_magic23<3>(lo)), zp);
            r = ffma2(f, aa, make_float2(st.a[4 * i + 2], st.a[4 * i + 3]));
            st.a[4 * i + 2] = r.x; st.a[4 * i + 3] = r.y;
            f = fadd2(make_float2(byte_magic23<0>(hi), byte_magic23<1>(hi)), zp);
            r = ffma2(f, aa, make_float2(st.a[16 + 4 * i], st.a[16 + 4 * i + 1]));
            st.a[16 + 4 * i] = r.x; st.a[16 + 4 * i + 1] = r.y;
            f = fadd2(make_float2(byte_magic23<2>(hi), byte_magic23<3>(hi)), zp);
            r = ffma2(f, aa, make_float2(st.a[16 + 4 * i + 2], st.a[16 + 4 * i + 3]));
            st.a[16 + 4 * i + 2] = r.x; st.a[16 + 4 * i + 3] = r.y;
        }
    } else {  // F_Q6_K
        // unit u: super-block b, half h, byte group gq; element 8 r + i is
        // weight 128 h + 32 r + 8 gq + i, with scale scales[8 h + 2 r + gq / 2]
        const int b = u >> 3, h = (u >> 2) & 1, gq = u & 3;
        const uint32_t sb = rowa + 210u * b;
        uint32_t A[2], B[2], H[2], S[2];
        lds_words_a2<2>(sb + 64u * h + 8u * gq, A);
        lds_words_a2<2>(sb + 64u * h + 32u + 8u * gq, B);
        lds_words_a2<2>(sb + 128u + 32u * h + 8u * gq, H);
        lds_words_a2<2>(sb + 192u + 8u * h, S);
        const float dd = dyj * f16_bits_to_f32(lds16(sb + 208u));
        float ar[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t pos = 8u * (2u * (uint32_t)(r & 1) + (uint32_t)(gq >> 1));
            int32_t scv;
            asm("bfe.s32 %0, %1, %2, 8;" : "=r"(scv) : "r"(S[r >> 1]), "r"(pos));
            ar[r] = dd * (float)scv;
        }
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
            const uint32_t q[4] = {
                (A[wi] & 0x0F0F0F0Fu) | ((H[wi] << 4) & 0x30303030u),
                (B[wi] & 0x0F0F0F0Fu) | ((H[wi] << 2) & 0x30303030u),
                ((A[wi] >> 4) & 0x0F0F0F0Fu) | (H[wi] & 0x30303030u),
                ((B[wi] >> 4) & 0x0F0F0F0Fu) | ((H[wi] >> 2) & 0x30303030u)};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 aa = make_float2(ar[r], ar[r]);
                const int e = 8 * r + 4 * wi;
                // q - 32 exactly as 2^23 + q - (2^23 + 32)
                const float2 zp = make_float2(-8388640.0f, -8388640.0f);
                float2 v, f;
                f = fadd2(make_float2(byte_magic23<0>(q[r]), byte_magic23<1>(q[r])), zp);
                v = ffma2(f, aa, make_float2(st.a[e], st.a[e + 1]));
                st.a[e] = v.x; st.a[e + 1] = v.y;
                f = fadd2(make_float2(byte_magic23<2>(q[r]), byte_magic23<3>(q[r])), zp);
                v = ffma2(f, aa, make_float2(st.a[e + 2], st.a[e + 3]));
                st.a[e + 2] = v.x; st.a[e + 3] = v.y;
            }
        }
    }
}

// Final dx value of element e of unit u, and its k index.
template <int FMT>
__device__ __forceinline__ void unit_result(const BAcc<FMT> &st, int u, int e, float &v,
                                            int64_t &kidx) {
    if (FMT == F_BF16 || FMT == F_F16) {
        v = st.a[e];
        kidx = 8 * (int64_t)u + e;
    } else if (FMT == F_Q4_0 || FMT == F_Q8_0 || FMT == F_Q5_0) {
        v = st.a[e];  // exact q - z: no carrier
        kidx = 32 * (int64_t)u + e;
    } else if (FMT == F_Q4_K) {
        // sum (a q - dy dm) = 256 sum a (0.5 + q/256) - 128 sum a - sum dy dm
        v = fmaf(256.0f, st.a[e], -fmaf(128.0f, st.s0, st.s1));
        kidx = 32 * (int64_t)u + e;
    } else {
        const int r = e >> 3, i = e & 7;
        v = st.a[e];  // exact q - 32
        const int b = u >> 3, h = (u >> 2) & 1, gq = u & 3;
        kidx = 256 * (int64_t)b + 128 * h + 32 * r + 8 * gq + i;
    }
}

template <int FMT>
__global__ void __launch_bounds__(kBwThreads, 2) back_input_kernel(const BackParams p) {
    constexpr int UK = BUnitK<FMT>::value;
    extern __shared__ __align__(128) uint8_t smem[];
    const int NS = p.NS, SR = p.SR, SB = p.SB;
    const uint32_t bar0 = smem_addr(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 16 * NS);
    float *dys = reinterpret_cast<float *>(smem + ((16 * NS + 16 + 127) & ~127));
    const uint32_t stage_off =
        (uint32_t)((((16 * NS + 16 + 127) & ~127) + 4 * p.dy_cap + 127) & ~127);
    uint8_t *stages = smem + stage_off;
    const uint32_t stage0 = bar0 + stage_off;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (NS + s); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int64_t r0 = p.j0 + (int64_t)cta * p.rows_base + (cta < p.rows_rem ? cta : p.rows_rem);
    const int64_t nrows = p.rows_base + (cta < p.rows_rem ? 1 : 0);
    const int nst = (int)((nrows + SR - 1) / SR);
    const int64_t R = p.row_bytes;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kBwWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // the sum kernel that follows may start launching; it waits for this grid
    pdl_launch_dependents();

    if (warp == kBwWarps) {
        // ---------------- producer: one lane streams the weight bytes ----------------
        if (lane != 0) return;
        const int64_t lim = p.w_total & ~(int64_t)15;
        int issued = 0;
        for (int s = 0; s < nst; ++s) {
            const int slot = s % NS;
            if (s >= NS && !mbar_wait(empty(slot), ((s / NS) + 1) & 1)) {
                record_error(p.err, DERR_GEMV_EMPTY);
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            const int64_t ra = r0 + (int64_t)s * SR;
            const int64_t rb = min(ra + SR, r0 + nrows);
            const int64_t A = ra * R, B = rb * R;
            const int64_t a16 = A & ~(int64_t)15, b16 = (B + 15) & ~(int64_t)15;
            const int64_t tend = min(b16, lim);
            if (B > lim) {  // bytes after the last whole 16-byte chunk of W
                for (int64_t q = max(a16, lim); q < B; ++q)
                    stages[(int64_t)slot * SB + (q - a16)] = p.w[q];
            }
            const uint32_t tx = tend > a16 ? (uint32_t)(tend - a16) : 0u;
            mbar_arrive_expect_tx(full(slot), tx);
            if (tx) bulk_g2s(stage0 + (uint32_t)slot * SB, p.w + a16, tx, full(slot));
            ++issued;
        }
        // no copy may land after this CTA exits
        for (int s = max(0, issued - NS); s < issued; ++s)
            if (!mbar_wait(full(s % NS), (s / NS) & 1)) record_error(p.err, DERR_TEARDOWN);
        return;
    }

    // ---------------- consumers ----------------
    // Under programmatic launch the weight stream starts while the preceding
    // kernel finishes; dy is read after it unless the caller vouched that it
    // does not write dy.
    if (!p.x_ready) pdl_wait_prev();
    for (int64_t i = tid; i < nrows; i += kBwCons) dys[i] = __ldg(p.dy + r0 + i);
    named_barrier(1, kBwCons);
    const int U = p.U, G = p.G;
    // thread -> (row group g, unit u); units beyond U (G * U < 256) idle
    const int g = tid / U;
    const int u = tid - g * U;
    const bool active = g < G;
    BAcc<FMT> st;
#pragma unroll
    for (int e = 0; e < UK; ++e) st.a[e] = 0.0f;
    st.s0 = st.s1 = 0.0f;
    {
        const uint32_t sbk = (uint32_t)(u & 7);  // Q4_K: sub-block of the unit
        st.lowgrp = sbk < 4;
        const uint32_t t = st.lowgrp ? sbk : sbk - 4u;
        st.p0 = t | ((t + 4u) << 4);
        st.p1 = st.lowgrp ? 0x3F3Fu : 0x0F0Fu;
        st.p2 = st.lowgrp ? 0u : 0x3030u;
        st.sh = (sbk & 1) ? 4u : 0u;
    }
    bool failed = false;
    for (int s = 0; s < nst; ++s) {
        const int slot = s % NS;
        if (!failed && !mbar_wait(full(slot), (s / NS) & 1)) {
            failed = true;
            *abort_flag = 1;
            record_error(p.err, DERR_GEMV_FULL);
        }
        const int64_t ra = r0 + (int64_t)s * SR;
        const int64_t rb = min(ra + SR, r0 + nrows);
        const int rows_in = (int)(rb - ra);
        const int64_t a16 = (ra * R) & ~(int64_t)15;
        const uint32_t sbase = stage0 + (uint32_t)slot * SB;
        if (!failed && active) {
            for (int rr = g; rr < rows_in; rr += G) {
                const uint32_t rowa = sbase + (uint32_t)((ra + rr) * R - a16);
                unit_axpy<FMT>(rowa, u, dys[ra - r0 + rr], st);
            }
        }
        // the stage is refilled by a bulk copy (the async proxy) once every
        // consumer warp has arrived: order this thread's reads of it first
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(slot));
    }
    // row groups -> one partial per k index, through shared memory (the ring
    // is idle: every stage has been consumed)
    named_barrier(1, kBwCons);
    // [G][k + k/32] floats: one padding word per 32 keeps a warp's writes
    // (32 units at the same element) on distinct banks
    float *red = reinterpret_cast<float *>(stages);
    const int64_t k = p.k;
    const int64_t kpad = k + k / 32;
    if (active) {
#pragma unroll
        for (int e = 0; e < UK; ++e) {
            float v;
            int64_t ki;
            unit_result<FMT>(st, u, e, v, ki);
            red[(int64_t)g * kpad + ki + (ki >> 5)] = v;
        }
    }
    named_barrier(1, kBwCons);
    // the partials' workspace may still be read by the preceding call's sum
    pdl_wait_prev();
    float *out = p.part + (int64_t)cta * k;
    for (int64_t i = tid; i < k; i += kBwCons) {
        float v = 0.0f;
        for (int gg = 0; gg < G; ++gg) v += red[(int64_t)gg * kpad + i + (i >> 5)];
        out[i] = (failed || *abort_flag) ? 0.0f : v;
    }
}

// dx[i] (+)= sum over CTAs c of part[c][i], in a fixed order: a CTA takes 32
// consecutive i; warp w sums the partials c = w, w + 8, ... (four loads in
// flight), then one warp adds the eight warp sums in order.
__global__ void __launch_bounds__(256) back_input_sum_kernel(const float *__restrict__ part,
                                                             int parts, int64_t k, float *dx,
                                                             int accumulate) {
    __shared__ float ws[8][33];
    // launched as a programmatic dependent of the partials' kernel: wait for
    // it before reading; a following call's kernels may start streaming now
    pdl_wait_prev();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t i = (int64_t)blockIdx.x * 32 + lane;
    float v = 0.0f;
    if (i < k) {
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        int c = w;
        for (; c + 24 < parts; c += 32) {
            a0 += __ldg(part + (int64_t)c * k + i);
            a1 += __ldg(part + (int64_t)(c + 8) * k + i);
            a2 += __ldg(part + (int64_t)(c + 16) * k + i);
            a3 += __ldg(part + (int64_t)(c + 24) * k + i);
        }
        for (; c < parts; c += 8) a0 += __ldg(part + (int64_t)c * k + i);
        v = (a0 + a1) + (a2 + a3);
    }
    ws[w][lane] = v;
    __syncthreads();
    if (w == 0 && i < k) {
        float t = accumulate ? dx[i] : 0.0f;
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) sum += ws[j][lane];
        dx[i] = t + sum;
    }
}

template <int FMT>
cudaError_t launch_bw_t(const BackParams &p, int grid, size_t smem, cudaStream_t s, bool overlap) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(back_input_kernel<FMT>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (!overlap) {
        back_input_kernel<FMT><<<grid, kBwThreads, smem, s>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kBwThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, back_input_kernel<FMT>, p);
}

int unit_k_of(int fmt) { return (fmt == F_BF16 || fmt == F_F16) ? 8 : 32; }

}  // namespace

bool back_input_supports(int fmt, int64_t k) {
    if (fmt < F_BF16 || fmt > kLastFmt || k <= 0) return false;
    const int uk = unit_k_of(fmt);
    return k % uk == 0 && k / uk <= kBwCons;
}

static int64_t bw_plan(int fmt, int64_t k, int64_t R, int64_t M, int sm_count, int *grid_out,
                       int64_t *SR_out, int *NS_out, int *SB_out, size_t *smem_out,
                       int *dy_cap_out) {
    const int uk = unit_k_of(fmt);
    const int U = (int)(k / uk);
    const int G = kBwCons / U;
    const int ctas_target = 2 * sm_count;
    const int64_t per_cta = (M + ctas_target - 1) / ctas_target;
    int64_t SR = std::max<int64_t>(G, 32768 / R / G * G);
    if (per_cta < SR) SR = std::max<int64_t>(G, (per_cta + G - 1) / G * G);
    const int SB = (int)(((SR * R + 32) + 127) & ~(int64_t)127);
    const int64_t nstage_total = (M + SR - 1) / SR;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(nstage_total, ctas_target));
    const int64_t rows_max = (M + grid - 1) / grid;
    const int dy_cap = (int)rows_max;
    const size_t fixed = (size_t)(((16 * 8 + 16 + 127) & ~127) + 4 * dy_cap + 127) & ~(size_t)127;
    // the reduction reuses the ring: it must hold G x k floats
    const size_t red = (size_t)4 * G * (k + k / 32);
    int NS = 2;
    while (NS < 8 && fixed + (size_t)(NS + 1) * SB <= 110 * 1024) ++NS;
    while ((size_t)NS * SB < red && NS < 16) ++NS;
    *grid_out = grid;
    *SR_out = SR;
    *NS_out = NS;
    *SB_out = SB;
    *dy_cap_out = dy_cap;
    *smem_out = fixed + (size_t)NS * SB;
    return (int64_t)grid * k * 4;
}

size_t back_input_workspace_bytes(int fmt, int64_t k, int64_t n, int64_t j0, int64_t j1,
                                  const DeviceInfo &dev) {
    if (!back_input_supports(fmt, k) || j1 <= j0) return 0;
    int grid, NS, SB, dy_cap;
    int64_t SR;
    size_t smem;
    const int64_t R = (k / block_elems(fmt)) * block_bytes(fmt);
    (void)n;
    return (size_t)bw_plan(fmt, k, R, j1 - j0, dev.sm_count, &grid, &SR, &NS, &SB, &smem, &dy_cap);
}

cudaError_t launch_back_input(const BackLaunch &b, const DeviceInfo &dev, cudaStream_t s) {
    if (!back_input_supports(b.fmt, b.k)) return cudaErrorNotSupported;
    const int64_t M = b.j1 - b.j0;
    if (M <= 0) return cudaSuccess;
    int grid, NS, SB, dy_cap;
    int64_t SR;
    size_t smem;
    bw_plan(b.fmt, b.k, b.row_bytes, M, dev.sm_count, &grid, &SR, &NS, &SB, &smem, &dy_cap);
    if (smem > 200 * 1024) return cudaErrorNotSupported;
    BackParams p;
    p.w = b.w;
    p.dy = b.dy;
    p.part = static_cast<float *>(b.workspace);
    p.k = b.k;
    p.row_bytes = b.row_bytes;
    p.w_total = b.row_bytes * b.n;
    p.j0 = b.j0;
    p.rows_base = M / grid;
    p.rows_rem = (int)(M % grid);
    p.U = (int)(b.k / unit_k_of(b.fmt));
    p.G = kBwCons / p.U;
    p.SR = (int)SR;
    p.SB = SB;
    p.NS = NS;
    p.dy_cap = dy_cap;
    p.x_ready = b.x_ready ? 1 : 0;
    p.err = dev.err;
    cudaError_t e;
    switch (b.fmt) {
    case F_BF16: e = launch_bw_t<F_BF16>(p, grid, smem, s, b.overlap_prev); break;
    case F_F16: e = launch_bw_t<F_F16>(p, grid, smem, s, b.overlap_prev); break;
    case F_Q4_0: e = launch_bw_t<F_Q4_0>(p, grid, smem, s, b.overlap_prev); break;
    case F_Q4_K: e = launch_bw_t<F_Q4_K>(p, grid, smem, s, b.overlap_prev); break;
    case F_Q6_K: e = launch_bw_t<F_Q6_K>(p, grid, smem, s, b.overlap_prev); break;
    case F_Q8_0: e = launch_bw_t<F_Q8_0>(p, grid, smem, s, b.overlap_prev); break;
    case F_Q5_0: e = launch_bw_t<F_Q5_0>(p, grid, smem, s, b.overlap_prev); break;
    default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    // the sum: a programmatic dependent of the partials' kernel (it waits for it)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((b.k + 31) / 32));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float *part = p.part;
    const int parts = grid;
    const int64_t kk = b.k;
    float *dx = b.dx;
    const int acc = b.accumulate;
    return cudaLaunchKernelEx(&cfg, back_input_sum_kernel, part, parts, kk, dx, acc);
}

}  // namespace qmm
