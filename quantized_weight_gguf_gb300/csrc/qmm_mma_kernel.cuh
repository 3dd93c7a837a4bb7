// qmm_mma_kernel.cuh -- N-token fused dequantize + tensor-core product on sm_103a:
// Y[t][j] = sum_i X[t][i] W[j][i] for a tile of 128 output columns j and BN
// tokens t per CTA.
//
// CTAs run in clusters of two: the pair works on adjacent 128-row tiles of W
// and the same tokens, and each CTA fetches half of every X tile with a TMA
// multicast into both CTAs' shared memory, halving the L2 traffic for X.
// Pipeline per CTA (one CTA per SM, warp-specialised):
//   warp 0      TMA producer: its half of each fp16 X tile [BN tokens x 64 k]
//               -> shared memory of both CTAs (128-byte swizzle);
//   warp 1      allocates the fp32 accumulator in tensor memory (TMEM) and one
//               lane issues tcgen05.mma (M=128, N=BN, K=16, fp16 in, fp32 acc);
//   warps 2..17 dequantize W in two groups of 8 warps that take alternate
//               k-steps: thread (r, h) turns 32 weights of row r per k-step
//               into fp16 and stores them in the same swizzled K-major layout
//               the MMA descriptor describes; after the k-loop all 16 warps
//               drain the accumulator TMEM -> registers -> y;
//   warp 18     raw-tile formats: streams raw W tiles (128 rows x a 256-wide
//               k slice) ahead of the dequant warps, by TMA (Q6_K rows by
//               16-byte cp.async copies of its 32 lanes).
// X is converted to fp16 once per call by a small kernel that also scales each
// token row by a power of two (exact) so it fits fp16's range; the epilogue
// multiplies by the inverse power.
//
// Precision modes (fp16 operands round each product's inputs to 11 bits):
//   MODE 1  W16 . X16                      one product per output; the
//           templates keep it but nothing instantiates it: a single fp16 copy
//           of a structured x (a constant row, all-positive terms) errs
//           coherently by up to 2^-12 of sum |x w| at any k
//   MODE 2  W16 . (X_hi + X_lo)            x split into two fp16 terms: the B
//           tile holds BN/2 tokens' hi rows then their lo rows, and the
//           epilogue adds column c and c + BN/2 (exact for fp16-exact W)
//   MODE 3  (W_hi + W_lo) . (X_hi + X_lo)  also w split: the A tile holds 64
//           rows' hi parts then their lo parts; the epilogue adds the row
//           pair through shared memory.
//
// The kernel and its launch templates live here; qmm_mma.cu holds the host
// planning and the x conversion, and the qmm_mma_inst_*.cu units instantiate
// the kernel for groups of formats (compiled in parallel).
#pragma once
#include <cuda.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "qmm_decode.cuh"
#include "qmm_internal.h"

namespace qmm {

constexpr int kDeqWarps = 16;                     // two groups of 8, alternate k-steps
constexpr int kRawWarp = 2 + kDeqWarps;             // streams raw W tiles
constexpr int kMmaThreads = 32 * (kRawWarp + 1);
constexpr int kBM = 128;
constexpr int kBK = 64;

struct MmaParams {
    const uint8_t *w;
    float *y;
    const float *xscale;
    int64_t k, n, n_tokens, row_bytes;
    int64_t j0, j1;
    int KS;
    int accumulate;
    int pairs;       // pairs of 128-row tiles (a cluster of two CTAs takes one pair)
    int tiles_n;     // token tiles
    int full_units;  // pair-tiles computed whole (the first units)
    int split;       // the remaining pair-tiles are computed as `split` k-ranges each
    int n_units;     // full_units + (pairs * tiles_n - full_units) * split
    unsigned int *err;
    // gated pairs: y = act(gate) * (this product); act 1 SwiGLU, 2 GeGLU, 0 none
    const float *gate;
    int glu;
    int tma_epi;  // y written through shared memory by tensor stores (map tmy)
    int64_t w_rows;  // rows of the W buffer (n, or n_experts slices of n)
    int ss;          // 16-bit W tiles read as the MMA's A operand from shared memory (mma_ssable)
};

// Affine formats also read a bf16 scale and bias per group of 64 from two
// arrays [n][k/64] (aux_row_bytes per row). A separate parameter type: the
// other formats' kernels keep their parameters as they are.
struct MmaAffFields {
    const uint8_t *sc, *bi;
    int64_t aux_row_bytes;
};
struct MmaAffParams : MmaParams, MmaAffFields {};

// Expert-grouped products (mixture of experts over many positions): the
// (position, slot) pairs are routed on the device into expert-sorted rows of
// x; x row i of the sorted order goes to y row perm[i]. Expert e owns the
// sorted rows [row_off[e], row_off[e + 1]) and the units
// [unit_off[e], unit_off[e + 1]) of the schedule (its token tiles times the
// row pairs), and W rows e * slice_rows + j. GGUF formats only.
struct MmaGrpFields {
    const int *row_off, *unit_off, *perm;
    int n_experts;
    int64_t slice_rows;
};
struct MmaGrpParams : MmaParams, MmaGrpFields {};
// everything the host fills in
struct MmaHostParams : MmaAffParams, MmaGrpFields {};
template <int FMT, bool GRP = false>
using MmaParamsOf = typename std::conditional<
    GRP, MmaGrpParams,
    typename std::conditional<is_affine(FMT), MmaAffParams, MmaParams>::type>::type;

// Q4_K super-blocks of 128 rows staged raw by TMA (one 128 x 144-byte box per
// 256-wide slice of k), then decoded from shared memory.
constexpr int kRawBytes = kBM * 144;

// Raw W tiles (128 rows of a 256-wide k slice each): staged by TMA for Q4_K
// super-blocks (144 B), eight 32-weight blocks of Q4_0 (144 B), Q5_0 (176 B)
// or Q8_0 (272 B), and affine code words (128 B at 4 bits, 256 B at 8; their
// scales and biases come from global memory per thread). Q6_K's 210-byte
// super-blocks start on 2-byte boundaries, which no TMA box can: the raw
// loader's 32 lanes copy each row's 224 bytes from the 16-byte boundary at or
// below its super-block, into a 240-byte row of the tile, in 16-byte cp.async
// copies (one arrival a lane on the slot's barrier). MODE 3
// (rows split into hi / lo halves) decodes from registers; so do the block
// formats when k % 256 != 0.
__host__ __device__ constexpr int raw_slice_bytes(int fmt, int mode) {
    return mode == 3 ? 0
           : fmt == F_Q4_K ? 144
           : fmt == F_AFF4 ? 128
           : fmt == F_AFF8 ? 256
           : fmt == F_Q4_0 ? 144
           : fmt == F_Q5_0 ? 176
           : fmt == F_Q8_0 ? 272
           : fmt == F_Q6_K ? 240 : 0;
}
// Raw tiles filled row by row by the loader lanes (no tensor map)
__host__ __device__ constexpr bool raw_rowcopy(int fmt) { return fmt == F_Q6_K; }
// 16-bit formats in split-x mode (ungrouped) can take their W tiles as the
// MMA's A operand straight from shared memory: nothing to decode. The raw
// ring then holds one 128 x 64 tile per k-step (16 KB, 128-byte swizzled,
// the layout of the x tiles). A call takes that form (MmaParams::ss) when its
// rows admit a tensor map (k % 8 == 0); otherwise the same instance decodes
// from per-thread loads.
__host__ __device__ constexpr bool mma_ssable(int fmt, int mode, bool grp) {
    return (fmt == F_BF16 || fmt == F_F16) && mode == 2 && !grp;
}
__host__ __device__ constexpr int mma_ring_bytes(int fmt, int mode, bool grp) {
    return mma_ssable(fmt, mode, grp) ? kBM * kBK * 2 : kBM * raw_slice_bytes(fmt, mode);
}
constexpr int kQ6kWindow = 224;  // bytes copied per row: covers 210 from any even offset below 16
// Block formats whose raw tiles hold whole 32-weight blocks (read with
// realigning loads: a block starts on a 2-byte boundary)
__host__ __device__ constexpr bool raw_block32(int fmt) {
    return fmt == F_Q4_0 || fmt == F_Q5_0 || fmt == F_Q8_0;
}
// Element size of the raw tiles' tensor map: a box row is at most 256
// elements, so Q8_0's 272-byte slices go as 136 16-bit elements
__host__ __device__ constexpr int raw_elem_bytes(int fmt) { return fmt == F_Q8_0 ? 2 : 1; }

// Tensor memory (512 columns x 128 lanes of 32 bits, all taken by the one CTA
// on the SM): the fp32 accumulator(s) first, then a ring of NA dequantized W
// stages (A operand: row r on lane r, k pairs packed per column, 32 columns
// per 64-wide k-step). Shared memory: a ring of NB x stages (streamed from
// L2 by TMA) and, for the raw-tile formats, kNR raw W tiles of 128 rows.
//
// A stage is KA = 4 k-steps (one 256-wide super-block): each dequant thread
// then pays one raw-tile wait, one slot wait and one arrival per two decoded
// chunks. An x stage is KB k-steps, 32 KB at most (the x tile of 256 tokens
// is 32 KB per k-step).
// The epilogue stages y in shared memory and writes it with tensor stores
// (split x mode, ungrouped products): each of the 16 dequant warps owns
// 2 KB, 32 rows x 16 tokens of fp32.
constexpr int kEpiStageBytes = 16 * 2048;
__host__ __device__ constexpr bool mma_tma_epilogue(int mode, bool grp) { return mode == 2 && !grp; }

// EPI: bytes of the epilogue's staging area (0: y stored from registers).
// RAWB: bytes of one raw W tile (0: no raw ring); DEEP: a deeper raw ring
template <int BN, int RAWB, int EPI = 0, bool DEEP = false>
struct MmaCfg {
    static constexpr bool RAW = RAWB > 0;
    static constexpr int KA = 4;
    static constexpr int KB = BN >= 256 ? 1 : (BN >= 128 ? 2 : 4);
    static constexpr int kBBytes = BN * kBK * 2;            // one k-step of x
    static constexpr int kBStage = KB * kBBytes;
    static constexpr int kAccCols = BN < 32 ? 32 : BN;      // one accumulator
    // Accumulators that the K = 16 steps of a k-step go to in turn (summed
    // in the epilogue). One: back-to-back MMAs into the same accumulator run
    // at the full rate (16 cycles each at N = 32, measured alone), and one
    // accumulator leaves TMEM to a three-stage A ring at every tile width.
    static constexpr int kNAcc = 1;
    static constexpr int kACol0 = kNAcc * kAccCols;         // first A column
    static constexpr int kAStageCols = KA * 32;
    static constexpr int kNAFit = (512 - kACol0) / kAStageCols;
    static constexpr int NA = kNAFit > 3 ? 3 : kNAFit;
    static constexpr int kCols = 512;
    // raw W stages: as many as fit, up to 4, next to a minimum x ring of four
    // k-steps (two stages at least); HBM latency is hidden by the raw ring, L2
    // latency by the x ring (8 raw stages at small token tiles measured no
    // faster at N <= 32 and slower at N = 64)
    // The rings and the epilogue staging area share kBudget bytes (the rest
    // of the 227 KB goes to alignment, barriers and token scales). At
    // BN = 256 the x ring keeps four one-k-step stages (three measured 50 %
    // slower k-loops: L2 latency is no longer covered); the raw ring then
    // gets what is left, three or four stages (two x stages fewer only when
    // a raw tile is so large that fewer than two would fit).
    static constexpr int kBudget = 220 * 1024;
    static constexpr int kNBWant = (4 + KB - 1) / KB < 2 ? 2 : (4 + KB - 1) / KB;
    static constexpr bool kShrinkX =
        RAW && KB == 1 && (kBudget - kNBWant * kBStage - EPI) / RAWB < 2;
    static constexpr int kNBMin = kShrinkX ? kNBWant - 1 : kNBWant;
    static constexpr int kRawFit = RAW ? (kBudget - kNBMin * kBStage - EPI) / RAWB : 0;
    // 16-bit tiles read as A (DEEP) need no decode, so only the ring's depth
    // keeps HBM busy: up to 8 slots
    static constexpr int kNRMax = DEEP ? 8 : 4;
    static constexpr int kNR = RAW ? (kRawFit > kNRMax ? kNRMax : kRawFit) : 1;
    static_assert(!RAW || kNR >= 2, "raw W ring too shallow");
    static constexpr int kAvail = kBudget - (RAW ? kNR * RAWB : 0) - EPI;
    static constexpr int NB = (kAvail / kBStage) > 8 ? 8 : (kAvail / kBStage);
    static constexpr size_t kSmemUsed = (size_t)NB * kBStage +
                                        (RAW ? (size_t)kNR * RAWB : 0) + EPI + 1024 /*align*/ +
                                        512 /*barriers*/ + 2048 /*token scales*/;
    // at least half of the SM's shared memory, so that no second CTA can be
    // resident and block in its TMEM allocation (every CTA takes all 512
    // columns) while holding resources its cluster peer waits for
    static constexpr size_t kSmem = kSmemUsed < 120 * 1024 ? 120 * 1024 : kSmemUsed;
    // MODE 3 parks its low rows' sums ([BN/2 tokens][64 rows] fp32) over the x ring
    static_assert(NB * kBStage >= BN * 128, "x ring too small for the MODE 3 epilogue");
    static_assert(NB >= 2 && NA >= 2, "rings too shallow");
};

__device__ __forceinline__ bool wait_abortable(uint32_t bar, uint32_t parity,
                                               volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 32 weights -> 16 fp16x2 words, generic formats: exact fp32, then RN to fp16.
template <int FMT>
__device__ __forceinline__ void to_half_words(const Raw32<FMT> &raw, uint32_t (&hw)[16]) {
    float v[32];
    raw.decode(v);
#pragma unroll
    for (int i = 0; i < 16; ++i) hw[i] = pack_half2(v[2 * i], v[2 * i + 1]);
}

// Q4_K: w = ds*q - dm computed as (256 ds) * (0.5 + q/256) - (128 ds + dm),
// one fp32 fma per weight, then RN to fp16 (the fp16 rounding dominates).
template <>
__device__ __forceinline__ void to_half_words<F_Q4_K>(const Raw32<F_Q4_K> &raw,
                                                      uint32_t (&hw)[16]) {
    uint32_t sc, m;
    q4k_scale_min(raw.hdr.y, raw.hdr.z, raw.hdr.w, raw.s, sc, m);
    const float d = f16_bits_to_f32(raw.hdr.x & 0xFFFFu);
    const float dmin = f16_bits_to_f32(raw.hdr.x >> 16);
    const float ds = d * (float)sc;
    const float a = 256.0f * ds;
    const float c = -fmaf(128.0f, ds, dmin * (float)m);
    const float2 av = make_float2(a, a), cv = make_float2(c, c);
    const uint32_t sh = (raw.s & 1) ? 4u : 0u;
    const uint32_t wd[8] = {raw.qs[0].x, raw.qs[0].y, raw.qs[0].z, raw.qs[0].w,
                            raw.qs[1].x, raw.qs[1].y, raw.qs[1].z, raw.qs[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t nib = (wd[i] >> sh) & 0x0F0F0F0Fu;
        const float2 f01 = ffma2(av, make_float2(byte_half_plus<0>(nib), byte_half_plus<1>(nib)), cv);
        const float2 f23 = ffma2(av, make_float2(byte_half_plus<2>(nib), byte_half_plus<3>(nib)), cv);
        hw[2 * i] = pack_half2(f01.x, f01.y);
        hw[2 * i + 1] = pack_half2(f23.x, f23.y);
    }
}

// Affine 4-bit: w = q s + b as (256 s) (0.5 + q/256) + (b - 128 s), the
// code riding the exact byte carrier, two weights per packed fp32 fma, then
// RN to fp16 (b - 128 s rounds in fp32, far below the fp16 rounding of w).
// Word i holds elements 8i .. 8i+7, lowest nibble first: byte j of the
// low-nibble mask is element 8i + 2j, of the high-nibble mask 8i + 2j + 1,
// so each (low, high) byte pair is one fp16x2 word of consecutive k.
template <>
__device__ __forceinline__ void to_half_words<F_AFF4>(const Raw32<F_AFF4> &raw,
                                                      uint32_t (&hw)[16]) {
    const float sc = __uint_as_float(raw.sbits << 16), bi = __uint_as_float(raw.bbits << 16);
    const float a = 256.0f * sc, c = fmaf(-128.0f, sc, bi);
    const float2 av = make_float2(a, a), cv = make_float2(c, c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = raw.qw[i] & 0x0F0F0F0Fu, hi = (raw.qw[i] >> 4) & 0x0F0F0F0Fu;
        float2 f;
        f = ffma2(make_float2(byte_half_plus<0>(lo), byte_half_plus<0>(hi)), av, cv);
        hw[4 * i] = pack_half2(f.x, f.y);
        f = ffma2(make_float2(byte_half_plus<1>(lo), byte_half_plus<1>(hi)), av, cv);
        hw[4 * i + 1] = pack_half2(f.x, f.y);
        f = ffma2(make_float2(byte_half_plus<2>(lo), byte_half_plus<2>(hi)), av, cv);
        hw[4 * i + 2] = pack_half2(f.x, f.y);
        f = ffma2(make_float2(byte_half_plus<3>(lo), byte_half_plus<3>(hi)), av, cv);
        hw[4 * i + 3] = pack_half2(f.x, f.y);
    }
}

// Affine 8-bit: q exactly as (2^23 + q) - 2^23, then fma(q, s, b) two weights
// at a time and RN to fp16; byte j of word i is element 4i + j.
template <>
__device__ __forceinline__ void to_half_words<F_AFF8>(const Raw32<F_AFF8> &raw,
                                                      uint32_t (&hw)[16]) {
    const float sc = __uint_as_float(raw.sbits << 16), bi = __uint_as_float(raw.bbits << 16);
    const float2 sv = make_float2(sc, sc), bv = make_float2(bi, bi);
    const float2 zp = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = raw.qw[i];
        const float2 q01 = fadd2(make_float2(byte_magic23<0>(w), byte_magic23<1>(w)), zp);
        const float2 q23 = fadd2(make_float2(byte_magic23<2>(w), byte_magic23<3>(w)), zp);
        const float2 f01 = ffma2(q01, sv, bv), f23 = ffma2(q23, sv, bv);
        hw[2 * i] = pack_half2(f01.x, f01.y);
        hw[2 * i + 1] = pack_half2(f23.x, f23.y);
    }
}

__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) {
    return *reinterpret_cast<const __half2 *>(&v);
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Q4_K, per super-block: the fp16x2 constants of its four 64-weight chunks
// (chunk c holds sub-block 2c in the low nibbles, 2c + 1 in the high ones).
// The 6-bit scales sc[0..7] and mins m[0..7] are first gathered as bytes of
// four words from the header words y (scales[0..3]), z (scales[4..7]) and
// w (scales[8..11]): sc[s] = y byte s & 63 and m[s] = z byte s & 63 for
// s < 4; for s = 4 + t, the low / high nibble of w byte t below the top two
// bits of y / z byte t.
struct Q4KChunk {
    __half2 s0, n0, s1, n1, e0, e1;
};

__device__ __forceinline__ void q4k_superblock_consts(const uint4 &hdr, __half2 &d2,
                                                      Q4KChunk (&cc)[4]) {
    const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, m_lo = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    d2 = u32_as_h2((hdr.x & 0xFFFFu) * 0x10001u);
    const __half2 ndmin2 = __hneg2(u32_as_h2((hdr.x >> 16) * 0x10001u));
    const __half2 k1024 = u32_as_h2(0x64006400u);
    // byte j of v (< 64) as the exact fp16 pair (v, v): (1024 + v) - 1024
    auto byte_h2 = [&](uint32_t v, uint32_t j) {
        return __hsub2(u32_as_h2(prmt(v, 0x64646464u, j | 0x40u | (j << 8) | 0x4000u)), k1024);
    };
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t scw = c < 2 ? sc_lo : sc_hi, mw = c < 2 ? m_lo : m_hi;
        const uint32_t j = 2u * (uint32_t)(c & 1);
        const __half2 sa = byte_h2(scw, j), sb = byte_h2(scw, j + 1);
        cc[c].s0 = sa;
        cc[c].n0 = __hmul2(sa, u32_as_h2(0xE400E400u));   // * -1024
        cc[c].s1 = __hmul2(sb, u32_as_h2(0x2C002C00u));   // / 16
        cc[c].n1 = __hmul2(sb, u32_as_h2(0xD400D400u));   // * -64
        // -fp16(dmin m): the exact product rounded once
        cc[c].e0 = __hmul2(ndmin2, byte_h2(mw, j));
        cc[c].e1 = __hmul2(ndmin2, byte_h2(mw, j + 1));
    }
}

// Half h of a Q4_K 64-weight chunk: quant bytes 16h .. 16h+15 of the chunk (q),
// i.e. weights 16h + 0..15 (low nibbles, sub-block 2c) and 32 + 16h + 0..15
// (high nibbles, sub-block 2c+1) -> 16 fp16x2 words: 0..7 low, 8..15 high.
//
// All in fp16x2 arithmetic, two weights per instruction:
//   a nibble pair becomes (1024 + q) exactly by OR-ing it into the fp16
//   pattern of 1024 (a high nibble, kept in place, gives 1024 + 16 q);
//   sc * q = (1024 + q) * sc - 1024 sc is exact in one fma (the result is an
//   integer below 2048; 1024 sc and sc / 16 are exact in fp16);
//   w = d * (sc q) - fp16(dmin m) is then rounded once.
// Only dmin * m picks up an extra fp16 rounding against RN(ds q - dm); the
// error stays at the level of rounding w itself.
__device__ __forceinline__ void q4k_half_chunk_to_half(const Q4KChunk &k, const __half2 d2,
                                                       const uint4 &q, uint32_t (&hw)[16]) {
    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bytes (0, 2, 1, 3): weights 4i, 4i+1 in the two 16-bit halves of t,
        // 4i+2, 4i+3 in those of t >> 8
        const uint32_t t = prmt(wd[i], 0u, 0x3120u);
        const uint32_t u = t >> 8;
        const __half2 l01 = u32_as_h2((t & 0x000F000Fu) | 0x64006400u);
        const __half2 l23 = u32_as_h2((u & 0x000F000Fu) | 0x64006400u);
        const __half2 h01 = u32_as_h2((t & 0x00F000F0u) | 0x64006400u);
        const __half2 h23 = u32_as_h2((u & 0x00F000F0u) | 0x64006400u);
        hw[2 * i] = h2_as_u32(__hfma2(__hfma2(l01, k.s0, k.n0), d2, k.e0));
        hw[2 * i + 1] = h2_as_u32(__hfma2(__hfma2(l23, k.s0, k.n0), d2, k.e0));
        hw[8 + 2 * i] = h2_as_u32(__hfma2(__hfma2(h01, k.s1, k.n1), d2, k.e1));
        hw[8 + 2 * i + 1] = h2_as_u32(__hfma2(__hfma2(h23, k.s1, k.n1), d2, k.e1));
    }
}

template <int FMT>
struct Prefetch {
    static constexpr int value = (FMT == F_Q4_K || FMT == F_Q4_0) ? 4
                                 : (FMT == F_Q6_K || FMT == F_BF16 || FMT == F_F16) ? 2 : 3;
};

__device__ __forceinline__ void split_half_words(const float (&v)[32], bool lo, uint32_t (&hw)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        if (!lo) {
            hw[i] = *reinterpret_cast<const uint32_t *>(&h);
        } else {
            const float2 f = __half22float2(h);
            hw[i] = pack_half2(v[2 * i] - f.x, v[2 * i + 1] - f.y);
        }
    }
}

template <int FMT, int BN, int MODE, bool GRP = false>
__global__ void __launch_bounds__(kMmaThreads, 1)
    mma_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmx_lo,
               const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmy,
               const MmaParamsOf<FMT, GRP> p) {
    static_assert(!GRP || (!is_affine(FMT) && MODE == 2), "grouped products: GGUF formats, x split");
    constexpr int kRowsOut = MODE == 3 ? 64 : kBM;   // output rows per CTA
    constexpr int kTokOut = MODE == 1 ? BN : BN / 2;  // tokens per CTA
    constexpr int kSliceB = raw_slice_bytes(FMT, MODE);  // raw W tiles by TMA
    constexpr bool kRaw = kSliceB > 0;                    // decoded from the raw ring
    constexpr bool kSSable = mma_ssable(FMT, MODE, GRP);
    constexpr int kRawB = mma_ring_bytes(FMT, MODE, GRP);  // one slot of the raw ring
    // y through shared memory and tensor stores (the host enables it per call)
    constexpr bool kTmaEpi = mma_tma_epilogue(MODE, GRP);
    constexpr int kEpiB = kTmaEpi ? kEpiStageBytes : 0;
    using C = MmaCfg<BN, kRawB, kEpiB, kSSable>;
    constexpr int NA = C::NA, NB = C::NB, kNR = C::kNR, KA = C::KA, KB = C::KB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
    const uint32_t B0 = sbase;                                     // x ring
    const uint32_t W0 = B0 + NB * C::kBStage;                      // raw W stages (kRaw)
    const uint32_t E0 = W0 + (kRawB > 0 ? kNR * kRawB : 0);         // epilogue staging (kTmaEpi)
    const uint32_t bar0 = E0 + kEpiB;
    auto fullA = [&](int s) { return bar0 + 8u * s; };
    auto emptyA = [&](int s) { return bar0 + 8u * (NA + s); };
    auto fullB = [&](int s) { return bar0 + 8u * (2 * NA + s); };
    auto emptyB = [&](int s) { return bar0 + 8u * (2 * NA + NB + s); };
    auto rawFull = [&](int s) { return bar0 + 8u * (2 * NA + 2 * NB + s); };
    auto rawEmpty = [&](int s) { return bar0 + 8u * (2 * NA + 2 * NB + kNR + s); };
    const uint32_t accFull = bar0 + 8u * (2 * NA + 2 * NB + 2 * kNR);
    const uint32_t accEmpty = accFull + 8u;
    auto xsFull = [&](int b) { return accFull + 8u * (2 + b); };
    auto xsFree = [&](int b) { return accFull + 8u * (4 + b); };
    const uint32_t scrReady = accFull + 8u * 6;  // MODE 3: lo rows parked in scratch
    const uint32_t slot_off = 8u * (2 * NA + 2 * NB + 2 * kNR + 7);
    const uint32_t slot_addr = bar0 + slot_off;
    uint8_t *gen = smem_raw + (bar0 - raw_addr);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gen + slot_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gen + slot_off + 8);
    // token scales of the tile in flight, double-buffered: [2][kTokOut]
    float *xs_s = reinterpret_cast<float *>(gen + 512);
    // Two groups of 8 dequant warps take alternate k-steps; an A stage (KA = 4
    // k-steps) is done when both groups have arrived.
    constexpr int kGroups = 2;
    // raw W tiles: one group fills a whole stage; otherwise both groups
    constexpr int kFullACount = kRaw ? kDeqWarps / kGroups : kDeqWarps;
    static_assert(KA % kGroups == 0, "every group needs a k-step in every A stage");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool ss = kSSable && p.ss != 0;  // A tiles straight from the raw ring
    const uint32_t crank = cluster_ctarank();  // 0 or 1 within the CTA pair
    const int KS = p.KS;                     // 64-wide k-steps
    // Tiles: the pair of CTAs takes 128-row tiles 2q and 2q + 1 of token tile
    // nt together; pair-tile v = q * tiles_n + nt (the token tiles of one W
    // row pair run side by side on neighbouring clusters, so W is read from
    // HBM about once). Units: the first full_units pair-tiles whole, then the
    // rest in split = 2 super-block-aligned k-halves each, so that the last
    // round keeps every cluster busy; the halves add into a y region the
    // conversion kernel zeroed (0 + a + b is the same in either order, so the
    // result does not depend on which half lands first). Cluster c of C takes
    // units c, c + C, ...
    //
    // Grouped products take units expert by expert (unit_off, written by the
    // routing kernel before this grid started): unit u of expert e is row
    // pair q and token tile nt of e's sorted rows, never split.
    const int c0 = (int)(blockIdx.x >> 1), cstep = (int)(gridDim.x >> 1);
    struct Tile {
        int64_t m0;      // first output column (row of W within its slice)
        int64_t wrow;    // first row of W in the stacked weights
        int n0, rot;     // first x row (sorted order for grouped products)
        int tok_end;     // end of this tile's valid x rows
        int k_lo, k_hi;  // k-steps of this unit
        int part;        // k-range index, or -1 for a whole tile
    };
    int n_units = p.n_units;
    if constexpr (GRP) n_units = __ldg(p.unit_off + p.n_experts);
    auto tile_of = [&](int u) {
        int v = u, part = -1;
        int q, nt;
        Tile t;
        if constexpr (GRP) {
            // expert e: the last with unit_off[e] <= u (experts without rows
            // own no units)
            int lo = 0, hi = p.n_experts;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(p.unit_off + mid) <= u) lo = mid; else hi = mid;
            }
            const int r0 = __ldg(p.row_off + lo), r1 = __ldg(p.row_off + lo + 1);
            const int ntile = (r1 - r0 + kTokOut - 1) / kTokOut;
            const int local = u - __ldg(p.unit_off + lo);
            q = local / ntile;
            nt = local - q * ntile;
            t.n0 = r0 + nt * kTokOut;
            t.tok_end = r1;
            t.m0 = p.j0 + (int64_t)(2 * q + (int)crank) * kRowsOut;
            t.wrow = (int64_t)lo * p.slice_rows + t.m0;
        } else {
            if (u >= p.full_units) {
                const int w = u - p.full_units;
                v = p.full_units + w / p.split;
                part = w % p.split;
            }
            q = v / p.tiles_n;
            nt = v - q * p.tiles_n;
            t.n0 = nt * kTokOut;
            t.tok_end = (int)p.n_tokens;
            t.m0 = p.j0 + (int64_t)(2 * q + (int)crank) * kRowsOut;
            t.wrow = t.m0;
        }
        t.part = part;
        if (part < 0) {
            t.k_lo = 0;
            t.k_hi = KS;
            // each whole tile walks k in its own rotated order (whole super-blocks)
            // so that the CTAs do not all fetch the same x tile at the same
            // moment; the sum is the same up to rounding order
            t.rot = (KS % 4 == 0) ? 4 * (q % (KS / 4)) : 0;
        } else {
            const int nsb = (KS + 3) / 4;
            t.k_lo = 4 * (part * nsb / p.split);
            t.k_hi = std::min(KS, 4 * ((part + 1) * nsb / p.split));
            t.rot = 0;
        }
        return t;
    };
    auto kx = [&](const Tile &t, int ks) { return t.rot ? (ks + t.rot) % KS : ks; };
    auto nks = [&](const Tile &t) { return t.k_hi - t.k_lo; };
    // A stages (the last may be padded) and x stages of a unit
    auto nsa = [&](const Tile &t) { return (nks(t) + KA - 1) / KA; };
    auto nsb = [&](const Tile &t) { return (nks(t) + KB - 1) / KB; };

    if (tid == 0) {
        for (int s = 0; s < NA; ++s) {
            mbar_init(fullA(s), kFullACount);
            mbar_init(emptyA(s), 1);
        }
        for (int s = 0; s < NB; ++s) {
            mbar_init(fullB(s), 1);
            mbar_init(emptyB(s), 2);  // both CTAs of the pair have consumed the stage
        }
        for (int s = 0; s < kNR; ++s) {
            mbar_init(rawFull(s), raw_rowcopy(FMT) ? 32 : 1);
            // the group that decodes it, or the MMAs that read it as A
            mbar_init(rawEmpty(s), ss ? 1 : kDeqWarps / kGroups);
        }
        mbar_init(accFull, 1);
        mbar_init(accEmpty, kDeqWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(xsFull(b), 1);
            mbar_init(xsFree(b), kDeqWarps);
        }
        mbar_init(scrReady, kDeqWarps / 2);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(slot_addr, C::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before any multicast reaches them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The next grid in the stream may begin launching now; whatever it reads
    // of this product (y, the workspace) it reads after its griddepcontrol.wait,
    // which returns once this grid has completed (the library's conversion
    // kernel and programmatic GEMVs do so).
    pdl_launch_dependents();

    if (warp == 0) {
        // ------------------ token scales + x tiles via TMA ------------------
        // x16 and the scales come from the conversion kernel just before this
        // one, which lets this grid start early: only this warp waits for it
        pdl_wait_prev();
        if (lane == 0) {
            prefetch_tmap(&tmx);
            if (MODE != 1) prefetch_tmap(&tmx_lo);
        }
        int bcount = 0;  // x stages issued so far (all tiles)
        int it = 0;
        for (int u = c0; u < n_units; u += cstep, ++it) {
            if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
            const Tile t = tile_of(u);
            // the tile's token scales (2^e of each token's fp16 conversion) for
            // its epilogue, into buffer it & 1 once the tile two back is done
            const int xb = it & 1;
            if (it >= 2) {
                const bool ok = wait_abortable(xsFree(xb), ((it >> 1) + 1) & 1, abort_flag);
                if (__all_sync(0xFFFFFFFFu, ok) == 0) {
                    if (lane == 0) { record_error(p.err, DERR_MMA_EMPTY); *abort_flag = 1; }
                    break;
                }
            }
            // the scale loads are issued now and stored after the tile's x
            // stages have gone out (the epilogue needs them only at the end)
            constexpr int kScl = (kTokOut + 31) / 32;
            float scl[kScl];
#pragma unroll
            for (int j = 0; j < kScl; ++j) {
                const int i = lane + 32 * j;
                scl[j] = i < kTokOut && t.n0 + i < t.tok_end ? __ldg(p.xscale + t.n0 + i) : 0.0f;
            }
            if (lane == 0) {
                const int NSB = nsb(t);
                for (int st = 0; st < NSB; ++st, ++bcount) {
                    const int slot = bcount % NB;
                    if (bcount >= NB &&
                        !wait_abortable(emptyB(slot), ((bcount / NB) + 1) & 1, abort_flag)) {
                        record_error(p.err, DERR_MMA_EMPTY);
                        *abort_flag = 1;
                        break;
                    }
                    // the whole stage lands here: this CTA's halves and the peer's halves
                    mbar_arrive_expect_tx(fullB(slot), C::kBStage);
                    for (int sub = 0; sub < KB; ++sub) {
                        // past k_hi: not used; past KS: zero-filled by the map
                        const int ks = t.k_lo + st * KB + sub;
                        const int kc = ks < KS ? kx(t, ks) : ks;
                        // MODE 1: this CTA fetches token rows [n0 + crank BN/2, +BN/2);
                        // MODE 2/3: CTA 0 the hi rows, CTA 1 the lo rows of the tile's tokens
                        const uint32_t dst =
                            B0 + slot * C::kBStage + sub * C::kBBytes + crank * (BN / 2) * 128;
                        if (MODE == 1)
                            tma_load_2d_multicast(dst, &tmx, kc * kBK,
                                                  t.n0 + (int)crank * (BN / 2), fullB(slot),
                                                  (uint16_t)3);
                        else
                            tma_load_2d_multicast(
                                dst, crank ? (const void *)&tmx_lo : (const void *)&tmx, kc * kBK,
                                t.n0, fullB(slot), (uint16_t)3);
                    }
                }
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kScl; ++j)
                if (lane + 32 * j < kTokOut) xs_s[xb * kTokOut + lane + 32 * j] = scl[j];
            __syncwarp();
            if (lane == 0) mbar_arrive(xsFull(xb));
        }
        // no copy may land after this CTA exits
        if (lane == 0)
            for (int s = std::max(0, bcount - NB); s < bcount; ++s)
                if (!mbar_wait(fullB(s % NB), (s / NB) & 1)) record_error(p.err, DERR_TEARDOWN);
    } else if (warp == 1) {
        // ------------------------------ MMA issue ------------------------------
        // One elected lane runs the whole loop: its waits, the MMAs and their
        // commits (the other lanes wait at the end). The loop goes A stage by
        // A stage: an x stage (KB k-steps, KB | KA) starts at a multiple of KB
        // inside it, so every wait and commit sits at a position known at
        // compile time, and ring slots and phases are running counters.
        // Measured at 32 columns (a k-step of 4 MMAs is 64 cycles of tensor
        // work): issuing a k-step takes about 106 cycles this way against 230
        // for a loop that the whole warp ran and converged at every k-step;
        // either way small token tiles are paced by the decode (about 2300
        // cycles per super-block and group, the two groups overlapping).
        constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
        const bool mma_leader = elect_one();  // the whole warp elects once
        if (mma_leader && ss) {
            // A from the raw ring, one k-step a slot: each k-step waits for its
            // W tile (and, at a stage start, its x stage), issues its four
            // K = 16 MMAs and frees the slot
            const uint32_t idesc_ss = FMT == F_BF16 ? idesc_bf16_f32(kBM, BN) : idesc;
            int sr = 0, sb = 0;
            uint32_t phr = 0, phb = 0;
            int it = 0;
            bool failed = false;
            for (int u = c0; u < n_units && !failed; u += cstep, ++it) {
                const Tile t = tile_of(u);
                const int KSu = nks(t);
                if (it > 0) {  // the epilogue has drained the accumulator
                    if (!wait_abortable(accEmpty, (it - 1) & 1, abort_flag)) {
                        record_error(p.err, DERR_MMA_ACC);
                        *abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                }
                for (int ks = 0; ks < KSu; ++ks) {
                    if (!wait_abortable(rawFull(sr), phr, abort_flag)) {
                        record_error(p.err, DERR_MMA_A);
                        *abort_flag = 1;
                        failed = true;
                        break;
                    }
                    if (ks % KB == 0 && !wait_abortable(fullB(sb), phb, abort_flag)) {
                        record_error(p.err, DERR_MMA_B);
                        *abort_flag = 1;
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const bool last = ks == KSu - 1;
                    const uint64_t ad = sdesc_sw128(W0 + sr * kRawB);
                    const uint64_t bd = sdesc_sw128(B0 + sb * C::kBStage + (ks % KB) * C::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)  // K = 16: 32 bytes of A and of B
                        tc_mma_f16_ss(tmem, ad + 2 * kk, bd + 2 * kk, idesc_ss, ks > 0 || kk > 0);
                    tc_commit(rawEmpty(sr));
                    if (++sr == kNR) { sr = 0; phr ^= 1u; }
                    if (ks % KB == KB - 1 || last) {
                        tc_commit_multicast(emptyB(sb), (uint16_t)3);  // both CTAs may refill
                        if (++sb == NB) { sb = 0; phb ^= 1u; }
                    }
                    if (last) tc_commit(accFull);  // the tile's product is complete
                }
            }
        } else if (mma_leader) {
            int sa = 0, sb = 0;        // A / x ring slots
            uint32_t pha = 0, phb = 0; // their phase parities
            int it = 0;
            bool failed = false;
            for (int u = c0; u < n_units && !failed; u += cstep, ++it) {
                const Tile t = tile_of(u);
                const int KSu = nks(t);
                if (it > 0) {  // the epilogue has drained the accumulator
                    if (!wait_abortable(accEmpty, (it - 1) & 1, abort_flag)) {
                        record_error(p.err, DERR_MMA_ACC);
                        *abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                }
                for (int ks0 = 0; ks0 < KSu; ks0 += KA) {
                    if (!wait_abortable(fullA(sa), pha, abort_flag)) {
                        record_error(p.err, DERR_MMA_A);
                        *abort_flag = 1;
                        failed = true;
                        break;
                    }
                    const uint32_t at0 = tmem + (uint32_t)(C::kACol0 + sa * C::kAStageCols);
#pragma unroll
                    for (int j = 0; j < KA; ++j) {
                        const int ks = ks0 + j;
                        if (ks >= KSu) break;  // a padded last A stage
                        if (j % KB == 0 && !wait_abortable(fullB(sb), phb, abort_flag)) {
                            record_error(p.err, DERR_MMA_B);
                            *abort_flag = 1;
                            failed = true;
                            break;
                        }
                        // order the MMAs after this stage's barrier waits
                        if (j % KB == 0) tc_fence_after();
                        const bool last = ks == KSu - 1;
                        const uint64_t bd = sdesc_sw128(B0 + sb * C::kBStage + (j % KB) * C::kBBytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {  // K = 16: 8 A columns, 32 B bytes
                            // K step kk goes to accumulator kk % kNAcc; the tile's
                            // first MMA into each accumulator overwrites it
                            const int a = kk % C::kNAcc;
                            tc_mma_f16_ts(tmem + (uint32_t)(a * C::kAccCols), at0 + 32 * j + 8 * kk,
                                          bd + 2 * kk, idesc, ks > 0 || kk >= C::kNAcc);
                        }
                        if (j % KB == KB - 1 || last) {
                            tc_commit_multicast(emptyB(sb), (uint16_t)3);  // both CTAs may refill
                            if (++sb == NB) { sb = 0; phb ^= 1u; }
                        }
                        if (j == KA - 1 || last) tc_commit(emptyA(sa));
                        if (last) tc_commit(accFull);  // the tile's product is complete
                    }
                    if (failed) break;
                    if (++sa == NA) { sa = 0; pha ^= 1u; }
                }
            }
        }
        __syncwarp();
    } else if (warp == kRawWarp) {
        // ------------------------- raw W tiles (Q4_K, affine codes) via TMA -------------------------
        // its own warp, so that the raw ring runs as far ahead of the dequant
        // warps as it is deep (into the next tile), whatever the x ring does
        if (ss) {
            // 16-bit W: one 128-row x 64-wide tile a k-step, in the order the
            // MMA lane consumes them
            if (lane == 0) {
                prefetch_tmap(&tmw);
                int rcount = 0;
                for (int u = c0; u < n_units; u += cstep) {
                    if (*abort_flag) break;
                    const Tile t = tile_of(u);
                    bool ok = true;
                    for (int ks = t.k_lo; ks < t.k_hi; ++ks, ++rcount) {
                        const int rs = rcount % kNR;
                        if (rcount >= kNR &&
                            !wait_abortable(rawEmpty(rs), ((rcount / kNR) + 1) & 1, abort_flag)) {
                            record_error(p.err, DERR_MMA_EMPTY);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(rawFull(rs), kRawB);
                        tma_load_2d(W0 + rs * kRawB, &tmw, kBK * kx(t, ks), (int)t.wrow, rawFull(rs));
                    }
                    if (!ok) break;
                }
                // no copy may land after this CTA exits
                for (int s = std::max(0, rcount - kNR); s < rcount; ++s)
                    if (!mbar_wait(rawFull(s % kNR), (s / kNR) & 1)) record_error(p.err, DERR_TEARDOWN);
            }
        } else if (kRaw && raw_rowcopy(FMT)) {
            // Q6_K: lane l copies 16-byte chunks l, l + 32, ... of the slot,
            // chunk c = 14 r + q being bytes 16 q .. 16 q + 15 of row r's
            // window, which starts at (w + j R + 210 sb) & ~15 for row j of W.
            // Rows past the matrix and bytes past the end of W are zero-filled.
            // (One 1-D bulk copy a row kept the tensor-copy unit so busy that
            // a tile took about 1.35x as long.)
            constexpr int kCh = kQ6kWindow / 16;
            constexpr int kPerLane = kBM * kCh / 32;
            constexpr int kDr = 32 / kCh, kDq = 32 % kCh;  // (r, q) step of c + 32
            static_assert(kBM * kCh % 32 == 0 && kCh <= 32, "chunks per lane");
            const uintptr_t wbase = reinterpret_cast<uintptr_t>(p.w);
            const uintptr_t wend = wbase + (uintptr_t)(p.row_bytes * p.w_rows);
            const uintptr_t R = (uintptr_t)p.row_bytes;
            int rcount = 0;
            for (int u = c0; u < n_units; u += cstep) {
                if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
                const Tile t = tile_of(u);
                const int rows_ok = (int)std::min<int64_t>(kBM, p.w_rows - t.wrow);
                bool ok = true;
                for (int b = t.k_lo / 4; b < t.k_hi / 4; ++b, ++rcount) {  // k % 256 == 0
                    const int rs = rcount % kNR;
                    bool free_ok = true;
                    if (lane == 0 && rcount >= kNR)
                        free_ok = wait_abortable(rawEmpty(rs), ((rcount / kNR) + 1) & 1, abort_flag);
                    if (!__shfl_sync(0xFFFFFFFFu, (int)free_ok, 0)) {
                        if (lane == 0) {
                            record_error(p.err, DERR_MMA_EMPTY);
                            *abort_flag = 1;
                        }
                        ok = false;
                        break;
                    }
                    const int64_t sbg = kx(t, 4 * b) >> 2;  // super-block index along the row
                    const uint32_t slot = W0 + rs * kRawB;
                    int r = lane / kCh, q = lane - (lane / kCh) * kCh;
                    uintptr_t rb = wbase + (uintptr_t)((t.wrow + r) * p.row_bytes) + (uintptr_t)(210 * sbg);
#pragma unroll 4
                    for (int i = 0; i < kPerLane; ++i) {
                        const uintptr_t a = (rb & ~(uintptr_t)15) + 16u * (uint32_t)q;
                        uintptr_t src = wbase;  // nothing is read for a zero-filled chunk
                        uint32_t valid = 0;
                        if (r < rows_ok && a < wend) {
                            src = a;
                            valid = wend - a < 16 ? (uint32_t)(wend - a) : 16u;
                        }
                        cp_async16(slot + (uint32_t)(r * kSliceB + 16 * q),
                                   reinterpret_cast<const void *>(src), valid);
                        r += kDr;
                        q += kDq;
                        rb += kDr * R;
                        if (q >= kCh) {
                            q -= kCh;
                            ++r;
                            rb += R;
                        }
                    }
                    cp_async_arrive(rawFull(rs));
                }
                if (!ok) break;
            }
            // no copy may land after this CTA exits
            if (lane == 0)
                for (int s = std::max(0, rcount - kNR); s < rcount; ++s)
                    if (!mbar_wait(rawFull(s % kNR), (s / kNR) & 1)) record_error(p.err, DERR_TEARDOWN);
        } else if (kRaw && lane == 0) {
            prefetch_tmap(&tmw);
            int rcount = 0;
            for (int u = c0; u < n_units; u += cstep) {
                if (*abort_flag) break;
                const Tile t = tile_of(u);
                bool ok = true;
                for (int b = t.k_lo / 4; b < t.k_hi / 4; ++b, ++rcount) {  // k % 256 == 0
                    const int rs = rcount % kNR;
                    if (rcount >= kNR &&
                        !wait_abortable(rawEmpty(rs), ((rcount / kNR) + 1) & 1, abort_flag)) {
                        record_error(p.err, DERR_MMA_EMPTY);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    // boxes of at most 128 bytes a row when swizzled (8-bit
                    // affine rows take two)
                    constexpr int kBoxes = FMT == F_AFF8 ? 2 : 1;
                    mbar_arrive_expect_tx(rawFull(rs), kRawB);
#pragma unroll
                    for (int bx = 0; bx < kBoxes; ++bx)
                        tma_load_2d(W0 + rs * kRawB + (uint32_t)bx * (kRawB / kBoxes), &tmw,
                                    (kSliceB * (kx(t, 4 * b) >> 2) + bx * (kSliceB / kBoxes)) /
                                        raw_elem_bytes(FMT),
                                    (int)t.wrow, rawFull(rs));
                }
                if (!ok) break;
            }
            // no copy may land after this CTA exits
            for (int s = std::max(0, rcount - kNR); s < rcount; ++s)
                if (!mbar_wait(rawFull(s % kNR), (s / kNR) & 1)) record_error(p.err, DERR_TEARDOWN);
        }
    } else {
        // ------------------------------ W dequant producers ------------------------------
        // Warp w (2..17) owns TMEM lanes 32 (w % 4) .. +31, i.e. rows r of the
        // tile; (w - 2) / 4 picks the half h of each 64-wide k-step and the
        // group g (k-step parity) it takes. Each group's first k-step in a
        // stage waits for the stage to be free, its last one signals it.
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;
        const int dq = (warp - 2) >> 2;
        const int h = dq & 1;
        const int g = dq >> 1;
        const uint32_t tlane = tmem + ((uint32_t)(32 * quarter) << 16);
        bool failed = false;
        int abase = 0;   // A stages of earlier tiles
        int rcount = 0;  // raw super-blocks consumed (all tiles)
        // k-step ks of the tile: wait for its A slot (when first in the stage)
        // and return the TMEM address of its 32 columns
        auto a_slot = [&](int ks) {
            const int st = abase + ks / KA, sub = ks % KA;
            const int slot = st % NA;
            if (sub < kGroups && st >= NA) {
                const bool ok = wait_abortable(emptyA(slot), ((st / NA) + 1) & 1, abort_flag);
                if (__all_sync(0xFFFFFFFFu, ok) == 0) {
                    if (!failed) record_error(p.err, DERR_MMA_EMPTY);
                    failed = true;
                    *abort_flag = 1;
                }
                tc_fence_after();  // the MMAs that read the slot are done
            }
            return tlane + (uint32_t)(C::kACol0 + slot * C::kAStageCols + sub * 32);
        };
        auto a_done = [&](int ks) {
            const int st = abase + ks / KA, sub = ks % KA;
            if (sub + kGroups >= KA) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && !failed) mbar_arrive(fullA(st % NA));
            }
        };
        int it = 0;
        for (int u = c0; u < n_units && !failed; u += cstep, ++it) {
            const Tile t = tile_of(u);
            const int KSu = nks(t);
            // ss: the A operand is the raw ring itself, nothing to decode
            if (!ss) {
            if constexpr (kRaw) {
                // Super-block b is one A stage. Group g takes the super-blocks
                // whose global index has parity g, so the two groups run out of
                // phase: thread (r, h) decodes half h of all four 64-weight
                // chunks of row r.
                const bool row_ok = t.m0 + r < p.j1;
                const int NSBLK = KSu / 4;  // k % 256 == 0: whole super-blocks
                const int rbase = rcount;   // global index of the unit's first super-block
                for (int b = (g - rbase) & 1; b < NSBLK && !failed; b += 2) {
                    const int rc = rbase + b;
                    const int rs = rc % kNR;
                    // affine: the row's four scales and biases of this slice come
                    // from global memory; their loads overlap the raw-tile wait
                    uint2 sc4 = make_uint2(0u, 0u), bi4 = make_uint2(0u, 0u);
                    if constexpr (is_affine(FMT)) {
                        if (row_ok) {
                            // the unit's super-block b is k-step t.k_lo + 4 b (before rotation)
                            const int64_t ao = (t.wrow + r) * p.aux_row_bytes +
                                               8 * (kx(t, t.k_lo + 4 * b) >> 2);
                            sc4 = __ldg(reinterpret_cast<const uint2 *>(p.sc + ao));
                            bi4 = __ldg(reinterpret_cast<const uint2 *>(p.bi + ao));
                        }
                    }
                    // Q6_K: where this row's super-block starts in its tile row
                    // (its global address modulo 16, as the loader cut it)
                    uint32_t q6_rem = 0;
                    if constexpr (raw_rowcopy(FMT)) {
                        const int64_t sbg = kx(t, t.k_lo + 4 * b) >> 2;
                        q6_rem = (uint32_t)((reinterpret_cast<uintptr_t>(p.w) +
                                             (uintptr_t)((t.wrow + r) * p.row_bytes + 210 * sbg)) &
                                            15u);
                    }
                    const bool ok = wait_abortable(rawFull(rs), (rc / kNR) & 1, abort_flag);
                    if (__all_sync(0xFFFFFFFFu, ok) == 0) {
                        record_error(p.err, DERR_MMA_A);
                        failed = true;
                        *abort_flag = 1;
                        break;
                    }
                    // Q4_K: the super-block header and this half of each chunk;
                    // affine: this half of each k-step's codes (128-byte swizzled
                    // rows: 16-byte chunk q of row r sits at chunk q ^ (r & 7) of
                    // its 128-byte line)
                    // Rows past j1 are decoded like the others (their raw bytes
                    // are in the tile, rows past the matrix being the map's zero
                    // fill; affine scales and biases past j1 stay 0): the
                    // accumulator rows they feed are never stored.
                    uint4 hdr, qv[4], qv2[4];
                    if constexpr (FMT == F_Q4_K) {
                        const uint32_t rb = W0 + rs * kRawB + (uint32_t)r * 144u;
                        hdr = lds128(rb);
#pragma unroll
                        for (int c = 0; c < 4; ++c) qv[c] = lds128(rb + 16u + 32u * c + 16u * h);
                    } else if constexpr (raw_block32(FMT) || raw_rowcopy(FMT)) {
                        // read block by block during the decode below; the raw
                        // slot is released after it
                    } else {
                        const uint32_t sw = (uint32_t)(r & 7);
                        {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                if (FMT == F_AFF4) {
                                    const uint32_t rb = W0 + rs * kRawB + (uint32_t)r * 128u;
                                    qv[c] = lds128(rb + 16u * (((uint32_t)(2 * c + h)) ^ sw));
                                } else {
                                    // 256-byte rows as two 128-byte sub-tiles
                                    const uint32_t rb = W0 + rs * kRawB + (uint32_t)(c >> 1) * (kBM * 128u) +
                                                        (uint32_t)r * 128u;
                                    const uint32_t q0 = (uint32_t)(4 * (c & 1) + 2 * h);
                                    qv[c] = lds128(rb + 16u * (q0 ^ sw));
                                    qv2[c] = lds128(rb + 16u * ((q0 + 1u) ^ sw));
                                }
                            }
                        }
                    }
                    // the raw slot is refilled by TMA (the async proxy) once every
                    // reader has arrived: order this thread's reads of it first
                    if constexpr (!raw_block32(FMT) && !raw_rowcopy(FMT)) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rawEmpty(rs));  // raw tile read
                    }
                    // the stage's slot, once the MMAs that read it last are done
                    const int st = abase + b, slot = st % NA;
                    if (st >= NA) {
                        const bool ok2 =
                            wait_abortable(emptyA(slot), ((st / NA) + 1) & 1, abort_flag);
                        if (__all_sync(0xFFFFFFFFu, ok2) == 0) {
                            record_error(p.err, DERR_MMA_EMPTY);
                            failed = true;
                            *abort_flag = 1;
                        }
                        tc_fence_after();
                    }
                    const uint32_t ta = tlane + (uint32_t)(C::kACol0 + slot * C::kAStageCols);
                    Q4KChunk kc[4];
                    __half2 d2;
                    if constexpr (FMT == F_Q4_K) q4k_superblock_consts(hdr, d2, kc);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t hw[16];
                        if constexpr (FMT == F_Q4_K) {
                            q4k_half_chunk_to_half(kc[c], d2, qv[c], hw);
                        } else if constexpr (raw_block32(FMT)) {
                            // chunk c = blocks 2c and 2c + 1 of the slice; this
                            // thread's half is block 2c + h (weights 32h + 0..31)
                            Raw32<FMT> ra;
                            ra.load_shared(W0 + rs * kRawB + (uint32_t)r * (uint32_t)kSliceB +
                                           (uint32_t)(2 * c + h) * (uint32_t)(kSliceB / 8));
                            to_half_words<FMT>(ra, hw);
                        } else if constexpr (raw_rowcopy(FMT)) {
                            // this row's super-block starts q6_rem bytes into its
                            // tile row; weights 64c + 32h + 0..31 of it
                            Raw32<FMT> ra;
                            ra.load_shared(W0 + rs * kRawB + (uint32_t)r * (uint32_t)kSliceB + q6_rem,
                                           64 * c + 32 * h);
                            to_half_words<FMT>(ra, hw);
                        } else {
                            Raw32<FMT> ra;
                            ra.qw[0] = qv[c].x; ra.qw[1] = qv[c].y; ra.qw[2] = qv[c].z; ra.qw[3] = qv[c].w;
                            if constexpr (FMT == F_AFF8) {
                                ra.qw[4] = qv2[c].x; ra.qw[5] = qv2[c].y;
                                ra.qw[6] = qv2[c].z; ra.qw[7] = qv2[c].w;
                            }
                            ra.sbits = ((c < 2 ? sc4.x : sc4.y) >> (16 * (c & 1))) & 0xFFFFu;
                            ra.bbits = ((c < 2 ? bi4.x : bi4.y) >> (16 * (c & 1))) & 0xFFFFu;
                            to_half_words<FMT>(ra, hw);
                        }
                        if constexpr (FMT == F_Q4_K) {
                            // chunk c = k-step c of the stage: weights 16h + 0..15 ->
                            // columns 8h..8h+7, 32 + 16h + 0..15 -> 16 + 8h..
                            tmem_st8(ta + 32u * c + 8u * h, hw);
                            tmem_st8(ta + 32u * c + 16u + 8u * h, hw + 8);
                        } else {
                            // k-step c, weights 32h + 0..31 -> columns 16h..
                            tmem_st16(ta + 32u * c + 16u * h, hw);
                        }
                    }
                    if constexpr (raw_block32(FMT) || raw_rowcopy(FMT)) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rawEmpty(rs));  // raw tile read
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0 && !failed) mbar_arrive(fullA(slot));
                }
                rcount = rbase + NSBLK;
            } else {
                const bool lo_part = MODE == 3 && r >= 64;  // MODE 3: rows 64..127 hold W_lo
                const int64_t rj = MODE == 3 ? (r & 63) : r;
                const int64_t j = t.m0 + rj;
                const bool row_ok = j < p.j1;
                const uint8_t *rowp = p.w + (row_ok ? t.wrow + rj : 0) * p.row_bytes;
                // 32 weights of this row at k0 (affine: with the group's scale and bias)
                auto load_raw = [&](Raw32<FMT> &r, int64_t k0, int nv) {
                    if constexpr (is_affine(FMT)) {
                        const int64_t ao = (row_ok ? t.wrow + rj : 0) * p.aux_row_bytes;
                        r.load(rowp, p.sc + ao, p.bi + ao, k0);
                    } else {
                        r.load(rowp, k0, nv);
                    }
                };
                constexpr int PD = Prefetch<FMT>::value;
                Raw32<FMT> ring[PD];
                // this thread's i-th k-step is g + 2 i
                auto ks_of = [&](int i) { return g + 2 * i; };
                // unit-relative k-step -> first weight index; past the unit's
                // range: beyond k (nothing loaded, zeros stored)
                auto k0_of = [&](int i) {
                    const int ks = t.k_lo + ks_of(i);
                    return ks < t.k_hi ? (int64_t)kx(t, ks) * kBK + 32 * h : p.k;
                };
                auto nvalid_of = [&](int64_t k0) {
                    const int64_t v = p.k - k0;
                    return (int)(v < 0 ? 0 : (v > 32 ? 32 : v));
                };
                // k-steps of this group over the stage-padded range: a k-step
                // past k stores zeros (the MMA skips it) but still takes part
                // in its stage's arrival count
                const int NI = (nsa(t) * KA - g + 1) / 2;
#pragma unroll
                for (int q = 0; q < PD; ++q) {
                    const int64_t k0 = k0_of(q);
                    const int nv = nvalid_of(k0);
                    if (q < NI && row_ok && nv > 0) load_raw(ring[q], k0, nv);
                }
                for (int i0 = 0; i0 < NI && !failed; i0 += PD) {
#pragma unroll
                    for (int q = 0; q < PD; ++q) {
                        const int i = i0 + q;
                        if (i < NI) {
                            const int ks = ks_of(i);
                            const int64_t k0 = k0_of(i);
                            const int nv = nvalid_of(k0);
                            uint32_t hw[16];
                            if (row_ok && nv > 0) {
                                if (MODE == 3) {
                                    float v[32];
                                    ring[q].decode(v);
                                    split_half_words(v, lo_part, hw);
                                } else {
                                    to_half_words<FMT>(ring[q], hw);
                                }
                                if (nv < 32) {
#pragma unroll
                                    for (int e = 0; e < 16; ++e)
                                        if (2 * e >= nv) hw[e] = 0u;  // nv is even
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 16; ++e) hw[e] = 0u;
                            }
                            const int64_t kn = k0_of(i + PD);
                            const int nvn = nvalid_of(kn);
                            if (i + PD < NI && row_ok && nvn > 0) load_raw(ring[q], kn, nvn);
                            const uint32_t ta = a_slot(ks);
                            tmem_st16(ta + 16u * h, hw);  // weights 32h + 0..31 -> columns 16h..
                            a_done(ks);
                        }
                    }
                }
            }
            }  // !ss
            abase += nsa(t);
            if (failed) break;
            // ------------------------------ epilogue ------------------------------
            // TMEM -> registers -> y: per warp store, 32 consecutive rows of one
            // token (128 contiguous bytes)
            const int xb = it & 1;
            const bool acc_ok = mbar_wait(accFull, it & 1) && mbar_wait(xsFull(xb), (it >> 1) & 1);
            if (!acc_ok) {
                record_error(p.err, DERR_MMA_ACC);
                *abort_flag = 1;
                failed = true;
                break;
            }
            tc_fence_after();
            const float *xsc = xs_s + xb * kTokOut;
            const int slice = dq;  // 0..3: which part of the token columns
            constexpr int kSlices = kTokOut >= 64 ? 4 : (kTokOut >= 32 ? 2 : 1);
            constexpr int kSliceCols = kTokOut / kSlices;
            const int c_lo = slice < kSlices ? slice * kSliceCols : 0;
            const int c_hi = slice < kSlices ? c_lo + kSliceCols : 0;
            const int64_t je = t.m0 + (MODE == 3 ? (r & 63) : r);
            const bool store_ok = !*abort_flag && je < p.j1;
            // the k-halves of a split tile add into zeros
            const bool split = t.part >= 0;
            if (split) pdl_wait_prev();  // the conversion kernel zeroed the region
            // MODE 3 row-pair scratch [col][64] over the x ring (MODE 3 CTAs
            // take one tile each: nothing is prefetched into the ring)
            float *scratch = reinterpret_cast<float *>(smem_raw + (B0 - raw_addr));
            // the accumulators are summed here (every one was written: a
            // k-step has four K steps); one accumulator's hi and lo columns at
            // a time, 32 registers live
            auto load_acc = [&](int col, float (&acc)[16]) {
#pragma unroll
                for (int a = 0; a < C::kNAcc; ++a) {
                    uint32_t v[16], v2[16];
                    const uint32_t base = tlane + (uint32_t)(a * C::kAccCols + col);
                    tmem_ld16(base, v);
                    if (MODE != 1) tmem_ld16(base + (uint32_t)(BN / 2), v2);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float d = MODE != 1 ? __uint_as_float(v[i]) + __uint_as_float(v2[i])
                                                  : __uint_as_float(v[i]);
                        acc[i] = a == 0 ? d : acc[i] + d;
                    }
                }
            };
            if (MODE == 3 && quarter >= 2) {
                // lo rows: park (D[r][c] + D[r][c + BN/2]) for the hi warps
                for (int col = c_lo; col < c_hi; col += 16) {
                    float acc[16];
                    load_acc(col, acc);
#pragma unroll
                    for (int i = 0; i < 16; ++i) scratch[(col + i) * 64 + (r & 63)] = acc[i];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(scrReady);
            }
            bool scr_ok = true;
            if (MODE == 3 && quarter < 2) {
                scr_ok = mbar_wait(scrReady, 0);  // one tile per CTA in MODE 3
                if (!scr_ok) {
                    record_error(p.err, DERR_MMA_ACC);
                    *abort_flag = 1;
                }
            }
            if (kTmaEpi && p.tma_epi) {
                // each warp: its 32 rows x 16 tokens through its 2 KB staging
                // area (token-major: the layout of y) and one tensor store (or
                // add); the stores run on while the warps decode the next
                // tile. Tokens past n_tokens and columns past j1 fall outside
                // the tensor map and are not written.
                const uint32_t ereg = E0 + (uint32_t)(warp - 2) * 2048u;
                const bool add = p.accumulate || split;
                for (int col = c_lo; col < c_hi; col += 16) {
                    float acc[16];
                    load_acc(col, acc);
                    if (p.glu) {
                        // gated pair: y (+)= act(gate) * (this product); the
                        // gate values of rows and tokens outside the tile are
                        // not read (the tensor store drops those elements)
                        // all 16 loads are issued before any is used
                        float gv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int64_t tt = t.n0 + col + i;
                            gv[i] = tt < t.tok_end && je < p.j1 ? __ldg(p.gate + tt * p.n + je) : 0.0f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[i] *= glu_gate(gv[i], glu_arg(p.glu, gv[i]));
                    }
                    if (lane == 0) bulk_wait_group_read0();  // the area's last store has read it
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        sts32f(ereg + (uint32_t)(128 * i + 4 * lane), acc[i] * xsc[col + i]);
                    fence_proxy_async_smem();  // visible to the tensor store
                    __syncwarp();
                    if (lane == 0 && !*abort_flag) {
                        const int cx = (int)(t.m0 + 32 * quarter), cy = t.n0 + col;
                        if (add)
                            tma_reduce_add_2d(&tmy, cx, cy, ereg);
                        else
                            tma_store_2d(&tmy, cx, cy, ereg);
                        bulk_commit_group();
                    }
                }
            } else if ((MODE != 3 || quarter < 2) && scr_ok) {
                for (int col = c_lo; col < c_hi; col += 16) {
                    float acc[16];
                    load_acc(col, acc);
                    if (MODE == 3) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[i] += scratch[(col + i) * 64 + (r & 63)];
                    }
                    if (store_ok) {
                        const int64_t t0 = t.n0 + col;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (t0 + i < t.tok_end) {
                                float val = acc[i] * xsc[col + i];
                                // grouped products: sorted x row -> its y row
                                int64_t yrow = t0 + i;
                                if constexpr (GRP) yrow = __ldg(p.perm + t0 + i);
                                if (p.glu) {
                                    // act(g) u is linear in u: split k-halves add their share
                                    const float g = __ldg(p.gate + yrow * p.n + je);
                                    val *= glu_gate(g, glu_arg(p.glu, g));
                                }
                                float *yq = p.y + yrow * p.n + je;
                                if (split)
                                    atomicAdd(yq, val);
                                else
                                    *yq = p.accumulate ? *yq + val : val;
                            }
                        }
                    }
                }
            }
            // accumulator and token scales free for the next tile
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(accEmpty);
                mbar_arrive(xsFree(xb));
            }
        }
        // this warp's tensor stores of y complete before the CTA exits
        if (kTmaEpi && p.tma_epi && lane == 0) bulk_wait_group0();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no multicast or remote arrival is still headed for this CTA
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kCols);
    }
}

struct Maps {
    CUtensorMap x, xlo, w, y;
};

// Clusters of two CTAs that can be resident at once (defined beside the Q4_K
// instances, whose footprint it queries).
int mma_clusters(const DeviceInfo &dev);

// Persistent grid: clusters of two CTAs, as many as can be resident at once
// (one CTA per SM), capped by the number of row-tile pairs x token tiles.
// MODE 3 keeps one tile per CTA (its epilogue scratch lives in the x ring).
template <int FMT, int BN, int MODE, bool GRP = false>
static cudaError_t launch_t(const Maps &mp, const MmaHostParams &h, const DeviceInfo &dev,
                            cudaStream_t s) {
    MmaParamsOf<FMT, GRP> p;
    if constexpr (GRP) {
        static_cast<MmaParams &>(p) = static_cast<const MmaParams &>(h);
        static_cast<MmaGrpFields &>(p) = static_cast<const MmaGrpFields &>(h);
    } else {
        p = static_cast<const MmaParamsOf<FMT> &>(static_cast<const MmaAffParams &>(h));
    }
    using C = MmaCfg<BN, mma_ring_bytes(FMT, MODE, GRP),
                     mma_tma_epilogue(MODE, GRP) ? kEpiStageBytes : 0, mma_ssable(FMT, MODE, GRP)>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int max_clusters = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(mma_kernel<FMT, BN, MODE, GRP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
        if (attr_err != cudaSuccess) return;
        cudaLaunchConfig_t q = cfg;
        q.gridDim = dim3(2 * (unsigned)(dev.sm_count / 2));
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mma_kernel<FMT, BN, MODE, GRP>, &q) != cudaSuccess ||
            n <= 0) {
            (void)cudaGetLastError();
            n = dev.sm_count / 2;
        }
        max_clusters = std::min(n, mma_clusters(dev));
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int P = p.pairs * p.tiles_n;
    // grouped products: n_units is an upper bound (the routed count is on the device)
    const int clusters = MODE == 3 ? P : std::min(p.n_units, max_clusters);
    cfg.gridDim = dim3(2 * (unsigned)clusters);
    // programmatic launch after the x conversion kernel (see pdl_wait_prev)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, mma_kernel<FMT, BN, MODE, GRP>, mp.x, mp.xlo, mp.w, mp.y, p);
}

template <int FMT, int MODE, bool GRP = false>
static cudaError_t launch_bn(int bn, const Maps &mp, const MmaHostParams &p, const DeviceInfo &dev,
                             cudaStream_t s) {
    switch (bn) {
    case 16:
        if constexpr (MODE == 1) return launch_t<FMT, 16, MODE, GRP>(mp, p, dev, s);
        break;
    case 32: return launch_t<FMT, 32, MODE, GRP>(mp, p, dev, s);
    case 64: return launch_t<FMT, 64, MODE, GRP>(mp, p, dev, s);
    case 128: return launch_t<FMT, 128, MODE, GRP>(mp, p, dev, s);
    case 256: return launch_t<FMT, 256, MODE, GRP>(mp, p, dev, s);
    default: break;
    }
    return cudaErrorInvalidValue;
}

// Instantiated (explicitly) by the qmm_mma_inst_*.cu units, one group of
// formats each.
template <int FMT>
cudaError_t launch_fmt(int mode, int bn, const Maps &mp, const MmaHostParams &p,
                       const DeviceInfo &dev, cudaStream_t s) {
    constexpr bool quant = FMT != F_BF16 && FMT != F_F16;
    if (mode == 2) return launch_bn<FMT, 2>(bn, mp, p, dev, s);
    if (quant && mode == 3) return launch_bn<FMT, quant ? 3 : 2>(bn, mp, p, dev, s);
    return cudaErrorInvalidValue;
}

// The expert-grouped instances (split x only), in units of their own.
template <int FMT>
cudaError_t launch_fmt_grouped(int bn, const Maps &mp, const MmaHostParams &p,
                               const DeviceInfo &dev, cudaStream_t s) {
    if constexpr (is_affine(FMT)) {
        return cudaErrorNotSupported;
    } else {
        return launch_bn<FMT, 2, true>(bn, mp, p, dev, s);
    }
}

#define QMM_MMA_INSTANTIATE(F)                                                               \
    template cudaError_t launch_fmt<F>(int, int, const Maps &, const MmaHostParams &,         \
                                       const DeviceInfo &, cudaStream_t)
#define QMM_MMA_INSTANTIATE_GROUPED(F)                                                       \
    template cudaError_t launch_fmt_grouped<F>(int, const Maps &, const MmaHostParams &,      \
                                               const DeviceInfo &, cudaStream_t)

}  // namespace qmm
