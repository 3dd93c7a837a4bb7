// qmm_decode.cuh -- element-exact decoding of 32 consecutive weights of one
// packed row, straight from global memory. Used by the standalone dequant
// kernel and by the weight producers of the tensor-core path.
//
// Values are bit-identical to "the exact value rounded once to fp32":
// every product below is exact in fp32 (Q4_0: 4+11 bits; Q6_K: 11+8+6 bits;
// Q4_K: d*sc and dmin*m are 17-bit products), so only Q4_K's final
// d*sc*q - dmin*m rounds, and it does so once inside an explicit fma.
//
// Layouts (little-endian; block sizes from the rullama matmul.rs dispatchers,
// field order inside K-quant blocks from the standard ggml layout):
//   BF16 / F16: 2 bytes per weight.
//   Q4_0  (32 w, 18 B): f16 d | 16 bytes; weight i < 16 = low nibble of byte i,
//                       weight i + 16 = its high nibble; w = (q - 8) * d.
//   Q4_K (256 w, 144 B): f16 d | f16 dmin | 12 bytes of 6-bit scales and mins
//                       | 128 nibble bytes; weights 64c..64c+31 are the low
//                       nibbles of bytes 32c..32c+31, 64c+32..64c+63 their high
//                       nibbles; sub-block s = weight / 32; w = d*sc_s*q - dmin*m_s.
//   Q8_0  (32 w, 34 B): f16 d | 32 signed bytes q; w = q * d.
//   Q5_0  (32 w, 22 B): f16 d | u32 qh | 16 bytes; weight i < 16 = low nibble of
//                       byte i with bit i of qh as bit 4, weight i + 16 = its
//                       high nibble with bit i + 16 of qh; w = (q - 16) * d.
//   AFF4 / AFF8 (MLX-style affine, groups of 64): three arrays per matrix --
//                       codes in little-endian u32 words (8 four-bit or 4
//                       eight-bit codes per word, lowest bits first), a bf16
//                       scale and a bf16 bias per group ([n][k/64] each);
//                       w = fma(q, scale, bias) (q * scale is exact in fp32).
//   Q6_K (256 w, 210 B): ql[128] | qh[64] | int8 scales[16] | f16 d; for half h and
//                       l < 32, weight 128h + 32r + l takes nibble (r < 2: low,
//                       else high) of ql[64h + 32(r & 1) + l] and bits 2r..2r+1 of
//                       qh[32h + l] as its top two bits; w = d * scales[w/16] * (q - 32).
#pragma once

#include "qmm_device.cuh"

namespace qmm {

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned short *>(p));
}
__device__ __forceinline__ uint32_t ldg_u32(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}
__device__ __forceinline__ uint4 ldg_u128(const uint8_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// 6-bit scale and min of sub-block s (0..7) from the 12 packed bytes held in
// three little-endian words s0 (bytes 0..3), s1 (4..7), s2 (8..11).
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int s,
                                              uint32_t &sc, uint32_t &m) {
    if (s < 4) {
        sc = (s0 >> (8 * s)) & 63u;
        m = (s1 >> (8 * s)) & 63u;
    } else {
        const int t = s - 4;
        sc = ((s2 >> (8 * t)) & 15u) | (((s0 >> (8 * t + 6)) & 3u) << 4);
        m = ((s2 >> (8 * t + 4)) & 15u) | (((s1 >> (8 * t + 6)) & 3u) << 4);
    }
}

template <int FMT>
struct Raw32;

// BF16 and F16: 64 bytes (fewer at a ragged row end; k is even).
template <int FMT>
struct Raw16bit {
    uint32_t wd[16];
    __device__ __forceinline__ void load(const uint8_t *row, int64_t k0, int nvalid) {
        const uint8_t *p = row + 2 * k0;
        if (nvalid == 32 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 v = ldg_u128(p + 16 * q);
                wd[4 * q] = v.x; wd[4 * q + 1] = v.y; wd[4 * q + 2] = v.z; wd[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) wd[i] = (2 * i < nvalid) ? ldg_u32(p + 4 * i) : 0u;
        }
    }
    __device__ __forceinline__ void decode(float (&w)[32]) const {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (FMT == F_BF16) {
                w[2 * i] = bf16_bits_to_f32(wd[i] & 0xFFFFu);
                w[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
            } else {
                w[2 * i] = f16_bits_to_f32(wd[i] & 0xFFFFu);
                w[2 * i + 1] = f16_bits_to_f32(wd[i] >> 16);
            }
        }
    }
};
template <> struct Raw32<F_BF16> : Raw16bit<F_BF16> {};
template <> struct Raw32<F_F16> : Raw16bit<F_F16> {};

template <>
struct Raw32<F_Q4_0> {
    uint32_t dbits;   // f16 d
    uint32_t qw[4];   // the 16 quant bytes, packed little-endian
    __device__ __forceinline__ void load(const uint8_t *row, int64_t k0, int) {
        const uint8_t *p = row + 18 * (k0 >> 5);
        dbits = ldg_u16(p);
#pragma unroll
        for (int i = 0; i < 4; ++i) qw[i] = ldg_u16(p + 2 + 4 * i) | (ldg_u16(p + 4 + 4 * i) << 16);
    }
    // the block at shared address a (2-byte aligned), from a raw W tile: a
    // row's blocks alternate between 2 mod 4 and 0 mod 4 starts, the last
    // one aligned, so no read leaves the row
    __device__ __forceinline__ void load_shared(uint32_t a) {
        dbits = lds16(a);
        lds_words_a2_exact<4>(a + 2, qw);
    }
    __device__ __forceinline__ void decode(float (&w)[32]) const {
        const float d = f16_bits_to_f32(dbits);
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const uint32_t q = (qw[b >> 2] >> (8 * (b & 3))) & 0xFFu;
            w[b] = __fmul_rn((float)((int)(q & 15u) - 8), d);
            w[b + 16] = __fmul_rn((float)((int)(q >> 4) - 8), d);
        }
    }
};

template <>
struct Raw32<F_Q4_K> {
    uint4 hdr;     // d | dmin | scales[0..11]
    uint4 qs[2];   // the 32 quant bytes shared by sub-blocks 2c and 2c+1
    int s;         // sub-block of these 32 weights
    __device__ __forceinline__ void load(const uint8_t *row, int64_t k0, int) {
        const uint8_t *p = row + 144 * (k0 >> 8);
        s = (int)((k0 & 255) >> 5);
        hdr = ldg_u128(p);
        qs[0] = ldg_u128(p + 16 + 32 * (s >> 1));
        qs[1] = ldg_u128(p + 32 + 32 * (s >> 1));
    }
    __device__ __forceinline__ void decode(float (&w)[32]) const {
        uint32_t sc, m;
        q4k_scale_min(hdr.y, hdr.z, hdr.w, s, sc, m);
        const float d = f16_bits_to_f32(hdr.x & 0xFFFFu);
        const float dmin = f16_bits_to_f32(hdr.x >> 16);
        const float ds = __fmul_rn(d, (float)sc);
        const float ndm = -__fmul_rn(dmin, (float)m);
        const uint32_t sh = (s & 1) ? 4u : 0u;
        const uint32_t words[8] = {qs[0].x, qs[0].y, qs[0].z, qs[0].w,
                                   qs[1].x, qs[1].y, qs[1].z, qs[1].w};
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const uint32_t q = (words[l >> 2] >> (8 * (l & 3) + sh)) & 15u;
            w[l] = __fmaf_rn(ds, (float)q, ndm);
        }
    }
};

template <>
struct Raw32<F_Q6_K> {
    uint32_t ql[8], qh[8];  // the 32 ql and 32 qh bytes used, packed little-endian
    uint32_t sc2, dbits;    // the two int8 scales of these 32 weights; f16 d
    int r;                  // which quarter of the half (selects nibble and qh bits)
    __device__ __forceinline__ void load(const uint8_t *row, int64_t k0, int) {
        const uint8_t *p = row + 210 * (k0 >> 8);
        const int e0 = (int)(k0 & 255);
        const int h = e0 >> 7;
        r = (e0 & 127) >> 5;
        const uint8_t *pl = p + 64 * h + 32 * (r & 1);
        const uint8_t *ph = p + 128 + 32 * h;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ql[i] = ldg_u16(pl + 4 * i) | (ldg_u16(pl + 4 * i + 2) << 16);
            qh[i] = ldg_u16(ph + 4 * i) | (ldg_u16(ph + 4 * i + 2) << 16);
        }
        sc2 = ldg_u16(p + 192 + 8 * h + 2 * r);
        dbits = ldg_u16(p + 208);
    }
    // weights e0 .. e0 + 31 (e0 a multiple of 32) of the super-block at shared
    // address sb (2-byte aligned), from a raw W tile; every read stays within
    // the super-block's 210 bytes
    __device__ __forceinline__ void load_shared(uint32_t sb, int e0) {
        const int h = e0 >> 7;
        r = (e0 & 127) >> 5;
        lds_words_a2_exact<8>(sb + 64u * h + 32u * (r & 1), ql);
        lds_words_a2_exact<8>(sb + 128u + 32u * h, qh);
        sc2 = lds16(sb + 192u + 8u * h + 2u * r);
        dbits = lds16(sb + 208u);
    }
    __device__ __forceinline__ void decode(float (&w)[32]) const {
        const float d = f16_bits_to_f32(dbits);
        const float ds0 = __fmul_rn(d, (float)(int)(int8_t)(sc2 & 0xFFu));
        const float ds1 = __fmul_rn(d, (float)(int)(int8_t)(sc2 >> 8));
        const uint32_t nsh = (r >= 2) ? 4u : 0u;
        const uint32_t hsh = 2u * (uint32_t)r;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const uint32_t lo = (ql[l >> 2] >> (8 * (l & 3))) & 0xFFu;
            const uint32_t hi = (qh[l >> 2] >> (8 * (l & 3))) & 0xFFu;
            const int q = (int)(((lo >> nsh) & 15u) | (((hi >> hsh) & 3u) << 4));
            w[l] = __fmul_rn(l < 16 ? ds0 : ds1, (float)(q - 32));
        }
    }
};

template <>
struct Raw32<F_Q8_0> {
    uint32_t dbits;
    uint32_t qw[8];   // the 32 code bytes, packed little-endian
    __device__ __forceinline__ void load(const uint8_t *row, int64_t k0, int) {
        const uint8_t *p = row + 34 * (k0 >> 5);
        dbits = ldg_u16(p);
#pragma unroll
        for (int i = 0; i < 8; ++i) qw[i] = ldg_u16(p + 2 + 4 * i) | (ldg_u16(p + 4 + 4 * i) << 16);
    }
    __device__ __forceinline__ void load_shared(uint32_t a) {
        dbits = lds16(a);
        lds_words_a2_exact<8>(a + 2, qw);
    }
    __device__ __forceinline__ void decode(float (&w)[32]) const {
        const float d = f16_bits_to_f32(dbits);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int q = (int)(int8_t)((qw[i >> 2] >> (8 * (i & 3))) & 0xFFu);
            w[i] = __fmul_rn((float)q, d);
        }
    }
};

template <>
struct Raw32<F_Q5_0> {
    uint32_t dbits, qh;
    uint32_t qw[4];   // the 16 nibble bytes, packed little-endian
    __device__ __forceinline__ void load(const uint8_t *row, int64_t k0, int) {
        const uint8_t *p = row + 22 * (k0 >> 5);
        dbits = ldg_u16(p);
        qh = ldg_u16(p + 2) | (ldg_u16(p + 4) << 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) qw[i] = ldg_u16(p + 6 + 4 * i) | (ldg_u16(p + 8 + 4 * i) << 16);
    }
    __device__ __forceinline__ void load_shared(uint32_t a) {
        dbits = lds16(a);
        uint32_t h[1];
        lds_words_a2_exact<1>(a + 2, h);
        qh = h[0];
        lds_words_a2_exact<4>(a + 6, qw);
    }
    __device__ __forceinline__ void decode(float (&w)[32]) const {
        const float d = f16_bits_to_f32(dbits);
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const uint32_t byte = (qw[b >> 2] >> (8 * (b & 3))) & 0xFFu;
            const int lo = (int)((byte & 15u) | (((qh >> b) & 1u) << 4));
            const int hi = (int)((byte >> 4) | (((qh >> (b + 16)) & 1u) << 4));
            w[b] = __fmul_rn((float)(lo - 16), d);
            w[b + 16] = __fmul_rn((float)(hi - 16), d);
        }
    }
};

// Affine formats: 32 codes (half a group) of row `row`, with the group's
// scale and bias from the rows `srow` / `brow` of the two bf16 arrays; k0 is
// a multiple of 32 and every 32-weight unit is whole (k % 64 == 0).
template <int BITS>
struct RawAffine {
    uint32_t qw[BITS];          // 32 codes: BITS words
    uint32_t sbits, bbits;      // bf16 patterns
    __device__ __forceinline__ void load(const uint8_t *row, const uint8_t *srow,
                                         const uint8_t *brow, int64_t k0) {
        const uint8_t *p = row + (k0 * BITS) / 8;
#pragma unroll
        for (int q = 0; q < BITS / 4; ++q) {
            const uint4 v = ldg_u128(p + 16 * q);
            qw[4 * q] = v.x; qw[4 * q + 1] = v.y; qw[4 * q + 2] = v.z; qw[4 * q + 3] = v.w;
        }
        sbits = ldg_u16(srow + 2 * (k0 >> 6));
        bbits = ldg_u16(brow + 2 * (k0 >> 6));
    }
    __device__ __forceinline__ void decode(float (&w)[32]) const {
        const float sc = __uint_as_float(sbits << 16), bi = __uint_as_float(bbits << 16);
        constexpr int per = 32 / BITS;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t q = (qw[i / per] >> (BITS * (i % per))) & ((1u << BITS) - 1u);
            w[i] = __fmaf_rn((float)q, sc, bi);
        }
    }
};
template <> struct Raw32<F_AFF4> : RawAffine<4> {};
template <> struct Raw32<F_AFF8> : RawAffine<8> {};

}  // namespace qmm
