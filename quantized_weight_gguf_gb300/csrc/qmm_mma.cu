// qmm_mma.cu -- N-token fused dequantize + tensor-core product on sm_103a:
// Y[t][j] = sum_i X[t][i] W[j][i] for a tile of 128 output columns j and BN
// tokens t per CTA.
//
// Pipeline per CTA (one CTA per SM, warp-specialised):
//   warp 0      TMA producer: fp16 X tiles [BN tokens x 64 k] -> shared memory
//               (128-byte swizzle) through a tensor map;
//   warp 1      allocates the fp32 accumulator in tensor memory (TMEM) and one
//               lane issues tcgen05.mma (M=128, N=BN, K=16, fp16 in, fp32 acc);
//   warps 2..9  dequantize W: thread (r, h) turns 32 weights of row r per
//               k-step into fp16 and stores them in the same swizzled K-major
//               layout the MMA descriptor describes; after the k-loop they
//               drain the accumulator TMEM -> registers -> y.
// X is converted to fp16 once per call by a small kernel that also scales each
// token row by a power of two (exact) so it fits fp16's range; the epilogue
// multiplies by the inverse power.
//
// Precision modes (fp16 operands round each product's inputs to 11 bits; the
// resulting error relative to sum |x w| shrinks like 1/sqrt(k)):
//   MODE 1  W16 . X16                      one product per output
//   MODE 2  W16 . (X_hi + X_lo)            x split into two fp16 terms: the B
//           tile holds BN/2 tokens' hi rows then their lo rows, and the
//           epilogue adds column c and c + BN/2 (exact for fp16-exact W)
//   MODE 3  (W_hi + W_lo) . (X_hi + X_lo)  also w split: the A tile holds 64
//           rows' hi parts then their lo parts; the epilogue adds the row
//           pair through shared memory.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "qmm_decode.cuh"
#include "qmm_internal.h"

namespace qmm {

constexpr int kMmaThreads = 320;
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB per stage

struct MmaParams {
    const uint8_t *w;
    float *y;
    const float *xscale;
    int64_t k, n, n_tokens, row_bytes;
    int64_t j0, j1;
    int KS;
    int accumulate;
    unsigned int *err;
};

template <int BN>
struct MmaCfg {
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStage = kABytes + kBBytes;
    static constexpr int NS = (192 * 1024 / kStage) > 8 ? 8 : (192 * 1024 / kStage);
    static constexpr int kCols = BN < 32 ? 32 : BN;  // TMEM columns (power of two >= 32)
    static constexpr size_t kSmem = (size_t)NS * kStage + 1024 /*align*/ + 256 /*barriers*/;
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

template <int FMT>
struct Prefetch {
    static constexpr int value = (FMT == F_Q4_K || FMT == F_Q4_0) ? 4 : 3;
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

template <int FMT, int BN, int MODE>
__global__ void __launch_bounds__(kMmaThreads, 1)
    mma_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmx_lo,
               const MmaParams p) {
    constexpr int kRowsOut = MODE == 3 ? 64 : kBM;   // output rows per CTA
    constexpr int kTokOut = MODE == 1 ? BN : BN / 2;  // tokens per CTA
    using C = MmaCfg<BN>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
    const uint32_t A0 = sbase;
    const uint32_t B0 = sbase + NS * kABytes;
    const uint32_t bar0 = B0 + NS * C::kBBytes;
    auto fullA = [&](int s) { return bar0 + 8u * s; };
    auto fullB = [&](int s) { return bar0 + 8u * (NS + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * NS + s); };
    const uint32_t accb = bar0 + 8u * (3 * NS);
    const uint32_t slot_addr = accb + 8u;
    uint8_t *gen = smem_raw + (bar0 - raw_addr);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gen + 8 * (3 * NS) + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gen + 8 * (3 * NS) + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t m0 = p.j0 + (int64_t)blockIdx.x * kRowsOut;
    const int n0 = blockIdx.y * kTokOut;
    const int KS = p.KS;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(fullA(s), 8);
            mbar_init(fullB(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(accb, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(slot_addr, C::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------ X tiles via TMA ------------------------------
        if (lane == 0) {
            prefetch_tmap(&tmx);
            if (MODE != 1) prefetch_tmap(&tmx_lo);
            int issued = 0;
            for (int ks = 0; ks < KS; ++ks) {
                const int slot = ks % NS;
                if (ks >= NS && !wait_abortable(empty(slot), ((ks / NS) + 1) & 1, abort_flag)) {
                    record_error(p.err, DERR_MMA_EMPTY);
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(fullB(slot), C::kBBytes);
                if (MODE == 1) {
                    tma_load_2d(B0 + slot * C::kBBytes, &tmx, ks * kBK, n0, fullB(slot));
                } else {  // hi rows then lo rows of the same tokens
                    tma_load_2d(B0 + slot * C::kBBytes, &tmx, ks * kBK, n0, fullB(slot));
                    tma_load_2d(B0 + slot * C::kBBytes + (BN / 2) * 128, &tmx_lo, ks * kBK, n0,
                                fullB(slot));
                }
                ++issued;
            }
            for (int s = std::max(0, issued - NS); s < issued; ++s)
                if (!mbar_wait(fullB(s % NS), (s / NS) & 1)) record_error(p.err, DERR_TEARDOWN);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issue ------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
            for (int ks = 0; ks < KS; ++ks) {
                const int slot = ks % NS;
                const uint32_t par = (ks / NS) & 1;
                if (!wait_abortable(fullA(slot), par, abort_flag)) {
                    record_error(p.err, DERR_MMA_A);
                    *abort_flag = 1;
                    break;
                }
                if (!wait_abortable(fullB(slot), par, abort_flag)) {
                    record_error(p.err, DERR_MMA_B);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sdesc_sw128(A0 + slot * kABytes);
                const uint64_t bd = sdesc_sw128(B0 + slot * C::kBBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)  // K = 16 per instruction: +32 bytes
                    tc_mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (ks | kk) != 0);
                tc_commit(empty(slot));
            }
            tc_commit(accb);  // fires when every MMA issued above has completed
        }
    } else {
        // ------------------------------ W dequant producers ------------------------------
        const int dt = tid - 64;
        const int r = dt & (kBM - 1);
        const int h = dt >> 7;
        const bool lo_part = MODE == 3 && r >= 64;   // MODE 3: rows 64..127 hold W_lo
        const int64_t j = m0 + (MODE == 3 ? (r & 63) : r);
        const bool row_ok = j < p.j1;
        const uint8_t *rowp = p.w + (row_ok ? j : 0) * p.row_bytes;
        const uint32_t swz = (uint32_t)(r & 7);
        constexpr int PD = Prefetch<FMT>::value;
        Raw32<FMT> ring[PD];
        auto k0_of = [&](int ks) { return (int64_t)ks * kBK + 32 * h; };
        auto nvalid_of = [&](int64_t k0) {
            const int64_t v = p.k - k0;
            return (int)(v < 0 ? 0 : (v > 32 ? 32 : v));
        };
#pragma unroll
        for (int q = 0; q < PD; ++q) {
            const int64_t k0 = k0_of(q);
            const int nv = nvalid_of(k0);
            if (q < KS && row_ok && nv > 0) ring[q].load(rowp, k0, nv);
        }
        bool failed = false;
        for (int ks0 = 0; ks0 < KS; ks0 += PD) {
#pragma unroll
            for (int q = 0; q < PD; ++q) {
                const int ks = ks0 + q;
                if (ks < KS) {
                    const int64_t k0 = k0_of(ks);
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
                            for (int i = 0; i < 16; ++i)
                                if (2 * i >= nv) hw[i] = 0u;  // nv is even
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) hw[i] = 0u;
                    }
                    const int64_t kn = k0_of(ks + PD);
                    const int nvn = nvalid_of(kn);
                    if (ks + PD < KS && row_ok && nvn > 0) ring[q].load(rowp, kn, nvn);
                    const int slot = ks % NS;
                    if (!failed && ks >= NS &&
                        !wait_abortable(empty(slot), ((ks / NS) + 1) & 1, abort_flag)) {
                        failed = true;
                        *abort_flag = 1;
                        record_error(p.err, DERR_MMA_EMPTY);
                    }
                    if (!failed) {
                        const uint32_t arow = A0 + slot * kABytes + (uint32_t)r * 128u;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t chunk = (uint32_t)(4 * h + c) ^ swz;
                            sts128(arow + chunk * 16u, hw[4 * c], hw[4 * c + 1], hw[4 * c + 2],
                                   hw[4 * c + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && !failed) mbar_arrive(fullA(slot));
                }
            }
        }
        // ------------------------------ epilogue ------------------------------
        __syncwarp();
        const bool acc_ok = mbar_wait(accb, 0);
        if (!acc_ok) record_error(p.err, DERR_MMA_ACC);
        tc_fence_after();
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        // token columns of this warp within [0, kTokOut)
        int c_lo, c_hi;
        if (kTokOut >= 32) {
            c_lo = half * (kTokOut / 2);
            c_hi = c_lo + kTokOut / 2;
        } else {
            c_lo = 0;
            c_hi = half == 0 ? kTokOut : 0;
        }
        const int rl = 32 * quarter + lane;                 // accumulator row (TMEM lane)
        const int64_t je = m0 + (MODE == 3 ? (rl & 63) : rl);
        const bool store_ok = acc_ok && !*abort_flag && je < p.j1;
        const uint32_t tbase = tmem + ((uint32_t)(32 * quarter) << 16);
        float *scratch = reinterpret_cast<float *>(smem_raw + (A0 - raw_addr));  // [col][64]
        if (MODE == 3 && quarter >= 2) {
            // lo rows: park (D[r][c] + D[r][c + BN/2]) for the hi warps
            __syncwarp();
            for (int col = c_lo; col < c_hi; col += 16) {
                uint32_t v[16], w2[16];
                tmem_ld16(tbase + (uint32_t)col, v);
                tmem_ld16(tbase + (uint32_t)(col + BN / 2), w2);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    scratch[(col + i) * 64 + (rl & 63)] = __uint_as_float(v[i]) + __uint_as_float(w2[i]);
            }
        }
        if (MODE == 3) named_barrier(2, 256);
        if (MODE != 3 || quarter < 2) {
            __syncwarp();
            for (int col = c_lo; col < c_hi; col += 16) {
                uint32_t v[16];
                tmem_ld16(tbase + (uint32_t)col, v);
                float acc[16];
                if (MODE == 1) {
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = __uint_as_float(v[i]);
                } else {
                    uint32_t w2[16];
                    tmem_ld16(tbase + (uint32_t)(col + BN / 2), w2);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = __uint_as_float(v[i]) + __uint_as_float(w2[i]);
                    if (MODE == 3) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[i] += scratch[(col + i) * 64 + (rl & 63)];
                    }
                }
                if (store_ok) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int64_t t = n0 + col + i;
                        if (t < p.n_tokens) {
                            const float val = acc[i] * __ldg(p.xscale + t);
                            float *yp = p.y + t * p.n + je;
                            *yp = p.accumulate ? *yp + val : val;
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kCols);
    }
}

// X [N][k] fp32 -> X16 [N][kp] fp16 (zero padded) scaled by 2^-e per row so the
// row's largest magnitude lands in [2^14, 2^15); xscale[t] = 2^e. With x16lo,
// also the fp16 rounding of what X16 missed (x = hi + lo to ~22 bits).
__global__ void __launch_bounds__(256) x_to_f16_kernel(const float *__restrict__ x, int64_t k,
                                                       int64_t kp, __half *__restrict__ x16,
                                                       __half *__restrict__ x16lo,
                                                       float *__restrict__ xscale) {
    __shared__ float red[8];
    const int64_t t = blockIdx.x;
    const float *xt = x + t * k;
    float m = 0.0f;
    for (int64_t i = threadIdx.x; i < k; i += blockDim.x) m = fmaxf(m, fabsf(__ldg(xt + i)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    m = red[0];
    int e = 0;
    if (m > 0.0f && isfinite(m)) {
        int E;
        frexpf(m, &E);
        e = E - 15;
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
    }
    __half *ot = x16 + t * kp;
    __half *ol = x16lo ? x16lo + t * kp : nullptr;
    for (int64_t i = threadIdx.x; i < kp; i += blockDim.x) {
        const float v = i < k ? ldexpf(__ldg(xt + i), -e) : 0.0f;
        const __half hv = __float2half_rn(v);
        ot[i] = hv;
        if (ol) ol[i] = __float2half_rn(v - __half2float(hv));
    }
    if (threadIdx.x == 0) xscale[t] = ldexpf(1.0f, e);
}

// ------------------------------------------------------------------ host ----

static int64_t kpad(int64_t k) { return (k + kBK - 1) / kBK * kBK; }
static size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

int mma_mode(int fmt, int64_t k) {
    if (fmt == F_BF16 || fmt == F_F16) return 2;  // W is fp16-exact: split x only
    if (k >= 4096) return 1;
    if (k >= 1024) return 2;
    return 3;
}

size_t mma_workspace_bytes(int fmt, int64_t n_tokens, int64_t k) {
    const size_t one = round256((size_t)n_tokens * (size_t)kpad(k) * 2);
    return (mma_mode(fmt, k) >= 2 ? 2 : 1) * one + round256((size_t)n_tokens * 4);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

template <int FMT, int BN, int MODE>
static cudaError_t launch_t(const CUtensorMap &tm, const CUtensorMap &tl, const MmaParams &p,
                            dim3 grid, cudaStream_t s) {
    using C = MmaCfg<BN>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(mma_kernel<FMT, BN, MODE>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    mma_kernel<FMT, BN, MODE><<<grid, kMmaThreads, C::kSmem, s>>>(tm, tl, p);
    return cudaGetLastError();
}

template <int FMT, int MODE>
static cudaError_t launch_bn(int bn, const CUtensorMap &tm, const CUtensorMap &tl,
                             const MmaParams &p, dim3 grid, cudaStream_t s) {
    switch (bn) {
    case 16: if (MODE == 1) return launch_t<FMT, 16, MODE>(tm, tl, p, grid, s); break;
    case 32: return launch_t<FMT, 32, MODE>(tm, tl, p, grid, s);
    case 64: return launch_t<FMT, 64, MODE>(tm, tl, p, grid, s);
    case 128: return launch_t<FMT, 128, MODE>(tm, tl, p, grid, s);
    case 256: return launch_t<FMT, 256, MODE>(tm, tl, p, grid, s);
    default: break;
    }
    return cudaErrorInvalidValue;
}

template <int FMT>
static cudaError_t launch_fmt(int mode, int bn, const CUtensorMap &tm, const CUtensorMap &tl,
                              const MmaParams &p, dim3 grid, cudaStream_t s) {
    constexpr bool quant = FMT != F_BF16 && FMT != F_F16;
    if (mode == 2) return launch_bn<FMT, 2>(bn, tm, tl, p, grid, s);
    if (quant && mode == 1) return launch_bn<FMT, quant ? 1 : 2>(bn, tm, tl, p, grid, s);
    if (quant && mode == 3) return launch_bn<FMT, quant ? 3 : 2>(bn, tm, tl, p, grid, s);
    return cudaErrorInvalidValue;
}

static bool encode_x_map(EncodeTiledFn encode, CUtensorMap *tm, void *base, int64_t kp,
                         int64_t n_tokens, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)kp, (cuuint64_t)n_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)kp * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_mma(const MmaLaunch &m, const DeviceInfo &dev, cudaStream_t s) {
    const int64_t M = m.j1 - m.j0;
    if (M <= 0 || m.n_tokens <= 0) return cudaSuccess;
    EncodeTiledFn encode = get_encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const int mode = mma_mode(m.fmt, m.k);
    const int64_t kp = kpad(m.k);
    const size_t one = round256((size_t)m.n_tokens * kp * 2);
    uint8_t *ws = reinterpret_cast<uint8_t *>(m.workspace);
    __half *x16 = reinterpret_cast<__half *>(ws);
    __half *x16lo = mode >= 2 ? reinterpret_cast<__half *>(ws + one) : nullptr;
    float *xscale = reinterpret_cast<float *>(ws + (mode >= 2 ? 2 : 1) * one);
    x_to_f16_kernel<<<(unsigned)m.n_tokens, 256, 0, s>>>(m.x, m.k, kp, x16, x16lo, xscale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // tokens per CTA tile: up to 256 (MODE 1) or 128 (hi + lo rows share the tile)
    const int tok_max = mode == 1 ? 256 : 128;
    int tok = tok_max;
    if (m.n_tokens < tok_max) {
        tok = 16;
        while (tok < m.n_tokens) tok <<= 1;
    }
    const int bn = mode == 1 ? tok : 2 * tok;
    CUtensorMap tm, tl;
    if (!encode_x_map(encode, &tm, x16, kp, m.n_tokens, tok)) return cudaErrorInvalidValue;
    if (mode >= 2) {
        if (!encode_x_map(encode, &tl, x16lo, kp, m.n_tokens, tok)) return cudaErrorInvalidValue;
    } else {
        tl = tm;
    }
    MmaParams p;
    p.w = m.w; p.y = m.y; p.xscale = xscale;
    p.k = m.k; p.n = m.n; p.n_tokens = m.n_tokens; p.row_bytes = m.row_bytes;
    p.j0 = m.j0; p.j1 = m.j1;
    p.KS = (int)(kp / kBK);
    p.accumulate = m.accumulate;
    p.err = dev.err;
    const int rows_out = mode == 3 ? 64 : kBM;
    const dim3 grid((unsigned)((M + rows_out - 1) / rows_out),
                    (unsigned)((m.n_tokens + tok - 1) / tok));
    switch (m.fmt) {
    case F_BF16: return launch_fmt<F_BF16>(mode, bn, tm, tl, p, grid, s);
    case F_F16: return launch_fmt<F_F16>(mode, bn, tm, tl, p, grid, s);
    case F_Q4_0: return launch_fmt<F_Q4_0>(mode, bn, tm, tl, p, grid, s);
    case F_Q4_K: return launch_fmt<F_Q4_K>(mode, bn, tm, tl, p, grid, s);
    case F_Q6_K: return launch_fmt<F_Q6_K>(mode, bn, tm, tl, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
