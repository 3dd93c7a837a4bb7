// qmm_mma.cu -- host side of the N-token tensor-core product: the x
// conversion kernel (fp16 copy of x with a power-of-two scale per token), the
// precision mode and workspace rules, the tensor maps and the persistent
// schedule. The kernel itself is in qmm_mma_kernel.cuh; its instances are
// compiled in the qmm_mma_inst_*.cu units.
#include "qmm_mma_kernel.cuh"

namespace qmm {

extern template cudaError_t launch_fmt<F_BF16>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_F16>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q4_0>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q4_K>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q6_K>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q8_0>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q5_0>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_AFF4>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_AFF8>(int, int, const Maps &, const MmaAffParams &,
                                            const DeviceInfo &, cudaStream_t);

// y columns that split tiles add into: zeroed per token by the conversion kernel
struct SplitZero {
    float *y;          // null: no split tiles
    int64_t n, j0, j1;
    int first;         // first split pair-tile
    int pairs, tiles_n, tok, rows;
};

// X [N][k] fp32 -> X16 [N][kp] fp16 (zero padded) scaled by 2^-e per row so the
// row's largest magnitude lands in [2^14, 2^15); xscale[t] = 2^e. With x16lo,
// also the fp16 rounding of what X16 missed (x = hi + lo to ~22 bits).
__global__ void __launch_bounds__(256) x_to_f16_kernel(const float *__restrict__ x, int64_t k,
                                                       int64_t kp, __half *__restrict__ x16,
                                                       __half *__restrict__ x16lo,
                                                       float *__restrict__ xscale,
                                                       const SplitZero z) {
    __shared__ float red[8];
    pdl_launch_dependents();  // the product kernel may start its W pipeline now
    if (z.y) {
        // split pair-tiles v >= first (v = q * tiles_n + nt) of this token's
        // token tile start at the first such v; they run to the last row tile
        const int nt = (int)(blockIdx.x / z.tok);
        const int v0 = z.first + ((nt - z.first % z.tiles_n) % z.tiles_n + z.tiles_n) % z.tiles_n;
        if (v0 < z.pairs * z.tiles_n) {
            const int64_t c0 = z.j0 + (int64_t)(v0 / z.tiles_n) * 2 * z.rows;
            float *yt = z.y + (int64_t)blockIdx.x * z.n;
            for (int64_t j = c0 + threadIdx.x; j < z.j1; j += blockDim.x) yt[j] = 0.0f;
        }
    }
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

// Precision mode of a call. x is always split into two fp16 terms (about 22
// significant bits), so its rounding cannot add up over k whatever x holds
// (a single fp16 copy errs by up to 2^-12 per element, coherently for
// constant or repeated activations: 2.4e-4 of sum |x w| for x = 0.1). W is
// rounded once to fp16 (16-bit formats are exact in fp16 within its range);
// for k < 1024 it is split too, since fewer products average its rounding.
int mma_mode(int fmt, int64_t k) {
    if (fmt == F_BF16 || fmt == F_F16) return 2;
    // affine rows take the raw-tile path in whole 256-wide slices; other k
    // decode from registers with both operands split
    if (is_affine(fmt) && k % 256 != 0) return 3;
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
    // tokens per CTA tile: up to 256 (MODE 1) or 128 (hi + lo rows share the tile)
    const int tok_max = mode == 1 ? 256 : 128;
    int tok = tok_max;
    if (m.n_tokens < tok_max) {
        tok = 16;
        while (tok < m.n_tokens) tok <<= 1;
    }
    // schedule: P pair-tiles over NC resident clusters; when the last round is
    // at most half full, its R pair-tiles run as two k-halves each
    const int rows_out = mode == 3 ? 64 : kBM;
    const int64_t tiles_m = (M + rows_out - 1) / rows_out;
    const int pairs = (int)((tiles_m + 1) / 2);
    const int tiles_n = (int)((m.n_tokens + tok - 1) / tok);
    const int P = pairs * tiles_n, NC = mma_clusters(dev);
    const int R = P % NC;
    const int KS = (int)(kp / kBK);
    const bool split = mode != 3 && !m.accumulate && R > 0 && 2 * R <= NC && (KS + 3) / 4 >= 2;
    SplitZero z = {};
    if (split) {
        z.y = m.y;
        z.n = m.n; z.j0 = m.j0; z.j1 = m.j1;
        z.first = P - R;
        z.pairs = pairs; z.tiles_n = tiles_n; z.tok = mode == 1 ? tok : tok;
        z.rows = rows_out;
    }
    x_to_f16_kernel<<<(unsigned)m.n_tokens, 256, 0, s>>>(m.x, m.k, kp, x16, x16lo, xscale, z);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int bn = mode == 1 ? tok : 2 * tok;
    // each CTA of a pair fetches half of an x tile: BN/2 token rows
    const int box_rows = bn / 2;
    Maps mp;
    if (!encode_x_map(encode, &mp.x, x16, kp, m.n_tokens, box_rows)) return cudaErrorInvalidValue;
    if (mode >= 2) {
        if (!encode_x_map(encode, &mp.xlo, x16lo, kp, m.n_tokens, box_rows))
            return cudaErrorInvalidValue;
    } else {
        mp.xlo = mp.x;
    }
    CUtensorMap &tm = mp.x;
    CUtensorMap &tw = mp.w;
    // raw W tiles: the packed rows as a 2-D byte tensor [n][row_bytes]
    tw = tm;
    if (raw_slice_bytes(m.fmt, mode) > 0) {
        // raw W tiles: Q4_K boxes of 128 rows x one 144-byte super-block;
        // affine code boxes of 128 rows x 128 bytes, 128-byte swizzled (the
        // dequant warps read 16-byte chunks of 32 consecutive rows)
        const bool aff = is_affine(m.fmt);
        const cuuint64_t dims[2] = {(cuuint64_t)m.row_bytes, (cuuint64_t)m.n};
        const cuuint64_t strides[1] = {(cuuint64_t)m.row_bytes};
        const cuuint32_t box[2] = {aff ? 128u : 144u, (cuuint32_t)kBM};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(m.w), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   aff ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    MmaAffParams p;
    p.w = m.w; p.y = m.y; p.xscale = xscale;
    p.sc = m.sc;
    p.bi = m.bi;
    p.aux_row_bytes = (m.k / 64) * 2;
    p.k = m.k; p.n = m.n; p.n_tokens = m.n_tokens; p.row_bytes = m.row_bytes;
    p.j0 = m.j0; p.j1 = m.j1;
    p.KS = (int)(kp / kBK);
    p.accumulate = m.accumulate;
    p.err = dev.err;
    p.pairs = pairs;
    p.tiles_n = tiles_n;
    p.full_units = split ? P - R : P;
    p.split = split ? 2 : 1;
    p.n_units = p.full_units + (P - p.full_units) * p.split;
    switch (m.fmt) {
    case F_BF16: return launch_fmt<F_BF16>(mode, bn, mp, p, dev, s);
    case F_F16: return launch_fmt<F_F16>(mode, bn, mp, p, dev, s);
    case F_Q4_0: return launch_fmt<F_Q4_0>(mode, bn, mp, p, dev, s);
    case F_Q4_K: return launch_fmt<F_Q4_K>(mode, bn, mp, p, dev, s);
    case F_Q6_K: return launch_fmt<F_Q6_K>(mode, bn, mp, p, dev, s);
    case F_Q8_0: return launch_fmt<F_Q8_0>(mode, bn, mp, p, dev, s);
    case F_Q5_0: return launch_fmt<F_Q5_0>(mode, bn, mp, p, dev, s);
    case F_AFF4: return launch_fmt<F_AFF4>(mode, bn, mp, p, dev, s);
    case F_AFF8: return launch_fmt<F_AFF8>(mode, bn, mp, p, dev, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
