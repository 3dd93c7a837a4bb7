// qmm_mma.cu -- host side of the N-token tensor-core product: the x
// conversion kernel (fp16 copy of x with a power-of-two scale per token), the
// precision mode and workspace rules, the tensor maps and the persistent
// schedule. The kernel itself is in qmm_mma_kernel.cuh; its instances are
// compiled in the qmm_mma_inst_*.cu units.
#include "qmm_mma_kernel.cuh"

#include <cuda_bf16.h>

namespace qmm {

extern template cudaError_t launch_fmt<F_BF16>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_F16>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q4_0>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q4_K>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q6_K>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q8_0>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_Q5_0>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_AFF4>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
extern template cudaError_t launch_fmt<F_AFF8>(int, int, const Maps &, const MmaHostParams &,
                                            const DeviceInfo &, cudaStream_t);
#define QMM_EXTERN_GROUPED(F)                                                                \
    extern template cudaError_t launch_fmt_grouped<F>(int, const Maps &, const MmaHostParams &, \
                                                      const DeviceInfo &, cudaStream_t)
QMM_EXTERN_GROUPED(F_BF16);
QMM_EXTERN_GROUPED(F_F16);
QMM_EXTERN_GROUPED(F_Q4_0);
QMM_EXTERN_GROUPED(F_Q4_K);
QMM_EXTERN_GROUPED(F_Q6_K);
QMM_EXTERN_GROUPED(F_Q8_0);
QMM_EXTERN_GROUPED(F_Q5_0);
#undef QMM_EXTERN_GROUPED

// y columns that split tiles add into: zeroed per token by the conversion kernel
struct SplitZero {
    float *y;          // null: no split tiles
    int64_t n, j0, j1;
    int first;         // first split pair-tile
    int pairs, tiles_n, tok, rows;
};

// Rows of x in another order (expert-grouped products): x16 row t is x row
// src[t] / top_k for t < *count, zeros beyond.
struct XGather {
    const int *src;     // null: row t is x row t
    const int *count;
    int top_k;
};

// X [N][k] fp32 -> X16 [N][kp] fp16 (zero padded) scaled by 2^-e per row so the
// row's largest magnitude lands in [2^14, 2^15); xscale[t] = 2^e. With x16lo,
// also the fp16 rounding of what X16 missed (x = hi + lo to ~22 bits). With
// bf16 set, both terms are bf16 instead (x = hi + lo to ~16 bits), for
// products whose W tiles are bf16.
__global__ void __launch_bounds__(256) x_to_f16_kernel(const float *__restrict__ x, int64_t k,
                                                       int64_t kp, __half *__restrict__ x16,
                                                       __half *__restrict__ x16lo,
                                                       float *__restrict__ xscale,
                                                       const SplitZero z, const XGather gx,
                                                       const int bf16) {
    __shared__ float red[8];
    // Launched as a programmatic dependent: the product kernel that follows may
    // start its W pipeline now; everything this kernel reads (x, the routing)
    // or writes (the workspace, y's split columns) waits for the preceding
    // grid, which may still be reading the workspace, to complete.
    pdl_launch_dependents();
    pdl_wait_prev();
    int64_t src_row = blockIdx.x;
    if (gx.src) {
        const int64_t t = blockIdx.x;
        if (t >= *gx.count) {  // past the routed rows (block-uniform)
            for (int64_t i = threadIdx.x; i < kp; i += blockDim.x) {
                x16[t * kp + i] = __float2half_rn(0.0f);
                x16lo[t * kp + i] = __float2half_rn(0.0f);
            }
            if (threadIdx.x == 0) xscale[t] = 1.0f;
            return;
        }
        src_row = gx.src[t] / gx.top_k;
    }
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
    const float *xt = x + src_row * k;
    // Rows of up to kXRegs float4 per thread (k <= 8192, 16-byte aligned) are
    // read once, with 16-byte loads, and kept in registers for the
    // conversion; 8-byte stores write four halves at a time. Other rows are
    // read twice (the second pass from L2) element by element. Both forms
    // round every element the same way.
    constexpr int kXRegs = 8;
    const bool in_regs = (reinterpret_cast<uintptr_t>(xt) & 15u) == 0 && (k & 3) == 0 &&
                         kp <= 4 * 256 * kXRegs && blockDim.x == 256;
    float4 xv[kXRegs];
    float m = 0.0f;
    if (in_regs) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xt);
        const int64_t k4 = k >> 2;
#pragma unroll
        for (int j = 0; j < kXRegs; ++j) {
            const int64_t i = threadIdx.x + 256 * j;
            xv[j] = i < k4 ? __ldg(x4 + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(xv[j].x), fabsf(xv[j].y)),
                               fmaxf(fabsf(xv[j].z), fabsf(xv[j].w))));
        }
    } else {
        for (int64_t i = threadIdx.x; i < k; i += blockDim.x) m = fmaxf(m, fabsf(__ldg(xt + i)));
    }
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
    if (in_regs) {
        // kp is a multiple of 64 and the rows start 256-byte aligned: every
        // group of four halves is one aligned 8-byte store
        const int64_t kp4 = kp >> 2;
#pragma unroll
        for (int j = 0; j < kXRegs; ++j) {
            const int64_t i = threadIdx.x + 256 * j;
            if (i < kp4) {
                const float v0 = ldexpf(xv[j].x, -e), v1 = ldexpf(xv[j].y, -e);
                const float v2 = ldexpf(xv[j].z, -e), v3 = ldexpf(xv[j].w, -e);
                uint2 hw, lw;
                float2 f01, f23;
                if (bf16) {
                    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v0, v1);
                    const __nv_bfloat162 h23 = __floats2bfloat162_rn(v2, v3);
                    f01 = __bfloat1622float2(h01);
                    f23 = __bfloat1622float2(h23);
                    hw.x = *reinterpret_cast<const uint32_t *>(&h01);
                    hw.y = *reinterpret_cast<const uint32_t *>(&h23);
                } else {
                    const __half2 h01 = __floats2half2_rn(v0, v1), h23 = __floats2half2_rn(v2, v3);
                    f01 = __half22float2(h01);
                    f23 = __half22float2(h23);
                    hw.x = *reinterpret_cast<const uint32_t *>(&h01);
                    hw.y = *reinterpret_cast<const uint32_t *>(&h23);
                }
                *reinterpret_cast<uint2 *>(ot + 4 * i) = hw;
                if (ol) {
                    if (bf16) {
                        const __nv_bfloat162 l01 = __floats2bfloat162_rn(v0 - f01.x, v1 - f01.y);
                        const __nv_bfloat162 l23 = __floats2bfloat162_rn(v2 - f23.x, v3 - f23.y);
                        lw.x = *reinterpret_cast<const uint32_t *>(&l01);
                        lw.y = *reinterpret_cast<const uint32_t *>(&l23);
                    } else {
                        const __half2 l01 = __floats2half2_rn(v0 - f01.x, v1 - f01.y);
                        const __half2 l23 = __floats2half2_rn(v2 - f23.x, v3 - f23.y);
                        lw.x = *reinterpret_cast<const uint32_t *>(&l01);
                        lw.y = *reinterpret_cast<const uint32_t *>(&l23);
                    }
                    *reinterpret_cast<uint2 *>(ol + 4 * i) = lw;
                }
            }
        }
    } else {
        for (int64_t i = threadIdx.x; i < kp; i += blockDim.x) {
            const float v = i < k ? ldexpf(__ldg(xt + i), -e) : 0.0f;
            if (bf16) {
                const __nv_bfloat16 hv = __float2bfloat16_rn(v);
                const __nv_bfloat16 lv = __float2bfloat16_rn(v - __bfloat162float(hv));
                ot[i] = *reinterpret_cast<const __half *>(&hv);
                if (ol) ol[i] = *reinterpret_cast<const __half *>(&lv);
            } else {
                const __half hv = __float2half_rn(v);
                ot[i] = hv;
                if (ol) ol[i] = __float2half_rn(v - __half2float(hv));
            }
        }
    }
    if (threadIdx.x == 0) xscale[t] = ldexpf(1.0f, e);
}

// The conversion as a programmatic dependent of the preceding grid (see the
// kernel's first lines).
static cudaError_t launch_x_to_f16(unsigned blocks, cudaStream_t s, int bf16, const float *x, int64_t k,
                                   int64_t kp, __half *x16, __half *x16lo, float *xscale,
                                   const SplitZero &z, const XGather &gx) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, x_to_f16_kernel, x, k, kp, x16, x16lo, xscale, z, gx, bf16);
}

// ------------------------------------------------------------------ host ----

static int64_t kpad(int64_t k) { return (k + kBK - 1) / kBK * kBK; }
static size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

// Precision mode of a call. x is always split into two fp16 terms (about 22
// significant bits), so its rounding cannot add up over k whatever x holds
// (a single fp16 copy errs by up to 2^-12 per element, coherently for
// constant or repeated activations: 2.4e-4 of sum |x w| for x = 0.1). W is
// rounded once to fp16 (16-bit formats are exact in fp16 within its range);
// for k < 1024 it is split too, since fewer products average its rounding,
// and at any k when the caller asks (QMM_FLAG_SPLIT_W: rows that repeat one
// weight value add its rounding up coherently).
int mma_mode(int fmt, int64_t k, bool split_w) {
    if (fmt == F_BF16 || fmt == F_F16) return 2;
    if (split_w) return 3;
    // affine and block-format rows take the raw-tile path in whole 256-wide
    // slices; other k decode from registers with both operands split
    if ((is_affine(fmt) || raw_block32(fmt)) && k % 256 != 0) return 3;
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

// Raw W tiles: the packed rows as a 2-D tensor [rows][row_bytes] (16-bit
// elements for Q8_0, bytes otherwise), boxes of 128 rows x one 256-wide k
// slice (Q4_K 144 B, Q4_0 144, Q5_0 176, Q8_0 272: multiples of 16 bytes, as
// are the row strides for k % 256 == 0); affine code boxes of 128 rows x
// 128 bytes, 128-byte swizzled (the dequant warps read 16-byte chunks of 32
// consecutive rows).
static bool encode_raw_w_map(EncodeTiledFn encode, CUtensorMap *tm, const uint8_t *w, int fmt,
                             int64_t row_bytes, int64_t rows) {
    const bool aff = is_affine(fmt);
    const int eb = raw_elem_bytes(fmt);
    const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / eb), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {aff ? 128u : (cuuint32_t)(raw_slice_bytes(fmt, 2) / eb),
                               (cuuint32_t)kBM};
    const cuuint32_t estr[2] = {1, 1};
    return encode(tm, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<uint8_t *>(w), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  aff ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    const int mode = mma_mode(m.fmt, m.k, m.split_w != 0);
    // 16-bit W tiles as the MMA's A operand from shared memory: rows a tensor
    // map can describe (2 k bytes a multiple of 16)
    const bool ss = (m.fmt == F_BF16 || m.fmt == F_F16) && mode == 2 && m.k % 8 == 0;
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
    // (not for the gated up product: a saturated gate makes act(g) * u_half
    // subnormal, and fp32 atomic adds flush subnormals to zero)
    const bool split = mode != 3 && !m.accumulate && !m.glu && R > 0 && 2 * R <= NC &&
                       (KS + 3) / 4 >= 2;
    SplitZero z = {};
    if (split) {
        z.y = m.y;
        z.n = m.n; z.j0 = m.j0; z.j1 = m.j1;
        z.first = P - R;
        z.pairs = pairs; z.tiles_n = tiles_n; z.tok = mode == 1 ? tok : tok;
        z.rows = rows_out;
    }
    cudaError_t e = launch_x_to_f16((unsigned)m.n_tokens, s, ss && m.fmt == F_BF16 ? 1 : 0, m.x, m.k,
                                    kp, x16, x16lo, xscale, z,
                                    XGather{});
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
    if (raw_slice_bytes(m.fmt, mode) > 0 && !raw_rowcopy(m.fmt) &&
        !encode_raw_w_map(encode, &tw, m.w, m.fmt, m.row_bytes, m.n))
        return cudaErrorInvalidValue;
    if (ss) {
        // 16-bit W as [n][k] elements, 128-row x 64-wide boxes, 128-byte
        // swizzled: the A operand's shared-memory layout (that of the x tiles)
        const cuuint64_t dims[2] = {(cuuint64_t)m.k, (cuuint64_t)m.n};
        const cuuint64_t strides[1] = {(cuuint64_t)m.row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tw,
                   m.fmt == F_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   2, const_cast<uint8_t *>(m.w), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // y through shared memory and tensor stores: split-x mode, rows of y
    // 16-byte aligned (n % 4 == 0) and the column tile starting on a 16-byte
    // boundary; the map's columns end at j1, so the stores never touch
    // columns outside the tile
    const bool tma_epi = mode == 2 && m.n % 4 == 0 && m.j0 % 4 == 0 &&
                         (reinterpret_cast<uintptr_t>(m.y) & 15u) == 0;
    mp.y = mp.x;
    if (tma_epi) {
        const cuuint64_t dims[2] = {(cuuint64_t)m.j1, (cuuint64_t)m.n_tokens};
        const cuuint64_t strides[1] = {(cuuint64_t)m.n * 4};
        const cuuint32_t box[2] = {32u, 16u};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&mp.y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, m.y, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    MmaHostParams p = {};
    p.tma_epi = tma_epi ? 1 : 0;
    p.w = m.w; p.y = m.y; p.xscale = xscale;
    p.sc = m.sc;
    p.bi = m.bi;
    p.aux_row_bytes = (m.k / 64) * 2;
    p.k = m.k; p.n = m.n; p.n_tokens = m.n_tokens; p.row_bytes = m.row_bytes;
    p.w_rows = m.n;
    p.ss = ss ? 1 : 0;
    p.j0 = m.j0; p.j1 = m.j1;
    p.KS = (int)(kp / kBK);
    p.accumulate = m.accumulate;
    p.err = dev.err;
    p.gate = m.gate;
    p.glu = m.glu;
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

// ------------------------------------------------ expert-grouped products ----

// One block: counts the valid (position, slot) pairs of each expert, lays the
// experts' rows out one after another (row_off[e] .. row_off[e + 1]), gives
// expert e ceil(count / tok) token tiles times `row_pairs` row pairs of
// schedule units (unit_off), and scatters each pair's index to a row of its
// expert (perm). The order within an expert is whatever the atomics give:
// each output row is computed from its own x row alone, so the results do not
// depend on it. Ids outside [0, E) are left out (their y rows untouched) and
// reported through the device error word.
constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads)
    expert_route_kernel(const int32_t *__restrict__ ids, int pairs, int E, int tok, int row_pairs,
                        int *__restrict__ row_off, int *__restrict__ unit_off,
                        int *__restrict__ perm, unsigned int *err) {
    __shared__ int cnt[kMaxGroupedExperts];
    __shared__ int wr[32], wu[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kRouteThreads) cnt[e] = 0;
    __syncthreads();
    for (int i = tid; i < pairs; i += kRouteThreads) {
        const int e = ids[i];
        if (e >= 0 && e < E)
            atomicAdd(&cnt[e], 1);
        else
            record_error(err, DERR_BAD_ID);
    }
    __syncthreads();
    // exclusive scans of rows and units: thread t takes experts [t * per, +per)
    const int per = (E + kRouteThreads - 1) / kRouteThreads;
    const int e0 = tid * per;
    int sr = 0, su = 0;
    for (int j = 0; j < per; ++j) {
        const int e = e0 + j;
        if (e < E) {
            sr += cnt[e];
            su += (cnt[e] + tok - 1) / tok * row_pairs;
        }
    }
    int ir = sr, iu = su;  // inclusive within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xFFFFFFFFu, ir, o), b = __shfl_up_sync(0xFFFFFFFFu, iu, o);
        if (lane >= o) { ir += a; iu += b; }
    }
    if (lane == 31) { wr[warp] = ir; wu[warp] = iu; }
    __syncthreads();
    if (warp == 0) {
        int a = wr[lane], b = wu[lane];  // 32 warps of 32 threads
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int c = __shfl_up_sync(0xFFFFFFFFu, a, o), d = __shfl_up_sync(0xFFFFFFFFu, b, o);
            if (lane >= o) { a += c; b += d; }
        }
        wr[lane] = a;
        wu[lane] = b;
    }
    __syncthreads();
    int br = (warp ? wr[warp - 1] : 0) + ir - sr, bu = (warp ? wu[warp - 1] : 0) + iu - su;
    for (int j = 0; j < per; ++j) {
        const int e = e0 + j;
        if (e < E) {
            const int c = cnt[e];
            row_off[e] = br;
            unit_off[e] = bu;
            cnt[e] = br;  // becomes the expert's scatter cursor
            br += c;
            bu += (c + tok - 1) / tok * row_pairs;
        }
    }
    if (tid == kRouteThreads - 1) {
        row_off[E] = wr[31];
        unit_off[E] = wu[31];
    }
    __syncthreads();
    for (int i = tid; i < pairs; i += kRouteThreads) {
        const int e = ids[i];
        if (e >= 0 && e < E) perm[atomicAdd(&cnt[e], 1)] = i;
    }
}

int grouped_token_tile(int64_t pairs, int64_t n_experts) {
    const int64_t avg = (pairs + n_experts - 1) / n_experts;
    int tok = 16;
    while (tok < avg && tok < 128) tok <<= 1;
    return tok;
}

size_t mma_grouped_workspace_bytes(int fmt, int64_t pairs, int64_t k, int64_t n_experts) {
    return mma_workspace_bytes(fmt, pairs, k) + 2 * round256((size_t)(n_experts + 1) * 4) +
           round256((size_t)pairs * 4);
}

cudaError_t launch_mma_grouped(const MmaGroupedLaunch &m, const DeviceInfo &dev, cudaStream_t s) {
    const int64_t M = m.j1 - m.j0;
    const int64_t P = m.n_pos * m.top_k;
    if (M <= 0 || P <= 0) return cudaSuccess;
    if (mma_mode(m.fmt, m.k) != 2 || is_affine(m.fmt) || m.n_experts > kMaxGroupedExperts)
        return cudaErrorNotSupported;
    EncodeTiledFn encode = get_encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const int64_t kp = kpad(m.k);
    const size_t one = round256((size_t)P * kp * 2);
    uint8_t *ws = reinterpret_cast<uint8_t *>(m.workspace);
    __half *x16 = reinterpret_cast<__half *>(ws);
    __half *x16lo = reinterpret_cast<__half *>(ws + one);
    float *xscale = reinterpret_cast<float *>(ws + 2 * one);
    uint8_t *tail = ws + 2 * one + round256((size_t)P * 4);
    const size_t eb = round256((size_t)(m.n_experts + 1) * 4);
    int *row_off = reinterpret_cast<int *>(tail);
    int *unit_off = reinterpret_cast<int *>(tail + eb);
    int *perm = reinterpret_cast<int *>(tail + 2 * eb);
    const int tok = grouped_token_tile(P, m.n_experts);
    const int bn = 2 * tok;
    const int64_t tiles_m = (M + kBM - 1) / kBM;
    const int row_pairs = (int)((tiles_m + 1) / 2);
    expert_route_kernel<<<1, kRouteThreads, 0, s>>>(m.ids, (int)P, (int)m.n_experts, tok,
                                                     row_pairs, row_off, unit_off, perm, dev.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    XGather gx;
    gx.src = perm;
    gx.count = row_off + m.n_experts;
    gx.top_k = (int)m.top_k;
    {
        const cudaError_t ce =
            launch_x_to_f16((unsigned)P, s, 0, m.x, m.k, kp, x16, x16lo, xscale, SplitZero{}, gx);
        if (ce != cudaSuccess) return ce;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    Maps mp;
    if (!encode_x_map(encode, &mp.x, x16, kp, P, bn / 2) ||
        !encode_x_map(encode, &mp.xlo, x16lo, kp, P, bn / 2))
        return cudaErrorInvalidValue;
    mp.w = mp.x;
    mp.y = mp.x;  // rows of y are scattered: stored from registers
    // the stacked slices as one 2-D tensor [n_experts * n][row_bytes]
    if (raw_slice_bytes(m.fmt, 2) > 0 && !raw_rowcopy(m.fmt) &&
        !encode_raw_w_map(encode, &mp.w, m.w, m.fmt, m.row_bytes, m.n * m.n_experts))
        return cudaErrorInvalidValue;
    MmaHostParams p = {};
    p.w = m.w; p.y = m.y; p.xscale = xscale;
    p.k = m.k; p.n = m.n; p.n_tokens = P; p.row_bytes = m.row_bytes;
    p.w_rows = m.n * m.n_experts;
    p.j0 = m.j0; p.j1 = m.j1;
    p.KS = (int)(kp / kBK);
    p.accumulate = m.accumulate;
    p.err = dev.err;
    p.pairs = row_pairs;
    p.tiles_n = 1;
    p.split = 1;
    // an upper bound on the routed units (each expert with rows adds at most
    // one partial token tile): the grid size; the kernel reads the count
    const int64_t bound = (int64_t)row_pairs * ((P + tok - 1) / tok + std::min<int64_t>(m.n_experts, P));
    p.n_units = (int)std::min<int64_t>(bound, 1 << 30);
    p.full_units = p.n_units;
    p.row_off = row_off;
    p.unit_off = unit_off;
    p.perm = perm;
    p.n_experts = (int)m.n_experts;
    p.slice_rows = m.n;
    switch (m.fmt) {
    case F_BF16: return launch_fmt_grouped<F_BF16>(bn, mp, p, dev, s);
    case F_F16: return launch_fmt_grouped<F_F16>(bn, mp, p, dev, s);
    case F_Q4_0: return launch_fmt_grouped<F_Q4_0>(bn, mp, p, dev, s);
    case F_Q4_K: return launch_fmt_grouped<F_Q4_K>(bn, mp, p, dev, s);
    case F_Q6_K: return launch_fmt_grouped<F_Q6_K>(bn, mp, p, dev, s);
    case F_Q8_0: return launch_fmt_grouped<F_Q8_0>(bn, mp, p, dev, s);
    case F_Q5_0: return launch_fmt_grouped<F_Q5_0>(bn, mp, p, dev, s);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace qmm
