// qmm_dequant.cu -- standalone dequantization (packed bytes -> fp32 [n][k]),
// bit-exact, plus the small helper that zeroes a column tile of y.
#include "qmm_decode.cuh"
#include "qmm_internal.h"

namespace qmm {

// One thread per 32-weight unit (row j, weights 32u .. 32u+31).
// Affine formats also read their scale and bias rows (aux_row_bytes apart).
template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ w, int64_t k,
                                                      int64_t n, int64_t row_bytes,
                                                      float *__restrict__ out,
                                                      const uint8_t *__restrict__ sc,
                                                      const uint8_t *__restrict__ bi,
                                                      int64_t aux_row_bytes) {
    const int64_t units_per_row = (k + 31) / 32;
    const int64_t total = units_per_row * n;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = idx / units_per_row;
        const int64_t u = idx - j * units_per_row;
        const int64_t k0 = 32 * u;
        const int nvalid = (int)((k - k0) < 32 ? (k - k0) : 32);
        Raw32<FMT> raw;
        if constexpr (is_affine(FMT))
            raw.load(w + j * row_bytes, sc + j * aux_row_bytes, bi + j * aux_row_bytes, k0);
        else
            raw.load(w + j * row_bytes, k0, nvalid);
        float v[32];
        raw.decode(v);
        float *o = out + j * k + k0;
        if (nvalid == 32 && (reinterpret_cast<uintptr_t>(o) & 15u) == 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4 *>(o)[q] =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < nvalid) o[i] = v[i];
        }
    }
}

cudaError_t launch_dequant(int fmt, const uint8_t *w, int64_t k, int64_t n, int64_t row_bytes,
                           float *out, cudaStream_t s, const uint8_t *sc, const uint8_t *bi) {
    const int64_t ab = (k / 64) * 2;
    const int64_t total = ((k + 31) / 32) * n;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)1 << 20) blocks = (int64_t)1 << 20;
    const dim3 grid((unsigned)blocks), block(256);
    switch (fmt) {
    case F_BF16: dequant_kernel<F_BF16><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_F16: dequant_kernel<F_F16><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_Q4_0: dequant_kernel<F_Q4_0><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_Q4_K: dequant_kernel<F_Q4_K><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_Q6_K: dequant_kernel<F_Q6_K><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_Q8_0: dequant_kernel<F_Q8_0><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_Q5_0: dequant_kernel<F_Q5_0><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_AFF4: dequant_kernel<F_AFF4><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    case F_AFF8: dequant_kernel<F_AFF8><<<grid, block, 0, s>>>(w, k, n, row_bytes, out, sc, bi, ab); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

__global__ void zero_cols_kernel(float *y, int64_t n_tokens, int64_t n, int64_t j0, int64_t j1) {
    const int64_t width = j1 - j0;
    const int64_t total = width * n_tokens;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / width;
        y[t * n + j0 + (i - t * width)] = 0.0f;
    }
}

cudaError_t launch_zero_cols(float *y, int64_t n_tokens, int64_t n, int64_t j0, int64_t j1,
                             cudaStream_t s) {
    const int64_t total = (j1 - j0) * n_tokens;
    if (total <= 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    zero_cols_kernel<<<(unsigned)blocks, 256, 0, s>>>(y, n_tokens, n, j0, j1);
    return cudaGetLastError();
}

// Check of the bounded waits every pipeline relies on: one thread waits on an
// mbarrier that nothing ever arrives on. The wait gives up after limit_ns,
// the kernel records DERR_WAIT_PROBE and returns: no fault and no hang, and
// the context stays usable.
__global__ void bounded_wait_probe_kernel(unsigned int *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(b, 0, limit_ns)) record_error(err, DERR_WAIT_PROBE);
}

cudaError_t launch_bounded_wait_probe(unsigned int *err, uint64_t limit_ns, cudaStream_t s) {
    bounded_wait_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace qmm
