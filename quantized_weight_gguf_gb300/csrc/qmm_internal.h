// qmm_internal.h -- host-side interfaces between the C ABI (qmm_api.cu) and
// the kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qmm {

struct DeviceInfo {
    int sm_count = 0;
    int major = 0, minor = 0;
    size_t smem_optin = 0;   // max dynamic shared memory per block
    unsigned int *err = nullptr;  // device error word
};

// One GEMV launch: y[j] (+)= sum_i w[j][i] x[i] for j in [j0, j1), one token.
struct GemvLaunch {
    int fmt;
    const uint8_t *w;
    const float *x;
    float *y;
    int64_t k, n, row_bytes;
    int64_t j0, j1;
    int accumulate;
    bool overlap_prev;   // programmatic dependent launch (W is not written by the previous kernel)
    bool x_ready;        // x is not written by the previous kernel either: only y waits
    // expert-indexed calls: w holds n_experts slices of n rows; GEMV number
    // q < pairs uses slice ids[q], x row q / top_k and y row q (device ids)
    const int32_t *ids = nullptr;
    int n_experts = 0, top_k = 1, pairs = 1;
    // affine formats: bf16 scale and bias arrays [n][k/64]
    const uint8_t *sc = nullptr, *bi = nullptr;
    // gated pair (glu 1: SwiGLU, 2: GeGLU): w is the gate matrix, w2 the up
    // matrix; y = act(x Wg) * (x Wu)
    const uint8_t *w2 = nullptr;
    int glu = 0;
};
// Returns cudaSuccess or the launch error; cudaErrorNotSupported when no
// GEMV variant takes the shape (the caller then uses the tensor-core path).
cudaError_t launch_gemv(const GemvLaunch &g, const DeviceInfo &dev, cudaStream_t s);
bool gemv_supports(int fmt, int64_t k);

// N-token tensor-core product over [j0, j1) for all tokens.
struct MmaLaunch {
    int fmt;
    const uint8_t *w;
    const float *x;
    float *y;
    int64_t k, n, n_tokens, row_bytes;
    int64_t j0, j1;
    int accumulate;
    void *workspace;        // >= mma_workspace_bytes(fmt, n_tokens, k)
    // affine formats: bf16 scale and bias arrays [n][k/64]
    const uint8_t *sc = nullptr, *bi = nullptr;
    // gated pairs (glu 1: SwiGLU, 2: GeGLU): this is the up product, and the
    // epilogue writes act(gate[t][j]) * (x Wu)[t][j] (gate: [N][n], row stride n)
    const float *gate = nullptr;
    int glu = 0;
    // 1: a quantized W is split into two fp16 terms as well (precision mode 3
    // at every k); 16-bit formats are exact in the operand type either way
    int split_w = 0;
};
size_t mma_workspace_bytes(int fmt, int64_t n_tokens, int64_t k);
// precision mode: 2 x split into two fp16 terms, 3 w and x split
int mma_mode(int fmt, int64_t k, bool split_w = false);
cudaError_t launch_mma(const MmaLaunch &m, const DeviceInfo &dev, cudaStream_t s);

// Expert-grouped N-token product: the (position, slot) pairs are routed on
// the device into expert-sorted rows, then one tensor-core pass multiplies
// each expert's rows by its slice; y row p * top_k + s as for the GEMV form.
constexpr int kMaxGroupedExperts = 4096;
struct MmaGroupedLaunch {
    int fmt;
    const uint8_t *w;           // n_experts stacked slices of n rows
    const float *x;             // [n_pos][k]
    const int32_t *ids;         // [n_pos][top_k], device
    float *y;                   // [n_pos * top_k][n]
    int64_t k, n, n_pos, top_k, n_experts, row_bytes;
    int64_t j0, j1;
    int accumulate;
    void *workspace;            // >= mma_grouped_workspace_bytes(...)
};
size_t mma_grouped_workspace_bytes(int fmt, int64_t pairs, int64_t k, int64_t n_experts);
cudaError_t launch_mma_grouped(const MmaGroupedLaunch &m, const DeviceInfo &dev, cudaStream_t s);

// Backward with respect to the input, one vector:
// dx[i] (+)= sum_{j in [j0, j1)} dy[j] w[j][i].
struct BackLaunch {
    int fmt;
    const uint8_t *w;
    const float *dy;        // n entries
    float *dx;              // k entries
    int64_t k, n, row_bytes;
    int64_t j0, j1;         // rows of the sum axis
    int accumulate;
    void *workspace;        // >= back_input_workspace_bytes(...): per-CTA partials
    bool overlap_prev = false;  // programmatic launch (W is not written by the previous kernel)
    bool x_ready = false;       // dy is not written by the previous kernel either
};
bool back_input_supports(int fmt, int64_t k);
size_t back_input_workspace_bytes(int fmt, int64_t k, int64_t n, int64_t j0, int64_t j1,
                                  const DeviceInfo &dev);
cudaError_t launch_back_input(const BackLaunch &b, const DeviceInfo &dev, cudaStream_t s);

// Standalone dequantization of n rows into out[n][k].
// Affine formats pass their bf16 scale and bias arrays ([n][k/64] each).
cudaError_t launch_dequant(int fmt, const uint8_t *w, int64_t k, int64_t n, int64_t row_bytes,
                           float *out, cudaStream_t s, const uint8_t *sc = nullptr,
                           const uint8_t *bi = nullptr);

// y[t][j] = 0 for j in [j0, j1) (k == 0 with accumulate == 0).
cudaError_t launch_zero_cols(float *y, int64_t n_tokens, int64_t n, int64_t j0, int64_t j1,
                             cudaStream_t s);

// One block waiting on a barrier nothing satisfies; it gives up after
// limit_ns and records an error in *err (see qmm_check_bounded_wait).
cudaError_t launch_bounded_wait_probe(unsigned int *err, uint64_t limit_ns, cudaStream_t s);
// Record a status and message for qmm_last_error() on this host thread; returns status.
int set_error(int status, const char *fmt, ...);

}  // namespace qmm
