// qmm_api.cu -- the C ABI declared in include/qmm.h: host-side validation,
// path policy, workspace, stream handling and error reporting. Launches only;
// no host synchronisation on the compute path.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "qmm.h"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace {

// Device error word: kernels record the first barrier timeout here.
__device__ unsigned int g_err_word;

thread_local char t_err[512] = "";
thread_local cudaStream_t t_stream = nullptr;

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return status;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
qmm::DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices];

// Library-owned grow-only workspace per device (used when the caller passes none).
void *g_ws[kMaxDevices];
size_t g_ws_bytes[kMaxDevices];

// Largest token count for which the GEMV path (one launch per token) is used
// by default; above it the tensor-core path wins. Measured on the Q4_K FFN
// shape (k = 4096, n = 14336): one GEMV 10.7 us, so two tokens 21.5 us against
// 20.4-21.0 us for the tensor-core call at N <= 32 (two tokens stay on the
// GEMV, within 5 %, for its exact fp32 products); three tokens 32 us.
constexpr int64_t kGemvMaxTokens = 2;
// With QMM_FLAG_SPLIT_W (a quantized W carried as two fp16 terms on the
// tensor cores, precision mode 3) the tensor-core call costs about ten
// GEMVs at these sizes (Q4_K k = 4096, n = 14336: 106 us at 8 tokens, one
// GEMV 10.7 us), and the GEMV's fp32 products are exact: up to 8 tokens take
// one GEMV each.
constexpr int64_t kGemvMaxTokensSplitW = 8;

int device_info(qmm::DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(QMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(QMM_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_ok[dev]) {
        qmm::DeviceInfo d;
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess)
            return fail(QMM_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
        d.sm_count = prop.multiProcessorCount;
        d.major = prop.major;
        d.minor = prop.minor;
        d.smem_optin = prop.sharedMemPerBlockOptin;
        if (d.major != 10 || d.minor != 3)
            return fail(QMM_ERR_UNSUPPORTED,
                        "libqmm is built for sm_103a only; device %d is compute capability %d.%d",
                        dev, d.major, d.minor);
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_err_word);
        if (e != cudaSuccess)
            return fail(QMM_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        d.err = static_cast<unsigned int *>(p);
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    *out = &g_dev[dev];
    return QMM_OK;
}

int64_t row_bytes_of(int fmt, int64_t k) {
    switch (fmt) {
    case QMM_BF16:
    case QMM_F16: return (k % 2 == 0) ? 2 * k : -1;
    case QMM_Q4_0: return (k % 32 == 0) ? (k / 32) * 18 : -1;
    case QMM_Q4_K: return (k % 256 == 0) ? (k / 256) * 144 : -1;
    case QMM_Q6_K: return (k % 256 == 0) ? (k / 256) * 210 : -1;
    case QMM_Q8_0: return (k % 32 == 0) ? (k / 32) * 34 : -1;
    case QMM_Q5_0: return (k % 32 == 0) ? (k / 32) * 22 : -1;
    case QMM_AFFINE4: return (k % 64 == 0) ? k / 2 : -1;
    case QMM_AFFINE8: return (k % 64 == 0) ? k : -1;
    default: return -1;
    }
}

const char *fmt_name(int fmt) {
    static const char *names[] = {"BF16", "F16", "Q4_0", "Q4_K", "Q6_K", "Q8_0", "Q5_0",
                                  "AFFINE4", "AFFINE8"};
    return (fmt >= 0 && fmt <= 8) ? names[fmt] : "?";
}

// Shape/pointer validation shared by the entry points. On success fills the
// effective tile and row bytes.
int validate(const qmm_args *a, int64_t *j0, int64_t *j1, int64_t *rb, bool check_ptrs) {
    if (!a) return fail(QMM_ERR_NULL, "args is NULL");
    if (a->fmt < QMM_BF16 || a->fmt > QMM_AFFINE8)
        return fail(QMM_ERR_FORMAT, "unknown format code %d", a->fmt);
    if (a->k < 0 || a->n < 0) return fail(QMM_ERR_SHAPE, "negative k or n (k=%lld n=%lld)",
                                          (long long)a->k, (long long)a->n);
    if (a->n_tokens < 1) return fail(QMM_ERR_SHAPE, "n_tokens %lld < 1", (long long)a->n_tokens);
    const int64_t r = row_bytes_of(a->fmt, a->k);
    if (r < 0) {
        const char *need = (a->fmt == QMM_Q4_0 || a->fmt == QMM_Q8_0 || a->fmt == QMM_Q5_0)
                               ? "a multiple of 32"
                           : (a->fmt == QMM_Q4_K || a->fmt == QMM_Q6_K) ? "a multiple of 256"
                           : (a->fmt == QMM_AFFINE4 || a->fmt == QMM_AFFINE8) ? "a multiple of 64"
                                                                              : "even";
        return fail(QMM_ERR_SHAPE, "k %lld must be %s for %s matmul", (long long)a->k, need,
                    fmt_name(a->fmt));
    }
    if (a->w_len != 0 && a->w_len != (size_t)(r * a->n))
        return fail(QMM_ERR_SIZE, "%s W bytes %zu != row_bytes*n = %lld", fmt_name(a->fmt),
                    a->w_len, (long long)(r * a->n));
    int64_t s = a->j_start, e = a->j_end;
    if (s == 0 && e == 0) e = a->n;
    if (s < 0 || s > e || e > a->n)
        return fail(QMM_ERR_RANGE, "tile [%lld, %lld) not within [0, %lld]", (long long)s,
                    (long long)e, (long long)a->n);
    *j0 = s;
    *j1 = e;
    *rb = r;
    if (check_ptrs && e > s) {
        if (!a->y) return fail(QMM_ERR_NULL, "y is NULL");
        if (a->k > 0 && (!a->w || !a->x)) return fail(QMM_ERR_NULL, "w or x is NULL");
        if (a->k > 0 && (reinterpret_cast<uintptr_t>(a->w) & 15u))
            return fail(QMM_ERR_ALIGN, "w must be 16-byte aligned");
        if ((a->k > 0 && (reinterpret_cast<uintptr_t>(a->x) & 3u)) ||
            (reinterpret_cast<uintptr_t>(a->y) & 3u))
            return fail(QMM_ERR_ALIGN, "x and y must be 4-byte aligned");
    }
    if (a->path < QMM_PATH_AUTO || a->path > QMM_PATH_MMA)
        return fail(QMM_ERR_SHAPE, "unknown path %d", a->path);
    if (a->flags & ~(QMM_FLAG_OVERLAP_PREV | QMM_FLAG_X_READY | QMM_FLAG_SPLIT_W))
        return fail(QMM_ERR_SHAPE, "unknown flags 0x%x", a->flags);
    return QMM_OK;
}

int choose_path(const qmm_args *a) {
    if (a->path == QMM_PATH_GEMV) return QMM_PATH_GEMV;
    if (a->path == QMM_PATH_MMA) return QMM_PATH_MMA;
    const bool split_w = (a->flags & QMM_FLAG_SPLIT_W) && a->fmt != QMM_BF16 && a->fmt != QMM_F16;
    const int64_t gemv_max = split_w ? kGemvMaxTokensSplitW : kGemvMaxTokens;
    if (a->n_tokens <= gemv_max && qmm::gemv_supports(a->fmt, a->k)) return QMM_PATH_GEMV;
    return QMM_PATH_MMA;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(QMM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The library-owned grow-only scratch of the current device, at least `need` bytes.
int library_workspace(size_t need, void **out) {
    int d = 0;
    cudaGetDevice(&d);
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ws_bytes[d] < need) {
        // grow-only; the old buffer may still be in use by queued work
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "workspace grow sync");
        if (g_ws[d]) cudaFree(g_ws[d]);
        g_ws[d] = nullptr;
        g_ws_bytes[d] = 0;
        e = cudaMalloc(&g_ws[d], need);
        if (e != cudaSuccess) return cuda_fail(e, "workspace cudaMalloc");
        g_ws_bytes[d] = need;
    }
    *out = g_ws[d];
    return QMM_OK;
}

bool affine_fmt(int fmt) { return fmt == QMM_AFFINE4 || fmt == QMM_AFFINE8; }

// A caller workspace for the tensor-core path: large enough, 256-byte
// aligned, and device memory of the current device. The kernel reads its x
// tiles from it with tensor copies that the two CTAs of a cluster share, so
// the tensor map must cover this GPU's own memory only (not host, managed
// or another device's memory).
int check_mma_workspace(const void *ws, size_t have, size_t need) {
    if (have < need)
        return fail(QMM_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", have, need);
    if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return fail(QMM_ERR_ALIGN, "workspace must be 256-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(QMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    cudaPointerAttributes at;
    e = cudaPointerGetAttributes(&at, ws);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(QMM_ERR_UNSUPPORTED, "workspace is not CUDA device memory (%s)",
                    cudaGetErrorString(e));
    }
    if (at.type != cudaMemoryTypeDevice || at.device != dev)
        return fail(QMM_ERR_UNSUPPORTED,
                    "workspace must be device memory of the current device %d (memory type %d, "
                    "device %d)",
                    dev, (int)at.type, at.device);
    return QMM_OK;
}

// The product of every entry point. Affine formats come with their scale and
// bias arrays (sc, bi), which only qmm_matmul_affine passes (affine_entry).
int run(const qmm_args *a, const void *sc = nullptr, const void *bi = nullptr,
        bool affine_entry = false) {
    int64_t j0, j1, rb;
    int st = validate(a, &j0, &j1, &rb, true);
    if (st != QMM_OK) return st;
    if (affine_fmt(a->fmt) != affine_entry)
        return fail(QMM_ERR_FORMAT, affine_entry
                                        ? "qmm_matmul_affine takes QMM_AFFINE4 or QMM_AFFINE8"
                                        : "affine weights need their scales and biases: use "
                                          "qmm_matmul_affine");
    if (j1 <= j0) return QMM_OK;
    if (affine_fmt(a->fmt) && a->k > 0) {
        if (!sc || !bi) return fail(QMM_ERR_NULL, "scales or biases is NULL");
        if ((reinterpret_cast<uintptr_t>(sc) & 15u) || (reinterpret_cast<uintptr_t>(bi) & 15u))
            return fail(QMM_ERR_ALIGN, "scales and biases must be 16-byte aligned");
    }
    qmm::DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(a->stream);
    if (a->k == 0) {
        if (a->accumulate) return QMM_OK;
        cudaError_t e = qmm::launch_zero_cols(a->y, a->n_tokens, a->n, j0, j1, s);
        return e == cudaSuccess ? QMM_OK : cuda_fail(e, "zero-fill launch");
    }
    const int path = choose_path(a);
    if (path == QMM_PATH_GEMV) {
        if (!qmm::gemv_supports(a->fmt, a->k))
            return fail(QMM_ERR_UNSUPPORTED, "GEMV path cannot take %s with k=%lld",
                        fmt_name(a->fmt), (long long)a->k);
        for (int64_t t = 0; t < a->n_tokens; ++t) {
            qmm::GemvLaunch g;
            g.fmt = a->fmt;
            g.w = static_cast<const uint8_t *>(a->w);
            g.x = a->x + t * a->k;
            g.y = a->y + t * a->n;
            g.k = a->k; g.n = a->n; g.row_bytes = rb;
            g.j0 = j0; g.j1 = j1;
            g.accumulate = a->accumulate;
            g.overlap_prev = (a->flags & QMM_FLAG_OVERLAP_PREV) != 0;
            g.x_ready = g.overlap_prev && (a->flags & QMM_FLAG_X_READY) != 0;
            g.sc = static_cast<const uint8_t *>(sc);
            g.bi = static_cast<const uint8_t *>(bi);
            cudaError_t e = qmm::launch_gemv(g, *dev, s);
            if (e != cudaSuccess) return cuda_fail(e, "GEMV launch");
        }
        return QMM_OK;
    }
    const size_t need = qmm::mma_workspace_bytes(a->fmt, a->n_tokens, a->k);
    void *ws = a->workspace;
    if (ws) {
        st = check_mma_workspace(ws, a->workspace_bytes, need);
        if (st != QMM_OK) return st;
    } else {
        st = library_workspace(need, &ws);
        if (st != QMM_OK) return st;
    }
    qmm::MmaLaunch m;
    m.fmt = a->fmt;
    m.w = static_cast<const uint8_t *>(a->w);
    m.x = a->x;
    m.y = a->y;
    m.k = a->k; m.n = a->n; m.n_tokens = a->n_tokens; m.row_bytes = rb;
    m.j0 = j0; m.j1 = j1;
    m.accumulate = a->accumulate;
    m.workspace = ws;
    m.sc = static_cast<const uint8_t *>(sc);
    m.bi = static_cast<const uint8_t *>(bi);
    m.split_w = (a->flags & QMM_FLAG_SPLIT_W) != 0;
    cudaError_t e = qmm::launch_mma(m, *dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core launch");
    return QMM_OK;
}

size_t round256_bytes(size_t v) { return (v + 255) & ~(size_t)255; }

// One token on the GEMV path: the fused gated GEMV; otherwise the gate
// product into scratch, then the up product whose epilogue applies the
// activation to the gate values and writes y.
bool glu_fused(const qmm_args *a) {
    return a->n_tokens == 1 && a->path != QMM_PATH_MMA && qmm::gemv_supports(a->fmt, a->k);
}

size_t glu_scratch_bytes(const qmm_args *a) {
    const size_t one = round256_bytes((size_t)a->n_tokens * (size_t)a->n * 4);
    return one + qmm::mma_workspace_bytes(a->fmt, a->n_tokens, a->k);
}
// Whether an expert-indexed call runs as the grouped tensor-core product
// (pairs routed by expert on the device, one pass over the sorted rows) or
// as one GEMV per (position, slot). The grouped form takes GGUF formats whose
// k the split-x tensor-core mode takes. AUTO groups the formats whose W tiles
// stream raw by TMA (Q4_K, Q8_0, Q5_0, Q4_0) once there are several positions
// and on average at least two pairs per expert (top 8 of 64 experts, k = 2048,
// n = 768; 64 positions: Q4_K 37 against 189 us in the per-pair GEMV form,
// Q8_0 46 against 211, Q5_0 60 against 222; 16 positions: Q4_K 36 against 53,
// Q8_0 42 against 60). Q6_K's grouped form costs about the same from 16
// positions on (its exact fp32 decode paces it: 106-109 us from 16 to 64
// positions, against 67, 131, 204 and 255 us per pair at 16, 24, 40 and 64),
// so it groups from three pairs per expert.
// With QMM_FLAG_SPLIT_W the pairs take the GEMV (exact fp32 products).
bool experts_grouped_ok(const qmm_args *a, int64_t n_experts) {
    return !affine_fmt(a->fmt) && a->k > 0 && qmm::mma_mode(a->fmt, a->k) == 2 &&
           !(a->flags & QMM_FLAG_SPLIT_W) && n_experts <= qmm::kMaxGroupedExperts;
}
bool experts_grouped(const qmm_args *a, int64_t n_experts, int64_t top_k) {
    if (a->path == QMM_PATH_GEMV || !experts_grouped_ok(a, n_experts)) return false;
    if (a->path == QMM_PATH_MMA) return true;
    if (a->n_tokens <= 1) return false;
    const int64_t pairs = a->n_tokens * top_k;
    if (a->fmt == QMM_Q6_K) return pairs >= 3 * n_experts;
    const bool raw_tiles = a->fmt == QMM_Q4_K || a->fmt == QMM_Q8_0 || a->fmt == QMM_Q5_0 ||
                           a->fmt == QMM_Q4_0;
    return raw_tiles && pairs >= 2 * n_experts;
}

// The expert-indexed product of both entry points; affine matrices come with
// their stacked scale and bias arrays (affine_entry).
int experts_impl(const qmm_args *a, const int32_t *ids, int64_t n_experts, int64_t top_k,
                 const void *sc, const void *bi, bool affine_entry) {
    if (!a) return fail(QMM_ERR_NULL, "args is NULL");
    if (n_experts < 1 || top_k < 1)
        return fail(QMM_ERR_SHAPE, "n_experts %lld and top_k %lld must be >= 1",
                    (long long)n_experts, (long long)top_k);
    if (a->path == QMM_PATH_MMA && !experts_grouped_ok(a, n_experts))
        return fail(QMM_ERR_UNSUPPORTED,
                    "the grouped tensor-core expert product takes GGUF formats with k >= 1024 "
                    "and at most %d experts", qmm::kMaxGroupedExperts);
    if (affine_fmt(a->fmt) != affine_entry)
        return fail(QMM_ERR_FORMAT, affine_entry
                                        ? "qmm_matmul_experts_affine takes QMM_AFFINE4 or QMM_AFFINE8"
                                        : "affine experts need their scales and biases: use "
                                          "qmm_matmul_experts_affine");
    // shape checks of one expert slice (w_len is checked against all slices below)
    qmm_args one = *a;
    one.w_len = 0;
    int64_t j0, j1, rb;
    int st = validate(&one, &j0, &j1, &rb, true);
    if (st != QMM_OK) return st;
    const int64_t slice = rb * a->n;
    if (a->w_len != 0 && a->w_len != (size_t)(slice * n_experts))
        return fail(QMM_ERR_SIZE, "%s W bytes %zu != n_experts*row_bytes*n = %lld",
                    fmt_name(a->fmt), a->w_len, (long long)(slice * n_experts));
    const int64_t pairs = a->n_tokens * top_k;
    if (pairs > 65535)
        return fail(QMM_ERR_SHAPE, "n_tokens * top_k = %lld exceeds 65535", (long long)pairs);
    if (j1 <= j0) return QMM_OK;
    if (!ids) return fail(QMM_ERR_NULL, "ids is NULL");
    if (reinterpret_cast<uintptr_t>(ids) & 3u) return fail(QMM_ERR_ALIGN, "ids must be 4-byte aligned");
    if (affine_entry && a->k > 0) {
        if (!sc || !bi) return fail(QMM_ERR_NULL, "scales or biases is NULL");
        if ((reinterpret_cast<uintptr_t>(sc) & 15u) || (reinterpret_cast<uintptr_t>(bi) & 15u))
            return fail(QMM_ERR_ALIGN, "scales and biases must be 16-byte aligned");
    }
    if (a->k > 0 && !experts_grouped(a, n_experts, top_k) && !qmm::gemv_supports(a->fmt, a->k))
        return fail(QMM_ERR_UNSUPPORTED, "expert GEMV cannot take %s with k=%lld", fmt_name(a->fmt),
                    (long long)a->k);
    qmm::DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(a->stream);
    if (a->k == 0) {
        if (a->accumulate) return QMM_OK;
        cudaError_t e = qmm::launch_zero_cols(a->y, pairs, a->n, j0, j1, s);
        return e == cudaSuccess ? QMM_OK : cuda_fail(e, "zero-fill launch");
    }
    if (experts_grouped(a, n_experts, top_k)) {
        const size_t need = qmm::mma_grouped_workspace_bytes(a->fmt, pairs, a->k, n_experts);
        void *ws = a->workspace;
        if (ws) {
            st = check_mma_workspace(ws, a->workspace_bytes, need);
            if (st != QMM_OK) return st;
        } else {
            st = library_workspace(need, &ws);
            if (st != QMM_OK) return st;
        }
        qmm::MmaGroupedLaunch m;
        m.fmt = a->fmt;
        m.w = static_cast<const uint8_t *>(a->w);
        m.x = a->x;
        m.ids = ids;
        m.y = a->y;
        m.k = a->k; m.n = a->n; m.n_pos = a->n_tokens; m.top_k = top_k;
        m.n_experts = n_experts; m.row_bytes = rb;
        m.j0 = j0; m.j1 = j1;
        m.accumulate = a->accumulate;
        m.workspace = ws;
        cudaError_t e = qmm::launch_mma_grouped(m, *dev, s);
        return e == cudaSuccess ? QMM_OK : cuda_fail(e, "grouped expert launch");
    }
    qmm::GemvLaunch g;
    g.fmt = a->fmt;
    g.w = static_cast<const uint8_t *>(a->w);
    g.x = a->x;
    g.y = a->y;
    g.k = a->k; g.n = a->n; g.row_bytes = rb;
    g.j0 = j0; g.j1 = j1;
    g.accumulate = a->accumulate;
    g.overlap_prev = (a->flags & QMM_FLAG_OVERLAP_PREV) != 0;
    g.x_ready = g.overlap_prev && (a->flags & QMM_FLAG_X_READY) != 0;
    g.ids = ids;
    g.sc = static_cast<const uint8_t *>(sc);
    g.bi = static_cast<const uint8_t *>(bi);
    g.n_experts = (int)n_experts;
    g.top_k = (int)top_k;
    g.pairs = (int)pairs;
    cudaError_t e = qmm::launch_gemv(g, *dev, s);
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "expert GEMV launch");
}

}  // namespace

namespace qmm {
int set_error(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return status;
}
}  // namespace qmm

extern "C" {

size_t qmm_weight_bytes(int fmt, int64_t k, int64_t n) {
    if (k < 0 || n < 0) return 0;
    const int64_t r = row_bytes_of(fmt, k);
    return r < 0 ? 0 : (size_t)(r * n);
}

void qmm_set_stream(void *stream) { t_stream = static_cast<cudaStream_t>(stream); }

int qmm_matmul(int fmt, const void *w, const float *x, int64_t k, int64_t n, int64_t n_tokens,
               float *y) {
    qmm_args a;
    std::memset(&a, 0, sizeof a);
    a.fmt = fmt;
    a.w = w;
    a.x = x;
    a.y = y;
    a.k = k;
    a.n = n;
    a.n_tokens = n_tokens;
    a.stream = t_stream;
    t_err[0] = 0;
    return run(&a);
}

int qmm_matmul_ex(const qmm_args *a) {
    t_err[0] = 0;
    return run(a);
}

size_t qmm_workspace_bytes(const qmm_args *a) {
    int64_t j0, j1, rb;
    if (validate(a, &j0, &j1, &rb, false) != QMM_OK) return 0;
    if (a->k == 0 || j1 <= j0 || choose_path(a) != QMM_PATH_MMA) return 0;
    return qmm::mma_workspace_bytes(a->fmt, a->n_tokens, a->k);
}

int qmm_select_path(const qmm_args *a) {
    int64_t j0, j1, rb;
    if (validate(a, &j0, &j1, &rb, false) != QMM_OK) return -1;
    return choose_path(a);
}

int qmm_matmul_host(const qmm_args *a, void *dev_w, float *dev_x, float *dev_y) {
    t_err[0] = 0;
    int64_t j0, j1, rb;
    int st = validate(a, &j0, &j1, &rb, true);
    if (st != QMM_OK) return st;
    if (j1 <= j0) return QMM_OK;
    if (!dev_w || !dev_x || !dev_y) return fail(QMM_ERR_NULL, "device staging buffer is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(a->stream);
    const size_t wb = (size_t)(rb * a->n), xb = (size_t)(a->k * a->n_tokens) * 4,
                 yb = (size_t)(a->n * a->n_tokens) * 4;
    cudaError_t e;
    if (wb && (e = cudaMemcpyAsync(dev_w, a->w, wb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "copy W to device");
    if (xb && (e = cudaMemcpyAsync(dev_x, a->x, xb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "copy x to device");
    if (a->accumulate &&
        (e = cudaMemcpyAsync(dev_y, a->y, yb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "copy y to device");
    qmm_args d = *a;
    d.w = dev_w;
    d.x = dev_x;
    d.y = dev_y;
    st = run(&d);
    if (st != QMM_OK) return st;
    if ((e = cudaMemcpyAsync(a->y, dev_y, yb, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "copy y to host");
    return QMM_OK;
}

int qmm_matmul_backward_input(const qmm_args *a) {
    t_err[0] = 0;
    if (!a) return fail(QMM_ERR_NULL, "args is NULL");
    if (a->n_tokens != 1)
        return fail(QMM_ERR_SHAPE, "backward-input takes one dy vector (n_tokens %lld != 1)",
                    (long long)a->n_tokens);
    if (affine_fmt(a->fmt))
        return fail(QMM_ERR_FORMAT, "backward-input takes single-stream (GGUF) formats");
    int64_t j0, j1, rb;
    // x = dy (n entries), y = dx (k entries): the pointer checks of validate()
    // hold for the swapped lengths too
    int st = validate(a, &j0, &j1, &rb, true);
    if (st != QMM_OK) return st;
    if (a->k == 0) return QMM_OK;
    if (!a->y) return fail(QMM_ERR_NULL, "dx (y) is NULL");
    if (a->n > 0 && (!a->w || !a->x)) return fail(QMM_ERR_NULL, "w or dy (x) is NULL");
    if (!qmm::back_input_supports(a->fmt, a->k))
        return fail(QMM_ERR_UNSUPPORTED, "backward-input cannot take %s with k=%lld",
                    fmt_name(a->fmt), (long long)a->k);
    qmm::DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(a->stream);
    if (j1 <= j0) {  // empty sum: dx = 0, or unchanged when accumulating
        if (a->accumulate) return QMM_OK;
        cudaError_t e = qmm::launch_zero_cols(a->y, 1, a->k, 0, a->k, s);
        return e == cudaSuccess ? QMM_OK : cuda_fail(e, "zero-fill launch");
    }
    const size_t need = qmm::back_input_workspace_bytes(a->fmt, a->k, a->n, j0, j1, *dev);
    void *ws = a->workspace;
    if (ws) {
        if (a->workspace_bytes < need)
            return fail(QMM_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", a->workspace_bytes,
                        need);
        if (reinterpret_cast<uintptr_t>(ws) & 255u)
            return fail(QMM_ERR_ALIGN, "workspace must be 256-byte aligned");
    } else {
        st = library_workspace(need, &ws);
        if (st != QMM_OK) return st;
    }
    qmm::BackLaunch b;
    b.fmt = a->fmt;
    b.w = static_cast<const uint8_t *>(a->w);
    b.dy = a->x;
    b.dx = a->y;
    b.k = a->k; b.n = a->n; b.row_bytes = rb;
    b.j0 = j0; b.j1 = j1;
    b.accumulate = a->accumulate;
    b.workspace = ws;
    b.overlap_prev = (a->flags & QMM_FLAG_OVERLAP_PREV) != 0;
    b.x_ready = b.overlap_prev && (a->flags & QMM_FLAG_X_READY) != 0;
    cudaError_t e = qmm::launch_back_input(b, *dev, s);
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "backward-input launch");
}

int qmm_matmul_experts(const qmm_args *a, const int32_t *ids, int64_t n_experts, int64_t top_k) {
    t_err[0] = 0;
    return experts_impl(a, ids, n_experts, top_k, nullptr, nullptr, false);
}

size_t qmm_experts_workspace_bytes(const qmm_args *a, int64_t n_experts, int64_t top_k) {
    if (!a || n_experts < 1 || top_k < 1) return 0;
    qmm_args one = *a;
    one.w_len = 0;
    int64_t j0, j1, rb;
    if (validate(&one, &j0, &j1, &rb, false) != QMM_OK || a->k == 0 || j1 <= j0) return 0;
    if (!experts_grouped(a, n_experts, top_k)) return 0;
    return qmm::mma_grouped_workspace_bytes(a->fmt, a->n_tokens * top_k, a->k, n_experts);
}

int qmm_matmul_experts_affine(const qmm_args *a, const int32_t *ids, int64_t n_experts,
                              int64_t top_k, const void *scales, const void *biases) {
    t_err[0] = 0;
    return experts_impl(a, ids, n_experts, top_k, scales, biases, true);
}

size_t qmm_backward_input_workspace_bytes(const qmm_args *a) {
    int64_t j0, j1, rb;
    if (!a || a->n_tokens != 1 || validate(a, &j0, &j1, &rb, false) != QMM_OK) return 0;
    if (a->k == 0 || j1 <= j0 || !qmm::back_input_supports(a->fmt, a->k)) return 0;
    qmm::DeviceInfo *dev = nullptr;
    if (device_info(&dev) != QMM_OK) return 0;
    return qmm::back_input_workspace_bytes(a->fmt, a->k, a->n, j0, j1, *dev);
}

int qmm_dequant(int fmt, const void *w, int64_t k, int64_t n, float *out, void *stream) {
    t_err[0] = 0;
    if (affine_fmt(fmt))
        return fail(QMM_ERR_FORMAT, "%s weights need their scales and biases: use qmm_dequant_affine",
                    fmt_name(fmt));
    if (fmt < QMM_BF16 || fmt > QMM_Q5_0) return fail(QMM_ERR_FORMAT, "unknown format code %d", fmt);
    if (k < 0 || n < 0) return fail(QMM_ERR_SHAPE, "negative k or n");
    const int64_t r = row_bytes_of(fmt, k);
    if (r < 0) return fail(QMM_ERR_SHAPE, "k %lld does not fit %s blocks", (long long)k, fmt_name(fmt));
    if (k == 0 || n == 0) return QMM_OK;
    if (!w || !out) return fail(QMM_ERR_NULL, "w or out is NULL");
    if ((reinterpret_cast<uintptr_t>(w) & 15u)) return fail(QMM_ERR_ALIGN, "w must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(out) & 3u)) return fail(QMM_ERR_ALIGN, "out must be 4-byte aligned");
    qmm::DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaError_t e = qmm::launch_dequant(fmt, static_cast<const uint8_t *>(w), k, n, r, out,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "dequant launch");
}


size_t qmm_glu_workspace_bytes(const qmm_args *a) {
    int64_t j0, j1, rb;
    if (!a || affine_fmt(a->fmt) || validate(a, &j0, &j1, &rb, false) != QMM_OK) return 0;
    if (a->k == 0 || j1 <= j0 || glu_fused(a)) return 0;
    return glu_scratch_bytes(a);
}

int qmm_matmul_glu(const qmm_args *a, const void *w_up, int act) {
    t_err[0] = 0;
    if (!a) return fail(QMM_ERR_NULL, "args is NULL");
    if (act != QMM_ACT_SWIGLU && act != QMM_ACT_GEGLU)
        return fail(QMM_ERR_FORMAT, "unknown activation %d", act);
    if (affine_fmt(a->fmt))
        return fail(QMM_ERR_FORMAT, "gated products take single-stream (GGUF) formats");
    int64_t j0, j1, rb;
    int st = validate(a, &j0, &j1, &rb, true);
    if (st != QMM_OK) return st;
    if (j1 <= j0) return QMM_OK;
    if (a->k > 0) {
        if (!w_up) return fail(QMM_ERR_NULL, "w_up is NULL");
        if (reinterpret_cast<uintptr_t>(w_up) & 15u)
            return fail(QMM_ERR_ALIGN, "w_up must be 16-byte aligned");
    }
    if (a->n_tokens == 1 && a->path == QMM_PATH_GEMV && !qmm::gemv_supports(a->fmt, a->k))
        return fail(QMM_ERR_UNSUPPORTED, "GEMV path cannot take %s with k=%lld", fmt_name(a->fmt),
                    (long long)a->k);
    qmm::DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(a->stream);
    if (a->k == 0) {  // gate = up = 0: y = 0 (unchanged when accumulating)
        if (a->accumulate) return QMM_OK;
        cudaError_t e = qmm::launch_zero_cols(a->y, a->n_tokens, a->n, j0, j1, s);
        return e == cudaSuccess ? QMM_OK : cuda_fail(e, "zero-fill launch");
    }
    if (glu_fused(a)) {
        qmm::GemvLaunch g;
        g.fmt = a->fmt;
        g.w = static_cast<const uint8_t *>(a->w);
        g.w2 = static_cast<const uint8_t *>(w_up);
        g.glu = act;
        g.x = a->x;
        g.y = a->y;
        g.k = a->k; g.n = a->n; g.row_bytes = rb;
        g.j0 = j0; g.j1 = j1;
        g.accumulate = a->accumulate;
        g.overlap_prev = (a->flags & QMM_FLAG_OVERLAP_PREV) != 0;
        g.x_ready = g.overlap_prev && (a->flags & QMM_FLAG_X_READY) != 0;
        cudaError_t e = qmm::launch_gemv(g, *dev, s);
        return e == cudaSuccess ? QMM_OK : cuda_fail(e, "gated GEMV launch");
    }
    const size_t need = glu_scratch_bytes(a);
    void *ws = a->workspace;
    if (ws) {
        st = check_mma_workspace(ws, a->workspace_bytes, need);
        if (st != QMM_OK) return st;
    } else {
        st = library_workspace(need, &ws);
        if (st != QMM_OK) return st;
    }
    const size_t one = round256_bytes((size_t)a->n_tokens * (size_t)a->n * 4);
    float *gbuf = static_cast<float *>(ws);
    void *mws = static_cast<uint8_t *>(ws) + one;
    // gate = x Wg into scratch; then y (+)= act(gate) * (x Wu) in the up
    // product's epilogue (no up vector is stored, no combine launch)
    for (int m = 0; m < 2; ++m) {
        qmm::MmaLaunch ml;
        ml.fmt = a->fmt;
        ml.w = static_cast<const uint8_t *>(m ? w_up : a->w);
        ml.x = a->x;
        ml.y = m ? a->y : gbuf;
        ml.k = a->k; ml.n = a->n; ml.n_tokens = a->n_tokens; ml.row_bytes = rb;
        ml.j0 = j0; ml.j1 = j1;
        ml.accumulate = m ? a->accumulate : 0;
        ml.workspace = mws;
        ml.split_w = (a->flags & QMM_FLAG_SPLIT_W) != 0;
        if (m) {
            ml.gate = gbuf;
            ml.glu = act;
        }
        cudaError_t e = qmm::launch_mma(ml, *dev, s);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core launch");
    }
    return QMM_OK;
}

int qmm_matmul_affine(const qmm_args *a, const void *scales, const void *biases) {
    t_err[0] = 0;
    if (!a) return fail(QMM_ERR_NULL, "args is NULL");
    return run(a, scales, biases, true);
}

int qmm_dequant_affine(int fmt, const void *w, const void *scales, const void *biases, int64_t k,
                       int64_t n, float *out, void *stream) {
    t_err[0] = 0;
    if (!affine_fmt(fmt))
        return fail(QMM_ERR_FORMAT, "qmm_dequant_affine takes QMM_AFFINE4 or QMM_AFFINE8 (got %d)", fmt);
    if (k < 0 || n < 0) return fail(QMM_ERR_SHAPE, "negative k or n");
    const int64_t r = row_bytes_of(fmt, k);
    if (r < 0) return fail(QMM_ERR_SHAPE, "k %lld must be a multiple of 64 for %s", (long long)k,
                           fmt_name(fmt));
    if (k == 0 || n == 0) return QMM_OK;
    if (!w || !scales || !biases || !out) return fail(QMM_ERR_NULL, "w, scales, biases or out is NULL");
    if ((reinterpret_cast<uintptr_t>(w) & 15u)) return fail(QMM_ERR_ALIGN, "w must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(scales) & 1u) || (reinterpret_cast<uintptr_t>(biases) & 1u))
        return fail(QMM_ERR_ALIGN, "scales and biases must be 2-byte aligned");
    if ((reinterpret_cast<uintptr_t>(out) & 3u)) return fail(QMM_ERR_ALIGN, "out must be 4-byte aligned");
    qmm::DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaError_t e = qmm::launch_dequant(fmt, static_cast<const uint8_t *>(w), k, n, r, out,
                                        static_cast<cudaStream_t>(stream),
                                        static_cast<const uint8_t *>(scales),
                                        static_cast<const uint8_t *>(biases));
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "dequant launch");
}

int qmm_check_bounded_wait(void *stream) {
    t_err[0] = 0;
    qmm::DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaError_t e = qmm::launch_bounded_wait_probe(dev->err, 50000000ull /* 50 ms */,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QMM_OK : cuda_fail(e, "bounded-wait check launch");
}

int qmm_device_status(void *stream) {
    t_err[0] = 0;
    qmm::DeviceInfo *dev = nullptr;
    int st = device_info(&dev);
    if (st != QMM_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned int v = 0;
    e = cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (v != 0) {
        const unsigned int zero = 0;
        cudaMemcpy(dev->err, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (v == qmm::DERR_BAD_ID)
            return fail(QMM_ERR_BAD_ID, "an expert id was outside [0, n_experts)");
        return fail(QMM_ERR_DEVICE_TIMEOUT, "a kernel gave up waiting on a pipeline barrier (code %u)", v);
    }
    return QMM_OK;
}

const char *qmm_last_error(void) { return t_err; }

int qmm_version(void) { return 100; }

}  // extern "C"
