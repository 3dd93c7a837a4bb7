// qmm_noalloc.cu -- qmm_matmul_noalloc: the tensor-core product for callers
// that cannot allocate device memory themselves (they have no CUDA allocator
// of their own, for instance a host program that reaches libqmm only through
// this C interface, or they must not make the allocation calls, which
// synchronize the device, on their hot path). The scratch that the
// tensor-core path needs (the fp16 copies of x and one scale per token) lives
// in a fixed array in device memory that this library defines, so the call
// allocates nothing.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "qmm.h"
#include "qmm_internal.h"

namespace {

// Every GPU that loads libqmm holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDev];

// Device address of the scratch array on the current device. The array's
// name is only a host-side stand-in in host code; the address comes from the
// runtime, once per device, with that device current.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDev) return QMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return QMM_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QMM_OK;
}

}  // namespace

extern "C" int qmm_matmul_noalloc(const qmm_args *a) {
    if (!a) return qmm_matmul_ex(a);  // reports QMM_ERR_NULL
    qmm_args b;
    std::memcpy(&b, a, sizeof b);
    b.path = QMM_PATH_MMA;
    b.workspace = nullptr;
    b.workspace_bytes = 0;
    if (qmm_select_path(&b) < 0) return qmm_matmul_ex(&b);  // invalid: same status and message
    const size_t need = qmm_workspace_bytes(&b);
    if (need > kNoAllocScratchBytes)
        return qmm::set_error(QMM_ERR_WORKSPACE,
                              "qmm_matmul_noalloc: this call needs %zu bytes of scratch; the "
                              "fixed scratch array holds %zu bytes (reduce n_tokens or k)",
                              need, kNoAllocScratchBytes);
    if (need > 0) {
        void *p = nullptr;
        if (scratch_address(&p) != QMM_OK)
            return qmm::set_error(QMM_ERR_CUDA,
                                  "qmm_matmul_noalloc: cudaGetSymbolAddress of the scratch array failed");
        b.workspace = p;
        b.workspace_bytes = kNoAllocScratchBytes;
    }
    return qmm_matmul_ex(&b);
}
