// qmm_device.cuh -- device-side building blocks shared by the libqmm kernels:
// format geometry, 16-bit float decoding, and thin inline-PTX wrappers for
// mbarriers, bulk / tensor copies (TMA) and the tcgen05 tensor-core path of
// sm_103a. Every barrier wait is bounded by wall-clock time (%globaltimer) so a
// broken pipeline reports an error instead of hanging the GPU.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmm {

enum Fmt : int {
    F_BF16 = 0, F_F16 = 1, F_Q4_0 = 2, F_Q4_K = 3, F_Q6_K = 4, F_Q8_0 = 5, F_Q5_0 = 6,
    F_AFF4 = 7, F_AFF8 = 8  // MLX-style affine: code words + bf16 scale and bias per 64
};
constexpr int kLastFmt = F_Q5_0;  // the last single-stream (GGUF) format
__host__ __device__ constexpr bool is_affine(int f) { return f == F_AFF4 || f == F_AFF8; }

// Error codes written to the device error word (first fault wins).
enum DevErr : unsigned int {
    DERR_NONE = 0,
    DERR_GEMV_FULL = 1,    // GEMV consumer gave up waiting for a stage's bytes
    DERR_GEMV_EMPTY = 2,   // GEMV producer gave up waiting for a free stage
    DERR_MMA_A = 3,        // MMA issuer gave up waiting for a dequantized W tile
    DERR_MMA_B = 4,        // MMA issuer gave up waiting for an x tile
    DERR_MMA_EMPTY = 5,    // a producer gave up waiting for a free stage
    DERR_MMA_ACC = 6,      // epilogue gave up waiting for the accumulator
    DERR_TEARDOWN = 7,     // copies still in flight at exit after a fault
    DERR_BAD_ID = 8,       // an expert id outside [0, n_experts)
    DERR_WAIT_PROBE = 9    // the bounded-wait check gave up, as it must
};

// Block geometry (elements per block, bytes per block) of each format.
__host__ __device__ constexpr int block_elems(int f) {
    return (f == F_Q4_0 || f == F_Q8_0 || f == F_Q5_0) ? 32
           : (f == F_Q4_K || f == F_Q6_K) ? 256
           : is_affine(f) ? 64 : 1;
}
__host__ __device__ constexpr int block_bytes(int f) {
    return f == F_Q4_0 ? 18 : f == F_Q4_K ? 144 : f == F_Q6_K ? 210 : f == F_Q8_0 ? 34
           : f == F_Q5_0 ? 22 : f == F_AFF4 ? 32 : f == F_AFF8 ? 64 : 2;
}

// ------------------------------------------------------------ numbers ----

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) {
    return __uint_as_float(h16 << 16);
}
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h16) {
    return __half2float(__ushort_as_half((unsigned short)h16));
}

// Two fp32 multiply-adds in one packed instruction (sm_100 family f32x2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

// A pair of fp32 values as one 64-bit register (the packed instructions'
// operand form).
__device__ __forceinline__ uint64_t pack_f2(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
// As above with b already packed.
__device__ __forceinline__ float2 ffma2(float2 a, uint64_t b, float2 c) {
    uint64_t ra, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(b), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

// Two fp32 additions in one packed instruction.
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Byte i (0..3) of `v`, which must be < 128, as the float 0.5 + v/256:
// the byte lands in mantissa bits 16..22 under the exponent of 0.5.
template <int I>
__device__ __forceinline__ float byte_half_plus(uint32_t v) {
    return __uint_as_float(prmt(v, 0x3F000000u, 0x7054u | (I << 8)));
}
// Byte i of `v` as the float 2^23 + v (exact for any byte value).
template <int I>
__device__ __forceinline__ float byte_magic23(uint32_t v) {
    return __uint_as_float(prmt(v, 0x4B000000u, 0x7650u | I));
}

// Gate activations of gated FFN pairs, out = act(gate) * up: ACT 1 silu,
// g s(g); ACT 2 GELU in its tanh form, g/2 (1 + tanh z) with z = sqrt(2/pi)
// (g + 0.044715 g^3), evaluated as g s(2z) (the same function:
// 1 + tanh z = 2 s(2z)). The logistic s(t) is taken from e = exp(-|t|)
// (fp32 library exp, never overflows): r = 1 / (1 + e) correctly rounded,
// s = r for t >= 0 and e r for t < 0, so neither tail cancels and there is
// no divergent branch.
__device__ __forceinline__ float glu_arg(int act, float g) {
    return act == 1 ? g : 1.5957691216057308f * fmaf(0.044715f * g, g * g, g);
}
__device__ __forceinline__ float glu_gate(float g, float t) {
    const float e = expf(-fabsf(t));
    const float r = __frcp_rn(1.0f + e);
    return g * (t >= 0.0f ? r : e * r);
}
template <int ACT>
__device__ __forceinline__ float glu_act(float g) {
    return glu_gate(g, glu_arg(ACT, g));
}

// ------------------------------------------------------------- timing ----

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per barrier wait

__device__ __forceinline__ void record_error(unsigned int *err, unsigned int code) {
    if (err) atomicCAS(err, 0u, code);
}

// ------------------------------------------------------------- smem -----

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// Test the phase with parity `parity`; if it has not completed, the thread
// is suspended until it does or about 1 ms passes (no busy polling).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}
// Wait for the phase with parity `parity` to complete; false after
// `limit_ns` (2 s unless a caller asks otherwise).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy ones (tensor-core operand reads, bulk and tensor copies): its
// writes become visible to them, and its reads of a buffer that a copy will
// refill complete first (without it a refill released by an mbarrier arrival
// was seen to overwrite data still being read).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start
// launching / wait until the preceding kernel has completed and flushed.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prev() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 16-byte asynchronous copy global -> shared on the load path (cp.async,
// L1 bypassed), not the tensor-copy unit: `valid` bytes (0..16) are read from
// src, the rest of the 16 are zero-filled. dst and src 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid)
                 : "memory");
}
// One arrival on `bar` once every earlier cp.async of this thread has landed
// (.noinc: it counts against the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 2-D tiled tensor copy global -> shared (TMA) through a tensor map.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 2-D tiled tensor load delivered to the same shared offset of every CTA in
// `mask` within this CTA's cluster, completing bytes on each CTA's `bar`.
__device__ __forceinline__ void tma_load_2d_multicast(uint32_t dst, const void *tmap, int c0, int c1,
                                                      uint32_t bar, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar), "h"(mask)
        : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// 2-D tiled tensor store / reduce-add shared -> global (TMA), bulk-group completion.
__device__ __forceinline__ void tma_store_2d(const void *tmap, int c0, int c1, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap),
        "r"(c0), "r"(c1), "r"(src)
        : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const void *tmap, int c0, int c1, uint32_t src) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            tmap),
        "r"(c0), "r"(c1), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk group has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk group has completed (its writes performed).
__device__ __forceinline__ void bulk_wait_group0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts32f(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Read `NW` consecutive 32-bit words starting at a 2-byte-aligned shared
// address: aligned-down word loads, then a byte permute per word.
template <int NW>
__device__ __forceinline__ void lds_words_a2(uint32_t addr, uint32_t (&out)[NW]) {
    const uint32_t base = addr & ~3u;
    const uint32_t sel = (addr & 2u) ? 0x5432u : 0x3210u;
    uint32_t w[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) w[i] = lds32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < NW; ++i) out[i] = prmt(w[i], w[i + 1], sel);
}

// As lds_words_a2, reading no word past the last byte it returns: an
// aligned address takes NW words, an address 2 mod 4 the NW + 1 that cover
// it (one of them reaching 2 bytes past the data).
template <int NW>
__device__ __forceinline__ void lds_words_a2_exact(uint32_t addr, uint32_t (&out)[NW]) {
    const uint32_t base = addr & ~3u;
    const bool odd = (addr & 2u) != 0;
    const uint32_t sel = odd ? 0x5432u : 0x3210u;
    uint32_t w[NW + 1];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = lds32(base + 4 * i);
    w[NW] = odd ? lds32(base + 4 * NW) : 0u;
#pragma unroll
    for (int i = 0; i < NW; ++i) out[i] = prmt(w[i], w[i + 1], sel);
}

// ------------------------------------------------------------ tcgen05 ----

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, fp16 operands, fp32 accumulator.
__device__ __forceinline__ void tc_mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Load with acquire semantics at GPU scope (pairs with a release or a fence
// + atomic by another CTA).
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(pred));
    return pred != 0;
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M = 128 rows on the 128 TMEM lanes,
// two fp16 of consecutive k per 32-bit column, 8 columns per K = 16), B by
// descriptor, fp32 accumulator.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// As above with A from shared memory too (a K-major, 128-byte swizzled tile
// described like B).
__device__ __forceinline__ void tc_mma_f16_ss(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Registers -> tensor memory: thread t of the warp writes 8 (16) consecutive
// 32-bit columns of TMEM lane (lane field of taddr) + t. The warp may only
// address its own quarter of the lanes: 32 * (warp id % 4) ...
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
// Wait until this thread's tcgen05.st writes have completed.
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}
// As tc_commit, arriving on the barrier at the same offset in every CTA of `mask`.
__device__ __forceinline__ void tc_commit_multicast(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns of tensor memory into registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: 8-row x 128-byte atoms stacked every 1024 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address (16-byte units)
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused with swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset between 8-row groups
    d |= (uint64_t)1 << 46;                    // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                    // swizzle mode: 128-byte
    return d;
}

// Instruction descriptor: kind::f16 with fp16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
    return (1u << 4)                        // D format fp32
           | (0u << 7) | (0u << 10)         // A, B format fp16
           | ((uint32_t)(n >> 3) << 17)     // N / 8
           | ((uint32_t)(m >> 4) << 24);    // M / 16
}
// The same with A and B in bf16.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
    return idesc_f16_f32(m, n) | (1u << 7) | (1u << 10);
}

}  // namespace qmm
