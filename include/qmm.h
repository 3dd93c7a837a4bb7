/*
 * qmm.h -- C ABI of libqmm: fused dequantize-and-multiply y = x @ W on one
 * NVIDIA GB300 GPU (sm_103a), with W kept in its GGUF/ggml packed bytes.
 *
 * The operation (rullama 0.5.0, src/backend/matmul.rs, module doc and the
 * `matmul_bf16` / `matmul_f16` / `matmul_q4_0` / `matmul_q4_k` /
 * `matmul_q6_k` dispatchers): W is n rows of k weights, row-major; row j
 * holds the k weights of output column j, packed in one of the formats
 * below (the five GGUF formats of those dispatchers, Q8_0 and Q5_0 from the
 * expert-matmul tests of rullama src/backend/dispatch/mod.rs, and the
 * MLX-style affine matrices of moeflux tests/graph_diff_oracle.rs). Further
 * entry points: the backward with respect to the input, the expert-indexed
 * product, gated FFN pairs (SwiGLU / GeGLU) and the affine products.
 * x holds n_tokens rows of k fp32 activations (the batched tests of the same
 * page stack tokens as X[N x k] -> Y[N x n]); y[t][j] = sum_i x[t][i] *
 * w[j][i], fp32. Output-axis tiling follows `MatmulBackInputParams` in
 * rullama src/backend/dispatch/mod.rs: only columns j in [j_start, j_end)
 * are computed; the first tile writes (accumulate = 0), later tiles add
 * (accumulate = 1).
 *
 * Conventions shared by every entry point:
 *  - Data pointers are DEVICE pointers owned by the caller (except in
 *    qmm_matmul_host). The library keeps no reference after a call returns.
 *  - Calls are stream-ordered and asynchronous: they validate on the host,
 *    enqueue kernels on the given stream and return. Nothing is copied to
 *    or from the host and nothing synchronizes, except the documented
 *    first-use set-up.
 *  - Invalid arguments are rejected on the host before anything is
 *    enqueued; the call returns a qmm_status and qmm_last_error() holds a
 *    message (per host thread).
 *  - Layouts: w is n * qmm_weight_bytes(fmt, k, 1) bytes; x is [n_tokens][k]
 *    fp32 row-major; y is [n_tokens][n] fp32 row-major (row stride n even
 *    when only a column tile is computed).
 *  - Alignment: w must be 16-byte aligned (its rows are streamed with bulk
 *    copies); x and y must be 4-byte aligned. Otherwise QMM_ERR_ALIGN.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats. Block geometry from the rullama matmul.rs dispatchers:
 * BF16 / F16: 2 bytes per weight, k even.
 * Q4_0: blocks of 32 weights in 18 bytes (f16 d + 16 nibble bytes), k % 32 == 0.
 * Q4_K: super-blocks of 256 weights in 144 bytes (f16 d, f16 dmin,
 *       12 bytes of 6-bit scales/mins, 128 nibble bytes), k % 256 == 0.
 * Q6_K: super-blocks of 256 weights in 210 bytes (128 low-nibble bytes,
 *       64 high-bit bytes, 16 int8 scales, f16 d), k % 256 == 0.
 * Q8_0: blocks of 32 weights in 34 bytes (f16 d + 32 signed bytes), k % 32 == 0.
 * Q5_0: blocks of 32 weights in 22 bytes (f16 d, a 32-bit word of fifth
 *       bits, 16 nibble bytes), k % 32 == 0 (rullama dispatch/mod.rs expert tests).
 * Inside the blocks the fields follow the standard ggml layouts.
 * AFFINE4 / AFFINE8: MLX-style affine matrices (moeflux
 *       tests/graph_diff_oracle.rs, the EmbedGatherNTokens test and the
 *       MatvecNTokens op it names), three arrays: the codes (w, k/2 or k bytes
 *       per row: little-endian 32-bit words of 8 four-bit or 4 eight-bit codes,
 *       lowest bits first), and a bf16 scale and a bf16 bias per group of 64
 *       consecutive weights of a row ([n][k/64] each); weight = code * scale +
 *       bias, rounded once to fp32; k % 64 == 0. Only qmm_matmul_affine,
 *       qmm_matmul_experts_affine and qmm_dequant_affine take them;
 *       qmm_weight_bytes counts the code bytes. */
typedef enum qmm_format {
    QMM_BF16 = 0,
    QMM_F16 = 1,
    QMM_Q4_0 = 2,
    QMM_Q4_K = 3,
    QMM_Q6_K = 4,
    QMM_Q8_0 = 5,
    QMM_Q5_0 = 6,
    QMM_AFFINE4 = 7,
    QMM_AFFINE8 = 8
} qmm_format;

typedef enum qmm_status {
    QMM_OK = 0,
    QMM_ERR_FORMAT = 1,          /* unknown format code */
    QMM_ERR_SHAPE = 2,           /* k not a multiple of the block, negative sizes, n_tokens < 1 */
    QMM_ERR_SIZE = 3,            /* w_len given and != n * row bytes */
    QMM_ERR_RANGE = 4,           /* not 0 <= j_start <= j_end <= n */
    QMM_ERR_NULL = 5,            /* a pointer needed for the call is NULL */
    QMM_ERR_ALIGN = 6,           /* w not 16-byte aligned, or x / y not 4-byte aligned */
    QMM_ERR_CUDA = 7,            /* a CUDA runtime call failed (message has the CUDA error) */
    QMM_ERR_DEVICE_TIMEOUT = 8,  /* a kernel gave up waiting on a pipeline barrier (reported by qmm_device_status) */
    QMM_ERR_WORKSPACE = 9,       /* workspace given but smaller than qmm_workspace_bytes() */
    QMM_ERR_UNSUPPORTED = 10,    /* current device is not compute capability 10.3, the path cannot take the shape,
                                    or a caller workspace is not device memory of the current device */
    QMM_ERR_BAD_ID = 11          /* an expert id outside [0, n_experts) (reported by qmm_device_status) */
} qmm_status;

/* Kernel path selection for qmm_args.path. */
typedef enum qmm_path {
    QMM_PATH_AUTO = 0,   /* by n_tokens: GEMV for small N, tensor-core (tcgen05) MMA above the crossover */
    QMM_PATH_GEMV = 1,   /* force the streaming GEMV kernel (one launch per token) */
    QMM_PATH_MMA = 2     /* force the tcgen05 N-token kernel */
} qmm_path;

typedef struct qmm_args {
    int fmt;                 /* qmm_format */
    const void *w;           /* device, n * row_bytes packed weight bytes, 16-byte aligned */
    size_t w_len;            /* bytes the caller holds at w; 0 = not checked */
    const float *x;          /* device, [n_tokens][k] */
    float *y;                /* device, [n_tokens][n]; read too when accumulate != 0 */
    int64_t k;               /* weights per row (reduction length) */
    int64_t n;               /* rows of W = output columns */
    int64_t n_tokens;        /* rows of x and y, >= 1 */
    int64_t j_start, j_end;  /* output columns computed; both 0 means [0, n) */
    int accumulate;          /* 0: y[t][j] = sum; else y[t][j] += sum (columns outside the tile untouched) */
    int path;                /* qmm_path */
    void *workspace;         /* device scratch for the MMA path, or NULL (library-owned grow-only buffer) */
    size_t workspace_bytes;  /* bytes at workspace */
    void *stream;            /* cudaStream_t; NULL = legacy default stream */
    int flags;               /* bitwise OR of qmm_flags; 0 = none */
} qmm_args;

/* qmm_args.flags */
typedef enum qmm_flags {
    /* W is not written by the kernel that precedes this call in the stream.
     * The GEMV kernel is then launched as a programmatic dependent of that
     * kernel: it may start streaming W into shared memory while the
     * preceding kernel is still running, and waits for that kernel to finish
     * (and its writes to become visible) before it reads x or touches y.
     * Without the flag the GEMV is launched the same way but waits for the
     * preceding kernel before it reads W as well: stream order holds, and only
     * the launch latency is hidden. */
    QMM_FLAG_OVERLAP_PREV = 1,
    /* With QMM_FLAG_OVERLAP_PREV: x is not written by the preceding kernel
     * either (for instance several projections of the same activations, or
     * x produced two kernels back). The GEMV then also stages x and computes
     * its partial sums before that kernel has finished; only its stores to y
     * wait for it. */
    QMM_FLAG_X_READY = 2,
    /* Tensor-core (N-token) calls on a quantized format: W is split into two
     * fp16 terms as well as x, at every k (precision mode 3; by default W is
     * one fp16 term for k >= 1024). Each weight is then carried with about 22
     * significant bits instead of 11. Without the flag the product's error
     * bound rests on W's fp16 rounding errors not adding up coherently along
     * k: a row whose weights repeat one value (a constant row, codes at one
     * level under one scale) times activations of one sign errs by about
     * 2^-11 of sum_i |x_i w_ij| (measured 4.9e-4), and by more (4.9e-3
     * measured) on Q4_K rows whose weight d q - dmin m nearly cancels, above
     * the 1e-4 bar of the problem statement; with the flag such rows hold the
     * bar. Costs about 5x the
     * time of the default tensor-core call (Q4_K k=4096 n=14336: 106 against
     * 22 us at 8 tokens, 411 against 83 us at 512), so with the flag
     * QMM_PATH_AUTO sends calls of up to 8 tokens to the GEMV path (one
     * launch per token, exact fp32 products, 10.7 us each on that shape).
     * Expert-indexed calls with the flag take the one-GEMV-per-pair form. The
     * GEMV path and 16-bit formats are unaffected: their products are exact
     * in their operand types. */
    QMM_FLAG_SPLIT_W = 4
} qmm_flags;
/* Independent of the flags, the tensor-core (N-token) path lets the launches
 * after it begin early: its x conversion runs as a programmatic dependent of
 * the preceding kernel (it waits for that kernel to finish before it reads x
 * or writes anything, so ordinary stream order holds), and the product kernel
 * allows the next kernel to launch while it runs. A caller's own kernel
 * launched with programmatic stream serialization after a tensor-core call
 * must therefore wait (griddepcontrol.wait / cudaGridDependencySynchronize)
 * before it reads y; ordinary launches are unaffected. */

/* Bytes of n packed rows of k weights: (k/32)*18*n (Q4_0), (k/256)*144*n
 * (Q4_K), (k/256)*210*n (Q6_K), 2*k*n (BF16 / F16) as in the rullama
 * matmul.rs shape checks; (k/32)*34*n (Q8_0), (k/32)*22*n (Q5_0); the code
 * bytes k*n/2 or k*n of the affine formats. 0 when fmt is unknown, k does
 * not fit the format, or k/n is negative. Host only. */
size_t qmm_weight_bytes(int fmt, int64_t k, int64_t n);

/* y = x @ W over the whole output axis, on the stream last given to
 * qmm_set_stream (default: the legacy default stream), auto path, workspace
 * from the library's own grow-only buffer: the problem statement's plain
 * signature qmm_matmul(fmt, w_bytes, x, k, n, n_tokens, y). Returns a
 * qmm_status. */
int qmm_matmul(int fmt, const void *w, const float *x, int64_t k, int64_t n,
               int64_t n_tokens, float *y);

/* Stream used by qmm_matmul on the calling host thread (a cudaStream_t).
 * This is the chained model of rullama src/backend/dispatch/mod.rs
 * ("Chained dispatchers"): work is appended to a stream that the caller
 * owns and nothing waits for it; NULL selects the legacy default stream.
 * The library keeps the handle only as this thread's setting. */
void qmm_set_stream(void *stream);

/* Full form: column tile, accumulate, path, workspace and stream.
 * k == 0 writes zeros to the tile's columns (or leaves them when
 * accumulating); n == 0 or an empty tile enqueues nothing.
 * Scratch: with a->workspace NULL the tensor-core path uses one grow-only
 * buffer per device owned by the library (growing it synchronizes the
 * device once); calls that may run concurrently on different streams, or
 * that are captured into a CUDA graph, pass their own workspace. A caller
 * workspace must be 256-byte aligned device memory of the current device
 * (checked with cudaPointerGetAttributes: QMM_ERR_UNSUPPORTED otherwise),
 * since the tensor-core kernel reads its x tiles from it with copies that
 * each pair of CTAs shares. */
int qmm_matmul_ex(const qmm_args *a);

/* Device scratch bytes qmm_matmul_ex needs for *a (0 for the GEMV path).
 * The MMA path splits x into two fp16 terms (high part and rounding
 * remainder, k padded to a multiple of 64) scaled by one power of two per
 * token: 2 * round256(n_tokens * kp * 2) + round256(n_tokens * 4) bytes.
 * Host only. */
size_t qmm_workspace_bytes(const qmm_args *a);

/* Which kernel path qmm_matmul_ex would run for *a (a qmm_path value other
 * than AUTO), or -1 if *a is invalid. Host only. */
int qmm_select_path(const qmm_args *a);

/* Host-buffer form of qmm_matmul_ex, matching the pages' one-shot
 * dispatchers that take weight bytes and x from the host and return y
 * (rullama matmul.rs `dispatch_matmul`). a->w, a->x and a->y are HOST
 * pointers (page-locked memory makes the copies asynchronous); dev_w,
 * dev_x and dev_y are caller-owned device buffers at least as large as W,
 * x and y. Enqueues W -> dev_w, x -> dev_x (and y -> dev_y when
 * accumulating), the product, then dev_y -> y, all on a->stream; the caller
 * synchronizes the stream before reading y. */
int qmm_matmul_host(const qmm_args *a, void *dev_w, float *dev_x, float *dev_y);

/* Backward of y = x @ W with respect to the input, for one vector (rullama
 * src/backend/dispatch/mod.rs, `MatmulBackInputParams` and the
 * `matmul_q*_backward_input` dispatchers):
 *     dx[i] (+)= sum_{j in [j_start, j_end)} dy[j] * w[j][i],  i in [0, k)
 * The row range tiles the SUM axis (the reference's tiling of the vocabulary
 * head): the first tile writes dx (accumulate = 0), later tiles add to it
 * (accumulate = 1); j_start == j_end == 0 means all n rows, and an empty
 * range writes zeros (or leaves dx when accumulating). Fields: a->x is dy
 * (device, n floats), a->y is dx (device, k floats), a->n_tokens must be 1,
 * a->path is ignored; fmt, w, w_len, k, n, workspace, stream as for
 * qmm_matmul_ex. a->flags as for qmm_matmul_ex with dy in the role of x:
 * under QMM_FLAG_OVERLAP_PREV the partial-sum kernel starts streaming W
 * while the preceding kernel finishes, reads dy after it (unless
 * QMM_FLAG_X_READY) and always writes its partials after it. Within a call
 * the summing kernel is always launched as a programmatic dependent. Units of k are 32 weights (8 for 16-bit formats) and at
 * most 256 per row: k <= 8192 for the block formats, k <= 2048 for BF16/F16
 * (QMM_ERR_UNSUPPORTED beyond). The result is the same on every call (the
 * per-CTA partial sums are added in a fixed order). Stream-ordered, no
 * host synchronization; acceptance bar as for the forward product, with
 * S = sum_j |dy[j] w[j][i]|. */
int qmm_matmul_backward_input(const qmm_args *a);

/* Device scratch bytes qmm_matmul_backward_input needs for *a (one fp32
 * partial dx per CTA: grid * k * 4; 0 for an empty call or invalid
 * arguments). With a->workspace NULL the library's own grow-only buffer is
 * used. Host only (reads the device's SM count). */
size_t qmm_backward_input_workspace_bytes(const qmm_args *a);

/* Expert-indexed product (mixture of experts; rullama src/backend/dispatch/mod.rs,
 * tests `moe_expert_matmul_q5_0_gpu_vs_cpu` and `moe_expert_matmul_batched_gpu_vs_cpu`): W holds n_experts
 * slices of n rows stacked one after another (each qmm_weight_bytes(fmt, k, n)
 * bytes); a->x is [n_pos x k] with n_pos = a->n_tokens; ids is a DEVICE int32
 * array [n_pos x top_k]; a->y is [n_pos * top_k x n]:
 *     y[p * top_k + s][j] (+)= sum_i x[p][i] * w_{ids[p * top_k + s]}[j][i]
 * for j in [j_start, j_end). a->w_len, when nonzero, must be n_experts times
 * the slice bytes; n_pos * top_k <= 65535. Two forms, both reading the ids
 * on the device (nothing synchronizes):
 *  - GEMV form: each (position, slot) runs as one GEMV of the one-token
 *    path, side by side in one launch. a->flags as for qmm_matmul_ex, with
 *    ids counted as input: under QMM_FLAG_OVERLAP_PREV alone the kernel waits
 *    for the preceding one before it reads ids (so no weight byte moves
 *    before then); QMM_FLAG_X_READY vouches that neither x nor ids is written
 *    by the preceding kernel. Same formats and k limits as the one-token path.
 *  - grouped form (the batched expert matmul of the same page): a routing
 *    kernel sorts the pairs by expert on the device, then one tensor-core
 *    pass multiplies each expert's rows by its slice, so a slice chosen by
 *    many positions is decoded once per token tile instead of once per pair.
 *    GGUF formats with k >= 1024 (the split-x mode; Q4_0, Q5_0 and Q8_0
 *    also k % 256 == 0), n_experts <= 4096; scratch from a->workspace
 *    (qmm_experts_workspace_bytes) or the library's buffer. With
 *    QMM_FLAG_SPLIT_W the pairs take the GEMV form.
 * a->path GEMV or MMA forces a form (MMA: QMM_ERR_UNSUPPORTED where the
 * grouped form cannot take the call); AUTO takes the grouped form for Q4_K,
 * Q8_0, Q5_0 and Q4_0 when n_pos > 1 and n_pos * top_k >= 2 * n_experts, for
 * Q6_K (whose exact decode makes the grouped form cost about the same at any
 * position count) when n_pos * top_k >= 3 * n_experts, the GEMV form
 * otherwise. An id outside [0, n_experts)
 * leaves that y row untouched and records an error that qmm_device_status
 * reports as QMM_ERR_BAD_ID. */
int qmm_matmul_experts(const qmm_args *a, const int32_t *ids, int64_t n_experts, int64_t top_k);

/* Device scratch bytes qmm_matmul_experts needs for these arguments: 0 for
 * the GEMV form; for the grouped form the split fp16 copies of the routed x
 * rows, a scale per row, the routing tables and the row order
 * (2 * round256(P * kp * 2) + round256(P * 4) + 2 * round256((n_experts + 1) * 4)
 * + round256(P * 4) with P = n_pos * top_k, kp = k padded to 64). Host only. */
size_t qmm_experts_workspace_bytes(const qmm_args *a, int64_t n_experts, int64_t top_k);

/* The expert-indexed product for affine matrices (a->fmt = QMM_AFFINE4 or
 * QMM_AFFINE8; mixture-of-experts layers of MLX-style models): the code
 * words are stacked as above, and `scales` / `biases` stack the experts'
 * bf16 arrays the same way ([n_experts][n][k/64] each; device, 16-byte
 * aligned). Everything else as qmm_matmul_experts. */
int qmm_matmul_experts_affine(const qmm_args *a, const int32_t *ids, int64_t n_experts,
                              int64_t top_k, const void *scales, const void *biases);

/* Standalone dequantization, the GPU counterpart of the ggml-exact CPU
 * routines (`crate::gguf::quant::dequant_q4_0`, `dequant_q4_k`,
 * `dequant_q6_k`, `dequant_q8_0`, `dequant_q5_0`) that the tests of rullama
 * src/backend/matmul.rs and dispatch/mod.rs use as their reference:
 * out[j][i] = the fp32 value of weight i of row j, bit-identical to the
 * exact value rounded once to fp32 (only Q4_K's d*sc*q - dmin*m rounds;
 * every other product is exact). w is device memory (16-byte aligned), n
 * rows of qmm_weight_bytes(fmt, k, 1) bytes; out is caller-owned device
 * [n][k] fp32 (4-byte aligned). Errors as for qmm_matmul_ex (affine formats:
 * QMM_ERR_FORMAT, use qmm_dequant_affine); k == 0 or n == 0 enqueues
 * nothing. Stream-ordered, no host synchronization. */
int qmm_dequant(int fmt, const void *w, int64_t k, int64_t n, float *out, void *stream);

/* Gate activations of gated FFN pairs. */
typedef enum qmm_act {
    QMM_ACT_SWIGLU = 1,  /* silu(g) = g / (1 + e^-g) */
    QMM_ACT_GEGLU = 2    /* GELU, tanh form: g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) */
} qmm_act;

/* Gated pair (rullama src/backend/dispatch/mod.rs `silu_chained`,
 * `geglu_chained`; moeflux tests/graph_diff_oracle.rs `SwigluFusedBatched`):
 *     y[t][j] (+)= act((x Wg)[t][j]) * (x Wu)[t][j],  j in [j_start, j_end)
 * a->w is the gate matrix, w_up the up matrix (same format, k, n and w_len;
 * device, 16-byte aligned). One token on the GEMV path: one fused launch
 * that streams a CTA's rows of Wg, keeps the gate values on chip, streams
 * the same rows of Wu and writes only y. Several tokens: the gate product
 * goes through the tensor-core path into scratch (a->workspace of at least
 * qmm_glu_workspace_bytes(a) bytes, else the library's: the gate values
 * [n_tokens][n] fp32 plus qmm_workspace_bytes of the product), then the up
 * product's epilogue reads each gate value and writes act(gate) * up (or
 * adds it) to y; no up vector is stored and no combine kernel runs. GGUF
 * formats only (QMM_ERR_FORMAT for affine ones or an unknown act); flags as
 * for qmm_matmul_ex. */
int qmm_matmul_glu(const qmm_args *a, const void *w_up, int act);
size_t qmm_glu_workspace_bytes(const qmm_args *a);

/* y = x @ W for an affine matrix (a->fmt = QMM_AFFINE4 or QMM_AFFINE8):
 * a->w holds the code words, `scales` and `biases` the bf16 arrays [n][k/64]
 * (device memory, 16-byte aligned; NULL only when there is no work). Every
 * other field as for qmm_matmul_ex: tiles, accumulate, path (one token: the
 * GEMV; several: the tensor-core path), workspace, stream, flags. Errors as
 * for qmm_matmul_ex; QMM_ERR_FORMAT for any other format. */
int qmm_matmul_affine(const qmm_args *a, const void *scales, const void *biases);

/* out[j][i] = the fp32 weight i of row j of an affine matrix, bit-identical
 * to code * scale + bias rounded once. Device pointers; scales and biases
 * 2-byte aligned. Stream-ordered. */
int qmm_dequant_affine(int fmt, const void *w, const void *scales, const void *biases, int64_t k,
                       int64_t n, float *out, void *stream);

/* Health check of the device-side bounded waits: enqueues one small kernel
 * that waits on a barrier nothing satisfies; after about 50 ms the wait
 * gives up and the kernel records the fault and returns (no GPU fault, no
 * hang). The next qmm_device_status(stream) must then report
 * QMM_ERR_DEVICE_TIMEOUT (and clear it); the context stays usable. */
int qmm_check_bounded_wait(void *stream);

/* Synchronizes `stream`, then reports whether any kernel enqueued so far
 * timed out on a pipeline barrier (QMM_ERR_DEVICE_TIMEOUT) or met an expert
 * id out of range (QMM_ERR_BAD_ID), and clears the flag; QMM_OK otherwise,
 * QMM_ERR_CUDA if the synchronize failed. Every
 * barrier wait in the kernels is bounded (about 2 s); on expiry the kernel
 * records the fault, stops its pipeline, releases its tensor memory and
 * returns, so the context stays usable. */
int qmm_device_status(void *stream);

/* qmm_matmul_ex on the tensor-core path for callers that cannot allocate
 * device memory (no CUDA allocator of their own, or no allocation calls
 * allowed on their hot path because those synchronize the device). The
 * pages have no counterpart of this call. Its scratch (the fp16 copies of x
 * and the per-token scales, qmm_workspace_bytes() of the same arguments on
 * that path) lives in a fixed 16 MiB array in device memory that the library
 * defines; every GPU that loads libqmm holds that array until the process
 * exits. a->path, a->workspace and a->workspace_bytes are ignored; all other
 * fields mean what they mean for qmm_matmul_ex, and the caller still passes
 * w, x and y. A call that would need more than 16 MiB of scratch returns
 * QMM_ERR_WORKSPACE without enqueuing anything. The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine). The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current); make that first call before any stream capture.
 * Every call uses the same array and leaves its contents behind (each call
 * overwrites all the scratch it reads, so nothing needs clearing): calls
 * whose kernels can overlap on the GPU (different streams without ordering
 * between them) race on it. */
int qmm_matmul_noalloc(const qmm_args *a);

/* Message for the last non-OK status on this host thread ("" if none): the
 * text that the rullama matmul_* dispatchers (src/backend/matmul.rs) carry
 * in their `Err(RullamaError::Inference(..))` returns, here beside the
 * numeric qmm_status. The string is owned by the library and stays valid
 * until the next call on the same thread. */
const char *qmm_last_error(void);

/* ABI version (major * 100 + minor). */
int qmm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
