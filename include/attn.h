/*
 * attn.h: C ABI of the GB300 (sm_103a) exact multi-head attention library.
 *
 * The operation comes from "Self-attention, CUDA kernels and FlashAttention" (2026-11-15):
 *   section 1 "How self-attention works mathematically in a Vision Transformer":
 *       Scores = Q K^T / sqrt(d_k); a softmax along each row (each row sums to one);
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V; the same computation runs
 *       independently for every head.
 *   section 3 "FlashAttention: solving the Transformer memory bottleneck":
 *       tiled, fused evaluation that never stores the N x N matrix in HBM ("Tiling"), an
 *       online softmax ("The online softmax trick"), and a backward pass that keeps only
 *       small per-row normalisation statistics and recomputes the attention tiles on chip
 *       ("Recomputation in backpropagation").
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense, contiguous, row-major [B, H, N, d_k] bf16 (`const void *` / `void *`
 *     here, so that the header needs no CUDA half-precision types).  Row (b, h, i) starts at
 *     element ((b * H + h) * N + i) * d_k.  `lse` and the other per-row vectors are [B, H, N]
 *     fp32.  All pointers are device pointers, 16-byte aligned.
 *   - `scale` multiplies Q K^T before the softmax; pass 1/sqrt(d_k) for the article's
 *     formula.  It must be finite and > 0.
 *   - Supported: d_k in {64, 128}; B, H, N >= 1; B*H*N*d_k < 2^40 elements; N < 2^31.
 *   - Ownership: the caller allocates and owns every buffer, including the forward and
 *     backward workspaces.  The library allocates no device memory on these paths.
 *   - Calls enqueue work on `stream` and return without waiting; only
 *     attn_get_device_status() synchronises (that stream).  Outputs must not overlap inputs.
 *   - The compute calls allocate nothing and never synchronise, so they may be captured in a
 *     CUDA graph on `stream` and replayed (the captured pointers, sizes and scale are fixed).
 *   - Errors: every argument check runs before any launch; on failure the call returns a
 *     non-zero attn_status and launches nothing.  A kernel that cannot make progress does not
 *     hang the GPU: each of its waits gives up after a bounded time and records
 *     ATTN_ERR_TIMEOUT in a per-device status word, read by attn_get_device_status().
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,     /* null pointer, size < 1, bad scale, overlapping buffers */
    ATTN_ERR_UNSUPPORTED_DK = 2,  /* d_k not in {64, 128} */
    ATTN_ERR_MISALIGNED = 3,      /* a pointer not 16-byte aligned */
    ATTN_ERR_LAUNCH = 4,          /* the CUDA runtime refused a launch or a query */
    ATTN_ERR_TIMEOUT = 5,         /* a kernel wait gave up (reported by attn_get_device_status) */
    ATTN_ERR_WORKSPACE = 6,       /* workspace null, misaligned or smaller than required */
    ATTN_ERR_DEVICE = 7,          /* the current device is not an sm_103 GPU */
    ATTN_ERR_TOO_LARGE = 8        /* attn_bwd_noalloc: sizes need more than its fixed scratch */
} attn_status;

/*
 * Forward pass (section 1's Attention(Q,K,V); section 3's tiling and online softmax).
 *   q, k, v : [B,H,N,d_k] bf16 inputs.
 *   o       : [B,H,N,d_k] bf16 output, O = softmax(scale * Q K^T) V, rounded to nearest.
 *   lse     : [B,H,N] fp32 output, lse[b,h,i] = log(sum_j exp(scale * q_i . k_j)) (natural
 *             log): the per-row statistic the backward pass recomputes the tiles from.
 * Arithmetic: scores in fp32 (tensor cores), softmax statistics in fp32, and the product of
 * the weights with V on fp16 tensor cores: each weight is rounded to fp16 (relative error at
 * most 2^-11) and V is rounded to fp16, which is exact for |v| in [2^-14, 65504]; smaller
 * entries keep an absolute precision of 2^-25, and an entry of V above 65504 in magnitude
 * makes the O rows it contributes to non-finite.  O is normalised by the unrounded row sum.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H, int N, int d_k, float scale, cudaStream_t stream);

/*
 * Diagnostic forward: attn_fwd() (same o and lse, bitwise) that also writes O before it is
 * rounded to bf16, so that the arithmetic's own error can be told apart from the output
 * rounding (section 1's Attention(Q,K,V); the bf16 o is exactly o32 rounded to nearest).
 *   o32 : [B,H,N,d_k] fp32 device output, 16-byte aligned, written with per-row stores (slow:
 *         for tests and measurements, not for training).
 * Errors: as attn_fwd; ATTN_ERR_INVALID_ARG for a null o32 or one overlapping another buffer,
 * ATTN_ERR_MISALIGNED for a misaligned one.
 */
attn_status attn_fwd_diagnostic(const void *q, const void *k, const void *v, void *o, float *lse,
                                float *o32, int B, int H, int N, int d_k, float scale,
                                cudaStream_t stream);

/*
 * Bytes of device workspace attn_fwd_with_workspace() uses for these sizes: an fp16 copy of V
 * (B*H*N*d_k*2 bytes rounded up to a multiple of 256) where the sequence is long enough for
 * one rounding pass over V ahead of the forward kernel to cost less than rounding every V tile
 * in the shared memory of each CTA that reads it (d_k = 64: N >= 2048; d_k = 128: N >= 8192),
 * else 0.  Also 0 for sizes attn_fwd rejects.
 */
size_t attn_fwd_workspace_size(int B, int H, int N, int d_k);

/*
 * The forward pass of attn_fwd() with a caller workspace (section 3's tiled forward; the
 * operation, arguments, layouts, arithmetic and results are attn_fwd's, bitwise: V is rounded
 * to fp16 the same way, only in one pass over HBM into the workspace instead of in shared
 * memory).  Where attn_fwd_workspace_size() is 0 the call is attn_fwd() and `workspace` may
 * be null.
 *   workspace : caller-owned device memory of at least attn_fwd_workspace_size(B,H,N,d_k)
 *               bytes, 256-byte aligned, overwritten; it must not overlap q, k, v, o or lse.
 * Errors: as attn_fwd, plus ATTN_ERR_WORKSPACE (null, misaligned or too small where a
 * workspace is needed) and ATTN_ERR_INVALID_ARG for a workspace overlapping another buffer.
 */
attn_status attn_fwd_with_workspace(const void *q, const void *k, const void *v, void *o, float *lse,
                                    void *workspace, size_t workspace_bytes, int B, int H, int N,
                                    int d_k, float scale, cudaStream_t stream);

/*
 * Bytes of device workspace attn_bwd() needs for these sizes: two fp32 statistics per row
 * (-lse * log2(e) and -rowsum(dO o O), [B,H] x N rounded up to 128, stored interleaved per
 * pair of rows) and an fp32 dQ accumulator ([B,H,N,d_k]), each region 256-byte aligned.
 * Returns 0 if the sizes are unsupported.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d_k);

/*
 * Backward pass (section 3, "Recomputation in backpropagation": only the per-row statistic
 * `lse` from attn_fwd is kept; the probabilities are recomputed on chip).  With
 * P = exp(scale * Q K^T - lse) and D_i = sum_c dO_ic O_ic:
 *   dV = P^T dO;   dP = dO V^T;   dS = P o (dP - D);   dQ = scale * dS K;   dK = scale * dS^T Q.
 *   q, k, v, o, dout : [B,H,N,d_k] bf16 inputs (o is attn_fwd's output, dout = dL/dO).
 *   lse              : [B,H,N] fp32 from attn_fwd for the same q, k, scale.
 *   dq, dk, dv       : [B,H,N,d_k] bf16 outputs.
 *   workspace        : device memory of at least attn_bwd_workspace_size(B,H,N,d_k) bytes,
 *                      256-byte aligned, owned by the caller; its contents on entry do not
 *                      matter and on return are unspecified.
 * dQ is accumulated across key tiles with fp32 atomic additions, so its low-order bits may
 * differ from run to run; dK and dV are deterministic.  Exception: for d_k = 64 and N <= 256
 * over at most one head per SM (and N <= 128 or more heads than half the SMs) one kernel takes
 * each head whole and accumulates dQ on chip, without atomics: all three gradients are then
 * bitwise reproducible, and the workspace is not touched.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, void *dq, void *dk, void *dv,
                     void *workspace, size_t workspace_bytes, int B, int H, int N, int d_k,
                     float scale, cudaStream_t stream);

/*
 * The same backward pass with dQ computed without atomics, so that dQ, dK and dV are bitwise
 * reproducible from run to run (the article leaves the scheduling of the recomputation open;
 * this is the alternative to accumulating dQ with fp32 atomics).  Arguments, layouts, workspace
 * and errors are those of attn_bwd().  It runs the preprocess, the key-stationary kernel for dK
 * and dV alone, then a query-stationary pass that recomputes S = scale Q K^T and dP = dO V^T
 * tile by tile and accumulates dQ = scale * dS K in order, one CTA per 128 query rows.  It does
 * 14 instead of 10 B*H*N^2*d_k flops.  Where attn_bwd() takes heads whole (d_k = 64, short
 * sequences, few heads; see there) it runs that same kernel, which needs no atomics.
 */
attn_status attn_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                                   const void *dout, const float *lse, void *dq, void *dk,
                                   void *dv, void *workspace, size_t workspace_bytes, int B,
                                   int H, int N, int d_k, float scale, cudaStream_t stream);

/*
 * The three stream-ordered phases attn_bwd() runs, for callers that schedule or time them
 * separately.  Run on one stream, in this order, with the same sizes, scale and workspace,
 * they produce exactly what attn_bwd() produces.
 *
 * attn_bwd_preprocess: reads o, dout and lse; writes into the workspace -D_i, with
 *   D_i = sum_c dO_ic O_ic, and -lse_i * log2(e) (rows padded to a multiple of 128; padding rows
 *   get 0 and -inf, i.e. zero probability), and zeroes the workspace's fp32 dQ accumulator.
 * attn_bwd_main: for every 128-key tile, recomputes P = 2^(scale log2(e) q.k - lse log2(e))
 *   from q, k and the workspace, writes dk (= scale * dS^T Q) and dv (= P^T dO), and adds
 *   dS K into the dQ accumulator.  Reads q, k, v, dout and the workspace.
 * attn_bwd_dq_convert: dq = bf16(scale * accumulator).
 */
attn_status attn_bwd_preprocess(const void *o, const void *dout, const float *lse,
                                void *workspace, size_t workspace_bytes, int B, int H, int N,
                                int d_k, cudaStream_t stream);
attn_status attn_bwd_main(const void *q, const void *k, const void *v, const void *dout,
                          void *dk, void *dv, void *workspace, size_t workspace_bytes, int B,
                          int H, int N, int d_k, float scale, cudaStream_t stream);
attn_status attn_bwd_dq_convert(void *workspace, size_t workspace_bytes, void *dq, int B, int H,
                                int N, int d_k, float scale, cudaStream_t stream);

/*
 * Reads and clears the current device's status word after synchronising `stream`.
 * Returns ATTN_OK, ATTN_ERR_TIMEOUT if a kernel wait gave up since the last call, or
 * ATTN_ERR_LAUNCH if the stream reports a CUDA error.
 */
attn_status attn_get_device_status(cudaStream_t stream);

/* A static, human-readable name for a status code. */
const char *attn_status_string(attn_status status);

/*
 * The CUDA call behind the most recent ATTN_ERR_LAUNCH returned on the calling host thread,
 * with the runtime's error name and text ("no error" if there was none).  The string belongs
 * to the library and stays valid until the thread's next failing call.
 */
const char *attn_last_error_string(void);

/*
 * Diagnostics: launches one tiny kernel that waits, with the library's bounded-wait
 * routine, on a barrier nothing ever signals, giving up after `limit_us` microseconds
 * (1 ... 10^6).  The following attn_get_device_status() must then return ATTN_ERR_TIMEOUT.
 * Used to test the failure path without hanging or faulting the GPU.
 */
attn_status attn_debug_wait_timeout(unsigned limit_us, cudaStream_t stream);

/*
 * Query / key / value projection (section 1, "Generating queries, keys and values":
 * Q = X W_Q, K = X W_K, V = X W_V, each W in R^(D x d_k) per head): the step that feeds
 * attn_fwd.  The heads' weights side by side form one D x D matrix per projection; head h
 * takes its columns [h d_k, (h+1) d_k), and the outputs are written directly in the
 * [B, H, N, d_k] layout attn_fwd reads.
 *   x             : [B, N, D] bf16 (token rows).
 *   w_q, w_k, w_v : [D, D] bf16 row-major (input dimension x output columns).
 *   q, k, v       : [B, H, N, d_k] bf16 outputs (fp32 accumulation, rounded to nearest).
 * Requirements: D = H * d_k, D a multiple of 128, d_k in {64, 128}; pointers 16-byte aligned;
 * outputs overlap neither each other nor the inputs.
 */
attn_status attn_qkv_proj(const void *x, const void *w_q, const void *w_k, const void *w_v,
                          void *q, void *k, void *v, int B, int N, int D, int H, int d_k,
                          cudaStream_t stream);

/*
 * Backward of attn_qkv_proj for the gradients dq, dk, dv ([B, H, N, d_k] bf16, e.g. from
 * attn_bwd): dX = sum_t dY_t W_t^T ([B, N, D] bf16 output) and dW_t = X^T dY_t summed over all
 * B*N tokens ([D, D] fp32 outputs, written from zero).  Where too few dW tiles exist to fill
 * the GPU, the token rows are split across CTAs and their partial sums added with fp32 atomics,
 * so the last bits of dW may then vary between runs.
 * Same size rules as attn_qkv_proj.
 */
attn_status attn_qkv_proj_bwd(const void *x, const void *w_q, const void *w_k, const void *w_v,
                              const void *dq, const void *dk, const void *dv, void *dx,
                              float *dw_q, float *dw_k, float *dw_v, int B, int N, int D, int H,
                              int d_k, cudaStream_t stream);

/*
 * Bytes of device workspace attn_fwd_unfused() needs: the fp32 score matrix S [B,H,N,N] and the
 * bf16 probabilities P [B,H,N,N], each region 256-byte aligned (6 B H N^2 bytes and padding).
 * Returns 0 if the sizes are unsupported.
 */
size_t attn_fwd_unfused_workspace_size(int B, int H, int N, int d_k);

/*
 * Standard attention, the comparison point of section 3 ("memory bandwidth bottleneck"): the
 * same O and LSE as attn_fwd, computed the way the article says frameworks compute it before
 * FlashAttention: S = scale * Q K^T is written to HBM (fp32, by a batched cuBLAS GEMM), a softmax
 * pass reads S and writes P = softmax(S) to HBM (bf16, rounded after normalisation) and LSE, and
 * a second batched cuBLAS GEMM reads P back for O = P V (fp32 accumulation, bf16 output).
 * Memory grows as N^2 per head; the fused attn_fwd needs none.
 *   q, k, v, o, lse : as attn_fwd.  workspace : caller-owned device memory of at least
 *   attn_fwd_unfused_workspace_size() bytes, 256-byte aligned, overwritten.
 * Errors: as attn_fwd, plus ATTN_ERR_WORKSPACE; B*H*N must fit an int and B*H*N^2 stay below
 * 2^40 (ATTN_ERR_INVALID_ARG).  cuBLAS is loaded at the first call; if it cannot be loaded or
 * created the call returns ATTN_ERR_LAUNCH and attn_last_error_string() says why.  Calls are
 * serialised by a lock (one cuBLAS handle per device).
 */
attn_status attn_fwd_unfused(const void *q, const void *k, const void *v, void *o, float *lse,
                             void *workspace, size_t workspace_bytes, int B, int H, int N, int d_k,
                             float scale, cudaStream_t stream);

/*
 * Element-wise fp32 addition c[i] = a[i] + b[i], 0 <= i < n: the vector_add_cuda kernel of
 * section 2 ("Practical code comparison: raw CUDA C++ vs OpenAI Triton", the raw CUDA C++
 * version: one element per index, guarded by i < n), used here as the library's HBM bandwidth
 * probe (16-byte vector accesses, grid-stride over whole waves of the SMs).
 *   a, b : n fp32 device inputs;  c : n fp32 device output (may be a or b itself; no other
 *   overlap).  All 16-byte aligned.  n = 0 is a no-op; n < 0 is ATTN_ERR_INVALID_ARG.
 * Each c[i] is the correctly rounded fp32 sum, bit for bit what one fp32 addition gives.
 */
attn_status vector_add(const float *a, const float *b, float *c, long long n, cudaStream_t stream);

/*
 * attn_bwd_noalloc: the backward pass without any workspace argument, for callers that cannot
 * allocate device memory at the point where they run the backward: code that must not call
 * cudaMalloc (or an allocator built on it) there, for example because it runs under a memory
 * budget fixed up front or inside a framework that owns all device allocations.  The article
 * has no counterpart; this is a convenience of this library.
 *
 * Arguments and results are those of attn_bwd() without `workspace` / `workspace_bytes`.  The
 * scratch attn_bwd keeps in the workspace (attn_bwd_workspace_size(B,H,N,d_k) bytes) comes
 * instead from one array of 64 MiB compiled into the library; every GPU that loads the library
 * holds it until the process exits.  Sizes whose scratch exceeds 64 MiB are refused with
 * ATTN_ERR_TOO_LARGE before anything is launched.  The call allocates no device memory.
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) and
 * caches it; make that first call before any stream capture.  All calls share the one array:
 * calls whose work can overlap on the GPU (different streams, or different host threads without
 * ordering) race on it and produce wrong gradients; order them on one stream.  Each call
 * rewrites everything it reads from the array, so earlier contents do not matter.
 */
attn_status attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                             const void *dout, const float *lse, void *dq, void *dk, void *dv,
                             int B, int H, int N, int d_k, float scale, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
