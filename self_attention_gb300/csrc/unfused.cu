// "Standard attention", the comparison point of "Self-attention, CUDA kernels and
// FlashAttention", section 3 ("memory bandwidth bottleneck"): the score matrix is written to
// HBM, read back by a softmax pass that writes the probabilities to HBM, and those are read back
// once more by the product with V.  This is the O(N^2)-memory form the fused kernels avoid; it
// exists here so that the two can be timed on the same workloads.
//   1. S = scale * Q K^T   fp32 [BH][N][N], one batched library GEMM (bf16 in, fp32 out)
//   2. P = softmax(S)      bf16 [BH][N][N] and LSE fp32 [BH][N], the kernel below
//   3. O = P V             bf16 [BH][N][d], one batched library GEMM (bf16 in, fp32 accumulate)
// The two GEMMs are plain dense products, so they go to cuBLAS, loaded at the first call (the
// fused path never touches it).
#include <cublas_v2.h>
#include <dlfcn.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr float kLog2eU = 1.4426950408889634f;
constexpr float kLn2U = 0.6931471805599453f;
constexpr int kSoftmaxThreads = 256;

// One block per row of S (rows longer than kWarpRowMax, below): the row's maximum and sum by an
// online pass, then P = exp(S - m) / l rounded to bf16, and LSE = m + log l.  The row is read
// twice (the second time from L2).
__global__ void __launch_bounds__(kSoftmaxThreads)
    unfused_softmax_kernel(const float *__restrict__ s, __nv_bfloat16 *__restrict__ p, float *__restrict__ lse,
                           int n)
{
    __shared__ float red_m[kSoftmaxThreads / 32], red_l[kSoftmaxThreads / 32];
    const size_t row = blockIdx.x;
    const float *srow = s + row * n;
    __nv_bfloat16 *prow = p + row * n;
    float m = -INFINITY, l = 0.f;
    for (int j = threadIdx.x; j < n; j += kSoftmaxThreads) {
        const float x = srow[j] * kLog2eU;
        if (x > m) {
            l = l * exp2f(m - x) + 1.f;
            m = x;
        } else {
            l += exp2f(x - m);
        }
    }
    // combine (m, l) over the warp, then over the warps
    for (int off = 16; off > 0; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off), lo = __shfl_xor_sync(0xffffffffu, l, off);
        const float mn = fmaxf(m, mo);
        l = (m == -INFINITY ? 0.f : l * exp2f(m - mn)) + (mo == -INFINITY ? 0.f : lo * exp2f(mo - mn));
        m = mn;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red_m[warp] = m;
        red_l[warp] = l;
    }
    __syncthreads();
    m = red_m[0];
    l = red_l[0];
    for (int w = 1; w < kSoftmaxThreads / 32; ++w) {
        const float mn = fmaxf(m, red_m[w]);
        l = l * exp2f(m - mn) + red_l[w] * exp2f(red_m[w] - mn);
        m = mn;
    }
    const float inv_l = 1.f / l;
    for (int j = threadIdx.x; j < n; j += kSoftmaxThreads)
        prow[j] = __float2bfloat16_rn(exp2f(srow[j] * kLog2eU - m) * inv_l);
    if (threadIdx.x == 0) lse[row] = (m + log2f(l)) * kLn2U;
}

// Rows of at most kWarpRowMax: one warp per row (eight rows per block), the same two passes with
// warp shuffles only.
constexpr int kWarpRowMax = 2048;

__global__ void __launch_bounds__(256)
    unfused_softmax_warp_kernel(const float *__restrict__ s, __nv_bfloat16 *__restrict__ p,
                                float *__restrict__ lse, long long rows, int n)
{
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *srow = s + row * n;
    __nv_bfloat16 *prow = p + row * n;
    float m = -INFINITY, l = 0.f;
    for (int j = lane; j < n; j += 32) {
        const float x = srow[j] * kLog2eU;
        if (x > m) {
            l = l * exp2f(m - x) + 1.f;
            m = x;
        } else {
            l += exp2f(x - m);
        }
    }
    for (int off = 16; off > 0; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off), lo = __shfl_xor_sync(0xffffffffu, l, off);
        const float mn = fmaxf(m, mo);
        l = (m == -INFINITY ? 0.f : l * exp2f(m - mn)) + (mo == -INFINITY ? 0.f : lo * exp2f(mo - mn));
        m = mn;
    }
    const float inv_l = 1.f / l;
    for (int j = lane; j < n; j += 32) prow[j] = __float2bfloat16_rn(exp2f(srow[j] * kLog2eU - m) * inv_l);
    if (lane == 0) lse[row] = (m + log2f(l)) * kLn2U;
}

// cuBLAS entry points, resolved once from the shared library.
using CreateFn = cublasStatus_t (*)(cublasHandle_t *);
using SetStreamFn = cublasStatus_t (*)(cublasHandle_t, cudaStream_t);
using GemmFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int,
                                  const void *, const void *, cudaDataType, int, long long, const void *,
                                  cudaDataType, int, long long, const void *, void *, cudaDataType, int,
                                  long long, int, cublasComputeType_t, cublasGemmAlgo_t);

struct Blas {
    bool tried = false;
    CreateFn create = nullptr;
    SetStreamFn set_stream = nullptr;
    GemmFn gemm = nullptr;
    cublasHandle_t handle[64] = {};
};

std::mutex g_blas_mutex;
Blas g_blas;

const char *load_blas()
{
    if (!g_blas.tried) {
        g_blas.tried = true;
        void *lib = dlopen("libcublas.so.13", RTLD_NOW | RTLD_LOCAL);
        if (!lib) lib = dlopen("libcublas.so", RTLD_NOW | RTLD_LOCAL);
        if (lib) {
            g_blas.create = reinterpret_cast<CreateFn>(dlsym(lib, "cublasCreate_v2"));
            g_blas.set_stream = reinterpret_cast<SetStreamFn>(dlsym(lib, "cublasSetStream_v2"));
            g_blas.gemm = reinterpret_cast<GemmFn>(dlsym(lib, "cublasGemmStridedBatchedEx"));
        }
    }
    if (!g_blas.create || !g_blas.set_stream || !g_blas.gemm) return "cuBLAS (libcublas.so.13) not found";
    return nullptr;
}

}  // namespace

const char *launch_fwd_unfused(const FwdArgs &a, const void *q, const void *k, const void *v, float *s,
                               void *p, cudaStream_t stream, cudaError_t *err)
{
    *err = cudaSuccess;
    std::lock_guard<std::mutex> lock(g_blas_mutex);
    if (const char *why = load_blas()) return why;
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return "cudaGetDevice";
    if (dev < 0 || dev >= 64) return "device index out of range";
    cublasHandle_t &h = g_blas.handle[dev];
    if (!h && g_blas.create(&h) != CUBLAS_STATUS_SUCCESS) {
        h = nullptr;
        return "cublasCreate failed";
    }
    if (g_blas.set_stream(h, stream) != CUBLAS_STATUS_SUCCESS) return "cublasSetStream failed";
    const int n = a.n, d = a.d, bh = a.bh;
    const long long nd = (long long)n * d, nn = (long long)n * n;
    // Row-major matrices seen as column-major ones (their transposes): S^T = K Q^T, O^T = V^T P^T.
    const float alpha_s = a.scale, one = 1.f, zero = 0.f;
    if (g_blas.gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, n, n, d, &alpha_s, k, CUDA_R_16BF, d, nd, q, CUDA_R_16BF, d,
                    nd, &zero, s, CUDA_R_32F, n, nn, bh, CUBLAS_COMPUTE_32F,
                    CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
        return "cublasGemmStridedBatchedEx (S = Q K^T) failed";
    const long long rows = (long long)bh * n;
    if (n <= kWarpRowMax)
        unfused_softmax_warp_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
            s, reinterpret_cast<__nv_bfloat16 *>(p), a.lse, rows, n);
    else
        unfused_softmax_kernel<<<(unsigned)rows, kSoftmaxThreads, 0, stream>>>(
            s, reinterpret_cast<__nv_bfloat16 *>(p), a.lse, n);
    if ((*err = cudaGetLastError()) != cudaSuccess) return "softmax launch";
    if (g_blas.gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, d, n, n, &one, v, CUDA_R_16BF, d, nd, p, CUDA_R_16BF, n, nn,
                    &zero, a.o, CUDA_R_16BF, d, nd, bh, CUBLAS_COMPUTE_32F,
                    CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
        return "cublasGemmStridedBatchedEx (O = P V) failed";
    return nullptr;
}

}  // namespace attn
