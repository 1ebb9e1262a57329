// Element-wise fp32 vector addition, C = A + B: the kernel of "Self-attention, CUDA kernels and
// FlashAttention", section 2 ("Practical code comparison: raw CUDA C++ vs OpenAI Triton"),
// where one thread adds one element behind an index guard.  Here it serves as the HBM
// bandwidth probe of this library: 16-byte vector loads and stores with streaming cache hints,
// a grid-stride loop over whole waves of the SMs, and the same guard for the ragged tail.
#include "kernels.h"

#include <cuda_runtime.h>

namespace attn {
namespace {

__global__ void __launch_bounds__(256)
    vector_add_kernel(const float *__restrict__ a, const float *__restrict__ b, float *__restrict__ c,
                      long long n)
{
    const long long n4 = n / 4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    const float4 *a4 = reinterpret_cast<const float4 *>(a);
    const float4 *b4 = reinterpret_cast<const float4 *>(b);
    float4 *c4 = reinterpret_cast<float4 *>(c);
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    // two independent 16-byte loads per operand in flight per thread
    for (; i + stride < n4; i += 2 * stride) {
        const float4 x0 = __ldcs(a4 + i), y0 = __ldcs(b4 + i);
        const float4 x1 = __ldcs(a4 + i + stride), y1 = __ldcs(b4 + i + stride);
        __stcs(c4 + i, make_float4(x0.x + y0.x, x0.y + y0.y, x0.z + y0.z, x0.w + y0.w));
        __stcs(c4 + i + stride, make_float4(x1.x + y1.x, x1.y + y1.y, x1.z + y1.z, x1.w + y1.w));
    }
    if (i < n4) {
        const float4 x = __ldcs(a4 + i), y = __ldcs(b4 + i);
        __stcs(c4 + i, make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w));
    }
    // the last n % 4 elements, one thread each, behind the index guard
    const long long t = n4 * 4 + (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < n) c[t] = a[t] + b[t];
}

}  // namespace

cudaError_t launch_vector_add(const float *a, const float *b, float *c, long long n,
                              cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    // whole waves (8 CTAs of 256 threads per SM), fewer for small inputs
    const long long want = (n / 4 + 255) / 256 + 1;
    const long long blocks = want < 8LL * sms ? want : 8LL * sms;
    vector_add_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a, b, c, n);
    return cudaGetLastError();
}

}  // namespace attn
