// Host-side launchers of the attention kernels (internal to the library; the public C ABI
// in include/attn.h validates arguments and calls these).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cuda_bf16.h>

namespace attn {

struct FwdArgs {
    CUtensorMap tm_q, tm_k, tm_v;   // 3-D maps over [BH, N, d] bf16, 64 x rows boxes, 128-byte swizzle
    CUtensorMap tm_o;               // the same over O (128-row boxes), for tile stores
    void *o;                        // [BH, N, d] bf16
    float *lse;                     // [BH, N] fp32
    int bh, n, d;
    float scale;
    int v_f16;                      // 1: tm_v maps an fp16 copy of V (no rewrite in shared memory)
    float *o32;                     // null, or [BH, N, d] fp32: O before its bf16 rounding (diagnostic)
    int *status;                    // device status word
};

struct BwdArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    CUtensorMap tm_dk, tm_dv;       // dK and dV with 128-row boxes (tile stores, d = 64)
    const void *o, *dout;           // [BH, N, d] bf16
    const float *lse;               // [BH, N]
    void *dq, *dk, *dv;             // [BH, N, d] bf16
    // [BH, n_pad / 2] x 4 fp32 workspace, per pair of rows (2k, 2k + 1):
    // {-lse log2 e of both rows, -rowsum(dO o O) of both rows}; -inf and 0 past N.
    float *stats;
    float *dq_acc;                  // [BH, N, d]  workspace: fp32 dQ accumulator
    int bh, n, n_pad, d;
    float scale;
    int *status;
};

// Streaming multiprocessors of the current device (cached per device, safe to call from several
// host threads).
int device_sm_count();

cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t stream);
// v16[i] = v[i] rounded from bf16 to fp16, elems a multiple of 8, both 16-byte aligned.
cudaError_t launch_v_to_f16(const void *v, void *v16, long long elems, cudaStream_t stream);
// The three stream-ordered phases of the backward pass.
cudaError_t launch_bwd_preprocess(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_bwd_convert(const BwdArgs &a, cudaStream_t stream);
// Short sequences at d = 64 (N <= 256): the whole backward (statistics, dQ, dK, dV) in one
// kernel, one CTA per head, dQ accumulated on chip; used by attn_bwd and
// attn_bwd_deterministic where bwd_whole_heads(n, d, B*H) holds.
bool bwd_whole_heads(int n, int d, long long bh);
cudaError_t launch_bwd_heads(const BwdArgs &a, cudaStream_t stream);
// The deterministic backward: preprocess (no accumulator), the main kernel without its dQ part,
// then a query-stationary pass that computes dQ without atomics.
cudaError_t launch_bwd_deterministic(const BwdArgs &a, cudaStream_t stream);
// QKV projection (see proj.cu): tensor maps of the two operands (up to three each) and sizes.
struct ProjMaps {
    CUtensorMap a[3], b[3];
};
struct ProjArgs {
    int B, N, D, H, dk;
    __nv_bfloat16 *qkv[3];   // forward outputs Q, K, V [B,H,N,dk]
    __nv_bfloat16 *dx;       // [B,N,D]
    float *dw[3];            // [D,D] each
    int *status;
};
cudaError_t launch_proj_fwd(const ProjMaps &m, const ProjArgs &a, cudaStream_t stream);
cudaError_t launch_proj_dx(const ProjMaps &m, const ProjArgs &a, cudaStream_t stream);
cudaError_t launch_proj_dw(const ProjMaps &m, const ProjArgs &a, cudaStream_t stream);

// Standard attention (S and P through HBM; see unfused.cu): returns nullptr on success, else what
// failed (with *err set where a CUDA call failed).  s: [BH][N][N] fp32, p: [BH][N][N] bf16.
const char *launch_fwd_unfused(const FwdArgs &a, const void *q, const void *k, const void *v, float *s,
                               void *p, cudaStream_t stream, cudaError_t *err);

cudaError_t launch_vector_add(const float *a, const float *b, float *c, long long n,
                              cudaStream_t stream);
cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace attn
