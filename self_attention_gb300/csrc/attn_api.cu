// The C ABI declared in include/attn.h: argument validation, TMA descriptor construction and
// the device status word.  Compute happens only in the kernels this file launches.
#include "attn.h"
#include "common.cuh"
#include "kernels.h"

#include <cudaTypedefs.h>
#include <cmath>
#include <cstring>
#include <atomic>
#include <cstdio>
#include <mutex>

namespace attn {

// One status word per device (a __device__ variable lives in every device context).
__device__ int g_status_word;

int device_sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int sms = cached[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 148;
        cached[dev].store(sms, std::memory_order_relaxed);
    }
    return sms;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    bool supported = false;
    int *status = nullptr;  // device address of g_status_word on that device
};

std::mutex g_mutex;
thread_local char t_last_error[192] = "no error";

// Records a failed CUDA call for attn_last_error_string() and maps it to ATTN_ERR_LAUNCH.
attn_status fail(const char *what, cudaError_t e)
{
    std::snprintf(t_last_error, sizeof t_last_error, "%s: %s (%s)", what, cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return ATTN_ERR_LAUNCH;
}

attn_status fail_driver(const char *what, CUresult r)
{
    std::snprintf(t_last_error, sizeof t_last_error, "%s: CUresult %d", what, (int)r);
    return ATTN_ERR_LAUNCH;
}
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Resolves, once per device, whether it is an sm_103 part and where its status word is.
attn_status device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return fail("cudaGetDevice", cudaErrorInvalidDevice);
    // Bind the device's primary context to this host thread: the driver calls made below
    // (tensor-map encoding) need a current context, and a thread that has not used this
    // library's runtime before (e.g. an autograd worker) may have none.
    if ((e = cudaSetDevice(dev)) != cudaSuccess) return fail("cudaSetDevice", e);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &s = g_devices[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail("cudaDeviceGetAttribute", e);
        s.supported = (major == 10 && minor == 3);
        if (s.supported) {
            void *p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess)
                return fail("cudaGetSymbolAddress", e);
            s.status = static_cast<int *>(p);
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)",
                            e != cudaSuccess ? e : cudaErrorSymbolNotFound);
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        s.ready = true;
    }
    if (!s.supported) return ATTN_ERR_DEVICE;
    *out = &s;
    return ATTN_OK;
}

// 3-D map over [BH, N, d] bf16 (innermost first: d, N, BH), boxes of 64 x box_rows x 1 with
// the 128-byte swizzle.  Rows past N (or past a head) read as zeros.
CUresult make_map(CUtensorMap *m, const void *base, int bh, int n, int d, int box_rows,
                  CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)bh};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    return g_encode(m, type, 3, const_cast<void *>(base), dims, strides,
                    box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;
};

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

Range span(const void *p, size_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + bytes};
}

attn_status check_sizes(int B, int H, int N, int d_k, float scale)
{
    if (d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED_DK;
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    const long long bh = (long long)B * H;
    if (bh > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (bh * (long long)N * d_k >= (1LL << 40)) return ATTN_ERR_INVALID_ARG;
    // one CTA per 256 query rows of a head must fit a 1-D grid
    if (bh * (((long long)N + 255) / 256) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Whether the forward rounds V to fp16 in one pass ahead of the kernel (given a workspace)
// rather than in each CTA's shared memory.  The in-kernel rewrite costs shared-memory bandwidth
// per (query block, key tile) pair, the pass HBM traffic per element of V, so the pass pays
// from a sequence length on, which the per-CTA query rows set (256 at d = 128, 128 at d = 64).
// Measured crossovers (forward alone, GB300): d = 64 between N = 576 and N = 4096, d = 128
// between N = 4096 and N = 16384.
bool fwd_v_prepass(int N, int d_k) { return d_k == 64 ? N >= 2048 : N >= 8192; }

// The forward behind attn_fwd (v16 == nullptr), attn_fwd_with_workspace (v16: the fp16 copy of
// V) and attn_fwd_diagnostic (o32: O before its bf16 rounding as well).
attn_status run_fwd(const void *q, const void *k, const void *v, void *o, float *lse, void *v16,
                    size_t v16_bytes, int B, int H, int N, int d_k, float scale, cudaStream_t stream,
                    float *o32 = nullptr)
{
    attn_status st = check_sizes(B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    const long long bh = (long long)B * H;
    const size_t tbytes = (size_t)bh * N * d_k * 2, lbytes = (size_t)bh * N * 4;
    const Range ins[3] = {span(q, tbytes), span(k, tbytes), span(v, tbytes)};
    const Range ro = span(o, tbytes), rl = span(lse, lbytes);
    if (overlap(ro, rl)) return ATTN_ERR_INVALID_ARG;
    for (const Range &r : ins)
        if (overlap(r, ro) || overlap(r, rl)) return ATTN_ERR_INVALID_ARG;
    if (v16) {
        if ((reinterpret_cast<uintptr_t>(v16) & 255u) || v16_bytes < align256(tbytes)) return ATTN_ERR_WORKSPACE;
        const Range rw = span(v16, align256(tbytes));
        if (overlap(rw, ro) || overlap(rw, rl)) return ATTN_ERR_INVALID_ARG;
        for (const Range &r : ins)
            if (overlap(r, rw)) return ATTN_ERR_INVALID_ARG;
    }
    if (o32) {
        if (!aligned16(o32)) return ATTN_ERR_MISALIGNED;
        const Range r32 = span(o32, tbytes * 2);
        if (overlap(r32, ro) || overlap(r32, rl)) return ATTN_ERR_INVALID_ARG;
        for (const Range &r : ins)
            if (overlap(r, r32)) return ATTN_ERR_INVALID_ARG;
    }

    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    FwdArgs a;
    std::memset(&a, 0, sizeof a);
    CUresult r;
    if ((r = make_map(&a.tm_q, q, (int)bh, N, d_k, 128)) != CUDA_SUCCESS ||
        (r = make_map(&a.tm_k, k, (int)bh, N, d_k, 128)) != CUDA_SUCCESS ||
        (r = v16 ? make_map(&a.tm_v, v16, (int)bh, N, d_k, 128, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)
                 : make_map(&a.tm_v, v, (int)bh, N, d_k, 128)) != CUDA_SUCCESS ||
        (r = make_map(&a.tm_o, o, (int)bh, N, d_k, 128)) != CUDA_SUCCESS)
        return fail_driver("cuTensorMapEncodeTiled", r);
    a.o = o;
    a.lse = lse;
    a.bh = (int)bh;
    a.n = N;
    a.d = d_k;
    a.scale = scale;
    a.v_f16 = v16 ? 1 : 0;
    a.o32 = o32;
    a.status = dev->status;
    cudaError_t e;
    if (v16 && (e = launch_v_to_f16(v, v16, bh * N * d_k, stream)) != cudaSuccess)
        return fail("attn_fwd_with_workspace V to fp16 launch", e);
    e = launch_fwd(a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_fwd launch", e);
}

}  // namespace

extern "C" attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int H, int N, int d_k, float scale, cudaStream_t stream)
{
    return run_fwd(q, k, v, o, lse, nullptr, 0, B, H, N, d_k, scale, stream);
}

extern "C" attn_status attn_fwd_diagnostic(const void *q, const void *k, const void *v, void *o, float *lse,
                                           float *o32, int B, int H, int N, int d_k, float scale,
                                           cudaStream_t stream)
{
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return run_fwd(q, k, v, o, lse, nullptr, 0, B, H, N, d_k, scale, stream, o32);
}

extern "C" size_t attn_fwd_workspace_size(int B, int H, int N, int d_k)
{
    if (check_sizes(B, H, N, d_k, 1.0f) != ATTN_OK || !fwd_v_prepass(N, d_k)) return 0;
    return align256((size_t)B * H * N * d_k * 2);
}

extern "C" attn_status attn_fwd_with_workspace(const void *q, const void *k, const void *v, void *o,
                                               float *lse, void *workspace, size_t workspace_bytes, int B,
                                               int H, int N, int d_k, float scale, cudaStream_t stream)
{
    attn_status st = check_sizes(B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    if (!fwd_v_prepass(N, d_k)) return run_fwd(q, k, v, o, lse, nullptr, 0, B, H, N, d_k, scale, stream);
    if (!workspace) return ATTN_ERR_WORKSPACE;
    return run_fwd(q, k, v, o, lse, workspace, workspace_bytes, B, H, N, d_k, scale, stream);
}

namespace {

// Workspace layout (every region 256-byte aligned), with N_pad = N rounded up to 128:
//   stats [BH][N_pad / 2][4] fp32  per pair of rows: -lse * log2(e) of both rows, then
//                                  -rowsum(dO o O) of both; -inf and 0 in the padding
//                                  (probabilities there are 0)
//   dQacc [BH][N][d]          fp32  dQ accumulator (unscaled)
struct WorkspaceLayout {
    size_t stats_off, acc_off, total;
};

WorkspaceLayout workspace_layout(long long bh, int N, int d_k)
{
    const size_t n_pad = ((size_t)N + 127) / 128 * 128;
    WorkspaceLayout w;
    w.stats_off = 0;
    w.acc_off = align256((size_t)bh * n_pad * 8);
    w.total = w.acc_off + align256((size_t)bh * N * d_k * 4);
    return w;
}

}  // namespace

extern "C" size_t attn_bwd_workspace_size(int B, int H, int N, int d_k)
{
    if (check_sizes(B, H, N, d_k, 1.0f) != ATTN_OK) return 0;
    return workspace_layout((long long)B * H, N, d_k).total;
}

namespace {

enum Phase : unsigned { kPre = 1, kMain = 2, kConv = 4 };

// Validates what the requested backward phases need and fills `a`.  Operands a phase does
// not use may be null; they are neither checked nor mapped.  The workspace is always needed.
attn_status prepare_bwd(BwdArgs &a, unsigned phases, const void *q, const void *k, const void *v,
                        const void *o, const void *dout, const float *lse, void *dq, void *dk,
                        void *dv, void *workspace, size_t workspace_bytes, int B, int H, int N,
                        int d_k, float scale)
{
    attn_status st = check_sizes(B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    const bool pre = phases & kPre, main = phases & kMain, conv = phases & kConv;
    if ((pre && (!o || !dout || !lse)) || (main && (!q || !k || !v || !dout || !dk || !dv)) ||
        (conv && !dq))
        return ATTN_ERR_INVALID_ARG;
    const void *all[9] = {q, k, v, o, dout, lse, dq, dk, dv};
    const bool used[9] = {main, main, main, pre, pre || main, pre, conv, main, main};
    for (int i = 0; i < 9; ++i)
        if (used[i] && !aligned16(all[i])) return ATTN_ERR_MISALIGNED;
    const long long bh = (long long)B * H;
    const WorkspaceLayout wl = workspace_layout(bh, N, d_k);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < wl.total)
        return ATTN_ERR_WORKSPACE;
    const size_t tbytes = (size_t)bh * N * d_k * 2, lbytes = (size_t)bh * N * 4;
    // inputs: q k v o dout lse ; outputs: workspace dq dk dv
    Range outs[4];
    int n_out = 0;
    outs[n_out++] = span(workspace, wl.total);
    if (conv) outs[n_out++] = span(dq, tbytes);
    if (main) {
        outs[n_out++] = span(dk, tbytes);
        outs[n_out++] = span(dv, tbytes);
    }
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < 6; ++j)
            if (used[j] && overlap(span(all[j], j == 5 ? lbytes : tbytes), outs[i]))
                return ATTN_ERR_INVALID_ARG;
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(outs[i], outs[j])) return ATTN_ERR_INVALID_ARG;
    }

    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    std::memset(&a, 0, sizeof a);
    CUresult r;
    if (main && ((r = make_map(&a.tm_q, q, (int)bh, N, d_k, 64)) != CUDA_SUCCESS ||
                 (r = make_map(&a.tm_k, k, (int)bh, N, d_k, 128)) != CUDA_SUCCESS ||
                 (r = make_map(&a.tm_v, v, (int)bh, N, d_k, 128)) != CUDA_SUCCESS ||
                 (r = make_map(&a.tm_do, dout, (int)bh, N, d_k, 64)) != CUDA_SUCCESS ||
                 (r = make_map(&a.tm_dk, dk, (int)bh, N, d_k, 128)) != CUDA_SUCCESS ||
                 (r = make_map(&a.tm_dv, dv, (int)bh, N, d_k, 128)) != CUDA_SUCCESS))
        return fail_driver("cuTensorMapEncodeTiled", r);
    char *ws = static_cast<char *>(workspace);
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.stats = reinterpret_cast<float *>(ws + wl.stats_off);
    a.dq_acc = reinterpret_cast<float *>(ws + wl.acc_off);
    a.bh = (int)bh;
    a.n = N;
    a.n_pad = (N + 127) / 128 * 128;
    a.d = d_k;
    a.scale = scale;
    a.status = dev->status;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_bwd_preprocess(const void *o, const void *dout, const float *lse,
                                           void *workspace, size_t workspace_bytes, int B, int H,
                                           int N, int d_k, cudaStream_t stream)
{
    BwdArgs a;
    attn_status st = prepare_bwd(a, kPre, nullptr, nullptr, nullptr, o, dout, lse, nullptr, nullptr,
                                 nullptr, workspace, workspace_bytes, B, H, N, d_k, 1.0f);
    if (st != ATTN_OK) return st;
    const cudaError_t e = launch_bwd_preprocess(a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_bwd_preprocess launch", e);
}

extern "C" attn_status attn_bwd_main(const void *q, const void *k, const void *v, const void *dout,
                                     void *dk, void *dv, void *workspace, size_t workspace_bytes,
                                     int B, int H, int N, int d_k, float scale, cudaStream_t stream)
{
    BwdArgs a;
    attn_status st = prepare_bwd(a, kMain, q, k, v, nullptr, dout, nullptr, nullptr, dk, dv,
                                 workspace, workspace_bytes, B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    const cudaError_t e = launch_bwd_main(a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_bwd_main launch", e);
}

extern "C" attn_status attn_bwd_dq_convert(void *workspace, size_t workspace_bytes, void *dq,
                                           int B, int H, int N, int d_k, float scale,
                                           cudaStream_t stream)
{
    BwdArgs a;
    attn_status st = prepare_bwd(a, kConv, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq,
                                 nullptr, nullptr, workspace, workspace_bytes, B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    const cudaError_t e = launch_bwd_convert(a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_bwd_dq_convert launch", e);
}

extern "C" attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                                const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                void *workspace, size_t workspace_bytes, int B, int H, int N,
                                int d_k, float scale, cudaStream_t stream)
{
    BwdArgs a;
    attn_status st = prepare_bwd(a, kPre | kMain | kConv, q, k, v, o, dout, lse, dq, dk, dv,
                                 workspace, workspace_bytes, B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    // short sequences at d = 64 over few heads: one kernel, dQ accumulated on chip (the
    // workspace is unused)
    if (bwd_whole_heads(N, d_k, (long long)B * H)) {
        const cudaError_t e = launch_bwd_heads(a, stream);
        return e == cudaSuccess ? ATTN_OK : fail("attn_bwd launch", e);
    }
    cudaError_t e = launch_bwd_preprocess(a, stream);
    if (e == cudaSuccess) e = launch_bwd_main(a, stream);
    if (e == cudaSuccess) e = launch_bwd_convert(a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_bwd launch", e);
}

extern "C" attn_status attn_bwd_deterministic(const void *q, const void *k, const void *v,
                                              const void *o, const void *dout, const float *lse,
                                              void *dq, void *dk, void *dv, void *workspace,
                                              size_t workspace_bytes, int B, int H, int N, int d_k,
                                              float scale, cudaStream_t stream)
{
    BwdArgs a;
    attn_status st = prepare_bwd(a, kPre | kMain | kConv, q, k, v, o, dout, lse, dq, dk, dv,
                                 workspace, workspace_bytes, B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    // the whole-head kernel uses no atomics either
    const cudaError_t e = bwd_whole_heads(N, d_k, (long long)B * H) ? launch_bwd_heads(a, stream)
                                                                     : launch_bwd_deterministic(a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_bwd_deterministic launch", e);
}

extern "C" attn_status attn_get_device_status(cudaStream_t stream)
{
    DeviceState *dev = nullptr;
    attn_status st = device_state(&dev);
    if (st != ATTN_OK) return st;
    int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, dev->status, sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return fail("cudaMemcpyAsync(status)", e);
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return fail("cudaStreamSynchronize", e);
    if (word != 0) {
        if ((e = cudaMemsetAsync(dev->status, 0, sizeof(int), stream)) != cudaSuccess ||
            (e = cudaStreamSynchronize(stream)) != cudaSuccess)
            return fail("clearing the status word", e);
    }
    return word == 0 ? ATTN_OK : static_cast<attn_status>(word);
}

extern "C" const char *attn_status_string(attn_status status)
{
    switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED_DK: return "ATTN_ERR_UNSUPPORTED_DK: d_k must be 64 or 128";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED: pointers must be 16-byte aligned";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH: CUDA runtime error";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a kernel wait gave up";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE: the current device is not an sm_103 GPU";
    case ATTN_ERR_TOO_LARGE:
        return "ATTN_ERR_TOO_LARGE: the sizes need more scratch than attn_bwd_noalloc's fixed 64 MiB";
    }
    return "unknown attn_status";
}

extern "C" attn_status attn_debug_wait_timeout(unsigned limit_us, cudaStream_t stream)
{
    if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_INVALID_ARG;
    DeviceState *dev = nullptr;
    attn_status st = device_state(&dev);
    if (st != ATTN_OK) return st;
    const cudaError_t e = launch_wait_selftest(dev->status, (uint64_t)limit_us * 1000ull, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_debug_wait_timeout launch", e);
}

extern "C" const char *attn_last_error_string(void) { return t_last_error; }

namespace {

attn_status check_proj(const void *x, const void *const w[3], int B, int N, int D, int H, int d_k)
{
    if (d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED_DK;
    if (B < 1 || N < 1 || H < 1 || D != H * d_k || D % 128 != 0) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * N * D >= (1LL << 40) || (long long)B * H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    // the token rows B * N index the operand tensor maps as an int
    if ((long long)B * N > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if (!x || !w[0] || !w[1] || !w[2]) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w[0]) || !aligned16(w[1]) || !aligned16(w[2])) return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_qkv_proj(const void *x, const void *w_q, const void *w_k,
                                     const void *w_v, void *q, void *k, void *v, int B, int N,
                                     int D, int H, int d_k, cudaStream_t stream)
{
    const void *w[3] = {w_q, w_k, w_v};
    void *out[3] = {q, k, v};
    attn_status st = check_proj(x, w, B, N, D, H, d_k);
    if (st != ATTN_OK) return st;
    const size_t xbytes = (size_t)B * N * D * 2, wbytes = (size_t)D * D * 2;
    for (int t = 0; t < 3; ++t) {
        if (!out[t]) return ATTN_ERR_INVALID_ARG;
        if (!aligned16(out[t])) return ATTN_ERR_MISALIGNED;
        if (overlap(span(out[t], xbytes), span(x, xbytes))) return ATTN_ERR_INVALID_ARG;
        for (int u = 0; u < 3; ++u) {
            if (overlap(span(out[t], xbytes), span(w[u], wbytes))) return ATTN_ERR_INVALID_ARG;
            if (u > t && overlap(span(out[t], xbytes), span(out[u], xbytes))) return ATTN_ERR_INVALID_ARG;
        }
    }
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    ProjMaps m;
    std::memset(&m, 0, sizeof m);
    CUresult r = make_map(&m.a[0], x, 1, B * N, D, 128);            // X as [B*N, D]
    for (int t = 0; t < 3 && r == CUDA_SUCCESS; ++t) r = make_map(&m.b[t], w[t], 1, D, D, 64);
    if (r != CUDA_SUCCESS) return fail_driver("cuTensorMapEncodeTiled", r);
    m.a[1] = m.a[2] = m.a[0];
    ProjArgs a = {};
    a.B = B; a.N = N; a.D = D; a.H = H; a.dk = d_k; a.status = dev->status;
    for (int t = 0; t < 3; ++t) a.qkv[t] = static_cast<__nv_bfloat16 *>(out[t]);
    const cudaError_t e = launch_proj_fwd(m, a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_qkv_proj launch", e);
}

extern "C" attn_status attn_qkv_proj_bwd(const void *x, const void *w_q, const void *w_k,
                                         const void *w_v, const void *dq, const void *dk,
                                         const void *dv, void *dx, float *dw_q, float *dw_k,
                                         float *dw_v, int B, int N, int D, int H, int d_k,
                                         cudaStream_t stream)
{
    const void *w[3] = {w_q, w_k, w_v};
    const void *dy[3] = {dq, dk, dv};
    float *dw[3] = {dw_q, dw_k, dw_v};
    attn_status st = check_proj(x, w, B, N, D, H, d_k);
    if (st != ATTN_OK) return st;
    if (!dx) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(dx)) return ATTN_ERR_MISALIGNED;
    const size_t xbytes = (size_t)B * N * D * 2, wbytes = (size_t)D * D * 2, dwbytes = (size_t)D * D * 4;
    Range ins[7] = {span(x, xbytes), span(w[0], wbytes), span(w[1], wbytes), span(w[2], wbytes),
                    span(dy[0], xbytes), span(dy[1], xbytes), span(dy[2], xbytes)};
    Range outs[4] = {span(dx, xbytes), span(dw[0], dwbytes), span(dw[1], dwbytes), span(dw[2], dwbytes)};
    for (int t = 0; t < 3; ++t) {
        if (!dy[t] || !dw[t]) return ATTN_ERR_INVALID_ARG;
        if (!aligned16(dy[t]) || !aligned16(dw[t])) return ATTN_ERR_MISALIGNED;
    }
    for (int i = 0; i < 4; ++i) {
        for (const Range &r : ins)
            if (overlap(r, outs[i])) return ATTN_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (overlap(outs[i], outs[j])) return ATTN_ERR_INVALID_ARG;
    }
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    ProjArgs a = {};
    a.B = B; a.N = N; a.D = D; a.H = H; a.dk = d_k; a.status = dev->status;
    a.dx = static_cast<__nv_bfloat16 *>(dx);
    for (int t = 0; t < 3; ++t) a.dw[t] = dw[t];
    // dX = sum_t dY_t W_t^T: A = dY_t as [dk, N, B*H] (128-row boxes), B = W_t (128-row boxes)
    ProjMaps mx;
    std::memset(&mx, 0, sizeof mx);
    CUresult r = CUDA_SUCCESS;
    for (int t = 0; t < 3 && r == CUDA_SUCCESS; ++t) {
        r = make_map(&mx.a[t], dy[t], B * H, N, d_k, 128);
        if (r == CUDA_SUCCESS) r = make_map(&mx.b[t], w[t], 1, D, D, 128);
    }
    // dW_t = X^T dY_t: A = X as [D, N, B] (64-row boxes), B = dY_t (64-row boxes)
    ProjMaps mw;
    std::memset(&mw, 0, sizeof mw);
    if (r == CUDA_SUCCESS) r = make_map(&mw.a[0], x, B, N, D, 64);
    for (int t = 0; t < 3 && r == CUDA_SUCCESS; ++t) r = make_map(&mw.b[t], dy[t], B * H, N, d_k, 64);
    if (r != CUDA_SUCCESS) return fail_driver("cuTensorMapEncodeTiled", r);
    mw.a[1] = mw.a[2] = mw.a[0];
    cudaError_t e = launch_proj_dx(mx, a, stream);
    if (e == cudaSuccess) e = launch_proj_dw(mw, a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_qkv_proj_bwd launch", e);
}

extern "C" attn_status vector_add(const float *a, const float *b, float *c, long long n,
                                  cudaStream_t stream)
{
    if (n < 0) return ATTN_ERR_INVALID_ARG;
    if (n == 0) return ATTN_OK;
    if (!a || !b || !c) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return ATTN_ERR_MISALIGNED;
    const size_t bytes = (size_t)n * 4;
    // c may be a or b (in-place addition is element-wise safe); partial overlaps are not
    const Range rc = span(c, bytes), ra = span(a, bytes), rb = span(b, bytes);
    if ((overlap(rc, ra) && c != a) || (overlap(rc, rb) && c != b)) return ATTN_ERR_INVALID_ARG;
    DeviceState *dev = nullptr;
    attn_status st = device_state(&dev);
    if (st != ATTN_OK) return st;
    const cudaError_t e = launch_vector_add(a, b, c, n, stream);
    return e == cudaSuccess ? ATTN_OK : fail("vector_add launch", e);
}

// --------------------------------------------------------------------------------------------
// Standard attention (S and P materialised in HBM), the comparison point of the fused path.
namespace {

struct UnfusedLayout {
    size_t p_off, total;
};

UnfusedLayout unfused_layout(long long bh, int N)
{
    UnfusedLayout w;
    w.p_off = align256((size_t)bh * N * N * 4);
    w.total = w.p_off + align256((size_t)bh * N * N * 2);
    return w;
}

attn_status check_unfused(int B, int H, int N, int d_k, float scale)
{
    attn_status st = check_sizes(B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    // one softmax block per row; the library GEMMs take int sizes and long long strides
    if ((long long)B * H * N > 0x7fffffffLL || (long long)B * H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * H * N * N >= (1LL << 40)) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

}  // namespace

extern "C" size_t attn_fwd_unfused_workspace_size(int B, int H, int N, int d_k)
{
    if (check_unfused(B, H, N, d_k, 1.0f) != ATTN_OK) return 0;
    return unfused_layout((long long)B * H, N).total;
}

extern "C" attn_status attn_fwd_unfused(const void *q, const void *k, const void *v, void *o, float *lse,
                                        void *workspace, size_t workspace_bytes, int B, int H, int N,
                                        int d_k, float scale, cudaStream_t stream)
{
    attn_status st = check_unfused(B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    const long long bh = (long long)B * H;
    const UnfusedLayout lay = unfused_layout(bh, N);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < lay.total)
        return ATTN_ERR_WORKSPACE;
    const size_t tbytes = (size_t)bh * N * d_k * 2, lbytes = (size_t)bh * N * 4;
    const Range ins[3] = {span(q, tbytes), span(k, tbytes), span(v, tbytes)};
    const Range outs[3] = {span(o, tbytes), span(lse, lbytes), span(workspace, lay.total)};
    for (int i = 0; i < 3; ++i) {
        for (const Range &r : ins)
            if (overlap(r, outs[i])) return ATTN_ERR_INVALID_ARG;
        for (int j = i + 1; j < 3; ++j)
            if (overlap(outs[i], outs[j])) return ATTN_ERR_INVALID_ARG;
    }
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    FwdArgs a;
    std::memset(&a, 0, sizeof a);
    a.o = o;
    a.lse = lse;
    a.bh = (int)bh;
    a.n = N;
    a.d = d_k;
    a.scale = scale;
    a.status = dev->status;
    float *s = static_cast<float *>(workspace);
    void *p = static_cast<char *>(workspace) + lay.p_off;
    cudaError_t e = cudaSuccess;
    if (const char *why = launch_fwd_unfused(a, q, k, v, s, p, stream, &e)) {
        if (e != cudaSuccess) return fail(why, e);
        std::snprintf(t_last_error, sizeof t_last_error, "attn_fwd_unfused: %s", why);
        return ATTN_ERR_LAUNCH;
    }
    return ATTN_OK;
}

// --------------------------------------------------------------------------------------------
// The wait self-test kernel: one thread waits on an mbarrier that nothing arrives on.
namespace attn {
namespace {
__global__ void wait_selftest_kernel(int *status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_sh;
    abort_sh = 0;
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    const Guard g{&abort_sh, status, limit_ns};
    wait_bounded(&bar, 0, g);
}
}  // namespace

cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 1, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}
}  // namespace attn

// --------------------------------------------------------------------------------------------
// attn_bwd_noalloc: attn_bwd for callers that cannot allocate device memory.  Its scratch (the
// D and LSE2 vectors and the fp32 dQ accumulator that attn_bwd keeps in the caller's
// workspace) lives in one fixed array compiled into the library.
namespace attn {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

// Every GPU that loads this library holds this array (64 MiB) until the process exits.  In host
// code its name is only a stand-in for the symbol, never a device address: the address comes
// from cudaGetSymbolAddress, once per device, below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device
}  // namespace
}  // namespace attn

extern "C" attn_status attn_bwd_noalloc(const void *q, const void *k, const void *v,
                                        const void *o, const void *dout, const float *lse,
                                        void *dq, void *dk, void *dv, int B, int H, int N,
                                        int d_k, float scale, cudaStream_t stream)
{
    attn_status st = check_sizes(B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    const size_t need = attn_bwd_workspace_size(B, H, N, d_k);
    if (need > kNoAllocScratchBytes) return ATTN_ERR_TOO_LARGE;

    // device_state() makes this thread's current device current in the driver too, which
    // cudaGetSymbolAddress needs; the address is looked up once per device and cached.
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != ATTN_OK) return st;
    int id = 0;
    cudaError_t e = cudaGetDevice(&id);
    if (e != cudaSuccess) return fail("cudaGetDevice", e);
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (!g_scratch_addr[id]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) return fail("cudaGetSymbolAddress(g_noalloc_scratch)", e);
            g_scratch_addr[id] = p;
        }
        scratch = g_scratch_addr[id];
    }

    // The same three phases as attn_bwd; the preprocess phase rewrites every scratch byte the
    // later phases read (D, LSE2 and the zeroed accumulator), so what an earlier call left in
    // the array does not matter.
    BwdArgs a;
    st = prepare_bwd(a, kPre | kMain | kConv, q, k, v, o, dout, lse, dq, dk, dv, scratch,
                     kNoAllocScratchBytes, B, H, N, d_k, scale);
    if (st != ATTN_OK) return st;
    e = launch_bwd_preprocess(a, stream);
    if (e == cudaSuccess) e = launch_bwd_main(a, stream);
    if (e == cudaSuccess) e = launch_bwd_convert(a, stream);
    return e == cudaSuccess ? ATTN_OK : fail("attn_bwd_noalloc launch", e);
}
