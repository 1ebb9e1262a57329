// Backward pass of exact multi-head attention for sm_103a.
//
// "Self-attention, CUDA kernels and FlashAttention", section 3 ("Recomputation in
// backpropagation"): the forward pass keeps only a small per-row statistic (here LSE, the
// natural-log log-sum-exp of each row of scaled scores); the backward pass recomputes the
// attention tiles on chip from it instead of reading an N x N matrix from HBM.  The article
// prints no gradient formulas; these are the chain rule on section 1's formulas:
//   P = exp(scale * Q K^T - LSE),  dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
//   dS = P o (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three stream-ordered kernels:
//   1. preprocess: -D = -rowsum(dO o O) and -LSE2 = -LSE log2 e (fp32, rows padded to a
//      multiple of 128 with 0 and -inf so that padded queries get zero probability), and zero
//      the fp32 dQ accumulator.
//   2. main: one CTA per 128-key tile j of one head, looping over all 64-row query tiles i.
//        warp 12     TMA producer: K_j and V_j once; a ring of (Q_i, dO_i, LSE2_i, D_i).
//        warp 13     tcgen05 issuer, per query tile i (TMEM buffer b = i & 1):
//                      dV += P^T dO_i (P^T from TMEM), dQ_i^T = K_j^T dS^T (over P^T),
//                      dK += dS^T Q_i, then dP^T = V_j dO^T and S^T = K_j Q^T of tile i + 2.
//        warps 0-7   two warpgroups, alternating query tiles; thread = key row:
//                    P^T = 2^(S^T c - LSE log2 e), dS^T = P^T o (dP^T - D); P^T (bf16) goes back
//                    into TMEM over S^T, dS^T (bf16) into shared memory.  At the end group 0
//                    writes dK (times scale) and group 1 writes dV, in bf16.
//        warps 8-11  thread = one of the d columns: move dQ_i^T from TMEM to shared memory
//                    (transposed to dQ_i rows, two double-buffered halves) and add it into the
//                    fp32 accumulator with bulk reduce-adds (fp32 atomics in L2, whose
//                    throughput, ~6 TB/s on this part, bounds this loop; low bits of dQ vary
//                    from run to run).
//   3. convert: dQ = bf16(scale * accumulator).
// TMEM columns: dK [0,d), dV [d,2d), then two buffers of {S^T/P^T/dQ^T (64), dP^T (64)}.
// dQ^T has M = d rows; for d = 64 the MMA still runs with M = 128 and lanes 64-127 are unused.
//
// Further in this file: the d = 64 main kernels with 128-query tiles (one CTA per key block,
// and a persistent one over (head, key block) items), the deterministic mode's dK / dV pass for
// d = 128 and its query-stationary dQ pass, and, for short d = 64 sequences over few heads, a
// kernel that takes each head whole (statistics, all products and dQ, dK, dV in one launch,
// dQ accumulated in TMEM).
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
// Longest sequence for which the d = 64 backward runs as a persistent kernel.
constexpr int kBwdPersistentMaxN = 4096;

template <int D>
struct BwdCfg {
    static constexpr int BN = 128;   // keys per CTA (TMEM lanes of S^T, dP^T, dK, dV)
    static constexpr int BM = 64;    // queries per inner tile
    static constexpr int QST = (D == 64) ? 6 : 3;  // (Q, dO, LSE2, D) ring depth
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int STAGE_BYTES = 2 * Q_BYTES;   // Q_i then dO_i (swizzled tiles)
    static constexpr int LD_BYTES = 2 * BM * 4;       // LSE2_i then D_i (fp32) per stage
    static constexpr int DS_BYTES = BN * BM * 2;
    static constexpr int DQH_BYTES = (BM / 2) * D * 4;  // dQ staging: half a query tile
    static constexpr int SMEM_BYTES =
        2 * KV_BYTES + QST * STAGE_BYTES + 2 * DS_BYTES + 2 * DQH_BYTES + QST * LD_BYTES + 1024;
    static constexpr int THREADS = 448;
    static constexpr uint32_t TM_DK = 0, TM_DV = D, TM_BUF = 2 * D;
    __host__ __device__ static constexpr uint32_t tm_s(int b) { return TM_BUF + b * 128; }
    __host__ __device__ static constexpr uint32_t tm_dp(int b) { return TM_BUF + b * 128 + 64; }
};

// ------------------------------------------------------------------ 1. preprocess
// Over the padded rows (bh, i), i < n_pad, the negated statistics the later kernels add:
// -D = -sum_c dO_ic O_ic and -LSE2 = -lse log2(e) for i < n; 0 and -inf in the padding (zero
// probability there), interleaved per pair of rows as {-LSE2_2k, -LSE2_2k+1, -D_2k, -D_2k+1}
// so that one 16-byte load gives the packed operands for two queries.  Then zero the dQ
// accumulator.
// Layout: D / 8 consecutive threads share a row, 16 bytes of O and of dO each; a pass takes
// kPreRows rows per thread, all loads issued before any is reduced, so that each thread keeps
// several 16-byte loads in flight.  The padded row index g = h n_pad + i advances by a fixed
// stride, kept as (h, i) without a division per row.
constexpr int kPreRows = 4;

template <int D>
__global__ void __launch_bounds__(256, 4)
    bwd_preprocess_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                          const float *__restrict__ lse, float *__restrict__ stats,
                          float *__restrict__ dq_acc, int bh, int n,
                          int n_pad, int zero_acc)
{
    constexpr int TPR = D / 8;         // threads per row
    constexpr int RPW = 32 / TPR;      // rows per warp
    const int part = threadIdx.x % TPR;
    const long long rows = (long long)bh * n_pad;
    const long long stride = (long long)gridDim.x * (blockDim.x / TPR);   // rows per step
    const long long g_first = (long long)blockIdx.x * (blockDim.x / TPR) + threadIdx.x / TPR;
    // The loop tests the warp's first row, so whole warps run the same passes and the
    // shuffles below always see all 32 lanes.
    const long long g_warp = g_first - (threadIdx.x % 32) / TPR;
    const long long step_h = stride / n_pad;
    const int step_i = (int)(stride % n_pad);
    long long h = g_first / n_pad;
    int i = (int)(g_first % n_pad);
    for (long long gw = g_warp, g = g_first; gw < rows; gw += kPreRows * stride, g += kPreRows * stride) {
        uint4 a[kPreRows], b[kPreRows];
        float l[kPreRows];   // LSE of the row; +inf for a padding row, whose -LSE2 is -inf
#pragma unroll
        for (int u = 0; u < kPreRows; ++u) {
            const bool live = g + u * stride < rows && i < n;
            const long long row = h * n + i;
            a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
            l[u] = INFINITY;
            if (live) {
                a[u] = *reinterpret_cast<const uint4 *>(o + row * D + part * 8);
                b[u] = *reinterpret_cast<const uint4 *>(dout + row * D + part * 8);
                if (part == 0) l[u] = lse[row];
            }
            i += step_i;
            h += step_h;
            if (i >= n_pad) {
                i -= n_pad;
                ++h;
            }
        }
#pragma unroll
        for (int u = 0; u < kPreRows; ++u) {
            const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a[u]);
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&b[u]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = __bfloat1622float2(a2[e]);
                const float2 fb = __bfloat1622float2(b2[e]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const long long prow = g + u * stride;
            if (prow < rows && part == 0) {
                float *pair = stats + (prow >> 1) * 4 + (prow & 1);   // n_pad is even
                pair[0] = -l[u] * kLog2e;
                pair[2] = -acc;
            }
        }
    }
    static_assert(RPW * TPR == 32, "a warp covers whole rows");
    if (!zero_acc) return;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nthreads = (long long)gridDim.x * blockDim.x;
    float4 *acc4 = reinterpret_cast<float4 *>(dq_acc);
    const long long n4 = (long long)bh * n * D / 4;
    for (long long t = tid; t < n4; t += nthreads) acc4[t] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ 3. dQ convert
__global__ void __launch_bounds__(256)
    bwd_convert_dq_kernel(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dq,
                          float scale, long long n8)
{
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nthreads = (long long)gridDim.x * blockDim.x;
    for (long long t = tid; t < n8; t += nthreads) {
        const float4 a = reinterpret_cast<const float4 *>(dq_acc)[2 * t];
        const float4 b = reinterpret_cast<const float4 *>(dq_acc)[2 * t + 1];
        uint4 out;
        out.x = ptx::pack_bf16x2(a.x * scale, a.y * scale);
        out.y = ptx::pack_bf16x2(a.z * scale, a.w * scale);
        out.z = ptx::pack_bf16x2(b.x * scale, b.y * scale);
        out.w = ptx::pack_bf16x2(b.z * scale, b.w * scale);
        reinterpret_cast<uint4 *>(dq)[t] = out;
    }
}

// ------------------------------------------------------------------ 2. main
template <int D, bool WITH_DQ>
__global__ void __launch_bounds__(448, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const float *__restrict__ stats, float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dk,
                    __nv_bfloat16 *__restrict__ dv, int n, int n_pad, int n_kvblocks, float scale,
                    int *status)
{
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sK = smem;
    uint8_t *sV = sK + C::KV_BYTES;
    uint8_t *sQ = sV + C::KV_BYTES;                 // QST stages of {Q_i, dO_i}
    uint8_t *sDS = sQ + C::QST * C::STAGE_BYTES;    // two dS^T tiles
    float *sDQ = reinterpret_cast<float *>(sDS + 2 * C::DS_BYTES);  // 2 x dQ staging [BM/2][D]
    float *sLD = reinterpret_cast<float *>(sDS + 2 * C::DS_BYTES + 2 * C::DQH_BYTES);  // QST x {LSE2, D}

    __shared__ uint64_t bar_kv, bar_qf[C::QST], bar_qe[C::QST];
    __shared__ uint64_t bar_sdp[2], bar_ds_full[2], bar_ds_empty[2], bar_dq_full[2], bar_dq_empty[2];
    __shared__ uint64_t bar_dkv, bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / n_kvblocks;
    const int kv0 = (blockIdx.x % n_kvblocks) * C::BN;
    const int nq = (n + C::BM - 1) / C::BM;
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        ptx::mbar_init(&bar_kv, 1);
        for (int s = 0; s < C::QST; ++s) {
            ptx::mbar_init(&bar_qf[s], 1);
            ptx::mbar_init(&bar_qe[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bar_sdp[b], 1);
            ptx::mbar_init(&bar_ds_full[b], 128);
            ptx::mbar_init(&bar_ds_empty[b], 1);
            ptx::mbar_init(&bar_dq_full[b], 1);
            ptx::mbar_init(&bar_dq_empty[b], 128);
        }
        ptx::mbar_init(&bar_dkv, 1);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 13) {
        ptx::tmem_alloc(&tmem_sh, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == 12) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_do);
            ptx::mbar_arrive_expect_tx(&bar_kv, 2 * C::KV_BYTES);
            for (int h = 0; h < D / 64; ++h) {
                ptx::tma_load_3d(sK + h * C::BN * 128, &tm_k, &bar_kv, h * 64, kv0, bh);
                ptx::tma_load_3d(sV + h * C::BN * 128, &tm_v, &bar_kv, h * 64, kv0, bh);
            }
            for (int it = 0; it < nq; ++it) {
                const int s = it % C::QST;
                const uint32_t ph = (it / C::QST) & 1;
                wait_bounded(&bar_qe[s], ph ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_qf[s], C::STAGE_BYTES + C::LD_BYTES);
                uint8_t *stage = sQ + s * C::STAGE_BYTES;
                for (int h = 0; h < D / 64; ++h) {
                    ptx::tma_load_3d(stage + h * C::BM * 128, &tm_q, &bar_qf[s], h * 64, it * C::BM, bh);
                    ptx::tma_load_3d(stage + C::Q_BYTES + h * C::BM * 128, &tm_do, &bar_qf[s],
                                     h * 64, it * C::BM, bh);
                }
                const size_t rowvec = (size_t)bh * n_pad + (size_t)it * C::BM;
                ptx::bulk_load(sLD + s * 2 * C::BM, stats + rowvec * 2, C::BM * 8, &bar_qf[s]);
            }
            wait_bounded(&bar_kv, 0, g);
            for (int it = (nq > C::QST ? nq - C::QST : 0); it < nq; ++it)
                wait_bounded(&bar_qf[it % C::QST], (it / C::QST) & 1, g);
        }
    } else if (warp == 13) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idSdP = ptx::idesc_bf16_f32(128, C::BM, false, false);
            const uint32_t idKV = ptx::idesc_bf16_f32(128, D, false, true);
            const uint32_t idDQ = ptx::idesc_bf16_f32(128, C::BM, true, true);
            const uint32_t k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV);
            const uint32_t q_base = ptx::smem_u32(sQ), ds_base = ptx::smem_u32(sDS);
            auto qs = [&](int s) { return q_base + s * C::STAGE_BYTES; };
            auto dos = [&](int s) { return q_base + s * C::STAGE_BYTES + C::Q_BYTES; };
            // S^T = K_j Q_i^T and dP^T = V_j dO_i^T: all four operands K-major over d.
            auto issue_s = [&](int s, int b) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offa = (kk >> 2) * (C::BN * 128) + (kk & 3) * 32;
                    const uint32_t offb = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
                    ptx::mma_ss(tmem + C::tm_s(b), ptx::sdesc_sw128(k_base + offa, 16, 1024),
                                ptx::sdesc_sw128(qs(s) + offb, 16, 1024), idSdP, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_dp = [&](int s, int b) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offa = (kk >> 2) * (C::BN * 128) + (kk & 3) * 32;
                    const uint32_t offb = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
                    ptx::mma_ss(tmem + C::tm_dp(b), ptx::sdesc_sw128(v_base + offa, 16, 1024),
                                ptx::sdesc_sw128(dos(s) + offb, 16, 1024), idSdP, kk > 0 ? 1u : 0u);
                }
            };
            // dV += P^T dO_i: A = P^T (TMEM, 8 columns per 16 queries), B = dO_i MN-major.
            auto issue_dv = [&](int s, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ts(tmem + C::TM_DV, tmem + C::tm_s(b) + kk * 8,
                                ptx::sdesc_sw128(dos(s) + kk * 2048, C::BM * 128, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            // dK += dS^T Q_i: A = dS^T K-major (queries contiguous), B = Q_i MN-major.
            auto issue_dk = [&](int s, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DK, ptx::sdesc_sw128(ds_base + b * C::DS_BYTES + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(qs(s) + kk * 2048, C::BM * 128, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            // dQ_i^T = K_j^T dS^T into the S^T / P^T columns (free once dV has read P^T):
            // A = K_j MN-major (M = d; halves BN*128 bytes apart), B = dS^T MN-major (N = 64
            // queries), K = 128 keys.
            auto issue_dq = [&](int b) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    ptx::mma_ss(tmem + C::tm_s(b), ptx::sdesc_sw128(k_base + kk * 2048, C::BN * 128, 1024),
                                ptx::sdesc_sw128(ds_base + b * C::DS_BYTES + kk * 2048, C::BN * 128, 1024),
                                idDQ, kk > 0 ? 1u : 0u);
            };
            // Per query tile i (buffer b = i & 1): dV, dQ_i^T (over P^T), dK, then tile i + 2's
            // dP^T (its columns are free) and, once the dQ warps have drained dQ_i^T, its S^T.
            // The drain overlaps dK and dP^T; tile i + 1's products, issued one step earlier,
            // keep the other P / dS warpgroup busy meanwhile.
            wait_bounded(&bar_kv, 0, g);
            for (int j = 0; j < 2 && j < nq; ++j) {
                wait_bounded(&bar_qf[j % C::QST], (j / C::QST) & 1, g);
                ptx::tc_fence_after();
                issue_s(j % C::QST, j);
                issue_dp(j % C::QST, j);
                ptx::mma_commit(&bar_sdp[j]);
            }
            for (int it = 0; it < nq; ++it) {
                const int b = it & 1, s = it % C::QST;
                wait_bounded(&bar_ds_full[b], (it >> 1) & 1, g);
                ptx::tc_fence_after();
                issue_dv(s, b, it > 0);
                if constexpr (WITH_DQ) {
                    issue_dq(b);
                    ptx::mma_commit(&bar_dq_full[b]);
                }
                issue_dk(s, b, it > 0);
                ptx::mma_commit(&bar_qe[s]);
                ptx::mma_commit(&bar_ds_empty[b]);
                if (it + 2 < nq) {
                    const int s2 = (it + 2) % C::QST;
                    wait_bounded(&bar_qf[s2], ((it + 2) / C::QST) & 1, g);
                    ptx::tc_fence_after();
                    issue_dp(s2, b);
                    if constexpr (WITH_DQ)
                        wait_bounded(&bar_dq_empty[b], (it >> 1) & 1, g);   // dQ_i^T drained
                    ptx::tc_fence_after();
                    issue_s(s2, b);
                    ptx::mma_commit(&bar_sdp[b]);
                }
            }
            ptx::mma_commit(&bar_dkv);
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------------- P / dS warpgroups
        // Warpgroup wg takes the query tiles i = wg, wg + 2, ... (TMEM buffer b = wg), so the
        // two groups overlap their element-wise work.
        const int wg = warp >> 2, cw = warp & 3;
        const int r = cw * 32 + lane;       // key row within the tile = TMEM lane
        const bool key_ok = kv0 + r < n;
        const uint32_t lane_off = (uint32_t)(cw * 32) << 16;
        const float scale_log2 = scale * kLog2e;
        for (int it = wg; it < nq; it += 2) {
            const int b = wg, s = it % C::QST;
            const uint32_t ph = (it >> 1) & 1;
            // this query tile's -LSE2 (-inf past N) and -D (0 past N), loaded with the tile
            // this tile's {-LSE2 pair, -D pair} per two queries (-inf and 0 past N)
            const float *sst = sLD + s * 2 * C::BM;
            wait_bounded(&bar_sdp[b], ph, g);
            wait_bounded(&bar_ds_empty[b], ph ^ 1, g);
            ptx::tc_fence_after();
            const uint32_t rowp_a = ptx::smem_u32(sDS + b * C::DS_BYTES + r * 128);
            const uint32_t sst_a = ptx::smem_u32(sst);
            const uint32_t tS = tmem + lane_off + C::tm_s(b), tDP = tmem + lane_off + C::tm_dp(b);
            // 16 queries at a time; the next quarter's TMEM loads overlap this quarter's math.
            // P^T of quarter q goes to columns [8q, 8q + 8), over S^T columns already read.
            uint32_t sv[2][16], dpv[2][16];
            ptx::tmem_ld16(tS, sv[0]);
            ptx::tmem_ld16(tDP, dpv[0]);
            ptx::tmem_ld_wait();
            reg_fence(sv[0]);
            reg_fence(dpv[0]);
#pragma unroll
            for (int qt = 0; qt < 4; ++qt) {
                const int cur = qt & 1;
                if (qt < 3) {
                    ptx::tmem_ld16(tS + (qt + 1) * 16, sv[cur ^ 1]);
                    ptx::tmem_ld16(tDP + (qt + 1) * 16, dpv[cur ^ 1]);
                }
                uint32_t pp[8], dsp[8];
                const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2);
                uint4 st4[8];   // {-LSE2, -LSE2, -D, -D} of queries (c, c + 1), c = 0, 2, ..., 14
#pragma unroll
                for (int e = 0; e < 8; ++e) st4[e] = lds_u128(sst_a + (qt * 16 + 2 * e) * 8);
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const uint64_t nl = ((uint64_t)st4[c / 2].y << 32) | st4[c / 2].x;
                    const uint64_t nd = ((uint64_t)st4[c / 2].w << 32) | st4[c / 2].z;
                    const uint64_t x = ptx::fma_f32x2(
                        ptx::f2_pack(__uint_as_float(sv[cur][c]), __uint_as_float(sv[cur][c + 1])), c2, nl);
                    float x0, x1;
                    ptx::f2_unpack(x, x0, x1);
                    float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                    if (!key_ok) p0 = p1 = 0.f;
                    const uint64_t pq = ptx::f2_pack(p0, p1);
                    const uint64_t dsq = ptx::mul_f32x2(
                        pq, ptx::add_f32x2(ptx::f2_pack(__uint_as_float(dpv[cur][c]), __uint_as_float(dpv[cur][c + 1])), nd));
                    float ds0, ds1;
                    ptx::f2_unpack(dsq, ds0, ds1);
                    pp[c / 2] = ptx::pack_bf16x2(p0, p1);
                    dsp[c / 2] = ptx::pack_bf16x2(ds0, ds1);
                }
                ptx::tmem_st8(tS + qt * 8, pp);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
                    sts_u128(rowp_a + (((qt * 2 + cc) ^ (r & 7)) << 4),
                             make_uint4(dsp[4 * cc], dsp[4 * cc + 1], dsp[4 * cc + 2], dsp[4 * cc + 3]));
                if (qt < 3) {
                    ptx::tmem_ld_wait();
                    reg_fence(sv[cur ^ 1]);
                    reg_fence(dpv[cur ^ 1]);
                }
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_ds_full[b]);
        }
        // epilogue: dK = scale * acc, dV = acc, bf16, key rows < n
        wait_bounded(&bar_dkv, 0, g);
        ptx::tc_fence_after();
        const size_t row_off = ((size_t)bh * n + (key_ok ? kv0 + r : 0)) * D;
        {   // warpgroup 0 writes dK (times scale), warpgroup 1 writes dV
            const int which = wg;
            const float mul = which == 0 ? scale : 1.f;
            __nv_bfloat16 *dst_row = (which == 0 ? dk : dv) + row_off;
            const uint32_t col0 = which == 0 ? C::TM_DK : C::TM_DV;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + lane_off + col0 + c, v);
                ptx::tmem_ld_wait();
                reg_fence(v);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                if (key_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(dst_row + c);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                }
            }
        }
    } else {
        // ---------------------------------------------------------------- dQ warpgroup
        const int r = (warp - 8) * 32 + lane;   // d column = TMEM lane of dQ^T
        const uint32_t lane_off = (uint32_t)((warp - 8) * 32) << 16;
        const bool leader = threadIdx.x == 256;
        for (int it = 0; it < (WITH_DQ ? nq : 0); ++it) {
            const int b = it & 1;
            wait_bounded(&bar_dq_full[b], (it >> 1) & 1, g);
            ptx::tc_fence_after();
            uint32_t v0[32], v1[32];
            if ((warp - 8) * 32 < D) {
                ptx::tmem_ld32(tmem + lane_off + C::tm_s(b), v0);
                ptx::tmem_ld32(tmem + lane_off + C::tm_s(b) + 32, v1);
                ptx::tmem_ld_wait();
                reg_fence(v0);
                reg_fence(v1);
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_dq_empty[b]);
            // two halves of 32 query rows, each through its own 32 x D staging buffer, so that
            // filling one overlaps the bulk reduce-add still reading the other
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // halves past N (only in the last tile) are skipped by every dQ thread alike:
                // each staged half is one bulk group, which the buffer reuse below counts on
                const int q0 = it * C::BM + half * 32;
                if (q0 >= n) break;
                const int rows = (n - q0) < 32 ? (n - q0) : 32;
                float *stage = sDQ + half * (C::DQH_BYTES / 4);
                if (leader) ptx::bulk_wait_group_read<1>();   // this buffer's last reduce has read it
                ptx::named_bar(2, 128);
                if (r < D) {
                    const uint32_t base = opaque(ptx::smem_u32(stage) + r * 4);
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        sts_f32(base + c * D * 4, __uint_as_float(half == 0 ? v0[c] : v1[c]));
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar(2, 128);
                if (leader) {
                    ptx::bulk_reduce_add_f32(dq_acc + ((size_t)bh * n + q0) * D, stage, (uint32_t)rows * D * 4);
                    ptx::bulk_commit_group();
                }
            }
        }
        if (leader) ptx::bulk_wait_group<0>();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 2'. main, d = 64
// The same products as bwd_main_kernel with 128-query tiles, so that S^T, dP^T and dQ^T run
// at N = 128 (an M = 128, K = 16 MMA takes as long at N = 64 as at N = 128) and every per-tile
// latency is paid once per 128 queries instead of once per 64.
//   warp 10     TMA: K_j and V_j once; a ring of (Q_i, dO_i, LSE2_i, D_i), 128 rows each.
//   warp 11     tcgen05, per query tile i (S buffer b = i & 1), once P / dS of tile i are in:
//                 dP^T of tile i + 1 first, then dV += P^T dO_i, dQ_i^T = K_j^T dS^T (over
//                 S^T / P^T of tile i), dK += dS^T Q_i, and S^T of tile i + 2 into buffer b as
//                 soon as dQ_i^T has been drained from it.  S^T of the next tile is thus ready
//                 when the P / dS warps finish a tile; only dP^T is issued after.
//   warps 0-7   both warpgroups on the same tile, warpgroup w on its queries [64w, 64w + 64);
//               thread = key row.  First P^T from S^T (bf16 over the warpgroup's own S^T
//               columns, fp32 kept in registers), then, once dP^T is in, dS^T (bf16) into the
//               warpgroup's 64-query block of the shared dS^T tile.  At the end dK (warpgroup
//               0) and dV (warpgroup 1) go through the idle first (Q, dO) stage and leave with
//               one TMA tensor store each.
//   warps 8-9   dQ_i^T lanes 0-63 (the d rows; lanes 64-127 of the M = 128 product are
//               unused) from TMEM through shared memory into the fp32 accumulator with bulk
//               reduce-adds, 32 query rows at a time through two staging buffers.
// TMEM columns: dK [0,64), dV [64,128), dP^T [128,256), S^T_0 [256,384), S^T_1 [384,512).
struct WideCfg {
    static constexpr int D = 64;
    static constexpr int BN = 128;   // keys per CTA
    static constexpr int BM = 128;   // queries per tile
    static constexpr int QST = 3;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int STAGE_BYTES = 2 * Q_BYTES;
    static constexpr int LD_BYTES = 2 * BM * 4;
    static constexpr int DS_BYTES = BN * BM * 2;          // two 64-query blocks of BN rows
    static constexpr int DQC_BYTES = 32 * D * 4;          // dQ staging: 32 query rows
    static constexpr int SMEM_BYTES =
        2 * KV_BYTES + QST * STAGE_BYTES + 2 * DS_BYTES + 2 * DQC_BYTES + QST * LD_BYTES + 1024;
    static constexpr int THREADS = 384;
    static constexpr int TMA_WARP = 10, MMA_WARP = 11;
    static constexpr uint32_t TM_DK = 0, TM_DV = 64, TM_DP = 128;
    __host__ __device__ static constexpr uint32_t tm_s(int b) { return 256 + b * 128; }
};

template <bool WITH_DQ>
__global__ void __launch_bounds__(384, 1)
    bwd_main_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                         const float *__restrict__ stats, float *__restrict__ dq_acc, int n, int n_pad,
                         int n_kvblocks, float scale, int *status)
{
    using C = WideCfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sK = smem;
    uint8_t *sV = sK + C::KV_BYTES;
    uint8_t *sQ = sV + C::KV_BYTES;                 // QST stages of {Q_i, dO_i}
    uint8_t *sDS = sQ + C::QST * C::STAGE_BYTES;    // two dS^T tiles
    float *sDQ = reinterpret_cast<float *>(sDS + 2 * C::DS_BYTES);   // 2 x dQ staging [32][D]
    float *sLD = reinterpret_cast<float *>(sDS + 2 * C::DS_BYTES + 2 * C::DQC_BYTES);  // QST x {LSE2, D}

    __shared__ uint64_t bar_kv, bar_qf[C::QST], bar_qe[C::QST];
    __shared__ uint64_t bar_s_full[2], bar_dp_full, bar_ds_full, bar_ds_empty[2], bar_dq_full[2], bar_dq_empty[2];
    __shared__ uint64_t bar_dkv, bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / n_kvblocks;
    const int kv0 = (blockIdx.x % n_kvblocks) * C::BN;
    const int nq = (n + C::BM - 1) / C::BM;
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        ptx::mbar_init(&bar_kv, 1);
        for (int s = 0; s < C::QST; ++s) {
            ptx::mbar_init(&bar_qf[s], 1);
            ptx::mbar_init(&bar_qe[s], 1);
        }
        ptx::mbar_init(&bar_dp_full, 1);
        ptx::mbar_init(&bar_ds_full, 256);
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bar_s_full[b], 1);
            ptx::mbar_init(&bar_ds_empty[b], 1);
            ptx::mbar_init(&bar_dq_full[b], 1);
            ptx::mbar_init(&bar_dq_empty[b], 64);
        }
        ptx::mbar_init(&bar_dkv, 1);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(&tmem_sh, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == C::TMA_WARP) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_do);
            ptx::mbar_arrive_expect_tx(&bar_kv, 2 * C::KV_BYTES);
            ptx::tma_load_3d(sK, &tm_k, &bar_kv, 0, kv0, bh);
            ptx::tma_load_3d(sV, &tm_v, &bar_kv, 0, kv0, bh);
            for (int it = 0; it < nq; ++it) {
                const int s = it % C::QST;
                const uint32_t ph = (it / C::QST) & 1;
                wait_bounded(&bar_qe[s], ph ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_qf[s], C::STAGE_BYTES + C::LD_BYTES);
                uint8_t *stage = sQ + s * C::STAGE_BYTES;
                // the Q / dO maps have 64-row boxes: two per 128-row tile, contiguous in the
                // 128-byte-swizzled layout
                for (int h = 0; h < 2; ++h) {
                    ptx::tma_load_3d(stage + h * 64 * 128, &tm_q, &bar_qf[s], 0, it * C::BM + h * 64, bh);
                    ptx::tma_load_3d(stage + C::Q_BYTES + h * 64 * 128, &tm_do, &bar_qf[s], 0,
                                     it * C::BM + h * 64, bh);
                }
                const size_t rowvec = (size_t)bh * n_pad + (size_t)it * C::BM;
                ptx::bulk_load(sLD + s * 2 * C::BM, stats + rowvec * 2, C::BM * 8, &bar_qf[s]);
            }
            wait_bounded(&bar_kv, 0, g);
            for (int it = (nq > C::QST ? nq - C::QST : 0); it < nq; ++it)
                wait_bounded(&bar_qf[it % C::QST], (it / C::QST) & 1, g);
        }
    } else if (warp == C::MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idSdP = ptx::idesc_bf16_f32(128, C::BM, false, false);
            const uint32_t idKV = ptx::idesc_bf16_f32(128, D, false, true);
            const uint32_t idDQ = ptx::idesc_bf16_f32(128, C::BM, true, true);
            const uint32_t k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV);
            const uint32_t q_base = ptx::smem_u32(sQ), ds_base = ptx::smem_u32(sDS);
            auto qs = [&](int s) { return q_base + s * C::STAGE_BYTES; };
            auto dos = [&](int s) { return q_base + s * C::STAGE_BYTES + C::Q_BYTES; };
            // S^T = K_j Q_i^T and dP^T = V_j dO_i^T: K-major over d, N = 128 query rows.
            auto issue_s = [&](int s, int b) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::tm_s(b), ptx::sdesc_sw128(k_base + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(qs(s) + kk * 32, 16, 1024), idSdP, kk > 0 ? 1u : 0u);
            };
            auto issue_dp = [&](int s) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DP, ptx::sdesc_sw128(v_base + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(dos(s) + kk * 32, 16, 1024), idSdP, kk > 0 ? 1u : 0u);
            };
            // dV += P^T dO_i: P^T of queries [16kk, 16kk + 16) sits in the S^T columns of the
            // warpgroup that produced it (64 (kk / 4) + 8 (kk % 4)); dO_i MN-major.
            auto issue_dv = [&](int s, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ts(tmem + C::TM_DV, tmem + C::tm_s(b) + (kk >> 2) * 64 + (kk & 3) * 8,
                                ptx::sdesc_sw128(dos(s) + kk * 2048, C::BM * 128, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            // dK += dS^T Q_i: dS^T K-major (two 64-query blocks BN * 128 bytes apart), Q_i MN-major.
            auto issue_dk = [&](int s, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DK,
                                ptx::sdesc_sw128(ds_base + b * C::DS_BYTES + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32,
                                                 16, 1024),
                                ptx::sdesc_sw128(qs(s) + kk * 2048, C::BM * 128, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            // dQ_i^T = K_j^T dS^T over S^T / P^T of tile i: A = K_j MN-major with M = 128 (rows
            // 64-127 read V_j, which follows K_j in shared memory, and land in unused lanes),
            // B = dS^T MN-major, N = 128 queries in two blocks BN * 128 bytes apart.
            auto issue_dq = [&](int b) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    ptx::mma_ss(tmem + C::tm_s(b), ptx::sdesc_sw128(k_base + kk * 2048, C::BN * 128, 1024),
                                ptx::sdesc_sw128(ds_base + b * C::DS_BYTES + kk * 2048, C::BN * 128, 1024),
                                idDQ, kk > 0 ? 1u : 0u);
            };
            // S^T of tile i + 2 goes into buffer b as soon as tile i's dQ^T has been drained from
            // it, well before the P / dS warps finish tile i + 1; dP^T of tile i + 1 follows
            // the P / dS warps' last read of dP^T (tile i done).
            wait_bounded(&bar_kv, 0, g);
            wait_bounded(&bar_qf[0], 0, g);
            ptx::tc_fence_after();
            issue_s(0, 0);
            ptx::mma_commit(&bar_s_full[0]);
            issue_dp(0);
            ptx::mma_commit(&bar_dp_full);
            if (nq > 1) {
                wait_bounded(&bar_qf[1], 0, g);
                ptx::tc_fence_after();
                issue_s(1, 1);
                ptx::mma_commit(&bar_s_full[1]);
            }
            for (int it = 0; it < nq; ++it) {
                const int b = it & 1, s = it % C::QST;
                wait_bounded(&bar_ds_full, it & 1, g);
                ptx::tc_fence_after();
                if (it + 1 < nq) {
                    issue_dp((it + 1) % C::QST);   // its Q / dO stage was waited for with its S^T
                    ptx::mma_commit(&bar_dp_full);
                }
                issue_dv(s, b, it > 0);
                if constexpr (WITH_DQ) {
                    issue_dq(b);
                    ptx::mma_commit(&bar_dq_full[b]);
                }
                issue_dk(s, b, it > 0);
                ptx::mma_commit(&bar_qe[s]);
                ptx::mma_commit(&bar_ds_empty[b]);
                if (it + 2 < nq) {
                    const int s2 = (it + 2) % C::QST;
                    wait_bounded(&bar_qf[s2], ((it + 2) / C::QST) & 1, g);
                    if constexpr (WITH_DQ)
                        wait_bounded(&bar_dq_empty[b], (it >> 1) & 1, g);   // dQ_i^T drained
                    ptx::tc_fence_after();
                    issue_s(s2, b);
                    ptx::mma_commit(&bar_s_full[b]);
                }
            }
            ptx::mma_commit(&bar_dkv);
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------------- P / dS warpgroups
        const int wg = warp >> 2, cw = warp & 3;
        const int r = cw * 32 + lane;       // key row within the tile = TMEM lane
        const bool key_ok = kv0 + r < n;
        const uint32_t lane_off = (uint32_t)(cw * 32) << 16;
        const float scale_log2 = scale * kLog2e;
        const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2);
        for (int it = 0; it < nq; ++it) {
            const int b = it & 1, s = it % C::QST;
            // {-LSE2 pair, -D pair} per two of this warpgroup's queries
            const uint32_t sst_a = ptx::smem_u32(sLD + s * 2 * C::BM + wg * 128);
            const uint32_t rowp_a = ptx::smem_u32(sDS + b * C::DS_BYTES + wg * (C::BN * 128) + r * 128);
            const uint32_t tS = tmem + lane_off + C::tm_s(b) + wg * 64;
            const uint32_t tDP = tmem + lane_off + C::TM_DP + wg * 64;
            wait_bounded(&bar_s_full[b], (it >> 1) & 1, g);
            wait_bounded(&bar_ds_empty[b], ((it >> 1) & 1) ^ 1, g);
            ptx::tc_fence_after();
            // Phase 1, as soon as S^T is in: P^T = 2^(S^T c - LSE2) for 16 queries at a time
            // (the next 16 columns load meanwhile), bf16 back into TMEM over S^T columns
            // already read, fp32 kept for dS.
            float pf[64];
            {
                uint32_t sv[2][16];
                ptx::tmem_ld16(tS, sv[0]);
                ptx::tmem_ld_wait();
                reg_fence(sv[0]);
#pragma unroll
                for (int qt = 0; qt < 4; ++qt) {
                    const int cur = qt & 1;
                    if (qt < 3) ptx::tmem_ld16(tS + (qt + 1) * 16, sv[cur ^ 1]);
                    uint2 nl[8];   // -LSE2 of queries (c, c + 1), c = 0, 2, ..., 14
#pragma unroll
                    for (int e = 0; e < 8; ++e) nl[e] = lds_u64(sst_a + (qt * 16 + 2 * e) * 8);
                    uint32_t pp[8];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        const uint64_t x = ptx::fma_f32x2(
                            ptx::f2_pack(__uint_as_float(sv[cur][c]), __uint_as_float(sv[cur][c + 1])), c2,
                            ((uint64_t)nl[c / 2].y << 32) | nl[c / 2].x);
                        float x0, x1;
                        ptx::f2_unpack(x, x0, x1);
                        float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        if (!key_ok) p0 = p1 = 0.f;
                        pf[qt * 16 + c] = p0;
                        pf[qt * 16 + c + 1] = p1;
                        pp[c / 2] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st8(tS + qt * 8, pp);
                    if (qt < 3) {
                        ptx::tmem_ld_wait();
                        reg_fence(sv[cur ^ 1]);
                    }
                }
            }
            // Phase 2, once dP^T is in: dS^T = P^T o (dP^T - D), bf16 into shared memory.
            wait_bounded(&bar_dp_full, it & 1, g);
            ptx::tc_fence_after();
            {
                uint32_t dpv[2][16];
                ptx::tmem_ld16(tDP, dpv[0]);
                ptx::tmem_ld_wait();
                reg_fence(dpv[0]);
#pragma unroll
                for (int qt = 0; qt < 4; ++qt) {
                    const int cur = qt & 1;
                    if (qt < 3) ptx::tmem_ld16(tDP + (qt + 1) * 16, dpv[cur ^ 1]);
                    uint2 nd[8];   // -D of queries (c, c + 1)
#pragma unroll
                    for (int e = 0; e < 8; ++e) nd[e] = lds_u64(sst_a + (qt * 16 + 2 * e) * 8 + 8);
                    uint32_t dsp[8];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        const uint64_t dsq = ptx::mul_f32x2(
                            ptx::f2_pack(pf[qt * 16 + c], pf[qt * 16 + c + 1]),
                            ptx::add_f32x2(ptx::f2_pack(__uint_as_float(dpv[cur][c]), __uint_as_float(dpv[cur][c + 1])),
                                           ((uint64_t)nd[c / 2].y << 32) | nd[c / 2].x));
                        float ds0, ds1;
                        ptx::f2_unpack(dsq, ds0, ds1);
                        dsp[c / 2] = ptx::pack_bf16x2(ds0, ds1);
                    }
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
                        sts_u128(rowp_a + (((qt * 2 + cc) ^ (r & 7)) << 4),
                                 make_uint4(dsp[4 * cc], dsp[4 * cc + 1], dsp[4 * cc + 2], dsp[4 * cc + 3]));
                    if (qt < 3) {
                        ptx::tmem_ld_wait();
                        reg_fence(dpv[cur ^ 1]);
                    }
                }
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_ds_full);
        }
        // epilogue: dK = scale * acc (warpgroup 0), dV = acc (warpgroup 1), bf16, staged in the
        // now idle first (Q, dO) stage in the 128-byte-swizzled layout (16-byte chunk c of row r
        // at chunk c ^ (r % 8)) and stored with one TMA tensor store each (rows past N clipped)
        wait_bounded(&bar_dkv, 0, g);
        ptx::tc_fence_after();
        {
            const float mul = wg == 0 ? scale : 1.f;
            const uint32_t col0 = wg == 0 ? C::TM_DK : C::TM_DV;
            const uint32_t srow = ptx::smem_u32(sQ + wg * C::Q_BYTES) + r * 128;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + lane_off + col0 + c, v);
                ptx::tmem_ld_wait();
                reg_fence(v);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    sts_u128(srow + ((((c >> 3) + v4) ^ (r & 7)) << 4),
                             make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]));
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, 256);
            if (threadIdx.x == 0) {
                ptx::tma_store_3d(&tm_dk, sQ, 0, kv0, bh);
                ptx::tma_store_3d(&tm_dv, sQ + C::Q_BYTES, 0, kv0, bh);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group<0>();   // complete before the CTA exits
            }
        }
    } else if (WITH_DQ && warp < 10) {
        // ---------------------------------------------------------------- dQ warps
        const int r = (warp - 8) * 32 + lane;   // d column = TMEM lane of dQ^T
        const uint32_t lane_off = (uint32_t)((warp - 8) * 32) << 16;
        const bool leader = threadIdx.x == 256;
        int chunk = 0;   // staging buffer = chunk & 1
        for (int it = 0; it < nq; ++it) {
            const int b = it & 1;
            wait_bounded(&bar_dq_full[b], (it >> 1) & 1, g);
            ptx::tc_fence_after();
            uint32_t v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tmem + lane_off + C::tm_s(b) + c * 32, v[c]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence(v[c]);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_dq_empty[b]);
            // four chunks of 32 query rows, alternating between two 32 x D staging buffers so
            // that filling one overlaps the bulk reduce-add still reading the other
#pragma unroll
            for (int c = 0; c < 4; ++c, ++chunk) {
                // Chunks past N (only in the last tile) are skipped by every dQ thread alike:
                // each staged chunk is one bulk group, which the buffer reuse below counts on.
                const int q0 = it * C::BM + c * 32;
                if (q0 >= n) break;
                const int rows = (n - q0) < 32 ? (n - q0) : 32;
                float *stage = sDQ + (chunk & 1) * (C::DQC_BYTES / 4);
                if (leader) ptx::bulk_wait_group_read<1>();   // this buffer's last reduce has read it
                ptx::named_bar(2, 64);
                const uint32_t base = opaque(ptx::smem_u32(stage) + r * 4);
#pragma unroll
                for (int q = 0; q < 32; ++q) sts_f32(base + q * D * 4, __uint_as_float(v[c][q]));
                ptx::fence_proxy_async_smem();
                ptx::named_bar(2, 64);
                if (leader) {
                    ptx::bulk_reduce_add_f32(dq_acc + ((size_t)bh * n + q0) * D, stage, (uint32_t)rows * D * 4);
                    ptx::bulk_commit_group();
                }
            }
        }
        if (leader) ptx::bulk_wait_group<0>();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 2'''. main, d = 64, persistent
// For short sequences (few query tiles per key block) the wide kernel's fixed costs per CTA
// (start-up loads, the dK / dV epilogue, the last dQ reduce-adds) are as long as its products.
// This variant keeps one CTA per SM and runs its (head, key block) items as one sequence of
// query tiles, so that the tile pipeline's lookahead (dP^T one tile, S^T two tiles ahead)
// crosses item boundaries and the next item's loads and products overlap the previous item's
// tail.
//   warp 10     TMA: per item K into one of two buffers and V into one buffer (free once the
//               previous item's last dP^T has read it); per tile Q (+ statistics) through a
//               ring of three and dO through a ring of two.
//   warp 11     tcgen05, per tile t of the sequence, as the wide kernel; dK and dV restart
//               (accumulate off) on the first tile of each item.
//   warps 0-7   P / dS as the wide kernel; after the P phase of an item's first tile, the
//               previous item's dK (warpgroup 0, times scale) and dV (warpgroup 1) go from
//               TMEM through the idle dS^T buffer (the previous tile's, whose products are
//               done) to global memory by TMA tensor stores.
//   warps 8-9   dQ drain as the wide kernel (32 query rows per staged chunk; 16-row chunks,
//               which would leave room for a third dO buffer, drain ~1.3x slower).
// TMEM columns as the wide kernel.  Items (head, key block) are taken in a grid-stride order.
struct PersistBwdCfg {
    static constexpr int D = 64;
    static constexpr int BN = 128, BM = 128;
    static constexpr int QST = 3, DOST = 2;
    static constexpr int T_BYTES = 128 * D * 2;        // one 128-row tile
    static constexpr int LD_BYTES = 2 * BM * 4;
    static constexpr int DS_BYTES = BN * BM * 2;       // two 64-query blocks of BN rows
    static constexpr int DQC_ROWS = 32;
    static constexpr int DQC_BYTES = DQC_ROWS * D * 4; // dQ staging: 32 query rows
    static constexpr int SMEM_BYTES = 3 * T_BYTES + QST * T_BYTES + DOST * T_BYTES + 2 * DS_BYTES +
                                      2 * DQC_BYTES + QST * LD_BYTES + 1024;
    static constexpr int THREADS = 384;
    static constexpr int TMA_WARP = 10, MMA_WARP = 11;
    static constexpr uint32_t TM_DK = 0, TM_DV = 64, TM_DP = 128;
    __host__ __device__ static constexpr uint32_t tm_s(int b) { return 256 + b * 128; }
};

// Position of tile t of a CTA's sequence: item li (head bh, keys from kv0), query tile it.
struct TileCursor {
    int li, it, bh, kv0;
    __device__ void start(int first, int n_kvblocks, int bn)
    {
        li = 0;
        it = 0;
        bh = first / n_kvblocks;
        kv0 = (first % n_kvblocks) * bn;
    }
    __device__ void next(int nq, int first, int stride, int n_kvblocks, int bn)
    {
        if (++it == nq) {
            it = 0;
            ++li;
            const int item = first + li * stride;
            bh = item / n_kvblocks;
            kv0 = (item % n_kvblocks) * bn;
        }
    }
};

template <bool WITH_DQ>
__global__ void __launch_bounds__(384, 1)
    bwd_main_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                            const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                            const float *__restrict__ stats, float *__restrict__ dq_acc, int n, int n_pad,
                            int n_kvblocks, int n_items, float scale, int *status)
{
    using C = PersistBwdCfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sK = smem;                             // K_0, K_1, then V (dQ^T's unused rows read on)
    uint8_t *sV = sK + 2 * C::T_BYTES;
    uint8_t *sQ = sV + C::T_BYTES;                  // QST Q tiles
    uint8_t *sDO = sQ + C::QST * C::T_BYTES;        // DOST dO tiles
    uint8_t *sDS = sDO + C::DOST * C::T_BYTES;      // two dS^T tiles
    float *sDQ = reinterpret_cast<float *>(sDS + 2 * C::DS_BYTES);                       // 2 x [32][D]
    float *sLD = reinterpret_cast<float *>(sDS + 2 * C::DS_BYTES + 2 * C::DQC_BYTES);   // QST x stats

    __shared__ uint64_t bar_kf[2], bar_ke[2], bar_vf, bar_ve, bar_qf[C::QST], bar_qe[C::QST];
    __shared__ uint64_t bar_dof[C::DOST], bar_doe[C::DOST];
    __shared__ uint64_t bar_s_full[2], bar_dp_full, bar_ds_full, bar_ds_empty[2], bar_dq_full[2], bar_dq_empty[2];
    __shared__ uint64_t bar_dkv, bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nq = (n + C::BM - 1) / C::BM;
    const int first = blockIdx.x, stride = gridDim.x;
    const int n_mine = first < n_items ? (n_items - 1 - first) / stride + 1 : 0;
    const int T = n_mine * nq;                      // query tiles in this CTA's sequence
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bar_kf[b], 1);
            ptx::mbar_init(&bar_ke[b], 1);
            ptx::mbar_init(&bar_s_full[b], 1);
            ptx::mbar_init(&bar_ds_empty[b], 1);
            ptx::mbar_init(&bar_dq_full[b], 1);
            ptx::mbar_init(&bar_dq_empty[b], 64);
        }
        ptx::mbar_init(&bar_vf, 1);
        ptx::mbar_init(&bar_ve, 1);
        for (int s = 0; s < C::QST; ++s) {
            ptx::mbar_init(&bar_qf[s], 1);
            ptx::mbar_init(&bar_qe[s], 1);
        }
        for (int s = 0; s < C::DOST; ++s) {
            ptx::mbar_init(&bar_dof[s], 1);
            ptx::mbar_init(&bar_doe[s], 1);
        }
        ptx::mbar_init(&bar_dp_full, 1);
        ptx::mbar_init(&bar_ds_full, 256);
        ptx::mbar_init(&bar_dkv, 1);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(&tmem_sh, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == C::TMA_WARP) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_do);
            TileCursor c;
            c.start(first, n_kvblocks, C::BN);
            for (int t = 0; t < T; ++t) {
                if (c.it == 0) {   // K into buffer li % 2, once item li - 2 is done with it
                    const int kb = c.li & 1;
                    wait_bounded(&bar_ke[kb], ((c.li >> 1) & 1) ^ 1, g);
                    ptx::mbar_arrive_expect_tx(&bar_kf[kb], C::T_BYTES);
                    ptx::tma_load_3d(sK + kb * C::T_BYTES, &tm_k, &bar_kf[kb], 0, c.kv0, c.bh);
                }
                const int s = t % C::QST;
                wait_bounded(&bar_qe[s], ((t / C::QST) & 1) ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_qf[s], C::T_BYTES + C::LD_BYTES);
                // the Q / dO maps have 64-row boxes: two per 128-row tile, contiguous in the
                // 128-byte-swizzled layout
                for (int h = 0; h < 2; ++h)
                    ptx::tma_load_3d(sQ + s * C::T_BYTES + h * 64 * 128, &tm_q, &bar_qf[s], 0,
                                     c.it * C::BM + h * 64, c.bh);
                const size_t rowvec = (size_t)c.bh * n_pad + (size_t)c.it * C::BM;
                ptx::bulk_load(sLD + s * 2 * C::BM, stats + rowvec * 2, C::BM * 8, &bar_qf[s]);
                if (c.it == 0) {   // V, once the previous item's last dP^T has read it
                    wait_bounded(&bar_ve, (c.li & 1) ^ 1, g);
                    ptx::mbar_arrive_expect_tx(&bar_vf, C::T_BYTES);
                    ptx::tma_load_3d(sV, &tm_v, &bar_vf, 0, c.kv0, c.bh);
                }
                const int sd = t % C::DOST;
                wait_bounded(&bar_doe[sd], ((t / C::DOST) & 1) ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_dof[sd], C::T_BYTES);
                for (int h = 0; h < 2; ++h)
                    ptx::tma_load_3d(sDO + sd * C::T_BYTES + h * 64 * 128, &tm_do, &bar_dof[sd], 0,
                                     c.it * C::BM + h * 64, c.bh);
                c.next(nq, first, stride, n_kvblocks, C::BN);
            }
            // Do not leave the CTA with copies in flight (matters only after a timeout).
            for (int t = (T > C::QST ? T - C::QST : 0); t < T; ++t) wait_bounded(&bar_qf[t % C::QST], (t / C::QST) & 1, g);
            for (int t = (T > C::DOST ? T - C::DOST : 0); t < T; ++t)
                wait_bounded(&bar_dof[t % C::DOST], (t / C::DOST) & 1, g);
            for (int li = (n_mine > 2 ? n_mine - 2 : 0); li < n_mine; ++li)
                wait_bounded(&bar_kf[li & 1], (li >> 1) & 1, g);
            if (n_mine > 0) wait_bounded(&bar_vf, (n_mine - 1) & 1, g);
        }
    } else if (warp == C::MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idSdP = ptx::idesc_bf16_f32(128, C::BM, false, false);
            const uint32_t idKV = ptx::idesc_bf16_f32(128, D, false, true);
            const uint32_t idDQ = ptx::idesc_bf16_f32(128, C::BM, true, true);
            const uint32_t k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV);
            const uint32_t q_base = ptx::smem_u32(sQ), do_base = ptx::smem_u32(sDO);
            const uint32_t ds_base = ptx::smem_u32(sDS);
            // S^T = K Q_t^T and dP^T = V dO_t^T: K-major over d, N = 128 query rows.
            auto issue_s = [&](int kb, int s, int b) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::tm_s(b), ptx::sdesc_sw128(k_base + kb * C::T_BYTES + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(q_base + s * C::T_BYTES + kk * 32, 16, 1024), idSdP, kk > 0 ? 1u : 0u);
            };
            auto issue_dp = [&](int sd) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DP, ptx::sdesc_sw128(v_base + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(do_base + sd * C::T_BYTES + kk * 32, 16, 1024), idSdP,
                                kk > 0 ? 1u : 0u);
            };
            // dV += P^T dO_t: P^T of queries [16kk, 16kk + 16) in the S^T columns of the
            // warpgroup that produced it (64 (kk / 4) + 8 (kk % 4)); dO_t MN-major.
            auto issue_dv = [&](int sd, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ts(tmem + C::TM_DV, tmem + C::tm_s(b) + (kk >> 2) * 64 + (kk & 3) * 8,
                                ptx::sdesc_sw128(do_base + sd * C::T_BYTES + kk * 2048, C::BM * 128, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            // dK += dS^T Q_t: dS^T K-major (two 64-query blocks BN * 128 bytes apart), Q_t MN-major.
            auto issue_dk = [&](int s, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DK,
                                ptx::sdesc_sw128(ds_base + b * C::DS_BYTES + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32,
                                                 16, 1024),
                                ptx::sdesc_sw128(q_base + s * C::T_BYTES + kk * 2048, C::BM * 128, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            // dQ_t^T = K^T dS^T over S^T / P^T of tile t: A = K MN-major with M = 128 (rows
            // 64-127 read the next 16 KB of shared memory and land in unused lanes), B = dS^T
            // MN-major, N = 128 queries in two blocks BN * 128 bytes apart.
            auto issue_dq = [&](int kb, int b) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    ptx::mma_ss(tmem + C::tm_s(b), ptx::sdesc_sw128(k_base + kb * C::T_BYTES + kk * 2048, C::T_BYTES, 1024),
                                ptx::sdesc_sw128(ds_base + b * C::DS_BYTES + kk * 2048, C::BN * 128, 1024),
                                idDQ, kk > 0 ? 1u : 0u);
            };
            TileCursor c0, c1, c2;   // tiles t, t + 1, t + 2
            c0.start(first, n_kvblocks, C::BN);
            c1 = c0;
            c1.next(nq, first, stride, n_kvblocks, C::BN);
            c2 = c1;
            c2.next(nq, first, stride, n_kvblocks, C::BN);
            if (T > 0) {
                wait_bounded(&bar_kf[0], 0, g);
                wait_bounded(&bar_qf[0], 0, g);
                ptx::tc_fence_after();
                issue_s(0, 0, 0);
                ptx::mma_commit(&bar_s_full[0]);
                wait_bounded(&bar_vf, 0, g);
                wait_bounded(&bar_dof[0], 0, g);
                ptx::tc_fence_after();
                issue_dp(0);
                ptx::mma_commit(&bar_dp_full);
                if (nq == 1) ptx::mma_commit(&bar_ve);
            }
            if (T > 1) {
                if (c1.it == 0) wait_bounded(&bar_kf[c1.li & 1], (c1.li >> 1) & 1, g);
                wait_bounded(&bar_qf[1], 0, g);
                ptx::tc_fence_after();
                issue_s(c1.li & 1, 1, 1);
                ptx::mma_commit(&bar_s_full[1]);
            }
            for (int t = 0; t < T; ++t) {
                const int b = t & 1, s = t % C::QST, sd = t % C::DOST, kb = c0.li & 1;
                wait_bounded(&bar_ds_full, t & 1, g);
                ptx::tc_fence_after();
                if (t + 1 < T) {
                    if (c1.it == 0) wait_bounded(&bar_vf, c1.li & 1, g);   // the next item's V
                    wait_bounded(&bar_dof[(t + 1) % C::DOST], ((t + 1) / C::DOST) & 1, g);
                    ptx::tc_fence_after();
                    issue_dp((t + 1) % C::DOST);
                    ptx::mma_commit(&bar_dp_full);
                    if (c1.it == nq - 1) ptx::mma_commit(&bar_ve);          // its item's last read of V
                }
                issue_dv(sd, b, c0.it > 0);
                ptx::mma_commit(&bar_doe[sd]);
                if constexpr (WITH_DQ) {
                    issue_dq(kb, b);
                    ptx::mma_commit(&bar_dq_full[b]);
                }
                issue_dk(s, b, c0.it > 0);
                ptx::mma_commit(&bar_qe[s]);
                ptx::mma_commit(&bar_ds_empty[b]);
                if (c0.it == nq - 1) {   // the item's last products: K free, dK / dV complete
                    ptx::mma_commit(&bar_ke[kb]);
                    ptx::mma_commit(&bar_dkv);
                }
                if (t + 2 < T) {
                    const int s2 = (t + 2) % C::QST;
                    if (c2.it == 0) wait_bounded(&bar_kf[c2.li & 1], (c2.li >> 1) & 1, g);
                    wait_bounded(&bar_qf[s2], ((t + 2) / C::QST) & 1, g);
                    if constexpr (WITH_DQ)
                        wait_bounded(&bar_dq_empty[b], (t >> 1) & 1, g);   // dQ_t^T drained
                    ptx::tc_fence_after();
                    issue_s(c2.li & 1, s2, b);
                    ptx::mma_commit(&bar_s_full[b]);
                }
                c0 = c1;
                c1 = c2;
                c2.next(nq, first, stride, n_kvblocks, C::BN);
            }
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------------- P / dS warpgroups
        const int wg = warp >> 2, cw = warp & 3;
        const int r = cw * 32 + lane;       // key row within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(cw * 32) << 16;
        const float scale_log2 = scale * kLog2e;
        const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2);
        // dK = scale * acc (warpgroup 0) or dV = acc (warpgroup 1) of an item, bf16, into the
        // 32 KB staging area `stage` (dK then dV, 128-byte-swizzled rows: 16-byte chunk c of row
        // r at chunk c ^ (r % 8)), then one TMA tensor store each (rows past N clipped).  The
        // stores still read `stage` afterwards: `store_pending` says so to the caller.
        bool store_pending = false;
        auto epilogue = [&](int li, int bh, int kv0, uint8_t *stage) {
            if (store_pending) {   // earlier stores may still read either buffer
                if (threadIdx.x == 0) ptx::bulk_wait_group_read<0>();
                ptx::named_bar(1, 256);
            }
            wait_bounded(&bar_dkv, li & 1, g);
            ptx::tc_fence_after();
            const float mul = wg == 0 ? scale : 1.f;
            const uint32_t col0 = wg == 0 ? C::TM_DK : C::TM_DV;
            const uint32_t srow = ptx::smem_u32(stage + wg * C::T_BYTES) + r * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + lane_off + col0 + h * 32, v);
                ptx::tmem_ld_wait();
                reg_fence(v);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    sts_u128(srow + (((h * 4 + v4) ^ (r & 7)) << 4),
                             make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]));
            }
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, 256);
            if (threadIdx.x == 0) {
                ptx::tma_store_3d(&tm_dk, stage, 0, kv0, bh);
                ptx::tma_store_3d(&tm_dv, stage + C::T_BYTES, 0, kv0, bh);
                ptx::bulk_commit_group();
            }
            store_pending = true;
        };
        TileCursor c;
        c.start(first, n_kvblocks, C::BN);
        int prev_bh = 0, prev_kv0 = 0;
        for (int t = 0; t < T; ++t) {
            const int b = t & 1, s = t % C::QST;
            const bool key_ok = c.kv0 + r < n;
            // {-LSE2 pair, -D pair} per two of this warpgroup's queries
            const uint32_t sst_a = ptx::smem_u32(sLD + s * 2 * C::BM + wg * 128);
            const uint32_t rowp_a = ptx::smem_u32(sDS + b * C::DS_BYTES + wg * (C::BN * 128) + r * 128);
            const uint32_t tS = tmem + lane_off + C::tm_s(b) + wg * 64;
            const uint32_t tDP = tmem + lane_off + C::TM_DP + wg * 64;
            wait_bounded(&bar_s_full[b], (t >> 1) & 1, g);
            wait_bounded(&bar_ds_empty[b], ((t >> 1) & 1) ^ 1, g);
            ptx::tc_fence_after();
            // Phase 1, as soon as S^T is in: P^T = 2^(S^T c - LSE2), bf16 back into TMEM over S^T
            // columns already read, fp32 kept for dS.
            float pf[64];
            {
                uint32_t sv[2][16];
                ptx::tmem_ld16(tS, sv[0]);
                ptx::tmem_ld_wait();
                reg_fence(sv[0]);
#pragma unroll
                for (int qt = 0; qt < 4; ++qt) {
                    const int cur = qt & 1;
                    if (qt < 3) ptx::tmem_ld16(tS + (qt + 1) * 16, sv[cur ^ 1]);
                    uint2 nl[8];   // -LSE2 of queries (c, c + 1), c = 0, 2, ..., 14
#pragma unroll
                    for (int e = 0; e < 8; ++e) nl[e] = lds_u64(sst_a + (qt * 16 + 2 * e) * 8);
                    uint32_t pp[8];
#pragma unroll
                    for (int cc = 0; cc < 16; cc += 2) {
                        const uint64_t x = ptx::fma_f32x2(
                            ptx::f2_pack(__uint_as_float(sv[cur][cc]), __uint_as_float(sv[cur][cc + 1])), c2,
                            ((uint64_t)nl[cc / 2].y << 32) | nl[cc / 2].x);
                        float x0, x1;
                        ptx::f2_unpack(x, x0, x1);
                        float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        if (!key_ok) p0 = p1 = 0.f;
                        pf[qt * 16 + cc] = p0;
                        pf[qt * 16 + cc + 1] = p1;
                        pp[cc / 2] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st8(tS + qt * 8, pp);
                    if (qt < 3) {
                        ptx::tmem_ld_wait();
                        reg_fence(sv[cur ^ 1]);
                    }
                }
            }
            // The previous item's dK / dV, while this tile's dP^T and the previous tile's
            // products run; before this tile's dS^T, which lets its dV / dK restart the
            // accumulators.  Staged in the other dS^T buffer: the previous tile's dK and dQ^T,
            // complete once dK / dV are, have read it, and the next tile's dS^T waits for the
            // stores below.
            if (c.it == 0 && c.li > 0) {
                epilogue(c.li - 1, prev_bh, prev_kv0, sDS + (b ^ 1) * C::DS_BYTES);
            } else if (store_pending) {   // the stores issued one tile ago read this dS^T buffer
                if (threadIdx.x == 0) ptx::bulk_wait_group_read<0>();
                ptx::named_bar(1, 256);
                store_pending = false;
            }
            // Phase 2, once dP^T is in: dS^T = P^T o (dP^T - D), bf16 into shared memory.
            wait_bounded(&bar_dp_full, t & 1, g);
            ptx::tc_fence_after();
            {
                uint32_t dpv[2][16];
                ptx::tmem_ld16(tDP, dpv[0]);
                ptx::tmem_ld_wait();
                reg_fence(dpv[0]);
#pragma unroll
                for (int qt = 0; qt < 4; ++qt) {
                    const int cur = qt & 1;
                    if (qt < 3) ptx::tmem_ld16(tDP + (qt + 1) * 16, dpv[cur ^ 1]);
                    uint2 nd[8];   // -D of queries (c, c + 1)
#pragma unroll
                    for (int e = 0; e < 8; ++e) nd[e] = lds_u64(sst_a + (qt * 16 + 2 * e) * 8 + 8);
                    uint32_t dsp[8];
#pragma unroll
                    for (int cc = 0; cc < 16; cc += 2) {
                        const uint64_t dsq = ptx::mul_f32x2(
                            ptx::f2_pack(pf[qt * 16 + cc], pf[qt * 16 + cc + 1]),
                            ptx::add_f32x2(ptx::f2_pack(__uint_as_float(dpv[cur][cc]), __uint_as_float(dpv[cur][cc + 1])),
                                           ((uint64_t)nd[cc / 2].y << 32) | nd[cc / 2].x));
                        float ds0, ds1;
                        ptx::f2_unpack(dsq, ds0, ds1);
                        dsp[cc / 2] = ptx::pack_bf16x2(ds0, ds1);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        sts_u128(rowp_a + (((qt * 2 + h) ^ (r & 7)) << 4),
                                 make_uint4(dsp[4 * h], dsp[4 * h + 1], dsp[4 * h + 2], dsp[4 * h + 3]));
                    if (qt < 3) {
                        ptx::tmem_ld_wait();
                        reg_fence(dpv[cur ^ 1]);
                    }
                }
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_ds_full);
            prev_bh = c.bh;
            prev_kv0 = c.kv0;
            c.next(nq, first, stride, n_kvblocks, C::BN);
        }
        if (n_mine > 0) {
            epilogue(n_mine - 1, prev_bh, prev_kv0, sDS);   // every product is done: any buffer
            if (threadIdx.x == 0) ptx::bulk_wait_group<0>();   // complete before the CTA exits
        }
    } else if (WITH_DQ && warp < 10) {
        // ---------------------------------------------------------------- dQ warps
        const int r = (warp - 8) * 32 + lane;   // d column = TMEM lane of dQ^T
        const uint32_t lane_off = (uint32_t)((warp - 8) * 32) << 16;
        const bool leader = threadIdx.x == 256;
        int chunk = 0;   // staging buffer = chunk & 1
        TileCursor c;
        c.start(first, n_kvblocks, C::BN);
        for (int t = 0; t < T; ++t) {
            const int b = t & 1;
            wait_bounded(&bar_dq_full[b], (t >> 1) & 1, g);
            ptx::tc_fence_after();
            uint32_t v[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) ptx::tmem_ld32(tmem + lane_off + C::tm_s(b) + q * 32, v[q]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q) reg_fence(v[q]);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_dq_empty[b]);
            // chunks of DQC_ROWS query rows, alternating between two staging buffers so that
            // filling one overlaps the bulk reduce-add still reading the other
#pragma unroll
            for (int q = 0; q < C::BM / C::DQC_ROWS; ++q, ++chunk) {
                // Chunks past N (only in an item's last tile) are skipped by every dQ thread
                // alike: each staged chunk is one bulk group, which the buffer reuse counts on.
                const int q0 = c.it * C::BM + q * C::DQC_ROWS;
                if (q0 >= n) break;
                const int rows = (n - q0) < C::DQC_ROWS ? (n - q0) : C::DQC_ROWS;
                float *stage = sDQ + (chunk & 1) * (C::DQC_BYTES / 4);
                if (leader) ptx::bulk_wait_group_read<1>();   // this buffer's last reduce has read it
                ptx::named_bar(2, 64);
                const uint32_t base = opaque(ptx::smem_u32(stage) + r * 4);
#pragma unroll
                for (int qq = 0; qq < C::DQC_ROWS; ++qq)
                    sts_f32(base + qq * D * 4, __uint_as_float(v[q * C::DQC_ROWS / 32][(q * C::DQC_ROWS) % 32 + qq]));
                ptx::fence_proxy_async_smem();
                ptx::named_bar(2, 64);
                if (leader) {
                    ptx::bulk_reduce_add_f32(dq_acc + ((size_t)c.bh * n + q0) * D, stage, (uint32_t)rows * D * 4);
                    ptx::bulk_commit_group();
                }
            }
            c.next(nq, first, stride, n_kvblocks, C::BN);
        }
        if (leader) ptx::bulk_wait_group<0>();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 2''. dK / dV only, d = 128
// The deterministic mode's dK, dV pass for d = 128 with 128-query tiles, so that its four
// products run at N = 128 (S^T and dP^T at N = 64 take as long as at N = 128).  TMEM holds dK,
// dV, dP^T and one S^T buffer (4 x 128 columns).
//   warp 16     TMA: K_j and V_j once; Q_i (+ its statistics) in two slots, dO_i in one.
//   warp 17     tcgen05, per query tile i: once P^T is in, dV += P^T dO_i and S^T of tile
//               i + 1 (over P^T, after dV has read it); once dS^T is in, dK += dS^T Q_i and dP^T
//               of tile i + 1.
//   warps 0-15  four warpgroups on the same tile, warpgroup w on its queries [32w, 32w + 32);
//               thread = key row: P^T (bf16 over the group's S^T columns, fp32 kept), then dS^T
//               (bf16) into the dS^T tile.  At the end warpgroups 0-1 write dK (times scale) and
//               2-3 dV, 64 columns each, through the Q slots and TMA stores.
// TMEM columns: dK [0,128), dV [128,256), dP^T [256,384), S^T [384,512).
struct D128Cfg {
    static constexpr int D = 128;
    static constexpr int BN = 128;   // keys per CTA
    static constexpr int BM = 128;   // queries per tile
    static constexpr int QST = 2;    // Q slots
    static constexpr int T_BYTES = 128 * D * 2;       // one 128 x 128 bf16 tile, two 64-column blocks
    static constexpr int BLK = 128 * 128;             // bytes of one 64-column block of 128 rows
    static constexpr int LD_BYTES = 2 * BM * 4;       // statistics of one tile
    static constexpr int SMEM_BYTES = 2 * T_BYTES + QST * T_BYTES + T_BYTES + T_BYTES + QST * LD_BYTES + 1024;
    static constexpr int PDS_WARPS = 16;
    static constexpr int THREADS = 32 * (PDS_WARPS + 2);
    static constexpr int TMA_WARP = PDS_WARPS, MMA_WARP = PDS_WARPS + 1;
    static constexpr uint32_t TM_DK = 0, TM_DV = 128, TM_DP = 256, TM_S = 384;
};

__global__ void __launch_bounds__(D128Cfg::THREADS, 1)
    bwd_dkdv_d128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                         const float *__restrict__ stats, int n, int n_pad, int n_kvblocks, float scale,
                         int *status)
{
    using C = D128Cfg;
    constexpr int D = C::D;
    constexpr uint32_t PDS_THREADS = 32 * C::PDS_WARPS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sK = smem;
    uint8_t *sV = sK + C::T_BYTES;
    uint8_t *sQ = sV + C::T_BYTES;                  // QST slots of Q_i
    uint8_t *sDO = sQ + C::QST * C::T_BYTES;        // dO_i
    uint8_t *sDS = sDO + C::T_BYTES;                // dS^T, two 64-query blocks of 128 key rows
    float *sLD = reinterpret_cast<float *>(sDS + C::T_BYTES);   // QST x statistics

    __shared__ uint64_t bar_kv, bar_qf[C::QST], bar_qe[C::QST], bar_dof, bar_doe;
    __shared__ uint64_t bar_s_full, bar_p_full, bar_dp_full, bar_ds_full, bar_dkv, bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / n_kvblocks;
    const int kv0 = (blockIdx.x % n_kvblocks) * C::BN;
    const int nq = (n + C::BM - 1) / C::BM;
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        ptx::mbar_init(&bar_kv, 1);
        for (int s = 0; s < C::QST; ++s) {
            ptx::mbar_init(&bar_qf[s], 1);
            ptx::mbar_init(&bar_qe[s], 1);
        }
        ptx::mbar_init(&bar_dof, 1);
        ptx::mbar_init(&bar_doe, 1);
        ptx::mbar_init(&bar_s_full, 1);
        ptx::mbar_init(&bar_p_full, PDS_THREADS);
        ptx::mbar_init(&bar_dp_full, 1);
        ptx::mbar_init(&bar_ds_full, PDS_THREADS);
        ptx::mbar_init(&bar_dkv, 1);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(&tmem_sh, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == C::TMA_WARP) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_do);
            ptx::mbar_arrive_expect_tx(&bar_kv, 2 * C::T_BYTES);
            for (int h = 0; h < 2; ++h) {
                ptx::tma_load_3d(sK + h * C::BLK, &tm_k, &bar_kv, h * 64, kv0, bh);
                ptx::tma_load_3d(sV + h * C::BLK, &tm_v, &bar_kv, h * 64, kv0, bh);
            }
            // The Q / dO maps have 64-row boxes: four per tile (two column blocks x two row
            // halves), contiguous in the 128-byte-swizzled layout of each column block.
            for (int it = 0; it < nq; ++it) {
                const int s = it & 1;
                wait_bounded(&bar_qe[s], ((it >> 1) & 1) ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_qf[s], C::T_BYTES + C::LD_BYTES);
                uint8_t *slot = sQ + s * C::T_BYTES;
                for (int h = 0; h < 2; ++h)
                    for (int rr = 0; rr < 2; ++rr)
                        ptx::tma_load_3d(slot + h * C::BLK + rr * 64 * 128, &tm_q, &bar_qf[s], h * 64,
                                         it * C::BM + rr * 64, bh);
                const size_t rowvec = (size_t)bh * n_pad + (size_t)it * C::BM;
                ptx::bulk_load(sLD + s * 2 * C::BM, stats + rowvec * 2, C::BM * 8, &bar_qf[s]);
                wait_bounded(&bar_doe, (it & 1) ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_dof, C::T_BYTES);
                for (int h = 0; h < 2; ++h)
                    for (int rr = 0; rr < 2; ++rr)
                        ptx::tma_load_3d(sDO + h * C::BLK + rr * 64 * 128, &tm_do, &bar_dof, h * 64,
                                         it * C::BM + rr * 64, bh);
            }
            wait_bounded(&bar_kv, 0, g);
            for (int it = (nq > C::QST ? nq - C::QST : 0); it < nq; ++it)
                wait_bounded(&bar_qf[it & 1], (it >> 1) & 1, g);
            if (nq > 0) wait_bounded(&bar_dof, (nq - 1) & 1, g);
        }
    } else if (warp == C::MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idSdP = ptx::idesc_bf16_f32(128, C::BM, false, false);
            const uint32_t idKV = ptx::idesc_bf16_f32(128, D, false, true);
            const uint32_t k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV);
            const uint32_t q_base = ptx::smem_u32(sQ), do_base = ptx::smem_u32(sDO);
            const uint32_t ds_base = ptx::smem_u32(sDS);
            // S^T = K_j Q_i^T and dP^T = V_j dO_i^T: all four operands K-major over d (two
            // 64-column blocks), N = 128 queries.
            auto issue_s = [&](int s) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::BLK + (kk & 3) * 32;
                    ptx::mma_ss(tmem + C::TM_S, ptx::sdesc_sw128(k_base + off, 16, 1024),
                                ptx::sdesc_sw128(q_base + s * C::T_BYTES + off, 16, 1024), idSdP, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_dp = [&]() {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::BLK + (kk & 3) * 32;
                    ptx::mma_ss(tmem + C::TM_DP, ptx::sdesc_sw128(v_base + off, 16, 1024),
                                ptx::sdesc_sw128(do_base + off, 16, 1024), idSdP, kk > 0 ? 1u : 0u);
                }
            };
            // dV += P^T dO_i: P^T of queries [16kk, 16kk + 16) sits in the S^T columns of the
            // warpgroup that produced it (32 (kk / 2) + 8 (kk % 2)); dO_i MN-major (N = d in two
            // 64-column blocks BLK bytes apart).
            auto issue_dv = [&](bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ts(tmem + C::TM_DV, tmem + C::TM_S + (kk >> 1) * 32 + (kk & 1) * 8,
                                ptx::sdesc_sw128(do_base + kk * 2048, C::BLK, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            // dK += dS^T Q_i: dS^T K-major (two 64-query blocks BLK bytes apart), Q_i MN-major.
            auto issue_dk = [&](int s, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DK,
                                ptx::sdesc_sw128(ds_base + (kk >> 2) * C::BLK + (kk & 3) * 32, 16, 1024),
                                ptx::sdesc_sw128(q_base + s * C::T_BYTES + kk * 2048, C::BLK, 1024), idKV,
                                (acc || kk > 0) ? 1u : 0u);
            };
            wait_bounded(&bar_kv, 0, g);
            if (nq > 0) {
                wait_bounded(&bar_qf[0], 0, g);
                ptx::tc_fence_after();
                issue_s(0);
                ptx::mma_commit(&bar_s_full);
                wait_bounded(&bar_dof, 0, g);
                ptx::tc_fence_after();
                issue_dp();
                ptx::mma_commit(&bar_dp_full);
            }
            for (int it = 0; it < nq; ++it) {
                const int s = it & 1;
                const bool more = it + 1 < nq;
                wait_bounded(&bar_p_full, it & 1, g);
                ptx::tc_fence_after();
                issue_dv(it > 0);
                ptx::mma_commit(&bar_doe);                     // dO_i read (dP^T and dV)
                if (more) {   // over P^T, after dV has read it (in order)
                    wait_bounded(&bar_qf[s ^ 1], ((it + 1) >> 1) & 1, g);
                    ptx::tc_fence_after();
                    issue_s(s ^ 1);
                    ptx::mma_commit(&bar_s_full);
                }
                wait_bounded(&bar_ds_full, it & 1, g);
                ptx::tc_fence_after();
                issue_dk(s, it > 0);
                ptx::mma_commit(&bar_qe[s]);
                if (more) {   // dP^T is free: the P / dS warps have read it (dS^T is in)
                    wait_bounded(&bar_dof, (it + 1) & 1, g);
                    ptx::tc_fence_after();
                    issue_dp();
                    ptx::mma_commit(&bar_dp_full);
                }
            }
            ptx::mma_commit(&bar_dkv);
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else {
        // ---------------------------------------------------------------- P / dS warpgroups
        const int wg = warp >> 2, cw = warp & 3;
        const int r = cw * 32 + lane;       // key row within the tile = TMEM lane
        const bool key_ok = kv0 + r < n;
        const uint32_t lane_off = (uint32_t)(cw * 32) << 16;
        const float scale_log2 = scale * kLog2e;
        const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2);
        const uint32_t rowp_a = ptx::smem_u32(sDS + (wg >> 1) * C::BLK + r * 128);
        const int chunk0 = (wg & 1) * 4;    // the group's 32 queries: 16-byte chunks [chunk0, chunk0 + 4)
        const uint32_t tS = tmem + lane_off + C::TM_S + wg * 32;
        const uint32_t tDP = tmem + lane_off + C::TM_DP + wg * 32;
        for (int it = 0; it < nq; ++it) {
            const int s = it & 1;
            // {-LSE2 pair, -D pair} per two of this warpgroup's queries
            const uint32_t sst_a = ptx::smem_u32(sLD + s * 2 * C::BM + wg * 64);
            wait_bounded(&bar_s_full, it & 1, g);
            ptx::tc_fence_after();
            // Phase 1, as soon as S^T is in: P^T = 2^(S^T c - LSE2), 16 queries at a time (the
            // next 16 columns load meanwhile), bf16 back into TMEM over S^T columns already
            // read, fp32 kept for dS.
            float pf[32];
            {
                uint32_t sv[2][16];
                ptx::tmem_ld16(tS, sv[0]);
                ptx::tmem_ld16(tS + 16, sv[1]);
                ptx::tmem_ld_wait();
                reg_fence(sv[0]);
                reg_fence(sv[1]);
#pragma unroll
                for (int qt = 0; qt < 2; ++qt) {
                    uint2 nl[8];   // -LSE2 of queries (c, c + 1), c = 0, 2, ..., 14
#pragma unroll
                    for (int e = 0; e < 8; ++e) nl[e] = lds_u64(sst_a + (qt * 16 + 2 * e) * 8);
                    uint32_t pp[8];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        const uint64_t x = ptx::fma_f32x2(
                            ptx::f2_pack(__uint_as_float(sv[qt][c]), __uint_as_float(sv[qt][c + 1])), c2,
                            ((uint64_t)nl[c / 2].y << 32) | nl[c / 2].x);
                        float x0, x1;
                        ptx::f2_unpack(x, x0, x1);
                        float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        if (!key_ok) p0 = p1 = 0.f;
                        pf[qt * 16 + c] = p0;
                        pf[qt * 16 + c + 1] = p1;
                        pp[c / 2] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st8(tS + qt * 8, pp);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_p_full);
            // Phase 2, once dP^T is in (which also means tile i - 1's dK, issued before it, is
            // done with the dS^T tile): dS^T = P^T o (dP^T - D), bf16 into shared memory.
            wait_bounded(&bar_dp_full, it & 1, g);
            ptx::tc_fence_after();
            {
                uint32_t dpv[2][16];
                ptx::tmem_ld16(tDP, dpv[0]);
                ptx::tmem_ld16(tDP + 16, dpv[1]);
                ptx::tmem_ld_wait();
                reg_fence(dpv[0]);
                reg_fence(dpv[1]);
#pragma unroll
                for (int qt = 0; qt < 2; ++qt) {
                    uint2 nd[8];   // -D of queries (c, c + 1)
#pragma unroll
                    for (int e = 0; e < 8; ++e) nd[e] = lds_u64(sst_a + (qt * 16 + 2 * e) * 8 + 8);
                    uint32_t dsp[8];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        const uint64_t dsq = ptx::mul_f32x2(
                            ptx::f2_pack(pf[qt * 16 + c], pf[qt * 16 + c + 1]),
                            ptx::add_f32x2(ptx::f2_pack(__uint_as_float(dpv[qt][c]), __uint_as_float(dpv[qt][c + 1])),
                                           ((uint64_t)nd[c / 2].y << 32) | nd[c / 2].x));
                        float ds0, ds1;
                        ptx::f2_unpack(dsq, ds0, ds1);
                        dsp[c / 2] = ptx::pack_bf16x2(ds0, ds1);
                    }
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
                        sts_u128(rowp_a + (((chunk0 + qt * 2 + cc) ^ (r & 7)) << 4),
                                 make_uint4(dsp[4 * cc], dsp[4 * cc + 1], dsp[4 * cc + 2], dsp[4 * cc + 3]));
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_ds_full);
        }
        // epilogue: warpgroups 0-1 write dK = scale * acc, 2-3 dV = acc, 64 columns each, bf16,
        // staged in the now idle Q slots in the 128-byte-swizzled layout (16-byte chunk c of
        // row r at chunk c ^ (r % 8), one 64-column block per group) and stored with TMA tensor
        // stores (rows past N clipped)
        wait_bounded(&bar_dkv, 0, g);
        ptx::tc_fence_after();
        {
            const int which = wg >> 1, half = wg & 1;
            const float mul = which == 0 ? scale : 1.f;
            const uint32_t col0 = (which == 0 ? C::TM_DK : C::TM_DV) + half * 64;
            const uint32_t srow = ptx::smem_u32(sQ + which * C::T_BYTES + half * C::BLK) + r * 128;
#pragma unroll
            for (int c = 0; c < 64; c += 32) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + lane_off + col0 + c, v);
                ptx::tmem_ld_wait();
                reg_fence(v);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    sts_u128(srow + ((((c >> 3) + v4) ^ (r & 7)) << 4),
                             make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]));
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar(1, PDS_THREADS);
            if (threadIdx.x == 0) {
                for (int h = 0; h < 2; ++h) {
                    ptx::tma_store_3d(&tm_dk, sQ + h * C::BLK, h * 64, kv0, bh);
                    ptx::tma_store_3d(&tm_dv, sQ + C::T_BYTES + h * C::BLK, h * 64, kv0, bh);
                }
                ptx::bulk_commit_group();
                ptx::bulk_wait_group<0>();   // complete before the CTA exits
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 2'''. whole heads, d = 64, N <= 256
// Short sequences at d = 64 (N <= 256: at most two 128-row key blocks and query tiles per
// head): one CTA takes a whole head (in turn, should there be more heads than CTAs; the
// dispatch below keeps it to one), so that dQ accumulates in TMEM across the head's key
// blocks instead of in an fp32 accumulator in L2, and the row statistic D = rowsum(dO o O) is
// computed on chip.  dQ, dK and dV leave as bf16 straight
// from TMEM: no preprocess, zero-fill, reduce-add or convert pass, and no atomics (the result
// is bitwise reproducible).
//   warp 8      TMA: per head K, V (nkb 128-row key blocks) and Q, dO (nqt 128-row query tiles)
//               into fixed buffers, once every product of the previous head has read them.
//   warp 9      tcgen05, per step (key block kb, query tile qt): S^T = K_kb Q_qt^T and
//               dP^T = V_kb dO_qt^T; once P^T (TMEM) and dS^T (shared memory) are in:
//               dV_kb += P^T dO_qt, dK_kb += dS^T Q_qt and dQ_qt += dS K_kb; then the next
//               step's S^T and dP^T (in order after the products that read their columns).
//   warps 0-7   at each head the per-query statistics (thread = query: -LSE log2 e and -D, D
//               from O in global memory and dO in shared memory), then per step two
//               warpgroups on the tile (warpgroup g on queries [64g, 64g + 64), thread = key
//               row): P^T = 2^(S^T c - LSE2) (bf16 over S^T in TMEM) and dS^T = P^T o (dP^T - D)
//               (bf16 into shared memory); after each key block's last step dK (warpgroup 0,
//               times scale) and dV (warpgroup 1), after the head's last step dQ (warpgroup g:
//               query tile g, times scale), bf16, row by row to global memory.
// TMEM columns: dQ_0 [0,64), dQ_1 [64,128), dK [128,192), dV [192,256), S^T [256,384),
// dP^T [384,512).
struct HeadCfg {
    static constexpr int D = 64;
    static constexpr int T = 128;                  // rows of a key block / query tile
    static constexpr int TILE = T * D * 2;         // one 128-row tile, 16 KB (one 64-column block)
    static constexpr int STATS_BYTES = 2 * T * 8;  // {-LSE2, -D} of 256 queries, per pair of rows
    static constexpr int SMEM_BYTES = 10 * TILE + STATS_BYTES + 1024;   // K, V, Q, dO, dS^T: 2 tiles each
    static constexpr int PDS_WARPS = 8;
    static constexpr int THREADS = 32 * (PDS_WARPS + 2);
    static constexpr int TMA_WARP = PDS_WARPS, MMA_WARP = PDS_WARPS + 1;
    static constexpr uint32_t TM_DQ = 0, TM_DK = 128, TM_DV = 192, TM_S = 256, TM_DP = 384;
};

__global__ void __launch_bounds__(HeadCfg::THREADS, 1)
    bwd_head_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __nv_bfloat16 *__restrict__ o, const float *__restrict__ lse,
                    __nv_bfloat16 *__restrict__ dq, __nv_bfloat16 *__restrict__ dk,
                    __nv_bfloat16 *__restrict__ dv, int n, int n_heads, float scale, int *status)
{
    using C = HeadCfg;
    constexpr int D = C::D;
    constexpr uint32_t PDS_THREADS = 32 * C::PDS_WARPS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sK = smem;                       // key blocks 0, 1
    uint8_t *sV = sK + 2 * C::TILE;
    uint8_t *sQ = sV + 2 * C::TILE;           // query tiles 0, 1 (two 64-row boxes each)
    uint8_t *sDO = sQ + 2 * C::TILE;
    uint8_t *sDS = sDO + 2 * C::TILE;         // dS^T: two 64-query blocks of 128 key rows
    float *sLD = reinterpret_cast<float *>(sDS + 2 * C::TILE);

    __shared__ uint64_t bar_load, bar_head_done, bar_sdp, bar_ds, bar_kv_ready, bar_kv_read, bar_dq_read;
    __shared__ uint64_t bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = (n + C::T - 1) / C::T;     // key blocks = query tiles (1 or 2)
    const int first = blockIdx.x, stride = gridDim.x;
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        ptx::mbar_init(&bar_load, 1);
        ptx::mbar_init(&bar_head_done, 1);
        ptx::mbar_init(&bar_sdp, 1);
        ptx::mbar_init(&bar_ds, PDS_THREADS);
        ptx::mbar_init(&bar_kv_ready, 1);
        ptx::mbar_init(&bar_kv_read, PDS_THREADS);
        ptx::mbar_init(&bar_dq_read, PDS_THREADS);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(&tmem_sh, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == C::TMA_WARP) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_do);
            int hl = 0;
            for (int bh = first; bh < n_heads; bh += stride, ++hl) {
                if (hl > 0) wait_bounded(&bar_head_done, (hl - 1) & 1, g);   // the buffers are free
                ptx::mbar_arrive_expect_tx(&bar_load, 4 * nt * C::TILE);
                for (int t = 0; t < nt; ++t) {
                    ptx::tma_load_3d(sK + t * C::TILE, &tm_k, &bar_load, 0, t * C::T, bh);
                    ptx::tma_load_3d(sV + t * C::TILE, &tm_v, &bar_load, 0, t * C::T, bh);
                    for (int hh = 0; hh < 2; ++hh) {   // the Q / dO maps have 64-row boxes
                        ptx::tma_load_3d(sQ + t * C::TILE + hh * 64 * 128, &tm_q, &bar_load, 0,
                                         t * C::T + hh * 64, bh);
                        ptx::tma_load_3d(sDO + t * C::TILE + hh * 64 * 128, &tm_do, &bar_load, 0,
                                         t * C::T + hh * 64, bh);
                    }
                }
            }
            if (hl > 0) wait_bounded(&bar_load, (hl - 1) & 1, g);   // no copy in flight at exit
        }
    } else if (warp == C::MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idSdP = ptx::idesc_bf16_f32(128, C::T, false, false);
            const uint32_t idKV = ptx::idesc_bf16_f32(128, D, false, true);
            const uint32_t idDQ = ptx::idesc_bf16_f32(128, D, true, true);
            const uint32_t k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV);
            const uint32_t q_base = ptx::smem_u32(sQ), do_base = ptx::smem_u32(sDO);
            const uint32_t ds_base = ptx::smem_u32(sDS);
            // S^T = K_kb Q_qt^T, dP^T = V_kb dO_qt^T: K-major over d (one 64-column block)
            auto issue_sdp = [&](int kb, int qt) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_S, ptx::sdesc_sw128(k_base + kb * C::TILE + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(q_base + qt * C::TILE + kk * 32, 16, 1024), idSdP,
                                kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DP, ptx::sdesc_sw128(v_base + kb * C::TILE + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(do_base + qt * C::TILE + kk * 32, 16, 1024), idSdP,
                                kk > 0 ? 1u : 0u);
            };
            // K = 128 queries (dV, dK) or 128 keys (dQ), 16 per product
            auto issue_products = [&](int kb, int qt) {
                // dV += P^T dO: P^T of queries [16kk, 16kk + 16) in the S^T columns of warpgroup
                // kk / 4 (64 (kk / 4) + 8 (kk % 4)); dO MN-major (N = d)
#pragma unroll
                for (int kk = 0; kk < C::T / 16; ++kk)
                    ptx::mma_ts(tmem + C::TM_DV, tmem + C::TM_S + (kk >> 2) * 64 + (kk & 3) * 8,
                                ptx::sdesc_sw128(do_base + qt * C::TILE + kk * 2048, C::TILE, 1024), idKV,
                                (qt > 0 || kk > 0) ? 1u : 0u);
                // dK += dS^T Q: dS^T K-major (two 64-query blocks), Q MN-major
#pragma unroll
                for (int kk = 0; kk < C::T / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DK,
                                ptx::sdesc_sw128(ds_base + (kk >> 2) * C::TILE + (kk & 3) * 32, 16, 1024),
                                ptx::sdesc_sw128(q_base + qt * C::TILE + kk * 2048, C::TILE, 1024), idKV,
                                (qt > 0 || kk > 0) ? 1u : 0u);
                // dQ_qt += dS K_kb: A = dS (M = 128 queries) MN-major from the dS^T tile (its two
                // 64-query blocks TILE bytes apart), B = K_kb MN-major (N = d); K = 128 keys
#pragma unroll
                for (int kk = 0; kk < C::T / 16; ++kk)
                    ptx::mma_ss(tmem + C::TM_DQ + qt * 64, ptx::sdesc_sw128(ds_base + kk * 2048, C::TILE, 1024),
                                ptx::sdesc_sw128(k_base + kb * C::TILE + kk * 2048, C::TILE, 1024), idDQ,
                                (kb > 0 || kk > 0) ? 1u : 0u);
            };
            int hl = 0, step = 0, kbs = 0;
            for (int bh = first; bh < n_heads; bh += stride, ++hl) {
                wait_bounded(&bar_load, hl & 1, g);
                ptx::tc_fence_after();
                issue_sdp(0, 0);
                ptx::mma_commit(&bar_sdp);
                for (int kb = 0; kb < nt; ++kb) {
                    for (int qt = 0; qt < nt; ++qt, ++step) {
                        wait_bounded(&bar_ds, step & 1, g);
                        // the accumulators restart: dK / dV once the previous key block's
                        // epilogue has read them, dQ once the previous head's has
                        if (qt == 0 && kbs > 0) wait_bounded(&bar_kv_read, (kbs - 1) & 1, g);
                        if (kb == 0 && qt == 0 && hl > 0) wait_bounded(&bar_dq_read, (hl - 1) & 1, g);
                        ptx::tc_fence_after();
                        issue_products(kb, qt);
                        if (qt == nt - 1) ptx::mma_commit(&bar_kv_ready);
                        const bool last = kb == nt - 1 && qt == nt - 1;
                        if (!last) {   // over P^T and dP^T, after the products that read them
                            const int nkb = qt == nt - 1 ? kb + 1 : kb, nqt = qt == nt - 1 ? 0 : qt + 1;
                            issue_sdp(nkb, nqt);
                            ptx::mma_commit(&bar_sdp);
                        }
                    }
                    ++kbs;
                }
                ptx::mma_commit(&bar_head_done);   // Q, K, V, dO and dS^T read
            }
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else {
        // ---------------------------------------------------------------- P / dS warpgroups
        const int wg = warp >> 2, cw = warp & 3;
        const int r = cw * 32 + lane;       // key row of the block = TMEM lane (query row in the dQ epilogue)
        const uint32_t lane_off = (uint32_t)(cw * 32) << 16;
        const float scale_log2 = scale * kLog2e;
        const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2);
        const uint32_t tS = tmem + lane_off + C::TM_S + wg * 64, tDP = tmem + lane_off + C::TM_DP + wg * 64;
        const uint32_t rowp_a = ptx::smem_u32(sDS + wg * C::TILE + r * 128);
        const uint32_t ld_base = ptx::smem_u32(sLD);
        int hl = 0, step = 0, kbs = 0;
        for (int bh = first; bh < n_heads; bh += stride, ++hl) {
            wait_bounded(&bar_load, hl & 1, g);
            {   // per-query statistics: thread t takes query t; {-LSE2, -D} interleaved per pair
                const int qrow = (int)threadIdx.x;   // 0 .. 255
                float nl = -INFINITY, nd = 0.f;
                if (qrow < n) {
                    nl = -lse[(size_t)bh * n + qrow] * kLog2e;
                    const uint4 *orow = reinterpret_cast<const uint4 *>(o + ((size_t)bh * n + qrow) * D);
                    const uint32_t dorow = ptx::smem_u32(sDO + (qrow >> 7) * C::TILE + (qrow & 127) * 128);
                    float acc = 0.f;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 ov = __ldg(orow + c);
                        const uint4 dv4 = lds_u128(dorow + ((c ^ (qrow & 7)) << 4));
                        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc = fmaf(__uint_as_float(ow[e] << 16), __uint_as_float(dw[e] << 16), acc);
                            acc = fmaf(__uint_as_float(ow[e] & 0xffff0000u), __uint_as_float(dw[e] & 0xffff0000u), acc);
                        }
                    }
                    nd = -acc;
                }
                sts_f32(ld_base + (uint32_t)((qrow >> 1) * 4 + (qrow & 1)) * 4, nl);
                sts_f32(ld_base + (uint32_t)((qrow >> 1) * 4 + 2 + (qrow & 1)) * 4, nd);
                ptx::named_bar(1, PDS_THREADS);
            }
            for (int kb = 0; kb < nt; ++kb) {
                const bool key_ok = kb * C::T + r < n;
                for (int qt = 0; qt < nt; ++qt, ++step) {
                    // this warpgroup's 64 queries: {-LSE2 pair, -D pair} per two queries
                    const uint32_t sst_a = ld_base + (uint32_t)(qt * C::T + wg * 64) * 8;
                    wait_bounded(&bar_sdp, step & 1, g);
                    ptx::tc_fence_after();
                    // 16 queries at a time; the next quarter's TMEM loads overlap this quarter's
                    // math.  P^T of quarter q4 goes to columns [8 q4, 8 q4 + 8) over S^T columns
                    // already read.
                    uint32_t sv[2][16], dpv[2][16];
                    ptx::tmem_ld16(tS, sv[0]);
                    ptx::tmem_ld16(tDP, dpv[0]);
                    ptx::tmem_ld_wait();
                    reg_fence(sv[0]);
                    reg_fence(dpv[0]);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int cur = q4 & 1;
                        if (q4 < 3) {
                            ptx::tmem_ld16(tS + (q4 + 1) * 16, sv[cur ^ 1]);
                            ptx::tmem_ld16(tDP + (q4 + 1) * 16, dpv[cur ^ 1]);
                        }
                        uint32_t pp[8], dsp[8];
                        uint4 st4[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) st4[e] = lds_u128(sst_a + (q4 * 16 + 2 * e) * 8);
#pragma unroll
                        for (int c = 0; c < 16; c += 2) {
                            const uint64_t nl = ((uint64_t)st4[c / 2].y << 32) | st4[c / 2].x;
                            const uint64_t nd = ((uint64_t)st4[c / 2].w << 32) | st4[c / 2].z;
                            const uint64_t x = ptx::fma_f32x2(
                                ptx::f2_pack(__uint_as_float(sv[cur][c]), __uint_as_float(sv[cur][c + 1])), c2, nl);
                            float x0, x1;
                            ptx::f2_unpack(x, x0, x1);
                            float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                            if (!key_ok) p0 = p1 = 0.f;
                            const uint64_t pq = ptx::f2_pack(p0, p1);
                            const uint64_t dsq = ptx::mul_f32x2(
                                pq, ptx::add_f32x2(ptx::f2_pack(__uint_as_float(dpv[cur][c]), __uint_as_float(dpv[cur][c + 1])), nd));
                            float ds0, ds1;
                            ptx::f2_unpack(dsq, ds0, ds1);
                            pp[c / 2] = ptx::pack_bf16x2(p0, p1);
                            dsp[c / 2] = ptx::pack_bf16x2(ds0, ds1);
                        }
                        ptx::tmem_st8(tS + q4 * 8, pp);
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc)
                            sts_u128(rowp_a + (((q4 * 2 + cc) ^ (r & 7)) << 4),
                                     make_uint4(dsp[4 * cc], dsp[4 * cc + 1], dsp[4 * cc + 2], dsp[4 * cc + 3]));
                        if (q4 < 3) {
                            ptx::tmem_ld_wait();
                            reg_fence(sv[cur ^ 1]);
                            reg_fence(dpv[cur ^ 1]);
                        }
                    }
                    ptx::tmem_st_wait();
                    ptx::fence_proxy_async_smem();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(&bar_ds);
                }
                // the key block's dK (warpgroup 0, times scale) and dV (warpgroup 1), bf16, rows < n
                wait_bounded(&bar_kv_ready, kbs & 1, g);
                ptx::tc_fence_after();
                {
                    const float mul = wg == 0 ? scale : 1.f;
                    const uint32_t col0 = wg == 0 ? C::TM_DK : C::TM_DV;
                    __nv_bfloat16 *dst = (wg == 0 ? dk : dv) + ((size_t)bh * n + kb * C::T + r) * D;
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t v[32];
                        ptx::tmem_ld32(tmem + lane_off + col0 + c, v);
                        ptx::tmem_ld_wait();
                        reg_fence(v);
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                        if (key_ok) {
                            uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4)
                                d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                        }
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bar_kv_read);
                ++kbs;
            }
            // the head's dQ: warpgroup g takes query tile g (thread = query row), times scale
            if (wg < nt) {
                const int qrow = wg * C::T + r;
                __nv_bfloat16 *dst = dq + ((size_t)bh * n + qrow) * D;
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tmem + lane_off + C::TM_DQ + wg * 64 + c, v);
                    ptx::tmem_ld_wait();
                    reg_fence(v);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]) * scale, __uint_as_float(v[2 * e + 1]) * scale);
                    if (qrow < n) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_dq_read);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ 4. deterministic dQ pass
// dQ_i = scale * sum_j dS_ij K_j without atomics: one CTA owns 128 query rows of one head and
// walks the key tiles (128 keys each) in order, recomputing S = Q K^T and dP = dO V^T on chip.
// With 128-key steps S and dP run at N = 128 (an M = 128 MMA takes as long at N = 64).
//   warp 8      TMA: Q_i and dO_i once; a ring of K_j and a ring of V_j.
//   warp 9      tcgen05, per key tile j (S buffer b = j & 1), once dS_j is in: dP of tile
//               j + 1 first (the P / dS warps have read dP_j), then dQ += dS_j K_j (dS_j read
//               from TMEM, bf16 over S_j; K_j MN-major), then S of tile j + 2 into buffer b
//               (issued after the dQ product that reads it, so in order).
//   warps 0-7   both warpgroups on the same key tile, warpgroup h on its keys [64h, 64h + 64);
//               thread = query row, whose LSE and D sit in registers.  First P = 2^(S c - LSE
//               log2 e) as soon as S_j is in (fp32 kept), then dS = P o (dP - D) once dP_j is
//               in, bf16 over the warpgroup's own S columns (keys [64h, 64h + 64) -> columns
//               [64h, 64h + 32)).
// TMEM: S_0 [0,128), S_1 [128,256), dP [256,384), dQ [384,384+d).
template <int D>
struct DqCfg {
    static constexpr int BM = 128;   // query rows per CTA
    static constexpr int BN = 128;   // keys per step
    static constexpr int KST = (D == 64) ? 4 : 3;   // K ring
    static constexpr int VST = (D == 64) ? 3 : 2;   // V ring (V is read only by dP, one step ahead)
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int SMEM_BYTES = 2 * Q_BYTES + (KST + VST) * KV_BYTES + 1024;
    static constexpr int THREADS = 320;
    static constexpr uint32_t TM_DP = 256, TM_DQ = 384;
    __host__ __device__ static constexpr uint32_t tm_s(int b) { return b * 128; }
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const float *__restrict__ stats, __nv_bfloat16 *__restrict__ dq, int n, int n_pad,
                  int n_qblocks, float scale, int *status)
{
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sQ = smem;                      // Q_i: d / 64 column blocks of 128 rows
    uint8_t *sdO = sQ + C::Q_BYTES;          // dO_i, same layout
    uint8_t *sK = sdO + C::Q_BYTES;          // KST x K_j
    uint8_t *sV = sK + C::KST * C::KV_BYTES; // VST x V_j

    __shared__ uint64_t bar_q, bar_kf[C::KST], bar_ke[C::KST], bar_vf[C::VST], bar_ve[C::VST];
    __shared__ uint64_t bar_s_full[2], bar_dp_full, bar_ds_full, bar_dq, bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / n_qblocks;
    const int q0 = (blockIdx.x % n_qblocks) * C::BM;
    const int nk = (n + C::BN - 1) / C::BN;
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        ptx::mbar_init(&bar_q, 1);
        for (int s = 0; s < C::KST; ++s) {
            ptx::mbar_init(&bar_kf[s], 1);
            ptx::mbar_init(&bar_ke[s], 1);
        }
        for (int s = 0; s < C::VST; ++s) {
            ptx::mbar_init(&bar_vf[s], 1);
            ptx::mbar_init(&bar_ve[s], 1);
        }
        for (int b = 0; b < 2; ++b) ptx::mbar_init(&bar_s_full[b], 1);
        ptx::mbar_init(&bar_dp_full, 1);
        ptx::mbar_init(&bar_ds_full, 256);
        ptx::mbar_init(&bar_dq, 1);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 9) {
        ptx::tmem_alloc(&tmem_sh, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == 8) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_do);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            // the Q / dO maps have 64-row boxes: two per 128-row tile, contiguous in the
            // 128-byte-swizzled layout; d = 128 tiles are two 64-column blocks of 16 KB
            ptx::mbar_arrive_expect_tx(&bar_q, 2 * C::Q_BYTES);
            for (int h = 0; h < D / 64; ++h)
                for (int r = 0; r < 2; ++r) {
                    ptx::tma_load_3d(sQ + h * C::BM * 128 + r * 64 * 128, &tm_q, &bar_q, h * 64, q0 + r * 64, bh);
                    ptx::tma_load_3d(sdO + h * C::BM * 128 + r * 64 * 128, &tm_do, &bar_q, h * 64, q0 + r * 64, bh);
                }
            // K_j and V_j in key order; V runs at most VST tiles ahead of dP, K at most KST
            // tiles ahead of dQ
            for (int j = 0; j < nk; ++j) {
                const int sk = j % C::KST, sv = j % C::VST;
                wait_bounded(&bar_ke[sk], ((j / C::KST) & 1) ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_kf[sk], C::KV_BYTES);
                for (int h = 0; h < D / 64; ++h)
                    ptx::tma_load_3d(sK + sk * C::KV_BYTES + h * C::BN * 128, &tm_k, &bar_kf[sk], h * 64, j * C::BN, bh);
                wait_bounded(&bar_ve[sv], ((j / C::VST) & 1) ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_vf[sv], C::KV_BYTES);
                for (int h = 0; h < D / 64; ++h)
                    ptx::tma_load_3d(sV + sv * C::KV_BYTES + h * C::BN * 128, &tm_v, &bar_vf[sv], h * 64, j * C::BN, bh);
            }
            wait_bounded(&bar_q, 0, g);
            for (int j = (nk > C::VST ? nk - C::VST : 0); j < nk; ++j)
                wait_bounded(&bar_vf[j % C::VST], (j / C::VST) & 1, g);
            for (int j = (nk > C::KST ? nk - C::KST : 0); j < nk; ++j)
                wait_bounded(&bar_kf[j % C::KST], (j / C::KST) & 1, g);
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idSP = ptx::idesc_bf16_f32(128, C::BN, false, false);
            const uint32_t idQ = ptx::idesc_bf16_f32(128, D, false, true);
            const uint32_t q_base = ptx::smem_u32(sQ), do_base = ptx::smem_u32(sdO),
                           k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV);
            // S_j = Q K_j^T and dP_j = dO V_j^T: all operands K-major over d (64-column blocks
            // BM * 128 / BN * 128 bytes apart), N = 128 keys.
            auto issue_s = [&](int sk, int b) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offa = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
                    const uint32_t offb = (kk >> 2) * (C::BN * 128) + (kk & 3) * 32;
                    ptx::mma_ss(tmem + C::tm_s(b), ptx::sdesc_sw128(q_base + offa, 16, 1024),
                                ptx::sdesc_sw128(k_base + sk * C::KV_BYTES + offb, 16, 1024), idSP,
                                kk > 0 ? 1u : 0u);
                }
            };
            auto issue_dp = [&](int sv) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offa = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
                    const uint32_t offb = (kk >> 2) * (C::BN * 128) + (kk & 3) * 32;
                    ptx::mma_ss(tmem + C::TM_DP, ptx::sdesc_sw128(do_base + offa, 16, 1024),
                                ptx::sdesc_sw128(v_base + sv * C::KV_BYTES + offb, 16, 1024), idSP,
                                kk > 0 ? 1u : 0u);
                }
            };
            // dQ += dS_j K_j: A = dS_j from TMEM (keys [16kk, 16kk + 16) in the columns of the
            // warpgroup that wrote them: 64 (kk / 4) + 8 (kk % 4)), B = K_j MN-major (K = keys,
            // N = d; 64-column blocks BN * 128 bytes apart).
            auto issue_dq = [&](int sk, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    ptx::mma_ts(tmem + C::TM_DQ, tmem + C::tm_s(b) + (kk >> 2) * 64 + (kk & 3) * 8,
                                ptx::sdesc_sw128(k_base + sk * C::KV_BYTES + kk * 2048, C::BN * 128, 1024), idQ,
                                (acc || kk > 0) ? 1u : 0u);
            };
            auto start_s = [&](int j) {
                wait_bounded(&bar_kf[j % C::KST], (j / C::KST) & 1, g);
                ptx::tc_fence_after();
                issue_s(j % C::KST, j & 1);
                ptx::mma_commit(&bar_s_full[j & 1]);
            };
            auto start_dp = [&](int j) {
                wait_bounded(&bar_vf[j % C::VST], (j / C::VST) & 1, g);
                ptx::tc_fence_after();
                issue_dp(j % C::VST);
                ptx::mma_commit(&bar_dp_full);
                ptx::mma_commit(&bar_ve[j % C::VST]);
            };
            wait_bounded(&bar_q, 0, g);
            if (nk > 0) {
                start_s(0);
                start_dp(0);
            }
            if (nk > 1) start_s(1);
            for (int j = 0; j < nk; ++j) {
                const int b = j & 1, sk = j % C::KST;
                wait_bounded(&bar_ds_full, j & 1, g);
                ptx::tc_fence_after();
                if (j + 1 < nk) start_dp(j + 1);   // the P / dS warps have read dP_j
                issue_dq(sk, b, j > 0);
                ptx::mma_commit(&bar_ke[sk]);      // K_j: S_j and dQ_j done with it
                if (j + 2 < nk) start_s(j + 2);    // over dS_j, after the dQ product that reads it
            }
            ptx::mma_commit(&bar_dq);
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else {
        // ---------------------------------------------------------------- P / dS warpgroups
        const int h = warp >> 2, cw = warp & 3;
        const int row = q0 + cw * 32 + lane;    // query row = TMEM lane
        const bool row_ok = row < n;
        const uint32_t lane_off = (uint32_t)(cw * 32) << 16;
        const float scale_log2 = scale * kLog2e;
        const float *pair = stats + ((size_t)bh * n_pad + (row_ok ? row : 0)) / 2 * 4;
        const float nl2 = row_ok ? pair[row & 1] : -INFINITY;   // -LSE2
        const float nd = row_ok ? pair[2 + (row & 1)] : 0.f;    // -D
        const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2), nl22 = ptx::f2_pack(nl2, nl2),
                       nd2 = ptx::f2_pack(nd, nd);
        for (int j = 0; j < nk; ++j) {
            const int b = j & 1;
            const int valid = n - j * C::BN - h * 64;   // keys of this warpgroup below n
            const uint32_t tS = tmem + lane_off + C::tm_s(b) + h * 64, tDP = tmem + lane_off + C::TM_DP + h * 64;
            wait_bounded(&bar_s_full[b], (j >> 1) & 1, g);
            ptx::tc_fence_after();
            // phase 1, as soon as S_j is in: P for this warpgroup's 64 keys (fp32 kept)
            float pf[64];
#pragma unroll
            for (int c = 0; c < 64; c += 32) {
                uint32_t sv[32];
                ptx::tmem_ld32(tS + c, sv);
                ptx::tmem_ld_wait();
                reg_fence(sv);
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const uint64_t x = ptx::fma_f32x2(ptx::f2_pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2, nl22);
                    float x0, x1;
                    ptx::f2_unpack(x, x0, x1);
                    pf[c + i] = c + i < valid ? ptx::ex2(x0) : 0.f;
                    pf[c + i + 1] = c + i + 1 < valid ? ptx::ex2(x1) : 0.f;
                }
            }
            // phase 2, once dP_j is in: dS = P o (dP - D), bf16 over this warpgroup's S columns
            // (read in phase 1): keys [64h + c, +32) -> columns 64h + c / 2 + [0, 16)
            wait_bounded(&bar_dp_full, j & 1, g);
            ptx::tc_fence_after();
#pragma unroll
            for (int c = 0; c < 64; c += 32) {
                uint32_t dpv[32];
                ptx::tmem_ld32(tDP + c, dpv);
                ptx::tmem_ld_wait();
                reg_fence(dpv);
                uint32_t dsp[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const uint64_t dsq = ptx::mul_f32x2(
                        ptx::f2_pack(pf[c + i], pf[c + i + 1]),
                        ptx::add_f32x2(ptx::f2_pack(__uint_as_float(dpv[i]), __uint_as_float(dpv[i + 1])), nd2));
                    float ds0, ds1;
                    ptx::f2_unpack(dsq, ds0, ds1);
                    dsp[i / 2] = ptx::pack_bf16x2(ds0, ds1);
                }
                ptx::tmem_st16(tS + c / 2, dsp);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_ds_full);
        }
        // epilogue: dQ = scale * acc in bf16; warpgroup h writes columns [h*D/2, (h+1)*D/2)
        wait_bounded(&bar_dq, 0, g);
        ptx::tc_fence_after();
        __nv_bfloat16 *dst_row = dq + ((size_t)bh * n + (row_ok ? row : 0)) * D;
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) {
            const int col = h * (D / 2) + c;
            uint32_t v[32];
            ptx::tmem_ld32(tmem + lane_off + C::TM_DQ + col, v);
            ptx::tmem_ld_wait();
            reg_fence(v);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]) * scale, __uint_as_float(v[2 * e + 1]) * scale);
            if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(dst_row + col);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

int elementwise_blocks() { return 4 * device_sm_count(); }

template <int D>
cudaError_t launch_preprocess_d(const BwdArgs &a, bool zero_acc, cudaStream_t stream)
{
    bwd_preprocess_kernel<D><<<elementwise_blocks(), 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16 *>(a.o), reinterpret_cast<const __nv_bfloat16 *>(a.dout),
        a.lse, a.stats, a.dq_acc, a.bh, a.n, a.n_pad, zero_acc ? 1 : 0);
    return cudaGetLastError();
}

template <int D, bool WITH_DQ>
cudaError_t launch_main_d(const BwdArgs &a, cudaStream_t stream)
{
    using C = BwdCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D, WITH_DQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_kvblocks = (a.n + C::BN - 1) / C::BN;
    const long long ctas = (long long)n_kvblocks * a.bh;
    bwd_main_kernel<D, WITH_DQ><<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.stats, a.dq_acc,
        reinterpret_cast<__nv_bfloat16 *>(a.dk), reinterpret_cast<__nv_bfloat16 *>(a.dv), a.n,
        a.n_pad, n_kvblocks, a.scale, a.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs &a, cudaStream_t stream)
{
    return a.d == 64 ? launch_preprocess_d<64>(a, true, stream) : launch_preprocess_d<128>(a, true, stream);
}

template <bool WITH_DQ>
cudaError_t launch_main_wide(const BwdArgs &a, cudaStream_t stream)
{
    using C = WideCfg;
    cudaError_t e = cudaFuncSetAttribute(bwd_main_wide_kernel<WITH_DQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_kvblocks = (a.n + C::BN - 1) / C::BN;
    const long long ctas = (long long)n_kvblocks * a.bh;
    bwd_main_wide_kernel<WITH_DQ><<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dk, a.tm_dv, a.stats, a.dq_acc, a.n, a.n_pad, n_kvblocks,
        a.scale, a.status);
    return cudaGetLastError();
}


template <bool WITH_DQ>
cudaError_t launch_main_persist(const BwdArgs &a, cudaStream_t stream)
{
    using C = PersistBwdCfg;
    cudaError_t e = cudaFuncSetAttribute(bwd_main_persist_kernel<WITH_DQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_kvblocks = (a.n + C::BN - 1) / C::BN;
    const long long items = (long long)n_kvblocks * a.bh;
    const long long ctas = std::min<long long>(items, device_sm_count());
    bwd_main_persist_kernel<WITH_DQ><<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dk, a.tm_dv, a.stats, a.dq_acc, a.n, a.n_pad, n_kvblocks,
        (int)items, a.scale, a.status);
    return cudaGetLastError();
}

// d = 64 main kernel: the persistent variant where each key block has only a few query tiles.
template <bool WITH_DQ>
cudaError_t launch_main_d64(const BwdArgs &a, cudaStream_t stream)
{
    const int nq = (a.n + 127) / 128;
    if (nq >= 2 && a.n <= kBwdPersistentMaxN) return launch_main_persist<WITH_DQ>(a, stream);
    return launch_main_wide<WITH_DQ>(a, stream);
}

cudaError_t launch_dkdv_d128(const BwdArgs &a, cudaStream_t stream)
{
    using C = D128Cfg;
    cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_kvblocks = (a.n + C::BN - 1) / C::BN;
    const long long ctas = (long long)n_kvblocks * a.bh;
    bwd_dkdv_d128_kernel<<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dk, a.tm_dv, a.stats, a.n, a.n_pad, n_kvblocks, a.scale,
        a.status);
    return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdArgs &a, cudaStream_t stream)
{
    return a.d == 64 ? launch_main_d64<true>(a, stream) : launch_main_d<128, true>(a, stream);
}

template <int D>
cudaError_t launch_dq_d(const BwdArgs &a, cudaStream_t stream)
{
    using C = DqCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_qblocks = (a.n + C::BM - 1) / C::BM;
    const long long ctas = (long long)n_qblocks * a.bh;
    bwd_dq_kernel<D><<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.stats,
        reinterpret_cast<__nv_bfloat16 *>(a.dq), a.n, a.n_pad, n_qblocks, a.scale, a.status);
    return cudaGetLastError();
}

cudaError_t launch_bwd_deterministic(const BwdArgs &a, cudaStream_t stream)
{
    cudaError_t e = a.d == 64 ? launch_preprocess_d<64>(a, false, stream)
                              : launch_preprocess_d<128>(a, false, stream);
    if (e == cudaSuccess)
        e = a.d == 64 ? launch_main_d64<false>(a, stream) : launch_dkdv_d128(a, stream);
    if (e == cudaSuccess) e = a.d == 64 ? launch_dq_d<64>(a, stream) : launch_dq_d<128>(a, stream);
    return e;
}

// Where it measured faster than the three-kernel path: one head per CTA at most (its heads
// run one after another, without the other path's overlap of items), and either one key block
// per head or more heads than half the SMs (with two key blocks the other path runs two CTAs
// per head, which wins while there are few heads).
bool bwd_whole_heads(int n, int d, long long bh)
{
    if (d != 64 || n > 2 * HeadCfg::T) return false;
    const int sms = device_sm_count();
    return bh <= sms && (n <= HeadCfg::T || 2 * bh > sms);
}

cudaError_t launch_bwd_heads(const BwdArgs &a, cudaStream_t stream)
{
    using C = HeadCfg;
    cudaError_t e = cudaFuncSetAttribute(bwd_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long ctas = std::min<long long>(a.bh, device_sm_count());
    bwd_head_kernel<<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_do, reinterpret_cast<const __nv_bfloat16 *>(a.o), a.lse,
        reinterpret_cast<__nv_bfloat16 *>(a.dq), reinterpret_cast<__nv_bfloat16 *>(a.dk),
        reinterpret_cast<__nv_bfloat16 *>(a.dv), a.n, a.bh, a.scale, a.status);
    return cudaGetLastError();
}

cudaError_t launch_bwd_convert(const BwdArgs &a, cudaStream_t stream)
{
    bwd_convert_dq_kernel<<<elementwise_blocks(), 256, 0, stream>>>(
        a.dq_acc, reinterpret_cast<__nv_bfloat16 *>(a.dq), a.scale, (long long)a.bh * a.n * a.d / 8);
    return cudaGetLastError();
}

}  // namespace attn
