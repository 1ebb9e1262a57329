// Forward pass of exact multi-head attention, O = softmax(scale * Q K^T) V, plus the per-row
// log-sum-exp of the scaled scores, for sm_103a.
//
// "Self-attention, CUDA kernels and FlashAttention", section 1 defines the result (the
// "Scores" formula with the division by sqrt(d_k), the row softmax, Attention(Q,K,V) and
// independent heads).  Section 3 describes how to reach it without ever writing the N x N
// score matrix to HBM: Q, K and V are cut into blocks that fit on chip ("Tiling"), and the
// softmax runs online, keeping a running maximum and normaliser per row and rescaling the
// partial output when a new block raises the maximum ("The online softmax trick").  The
// per-row statistic the backward pass needs ("Recomputation in backpropagation") is stored
// as LSE = log sum_j exp(scale * q_i . k_j).
//
// Blackwell mapping of fwd_kernel<D, NQ> (one CTA = NQ query tiles of 128 rows of one head;
// used for d = 128 with NQ = 2, shown here.  d = 64, where the softmax work per tile equals the
// matrix work, runs one tile per CTA and two CTAs per SM: fwd_persistent_kernel, or
// fwd_sp_kernel where there are fewer tiles than resident CTAs, below):
//   warp 8      TMA producer: Q tiles once, then a ring of K tiles and a ring of V tiles (128
//               keys each).
//   warps 10-11 V converters: each V tile rewritten as fp16 in shared memory once it has landed
//               (or, where V was rounded to fp16 ahead of the kernel by v_to_f16_kernel, passed
//               on as it landed: v_f16).
//   warp 9      tcgen05 issuer: S_t = Q_t K_j^T into TMEM (fp32), then O_t += P_t V_j with
//               P_t read from TMEM (fp16, written over S_t) and V_j (fp16) from shared memory.
//   warps 0-7   two softmax warpgroups, one per query tile; thread = one query row.  They
//               read S_t from TMEM, update the running max m (log2 units, scale folded into
//               log2 e) and sum l, write P_t = 2^(x - m) as fp16 back into TMEM and rescale
//               O_t in TMEM when the maximum grew by more than kTau (exact: the final
//               division uses the same m).  The two tiles alternate on the tensor core, so
//               one tile's softmax overlaps the other tile's matrix products.
// P V runs in fp16 rather than bf16 (the two operands of one MMA share their type): an fp16
// weight is off by at most 2^-11 of itself where a bf16 one is off by 2^-8, and V's bf16 values
// are exact in fp16 across fp16's normal range.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [256+d,256+2d).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running maximum is only moved (and O rescaled) when a tile raises it by more than this
// many powers of two; in between, probabilities may reach 2^kTau, far from fp32/bf16 limits.
constexpr float kTau = 8.0f;
// P = 2^(x - m + kPOff) enters P V as fp16: with the maximum lagging by at most kTau the
// largest weight is 2^(kTau + kPOff) = 2^15, inside fp16's range, and the offset keeps weights
// down to 2^-31 of the row maximum out of fp16's flush-to-zero.  The row sum l adds the weights
// in fp32 before they are rounded; the offset cancels in O = acc / l, and LSE subtracts it.
constexpr float kPOff = 7.0f;

// Rewrites a shared tile of bf16 pairs as fp16 pairs, in place, 16 bytes at a time (the tile's
// swizzle permutes whole 16-byte chunks, so it is untouched): the NT calling threads take chunks
// ct, ct + NT, ... of the CHUNKS at `base`, PASS chunks per thread at a time with all of a pass's
// loads issued before its stores.  Rounding bf16 to fp16 is exact for magnitudes in fp16's
// normal range [2^-14, 65504]; smaller ones round to fp16's subnormal grid of 2^-24, larger ones
// become infinite.
template <int CHUNKS, int NT, int PASS>
__device__ __forceinline__ void tile_bf16_to_f16(uint32_t base, int ct)
{
    constexpr int PER_THREAD = CHUNKS / NT;
    static_assert(CHUNKS % NT == 0 && PER_THREAD % PASS == 0, "whole passes");
#pragma unroll 1
    for (int p = 0; p < PER_THREAD / PASS; ++p) {
        uint4 v[PASS];
#pragma unroll
        for (int k = 0; k < PASS; ++k) v[k] = lds_u128(base + (uint32_t)(ct + NT * (PASS * p + k)) * 16u);
#pragma unroll
        for (int k = 0; k < PASS; ++k)
            sts_u128(base + (uint32_t)(ct + NT * (PASS * p + k)) * 16u,
                     make_uint4(ptx::bf16x2_to_f16x2(v[k].x), ptx::bf16x2_to_f16x2(v[k].y),
                                ptx::bf16x2_to_f16x2(v[k].z), ptx::bf16x2_to_f16x2(v[k].w)));
    }
}

// Diagnostic output: 32 consecutive columns of a row of O before its bf16 rounding (acc / l
// in fp32), as attn_fwd_diagnostic returns them.
__device__ __forceinline__ void store_o32(float *dst, const uint32_t (&ov)[32], float inv_l)
{
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int v4 = 0; v4 < 8; ++v4)
        d4[v4] = make_float4(__uint_as_float(ov[4 * v4]) * inv_l, __uint_as_float(ov[4 * v4 + 1]) * inv_l,
                             __uint_as_float(ov[4 * v4 + 2]) * inv_l, __uint_as_float(ov[4 * v4 + 3]) * inv_l);
}

template <int D, int NQ_>
struct FwdCfg {
    static constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
    static constexpr int NQ = NQ_;  // query tiles per CTA
    static constexpr int BN = 128;  // keys per K/V tile
    // One tile per CTA (short sequences) keeps shared memory and TMEM small enough for two
    // CTAs per SM, which then hide each other's load and epilogue latency.
    static constexpr int STAGES = NQ == 1 ? 2 : (D == 64) ? 4 : 2;   // K ring
    // V ring: one stage deeper than the K ring, so that each V tile has landed, and has been
    // rewritten as fp16, well before its P V
    static constexpr int VSTAGES = STAGES + 1;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int SMEM_BYTES = NQ * Q_BYTES + (STAGES + VSTAGES) * KV_BYTES + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024 - 512, "dynamic + static shared memory over 227 KB");
    static constexpr int TMA_WARP = 4 * NQ, MMA_WARP = 4 * NQ + 1, CONV_WARP = 4 * NQ + 2;
    static constexpr int CONV_THREADS = 64, CONV_PASS = 16;   // 16 loads in flight per thread
    static constexpr int THREADS = 32 * (4 * NQ + 4);
    static constexpr uint32_t TM_O = NQ * 128;  // first O column
    static constexpr uint32_t TM_COLS = NQ == 1 ? 256 : 512;
    static constexpr int MIN_BLOCKS = NQ == 1 ? 2 : 1;
};

template <int D, int NQ>
__global__ void __launch_bounds__(FwdCfg<D, NQ>::THREADS, FwdCfg<D, NQ>::MIN_BLOCKS)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ o,
               float *__restrict__ lse, float *__restrict__ o32, int n, int n_qblocks, float scale_log2,
               int v_f16, int *status)
{
    using C = FwdCfg<D, NQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + C::NQ * C::Q_BYTES;
    uint8_t *sV = sK + C::STAGES * C::KV_BYTES;

    __shared__ uint64_t bar_q;
    __shared__ uint64_t bar_kf[C::STAGES], bar_ke[C::STAGES];
    __shared__ uint64_t bar_vf[C::VSTAGES], bar_ve[C::VSTAGES], bar_vc[C::VSTAGES];   // vc: V as fp16
    __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2], bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / n_qblocks;
    const int q0 = (blockIdx.x % n_qblocks) * (C::NQ * C::BM);
    const int nkv = (n + C::BN - 1) / C::BN;
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        ptx::mbar_init(&bar_q, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(&bar_kf[s], 1);
            ptx::mbar_init(&bar_ke[s], 1);
        }
        for (int s = 0; s < C::VSTAGES; ++s) {
            ptx::mbar_init(&bar_vf[s], 1);
            ptx::mbar_init(&bar_ve[s], 1);
            ptx::mbar_init(&bar_vc[s], C::CONV_THREADS);
        }
        for (int t = 0; t < C::NQ; ++t) {
            ptx::mbar_init(&bar_s[t], 1);
            ptx::mbar_init(&bar_p[t], 128);
            ptx::mbar_init(&bar_o[t], 1);
        }
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(&tmem_sh, C::TM_COLS);
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
            ptx::mbar_arrive_expect_tx(&bar_q, C::NQ * C::Q_BYTES);
            for (int t = 0; t < C::NQ; ++t)
                for (int h = 0; h < D / 64; ++h)
                    ptx::tma_load_3d(sQ + t * C::Q_BYTES + h * C::BM * 128, &tm_q, &bar_q, h * 64,
                                     q0 + t * C::BM, bh);
            for (int j = 0; j < nkv; ++j) {
                const int s = j % C::STAGES;
                const uint32_t ph = (j / C::STAGES) & 1;
                wait_bounded(&bar_ke[s], ph ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_kf[s], C::KV_BYTES);
                for (int h = 0; h < D / 64; ++h)
                    ptx::tma_load_3d(sK + s * C::KV_BYTES + h * C::BN * 128, &tm_k, &bar_kf[s],
                                     h * 64, j * C::BN, bh);
                const int sv = j % C::VSTAGES;
                wait_bounded(&bar_ve[sv], ((j / C::VSTAGES) & 1) ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_vf[sv], C::KV_BYTES);
                for (int h = 0; h < D / 64; ++h)
                    ptx::tma_load_3d(sV + sv * C::KV_BYTES + h * C::BN * 128, &tm_v, &bar_vf[sv],
                                     h * 64, j * C::BN, bh);
            }
            // Do not leave the CTA with copies in flight (matters only after a timeout).
            for (int j = (nkv > C::STAGES ? nkv - C::STAGES : 0); j < nkv; ++j)
                wait_bounded(&bar_kf[j % C::STAGES], (j / C::STAGES) & 1, g);
            for (int j = (nkv > C::VSTAGES ? nkv - C::VSTAGES : 0); j < nkv; ++j)
                wait_bounded(&bar_vf[j % C::VSTAGES], (j / C::VSTAGES) & 1, g);
        }
    } else if (warp == C::MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idS = ptx::idesc_bf16_f32(128, C::BN, false, false);
            const uint32_t idO = ptx::idesc_f16_f32(128, D, false, true);
            const uint32_t q_base = ptx::smem_u32(sQ), k_base = ptx::smem_u32(sK),
                           v_base = ptx::smem_u32(sV);
            // S_t = Q_t K^T: both operands K-major (d contiguous), 64-column halves for d=128.
            auto issue_s = [&](int t, int s) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
                    const uint64_t a = ptx::sdesc_sw128(q_base + t * C::Q_BYTES + off, 16, 1024);
                    const uint64_t b = ptx::sdesc_sw128(k_base + s * C::KV_BYTES + off, 16, 1024);
                    ptx::mma_ss(tmem + t * 128, a, b, idS, kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V: fp16 P from TMEM (8 columns = 16 keys per step), fp16 V MN-major (d
            // contiguous).
            auto issue_pv = [&](int t, int sv, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    const uint64_t b =
                        ptx::sdesc_sw128(v_base + sv * C::KV_BYTES + kk * 2048, C::BN * 128, 1024);
                    ptx::mma_ts(tmem + C::TM_O + t * D, tmem + t * 128 + kk * 8, b, idO,
                                (acc || kk > 0) ? 1u : 0u);
                }
            };
            wait_bounded(&bar_q, 0, g);
            wait_bounded(&bar_kf[0], 0, g);
            ptx::tc_fence_after();
#pragma unroll
            for (int t = 0; t < C::NQ; ++t) {
                issue_s(t, 0);
                ptx::mma_commit(&bar_s[t]);
            }
            ptx::mma_commit(&bar_ke[0]);
            // Per key tile j and query tile t: O_t += P_t V_j as soon as P_t is in TMEM, then
            // S_t of tile j + 1 into the same columns (the MMAs run in issue order, so P_t has
            // been read by then).  With two query tiles, one tile's products overlap the
            // other tile's softmax.
            for (int j = 0; j < nkv; ++j) {
                const int s = j % C::STAGES;
                const uint32_t ph = (j / C::STAGES) & 1;
                const int jn = j + 1;
                const int sn = jn % C::STAGES;
                const uint32_t phn = (jn / C::STAGES) & 1;
                const int sv = j % C::VSTAGES;
                wait_bounded(&bar_vc[sv], (j / C::VSTAGES) & 1, g);
#pragma unroll
                for (int t = 0; t < C::NQ; ++t) {
                    wait_bounded(&bar_p[t], j & 1, g);
                    ptx::tc_fence_after();
                    issue_pv(t, sv, j > 0);
                    if (t == C::NQ - 1) ptx::mma_commit(&bar_ve[sv]);
                    if (jn < nkv) {
                        if (t == 0) {
                            wait_bounded(&bar_kf[sn], phn, g);
                            ptx::tc_fence_after();
                        }
                        issue_s(t, sn);
                        ptx::mma_commit(&bar_s[t]);
                        if (t == C::NQ - 1) ptx::mma_commit(&bar_ke[sn]);
                    } else {
                        ptx::mma_commit(&bar_o[t]);
                    }
                }
            }
            // Every MMA must have finished before TMEM is released (matters after a timeout).
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else if (warp >= C::CONV_WARP) {
        // ---------------------------------------------------------------- V to fp16
        // each V tile rewritten as fp16 in place as soon as it has landed (passed on unchanged
        // when V is fp16 already)
        const int ct = (warp - C::CONV_WARP) * 32 + lane;
        for (int j = 0; j < nkv; ++j) {
            const int sv = j % C::VSTAGES;
            wait_bounded(&bar_vf[sv], (j / C::VSTAGES) & 1, g);
            if (!v_f16)
                tile_bf16_to_f16<C::KV_BYTES / 16, C::CONV_THREADS, C::CONV_PASS>(ptx::smem_u32(sV + sv * C::KV_BYTES), ct);
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bar_vc[sv]);
        }
    } else {
        // ---------------------------------------------------------------- softmax warpgroups
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int row = q0 + t * C::BM + quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + C::TM_O + t * D;
        float m = -INFINITY, l = 0.f;

        for (int j = 0; j < nkv; ++j) {
            wait_bounded(&bar_s[t], j & 1, g);
            ptx::tc_fence_after();
            uint32_t r[128];
            ptx::tmem_ld32_at<0>(tS + 0, r);
            ptx::tmem_ld32_at<32>(tS + 32, r);
            ptx::tmem_ld32_at<64>(tS + 64, r);
            ptx::tmem_ld32_at<96>(tS + 96, r);
            ptx::tmem_ld_wait();
            reg_fence(r);
            // keys >= n (only in the last tile) take no weight
            const int valid = n - j * C::BN;
            if (valid < C::BN) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= valid) r[i] = __float_as_uint(-INFINITY);
            }
            float mx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(r[u]);
#pragma unroll
            for (int i = 8; i < 128; i += 2)
                mx[(i >> 1) & 7] = ptx::max3(mx[(i >> 1) & 7], __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
            const float smax = ptx::max3(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], mx[5]),
                                         fmaxf(mx[6], mx[7]));
            const float mt = smax * scale_log2;
            float m_new = m, alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_new = mt;
            } else if (__any_sync(0xffffffffu, mt > m + kTau)) {
                m_new = fmaxf(m, mt);
                alpha = ptx::ex2(m - m_new);
                rescale = true;
            }
            const float neg_m = kPOff - m_new;
            // x c - m + kPOff for two scores per instruction (f32x2), 2^(.) on the MUFU, the row
            // sum two lanes at a time in fp32, then the weights rounded to fp16 pairs for P V
            const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2), nm2 = ptx::f2_pack(neg_m, neg_m);
            uint64_t sum2[2] = {ptx::f2_pack(0.f, 0.f), ptx::f2_pack(0.f, 0.f)};
            // P as fp16 pairs into TMEM over S_t, 32 keys (16 columns) at a time
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const uint64_t t = ptx::fma_f32x2(
                        ptx::f2_pack(__uint_as_float(r[ch * 32 + i]), __uint_as_float(r[ch * 32 + i + 1])), c2, nm2);
                    float t0, t1;
                    ptx::f2_unpack(t, t0, t1);
                    const float p0 = ptx::ex2(t0), p1 = ptx::ex2(t1);
                    sum2[(i >> 1) & 1] = ptx::add_f32x2(sum2[(i >> 1) & 1], ptx::f2_pack(p0, p1));
                    const uint32_t h = ptx::pack_f16x2(p0, p1);
                    pk[i >> 1] = h;
                }
                ptx::tmem_st16(tS + ch * 16, pk);
            }
            float sum[4];
            ptx::f2_unpack(sum2[0], sum[0], sum[1]);
            ptx::f2_unpack(sum2[1], sum[2], sum[3]);
            l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
            m = m_new;
            if (rescale) {
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t ov[32];
                    ptx::tmem_ld32(tO + c, ov);
                    ptx::tmem_ld_wait();
                    reg_fence(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    ptx::tmem_st32(tO + c, ov);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_p[t]);
        }

        // epilogue: O = O_acc / l (bf16), LSE = (m - kPOff + log2 l) ln 2
        wait_bounded(&bar_o[t], 0, g);
        ptx::tc_fence_after();
        const float inv_l = 1.f / l;
        __nv_bfloat16 *orow = o + ((size_t)bh * n + (row < n ? row : 0)) * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            ptx::tmem_ld32(tO + c, ov);
            ptx::tmem_ld_wait();
            reg_fence(ov);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = ptx::pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                                         __uint_as_float(ov[2 * i + 1]) * inv_l);
            if (o32 && row < n) store_o32(o32 + ((size_t)bh * n + row) * D + c, ov, inv_l);
            if (row < n) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
        }
        if (row < n) lse[(size_t)bh * n + row] = (m - kPOff + log2f(l)) * kLn2;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}

// fwd_sp_kernel: d = 64, one 128-row query tile per CTA, two CTAs per SM, with P in TMEM
// columns of its own instead of over S.  S of key tile j + 1 is then issued as soon as the
// softmax warps have read S_j out of TMEM, and runs under their exponentials; only P_j (and a
// rescale of O) waits for the P V product of tile j - 1.
//   warp 4      TMA producer: Q once, then a ring of K and V tiles.
//   warp 5      tcgen05 issuer: S_{j+1} = Q K_{j+1}^T once S_j has been read, O += P_j V_j once
//               P_j is in.
//   warps 6-7   V converters: each V tile rewritten as fp16 in shared memory once it has
//               landed (the other operand of P V), off the softmax warps' path.
//   warps 0-3   softmax, thread = query row: read S_j, running max and sum as fwd_kernel, P_j
//               (fp16) into the P columns once P V of tile j - 1 is done with them; at the end
//               O / l through the idle Q tile to global memory by one TMA tensor store.
// TMEM columns: S [0,128), O [128,192), P [192,256).
struct FwdSpCfg {
    static constexpr int D = 64;
    static constexpr int BM = 128, BN = 128;
    static constexpr int STAGES = 2;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int SMEM_BYTES = Q_BYTES + 2 * STAGES * KV_BYTES + 1024;
    static constexpr int THREADS = 256;
    static constexpr int TMA_WARP = 4, MMA_WARP = 5, CONV_WARP = 6, CONV_THREADS = 64;
    static constexpr int CONV_PASS = 8;   // 8 loads in flight per thread within 80 registers
    // two CTAs per SM launch with 128 registers a thread: softmax warpgroup 176, the other 80
    static constexpr uint32_t REG_SOFTMAX = 176, REG_OTHER = 80;
    static constexpr uint32_t TM_O = 128, TM_P = 192, TM_COLS = 256;
};

__global__ void __launch_bounds__(256, 2)
    fwd_sp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  float *__restrict__ lse, float *__restrict__ o32, int n, int n_qblocks, float scale_log2,
                  int v_f16, int *status)
{
    using C = FwdSpCfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + C::Q_BYTES;
    uint8_t *sV = sK + C::STAGES * C::KV_BYTES;

    __shared__ uint64_t bar_q;
    __shared__ uint64_t bar_kf[C::STAGES], bar_ke[C::STAGES], bar_vf[C::STAGES], bar_ve[C::STAGES];
    __shared__ uint64_t bar_vc[C::STAGES];   // V tile rewritten as fp16
    __shared__ uint64_t bar_s, bar_sread, bar_p, bar_pv, bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / n_qblocks;
    const int q0 = (blockIdx.x % n_qblocks) * C::BM;
    const int nkv = (n + C::BN - 1) / C::BN;
    const Guard g{&abort_sh, status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        ptx::mbar_init(&bar_q, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(&bar_kf[s], 1);
            ptx::mbar_init(&bar_ke[s], 1);
            ptx::mbar_init(&bar_vf[s], 1);
            ptx::mbar_init(&bar_ve[s], 1);
            ptx::mbar_init(&bar_vc[s], C::CONV_THREADS);
        }
        ptx::mbar_init(&bar_s, 1);
        ptx::mbar_init(&bar_sread, 128);
        ptx::mbar_init(&bar_p, 128);
        ptx::mbar_init(&bar_pv, 1);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(&tmem_sh, C::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    // The register split is taken inside each warpgroup's branch, so that the code of each role
    // is compiled to its own budget.
    if (warp >= 4) {
    ptx::setmaxnreg_dec<C::REG_OTHER>();
    if (warp == C::TMA_WARP) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::mbar_arrive_expect_tx(&bar_q, C::Q_BYTES);
            ptx::tma_load_3d(sQ, &tm_q, &bar_q, 0, q0, bh);
            for (int j = 0; j < nkv; ++j) {
                const int s = j % C::STAGES;
                const uint32_t ph = (j / C::STAGES) & 1;
                wait_bounded(&bar_ke[s], ph ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_kf[s], C::KV_BYTES);
                ptx::tma_load_3d(sK + s * C::KV_BYTES, &tm_k, &bar_kf[s], 0, j * C::BN, bh);
                wait_bounded(&bar_ve[s], ph ^ 1, g);
                ptx::mbar_arrive_expect_tx(&bar_vf[s], C::KV_BYTES);
                ptx::tma_load_3d(sV + s * C::KV_BYTES, &tm_v, &bar_vf[s], 0, j * C::BN, bh);
            }
            // Do not leave the CTA with copies in flight (matters only after a timeout).
            wait_bounded(&bar_q, 0, g);
            for (int j = (nkv > C::STAGES ? nkv - C::STAGES : 0); j < nkv; ++j) {
                wait_bounded(&bar_kf[j % C::STAGES], (j / C::STAGES) & 1, g);
                wait_bounded(&bar_vf[j % C::STAGES], (j / C::STAGES) & 1, g);
            }
        }
    } else if (warp == C::MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idS = ptx::idesc_bf16_f32(128, C::BN, false, false);
            const uint32_t idO = ptx::idesc_f16_f32(128, D, false, true);
            const uint32_t q_base = ptx::smem_u32(sQ), k_base = ptx::smem_u32(sK),
                           v_base = ptx::smem_u32(sV);
            // S = Q K_j^T: both operands K-major (d contiguous).
            auto issue_s = [&](int s) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem, ptx::sdesc_sw128(q_base + kk * 32, 16, 1024),
                                ptx::sdesc_sw128(k_base + s * C::KV_BYTES + kk * 32, 16, 1024), idS,
                                kk > 0 ? 1u : 0u);
            };
            // O += P V_j: fp16 P from its TMEM columns (8 columns = 16 keys per step), fp16 V
            // MN-major.
            auto issue_pv = [&](int s, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    ptx::mma_ts(tmem + C::TM_O, tmem + C::TM_P + kk * 8,
                                ptx::sdesc_sw128(v_base + s * C::KV_BYTES + kk * 2048, C::BN * 128, 1024), idO,
                                (acc || kk > 0) ? 1u : 0u);
            };
            wait_bounded(&bar_q, 0, g);
            wait_bounded(&bar_kf[0], 0, g);
            ptx::tc_fence_after();
            issue_s(0);
            ptx::mma_commit(&bar_s);
            ptx::mma_commit(&bar_ke[0]);
            for (int j = 0; j < nkv; ++j) {
                const int s = j % C::STAGES;
                if (j + 1 < nkv) {   // S_{j+1} over S_j once the softmax has read it
                    const int sn = (j + 1) % C::STAGES;
                    wait_bounded(&bar_sread, j & 1, g);
                    wait_bounded(&bar_kf[sn], ((j + 1) / C::STAGES) & 1, g);
                    ptx::tc_fence_after();
                    issue_s(sn);
                    ptx::mma_commit(&bar_s);
                    ptx::mma_commit(&bar_ke[sn]);
                }
                wait_bounded(&bar_vc[s], (j / C::STAGES) & 1, g);
                wait_bounded(&bar_p, j & 1, g);
                ptx::tc_fence_after();
                issue_pv(s, j > 0);
                ptx::mma_commit(&bar_pv);   // P and O free again; after the last tile: O final
                ptx::mma_commit(&bar_ve[s]);
            }
            // Every MMA must have finished before TMEM is released (matters after a timeout).
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else {
        // ---------------------------------------------------------------- V to fp16
        // each V tile rewritten as fp16 in place as soon as it has landed (passed on unchanged
        // when V is fp16 already)
        const int ct = (warp - C::CONV_WARP) * 32 + lane;
        for (int j = 0; j < nkv; ++j) {
            const int sv = j % C::STAGES;
            wait_bounded(&bar_vf[sv], (j / C::STAGES) & 1, g);
            if (!v_f16)
                tile_bf16_to_f16<C::KV_BYTES / 16, C::CONV_THREADS, C::CONV_PASS>(ptx::smem_u32(sV + sv * C::KV_BYTES), ct);
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bar_vc[sv]);
        }
    }
    } else {
        ptx::setmaxnreg_inc<C::REG_SOFTMAX>();
        // ---------------------------------------------------------------- softmax warpgroup
        const int r_local = warp * 32 + lane;   // row of the tile = TMEM lane
        const int row = q0 + r_local;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t tS = tmem + lane_off, tO = tmem + lane_off + C::TM_O, tP = tmem + lane_off + C::TM_P;
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < nkv; ++j) {
            wait_bounded(&bar_s, j & 1, g);
            ptx::tc_fence_after();
            uint32_t r[128];
            ptx::tmem_ld32_at<0>(tS + 0, r);
            ptx::tmem_ld32_at<32>(tS + 32, r);
            ptx::tmem_ld32_at<64>(tS + 64, r);
            ptx::tmem_ld32_at<96>(tS + 96, r);
            ptx::tmem_ld_wait();
            reg_fence(r);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_sread);   // S may take the next tile's product
            // keys >= n (only in the last tile) take no weight
            const int valid = n - j * C::BN;
            if (valid < C::BN) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= valid) r[i] = __float_as_uint(-INFINITY);
            }
            float mx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(r[u]);
#pragma unroll
            for (int i = 8; i < 128; i += 2)
                mx[(i >> 1) & 7] = ptx::max3(mx[(i >> 1) & 7], __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
            const float smax = ptx::max3(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], mx[5]),
                                         fmaxf(mx[6], mx[7]));
            const float mt = smax * scale_log2;
            float m_new = m, alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_new = mt;
            } else if (__any_sync(0xffffffffu, mt > m + kTau)) {
                m_new = fmaxf(m, mt);
                alpha = ptx::ex2(m - m_new);
                rescale = true;
            }
            const float neg_m = kPOff - m_new;
            const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2), nm2 = ptx::f2_pack(neg_m, neg_m);
            uint64_t sum2[2] = {ptx::f2_pack(0.f, 0.f), ptx::f2_pack(0.f, 0.f)};
            // P = 2^(x - m + kPOff) as fp16 pairs, packed into r[0, 64) (each pair lands at or
            // below the slots it was computed from)
#pragma unroll
            for (int i = 0; i < 128; i += 2) {
                const uint64_t t = ptx::fma_f32x2(ptx::f2_pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2, nm2);
                float t0, t1;
                ptx::f2_unpack(t, t0, t1);
                const float p0 = ptx::ex2(t0), p1 = ptx::ex2(t1);
                sum2[(i >> 1) & 1] = ptx::add_f32x2(sum2[(i >> 1) & 1], ptx::f2_pack(p0, p1));
                const uint32_t h = ptx::pack_f16x2(p0, p1);
                r[i >> 1] = h;
            }
            float sum[4];
            ptx::f2_unpack(sum2[0], sum[0], sum[1]);
            ptx::f2_unpack(sum2[1], sum[2], sum[3]);
            l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
            m = m_new;
            // P of tile j - 1 has been multiplied into O: its columns and O are ours again
            if (j > 0) wait_bounded(&bar_pv, (j - 1) & 1, g);
            ptx::tc_fence_after();
            if (rescale) {
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t ov[32];
                    ptx::tmem_ld32(tO + c, ov);
                    ptx::tmem_ld_wait();
                    reg_fence(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    ptx::tmem_st32(tO + c, ov);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = r[h * 32 + i];
                ptx::tmem_st32(tP + h * 32, pk);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_p);
        }

        // epilogue: O = O_acc / l (bf16) into the idle Q tile (128-byte swizzle: 16-byte chunk c
        // of row r at chunk c ^ (r % 8)), one TMA tensor store (rows past N clipped);
        // LSE = (m - kPOff + log2 l) ln 2
        wait_bounded(&bar_pv, (nkv - 1) & 1, g);
        ptx::tc_fence_after();
        const float inv_l = 1.f / l;
        const uint32_t srow = ptx::smem_u32(sQ) + r_local * 128;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            ptx::tmem_ld32(tO + c, ov);
            ptx::tmem_ld_wait();
            reg_fence(ov);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = ptx::pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
            if (o32 && row < n) store_o32(o32 + ((size_t)bh * n + row) * D + c, ov, inv_l);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
                sts_u128(srow + ((((c >> 3) + v4) ^ (r_local & 7)) << 4),
                         make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]));
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar(1, 128);
        if (threadIdx.x == 0) {
            ptx::tma_store_3d(&tm_o, sQ, 0, q0, bh);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group<0>();   // complete before the CTA exits
        }
        if (row < n) lse[(size_t)bh * n + row] = (m - kPOff + log2f(l)) * kLn2;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}

// Persistent variant for d = 64: one query tile per work item, items (head, 128-row block)
// taken in a grid-stride order by CTAs that stay resident (two per SM), so the loads of the
// next item, the tail of the previous one and the other CTA's work hide each other's latency.
//   warp 4      TMA: Q of each item into one of two Q buffers, K/V tiles through one ring that
//               runs across items; before a Q buffer takes its next Q, the O tile that the
//               softmax warps staged there leaves with one TMA tensor store (rows past N clipped).
//   warp 5      tcgen05: S = Q K_j^T, then O += P V_j; as in fwd_sp_kernel the next S, of this
//               item or the next, is issued as soon as the softmax warps have read S, and runs
//               under their exponentials.
//   warps 6-7   V converters: each V tile rewritten as fp16 in shared memory once it has
//               landed (the other operand of P V), off the softmax warps' path.
//   warps 0-3   softmax as fwd_sp_kernel (P in TMEM columns of its own), then the epilogue of
//               the item: the normalised bf16 tile goes into the item's Q buffer (free once the
//               item's last S has read it), in the 128-byte-swizzled layout, for the producer
//               to store.  The next item's first P V (accumulate off) follows the softmax warps'
//               next P, after this epilogue has read O.
// TMEM columns: S [0,128), O [128,128+d), P [128+d,128+d+64).
template <int D>
struct PersistCfg {
    static constexpr int BM = 128, BN = 128;
    static constexpr int STAGES = 2;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int SMEM_BYTES = 2 * Q_BYTES + 2 * STAGES * KV_BYTES + 1024;
    static constexpr int THREADS = 256;
    static constexpr int TMA_WARP = 4, MMA_WARP = 5, CONV_WARP = 6, CONV_THREADS = 64;
    static constexpr int CONV_PASS = 8;   // 8 loads in flight per thread within 80 registers
    // two CTAs per SM launch with 128 registers a thread; the softmax warpgroup takes 176 of
    // them (its code spills at 168), the producer / issuer / converter warpgroup gives back to
    // 80 (128 x 176 + 128 x 80 = 256 x 128)
    static constexpr uint32_t REG_SOFTMAX = 176, REG_OTHER = 80;
    static constexpr uint32_t TM_O = 128, TM_P = 128 + D;
    static constexpr uint32_t TM_COLS = 128 + D + 64 <= 256 ? 256 : 512;
};

template <int D>
__global__ void __launch_bounds__(256, 2)
    fwd_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                          float *__restrict__ lse, float *__restrict__ o32, int n, int n_qblocks, int n_items,
                          float scale_log2, int v_f16, int *status)
{
    using C = PersistCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sQ = smem;                         // two Q buffers
    uint8_t *sK = sQ + 2 * C::Q_BYTES;
    uint8_t *sV = sK + C::STAGES * C::KV_BYTES;

    __shared__ uint64_t bar_qf[2], bar_ost[2];   // Q loaded; O staged in the Q buffer
    __shared__ uint64_t bar_kf[C::STAGES], bar_ke[C::STAGES], bar_vf[C::STAGES], bar_ve[C::STAGES];
    __shared__ uint64_t bar_vc[C::STAGES];   // V tile rewritten as fp16
    __shared__ uint64_t bar_s, bar_sread, bar_p, bar_pv, bar_done;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkv = (n + C::BN - 1) / C::BN;
    const Guard g{&abort_sh, status, kWaitLimitNs};
    const int first = blockIdx.x, stride = gridDim.x;

    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bar_qf[b], 1);
            ptx::mbar_init(&bar_ost[b], 128);
        }
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(&bar_kf[s], 1);
            ptx::mbar_init(&bar_ke[s], 1);
            ptx::mbar_init(&bar_vf[s], 1);
            ptx::mbar_init(&bar_ve[s], 1);
            ptx::mbar_init(&bar_vc[s], C::CONV_THREADS);
        }
        ptx::mbar_init(&bar_s, 1);
        ptx::mbar_init(&bar_sread, 128);
        ptx::mbar_init(&bar_p, 128);
        ptx::mbar_init(&bar_pv, 1);
        ptx::mbar_init(&bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(&tmem_sh, C::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;
    // The register split is taken inside each warpgroup's branch, so that the code of each role
    // is compiled to its own budget.
    if (warp >= 4) {
    ptx::setmaxnreg_dec<C::REG_OTHER>();
    if (warp == C::TMA_WARP) {
        // ---------------------------------------------------------------- TMA producer
        if (ptx::elect_one()) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            // item li - 2's O, staged in Q buffer li % 2, out to global memory
            auto store_o = [&](int li) {
                const int item = first + li * stride;
                const int bh = item / n_qblocks, q0 = (item % n_qblocks) * C::BM;
                const int qb = li & 1;
                wait_bounded(&bar_ost[qb], (li >> 1) & 1, g);
                for (int h = 0; h < D / 64; ++h)
                    ptx::tma_store_3d(&tm_o, sQ + qb * C::Q_BYTES + h * C::BM * 128, h * 64, q0, bh);
                ptx::bulk_commit_group();
            };
            int kt = 0;   // K/V tiles loaded so far (ring position)
            int li = 0;
            for (int item = first; item < n_items; item += stride, ++li) {
                const int bh = item / n_qblocks, q0 = (item % n_qblocks) * C::BM;
                const int qb = li & 1;
                // Q buffer qb held item li - 2's Q, then its O: store that and let it be read
                if (li >= 2) {
                    store_o(li - 2);
                    ptx::bulk_wait_group_read<0>();
                }
                ptx::mbar_arrive_expect_tx(&bar_qf[qb], C::Q_BYTES);
                for (int h = 0; h < D / 64; ++h)
                    ptx::tma_load_3d(sQ + qb * C::Q_BYTES + h * C::BM * 128, &tm_q, &bar_qf[qb],
                                     h * 64, q0, bh);
                for (int j = 0; j < nkv; ++j, ++kt) {
                    const int s = kt % C::STAGES;
                    const uint32_t ph = (kt / C::STAGES) & 1;
                    wait_bounded(&bar_ke[s], ph ^ 1, g);
                    ptx::mbar_arrive_expect_tx(&bar_kf[s], C::KV_BYTES);
                    for (int h = 0; h < D / 64; ++h)
                        ptx::tma_load_3d(sK + s * C::KV_BYTES + h * C::BN * 128, &tm_k, &bar_kf[s],
                                         h * 64, j * C::BN, bh);
                    wait_bounded(&bar_ve[s], ph ^ 1, g);
                    ptx::mbar_arrive_expect_tx(&bar_vf[s], C::KV_BYTES);
                    for (int h = 0; h < D / 64; ++h)
                        ptx::tma_load_3d(sV + s * C::KV_BYTES + h * C::BN * 128, &tm_v, &bar_vf[s],
                                         h * 64, j * C::BN, bh);
                }
            }
            // the last two items' O, then every store complete before the CTA exits
            for (int l2 = (li > 2 ? li - 2 : 0); l2 < li; ++l2) store_o(l2);
            ptx::bulk_wait_group<0>();
            // Do not leave the CTA with copies in flight (matters only after a timeout).
            for (int t = (kt > C::STAGES ? kt - C::STAGES : 0); t < kt; ++t) {
                wait_bounded(&bar_kf[t % C::STAGES], (t / C::STAGES) & 1, g);
                wait_bounded(&bar_vf[t % C::STAGES], (t / C::STAGES) & 1, g);
            }
        }
    } else if (warp == C::MMA_WARP) {
        // ---------------------------------------------------------------- MMA issuer
        if (ptx::elect_one()) {
            const uint32_t idS = ptx::idesc_bf16_f32(128, C::BN, false, false);
            const uint32_t idO = ptx::idesc_f16_f32(128, D, false, true);
            const uint32_t q_base = ptx::smem_u32(sQ), k_base = ptx::smem_u32(sK),
                           v_base = ptx::smem_u32(sV);
            auto issue_s = [&](int qb, int s) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
                    const uint64_t a = ptx::sdesc_sw128(q_base + qb * C::Q_BYTES + off, 16, 1024);
                    const uint64_t b = ptx::sdesc_sw128(k_base + s * C::KV_BYTES + off, 16, 1024);
                    ptx::mma_ss(tmem, a, b, idS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int s, bool acc) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    const uint64_t b =
                        ptx::sdesc_sw128(v_base + s * C::KV_BYTES + kk * 2048, C::BN * 128, 1024);
                    ptx::mma_ts(tmem + C::TM_O, tmem + C::TM_P + kk * 8, b, idO, (acc || kk > 0) ? 1u : 0u);
                }
            };
            // S of global step kt (item li, key tile j)
            auto next_s = [&](int li, int j, int kt) {
                const int s = kt % C::STAGES;
                wait_bounded(&bar_kf[s], (kt / C::STAGES) & 1, g);
                if (j == 0) wait_bounded(&bar_qf[li & 1], (li >> 1) & 1, g);
                ptx::tc_fence_after();
                issue_s(li & 1, s);
                ptx::mma_commit(&bar_s);
                ptx::mma_commit(&bar_ke[s]);
            };
            if (first < n_items) next_s(0, 0, 0);
            int kt = 0, li = 0;
            for (int item = first; item < n_items; item += stride, ++li) {
                for (int j = 0; j < nkv; ++j, ++kt) {
                    const int s = kt % C::STAGES;
                    // the next S, of this item or the next, over S once the softmax has read it
                    if (j + 1 < nkv || item + stride < n_items) {
                        wait_bounded(&bar_sread, kt & 1, g);
                        if (j + 1 < nkv)
                            next_s(li, j + 1, kt + 1);
                        else
                            next_s(li + 1, 0, kt + 1);
                    }
                    wait_bounded(&bar_vc[s], (kt / C::STAGES) & 1, g);
                    wait_bounded(&bar_p, kt & 1, g);
                    ptx::tc_fence_after();
                    issue_pv(s, j > 0);
                    ptx::mma_commit(&bar_pv);   // P and O free again; after an item's last tile: O final
                    ptx::mma_commit(&bar_ve[s]);
                }
            }
            // Every MMA must have finished before TMEM is released (matters after a timeout).
            ptx::mma_commit(&bar_done);
            wait_bounded(&bar_done, 0, g);
        }
    } else {
        // ---------------------------------------------------------------- V to fp16
        // every V tile of this CTA's ring, in order, rewritten as fp16 in place once it has landed
        // (passed on unchanged when V is fp16 already)
        const int ct = (warp - C::CONV_WARP) * 32 + lane;
        const int n_steps = first < n_items ? ((n_items - first + stride - 1) / stride) * nkv : 0;
        for (int kv = 0; kv < n_steps; ++kv) {
            const int sv = kv % C::STAGES;
            wait_bounded(&bar_vf[sv], (kv / C::STAGES) & 1, g);
            if (!v_f16)
                tile_bf16_to_f16<C::KV_BYTES / 16, C::CONV_THREADS, C::CONV_PASS>(ptx::smem_u32(sV + sv * C::KV_BYTES), ct);
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bar_vc[sv]);
        }
    }
    } else {
        ptx::setmaxnreg_inc<C::REG_SOFTMAX>();
        // ---------------------------------------------------------------- softmax warpgroup
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t tS = tmem + lane_off, tO = tmem + lane_off + C::TM_O, tP = tmem + lane_off + C::TM_P;
        const int r_local = warp * 32 + lane;   // row of the tile = TMEM lane
        int kt = 0, li = 0;
        for (int item = first; item < n_items; item += stride, ++li) {
            const int bh = item / n_qblocks, q0 = (item % n_qblocks) * C::BM;
            const int row = q0 + r_local;
            const int qb = li & 1;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < nkv; ++j, ++kt) {
                wait_bounded(&bar_s, kt & 1, g);
                ptx::tc_fence_after();
                uint32_t r[128];
                ptx::tmem_ld32_at<0>(tS + 0, r);
                ptx::tmem_ld32_at<32>(tS + 32, r);
                ptx::tmem_ld32_at<64>(tS + 64, r);
                ptx::tmem_ld32_at<96>(tS + 96, r);
                ptx::tmem_ld_wait();
                reg_fence(r);
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bar_sread);   // S may take the next product
                const int valid = n - j * C::BN;
                if (valid < C::BN) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (i >= valid) r[i] = __float_as_uint(-INFINITY);
                }
                float mx[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(r[u]);
#pragma unroll
                for (int i = 8; i < 128; i += 2)
                    mx[(i >> 1) & 7] = ptx::max3(mx[(i >> 1) & 7], __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                const float smax = ptx::max3(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], mx[5]),
                                             fmaxf(mx[6], mx[7]));
                const float mt = smax * scale_log2;
                float m_new = m, alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m_new = mt;
                } else if (__any_sync(0xffffffffu, mt > m + kTau)) {
                    m_new = fmaxf(m, mt);
                    alpha = ptx::ex2(m - m_new);
                    rescale = true;
                }
                const float neg_m = kPOff - m_new;
                const uint64_t c2 = ptx::f2_pack(scale_log2, scale_log2), nm2 = ptx::f2_pack(neg_m, neg_m);
                uint64_t sum2[2] = {ptx::f2_pack(0.f, 0.f), ptx::f2_pack(0.f, 0.f)};
                // P = 2^(x - m + kPOff) as fp16 pairs, packed into r[0, 64)
#pragma unroll
                for (int i = 0; i < 128; i += 2) {
                    const uint64_t t = ptx::fma_f32x2(ptx::f2_pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), c2, nm2);
                    float t0, t1;
                    ptx::f2_unpack(t, t0, t1);
                    const float p0 = ptx::ex2(t0), p1 = ptx::ex2(t1);
                    sum2[(i >> 1) & 1] = ptx::add_f32x2(sum2[(i >> 1) & 1], ptx::f2_pack(p0, p1));
                    const uint32_t h = ptx::pack_f16x2(p0, p1);
                    r[i >> 1] = h;
                }
                float sum[4];
                ptx::f2_unpack(sum2[0], sum[0], sum[1]);
                ptx::f2_unpack(sum2[1], sum[2], sum[3]);
                l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
                m = m_new;
                // the previous P V is done with the P columns and O
                if (kt > 0) wait_bounded(&bar_pv, (kt - 1) & 1, g);
                ptx::tc_fence_after();
                if (rescale) {
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t ov[32];
                        ptx::tmem_ld32(tO + c, ov);
                        ptx::tmem_ld_wait();
                        reg_fence(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        ptx::tmem_st32(tO + c, ov);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) pk[i] = r[h * 32 + i];
                    ptx::tmem_st32(tP + h * 32, pk);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bar_p);
            }

            // epilogue of this item, once its last P V is done: O / l (bf16) into the Q buffer
            // (128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8)), then one TMA
            // store of the tile; LSE = (m - kPOff + log2 l) ln 2
            wait_bounded(&bar_pv, (kt - 1) & 1, g);
            ptx::tc_fence_after();
            const float inv_l = 1.f / l;
            const uint32_t srow = ptx::smem_u32(sQ + qb * C::Q_BYTES) + r_local * 128;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t ov[32];
                ptx::tmem_ld32(tO + c, ov);
                ptx::tmem_ld_wait();
                reg_fence(ov);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = ptx::pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l,
                                             __uint_as_float(ov[2 * i + 1]) * inv_l);
                if (o32 && row < n) store_o32(o32 + ((size_t)bh * n + row) * D + c, ov, inv_l);
                // columns [c, c + 32) of a 64-column box: chunks (c % 64) / 8 + v4
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    const int chunk = ((c & 63) >> 3) + v4;
                    sts_u128(srow + (c >> 6) * (C::BM * 128) + ((chunk ^ (r_local & 7)) << 4),
                             make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]));
                }
            }
            ptx::tc_fence_before();   // O read: the next item's first P V may overwrite it
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bar_ost[qb]);   // the producer stores the tile
            if (row < n) lse[(size_t)bh * n + row] = (m - kPOff + log2f(l)) * kLn2;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}


template <int D>
cudaError_t launch_fwd_persistent(const FwdArgs &a, cudaStream_t stream)
{
    using C = PersistCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(fwd_persistent_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_qblocks = (a.n + C::BM - 1) / C::BM;
    const long long items = (long long)n_qblocks * a.bh;
    // Two CTAs per SM: TMEM (256 columns each), shared memory and registers are sized for it.
    const long long ctas = std::min<long long>(items, 2LL * device_sm_count());
    fwd_persistent_kernel<D><<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.lse, a.o32, a.n, n_qblocks,
        (int)items, a.scale * kLog2e, a.v_f16, a.status);
    return cudaGetLastError();
}

template <int D, int NQ>
cudaError_t launch_fwd_d(const FwdArgs &a, cudaStream_t stream)
{
    using C = FwdCfg<D, NQ>;
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, NQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int rows_per_cta = C::NQ * C::BM;
    const int n_qblocks = (a.n + rows_per_cta - 1) / rows_per_cta;
    const long long ctas = (long long)n_qblocks * a.bh;
    fwd_kernel<D, NQ><<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, reinterpret_cast<__nv_bfloat16 *>(a.o), a.lse, a.o32, a.n, n_qblocks,
        a.scale * kLog2e, a.v_f16, a.status);
    return cudaGetLastError();
}

cudaError_t launch_fwd_sp(const FwdArgs &a, cudaStream_t stream)
{
    using C = FwdSpCfg;
    cudaError_t e = cudaFuncSetAttribute(fwd_sp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_qblocks = (a.n + C::BM - 1) / C::BM;
    const long long ctas = (long long)n_qblocks * a.bh;
    fwd_sp_kernel<<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.lse, a.o32, a.n, n_qblocks, a.scale * kLog2e, a.v_f16, a.status);
    return cudaGetLastError();
}

// V rounded to fp16 once, ahead of the forward kernel, for attn_fwd_with_workspace: the same
// rounding as tile_bf16_to_f16, over the whole [BH, N, d] tensor at HBM speed, so that the
// converter warps of every CTA reading V no longer rewrite each tile in shared memory (64
// CTAs read each V tile at d = 128 and N = 16384).  16-byte vectors, two in flight per
// thread, grid-stride over whole waves of the SMs; n16 = elements / 8.  V is read once more
// (by the backward) at most, so its loads stream; the fp16 copy is read right away by the
// forward kernel and is stored normally.
__global__ void __launch_bounds__(256)
    v_to_f16_kernel(const uint4 *__restrict__ v, uint4 *__restrict__ v16, long long n16)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    auto cvt = [](uint4 x) {
        return make_uint4(ptx::bf16x2_to_f16x2(x.x), ptx::bf16x2_to_f16x2(x.y), ptx::bf16x2_to_f16x2(x.z),
                          ptx::bf16x2_to_f16x2(x.w));
    };
    for (; i + stride < n16; i += 2 * stride) {
        const uint4 a = __ldcs(v + i), b = __ldcs(v + i + stride);
        v16[i] = cvt(a);
        v16[i + stride] = cvt(b);
    }
    if (i < n16) v16[i] = cvt(__ldcs(v + i));
}

}  // namespace

cudaError_t launch_v_to_f16(const void *v, void *v16, long long elems, cudaStream_t stream)
{
    const long long n16 = elems / 8;
    const long long want = (n16 + 255) / 256;
    const long long blocks = std::max(1LL, std::min<long long>(want, 8LL * device_sm_count()));
    v_to_f16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint4 *>(v), static_cast<uint4 *>(v16),
                                                          n16);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdArgs &a, cudaStream_t stream)
{
    if (a.d == 128) return launch_fwd_d<128, 2>(a, stream);
    // d = 64: one 128-row query tile per CTA, two CTAs per SM; persistent CTAs wherever there
    // are more tiles than resident CTAs (equal to one CTA per tile at long sequences, ahead
    // where items are short), else one CTA per tile
    const long long tiles = (long long)a.bh * ((a.n + 127) / 128);
    if (tiles > 2LL * device_sm_count()) return launch_fwd_persistent<64>(a, stream);
    return launch_fwd_sp(a, stream);
}

}  // namespace attn
