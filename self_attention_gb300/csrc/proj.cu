// The query / key / value projection of "Self-attention, CUDA kernels and FlashAttention",
// section 1 ("Generating queries, keys and values": Q = X W_Q, K = X W_K, V = X W_V with one
// d_k-wide block of columns of each W per head), and its backward, on tcgen05 tensor cores.
//
// One persistent GEMM skeleton, C[128 x BN tile] = sum over 64-wide K steps of A B (BN = 256
// when D is a multiple of 256, else 128), with three operand / epilogue policies:
//   ProjFwd : A = X [B*N, D] (K-major), B = W_t [D, D] (MN-major); the epilogue writes the
//             tile straight into the head-split [B, H, N, d_k] layout of Q, K or V.
//   ProjDx  : dX = sum_t dY_t W_t^T.  A = dY_t read from the head-split gradient (K-major,
//             query tiles within one batch row), B = W_t (K-major: W_t's rows are dX's columns).
//   ProjDw  : dW_t = X^T dY_t.  A = X^T (MN-major), B = dY_t (MN-major), K = the B*N token rows
//             taken 64 at a time within each batch.  A work item owns one 128 x 128 tile of dW
//             and stores it (fp32) once, unless splitting the token rows over several items
//             evens out the rounds of work items per SM; then dW is zeroed and the items add
//             their partial tiles with red.global.add.
// Each CTA (one per SM) walks the work items blockIdx.x, blockIdx.x + gridDim.x, ...:
// warp 0 TMA producer (a 4-stage ring of A and B tiles running across items), warp 1 tcgen05
// issuer (and TMEM owner), warps 4-7 epilogue (thread = row of the tile = TMEM lane).  The
// accumulator is double-buffered in TMEM (2 x BN columns), so the epilogue of one item
// overlaps the products of the next.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;            // A tile per stage (16 KB)
template <int BN>
struct Tile {
    // 192 KB of operand stages either way: the K loop is bound by L2 latency and bandwidth
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
    static constexpr uint32_t TM_COLS = 2 * BN;   // two accumulators
};

struct ProjParams {
    int B, N, D, H, dk;
    int n_mtiles, n_ntiles, ksplit, ksteps_per_split, n_items;
    __nv_bfloat16 *out[3];   // ProjFwd: Q, K, V
    __nv_bfloat16 *dx;       // ProjDx
    float *dw[3];            // ProjDw
    int *status;
};

// K-major tile of rows x 64 columns (boxes of 128 B rows): the k-th 16-wide slice starts 32 bytes in.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk)
{
    return ptx::sdesc_sw128(base + kk * 32, 16, 1024);
}
// MN-major tile of 64 rows (K) x (64 n) columns, stored as n 64-column blocks of 8 KB.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int kk)
{
    return ptx::sdesc_sw128(base + kk * 2048, 8192, 1024);
}

// ------------------------------------------------------------------ policies
struct ProjFwd {
    static constexpr bool A_MN = false, B_MN = true;
    // tile (m0 over B*N rows, n0 over the 3*D concatenated output columns; a tile lies in one W_t)
    __device__ static int ksteps(const ProjParams &p) { return p.D / BK; }
    template <int BN>
    __device__ static void load(const CUtensorMap *const *ma, const CUtensorMap *const *mb, const ProjParams &p,
                                int mt, int nt, int step, uint8_t *sa, uint8_t *sb, uint64_t *bar)
    {
        const int m0 = mt * BM, n0 = nt * BN, t = n0 / p.D, c0 = n0 % p.D, k0 = step * BK;
        ptx::tma_load_3d(sa, ma[0], bar, k0, m0, 0);
#pragma unroll
        for (int h = 0; h < BN / 64; ++h) ptx::tma_load_3d(sb + h * 8192, mb[t], bar, c0 + 64 * h, k0, 0);
    }
    template <int BN>
    __device__ static void store(const ProjParams &p, int mt, int nt, int ks, int lane_row,
                                 int c, const uint32_t (&v)[32])
    {
        const long long m = (long long)mt * BM + lane_row;
        if (m >= (long long)p.B * p.N) return;
        const int b = (int)(m / p.N), i = (int)(m % p.N);
        const int n0 = nt * BN, t = n0 / p.D, col = n0 % p.D + c;   // column within W_t
        const int h = col / p.dk, dd = col % p.dk;
        __nv_bfloat16 *dst = p.out[t] + (((size_t)b * p.H + h) * p.N + i) * p.dk + dd;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
};

struct ProjDx {
    static constexpr bool A_MN = false, B_MN = false;
    // tile (mt = batch b x query block, n0 over D input columns); K = 3 D gradient columns
    __device__ static int ksteps(const ProjParams &p) { return 3 * p.D / BK; }
    template <int BN>
    __device__ static void load(const CUtensorMap *const *ma, const CUtensorMap *const *mb, const ProjParams &p,
                                int mt, int nt, int step, uint8_t *sa, uint8_t *sb, uint64_t *bar)
    {
        const int qblocks = (p.N + BM - 1) / BM;
        const int b = mt / qblocks, i0 = (mt % qblocks) * BM;
        const int c = step * BK, t = c / p.D, ct = c % p.D, h = ct / p.dk, dd0 = ct % p.dk;
        ptx::tma_load_3d(sa, ma[t], bar, dd0, i0, b * p.H + h);
#pragma unroll
        for (int r = 0; r < BN / 128; ++r)   // 128-row boxes of W_t, contiguous
            ptx::tma_load_3d(sb + r * 16384, mb[t], bar, ct, nt * BN + 128 * r, 0);
    }
    template <int BN>
    __device__ static void store(const ProjParams &p, int mt, int nt, int ks, int lane_row,
                                 int c, const uint32_t (&v)[32])
    {
        const int qblocks = (p.N + BM - 1) / BM;
        const int b = mt / qblocks, i = (mt % qblocks) * BM + lane_row;
        if (i >= p.N) return;
        __nv_bfloat16 *dst = p.dx + ((size_t)b * p.N + i) * p.D + nt * BN + c;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
};

struct ProjDw {
    static constexpr bool A_MN = true, B_MN = true;
    // tile (m0 over D input rows j, n0 over the 3*D concatenated gradient columns); K = token
    // rows, 64 per step within one batch; split ks of p.ksplit takes a contiguous step range
    __device__ static int ksteps(const ProjParams &p) { return p.B * ((p.N + BK - 1) / BK); }
    template <int BN>
    __device__ static void load(const CUtensorMap *const *ma, const CUtensorMap *const *mb, const ProjParams &p,
                                int mt, int nt, int step, uint8_t *sa, uint8_t *sb, uint64_t *bar)
    {
        const int iblocks = (p.N + BK - 1) / BK;
        const int b = step / iblocks, i0 = (step % iblocks) * BK;
        const int j0 = mt * BM, n0 = nt * BN, t = n0 / p.D, ct = n0 % p.D;
        ptx::tma_load_3d(sa, ma[0], bar, j0, i0, b);
        ptx::tma_load_3d(sa + 8192, ma[0], bar, j0 + 64, i0, b);
#pragma unroll
        for (int g = 0; g < BN / 64; ++g) {
            const int col = ct + 64 * g, h = col / p.dk, dd0 = col % p.dk;
            ptx::tma_load_3d(sb + g * 8192, mb[t], bar, dd0, i0, b * p.H + h);
        }
    }
    template <int BN>
    __device__ static void store(const ProjParams &p, int mt, int nt, int ks, int lane_row,
                                 int c, const uint32_t (&v)[32])
    {
        const int j = mt * BM + lane_row, n0 = nt * BN, t = n0 / p.D, col = n0 % p.D + c;
        float *dst = p.dw[t] + (size_t)j * p.D + col;
        if (p.ksplit == 1) {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
            for (int q = 0; q < 8; ++q) d4[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst + e), "f"(__uint_as_float(v[e])) : "memory");
        }
    }
};

// ------------------------------------------------------------------ the GEMM skeleton
template <class P, int BN>
__global__ void __launch_bounds__(256, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                     const __grid_constant__ CUtensorMap a2, const __grid_constant__ CUtensorMap b0,
                     const __grid_constant__ CUtensorMap b1, const __grid_constant__ CUtensorMap b2,
                     const ProjParams p)
{
    using T = Tile<BN>;
    constexpr int STAGES = T::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ uint64_t bar_full[STAGES], bar_empty[STAGES], bar_acc_full[2], bar_acc_empty[2];
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = p.n_mtiles * p.n_ntiles;
    const int total = P::ksteps(p);
    // item -> (k split, m tile, n tile) and its K-step range
    auto decode = [&](int item, int &ks, int &mt, int &nt, int &k_begin, int &nk) {
        ks = item / tiles;
        const int tile = item % tiles;
        nt = tile % p.n_ntiles;
        mt = tile / p.n_ntiles;
        k_begin = ks * p.ksteps_per_split;
        const int k_end = (k_begin + p.ksteps_per_split < total) ? k_begin + p.ksteps_per_split : total;
        nk = k_end > k_begin ? k_end - k_begin : 0;
    };
    const Guard g{&abort_sh, p.status, kWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&bar_full[s], 1);
            ptx::mbar_init(&bar_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bar_acc_full[b], 1);
            ptx::mbar_init(&bar_acc_empty[b], 128);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&tmem_sh, T::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_sh;

    if (warp == 0) {
        if (ptx::elect_one()) {
            // pointers to the kernel-parameter maps (TMA reads a map from parameter space)
            const CUtensorMap *mas[3] = {&a0, &a1, &a2};
            const CUtensorMap *mbs[3] = {&b0, &b1, &b2};
            int j = 0;   // position in the stage ring, across items
            for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
                int ks, mt, nt, k_begin, nk;
                decode(item, ks, mt, nt, k_begin, nk);
                for (int q = 0; q < nk; ++q, ++j) {
                    const int s = j % STAGES;
                    const uint32_t ph = (j / STAGES) & 1;
                    wait_bounded(&bar_empty[s], ph ^ 1, g);
                    ptx::mbar_arrive_expect_tx(&bar_full[s], T::STAGE_BYTES);
                    uint8_t *sa = smem + s * T::STAGE_BYTES;
                    P::template load<BN>(mas, mbs, p, mt, nt, k_begin + q, sa, sa + A_BYTES, &bar_full[s]);
                }
            }
            for (int q = (j > STAGES ? j - STAGES : 0); q < j; ++q)
                wait_bounded(&bar_full[q % STAGES], (q / STAGES) & 1, g);
        }
    } else if (warp == 1) {
        if (ptx::elect_one()) {
            const uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, P::A_MN, P::B_MN);
            const uint32_t base = ptx::smem_u32(smem);
            int j = 0, li = 0;
            for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, ++li) {
                int ks, mt, nt, k_begin, nk;
                decode(item, ks, mt, nt, k_begin, nk);
                const int ab = li & 1;
                wait_bounded(&bar_acc_empty[ab], ((li >> 1) & 1) ^ 1, g);   // epilogue of item li-2 done
                ptx::tc_fence_after();
                for (int q = 0; q < nk; ++q, ++j) {
                    const int s = j % STAGES;
                    wait_bounded(&bar_full[s], (j / STAGES) & 1, g);
                    ptx::tc_fence_after();
                    const uint32_t sa = base + s * T::STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t da = P::A_MN ? desc_mnmajor(sa, kk) : desc_kmajor(sa, kk);
                        const uint64_t db = P::B_MN ? desc_mnmajor(sb, kk) : desc_kmajor(sb, kk);
                        ptx::mma_ss(tmem + ab * BN, da, db, idesc, (q > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(&bar_empty[s]);
                }
                ptx::mma_commit(&bar_acc_full[ab]);
            }
            // every MMA must have finished before TMEM is released (matters after a timeout)
            for (int b = 0; b < 2 && b < li; ++b) {
                const int last = li - 1 - ((li - 1 - b) & 1);   // the last item that used buffer b
                wait_bounded(&bar_acc_full[last & 1], (last >> 1) & 1, g);
            }
        }
    } else if (warp >= 4) {
        const int quarter = warp & 3, lane_row = quarter * 32 + lane;
        int li = 0;
        for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, ++li) {
            int ks, mt, nt, k_begin, nk;
            decode(item, ks, mt, nt, k_begin, nk);
            const int ab = li & 1;
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + ab * BN;
            wait_bounded(&bar_acc_full[ab], (li >> 1) & 1, g);
            ptx::tc_fence_after();
            if (nk > 0) {
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    ptx::tmem_ld32(taddr + c, v);
                    ptx::tmem_ld_wait();
                    reg_fence(v);
                    P::template store<BN>(p, mt, nt, ks, lane_row, c, v);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_acc_empty[ab]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, T::TM_COLS);
    }
}

__global__ void zero_f32_kernel(float *p, long long n)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0.f;
}

template <class P, int BN>
cudaError_t launch_gemm(const ProjMaps &m, ProjParams p, int sms, cudaStream_t stream)
{
    using T = Tile<BN>;
    cudaError_t e = cudaFuncSetAttribute(proj_gemm_kernel<P, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int ctas = p.n_items < sms ? p.n_items : sms;   // persistent: one CTA per SM
    proj_gemm_kernel<P, BN><<<ctas, 256, T::SMEM_BYTES, stream>>>(m.a[0], m.a[1], m.a[2], m.b[0], m.b[1],
                                                                  m.b[2], p);
    return cudaGetLastError();
}

int num_sms()
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

}  // namespace

cudaError_t launch_proj_fwd(const ProjMaps &m, const ProjArgs &a, cudaStream_t stream)
{
    ProjParams p = {};
    p.B = a.B; p.N = a.N; p.D = a.D; p.H = a.H; p.dk = a.dk; p.status = a.status;
    p.n_mtiles = (int)(((long long)a.B * a.N + BM - 1) / BM);
    const bool wide = a.D % 256 == 0;   // a 256-column tile must lie within one W_t
    p.n_ntiles = 3 * a.D / (wide ? 256 : 128);
    p.ksplit = 1;
    p.ksteps_per_split = a.D / BK;
    p.n_items = p.n_mtiles * p.n_ntiles;
    for (int t = 0; t < 3; ++t) p.out[t] = a.qkv[t];
    return wide ? launch_gemm<ProjFwd, 256>(m, p, num_sms(), stream)
                : launch_gemm<ProjFwd, 128>(m, p, num_sms(), stream);
}

cudaError_t launch_proj_dx(const ProjMaps &m, const ProjArgs &a, cudaStream_t stream)
{
    ProjParams p = {};
    p.B = a.B; p.N = a.N; p.D = a.D; p.H = a.H; p.dk = a.dk; p.status = a.status;
    p.n_mtiles = a.B * ((a.N + BM - 1) / BM);
    const bool wide = a.D % 256 == 0;
    p.n_ntiles = a.D / (wide ? 256 : 128);
    p.ksplit = 1;
    p.ksteps_per_split = 3 * a.D / BK;
    p.n_items = p.n_mtiles * p.n_ntiles;
    p.dx = a.dx;
    return wide ? launch_gemm<ProjDx, 256>(m, p, num_sms(), stream)
                : launch_gemm<ProjDx, 128>(m, p, num_sms(), stream);
}

cudaError_t launch_proj_dw(const ProjMaps &m, const ProjArgs &a, cudaStream_t stream)
{
    // dW is only D x 3D: 128-column tiles give the most work items (108 at D = 768)
    ProjParams p = {};
    p.B = a.B; p.N = a.N; p.D = a.D; p.H = a.H; p.dk = a.dk; p.status = a.status;
    p.n_mtiles = a.D / BM;
    p.n_ntiles = 3 * a.D / 128;
    const int tiles = p.n_mtiles * p.n_ntiles;
    const int total = a.B * ((a.N + BK - 1) / BK);
    const int sms = num_sms();
    // Rounds of items per SM, in units of one whole-K tile: ceil(tiles * s / sms) / s for s
    // splits.  The atomics of a split cost ~15-20 % (measured), so split two or three ways
    // only where that cuts the rounds by 1.4x or more.
    auto rounds = [&](int s) { return (double)((tiles * s + sms - 1) / sms) / s; };
    int ksplit = 1;
    for (int s = 2; s <= 3 && s <= total; ++s)
        if (rounds(1) >= 1.4 * rounds(s) && rounds(s) < rounds(ksplit)) ksplit = s;
    p.ksteps_per_split = (total + ksplit - 1) / ksplit;
    p.ksplit = (total + p.ksteps_per_split - 1) / p.ksteps_per_split;
    p.n_items = tiles * p.ksplit;
    for (int t = 0; t < 3; ++t) p.dw[t] = a.dw[t];
    if (p.ksplit > 1) {
        for (int t = 0; t < 3; ++t) {
            zero_f32_kernel<<<4 * sms, 256, 0, stream>>>(a.dw[t], (long long)a.D * a.D);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    return launch_gemm<ProjDw, 128>(m, p, sms, stream);
}

}  // namespace attn
