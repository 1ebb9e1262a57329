// Shared device helpers for the attention kernels: bounded mbarrier waits that report a
// timeout through a device status word instead of hanging, and small utilities.
#pragma once

#include "ptx.cuh"

namespace attn {

// Status codes written to the device status word; they match attn_status in include/attn.h.
constexpr int kStatusTimeout = 5;

// Longest a single wait may spin before the kernel gives up (nanoseconds of %globaltimer).
// Every wait in these kernels normally completes within microseconds.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Per-CTA failure state.  Once `abort` is set every later wait returns at once, so the CTA
// runs to its end quickly (its results are garbage and the status word says so).
struct Guard {
    int *abort_smem;   // shared-memory flag
    int *status;       // device status word (global)
    uint64_t limit_ns;
};

// Waits for the phase of `bar` with parity `parity` to complete.  Returns true on success,
// false if the wait timed out or the CTA had already aborted.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, const Guard &g)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*(volatile int *)g.abort_smem) return false;
        if (globaltimer_ns() - t0 > g.limit_ns) {
            *(volatile int *)g.abort_smem = 1;
            atomicCAS(g.status, 0, kStatusTimeout);
            return false;
        }
    }
}

// Keeps the compiler from using registers written by tcgen05.ld before tcgen05.wait::ld.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N])
{
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Returns `x` through an opaque move, so that addresses derived from it are recomputed where
// they are used instead of being hoisted out of a loop into dozens of live registers.
__device__ __forceinline__ uint32_t opaque(uint32_t x)
{
    uint32_t y;
    asm volatile("mov.b32 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void sts_f32(uint32_t addr, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Explicit shared-memory accesses: pointers derived from the aligned dynamic shared-memory
// base are generic to the compiler, and generic accesses take the slower L1TEX path.
__device__ __forceinline__ uint4 lds_u128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds_u64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_u128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace attn
