// Global-memory access helpers shared by the streaming kernels: 16-byte
// loads that bypass L1, L2 eviction-priority policies, and bulk L2
// prefetch.  All of them are plain PTX (sm_90+); the hints change only
// where lines are kept, never the values read or written.
#pragma once

#include <cstdint>

namespace moe {

// 16-byte read-only load that does not allocate in L1 (each line is used once).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte store whose line is among the first to leave L2.
__device__ __forceinline__ void st_evict_first(uint4 *p, const uint4 &v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p),
                 "r"(bytes), "l"(pol)
                 : "memory");
}

// Rows [0, pf_rows) of a row-major array go to L2 ahead of use: block b <
// pf_blocks has its thread 0 prefetch rows b, b + pf_blocks, ... with the
// evict-last policy.  A prefetch is only a hint and L2 is where every write
// lands, so it may be issued before the kernel waits for its predecessors.
__device__ __forceinline__ void prefetch_rows_l2(const void *base, int64_t row_bytes,
                                                 int64_t pf_rows, int pf_blocks) {
    if (threadIdx.x == 0 && (int)blockIdx.x < pf_blocks) {
        const uint64_t keep = l2_policy_evict_last();
        const unsigned char *b = static_cast<const unsigned char *>(base);
        for (int64_t r = blockIdx.x; r < pf_rows; r += pf_blocks)
            prefetch_l2(b + r * row_bytes, (uint32_t)row_bytes, keep);
    }
}

// Division of 32-bit dividends below 2^31 by a divisor fixed for a launch
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): with l = ceil(log2 d) and m = floor(2^32 (2^l - d)
// / d) + 1, n / d = (umulhi(n, m) + n) >> l.  The host computes (m, l) once;
// the kernel spends a multiply-high, an add and a shift per division.
struct FastDiv {
    uint32_t mul, shift;
};

inline FastDiv make_fast_div(uint32_t d) {  // d >= 1
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    const uint64_t m = (((1ull << 32) * ((1ull << l) - d)) / d) + 1;
    return FastDiv{(uint32_t)m, l};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

}  // namespace moe
