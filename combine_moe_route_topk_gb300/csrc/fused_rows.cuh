// Receive rows of the decode-fused dispatch's pack kernels (the bf16/f32
// pack in dispatch_pack.cu and the fp8-quantising pack in
// dispatch_pack_quant.cu): each pair's row, derived from what the fused
// route kernel leaves behind (see PackDerive in moe_internal.cuh), and the
// send counts of source ranks split over several route blocks.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Row of pair (g, k) with expert e and rank `rank` among its route block's
// pairs of e: d*cap + (start of e within rank d) + pairs of e in earlier
// chunks of 8 route blocks + pairs of e in the earlier blocks of this chunk
// + rank; -1 past the rank's capacity.  The rows of one expert follow the
// token order, as the count kernel lays them out.
__device__ __forceinline__ int fused_row(const PackDerive &D, int64_t g, int e, int rank) {
    const int gi = (int)g;
    const int b = D.ranks_per_block > 0 ? gi / (D.ranks_per_block * D.T)
                                        : (gi / D.T) * D.blocks_per_rank + (gi % D.T) / 32;
    const int d = e / D.L;
    const int c0 = b & ~7;  // first block of b's chunk of 8
    int local = __ldg(D.expert_offsets + e) - __ldg(D.expert_offsets + d * D.L) +
                (int)__ldg(D.chunk_prefix + (int64_t)(b >> 3) * D.Ep + e) + rank;
#pragma unroll
    for (int j = 0; j < 7; ++j)
        if (c0 + j < b) local += __ldg(D.block_hist + (int64_t)(c0 + j) * D.Ep + e);
    return local < D.cap ? d * D.cap + local : -1;
}

// Block s < N of a pack kernel writes row s of send_counts when source ranks
// are split over several route blocks (their per-block counts summed).
__device__ __forceinline__ void fused_send_counts(const PackDerive &D) {
    if (D.blocks_per_rank > 0 && (int)blockIdx.x < D.N) {
        const int s = (int)blockIdx.x, cps = D.blocks_per_rank;
        for (int d = threadIdx.x; d < D.N; d += blockDim.x) {
            int c = 0;
            for (int k = 0; k < cps; ++k) c += __ldg(D.block_send + (int64_t)(s * cps + k) * D.N + d);
            D.send_counts[(int64_t)s * D.N + d] = c;
        }
    }
}

}  // namespace moe
