// Route top-k: one warp per token.
//
// "Efficient and portable mixture-of-experts communication", section
// "Introduction": a small linear router produces a probability distribution
// over the experts; each token goes to its top-K experts, weighted by it.
// "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "MoE Router": the pages do this with a sort that
// carries the element indices.  Here a full sort is unnecessary: R rounds of
// a warp-wide arg-max select the same experts in the same order.
//
// Layout: lane l owns the J consecutive experts [l*J, l*J + J), J a
// compile-time constant with 32*J >= E.  Because lower lanes own lower
// expert ids, "highest key, then lowest lane, then lowest slot" is exactly
// "highest z, then lowest expert index" -- the tie rule of the definition.
//
// Keys: z = fl32(logit + bias) is mapped to an unsigned integer whose order
// is the float order (-0 is first turned into +0 so that the two zeros tie,
// as they compare equal).  A round is one warp max reduction (redux.sync)
// over each lane's best remaining key and a ballot for the lowest lane
// holding the maximum.  A lane with at most 8 keys sorts them once (bitonic
// network, key descending, slot ascending) and pops its head when it wins;
// a lane with 12 or more keeps only its best and second-best keys, promotes
// the runner-up when it wins and rescans its remaining keys only when it
// wins a third time (sorting 12 or more keys doubled the instructions per
// token on the 384-expert batch, where routing is bound by instruction
// issue: route 14.6 -> 12.3 us there; with 4 or 8 keys the sort is cheaper).
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "route_impl.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;  // 8 tokens per block

template <int J, bool kVec4>
__global__ void __launch_bounds__(kRouteThreads)
route_topk_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int64_t NT,
                  int E, int R, int score_fn, int renormalize, int32_t *__restrict__ topk_idx,
                  float *__restrict__ topk_w) {
    grid_dependency_wait();  // logits / outputs are shared with earlier kernels
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * (kRouteThreads / 32) + (threadIdx.x >> 5);
    if (g >= NT) return;  // uniform per warp
    route_impl::route_token<J, kVec4>(logits, bias, g, E, R, score_fn, renormalize, topk_idx,
                                      topk_w, lane);
}

template <int J, bool kVec4>
cudaError_t launch_jv(const float *logits, const float *bias, int64_t NT, int E, int R,
                      int score_fn, int renormalize, int32_t *topk_idx, float *topk_w,
                      cudaStream_t stream) {
    const int64_t blocks = (NT + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_topk_kernel<J, kVec4>, logits, bias, NT, E, R, score_fn,
                              renormalize, topk_idx, topk_w);
}

template <int J>
cudaError_t launch_j(const float *logits, const float *bias, int64_t NT, int E, int R, int score_fn,
                     int renormalize, int32_t *topk_idx, float *topk_w, cudaStream_t stream) {
    if constexpr (J % 4 == 0) {
        if (E % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0)
            return launch_jv<J, true>(logits, bias, NT, E, R, score_fn, renormalize, topk_idx,
                                      topk_w, stream);
    }
    return launch_jv<J, false>(logits, bias, NT, E, R, score_fn, renormalize, topk_idx, topk_w,
                               stream);
}

}  // namespace

cudaError_t launch_route_topk(const float *logits, const float *bias, int64_t NT, int E, int R,
                              int score_fn, int renormalize, int32_t *topk_idx, float *topk_w,
                              cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int need = (E + 31) / 32;  // slots per lane
#define MOE_ROUTE_CASE(JV) \
    if (need <= JV) return launch_j<JV>(logits, bias, NT, E, R, score_fn, renormalize, topk_idx, topk_w, stream);
    MOE_ROUTE_CASE(1)
    MOE_ROUTE_CASE(2)
    MOE_ROUTE_CASE(4)
    MOE_ROUTE_CASE(8)
    MOE_ROUTE_CASE(12)
    MOE_ROUTE_CASE(16)
    MOE_ROUTE_CASE(24)
    MOE_ROUTE_CASE(32)
#undef MOE_ROUTE_CASE
    return cudaErrorInvalidValue;  // E > 1024 is rejected before this point
}

}  // namespace moe
