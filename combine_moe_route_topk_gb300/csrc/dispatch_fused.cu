// Decode-fused dispatch: route top-k, dispatch count and dispatch pack in
// one call, as two kernels launched back to back with programmatic
// dependent launch and no grid-wide wait anywhere.
//
// "Hosting Qwen on Blackwell", section "Expert parallel": for decode the
// whole dispatch kernel is fused into one, while prefill splits it into
// several kernels because routing needs fewer blocks than the rest.
// "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "CUDA Graph": a fixed number of kernels splits the
// dynamically routed work.  "Enabling trillion-parameter models on AWS
// EFA", section "Dispatch and combine": per-expert counts, then their
// cumulative sum gives the offsets at which tokens are packed per
// destination.  The outputs are identical to those of the separate kernels
// (route_topk.cu, dispatch_count.cu, dispatch_pack.cu).
//
// Kernel 1, route_hist_kernel: B blocks of 1024 threads, block b owning a
// contiguous run of at most 32 tokens that never crosses a source rank
// boundary (whole ranks per block when T <= 32, else ceil(T/32) blocks per
// rank), so blocks in index order hold tokens in index order.
//   1. each warp routes one token (the route kernel's per-token body);
//   2. a 32-bit mask per expert marks the block's tokens that chose it: a
//      pair's rank among the block's pairs of its expert is the population
//      count of the mask below its token (stored in pos for now), the
//      block's count of the expert the population count of the whole mask
//      (one byte per expert, published to the workspace), and its send
//      counts per destination rank sums of those over the rank's experts
//      (written to send_counts directly when the block holds whole source
//      ranks, else published per block);
//   3. the block takes a ticket from the workspace's arrival counter (an
//      acquire-release atomic after a block barrier).  Every block but the
//      last one exits here: nothing waits.  The block holding the last
//      ticket has acquired every histogram: it computes, per expert, the
//      exclusive prefix of the counts over chunks of 8 blocks (u16, to the
//      workspace) and the totals, scans those into the expert and rank
//      offsets, checks the capacity and resets the counter for the next
//      call.  The pack kernel sums the per-block send counts of split ranks.
// Kernel 2 is the pack kernel of dispatch_pack.cu in its deriving form:
// pair (g, k) of expert e on rank d, in block b of chunk c = b / 8, lands at
//   d*cap + (expert_offsets[e] - expert_offsets[d*L]) + chunk_prefix[c][e]
//         + (histograms of blocks 8c .. b-1 at e) + rank,
// which is the count kernel's position: rows of one expert in token order.
// It is scheduled while kernel 1 runs; its blocks that find room beside it
// start pulling the x rows into L2, as in the three-call chain, and it
// starts writing as soon as kernel 1 has completed.  (Prefetches issued by
// the routing warps themselves, at any point, delayed their own loads and
// the ticket: routing took 10-11 us instead of 6 on the DeepSeek-V3 batch.)
//
// On GB300 the pack starts writing rows about 6 us earlier than in the
// three-call chain (where the count kernel runs alone on one cluster); the
// fused call takes 85.1 us against 86.2 us for the three calls on the
// DeepSeek-V3-shaped decode batch and 87.4 against 89.6 us on the
// Kimi-K2-shaped one.
//
// Scope: decode batches (N*T <= 4096), R <= 32, E <= 512 (the host rejects
// anything else with MOE_ERR_UNSUPPORTED: use the three separate calls).
// The workspace's arrival counter must be zero before the first call (the
// caller zero-fills the workspace once); every call leaves it zero.
#include <mutex>

#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "route_impl.cuh"

namespace moe {
namespace {

constexpr int kFThreads = 1024;  // 32 warps: one token per warp
constexpr int kFWarps = kFThreads / 32;
constexpr int kFTok = 32;        // tokens per block (32-bit masks)
constexpr int kFMaxR = 32;       // pairs per block <= 1024 = threads
constexpr int kFMaxE = 512;      // 16 experts per lane: the route body fits 64 registers
constexpr int kFMaxNT = 4096;
constexpr int kFMaxBlocks = 256;  // N*T <= 4096 never needs more (at least 16 tokens per block on average)
constexpr int kWsHeaderBytes = 256;  // word 0: arrival counter
constexpr int kChunk = 8;            // blocks per prefix chunk

__host__ __device__ inline int pad16(int v) { return (v + 15) & ~15; }
__host__ __device__ inline int64_t align256(int64_t v) { return (v + 255) & ~(int64_t)255; }

// How kernel 1 splits the tokens into blocks.
struct FusedGeom {
    int B;    // blocks
    int rpb;  // > 0: whole source ranks per block (T <= 32)
    int cps;  // > 0: blocks per source rank (T > 32)
};

__host__ __device__ inline FusedGeom fused_geom(int N, int T) {
    FusedGeom g;
    if (T <= kFTok) {
        g.rpb = kFTok / T;
        g.cps = 0;
        g.B = (N + g.rpb - 1) / g.rpb;
    } else {
        g.rpb = 0;
        g.cps = (T + kFTok - 1) / kFTok;
        g.B = N * g.cps;
    }
    return g;
}

__device__ __forceinline__ void block_tokens(const FusedGeom &geo, int b, int N, int T, int &tb, int &te) {
    if (geo.rpb > 0) {
        const int s0 = b * geo.rpb, s1 = min(N, s0 + geo.rpb);
        tb = s0 * T;
        te = s1 * T;
    } else {
        const int s = b / geo.cps, c = b - s * geo.cps;
        tb = s * T + c * kFTok;
        te = s * T + min(T, (c + 1) * kFTok);
    }
}

// Workspace: the arrival counter, then the byte histograms [B][Ep], the
// chunk prefixes (u16) [ceil(B/8)][Ep] and, for ranks split over blocks,
// the per-block send counts (u16) [B][N].
struct WsLayout {
    int64_t hist, cpre, sd, bytes;
};

__host__ __device__ inline int n_chunks(int B) { return (B + kChunk - 1) / kChunk; }

__host__ __device__ inline WsLayout ws_layout(int N, int T, int E) {
    const FusedGeom g = fused_geom(N, T);
    const int Ep = pad16(E);
    WsLayout w;
    w.hist = kWsHeaderBytes;
    w.cpre = w.hist + align256((int64_t)g.B * Ep);
    w.sd = w.cpre + align256((int64_t)n_chunks(g.B) * Ep * 2);
    w.bytes = w.sd + (g.cps > 0 ? align256((int64_t)g.B * N * 2) : 0);
    return w;
}

// Shared memory of kernel 1; every section starts on a 16-byte boundary.
// Only the last block uses the histogram copy and the chunk sums, but the
// launch gives every block the same amount.
struct FSmem {
    int mask, sel, hs, gs, tot, bytes;
};

__host__ __device__ inline FSmem f_smem_layout(int E, int R, int B) {
    const int Ep = pad16(E);
    FSmem s;
    int o = 0;
    auto take = [&o](int bytes) {
        const int at = o;
        o += pad16(bytes);
        return at;
    };
    s.sel = take(kFTok * R * 4);    // experts of the block's pairs (first: offset 0)
    s.mask = take(Ep * 4);          // u32 per expert: the block's tokens that chose it
    s.hs = take(B * Ep);            // last block: every block's histogram
    s.gs = take(n_chunks(B) * Ep * 4);  // last block: sums over chunks of 8 blocks
    s.tot = take((E + 1) * 4);      // last block: totals, then offsets
    s.bytes = o;
    return s;
}

struct FusedParams {
    const float *logits;
    const float *bias;
    int score_fn, renormalize;
    int N, T, E, R, cap;
    FusedGeom geo;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *expert_counts, *expert_offsets, *rank_counts, *rank_offsets, *send_counts, *pos,
        *status;
    unsigned char *ws;
};

// Ticket of a block: add 1 with acquire-release semantics at GPU scope (the
// block's earlier writes, ordered before it by a block barrier, are released
// with it; the holder of the last ticket acquires every other block's).
__device__ __forceinline__ int atomic_add_acq_rel(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

template <int J, bool kVec4>
__global__ void __launch_bounds__(kFThreads, 1)
route_hist_kernel(FusedParams P) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_last;
    __shared__ int s_wsum[kFWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int tb, te;
    block_tokens(P.geo, (int)blockIdx.x, P.N, P.T, tb, te);
    const int ntok = te - tb;  // 1..32
    // sel (the block's selections) sits at the start of shared memory, so
    // that little stays live across the routing below
    int *sel = reinterpret_cast<int *>(smem);

    grid_dependency_wait();  // outputs may still be read by earlier kernels
    grid_launch_dependents();

    // ---- 1. route: warp w takes token tb + w --------------------------------------
    // (no x prefetch from here: issued by the routing warps, it delays their
    // own loads; the pack kernel's blocks that wait beside this kernel do it)
    if (warp < ntok) {
        const int e = route_impl::route_token<J, kVec4>(P.logits, P.bias, (int64_t)(tb + warp), P.E, P.R,
                                                        P.score_fn, P.renormalize, P.topk_idx, P.topk_w, lane);
        if (lane < P.R) sel[warp * P.R + lane] = e;
    }
    const int N = P.N, T = P.T, E = P.E, R = P.R, L = E / N, Ep = pad16(E);
    const int B = P.geo.B, b = (int)blockIdx.x;
    const FSmem lay = f_smem_layout(E, R, B);
    const WsLayout wl = ws_layout(N, T, E);
    uint32_t *mask = reinterpret_cast<uint32_t *>(smem + lay.mask);
    unsigned char *ws_hist = P.ws + wl.hist;
    const int npair = ntok * R;
    for (int i = tid; i < Ep; i += kFThreads) mask[i] = 0u;
    __syncthreads();
    if (tid < npair) atomicOr(mask + sel[tid], 1u << (tid / R));
    __syncthreads();

    // ---- 2. ranks in the block, histogram, send counts ------------------------------
    if (tid < npair) {
        const int e = sel[tid];
        const uint32_t below = (1u << (tid / R)) - 1u;
        P.pos[(int64_t)tb * R + tid] = __popc(mask[e] & below);  // completed by the pack kernel
    }
    for (int q = tid; q < Ep / 4; q += kFThreads) {
        const uint32_t w = (uint32_t)__popc(mask[4 * q]) | ((uint32_t)__popc(mask[4 * q + 1]) << 8) |
                           ((uint32_t)__popc(mask[4 * q + 2]) << 16) | ((uint32_t)__popc(mask[4 * q + 3]) << 24);
        reinterpret_cast<uint32_t *>(ws_hist + (int64_t)b * Ep)[q] = w;
    }
    if (P.geo.rpb > 0) {
        // whole source ranks: their rows of send_counts
        const int s0 = tb / T, ns = ntok / T;
        for (int i = tid; i < ns * N; i += kFThreads) {
            const int sl = i / N, d = i - sl * N;
            const uint32_t rows = (T == 32 ? 0xffffffffu : ((1u << T) - 1u)) << (sl * T);
            int c = 0;
            for (int e = d * L; e < d * L + L; ++e) c += __popc(mask[e] & rows);
            P.send_counts[(int64_t)(s0 + sl) * N + d] = c;
        }
    } else {
        uint16_t *sd = reinterpret_cast<uint16_t *>(P.ws + wl.sd) + (int64_t)b * N;
        for (int d = tid; d < N; d += kFThreads) {
            int c = 0;
            for (int e = d * L; e < d * L + L; ++e) c += __popc(mask[e]);
            sd[d] = (uint16_t)c;
        }
    }

    // ---- 3. ticket; the last block scans ----------------------------------------------
    __syncthreads();  // the block's histogram and send counts, released by its ticket
    if (tid == 0) s_last = atomic_add_acq_rel(reinterpret_cast<int *>(P.ws), 1) == B - 1;
    __syncthreads();
    if (!s_last) return;

    // every block's histogram into shared memory (L2 reads: written by other SMs)
    unsigned char *hs = smem + lay.hs;
    for (int i = tid; i < B * Ep / 16; i += kFThreads)
        reinterpret_cast<uint4 *>(hs)[i] = __ldcg(reinterpret_cast<const uint4 *>(ws_hist) + i);
    __syncthreads();
    // chunk sums: item (c, q) adds the histograms of blocks [8c, 8c + 8) for
    // experts 4q..4q+3, two experts per 32-bit word in 16-bit halves (at
    // most 8 * 32 per half)
    const int nq = Ep / 4, nc = n_chunks(B);
    int *gs = reinterpret_cast<int *>(smem + lay.gs);
    for (int it = tid; it < nc * nq; it += kFThreads) {
        const int c = it / nq, q = it - c * nq;
        const int r1 = min(B, (c + 1) * kChunk);
        uint32_t ev = 0u, od = 0u;
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            const int r = c * kChunk + j;
            if (r < r1) {
                const uint32_t w = reinterpret_cast<const uint32_t *>(hs + r * Ep)[q];
                ev += w & 0x00ff00ffu;
                od += (w >> 8) & 0x00ff00ffu;
            }
        }
        int *o = gs + c * Ep + 4 * q;
        o[0] = (int)(ev & 0xffffu);
        o[1] = (int)(od & 0xffffu);
        o[2] = (int)(ev >> 16);
        o[3] = (int)(od >> 16);
    }
    __syncthreads();
    // per expert: exclusive prefix over the chunks (u16 to the workspace: an
    // expert has at most N*T <= 4096 pairs) and the total
    int *tot = reinterpret_cast<int *>(smem + lay.tot);
    uint16_t *cpre = reinterpret_cast<uint16_t *>(P.ws + wl.cpre);
    for (int e = tid; e < Ep; e += kFThreads) {
        int run = 0;
        for (int c = 0; c < nc; ++c) {
            cpre[c * Ep + e] = (uint16_t)run;
            run += gs[c * Ep + e];
        }
        if (e < E) tot[e] = run;
    }
    __syncthreads();
    // exclusive scan of the totals over experts (E <= 512 < threads)
    const int v0 = tid < E ? tot[tid] : 0;
    int xs = v0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xs, off);
        if (lane >= off) xs += y;
    }
    if (lane == 31) s_wsum[warp] = xs;
    __syncthreads();
    if (warp == 0) {
        int sv = s_wsum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, sv, off);
            if (lane >= off) sv += y;
        }
        s_wsum[lane] = sv;  // inclusive over warps
    }
    __syncthreads();
    const int excl = xs - v0 + (warp > 0 ? s_wsum[warp - 1] : 0);
    if (tid < E) {
        tot[tid] = excl;
        P.expert_counts[tid] = v0;
        P.expert_offsets[tid] = excl;
    }
    if (tid == 0) {
        tot[E] = s_wsum[kFWarps - 1];
        P.expert_offsets[E] = s_wsum[kFWarps - 1];
    }
    __syncthreads();
    int over = 0;
    for (int d = tid; d < N; d += kFThreads) {
        const int rc = tot[(d + 1) * L] - tot[d * L];
        P.rank_counts[d] = rc;
        P.rank_offsets[d] = tot[d * L];
        over |= rc > P.cap;
    }
    over = __syncthreads_or(over);
    if (tid == 0) {
        P.rank_offsets[N] = tot[E];
        *P.status = over ? MOE_ERR_CAPACITY : MOE_OK;
        atomicExch(reinterpret_cast<int *>(P.ws), 0);  // every ticket is taken: ready for the next call
    }
}

template <int J, bool kVec4>
cudaError_t launch_route_hist_jv(const FusedParams &P, cudaStream_t stream) {
    auto kern = route_hist_kernel<J, kVec4>;
    const size_t smem = (size_t)f_smem_layout(P.E, P.R, P.geo.B).bytes;
    // the shared-memory attribute belongs to the current context: set once
    // per host thread, device and context for the largest request seen
    static thread_local int cached_dev = -1;
    static thread_local unsigned long long cached_ctx = 0;
    static thread_local size_t cached_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = context_key();
    if (dev != cached_dev || ctx == 0 || ctx != cached_ctx || smem > cached_smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        cached_dev = dev;
        cached_ctx = context_key();
        cached_smem = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P.geo.B);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int J>
cudaError_t launch_route_hist_j(const FusedParams &P, cudaStream_t stream) {
    if constexpr (J % 4 == 0) {
        if (P.E % 4 == 0 && (reinterpret_cast<uintptr_t>(P.logits) & 15) == 0)
            return launch_route_hist_jv<J, true>(P, stream);
    }
    return launch_route_hist_jv<J, false>(P, stream);
}

// Limits of the two-kernel form ("" when it can run the batch).
const char *two_kernel_unsupported(int N, int T, int E, int R) {
    if (R > kFMaxR) return "R > 32";
    if (E > kFMaxE) return "E > 512";
    if ((int64_t)N * T > kFMaxNT) return "N*T > 4096 (not a decode batch)";
    if (fused_geom(N, T).B > kFMaxBlocks) return "more than 256 route blocks";  // not reached for N*T <= 4096
    return "";
}

}  // namespace

// Kernel 1 of the two-kernel form; fills *D with what the pack kernel needs
// to derive the rows.
static cudaError_t launch_route_hist(const float *logits, const float *bias, int score_fn, int renormalize, int N, int T,
                              int E, int R, int64_t cap, int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                              int32_t *expert_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                              int32_t *send_counts, int32_t *pos, int32_t *status, void *workspace,
                              cudaStream_t stream, PackDerive *D) {
    FusedParams P;
    P.logits = logits;
    P.bias = bias;
    P.score_fn = score_fn;
    P.renormalize = renormalize;
    P.N = N;
    P.T = T;
    P.E = E;
    P.R = R;
    P.cap = (int)cap;
    P.geo = fused_geom(N, T);
    P.topk_idx = topk_idx;
    P.topk_w = topk_w;
    P.expert_counts = expert_counts;
    P.expert_offsets = expert_offsets;
    P.rank_counts = rank_counts;
    P.rank_offsets = rank_offsets;
    P.send_counts = send_counts;
    P.pos = pos;
    P.status = status;
    P.ws = reinterpret_cast<unsigned char *>(workspace);
    const int need = (E + 31) / 32;
    // the same experts per lane as the route kernel, so that the softmax
    // denominator is summed in the same order and the weights agree bit for bit
    cudaError_t e;
    if (need <= 1) e = launch_route_hist_j<1>(P, stream);
    else if (need <= 2) e = launch_route_hist_j<2>(P, stream);
    else if (need <= 4) e = launch_route_hist_j<4>(P, stream);
    else if (need <= 8) e = launch_route_hist_j<8>(P, stream);
    else if (need <= 12) e = launch_route_hist_j<12>(P, stream);
    else e = launch_route_hist_j<16>(P, stream);
    if (e != cudaSuccess) return e;
    const WsLayout wl = ws_layout(N, T, E);
    D->topk_idx = topk_idx;
    D->expert_offsets = expert_offsets;
    D->chunk_prefix = reinterpret_cast<const uint16_t *>(P.ws + wl.cpre);
    D->block_hist = P.ws + wl.hist;
    D->block_send = reinterpret_cast<const uint16_t *>(P.ws + wl.sd);
    D->send_counts = send_counts;
    D->N = N;
    D->T = T;
    D->ranks_per_block = P.geo.rpb;
    D->blocks_per_rank = P.geo.cps;
    D->L = E / N;
    D->Ep = pad16(E);
    D->cap = (int)cap;
    D->route_blocks = P.geo.B;
    return cudaSuccess;
}

int64_t fused_workspace_bytes(int N, int T, int E) {
    if ((int64_t)N * T == 0 || two_kernel_unsupported(N, T, E, 1)[0] != '\0') return 0;
    return ws_layout(N, T, E).bytes;
}

// A batch runs fused if the single-cluster kernel takes it (no limit on T
// or R beyond the interface's) or else the two-kernel form does.
const char *fused_unsupported(int N, int T, int E, int R, int64_t row_bytes) {
    if ((int64_t)N * T == 0) return "";  // empty batch: only the (zero) counts are written
    if (dispatch_small_eligible((int64_t)N * T, E, R, row_bytes)) return "";
    return two_kernel_unsupported(N, T, E, R);
}

cudaError_t launch_dispatch_fused(const float *logits, const float *bias, int score_fn, int renormalize,
                                  const void *x, const float *x_scales, int N, int T, int E, int R,
                                  int64_t row_bytes, int spr, int64_t cap, int32_t *topk_idx,
                                  float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                                  int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts,
                                  int32_t *pos, int32_t *status, void *packed_x, float *packed_scales,
                                  int32_t *packed_src, void *workspace, cudaStream_t stream) {
    // An empty batch has nothing to route or pack: the count step alone
    // writes its zero counts and offsets and MOE_OK, as the separate calls do.
    if ((int64_t)N * T == 0)
        return launch_dispatch_count(topk_idx, N, T, E, R, cap, expert_counts, expert_offsets, rank_counts,
                                     rank_offsets, send_counts, pos, status, stream);
    // Small batches: one thread-block cluster, no workspace (the two-kernel
    // form below handles everything else, and takes over if the device
    // cannot schedule the cluster).
    if (dispatch_small_eligible((int64_t)N * T, E, R, row_bytes)) {
        cudaError_t e = launch_dispatch_small(logits, bias, score_fn, renormalize, x, x_scales, N, T, E, R,
                                              row_bytes, spr, cap, topk_idx, topk_w, expert_counts,
                                              expert_offsets, rank_counts, rank_offsets, send_counts, pos,
                                              status, packed_x, packed_scales, packed_src, stream);
        if (e != cudaErrorNotSupported) return e;
        if (two_kernel_unsupported(N, T, E, R)[0] != '\0') return cudaErrorNotSupported;
    }
    PackDerive D;
    cudaError_t e = launch_route_hist(logits, bias, score_fn, renormalize, N, T, E, R, cap, topk_idx, topk_w,
                                      expert_counts, expert_offsets, rank_counts, rank_offsets, send_counts, pos,
                                      status, workspace, stream, &D);
    if (e != cudaSuccess) return e;
    return launch_dispatch_pack_derive(x, x_scales, pos, (int64_t)N * T, R, row_bytes, spr, (int64_t)N * cap, D,
                                       packed_x, packed_scales, packed_src, stream);
}

const char *fused_quant_unsupported(int N, int T, int E, int R) {
    if ((int64_t)N * T == 0) return "";
    return two_kernel_unsupported(N, T, E, R);
}

cudaError_t launch_dispatch_fused_quant(const float *logits, const float *bias, int score_fn, int renormalize,
                                        const void *x, int N, int T, int E, int R, int H, int64_t cap,
                                        int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                                        int32_t *expert_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                                        int32_t *send_counts, int32_t *pos, int32_t *status, void *packed_q,
                                        float *packed_scales, int32_t *packed_src, void *workspace,
                                        cudaStream_t stream) {
    if ((int64_t)N * T == 0)
        return launch_dispatch_count(topk_idx, N, T, E, R, cap, expert_counts, expert_offsets, rank_counts,
                                     rank_offsets, send_counts, pos, status, stream);
    PackDerive D;
    cudaError_t e = launch_route_hist(logits, bias, score_fn, renormalize, N, T, E, R, cap, topk_idx, topk_w,
                                      expert_counts, expert_offsets, rank_counts, rank_offsets, send_counts, pos,
                                      status, workspace, stream, &D);
    if (e != cudaSuccess) return e;
    return launch_dispatch_pack_quant_derive(x, pos, (int64_t)N * T, R, H, (int64_t)N * cap, D, packed_q,
                                             packed_scales, packed_src, stream);
}

}  // namespace moe

// ---- self-test of a bounded wait --------------------------------------------
//
// A kernel that waits on a device word must give up after a bounded number
// of polls and report it instead of hanging.  Here one thread waits for
// status[1] to become nonzero (acquire loads, a sleep of 32 ns doubling to
// 128 ns between polls, at most `polls` polls); status[0] gets MOE_OK if it
// did and MOE_ERR_TIMEOUT if the wait gave up.  Nothing in the library
// writes status[1], so unless the caller set it beforehand the wait runs
// out: this shows on a given GPU that a wait which is never satisfied ends
// with a status the host can read, and leaves the context usable.
namespace moe {
namespace {

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Polls *word until it differs from `value`, at most `limit` times; false
// if it gave up.
__device__ bool wait_while_equal(const int *word, int value, long long limit) {
    long long it = 0;
    unsigned ns = 32;
    while (ld_acquire(word) == value) {
        if (++it > limit) return false;
        __nanosleep(ns);
        if (ns < 128) ns <<= 1;
    }
    return true;
}

__global__ void selftest_wait_kernel(int *status, long long polls) {
    if (threadIdx.x == 0 && blockIdx.x == 0)
        status[0] = wait_while_equal(status + 1, 0, polls) ? MOE_OK : MOE_ERR_TIMEOUT;
}
}  // namespace

cudaError_t launch_selftest_wait(int32_t *status, long long polls, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, polls);
    return cudaGetLastError();
}
}  // namespace moe

// ---- allocation-free variant -------------------------------------------------
//
// Some callers cannot allocate device memory at the point where they
// dispatch: a plug-in running inside another framework's execution loop has
// no allocator of its own, and serving code whose memory is fixed at
// start-up must not call cudaMalloc on its hot path (it synchronises the
// device and can fail under memory pressure).  For them the fused dispatch
// can use scratch that lives in the library itself: a fixed array in device
// memory, reserved on every GPU that loads the library for as long as the
// process runs.  Its size covers the workspace of every batch the fused
// dispatch accepts (N*T <= 4096 and E <= 512 need at most 216,064 bytes:
// N = 124, T = 33, E = 496), and it starts zero-filled, as the fused
// kernels require of a workspace before its first use.
namespace moe {

constexpr int64_t kStaticScratchBytes = 256 * 1024;
static __device__ __align__(256) unsigned char g_fused_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;

// The array's address belongs to the CUDA context the library's module was
// loaded into.  After cudaDeviceReset (or any other end of the primary
// context) the module is loaded again into a new context, possibly at
// another address, so the cached address is keyed on the context's unique
// id as well as on the device.
struct ScratchEntry {
    void *addr;
    unsigned long long ctx_id;
};
ScratchEntry g_scratch[kMaxScratchDevices] = {};

}  // namespace

int64_t fused_static_scratch_bytes() { return kStaticScratchBytes; }

// Device address of the scratch array in the current device's context.  In
// host code the array's name only stands in for it, so the address is
// looked up with the device current, once per context, and cached.  Where
// the driver cannot identify the context the lookup is simply repeated on
// every call.
cudaError_t fused_static_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    const unsigned long long id = context_key();
    if (id != 0 && g_scratch[dev].addr != nullptr && g_scratch[dev].ctx_id == id) {
        *out = g_scratch[dev].addr;
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fused_static_scratch);  // creates the context if needed
    if (e != cudaSuccess) return e;
    const unsigned long long id2 = context_key();
    if (id2 != 0) g_scratch[dev] = ScratchEntry{p, id2};
    *out = p;
    return cudaSuccess;
}

}  // namespace moe
