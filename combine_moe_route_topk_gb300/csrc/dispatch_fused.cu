// Decode-fused dispatch: route top-k, dispatch count and dispatch pack in
// one call, as two kernels: route and count in ONE cooperative launch, then
// the pack kernel of dispatch_pack.cu, launched with programmatic dependent
// launch so that it is scheduled while the first one runs.
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
// The route-count grid is G co-resident blocks (two per SM, launched
// cooperatively so that all of them are resident at once); block b owns the
// contiguous tokens [b*NT/G, (b+1)*NT/G), at most 32 of them.
//   1. route: one warp per token of the block; the selections stay in
//      shared memory, and a 32-bit mask per expert marks the block's tokens
//      that chose it (a pair's rank among the block's pairs of its expert is
//      a population count of the mask below its token);
//   2. count: the block publishes its per-expert histogram (one byte per
//      expert) to the workspace and takes a ticket from an arrival counter
//      (an acquire-release atomic after a block barrier).  The block that
//      draws the last ticket sums the histograms in chunks of 16 blocks,
//      scans the chunk sums into per-chunk prefixes and the expert totals
//      into the offsets, writes the count outputs and releases the others by
//      bumping a generation word.  The other blocks meanwhile bring their
//      own x rows into L2 (bulk prefetch, evict-last) and then wait for the
//      generation word to change (bounded);
//   3. rows: each block finishes the rows of its own pairs -- expert start
//      + its chunk's prefix + the histograms of the earlier blocks of its
//      chunk + the rank inside the block -- and writes pos and its send
//      counts.
// Nothing waits for more than one event: no grid-wide barrier, and the
// histogram exchange is one round trip through L2.  The wait is bounded: a
// wait that gives up leaves MOE_ERR_TIMEOUT in the status word.  The pack
// kernel, whose 4096 one-token blocks the hardware spreads over the SMs as
// they free up, then copies the rows from L2.  A single kernel that also
// packed (each block its own tokens) took 104 us on the DeepSeek-V3 decode
// batch: with a fixed share of tokens per block its blocks finished between
// 58 and 97 us.
//
// Scope: decode batches (N*T <= 4096), R <= 16, E <= 512; the host rejects
// anything else with MOE_ERR_UNSUPPORTED (use the three separate calls).
#include <mutex>

#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "route_impl.cuh"

namespace moe {
namespace {

constexpr int kCThreads = 512;                 // 16 warps
constexpr int kCWarps = kCThreads / 32;
constexpr int kCMaxTok = 32;                   // tokens per block (32-bit masks)
constexpr int kCMaxR = 16;                     // pairs per block <= 512 = threads
constexpr int kCMaxE = 512;
constexpr int kCMaxGrid = 320;                 // blocks the workspace is sized for
constexpr int kChunk = 16;                     // blocks per prefix chunk
constexpr int kMaxChunks = kCMaxGrid / kChunk;
constexpr int kCMaxNT = 4096;
constexpr int kSendSmem = 2048;                // ints of send-count staging per block
constexpr long long kSpinLimit = 1ll << 20;    // polls of the release wait (well under a second)

// workspace: words of the arrival counter, generation and error flag in
// separate 128-byte lines, then the byte histograms, the chunk prefixes
// (u16) and the expert offsets
constexpr int kWsArrive = 0, kWsGen = 32, kWsError = 64;
constexpr int kWsHeaderBytes = 512;

__host__ __device__ inline int pad16(int v) { return (v + 15) & ~15; }
__host__ __device__ inline int64_t ws_hist_off() { return kWsHeaderBytes; }
__host__ __device__ inline int64_t ws_cpre_off(int E) { return ws_hist_off() + (int64_t)kCMaxGrid * pad16(E); }
__host__ __device__ inline int64_t ws_eoff_off(int E) { return ws_cpre_off(E) + (int64_t)kMaxChunks * pad16(E) * 2; }
__host__ __device__ inline int64_t ws_bytes(int E) { return ws_eoff_off(E) + pad16((E + 1) * 4); }

struct FusedParams {
    const float *logits;
    const float *bias;
    int score_fn, renormalize;
    const uint4 *x;
    const float *x_scales;
    int nvec, spr;
    int N, T, E, R, cap;
    int64_t rows_total;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *expert_counts, *expert_offsets, *rank_counts, *rank_offsets, *send_counts, *pos,
        *status;
    uint4 *packed_x;
    float *packed_scales;
    int32_t *packed_src;
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

__device__ __forceinline__ void red_add_release(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Polls *word until it differs from `value`, at most `limit` times with a
// growing sleep between polls (32 ns doubling to 128 ns); false if it gave up.
__device__ bool wait_while_equal(const int *word, int value, long long limit) {
    long long it = 0;
    unsigned ns = 32;
    while (ld_acquire(word) == value) {
        if (++it > limit) return false;
        __nanosleep(ns);
        if (ns < 128) ns <<= 1;  // back off: hundreds of blocks poll one word
    }
    return true;
}

// Shared-memory layout of the cooperative kernel.  Every section starts on
// a 16-byte boundary.
struct CoopSmem {
    int mask, sel, send, csum, tot, bytes;
};

__host__ __device__ inline CoopSmem coop_smem_layout(int E) {
    CoopSmem s;
    int o = 0;
    auto take = [&o](int bytes) {
        const int at = o;
        o += pad16(bytes);
        return at;
    };
    s.mask = take(E * 4);                        // u32 per expert: tokens of the block that chose it
    s.sel = take(kCMaxTok * kCMaxR * 4);         // selected experts of the block's pairs
    s.send = take(kSendSmem * 4);                // send counts of the block's source ranks
    s.csum = take(kMaxChunks * pad16(E) * 2);    // last block: chunk sums (u16)
    s.tot = take((E + 1) * 4);                   // last block: totals, then offsets
    s.bytes = o;
    return s;
}

template <int J, bool kVec4>
__global__ void __launch_bounds__(kCThreads, 2)
route_count_kernel(FusedParams P) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_flag[4];  // [0] last ticket, [1] released, [2] generation seen at start
    __shared__ int s_wsum[kCWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NT = P.N * P.T, E = P.E, R = P.R, N = P.N, T = P.T, L = E / N;
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int Ep = pad16(E);
    const CoopSmem lay = coop_smem_layout(E);
    uint32_t *mask = reinterpret_cast<uint32_t *>(smem + lay.mask);
    int *sel = reinterpret_cast<int *>(smem + lay.sel);
    int *ssend = reinterpret_cast<int *>(smem + lay.send);
    int *ws_words = reinterpret_cast<int *>(P.ws);
    unsigned char *ws_hist = P.ws + ws_hist_off();
    uint16_t *ws_cpre = reinterpret_cast<uint16_t *>(P.ws + ws_cpre_off(E));
    int *ws_eoff = reinterpret_cast<int *>(P.ws + ws_eoff_off(E));

    const int tb = (int)((int64_t)b * NT / G), te = (int)((int64_t)(b + 1) * NT / G);
    const int ntok = te - tb;  // <= 32, checked by the launcher
    const int npair = ntok * R;
    const int s_first = tb / T;
    const int span = ntok > 0 ? (te - 1) / T - s_first + 1 : 0;
    const bool smem_send = span * N <= kSendSmem;

    // the pack kernel that follows may be scheduled now: it reads nothing of
    // this kernel's before its own grid-dependency wait
    grid_launch_dependents();
    if (tid == 0) s_flag[2] = ld_acquire(ws_words + kWsGen);  // before this block's ticket
    for (int i = tid; i < E; i += kCThreads) mask[i] = 0u;
    if (smem_send)
        for (int i = tid; i < span * N; i += kCThreads) ssend[i] = 0;
    __syncthreads();

    // ---- 1. route ---------------------------------------------------------------
    for (int t = warp; t < ntok; t += kCWarps) {
        const int e = route_impl::route_token<J, kVec4>(P.logits, P.bias, (int64_t)(tb + t), E, R, P.score_fn,
                                                        P.renormalize, P.topk_idx, P.topk_w, lane);
        if (lane < R) sel[t * R + lane] = e;
    }
    __syncthreads();
    if (tid < npair) atomicOr(mask + sel[tid], 1u << (tid / R));
    __syncthreads();

    // ---- 2. count: publish, ticket, the last block scans --------------------------
    for (int e = tid; e < Ep; e += kCThreads)
        ws_hist[(int64_t)b * Ep + e] = (unsigned char)(e < E ? __popc(mask[e]) : 0);
    __syncthreads();  // the block's histogram bytes, released by its ticket
    if (tid == 0) s_flag[0] = atomic_add_acq_rel(ws_words + kWsArrive, 1) == G - 1;
    __syncthreads();
    if (s_flag[0]) {
        // the last ticket acquired every other block's histogram
        uint16_t *csum = reinterpret_cast<uint16_t *>(smem + lay.csum);
        int *tot = reinterpret_cast<int *>(smem + lay.tot);
        const int C = (G + kChunk - 1) / kChunk;
        const int nv = Ep / 16;  // 16-byte vectors of a histogram row
        // chunk sums: item (chunk c, vector v) adds 16 blocks' 16 bytes
        for (int it = tid; it < C * nv; it += kCThreads) {
            const int c = it / nv, v = it - c * nv;
            uint4 h[kChunk];
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                const int bb = c * kChunk + j;
                h[j] = bb < G ? __ldcg(reinterpret_cast<const uint4 *>(ws_hist + (int64_t)bb * Ep) + v)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
            // bytes 0,2 / 1,3 of every word summed in 16-bit halves (a chunk
            // sum is at most 16 * 32 = 512)
            uint32_t ev[4] = {0u, 0u, 0u, 0u}, od[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                const uint32_t w4[4] = {h[j].x, h[j].y, h[j].z, h[j].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ev[q] += w4[q] & 0x00ff00ffu;
                    od[q] += (w4[q] >> 8) & 0x00ff00ffu;
                }
            }
            uint16_t *dst = csum + c * Ep + v * 16;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dst[4 * q + 0] = (uint16_t)(ev[q] & 0xffffu);
                dst[4 * q + 1] = (uint16_t)(od[q] & 0xffffu);
                dst[4 * q + 2] = (uint16_t)(ev[q] >> 16);
                dst[4 * q + 3] = (uint16_t)(od[q] >> 16);
            }
        }
        __syncthreads();
        // per expert: exclusive prefix over chunks (to the workspace) and total
        for (int e = tid; e < Ep; e += kCThreads) {
            int run = 0;
            for (int c = 0; c < C; ++c) {
                ws_cpre[c * Ep + e] = (uint16_t)run;
                run += csum[c * Ep + e];
            }
            if (e < E) tot[e] = run;
        }
        __syncthreads();
        // exclusive scan of the totals over experts (E <= 512: one per thread)
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
            int sv = lane < kCWarps ? s_wsum[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, sv, off);
                if (lane >= off) sv += y;
            }
            if (lane < kCWarps) s_wsum[lane] = sv;  // inclusive over warps
        }
        __syncthreads();
        const int excl = xs - v0 + (warp > 0 ? s_wsum[warp - 1] : 0);
        __syncthreads();  // every total read before it is overwritten
        if (tid < E) {
            tot[tid] = excl;
            P.expert_counts[tid] = v0;
            P.expert_offsets[tid] = excl;
            ws_eoff[tid] = excl;
            if (tid == E - 1) {
                tot[E] = excl + v0;
                P.expert_offsets[E] = excl + v0;
                ws_eoff[E] = excl + v0;
            }
        }
        __syncthreads();
        int over = 0;
        for (int d = tid; d < N; d += kCThreads) {
            const int rc = tot[(d + 1) * L] - tot[d * L];
            P.rank_counts[d] = rc;
            P.rank_offsets[d] = tot[d * L];
            over |= rc > P.cap;
        }
        over = __syncthreads_or(over);
        for (int i = tid; i < N * N; i += kCThreads) P.send_counts[i] = 0;  // filled after the release
        if (tid == 0) {
            P.rank_offsets[N] = tot[E];
            *P.status = over ? MOE_ERR_CAPACITY : MOE_OK;
        }
        __syncthreads();  // every thread's prefixes, offsets and zeroed send counts
        if (tid == 0) {
            atomicExch(ws_words + kWsArrive, 0);  // ready for the next launch
            red_add_release(ws_words + kWsGen, 1);  // release the others
            s_flag[1] = 1;
        }
    } else {
        // while the last block scans: this block's x rows into L2, then the wait
        if (warp == 0) {
            const uint64_t keep = l2_policy_evict_last();
            const uint32_t rb = (uint32_t)P.nvec * 16u;
            if (rb <= 65536u)
                for (int t = lane; t < ntok; t += 32) prefetch_l2(P.x + (int64_t)(tb + t) * P.nvec, rb, keep);
        }
        if (tid == 0) {
            const bool ok = wait_while_equal(ws_words + kWsGen, s_flag[2], kSpinLimit);
            if (!ok) atomicCAS(ws_words + kWsError, 0, MOE_ERR_TIMEOUT);
            s_flag[1] = ok;
        }
    }
    __syncthreads();
    if (!s_flag[1]) {
        if (tid == 0) *P.status = MOE_ERR_TIMEOUT;
        return;
    }

    // ---- 3. rows of this block's pairs, send counts -----------------------------
    if (tid < npair) {
        const int t = tid / R, k = tid - t * R;
        const int g = tb + t;
        const int e = sel[tid], d = e / L;
        const int c = b / kChunk;
        int base = __ldcg(ws_cpre + c * Ep + e);  // written by the last block before the release
        for (int bb = c * kChunk; bb < b; ++bb) base += __ldcg(ws_hist + (int64_t)bb * Ep + e);
        const int in_block = __popc(mask[e] & ((1u << t) - 1u));
        const int local = __ldcg(ws_eoff + e) - __ldcg(ws_eoff + d * L) + base + in_block;
        const int p = local < P.cap ? d * P.cap + local : -1;
        P.pos[(int64_t)g * R + k] = p;
        // counts report demand: the pair is counted whether or not it fits
        if (smem_send) atomicAdd(ssend + (g / T - s_first) * N + d, 1);
        else atomicAdd(P.send_counts + (int64_t)(g / T) * N + d, 1);
    }
    __syncthreads();
    if (smem_send)
        for (int i = tid; i < span * N; i += kCThreads)
            if (ssend[i]) atomicAdd(P.send_counts + (int64_t)(s_first + i / N) * N + (i - (i / N) * N), ssend[i]);

    // the last block's own rows (the others fetched theirs while waiting)
    if (s_flag[0] && warp == 0) {
        const uint64_t keep = l2_policy_evict_last();
        const uint32_t rb = (uint32_t)P.nvec * 16u;
        if (rb <= 65536u)
            for (int t = lane; t < ntok; t += 32) prefetch_l2(P.x + (int64_t)(tb + t) * P.nvec, rb, keep);
    }
}

template <int J, bool kVec4>
cudaError_t launch_fused_jv(FusedParams P, cudaStream_t stream) {
    auto kern = route_count_kernel<J, kVec4>;
    const size_t smem = (size_t)coop_smem_layout(P.E).bytes;
    // the shared-memory attribute and the occupancy it allows belong to the
    // current context: cached per host thread, device and context for the
    // largest request seen
    static thread_local int cached_dev = -1, cached_per_sm = 0;
    static thread_local unsigned long long cached_ctx = 0;
    static thread_local size_t cached_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = context_key();
    int per_sm = cached_per_sm;
    if (dev != cached_dev || ctx == 0 || ctx != cached_ctx || smem > cached_smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCThreads, smem);
        if (e != cudaSuccess) return e;
        cached_dev = dev;
        cached_ctx = context_key();
        cached_smem = smem;
        cached_per_sm = per_sm;
    }
    const int sms = sm_count();
    if (per_sm < 1 || sms < 1) return cudaErrorNotSupported;
    const int NT = P.N * P.T;
    int grid = sms * per_sm;
    if (grid > kCMaxGrid) grid = kCMaxGrid;
    if (grid > NT) grid = NT;
    if ((NT + grid - 1) / grid > kCMaxTok) return cudaErrorNotSupported;  // too few co-resident blocks
    e = cudaMemsetAsync(P.ws, 0, kWsHeaderBytes, stream);  // arrival counter, generation, flags
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int J>
cudaError_t launch_fused_j(FusedParams P, cudaStream_t stream) {
    if constexpr (J % 4 == 0) {
        if (P.E % 4 == 0 && (reinterpret_cast<uintptr_t>(P.logits) & 15) == 0)
            return launch_fused_jv<J, true>(P, stream);
    }
    return launch_fused_jv<J, false>(P, stream);
}

}  // namespace

int64_t fused_workspace_bytes(int E) { return ws_bytes(E); }

// Empty string when the fused kernel handles these dimensions, else why not.
namespace {
// Limits of the cooperative kernel ("" when it can run the batch).
const char *cooperative_unsupported(int N, int T, int E, int R) {
    const int64_t NT = (int64_t)N * T;
    if (R > kCMaxR) return "R > 16";
    if (E > kCMaxE) return "E > 512";
    if (NT > kCMaxNT) return "N*T > 4096 (not a decode batch)";
    (void)T;
    return "";
}
}  // namespace

// A batch runs fused if the single-cluster kernel takes it (no limit on T
// or R beyond the interface's) or else the cooperative kernel does.
const char *fused_unsupported(int N, int T, int E, int R, int64_t row_bytes) {
    if ((int64_t)N * T == 0) return "";  // empty batch: only the (zero) counts are written
    if (dispatch_small_eligible((int64_t)N * T, E, R, row_bytes)) return "";
    return cooperative_unsupported(N, T, E, R);
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
    // Small batches: one thread-block cluster, no grid-wide wait and no
    // workspace (the cooperative kernel below handles everything else, and
    // takes over if the device cannot schedule the cluster).
    if (dispatch_small_eligible((int64_t)N * T, E, R, row_bytes)) {
        cudaError_t e = launch_dispatch_small(logits, bias, score_fn, renormalize, x, x_scales, N, T, E, R,
                                              row_bytes, spr, cap, topk_idx, topk_w, expert_counts,
                                              expert_offsets, rank_counts, rank_offsets, send_counts, pos,
                                              status, packed_x, packed_scales, packed_src, stream);
        if (e != cudaErrorNotSupported) return e;
        // the device cannot schedule the cluster: the cooperative kernel, if
        // the batch is within its limits
        if (cooperative_unsupported(N, T, E, R)[0] != '\0') return cudaErrorNotSupported;
    }
    FusedParams P;
    P.logits = logits;
    P.bias = bias;
    P.score_fn = score_fn;
    P.renormalize = renormalize;
    P.x = reinterpret_cast<const uint4 *>(x);
    P.x_scales = x_scales;
    P.nvec = (int)(row_bytes / 16);
    P.spr = spr;
    P.N = N;
    P.T = T;
    P.E = E;
    P.R = R;
    P.cap = (int)cap;
    P.rows_total = (int64_t)N * cap;
    P.topk_idx = topk_idx;
    P.topk_w = topk_w;
    P.expert_counts = expert_counts;
    P.expert_offsets = expert_offsets;
    P.rank_counts = rank_counts;
    P.rank_offsets = rank_offsets;
    P.send_counts = send_counts;
    P.pos = pos;
    P.status = status;
    P.packed_x = reinterpret_cast<uint4 *>(packed_x);
    P.packed_scales = packed_scales;
    P.packed_src = packed_src;
    P.ws = reinterpret_cast<unsigned char *>(workspace);
    const int need = (E + 31) / 32;
    // the same experts per lane as the route kernel, so that the softmax
    // denominator is summed in the same order and the weights agree bit for bit
    cudaError_t e;
    if (need <= 1) e = launch_fused_j<1>(P, stream);
    else if (need <= 2) e = launch_fused_j<2>(P, stream);
    else if (need <= 4) e = launch_fused_j<4>(P, stream);
    else if (need <= 8) e = launch_fused_j<8>(P, stream);
    else if (need <= 12) e = launch_fused_j<12>(P, stream);
    else e = launch_fused_j<16>(P, stream);
    if (e != cudaSuccess) return e;
    // pack: scheduled while the cooperative kernel runs, it waits for it
    // (rows from pos) and then copies from L2 the x rows that the route-count
    // blocks prefetched while they waited
    return launch_dispatch_pack(x, x_scales, pos, (int64_t)N * T, R, row_bytes, spr, (int64_t)N * cap,
                                packed_x, packed_scales, packed_src, stream);
}

}  // namespace moe

// ---- self-test of the bounded wait -----------------------------------------
//
// One thread waits, through the same bounded poll as the route-count
// kernel's release wait, for status[1] to become nonzero; status[0] gets
// MOE_OK if it did and
// MOE_ERR_TIMEOUT if the wait gave up.  Nothing in the library writes
// status[1], so unless the caller set it beforehand the wait runs out: this
// shows on a given GPU that a wait which is never satisfied ends with a
// status the host can read, and leaves the context usable.
namespace moe {
namespace {
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
// kernel accepts (E <= 512 needs at most 164,288 bytes).
namespace moe {

constexpr int64_t kStaticScratchBytes = 192 * 1024;
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
