// C entry points of libmoe_route.so: argument validation on the host, then
// one launcher per step.  See include/moe_route.h for the contract.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>  // CUcontext and CUresult only: the two driver calls are fetched at run time

#include "moe_internal.cuh"

namespace moe {

namespace {
thread_local char g_err[512] = "";
}

int set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

namespace {
// Driver functions fetched through the runtime (no link against libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
struct CtxFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
    CtxFns() {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();
    }
};
}  // namespace

unsigned long long context_key() {
    static const CtxFns fns;  // initialised once, thread-safe
    if (fns.get_current == nullptr || fns.get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id + 1;  // never 0 for a real context
}

int sm_count() {
    static thread_local int dev_cached = -1, sms = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev != dev_cached) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 0;
        dev_cached = dev;
    }
    return sms;
}

int64_t l2_bytes() {
    static thread_local int dev_cached = -1, l2 = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev != dev_cached) {
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) l2 = 0;
        dev_cached = dev;
    }
    return l2;
}

namespace {

constexpr int64_t kI32Max = 2147483647;

struct Derived {
    int64_t NT, cap, rows_total, pairs, x_row_bytes, y_row_bytes;
    int scales_per_row;
};

int elem_bytes(int dtype) {
    switch (dtype) {
        case MOE_BF16: return 2;
        case MOE_F32: return 4;
        case MOE_FP8E4M3_BLK128: return 1;
        default: return 0;
    }
}

// Validates dims and fills the derived sizes.  `what` names the caller.
int check_dims(const MoeDims *d, Derived *out, const char *what) {
    g_err[0] = '\0';
    if (d == nullptr) return set_error(MOE_ERR_INVALID_ARG, "%s: dims is NULL", what);
    if (d->N < 1 || d->T < 0 || d->E < 1 || d->R < 1 || d->H < 1)
        return set_error(MOE_ERR_INVALID_ARG, "%s: need N>=1, T>=0, E>=1, R>=1, H>=1 (got N=%d T=%d E=%d R=%d H=%d)",
                         what, d->N, d->T, d->E, d->R, d->H);
    if (d->E % d->N != 0)
        return set_error(MOE_ERR_INVALID_ARG, "%s: E=%d is not a multiple of N=%d", what, d->E, d->N);
    if (d->R > d->E)
        return set_error(MOE_ERR_INVALID_ARG, "%s: R=%d exceeds E=%d", what, d->R, d->E);
    if (d->E > 1024 || d->R > 32)
        return set_error(MOE_ERR_UNSUPPORTED, "%s: this build supports E<=1024 and R<=32 (got E=%d R=%d)",
                         what, d->E, d->R);
    if (d->reserved != 0) return set_error(MOE_ERR_INVALID_ARG, "%s: dims.reserved must be 0", what);
    if (elem_bytes(d->x_dtype) == 0)
        return set_error(MOE_ERR_INVALID_ARG, "%s: unknown x_dtype %d", what, d->x_dtype);
    if (d->y_dtype != MOE_BF16 && d->y_dtype != MOE_F32)
        return set_error(MOE_ERR_INVALID_ARG, "%s: y_dtype must be MOE_BF16 or MOE_F32 (got %d)", what,
                         d->y_dtype);
    if (d->H % 8 != 0)
        return set_error(MOE_ERR_INVALID_ARG, "%s: H=%d must be a multiple of 8", what, d->H);
    if (d->H > (1 << 24))  // keeps per-row vector counts and in-row indices in 32 bits
        return set_error(MOE_ERR_UNSUPPORTED, "%s: this build supports H <= 2^24 (got H=%d)", what, d->H);
    if (d->x_dtype == MOE_FP8E4M3_BLK128 && d->H % 128 != 0)
        return set_error(MOE_ERR_INVALID_ARG, "%s: fp8 rows need H %% 128 == 0 (got H=%d)", what, d->H);
    if (d->cap_rows < 0) return set_error(MOE_ERR_INVALID_ARG, "%s: cap_rows < 0", what);
    Derived v;
    v.NT = (int64_t)d->N * d->T;
    const int64_t L = d->E / d->N;
    const int64_t bound = v.NT * (d->R > L ? d->R : L);
    v.cap = d->cap_rows > 0 ? d->cap_rows : bound;
    if (v.cap < 1) v.cap = 1;  // T == 0: keep the region arithmetic well defined
    v.pairs = v.NT * d->R;
    v.rows_total = (int64_t)d->N * v.cap;
    if (v.pairs > kI32Max || v.rows_total > kI32Max || v.NT > kI32Max - 65536)
        return set_error(MOE_ERR_UNSUPPORTED,
                         "%s: N*T*R=%lld and N*cap=%lld must stay below 2^31 (32-bit row indices)",
                         what, (long long)v.pairs, (long long)v.rows_total);
    v.x_row_bytes = (int64_t)d->H * elem_bytes(d->x_dtype);
    v.y_row_bytes = (int64_t)d->H * elem_bytes(d->y_dtype);
    v.scales_per_row = d->x_dtype == MOE_FP8E4M3_BLK128 ? d->H / 128 : 0;
    if (out) *out = v;
    return MOE_OK;
}

// Pack kernel choice: the register-path kernel by default (the faster of
// the two on GB300 at R = 8); the environment variable MOE_PACK_KERNEL=bulk
// selects bulk copies through shared memory (read once per process).
bool use_bulk_pack() {
    static const bool bulk = [] {
        const char *v = getenv("MOE_PACK_KERNEL");
        return v && strcmp(v, "bulk") == 0;
    }();
    return bulk;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int cuda_result(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MOE_OK;
    return set_error(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return MOE_VERSION; }

const char *moe_last_error(void) { return g_err; }

int moe_buffer_sizes(const MoeDims *dims, MoeSizes *out) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_buffer_sizes");
    if (rc != MOE_OK) return rc;
    if (out == nullptr) return set_error(MOE_ERR_INVALID_ARG, "moe_buffer_sizes: out is NULL");
    const int64_t N = dims->N, E = dims->E, H = dims->H;
    const int64_t L = E / N;
    memset(out, 0, sizeof(*out));
    out->bound_rows = v.NT * (dims->R > L ? dims->R : L);
    out->cap_rows = v.cap;
    out->total_pairs = v.pairs;
    out->logits_bytes = v.NT * E * 4;
    out->topk_idx_bytes = v.pairs * 4;
    out->topk_w_bytes = v.pairs * 4;
    out->pos_bytes = v.pairs * 4;
    out->expert_counts_bytes = E * 4;
    out->expert_offsets_bytes = (E + 1) * 4;
    out->rank_counts_bytes = N * 4;
    out->rank_offsets_bytes = (N + 1) * 4;
    out->send_counts_bytes = N * N * 4;
    out->x_bytes = v.NT * v.x_row_bytes;
    out->x_scales_bytes = v.NT * v.scales_per_row * 4;
    out->packed_x_bytes = v.rows_total * v.x_row_bytes;
    out->packed_scales_bytes = v.rows_total * v.scales_per_row * 4;
    out->packed_src_bytes = v.rows_total * 4;
    out->y_bytes = v.rows_total * v.y_row_bytes;
    out->out_bytes = v.NT * v.y_row_bytes;
    out->status_bytes = 4;
    out->partial_slots = dims->R < N ? dims->R : N;
    out->partial_bytes = v.NT * out->partial_slots * v.y_row_bytes;
    out->slot_rank_bytes = v.NT * out->partial_slots * 4;
    out->fused_workspace_bytes = fused_workspace_bytes(dims->N, dims->T, dims->E);
    (void)H;
    return MOE_OK;
}

static bool valid_score_fn(int score_fn) {
    const int fn = score_fn & ~MOE_BIAS_SELECT_ONLY;
    return fn == MOE_SOFTMAX || fn == MOE_SIGMOID;
}

int moe_route_topk(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                   int renormalize, int32_t *topk_idx, float *topk_w, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_route_topk");
    if (rc != MOE_OK) return rc;
    if (!valid_score_fn(score_fn))
        return set_error(MOE_ERR_INVALID_ARG, "moe_route_topk: unknown score_fn %d", score_fn);
    if (v.NT == 0) return MOE_OK;
    if (!logits || !topk_idx || !topk_w)
        return set_error(MOE_ERR_INVALID_ARG, "moe_route_topk: logits, topk_idx and topk_w must be non-NULL");
    if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) || (bias && !aligned(bias, 4)))
        return set_error(MOE_ERR_INVALID_ARG, "moe_route_topk: pointers must be 4-byte aligned");
    return cuda_result(launch_route_topk(logits, bias, v.NT, dims->E, dims->R, score_fn, renormalize ? 1 : 0,
                                         topk_idx, topk_w, (cudaStream_t)stream),
                       "moe_route_topk");
}

int moe_dispatch_count(const MoeDims *dims, const int32_t *topk_idx, int32_t *expert_counts,
                       int32_t *expert_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                       int32_t *send_counts, int32_t *pos, int32_t *status, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_dispatch_count");
    if (rc != MOE_OK) return rc;
    if (!expert_counts || !expert_offsets || !rank_counts || !rank_offsets || !send_counts || !status ||
        (v.NT > 0 && (!topk_idx || !pos)))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_count: a required pointer is NULL");
    const void *ptrs[] = {topk_idx, expert_counts, expert_offsets, rank_counts, rank_offsets,
                          send_counts, pos, status};
    for (const void *p : ptrs)
        if (p && !aligned(p, 4))
            return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_count: pointers must be 4-byte aligned");
    cudaError_t e = launch_dispatch_count(topk_idx, dims->N, dims->T, dims->E, dims->R, v.cap,
                                          expert_counts, expert_offsets, rank_counts, rank_offsets,
                                          send_counts, pos, status, (cudaStream_t)stream);
    if (e == cudaErrorNotSupported)
        return set_error(MOE_ERR_UNSUPPORTED,
                         "moe_dispatch_count: the device cannot schedule a thread-block cluster of this kernel");
    return cuda_result(e, "moe_dispatch_count");
}

int moe_dispatch_pack(const MoeDims *dims, const void *x, const float *x_scales, const int32_t *pos,
                      void *packed_x, float *packed_scales, int32_t *packed_src, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_dispatch_pack");
    if (rc != MOE_OK) return rc;
    if (v.NT == 0) return MOE_OK;
    const bool fp8 = dims->x_dtype == MOE_FP8E4M3_BLK128;
    if (!x || !pos || !packed_x || !packed_src || (fp8 && (!x_scales || !packed_scales)))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack: a required pointer is NULL");
    if (!aligned(x, 16) || !aligned(packed_x, 16))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack: x and packed_x must be 16-byte aligned");
    if (!aligned(pos, 4) || !aligned(packed_src, 4) || (fp8 && (!aligned(x_scales, 4) || !aligned(packed_scales, 4))))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack: index and scale pointers must be 4-byte aligned");
    if (use_bulk_pack() && pack_bulk_stages(v.x_row_bytes) > 0)
        return cuda_result(launch_dispatch_pack_bulk(x, fp8 ? x_scales : nullptr, pos, v.NT, dims->R,
                                                     v.x_row_bytes, v.scales_per_row, v.rows_total, packed_x,
                                                     fp8 ? packed_scales : nullptr, packed_src,
                                                     (cudaStream_t)stream),
                           "moe_dispatch_pack");
    return cuda_result(launch_dispatch_pack(x, fp8 ? x_scales : nullptr, pos, v.NT, dims->R, v.x_row_bytes,
                                            v.scales_per_row, v.rows_total, packed_x,
                                            fp8 ? packed_scales : nullptr, packed_src,
                                            (cudaStream_t)stream),
                       "moe_dispatch_pack");
}

int moe_dispatch_pack_quant(const MoeDims *dims, const void *x, const int32_t *pos, void *packed_q,
                            float *packed_scales, int32_t *packed_src, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_dispatch_pack_quant");
    if (rc != MOE_OK) return rc;
    if (dims->x_dtype != MOE_BF16)
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_quant: x_dtype must be MOE_BF16 (the rows it reads)");
    if (dims->H % 128 != 0)
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_quant: H=%d must be a multiple of 128", dims->H);
    if (v.NT == 0) return MOE_OK;
    if (!x || !pos || !packed_q || !packed_scales || !packed_src)
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_quant: a required pointer is NULL");
    if (!aligned(x, 16) || !aligned(packed_q, 16))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_quant: x and packed_q must be 16-byte aligned");
    if (!aligned(pos, 4) || !aligned(packed_scales, 4) || !aligned(packed_src, 4))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_quant: pos, packed_scales and packed_src must be 4-byte aligned");
    return cuda_result(launch_dispatch_pack_quant(x, pos, v.NT, dims->R, dims->H, v.rows_total, packed_q,
                                                  packed_scales, packed_src, (cudaStream_t)stream),
                       "moe_dispatch_pack_quant");
}

int moe_combine(const MoeDims *dims, const void *y, const int32_t *pos, const float *topk_w, void *out,
                void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_combine");
    if (rc != MOE_OK) return rc;
    if (v.NT == 0) return MOE_OK;
    if (!y || !pos || !topk_w || !out)
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine: a required pointer is NULL");
    if (!aligned(y, 16) || !aligned(out, 16))
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine: y and out must be 16-byte aligned");
    if (!aligned(pos, 4) || !aligned(topk_w, 4))
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine: pos and topk_w must be 4-byte aligned");
    return cuda_result(launch_combine(y, dims->y_dtype, pos, topk_w, v.NT, dims->R, dims->H, v.rows_total,
                                      out, (cudaStream_t)stream),
                       "moe_combine");
}

int moe_dispatch_pack_rank(const MoeDims *dims, int rank, const void *x, const float *x_scales,
                           const int32_t *pos, void *packed_x, float *packed_scales,
                           int32_t *packed_src, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_dispatch_pack_rank");
    if (rc != MOE_OK) return rc;
    if (rank < 0 || rank >= dims->N)
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_rank: rank %d outside [0, %d)", rank, dims->N);
    if (v.NT == 0) return MOE_OK;
    const bool fp8 = dims->x_dtype == MOE_FP8E4M3_BLK128;
    if (!x || !pos || !packed_x || !packed_src || (fp8 && (!x_scales || !packed_scales)))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_rank: a required pointer is NULL");
    if (!aligned(x, 16) || !aligned(packed_x, 16))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_rank: x and packed_x must be 16-byte aligned");
    if (!aligned(pos, 4) || !aligned(packed_src, 4) || (fp8 && (!aligned(x_scales, 4) || !aligned(packed_scales, 4))))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_pack_rank: index and scale pointers must be 4-byte aligned");
    return cuda_result(launch_pack_rank(x, fp8 ? x_scales : nullptr, pos, v.NT, dims->R, v.x_row_bytes,
                                        v.scales_per_row, (int64_t)rank * v.cap, (int64_t)(rank + 1) * v.cap,
                                        packed_x, fp8 ? packed_scales : nullptr, packed_src,
                                        (cudaStream_t)stream),
                       "moe_dispatch_pack_rank");
}

int moe_combine_rank(const MoeDims *dims, int rank, const void *y, const int32_t *pos,
                     const float *topk_w, void *out, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_combine_rank");
    if (rc != MOE_OK) return rc;
    if (rank < 0 || rank >= dims->N)
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_rank: rank %d outside [0, %d)", rank, dims->N);
    if (v.NT == 0) return MOE_OK;
    if (!y || !pos || !topk_w || !out)
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_rank: a required pointer is NULL");
    if (!aligned(y, 16) || !aligned(out, 16))
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_rank: y and out must be 16-byte aligned");
    if (!aligned(pos, 4) || !aligned(topk_w, 4))
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_rank: pos and topk_w must be 4-byte aligned");
    return cuda_result(launch_combine_rank(y, dims->y_dtype, pos, topk_w, v.NT, dims->R, dims->H,
                                           (int64_t)rank * v.cap, (int64_t)(rank + 1) * v.cap, out,
                                           (cudaStream_t)stream),
                       "moe_combine_rank");
}

int moe_combine_partials(const MoeDims *dims, const void *y, const int32_t *pos,
                         const float *topk_w, void *partial, int32_t *slot_rank, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_combine_partials");
    if (rc != MOE_OK) return rc;
    if (v.NT == 0) return MOE_OK;
    if (!y || !pos || !topk_w || !partial || !slot_rank)
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_partials: a required pointer is NULL");
    if (!aligned(y, 16) || !aligned(partial, 16))
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_partials: y and partial must be 16-byte aligned");
    if (!aligned(pos, 4) || !aligned(topk_w, 4) || !aligned(slot_rank, 4))
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_partials: pos, topk_w and slot_rank must be 4-byte aligned");
    const int P = dims->R < dims->N ? dims->R : dims->N;
    return cuda_result(launch_combine_partials(y, dims->y_dtype, pos, topk_w, v.NT, dims->R, dims->H, v.cap,
                                               v.rows_total, P, partial, slot_rank, (cudaStream_t)stream),
                       "moe_combine_partials");
}

int moe_combine_reduce_partials(const MoeDims *dims, const void *partial, const int32_t *slot_rank,
                                void *out, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_combine_reduce_partials");
    if (rc != MOE_OK) return rc;
    if (v.NT == 0) return MOE_OK;
    if (!partial || !slot_rank || !out)
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_reduce_partials: a required pointer is NULL");
    if (!aligned(partial, 16) || !aligned(out, 16) || !aligned(slot_rank, 4))
        return set_error(MOE_ERR_INVALID_ARG, "moe_combine_reduce_partials: misaligned pointer");
    const int P = dims->R < dims->N ? dims->R : dims->N;
    return cuda_result(launch_reduce_partials(partial, dims->y_dtype, slot_rank, v.NT, P, dims->H, out,
                                              (cudaStream_t)stream),
                       "moe_combine_reduce_partials");
}

int moe_dispatch_fused(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                       int renormalize, const void *x, const float *x_scales, int32_t *topk_idx,
                       float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                       int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts, int32_t *pos,
                       int32_t *status, void *packed_x, float *packed_scales, int32_t *packed_src,
                       void *workspace, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_dispatch_fused");
    if (rc != MOE_OK) return rc;
    if (!valid_score_fn(score_fn))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused: unknown score_fn %d", score_fn);
    const char *why = fused_unsupported(dims->N, dims->T, dims->E, dims->R, v.x_row_bytes);
    if (why[0] != '\0')
        return set_error(MOE_ERR_UNSUPPORTED, "moe_dispatch_fused: %s; use the separate calls", why);
    const bool fp8 = dims->x_dtype == MOE_FP8E4M3_BLK128;
    // an empty batch touches no workspace (its size is 0 there): NULL is fine
    if (!expert_counts || !expert_offsets || !rank_counts || !rank_offsets || !send_counts || !status ||
        (!workspace && v.NT > 0))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused: a required pointer is NULL");
    if (v.NT > 0 && (!logits || !x || !topk_idx || !topk_w || !pos || !packed_x || !packed_src ||
                     (fp8 && (!x_scales || !packed_scales))))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused: a required pointer is NULL");
    if ((x && !aligned(x, 16)) || (packed_x && !aligned(packed_x, 16)) || (workspace && !aligned(workspace, 16)))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused: x, packed_x and workspace must be 16-byte aligned");
    const void *ptrs4[] = {logits, bias, topk_idx, topk_w, expert_counts, expert_offsets, rank_counts,
                           rank_offsets, send_counts, pos, status, packed_src, x_scales, packed_scales};
    for (const void *p : ptrs4)
        if (p && !aligned(p, 4))
            return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused: pointers must be 4-byte aligned");
    cudaError_t e = launch_dispatch_fused(logits, bias, score_fn, renormalize ? 1 : 0, x, fp8 ? x_scales : nullptr,
                                          dims->N, dims->T, dims->E, dims->R, v.x_row_bytes, v.scales_per_row,
                                          v.cap, topk_idx, topk_w, expert_counts, expert_offsets, rank_counts,
                                          rank_offsets, send_counts, pos, status, packed_x,
                                          fp8 ? packed_scales : nullptr, packed_src, workspace,
                                          (cudaStream_t)stream);
    if (e == cudaErrorNotSupported)
        return set_error(MOE_ERR_UNSUPPORTED, "moe_dispatch_fused: the device cannot run this batch fused "
                                              "(thread-block cluster unavailable)");
    return cuda_result(e, "moe_dispatch_fused");
}

int moe_dispatch_fused_quant(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                             int renormalize, const void *x, int32_t *topk_idx, float *topk_w,
                             int32_t *expert_counts, int32_t *expert_offsets, int32_t *rank_counts,
                             int32_t *rank_offsets, int32_t *send_counts, int32_t *pos, int32_t *status,
                             void *packed_q, float *packed_scales, int32_t *packed_src, void *workspace,
                             void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_dispatch_fused_quant");
    if (rc != MOE_OK) return rc;
    if (!valid_score_fn(score_fn))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused_quant: unknown score_fn %d", score_fn);
    if (dims->x_dtype != MOE_BF16)
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused_quant: x_dtype must be MOE_BF16 (the rows it reads)");
    if (dims->H % 128 != 0)
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused_quant: H=%d must be a multiple of 128", dims->H);
    const char *why = fused_quant_unsupported(dims->N, dims->T, dims->E, dims->R);
    if (why[0] != '\0')
        return set_error(MOE_ERR_UNSUPPORTED, "moe_dispatch_fused_quant: %s; use the separate calls", why);
    // an empty batch touches no workspace (its size is 0 there): NULL is fine
    if (!expert_counts || !expert_offsets || !rank_counts || !rank_offsets || !send_counts || !status ||
        (!workspace && v.NT > 0))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused_quant: a required pointer is NULL");
    if (v.NT > 0 && (!logits || !x || !topk_idx || !topk_w || !pos || !packed_q || !packed_scales || !packed_src))
        return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused_quant: a required pointer is NULL");
    if ((x && !aligned(x, 16)) || (packed_q && !aligned(packed_q, 16)) || (workspace && !aligned(workspace, 16)))
        return set_error(MOE_ERR_INVALID_ARG,
                         "moe_dispatch_fused_quant: x, packed_q and workspace must be 16-byte aligned");
    const void *ptrs4[] = {logits, bias, topk_idx, topk_w, expert_counts, expert_offsets, rank_counts,
                           rank_offsets, send_counts, pos, status, packed_scales, packed_src};
    for (const void *p : ptrs4)
        if (p && !aligned(p, 4))
            return set_error(MOE_ERR_INVALID_ARG, "moe_dispatch_fused_quant: pointers must be 4-byte aligned");
    return cuda_result(launch_dispatch_fused_quant(logits, bias, score_fn, renormalize ? 1 : 0, x, dims->N, dims->T,
                                                   dims->E, dims->R, dims->H, v.cap, topk_idx, topk_w,
                                                   expert_counts, expert_offsets, rank_counts, rank_offsets,
                                                   send_counts, pos, status, packed_q, packed_scales, packed_src,
                                                   workspace, (cudaStream_t)stream),
                       "moe_dispatch_fused_quant");
}

int moe_dispatch_fused_static(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                              int renormalize, const void *x, const float *x_scales, int32_t *topk_idx,
                              float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                              int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts,
                              int32_t *pos, int32_t *status, void *packed_x, float *packed_scales,
                              int32_t *packed_src, void *stream) {
    Derived v;
    int rc = check_dims(dims, &v, "moe_dispatch_fused_static");
    if (rc != MOE_OK) return rc;
    const char *why = fused_unsupported(dims->N, dims->T, dims->E, dims->R, v.x_row_bytes);
    if (why[0] != '\0')
        return set_error(MOE_ERR_UNSUPPORTED, "moe_dispatch_fused_static: %s; use the separate calls", why);
    const int64_t need = fused_workspace_bytes(dims->N, dims->T, dims->E);
    if (v.NT > 0 && need > fused_static_scratch_bytes())  // an empty batch uses no scratch
        return set_error(MOE_ERR_UNSUPPORTED,
                         "moe_dispatch_fused_static: N=%d T=%d E=%d needs %lld bytes of scratch; the library's "
                         "static array holds %lld", dims->N, dims->T, dims->E, (long long)need,
                         (long long)fused_static_scratch_bytes());
    void *scratch = nullptr;
    cudaError_t e = fused_static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_result(e, "moe_dispatch_fused_static: scratch address");
    return moe_dispatch_fused(dims, logits, bias, score_fn, renormalize, x, x_scales, topk_idx, topk_w,
                              expert_counts, expert_offsets, rank_counts, rank_offsets, send_counts, pos,
                              status, packed_x, packed_scales, packed_src, scratch, stream);
}

int moe_selftest_bounded_wait(int32_t *status, int64_t polls, void *stream) {
    g_err[0] = '\0';
    if (!status || !aligned(status, 4))
        return set_error(MOE_ERR_INVALID_ARG, "moe_selftest_bounded_wait: status must be a 4-byte aligned pointer");
    if (polls < 1 || polls > ((int64_t)1 << 20))
        return set_error(MOE_ERR_INVALID_ARG, "moe_selftest_bounded_wait: polls %lld outside [1, 2^20]",
                         (long long)polls);
    return cuda_result(launch_selftest_wait(status, (long long)polls, (cudaStream_t)stream),
                       "moe_selftest_bounded_wait");
}

int moe_take_device_error(void *stream) {
    g_err[0] = '\0';
    int err = 0;
    cudaError_t e = take_device_error(&err, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_result(e, "moe_take_device_error");
    return err;
}

int moe_read_status(const int32_t *status, void *stream) {
    g_err[0] = '\0';
    if (!status) return set_error(MOE_ERR_INVALID_ARG, "moe_read_status: status is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_result(e, "moe_read_status");
    int32_t host = 0;
    e = cudaMemcpy(&host, status, sizeof(host), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_result(e, "moe_read_status");
    return host;
}

}  // extern "C"
