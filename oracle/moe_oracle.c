/*
 * CPU oracle for MoE token routing: route top-k, dispatch count, dispatch
 * pack, expert op (harness stand-in), combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * statement of what the routing path computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may call it.  It shares no
 * code, header, table or helper with the CUDA library; the only thing the two
 * have in common is the seeded input generator that feeds them.
 *
 * Floating point: routing weights and the combine sum are computed in double
 * and rounded once at the end.  The routing key z = logit + bias is a single
 * float addition (correctly rounded, hence identical on every IEEE machine),
 * so the selected indices are exact.
 *
 * Sources (page title, section):
 *   [P1] "Lower latency and higher throughput with multi-node DeepSeek
 *        deployment", sections "Expert Parallelism", "MoE Router",
 *        "Quantization".
 *   [P2] "Efficient and portable mixture-of-experts communication", sections
 *        "Introduction", "Portable kernels", "Dispatch", "Combine".
 *   [P4] "Hosting Qwen on Blackwell", section "Expert parallel".
 *   [P5] "Enabling trillion-parameter models on AWS EFA", sections "Send and
 *        receive buffers", "Dispatch and combine", "Evaluation".
 *
 * Build: gcc -O2 -fPIC -shared (no -ffast-math: the rounding must be IEEE).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_INVALID (-1)
#define OR_ERR_CAPACITY (-4)

#define OR_SOFTMAX 0
#define OR_SIGMOID 1
#define OR_BIAS_SELECT_ONLY 0x10 /* flag OR'ed into score_fn, see step 1 */

#define OR_BF16 0
#define OR_F32 1
#define OR_FP8 2

/* ------------------------------------------------------------------------ */
/* number formats, written from their definitions                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32. */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even; NaN stays NaN. */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* OCP fp8 e4m3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no inf. */
static double fp8e4m3_to_double(uint8_t b) {
    int s = (b >> 7) & 1, ex = (b >> 3) & 15, m = b & 7;
    double v;
    if (ex == 15 && m == 7) return NAN;
    if (ex == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, ex - 7);
    return s ? -v : v;
}

double oracle_fp8e4m3_decode(uint8_t b) { return fp8e4m3_to_double(b); }

/* binary32 -> e4m3, round to nearest with ties to the even code, saturating
 * at +-448: the code whose value is nearest to v (all 127 finite magnitudes
 * sorted ascending, found by bisection); a tie between two codes goes to
 * the one with mantissa lsb 0; magnitudes above 448 give 448.  The sign bit
 * is copied from v (so -0 and small negatives give 0x80).  v must not be
 * NaN. */
static uint8_t f32_to_fp8e4m3(float v) {
    static double mag[127];
    static int init = 0;
    if (!init) {
        for (int c = 0; c < 127; ++c) mag[c] = fp8e4m3_to_double((uint8_t)c);
        init = 1;
    }
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    if (a >= mag[126]) return (uint8_t)(sign | 126);
    int lo = 0, hi = 126; /* mag[lo] <= a < mag[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (mag[mid] <= a) lo = mid;
        else hi = mid;
    }
    const double dlo = a - mag[lo], dhi = mag[hi] - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = hi;
    else c = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | c);
}

uint8_t oracle_f32_to_fp8e4m3(float v) { return f32_to_fp8e4m3(v); }

/* ------------------------------------------------------------------------ */
/* next step: fp8 block quantisation of dispatched rows  ([P1] Quantization:
 * activations are quantised on the fly with one scaling factor per
 * 128-element vector; [P2] Dispatch: the message carries the block scaling
 * factors with the activations)
 *
 * For each row and each block of 128 consecutive elements:
 *   amax  = max |x| over the block (bf16 values are exact in float)
 *   scale = fl32(amax / 448)              (448: largest e4m3 value)
 *   code  = e4m3_RNE_sat(fl32(x / scale)), or 0 when amax == 0
 * ------------------------------------------------------------------------ */
int oracle_quantize_rows(int64_t rows, int64_t H, const uint16_t *x_bf16, uint8_t *codes,
                         float *scales) {
    if (H % 128 != 0) return OR_ERR_INVALID;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b0 = 0; b0 < H; b0 += 128) {
            float amax = 0.0f;
            for (int64_t h = b0; h < b0 + 128; ++h) {
                float a = fabsf(bf16_to_f32(x_bf16[r * H + h]));
                if (a > amax) amax = a;
            }
            float scale = amax / 448.0f;
            scales[r * (H / 128) + b0 / 128] = scale;
            for (int64_t h = b0; h < b0 + 128; ++h) {
                float v = bf16_to_f32(x_bf16[r * H + h]);
                codes[r * H + h] = (amax == 0.0f) ? (uint8_t)0 : f32_to_fp8e4m3(v / scale);
            }
        }
    }
    return OR_OK;
}
uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16(f); }

/* ------------------------------------------------------------------------ */
/* step 1: route top-k  ([P2] Introduction; [P1] MoE Router, Expert Parallelism)
 *
 * A linear router gives one logit per expert; each token goes to the R
 * experts with the highest scores and the router's probabilities give the
 * weights.  Here:  z_e = fl32(logit_e + bias_e)  (bias 0 when absent),
 * experts ordered by z descending, equal z broken towards the lower expert
 * index; the first R are selected in that order.  Scores: softmax over all
 * E experts (p_e = exp(z_e - max z) / sum_j exp(z_j - max z)) or the
 * logistic sigmoid p_e = 1 / (1 + exp(-z_e)).  Optional renormalisation
 * divides the selected p by their sum.  Weights are rounded to float once.
 *
 * With OR_BIAS_SELECT_ONLY (the DeepSeek-V3 router convention; the pages
 * do not say where the bias enters) the bias only moves the selection:
 * s_e = score of the raw logit (softmax over all E, or sigmoid), the key is
 * fl32(fl32(s_e) + bias_e) -- the selection is decided on float scores, as
 * a float kernel decides it -- ties again towards the lower index, and the
 * weights are the selected s_e (unrounded), optionally renormalised.
 * ------------------------------------------------------------------------ */

static const float *g_sort_z; /* key array for the comparator (single thread) */

static int cmp_expert(const void *a, const void *b) {
    int ea = *(const int *)a, eb = *(const int *)b;
    float za = g_sort_z[ea], zb = g_sort_z[eb];
    if (za > zb) return -1;
    if (za < zb) return 1;
    return (ea < eb) ? -1 : (ea > eb);
}

int oracle_route(int64_t NT, int E, int R, const float *logits, const float *bias,
                 int score_fn, int renorm, int32_t *topk_idx, float *topk_w,
                 double *topk_w64 /* nullable: unrounded weights */) {
    const int bias_select = (score_fn & OR_BIAS_SELECT_ONLY) != 0;
    const int fn = score_fn & ~OR_BIAS_SELECT_ONLY;
    if (E <= 0 || R <= 0 || R > E || (fn != OR_SOFTMAX && fn != OR_SIGMOID)) return OR_ERR_INVALID;
    float *z = (float *)malloc(sizeof(float) * (size_t)E);
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)R);
    double *sc = (double *)malloc(sizeof(double) * (size_t)E); /* raw-logit scores */
    for (int64_t g = 0; g < NT; ++g) {
        const float *lg = logits + g * E;
        if (bias_select) {
            if (fn == OR_SOFTMAX) {
                double lmax = (double)lg[0];
                for (int e = 1; e < E; ++e)
                    if ((double)lg[e] > lmax) lmax = (double)lg[e];
                double denom = 0.0;
                for (int e = 0; e < E; ++e) denom += exp((double)lg[e] - lmax);
                for (int e = 0; e < E; ++e) sc[e] = exp((double)lg[e] - lmax) / denom;
            } else {
                for (int e = 0; e < E; ++e) sc[e] = 1.0 / (1.0 + exp(-(double)lg[e]));
            }
        }
        for (int e = 0; e < E; ++e) {
            float b = bias ? bias[e] : 0.0f;
            if (bias_select) {
                float s_f = (float)sc[e];
                z[e] = s_f + b; /* float score plus bias, one float addition */
            } else {
                z[e] = lg[e] + b; /* one correctly rounded float addition */
            }
            order[e] = e;
        }
        g_sort_z = z;
        qsort(order, (size_t)E, sizeof(int), cmp_expert);

        if (bias_select) {
            for (int k = 0; k < R; ++k) p[k] = sc[order[k]];
        } else if (fn == OR_SOFTMAX) {
            double zmax = (double)z[order[0]];
            double denom = 0.0;
            for (int e = 0; e < E; ++e) denom += exp((double)z[e] - zmax);
            for (int k = 0; k < R; ++k) p[k] = exp((double)z[order[k]] - zmax) / denom;
        } else {
            for (int k = 0; k < R; ++k) p[k] = 1.0 / (1.0 + exp(-(double)z[order[k]]));
        }
        if (renorm) {
            double s = 0.0;
            for (int k = 0; k < R; ++k) s += p[k];
            for (int k = 0; k < R; ++k) p[k] = p[k] / s;
        }
        for (int k = 0; k < R; ++k) {
            topk_idx[g * R + k] = order[k];
            topk_w[g * R + k] = (float)p[k];
            if (topk_w64) topk_w64[g * R + k] = p[k];
        }
    }
    free(z);
    free(order);
    free(p);
    free(sc);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* step 2: dispatch count  ([P5] Dispatch and combine, Send and receive
 * buffers; [P2] Dispatch, Portable kernels)
 *
 * Experts are spread contiguously over the N ranks: expert e lives on rank
 * d = e / (E/N).  Token g = s*T + t belongs to source rank s.
 *   expert_counts[e]  = number of (g, k) with topk_idx[g][k] == e
 *   expert_offsets    = exclusive prefix sum of expert_counts over e
 *                       (E + 1 entries, last = total)
 *   rank_counts[d]    = sum of expert_counts over the experts of rank d
 *   rank_offsets      = exclusive prefix sum of rank_counts (N + 1 entries)
 *   send_counts[s][d] = number of (g, k) with g on rank s and the expert on d
 *   pos[g][k]         = row of rank d's receive region this pair lands in:
 *                       d*cap + (expert_offsets[e] - rank_offsets[d])
 *                             + #{(g', k') before (g, k) with topk_idx == e},
 *                       i.e. within a rank, rows are grouped by expert in
 *                       ascending order and, inside an expert, ordered by
 *                       token (hence by source rank) ascending.
 * A pair is invalid, gets pos = -1 and is not counted when its expert id is
 * outside [0, E) or repeats an earlier expert of the same token.  A pair
 * whose in-rank row would reach cap gets pos = -1 (it is still counted).
 * Status: invalid pairs => OR_ERR_INVALID, else a rank over capacity =>
 * OR_ERR_CAPACITY, else OR_OK.
 * ------------------------------------------------------------------------ */
int oracle_count(int N, int64_t T, int E, int R, int64_t cap, const int32_t *topk_idx,
                 int32_t *expert_counts, int32_t *expert_offsets, int32_t *rank_counts,
                 int32_t *rank_offsets, int32_t *send_counts, int32_t *pos) {
    if (N <= 0 || E <= 0 || E % N != 0 || R <= 0 || cap <= 0) return OR_ERR_INVALID;
    const int L = E / N;
    const int64_t NT = (int64_t)N * T;
    int any_invalid = 0, over = 0;

    /* validity of each pair */
    char *valid = (char *)malloc((size_t)(NT * R > 0 ? NT * R : 1));
    for (int64_t g = 0; g < NT; ++g) {
        for (int k = 0; k < R; ++k) {
            int e = topk_idx[g * R + k];
            int ok = (e >= 0 && e < E);
            for (int k2 = 0; ok && k2 < k; ++k2)
                if (topk_idx[g * R + k2] == e) ok = 0;
            valid[g * R + k] = (char)ok;
            if (!ok) any_invalid = 1;
        }
    }

    for (int e = 0; e < E; ++e) expert_counts[e] = 0;
    for (int s = 0; s < N; ++s)
        for (int d = 0; d < N; ++d) send_counts[s * N + d] = 0;
    for (int64_t g = 0; g < NT; ++g) {
        int s = (int)(g / T);
        for (int k = 0; k < R; ++k) {
            if (!valid[g * R + k]) continue;
            int e = topk_idx[g * R + k];
            expert_counts[e] += 1;
            send_counts[s * N + e / L] += 1;
        }
    }
    expert_offsets[0] = 0;
    for (int e = 0; e < E; ++e) expert_offsets[e + 1] = expert_offsets[e] + expert_counts[e];
    for (int d = 0; d < N; ++d) {
        int32_t c = 0;
        for (int e = d * L; e < (d + 1) * L; ++e) c += expert_counts[e];
        rank_counts[d] = c;
        if ((int64_t)c > cap) over = 1;
    }
    rank_offsets[0] = 0;
    for (int d = 0; d < N; ++d) rank_offsets[d + 1] = rank_offsets[d] + rank_counts[d];

    /* positions: walk the pairs in (g, k) order with one running counter per
     * expert, which is the "#earlier pairs with the same expert" term. */
    int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t g = 0; g < NT; ++g) {
        for (int k = 0; k < R; ++k) {
            if (!valid[g * R + k]) {
                pos[g * R + k] = -1;
                continue;
            }
            int e = topk_idx[g * R + k];
            int d = e / L;
            int64_t local = (int64_t)(expert_offsets[e] - rank_offsets[d]) + seen[e];
            seen[e] += 1;
            pos[g * R + k] = (local < cap) ? (int32_t)((int64_t)d * cap + local) : -1;
        }
    }
    free(seen);
    free(valid);
    if (any_invalid) return OR_ERR_INVALID;
    if (over) return OR_ERR_CAPACITY;
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* step 3: dispatch pack  ([P2] Dispatch; [P5] Dispatch and combine)
 *
 * Every routed pair (g, k) with pos >= 0 receives a byte copy of token row
 * x[g] (and, for block-scaled fp8, its H/128 float scales) plus the index of
 * its origin, g*R + k.  The oracle stores only occupied rows, compactly: the
 * region row (d, local) = pos is kept at compact row rank_offsets[d] + local
 * (rank_offsets from step 2; rows dropped for capacity leave unused gaps).
 * ------------------------------------------------------------------------ */
static int64_t compact_row(int32_t p, int64_t cap, const int32_t *rank_offsets) {
    int64_t d = (int64_t)p / cap, local = (int64_t)p % cap;
    return (int64_t)rank_offsets[d] + local;
}

int oracle_pack(int64_t NT, int R, int64_t row_bytes, int64_t scales_per_row, int64_t cap,
                const uint8_t *x, const float *x_scales, const int32_t *pos,
                const int32_t *rank_offsets, uint8_t *packed_x, float *packed_scales,
                int32_t *packed_src) {
    for (int64_t g = 0; g < NT; ++g) {
        for (int k = 0; k < R; ++k) {
            int32_t p = pos[g * R + k];
            if (p < 0) continue;
            int64_t c = compact_row(p, cap, rank_offsets);
            memcpy(packed_x + c * row_bytes, x + g * row_bytes, (size_t)row_bytes);
            if (scales_per_row > 0)
                memcpy(packed_scales + c * scales_per_row, x_scales + g * scales_per_row,
                       sizeof(float) * (size_t)scales_per_row);
            packed_src[c] = (int32_t)(g * R + k);
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* harness expert op on the compact rows (stands in for the grouped expert
 * GEMM; not part of the routing path):
 *   identity: y = x (bf16 -> bf16, f32 -> f32)
 *   scale:    y = round(float(x) * s_e), s_e = 1 + ((e mod 7) - 3)/16
 *   dequant:  y = bf16_RNE(fl32(decode_e4m3(q) * scale_block))
 * The expert of compact row c is topk_idx[packed_src[c]]; rows whose
 * packed_src is negative (never written: capacity gaps) are skipped.
 * ------------------------------------------------------------------------ */
int oracle_expert_op(int op /*0 identity, 1 scale, 2 dequant*/, int64_t rows, int64_t H,
                     int x_dtype, int y_dtype, const uint8_t *packed_x,
                     const float *packed_scales, const int32_t *packed_src,
                     const int32_t *topk_idx, void *y) {
    float fp8_value[256]; /* every e4m3 code decoded once (exact in float) */
    for (int b = 0; b < 256; ++b) fp8_value[b] = (float)fp8e4m3_to_double((uint8_t)b);
    for (int64_t c = 0; c < rows; ++c) {
        if (packed_src[c] < 0) continue;
        int e = topk_idx[packed_src[c]];
        float s = 1.0f + (float)((e % 7) - 3) / 16.0f;
        for (int64_t h = 0; h < H; ++h) {
            float v;
            if (x_dtype == OR_BF16) v = bf16_to_f32(((const uint16_t *)packed_x)[c * H + h]);
            else if (x_dtype == OR_F32) v = ((const float *)packed_x)[c * H + h];
            else v = fp8_value[packed_x[c * H + h]];
            if (op == 1) v = v * s;
            else if (op == 2) v = v * packed_scales[c * (H / 128) + h / 128];
            if (y_dtype == OR_BF16) ((uint16_t *)y)[c * H + h] = f32_to_bf16(v);
            else ((float *)y)[c * H + h] = v;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* step 4: combine  ([P2] Combine, Introduction; [P5] Dispatch and combine,
 * Evaluation)
 *
 * Each token's expert outputs come back to it and are summed with the
 * router weights:  out[g][h] = sum_k w[g][k] * y[pos[g][k]][h]  (pairs with
 * pos = -1 contribute nothing).  Accumulated in double; mag holds
 * sum_k |w * y| for the relative tolerance of float outputs.
 * ------------------------------------------------------------------------ */
int oracle_combine(int64_t NT, int R, int64_t H, int y_dtype, int64_t cap, const void *y,
                   const int32_t *pos, const int32_t *rank_offsets, const float *topk_w,
                   double *out, double *mag) {
    for (int64_t g = 0; g < NT; ++g) {
        for (int64_t h = 0; h < H; ++h) {
            out[g * H + h] = 0.0;
            if (mag) mag[g * H + h] = 0.0;
        }
        for (int k = 0; k < R; ++k) {
            int32_t p = pos[g * R + k];
            if (p < 0) continue;
            int64_t c = compact_row(p, cap, rank_offsets);
            double w = (double)topk_w[g * R + k];
            for (int64_t h = 0; h < H; ++h) {
                double v = (y_dtype == OR_BF16)
                               ? (double)bf16_to_f32(((const uint16_t *)y)[c * H + h])
                               : (double)((const float *)y)[c * H + h];
                out[g * H + h] += w * v;
                if (mag) mag[g * H + h] += fabs(w * v);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* next steps: accumulation of a token's pairs per destination rank
 * ([P5] Evaluation: accumulating on the send side reduces the data moved,
 * at some cost in accuracy; [P4] Expert parallel: with replicated inputs a
 * rank handles only the tokens routed to its own experts and accumulates
 * locally before an all-reduce)
 *
 * The rank of pair (g, k) is d = pos / cap (pairs with pos < 0 are skipped).
 *
 * oracle_combine_rank: out[g] = sum over pairs of g on rank `rank` of
 *   w * y[row], in double (0 for tokens with no pair there).  Summed over
 *   all ranks this is the combine.
 *
 * oracle_combine_partials: the distinct ranks of token g, in the order of
 *   their first pair k, get slots j = 0, 1, ...; partial[g][j] = sum over
 *   the pairs of g on that rank of w * y[row] in double, rounded to float
 *   and then to y_dtype (the 16-bit row a rank would send back);
 *   slot_rank[g][j] = that rank, or -1 for unused slots (zero rows); P =
 *   min(R, N) slots per token.
 *
 * oracle_reduce_partials: out[g] = sum over used slots of partial[g][j], in
 *   double.
 * ------------------------------------------------------------------------ */
int oracle_combine_rank(int64_t NT, int R, int64_t H, int y_dtype, int64_t cap, int rank,
                        const void *y, const int32_t *pos, const int32_t *rank_offsets,
                        const float *topk_w, double *out) {
    for (int64_t g = 0; g < NT; ++g) {
        for (int64_t h = 0; h < H; ++h) out[g * H + h] = 0.0;
        for (int k = 0; k < R; ++k) {
            int32_t p = pos[g * R + k];
            if (p < 0 || p / cap != rank) continue;
            int64_t c = compact_row(p, cap, rank_offsets);
            double w = (double)topk_w[g * R + k];
            for (int64_t h = 0; h < H; ++h) {
                double v = (y_dtype == OR_BF16)
                               ? (double)bf16_to_f32(((const uint16_t *)y)[c * H + h])
                               : (double)((const float *)y)[c * H + h];
                out[g * H + h] += w * v;
            }
        }
    }
    return OR_OK;
}

int oracle_combine_partials(int64_t NT, int R, int P, int64_t H, int y_dtype, int64_t cap,
                            const void *y, const int32_t *pos, const int32_t *rank_offsets,
                            const float *topk_w, void *partial, int32_t *slot_rank) {
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    for (int64_t g = 0; g < NT; ++g) {
        int nslot = 0;
        for (int j = 0; j < P; ++j) slot_rank[g * P + j] = -1;
        for (int k = 0; k < R; ++k) {
            int32_t p = pos[g * R + k];
            if (p < 0) continue;
            int d = (int)(p / cap), seen = 0;
            for (int j = 0; j < nslot; ++j)
                if (slot_rank[g * P + j] == d) seen = 1;
            if (!seen && nslot < P) slot_rank[g * P + nslot++] = d;
        }
        for (int j = 0; j < P; ++j) {
            for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
            for (int k = 0; k < R && j < nslot; ++k) {
                int32_t p = pos[g * R + k];
                if (p < 0 || p / cap != slot_rank[g * P + j]) continue;
                int64_t c = compact_row(p, cap, rank_offsets);
                double w = (double)topk_w[g * R + k];
                for (int64_t h = 0; h < H; ++h) {
                    double v = (y_dtype == OR_BF16)
                                   ? (double)bf16_to_f32(((const uint16_t *)y)[c * H + h])
                                   : (double)((const float *)y)[c * H + h];
                    acc[h] += w * v;
                }
            }
            for (int64_t h = 0; h < H; ++h) {
                int64_t o = (g * P + j) * H + h;
                if (y_dtype == OR_BF16) ((uint16_t *)partial)[o] = f32_to_bf16((float)acc[h]);
                else ((float *)partial)[o] = (float)acc[h];
            }
        }
    }
    free(acc);
    return OR_OK;
}

int oracle_reduce_partials(int64_t NT, int P, int64_t H, int y_dtype, const void *partial,
                           const int32_t *slot_rank, double *out) {
    for (int64_t g = 0; g < NT; ++g) {
        for (int64_t h = 0; h < H; ++h) {
            double s = 0.0;
            for (int j = 0; j < P; ++j) {
                if (slot_rank[g * P + j] < 0) continue;
                int64_t o = (g * P + j) * H + h;
                s += (y_dtype == OR_BF16) ? (double)bf16_to_f32(((const uint16_t *)partial)[o])
                                          : (double)((const float *)partial)[o];
            }
            out[g * H + h] = s;
        }
    }
    return OR_OK;
}
