// Per-token body of the route top-k step, shared by the route kernel and
// the decode-fused dispatch kernel.  See route_topk.cu for the method and
// its sources.
#pragma once

#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace route_impl {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Bitonic sort of a lane's (key, slot) pairs: key descending, slot
// ascending among equal keys, so the head is always the lane's next pick.
template <int JP>
__device__ __forceinline__ void sort_desc(uint32_t (&k)[JP], int (&sl)[JP]) {
#pragma unroll
    for (int size = 2; size <= JP; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < JP; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    // descending runs where (i & size) == 0, ascending otherwise
                    const bool desc = (i & size) == 0;
                    const bool i_first = k[i] > k[j] || (k[i] == k[j] && sl[i] < sl[j]);
                    if (desc != i_first) {
                        const uint32_t tk = k[i];
                        k[i] = k[j];
                        k[j] = tk;
                        const int ts = sl[i];
                        sl[i] = sl[j];
                        sl[j] = ts;
                    }
                }
            }
        }
    }
}

// Best live slot of a lane: the highest key, the lowest slot among equal
// keys (slots are scanned in ascending order and only a strictly higher key
// replaces the best).  s = -1 when no slot is live.
template <int J>
__device__ __forceinline__ void lane_best(const uint32_t (&key)[J], uint32_t live, uint32_t &h, int &s) {
    h = 0u;
    s = -1;
#pragma unroll
    for (int j = 0; j < J; ++j)
        if (((live >> j) & 1u) && (s < 0 || key[j] > h)) {
            h = key[j];
            s = j;
        }
}

// Route token g with the calling warp (all 32 lanes).  Returns, in lane
// k < R, the expert of pair k (what it writes to topk_idx[g][k]).
template <int J, bool kVec4>
__device__ __forceinline__ int route_token(const float *__restrict__ logits,
                                            const float *__restrict__ bias, int64_t g, int E, int R,
                                            int score_fn, int renormalize,
                                            int32_t *__restrict__ topk_idx,
                                            float *__restrict__ topk_w, int lane) {
    const float *row = logits + g * E;
    const int e0 = lane * J;
    float z[J];
#pragma unroll
    for (int j = 0; j < J; ++j) z[j] = 0.f;
    if (kVec4) {
        // E % 4 == 0 and J % 4 == 0: e0 + j is a multiple of 4, so the
        // 16-byte load is aligned and stays inside the row.
#pragma unroll
        for (int j = 0; j < J; j += 4) {
            if (e0 + j < E) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(row + e0 + j));
                z[j] = v.x;
                z[j + 1] = v.y;
                z[j + 2] = v.z;
                z[j + 3] = v.w;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (e0 + j < E) z[j] = __ldg(row + e0 + j);
    }
    const bool softmax = (score_fn & ~MOE_BIAS_SELECT_ONLY) == MOE_SOFTMAX;
    const bool bias_select = (score_fn & MOE_BIAS_SELECT_ONLY) != 0;
    // Bias for selection only: the scores s_e come from the raw logits and
    // the key is fl32(s_e + bias_e).  z[j] becomes s_j here; the bias is
    // added below as in the default mode.  The same expressions recompute
    // the winners' scores for the weights, so keys and weights agree.
    float lmax = 0.f, lsum = 0.f;  // softmax statistics of the raw logits
    if (bias_select) {
        if (softmax) {
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (e0 + j < E) m = fmaxf(m, z[j]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
            lmax = m;
            float t = 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (e0 + j < E) t += expf(__fsub_rn(z[j], lmax));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(kFull, t, off);
            lsum = t;
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (e0 + j < E) z[j] = __fdiv_rn(expf(__fsub_rn(z[j], lmax)), lsum);
        } else {
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (e0 + j < E) z[j] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z[j])));
        }
    }
    uint32_t valid = 0;
    uint32_t key[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        key[j] = 0u;
        if (e0 + j < E) {
            valid |= 1u << j;
            if (bias != nullptr) z[j] = __fadd_rn(z[j], __ldg(bias + e0 + j));
            key[j] = order_key(z[j]);
        }
    }
    // R rounds of a warp max reduction (redux.sync) over one key per lane (the
    // lane's best remaining key) and a ballot for the lowest lane holding the
    // maximum: highest key, then lowest lane, then lowest slot.  How a lane
    // keeps its best key depends on how many it holds:
    //   J <= 8: it sorts its keys once (bitonic network, key descending, slot
    //   ascending) and the winning lane shifts its sorted keys by one;
    //   J >= 12: it keeps its best and second-best keys, the winning lane
    //   promotes its runner-up, and only a lane that wins a third time
    //   rescans its remaining keys (sorting 12 or more keys per lane doubled
    //   the instructions per token on the 384-expert batch, where routing is
    //   bound by instruction issue; with 4 or 8 keys the sort is cheaper).
    float zmax = 0.f;
    int my_e = 0;
    float my_z = 0.f;
    if constexpr (J <= 8) {
        constexpr int JP = (J <= 1) ? 1 : (J <= 2) ? 2 : (J <= 4) ? 4 : 8;
        uint32_t sk[JP];
        int ss[JP];
#pragma unroll
        for (int j = 0; j < JP; ++j) {
            sk[j] = j < J ? key[j] : 0u;  // padding slots carry key 0 and sort last
            ss[j] = j;
        }
        sort_desc<JP>(sk, ss);
        int left = __popc(valid);  // live keys of this lane
        for (int k = 0; k < R; ++k) {
            const uint32_t v = (left > 0) ? sk[0] : 0u;
            const uint32_t kmax = __reduce_max_sync(kFull, v);
            const unsigned ball = __ballot_sync(kFull, left > 0 && v == kmax);
            const int wl = __ffs(ball) - 1;  // some lane always has a live key (R <= E)
            const int wj = __shfl_sync(kFull, ss[0], wl);
            const float wz = key_value(kmax);
            if (k == 0) zmax = wz;
            if (lane == k) {
                my_e = wl * J + wj;
                my_z = wz;
            }
            if (lane == wl) {
#pragma unroll
                for (int j = 0; j + 1 < JP; ++j) {
                    sk[j] = sk[j + 1];
                    ss[j] = ss[j + 1];
                }
                --left;
            }
        }
    } else {
        uint32_t live = valid;
        uint32_t h1 = 0u, h2 = 0u;
        int s1 = -1, s2 = -1;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            if ((live >> j) & 1u) {
                if (s1 < 0 || key[j] > h1) {
                    h2 = h1;
                    s2 = s1;
                    h1 = key[j];
                    s1 = j;
                } else if (s2 < 0 || key[j] > h2) {
                    h2 = key[j];
                    s2 = j;
                }
            }
        }
        bool second = true;  // (h2, s2) is the lane's runner-up (s2 = -1: none left)
        for (int k = 0; k < R; ++k) {
            const bool has = s1 >= 0;
            const uint32_t kmax = __reduce_max_sync(kFull, has ? h1 : 0u);
            const unsigned ball = __ballot_sync(kFull, has && h1 == kmax);
            const int wl = __ffs(ball) - 1;  // some lane always has a live key (R <= E)
            const int wj = __shfl_sync(kFull, s1, wl);
            const float wz = key_value(kmax);
            if (k == 0) zmax = wz;
            if (lane == k) {
                my_e = wl * J + wj;
                my_z = wz;
            }
            if (lane == wl) {
                live &= ~(1u << s1);
                if (second) {
                    h1 = h2;
                    s1 = s2;
                    second = false;
                } else {
                    lane_best<J>(key, live, h1, s1);
                }
            }
        }
    }

    float p = 0.f;
    if (bias_select) {
        if (lane < R) {
            const float l = __ldg(row + my_e);
            p = softmax ? __fdiv_rn(expf(__fsub_rn(l, lmax)), lsum)
                        : __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
        }
    } else if (softmax) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if ((valid >> j) & 1u) s += expf(key_value(key[j]) - zmax);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
        if (lane < R) p = expf(my_z - zmax) / s;
    } else {
        if (lane < R) p = 1.0f / (1.0f + expf(-my_z));
    }
    if (renormalize) {
        float t = p;  // lanes >= R hold 0
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(kFull, t, off);
        p = p / t;
    }
    if (lane < R) {
        topk_idx[g * R + lane] = my_e;
        topk_w[g * R + lane] = p;
    }
    return my_e;
}

}  // namespace route_impl
}  // namespace moe
