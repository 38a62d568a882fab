// 16-byte vectors of y rows for the accumulating kernels: 8 bf16 or 4 f32
// elements, widened to f32, accumulated with fused multiply-adds, and
// written back with one rounding (bf16: round to nearest even).
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

namespace moe {

template <int kBf16>
struct Vec;

template <>
struct Vec<1> {  // 8 x bf16
    static constexpr int kElems = 8;
    __device__ __forceinline__ static void fma(float (&a)[8], float w, const uint4 &v) {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), a[2 * i]);
            a[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xffff0000u), a[2 * i + 1]);
        }
    }
    __device__ __forceinline__ static void add(float (&a)[8], const uint4 &v) { fma(a, 1.0f, v); }
    __device__ __forceinline__ static uint4 pack(const float (&a)[8]) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
            u[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        return make_uint4(u[0], u[1], u[2], u[3]);
    }
};

template <>
struct Vec<0> {  // 4 x f32
    static constexpr int kElems = 4;
    __device__ __forceinline__ static void fma(float (&a)[4], float w, const uint4 &v) {
        a[0] = fmaf(w, __uint_as_float(v.x), a[0]);
        a[1] = fmaf(w, __uint_as_float(v.y), a[1]);
        a[2] = fmaf(w, __uint_as_float(v.z), a[2]);
        a[3] = fmaf(w, __uint_as_float(v.w), a[3]);
    }
    __device__ __forceinline__ static void add(float (&a)[4], const uint4 &v) {
        a[0] += __uint_as_float(v.x);
        a[1] += __uint_as_float(v.y);
        a[2] += __uint_as_float(v.z);
        a[3] += __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&a)[4]) {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    }
};

}  // namespace moe
