// Device helpers shared by the SpMM (forward, transposed) and SDDMM kernels.
#pragma once

#include "snk_internal.cuh"

namespace snk {

// Lane layout of a warp for a padded batch tile of BP columns:
//   VEC = floats of one operand row read by one lane (1, 2 or 4),
//   LPE = lanes that share one stored entry (they split its BP columns),
//   GPW = entries a warp handles side by side (groups per warp).
template <int BP>
struct Tile {
    static constexpr int VEC = BP < 4 ? BP : 4;
    static constexpr int LPE = BP / VEC;
    static constexpr int GPW = kWarp / LPE;
};

template <int VEC>
struct VecF;
template <>
struct VecF<1> {
    __device__ __forceinline__ static void load(const float* p, float (&x)[1]) { x[0] = *p; }
    __device__ __forceinline__ static void ldg(const float* p, float (&x)[1]) { x[0] = __ldg(p); }
};
template <>
struct VecF<2> {
    __device__ __forceinline__ static void load(const float* p, float (&x)[2]) {
        float2 t = *reinterpret_cast<const float2*>(p);
        x[0] = t.x;
        x[1] = t.y;
    }
    __device__ __forceinline__ static void ldg(const float* p, float (&x)[2]) {
        float2 t = __ldg(reinterpret_cast<const float2*>(p));
        x[0] = t.x;
        x[1] = t.y;
    }
};
template <>
struct VecF<4> {
    __device__ __forceinline__ static void load(const float* p, float (&x)[4]) {
        float4 t = *reinterpret_cast<const float4*>(p);
        x[0] = t.x;
        x[1] = t.y;
        x[2] = t.z;
        x[3] = t.w;
    }
    __device__ __forceinline__ static void ldg(const float* p, float (&x)[4]) {
        float4 t = __ldg(reinterpret_cast<const float4*>(p));
        x[0] = t.x;
        x[1] = t.y;
        x[2] = t.z;
        x[3] = t.w;
    }
};

// Four consecutive entries starting at a0 (a multiple of 4) of a stream of n
// elements; one 128-bit streaming load when all four exist, else scalar
// loads that stop at the end of the array.  Positions are 32-bit: the
// library keeps nnz below 2^31, so a0 + 4 never wraps.
__device__ __forceinline__ void stream4(const float* __restrict__ p, uint32_t a0, uint32_t n,
                                        float (&w)[4]) {
    if (a0 + 3 < n) {
        float4 t = __ldcs(reinterpret_cast<const float4*>(p + a0));
        w[0] = t.x;
        w[1] = t.y;
        w[2] = t.z;
        w[3] = t.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = (a0 + j < n) ? p[a0 + j] : 0.f;
    }
}

__device__ __forceinline__ void stream4(const int32_t* __restrict__ p, uint32_t a0, uint32_t n,
                                        int (&w)[4]) {
    if (a0 + 3 < n) {
        int4 t = __ldcs(reinterpret_cast<const int4*>(p + a0));
        w[0] = t.x;
        w[1] = t.y;
        w[2] = t.z;
        w[3] = t.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = (a0 + j < n) ? p[a0 + j] : 0;
    }
}

// Stage the operand transposed: dst[i*BP + beta] = src[beta*ld + i] for
// beta < b, 0 for b <= beta < BP, for i < n.  Reads are coalesced over i.
template <int BP>
__device__ __forceinline__ void stage_transposed(float* dst, const float* __restrict__ src,
                                                 int64_t ld, int b, int64_t n, int tid,
                                                 int nthreads) {
    for (int64_t i = tid; i < n; i += nthreads) {
        if constexpr (BP >= 4) {
#pragma unroll 4
            for (int q = 0; q < BP; q += 4) {
                float4 t;
                t.x = q + 0 < b ? src[(q + 0) * ld + i] : 0.f;
                t.y = q + 1 < b ? src[(q + 1) * ld + i] : 0.f;
                t.z = q + 2 < b ? src[(q + 2) * ld + i] : 0.f;
                t.w = q + 3 < b ? src[(q + 3) * ld + i] : 0.f;
                *reinterpret_cast<float4*>(dst + i * BP + q) = t;
            }
        } else if constexpr (BP == 2) {
            *reinterpret_cast<float2*>(dst + i * 2) =
                make_float2(src[i], b > 1 ? src[ld + i] : 0.f);
        } else {
            dst[i] = src[i];
        }
    }
}

}  // namespace snk
