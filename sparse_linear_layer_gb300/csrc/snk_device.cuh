// Device helpers shared by the SpMM (forward, transposed) and SDDMM kernels.
#pragma once

#include "snk_internal.cuh"

namespace snk {

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

// Lane layout of a warp for a padded batch tile of BP columns:
//   VEC = floats of one operand row read by one lane,
//   LPE = lanes that share one stored entry (they split its BP columns),
//   GPW = entries a warp handles side by side (groups per warp).
// Up to 16 columns a lane reads 4 (more entries side by side hide the
// latency of their loads); from 32 columns on it reads 8, so that a warp
// still holds 8 or more entries per step.  A lane's 8 columns are two chunks
// of 4, interleaved with the other lanes of its entry (lane sub holds
// columns 4 sub .. 4 sub + 3 and 4 (LPE + sub) .. + 3): each 128-bit load
// instruction of a group then covers 128 contiguous bytes of the row.
// Measured at 10000^2, 90%, b = 64: forward / dX / dW 154 / 201 / 278 us,
// against 204 / 271 / 356 with 4 columns per lane; 8 columns at b = 16 or 16
// columns at b = 64 were slower.
template <int BP>
struct Tile {
    static constexpr int VEC = BP < 4 ? BP : (BP >= 32 ? 8 : 4);
    static constexpr int LPE = BP / VEC;
    static constexpr int GPW = kWarp / LPE;
    // batch column of value j of lane sub
    __host__ __device__ static constexpr int beta(int sub, int j) {
        return VEC <= 4 ? sub * VEC + j : (j >> 2) * (4 * LPE) + sub * 4 + (j & 3);
    }
    // the lane's VEC values of an operand row (shared memory / read-only path)
    __device__ __forceinline__ static void load(const float* row, int sub, float (&x)[VEC]) {
        if constexpr (VEC <= 4) {
            VecF<VEC>::load(row + sub * VEC, x);
        } else {
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                const float4 t = reinterpret_cast<const float4*>(row)[q * LPE + sub];
                x[4 * q] = t.x;
                x[4 * q + 1] = t.y;
                x[4 * q + 2] = t.z;
                x[4 * q + 3] = t.w;
            }
        }
    }
    __device__ __forceinline__ static void ldg(const float* row, int sub, float (&x)[VEC]) {
        if constexpr (VEC <= 4) {
            VecF<VEC>::ldg(row + sub * VEC, x);
        } else {
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(row) + q * LPE + sub);
                x[4 * q] = t.x;
                x[4 * q + 1] = t.y;
                x[4 * q + 2] = t.z;
                x[4 * q + 3] = t.w;
            }
        }
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

// Index block of 4 consecutive entries: 16-bit indices (packed in two
// registers, read from a zero-padded library stream, no end test) or 32-bit
// indices (read with the end-of-array test).
template <bool IDX16>
struct IdxBlk;
template <>
struct IdxBlk<true> {
    uint32_t lo, hi;
    __device__ __forceinline__ void load(const uint16_t* p, uint32_t a0) {
        const uint2 t = __ldcs(reinterpret_cast<const uint2*>(p + a0));
        lo = t.x;
        hi = t.y;
    }
    __device__ __forceinline__ int get(int j) const {
        const uint32_t w = j < 2 ? lo : hi;
        return (int)((j & 1) ? (w >> 16) : (w & 0xffffu));
    }
};
template <>
struct IdxBlk<false> {
    int c[4];
    __device__ __forceinline__ void load(const int32_t* p, uint32_t a0, uint32_t n) {
        stream4(p, a0, n, c);
    }
    __device__ __forceinline__ int get(int j) const { return c[j]; }
};

// Four int32 entries of a zero-padded library stream (no end test).
__device__ __forceinline__ void padded4(const int32_t* __restrict__ p, uint32_t a0, int (&w)[4]) {
    const int4 t = __ldcs(reinterpret_cast<const int4*>(p + a0));
    w[0] = t.x;
    w[1] = t.y;
    w[2] = t.z;
    w[3] = t.w;
}

// ---- a band of the transposed operand into shared memory, by the TMA engine
// (one contiguous run: cp.async.bulk, issued by one thread, completed on an
// mbarrier that every thread then waits on, within a bounded number of
// cycles).
constexpr long long kStageWaitCycles = 4000000000LL;   // about two seconds at the boost clock
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void stage_bar_init(uint64_t* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// bytes: a multiple of 16, both addresses 16-byte aligned; copied in runs of
// at most 64 KB, all counted on the same barrier phase.
__device__ __forceinline__ void stage_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    for (uint32_t off = 0; off < bytes; off += 65536u) {
        const uint32_t n = min(65536u, bytes - off);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_addr(static_cast<char*>(dst) + off)),
                     "l"(static_cast<const char*>(src) + off), "r"(n), "r"(smem_addr(bar))
                     : "memory");
    }
}
// Wait for phase 0 of the barrier; false once `limit` cycles have passed.
__device__ __forceinline__ bool stage_wait(uint64_t* bar, long long limit) {
    long long t0 = 0;
    for (int spin = 0;; ++spin) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(smem_addr(bar))
            : "memory");
        if (ok) return true;
        if (spin == 0)
            t0 = clock64();
        else if (clock64() - t0 > limit)
            return false;
    }
}
// Rows [r0, r0 + rows) of a transposed operand xt[n][BP] into dst.  A wait
// that runs out records kStatLimit in *status and waits once more (for the
// copy still landing) before the block goes on; its results are then not
// to be trusted, and the caller learns it from the status word.
template <int BP>
__device__ __forceinline__ void stage_band(float* dst, const float* xt, int r0, int rows, uint64_t* bar,
                                           int32_t* status) {
    if (threadIdx.x == 0) stage_bar_init(bar);
    __syncthreads();
    if (rows <= 0) return;
    if (threadIdx.x == 0) stage_bulk(dst, xt + (int64_t)r0 * BP, (uint32_t)rows * BP * 4u, bar);
    if (!stage_wait(bar, kStageWaitCycles)) {
        if (status) atomicOr(status, kStatLimit);
        stage_wait(bar, kStageWaitCycles);
    }
}

// Component i (0..3, a runtime value) of a float4, without local memory.
__device__ __forceinline__ float f4_at(const float4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Stage the operand transposed: dst[i*BP + beta] = src[beta*ld + i] for
// beta < b, 0 for b <= beta < BP, for i < n.  When the rows of src are
// 16-byte aligned, groups of 4 columns are read with 128-bit loads (one per
// source row) and transposed in registers, so each thread issues 4x fewer
// loads; the remaining columns (and unaligned sources) use 32-bit loads.
// Several groups are loaded before any is stored, to keep loads in flight.
template <int BP, bool ROT = true>
__device__ __forceinline__ void stage_transposed(float* dst, const float* __restrict__ src,
                                                 int64_t ld, int b, int64_t n, int tid,
                                                 int nthreads) {
    int64_t n_vec = 0;
    if ((((uintptr_t)src) & 15) == 0 && (ld & 3) == 0) n_vec = n & ~(int64_t)3;
    const int64_t groups = n_vec >> 2;
    if constexpr (BP >= 4) {
        // Items (row group qb of 4 batch rows, column group g), all spread
        // over the threads at once: with one pass per row group, a 64-row
        // tile took 16 dependent rounds of loads with only the column groups'
        // threads busy.
        constexpr int QB = BP / 4;
        constexpr int U = 2;
        const int64_t items = groups * QB;
        for (int64_t i0 = tid; i0 < items; i0 += (int64_t)nthreads * U) {
            float4 t[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + (int64_t)u * nthreads;
                const int qb = (QB == 1 || i >= items) ? 0 : (int)(i / groups);
                const int64_t g = i - (int64_t)qb * groups;
                const int r0 = 4 * qb;
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
                    t[u][rr] = (i < items && r0 + rr < b)
                                   ? __ldg(reinterpret_cast<const float4*>(src + (r0 + rr) * ld) + g)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + (int64_t)u * nthreads;
                if (i < items) {
                    const int qb = QB == 1 ? 0 : (int)(i / groups);
                    const int64_t g = i - (int64_t)qb * groups;
                    float* d = dst + 4 * g * BP + 4 * qb;
                    // The 4 rows of group g, in an order rotated per
                    // thread (ROT): the lanes of a quarter-warp
                    // (consecutive g) then store to different banks
                    // (BP = 4: 8 distinct 16-byte slots of 128 bytes,
                    // where the plain order puts 4 lanes on the same
                    // banks).  The column sweep, which stages a phase
                    // at a time, measured no gain and keeps the plain
                    // order.  (Wider rows keep the plain order: the
                    // rotation buys little there and its selects cost
                    // registers.)
                    const int rot = !(ROT && BP <= 8) ? 0 : (BP == 4 ? (int)((g >> 1) & 3) : (int)(g & 3));
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int jj = (q + rot) & 3;
                        *reinterpret_cast<float4*>(d + jj * BP) =
                            make_float4(f4_at(t[u][0], jj), f4_at(t[u][1], jj), f4_at(t[u][2], jj), f4_at(t[u][3], jj));
                    }
                }
            }
        }
    } else {
        constexpr int U = BP == 2 ? 4 : 8;
        for (int64_t g0 = tid; g0 < groups; g0 += (int64_t)nthreads * U) {
            float4 t0[U], t1[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = g0 + (int64_t)u * nthreads;
                t0[u] = g < groups ? __ldg(reinterpret_cast<const float4*>(src) + g)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                if constexpr (BP == 2)
                    t1[u] = (g < groups && b > 1) ? __ldg(reinterpret_cast<const float4*>(src + ld) + g)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = g0 + (int64_t)u * nthreads;
                if (g < groups) {
                    if constexpr (BP == 2) {
                        float4* d = reinterpret_cast<float4*>(dst + 8 * g);
                        d[0] = make_float4(t0[u].x, t1[u].x, t0[u].y, t1[u].y);
                        d[1] = make_float4(t0[u].z, t1[u].z, t0[u].w, t1[u].w);
                    } else {
                        reinterpret_cast<float4*>(dst)[g] = t0[u];
                    }
                }
            }
        }
    }
    // remaining columns, 32-bit loads
    for (int64_t i = n_vec + tid; i < n; i += nthreads) {
#pragma unroll
        for (int beta = 0; beta < BP; ++beta) dst[i * BP + beta] = beta < b ? __ldg(src + beta * ld + i) : 0.f;
    }
}

// Row (segment) boundaries of one chunk, read 32 at a time: lane t holds the
// start of relative segment base+t and, optionally, that segment's bias.
// Queried warp-uniformly; moving forward reloads the window.
struct SegWindow {
    int r_begin, nrows, base;
    uint32_t start;
    float b;
    __device__ __forceinline__ void load(int rel, int lane, const int32_t* seg_ptr,
                                         const float* bias) {
        base = rel;
        const int t = rel + lane;
        start = t <= nrows ? (uint32_t)__ldg(seg_ptr + r_begin + t) : 0u;
        b = (bias && t < nrows) ? __ldg(bias + r_begin + t) : 0.f;
    }
    // start of relative segment i; the window is kept so that segment i-1's
    // bias stays readable
    __device__ __forceinline__ uint32_t bnd(int i, int lane, const int32_t* seg_ptr,
                                            const float* bias) {
        if (i - base >= 32) load(i - 1, lane, seg_ptr, bias);
        return __shfl_sync(0xffffffffu, start, i - base);
    }
    __device__ __forceinline__ float bias_of(int i) {
        return __shfl_sync(0xffffffffu, b, i - base);
    }
};

}  // namespace snk
