// Large-batch products on the tensor cores (tcgen05): Y = X W^T + b and
// dX = dY W (k_tc_spmm), and dW on the entries of W with db (k_tc_sddmm),
// for batches of hundreds of rows and more.
//
// "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
// GPU", appendix Table 13 (GAMLP training at batch 4096): at that batch the
// per-entry SpMM does b multiply-adds per stored weight and its operand
// traffic, not the weight stream, sets the time.  Here each 192-row x 64-column
// tile of the sparse operand is densified in shared memory from its own
// entries (W never exists densely in device memory) and multiplied on the
// tensor cores with a 128-row tile of the dense operand.
//
// Precision.  fp32 results within 1e-5 * sum|w||x| come from an fp16 split:
// every operand value x is scaled by a power of two per row (so the row's
// largest magnitude lands in [2^13, 2^14)), then written as hi = fp16(x) and
// lo = fp16(x - hi); the products hi*hi + hi*lo + lo*hi carry about 22 bits.
// The tensor core's fp32 accumulation truncates, so one accumulator is never
// chained over the whole reduction: two TMEM accumulators take turns, each
// over kTcPeriod windows, and every finished one is added into fp32 registers
// (round to nearest) while the other fills.  Rows and segments the split
// cannot carry (an inf or NaN; values spanning more than ~2^16, see
// tc_needs_exact) are flagged by the per-call passes and their outputs
// recomputed per stored entry by the kernels of snk_tc_exact.cu.
//
// Forward and dX, per call: the dense operand is scaled and split once into
// fp16 hi/lo arrays (k_tc_split), the values are put into tile order, scaled
// per segment and split (k_tc_values), after the segment scales are found
// (k_tc_seg_exp).  Then one CTA per 128 x 192 output tile, 11 warps:
//   warps 0-7  clear one of two sparse stages (the whole stage in denser
//              layers, the entries written there two windows ago in sparse
//              ones), write this window's entries, drain the accumulators and
//              store the output;
//   warp 8     loads the dense hi/lo tiles with TMA into one of two stages;
//   warp 9     issues the MMAs (one thread) and owns the TMEM allocation;
//   warp 10    stages each window's sparse entries (tile offsets and fp16
//              pieces, contiguous in tile order) into one of four shared-memory
//              slots with bulk copies, so the builders never wait on device
//              memory.
// The weight gradient is described at k_tc_sddmm.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "snk_internal.cuh"

namespace snk {

struct TcView {
    int32_t* perm_t = nullptr;    // [nnz] canonical slot of the j-th entry in tile order
    uint16_t* off = nullptr;      // [nnz + pad] byte offset of the entry in its swizzled fp16 tile
    int32_t* tile_ptr = nullptr;  // [n_tiles + 1] first entry of each (segment tile, window);
                                  // weight gradient: [n_tiles * kWGroups + 1], of each (block, group)
    int64_t n_tiles = 0;
    int n_win = 0;                // windows along the reduction dimension
    int n_nt = 0;                 // segment tiles
    int64_t version = -1;         // topology version the view was built for
};

struct TcState {
    // [0]: rows of W in 192 x 64 tiles (forward), [1]: its columns (dX),
    // [2]: 128-row x 192-column blocks of W (weight gradient)
    TcView view[3];
    uint32_t* hl = nullptr;       // [nnz + pad] scaled values in tile order as fp16 hi | lo << 16 (per call)
    int32_t* seg_exp = nullptr;   // [max(out, in)] scale exponent per segment
    int32_t* col_exp = nullptr;   // [in] weight gradient: scale exponent per column of X
    int32_t* run_start = nullptr; // view build: first position of each (tile, bank) run
    int32_t* row_exp = nullptr;   // [kTcChunk] scale exponent per dense row
    __half* dh = nullptr;         // [kTcChunk * k_stride] dense operand, scaled, high part
    __half* dl = nullptr;         // the low part
    int64_t k_stride = 0;         // row stride of dh / dl: max(out, in) rounded up to 8
    // outputs recomputed exactly (see tc_needs_exact): per segment of W (or,
    // for dW, per column of dY) and per column of X the flag bits; the
    // candidate segments; the flagged dense rows of the current chunk; the
    // flagged rows / columns of W for dW (list and set); and the counters and
    // maxima below
    int32_t* seg_code = nullptr;  // [max(out, in)]
    int32_t* col_code = nullptr;  // [in]
    int32_t* cand = nullptr;      // [max(out, in)]
    int32_t* frows = nullptr;     // [kTcChunk]
    int32_t* dw_flag = nullptr;   // [out + in]
    int32_t* dw_list = nullptr;   // [out + in]
    uint32_t* fix = nullptr;      // [kFixWords]
    float* part = nullptr;        // partial sums of split CTAs (small batches)
    int64_t part_len = 0;
};

// Words of TcState::fix: counters, and largest L1 norms and magnitudes as
// fp32 bit patterns (non-negative, so integer atomicMax orders them).  Each
// (L1, max) pair is adjacent: the exact kernels take a pointer to it.
enum {
    kFixRows = 0,     // flagged dense rows in the current chunk
    kFixCand = 1,     // candidate segments
    kFixSegL1 = 2,    // largest sum |v| over the segments of W
    kFixSegMax = 3,   // largest |v| in W
    kFixRowL1 = 4,    // largest sum |x| over the dense rows
    kFixRowMax = 5,   // largest |x| in the dense operand
    kFixDwList = 6,   // flagged rows / columns of W (weight gradient)
    kFixDyL1 = 8,     // weight gradient, per batch chunk: largest column sum of |dY|
    kFixDyMax = 9,    // largest |dY|
    kFixXL1 = 10,     // largest column sum of |X|
    kFixXMax = 11,    // largest |X|
    kFixWords = 12
};

namespace {

constexpr int kTcM = 128;          // dense rows per tile (TMEM lanes)
constexpr int kTcN = 192;          // segments per tile (accumulator columns)
constexpr int kTcK = 64;           // reduction window (128 bytes of fp16)
constexpr int kTcBuilders = 256;   // warps 0-7
constexpr int kTcThreads = kTcBuilders + 96;
constexpr int kTmaWarp = 8, kMmaWarp = 9, kRecWarp = 10;
constexpr int kStagesA = 2, kStagesB = 2;
constexpr int kRecSlots = 4;       // windows of sparse entries staged in shared memory
constexpr int kRecCap = 1536;      // entries staged per window (the rest are read from memory)
// Mean entries per window from which clearing the whole stage (48 KB of
// 16-byte stores) is cheaper than clearing the previous window's entries one
// by one (measured at 1200 entries per window: 13% faster; at 120: slower).
constexpr int64_t kZeroFillEntries = 400;
constexpr int kTcPeriod = 8;       // windows per accumulator turn
constexpr int kTcGroupM = 8;       // dense-row tiles per raster group
constexpr int kTcChunk = 8192;     // dense rows per launch
constexpr int kPieceA = kTcM * kTcK * 2;          // 16 KB
constexpr int kPieceB = kTcN * kTcK * 2;          // 24 KB
constexpr int kStageA = 2 * kPieceA, kStageB = 2 * kPieceB;
constexpr int kRecSlotBytes = kRecCap * 2 + kRecCap * 4;          // offsets, then fp16 pieces
constexpr int kTcSmem = kStagesA * kStageA + kStagesB * kStageB + kRecSlots * kRecSlotBytes + 1024;
constexpr uint32_t kAccStride = 256;              // TMEM columns between the two accumulators
constexpr uint32_t kTmemCols = 512;
constexpr int kColsPerThread = kTcN / 2;          // accumulator columns each builder drains
// Limit of a pipeline wait (about two seconds at the boost clock); a build
// may shorten it (SNK_TC_WAIT_CYCLES) to exercise the abort path.  A wait
// that runs out stops the CTA's pipeline: every role then waits, with the
// fixed drain limit, for the copies and MMAs it has issued, the outputs are
// written as NaN and the status word records kStatLimit.
#ifndef SNK_TC_WAIT_CYCLES
#define SNK_TC_WAIT_CYCLES 4000000000LL
#endif
constexpr long long kTcWaitCycles = SNK_TC_WAIT_CYCLES;
constexpr long long kTcDrainCycles = 4000000000LL;
// kind::f16 instruction descriptor: D fp32, A and B fp16, both K-major,
// N = kTcN, M = kTcM.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kTcN >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);

static_assert(kTcSmem <= 227 * 1024 - 4096, "pipeline stages exceed shared memory");
static_assert(kTcN % 64 == 0 && kTcN <= 256, "two builder halves of whole 32-column loads");
static_assert(kRecCap % 8 == 0, "staged ranges are whole 16-byte units");
constexpr int kTcPad = 16;         // entries readable past nnz in the tile-order arrays
// An fp16 piece of a sparse tile holds kTcN * kTcK / 64 = 192 words per bank,
// so fewer than kRankSpan entries of one window share a bank.
constexpr uint32_t kRankSpan = 512;
static_assert(kTcN * kTcK / 64 * 2 <= (int)kRankSpan, "rank within a bank fits its field");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Byte offset of fp16 element (row i, column k < 64) in a K-major tile with
// the 128-byte swizzle: 8-row atoms of 1024 bytes, 16-byte chunks XORed with
// the row within the atom (the layout a 128-byte-swizzled TMA load writes).
__device__ __forceinline__ uint32_t sw128(int i, int k) {
    return (uint32_t)((i >> 3) * 1024 + (i & 7) * 128 + (((k >> 3) ^ (i & 7)) << 4) + (k & 7) * 2);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
                 : "memory");
}
// Bounded wait on a phase; false once `limit` cycles have passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, long long limit = kTcWaitCycles) {
    long long t0 = 0;
    for (int spin = 0;; ++spin) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(smem_u32(b)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (spin == 0)
            t0 = clock64();
        else if (clock64() - t0 > limit)
            return false;
    }
}
// After a pipeline stopped early: wait for the last `issued` uses of a ring of
// `slots` barriers (window w used barrier w % slots in its (w / slots)-th
// phase), i.e. for every copy still landing in shared memory.
__device__ __forceinline__ bool drain_ring(uint64_t* bars, int slots, int issued) {
    bool ok = true;
    for (int w = issued > slots ? issued - slots : 0; w < issued; ++w)
        if (!mbar_wait(&bars[w % slots], (w / slots) & 1, kTcDrainCycles)) ok = false;
    return ok;
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// 32 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// OR of a flag over the 256 builder threads (named barrier 1).
__device__ __forceinline__ bool builders_any(bool flag) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.cta.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q; }"
        : "=r"(r)
        : "r"((uint32_t)flag), "n"(kTcBuilders)
        : "memory");
    return r != 0;
}

// Power-of-two exponent that brings the largest magnitude m into [2^13, 2^14).
__device__ __forceinline__ int tc_exponent(float m) {
    if (!(m > 0.f) || !isfinite(m)) return 0;
    int E;
    frexpf(m, &E);
    return min(120, max(-120, 14 - E));
}

// fp16 pieces of one scaled value: hi + lo carries about 22 bits.
__device__ __forceinline__ void split16(float x, __half& hi, __half& lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}

struct TcArgs {
    int b;                    // dense rows in this launch
    int64_t K_len;            // reduction length
    const int32_t* row_exp;   // [b]
    const uint16_t* off;      // sparse entries in tile order: tile offsets
    const uint32_t* hl;       // and fp16 pieces
    int zero_fill;            // clear whole stages (dense windows) or entry by entry
    const int32_t* tile_ptr;  // [n_nt * n_win + 1]
    const int32_t* seg_exp;   // [n_seg]
    int64_t n_seg;
    int n_win, n_mt, n_nt;
    const float* bias;        // [n_seg] or null
    float* Y;                 // [b, n_seg]
    int32_t* status;
    int full;                 // tiles computed whole by one CTA each (the first `full` in raster order)
    int split;                // CTAs sharing each remaining tile, each over a range of windows
    float* part;              // [(tile - full) * split + slice][kTcM][kTcN] their partial sums
};

// Output tile `id` in raster order: groups of kTcGroupM dense-row tiles
// sweep all segment tiles.
__device__ __forceinline__ void tc_tile_of(int id, int n_mt, int n_nt, int& mt, int& nt) {
    const int gsz = kTcGroupM * n_nt;
    const int first_m = (id / gsz) * kTcGroupM;
    const int gm = min(n_mt - first_m, kTcGroupM);
    mt = first_m + (id % gsz) % gm;
    nt = (id % gsz) / gm;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    k_tc_spmm(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_l,
              const TcArgs a) {
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    unsigned char* sa = tc_raw + ((1024 - (smem_u32(tc_raw) & 1023)) & 1023);  // A stages
    unsigned char* sb = sa + kStagesA * kStageA;                                // B stages
    unsigned char* sr = sb + kStagesB * kStageB;                                // staged entries
    __shared__ uint64_t full_a[kStagesA], empty_a[kStagesA], full_b[kStagesB], empty_b[kStagesB];
    __shared__ uint64_t rec_full[kRecSlots], rec_empty[kRecSlots];
    __shared__ uint64_t accf[2], acce[2], fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float pw_seg[kTcN];   // 2^e of each segment of the tile
    // per staging slot: the window's entries [j0, j1), offsets staged from
    // index ca up to ce, fp16 pieces from va up to ve
    __shared__ int rec_info[kRecSlots][6];

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    // CTAs below `full` take one whole tile each; the others share the
    // remaining tiles `split` ways, slice sk taking windows [w0, w1)
    const bool whole = (int)blockIdx.x < a.full;
    const int jt = whole ? 0 : (int)blockIdx.x - a.full;   // slot of a shared tile's slice
    const int id = whole ? (int)blockIdx.x : a.full + jt / a.split;
    const int sk = whole ? 0 : jt % a.split;
    const int spl = whole ? 1 : a.split;
    int mt, nt;
    tc_tile_of(id, a.n_mt, a.n_nt, mt, nt);
    const int64_t r0 = (int64_t)mt * kTcM;    // first dense row
    const int64_t s0 = (int64_t)nt * kTcN;    // first segment
    const int w0 = (int)((int64_t)a.n_win * sk / spl);
    const int n_win = (int)((int64_t)a.n_win * (sk + 1) / spl) - w0;   // windows of this CTA
    const int32_t* tp = a.tile_ptr + (int64_t)nt * a.n_win + w0;

    if (t == 0) {
        for (int i = 0; i < kStagesA; ++i) {
            mbar_init(&full_a[i], 1);
            mbar_init(&empty_a[i], 1);
        }
        for (int i = 0; i < kStagesB; ++i) {
            mbar_init(&full_b[i], kTcBuilders);
            mbar_init(&empty_b[i], 1);
        }
        for (int i = 0; i < kRecSlots; ++i) {
            mbar_init(&rec_full[i], 1);
            mbar_init(&rec_empty[i], kTcBuilders);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], kTcBuilders);
        }
        mbar_init(&fin, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (t < kTcN) {
        const int64_t sg = s0 + t;
        pw_seg[t] = ldexpf(1.f, sg < a.n_seg ? a.seg_exp[sg] : 0);
    }
    // the sparse stages start zeroed; later each is cleared before it is rewritten
    if (t < kTcBuilders) {
        uint4* pb = reinterpret_cast<uint4*>(sb);
        for (int i = t; i < kStagesB * kStageB / 16; i += kTcBuilders) pb[i] = make_uint4(0, 0, 0, 0);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    bool ok = true;   // this thread saw no wait run out

    if (warp == kTmaWarp) {
        // ---------------------------------------------------------------- dense tiles (TMA)
        if (lane == 0) {
            int w = 0;
            for (; w < n_win; ++w) {
                const int s = w % kStagesA;
                if (w >= kStagesA && !mbar_wait(&empty_a[s], ((w / kStagesA) - 1) & 1)) {
                    ok = false;
                    break;
                }
                unsigned char* st = sa + s * kStageA;
                mbar_expect_tx(&full_a[s], kStageA);
                tma_load_2d(st, &map_h, (w0 + w) * kTcK, (int)r0, &full_a[s]);
                tma_load_2d(st + kPieceA, &map_l, (w0 + w) * kTcK, (int)r0, &full_a[s]);
            }
            if (!ok) drain_ring(full_a, kStagesA, w);
        }
        __syncwarp();
    } else if (warp == kRecWarp) {
        // ---------------------------------------------------------------- sparse entries (bulk copies)
        if (lane == 0) {
            int w = 0;
            for (; w < n_win; ++w) {
                const int r = w % kRecSlots;
                if (w >= kRecSlots && !mbar_wait(&rec_empty[r], ((w / kRecSlots) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int j0 = tp[w], j1 = tp[w + 1];
                const int ca = j0 & ~7, ce = j1 > j0 ? min((j1 + 7) & ~7, ca + kRecCap) : ca;
                const int va = j0 & ~3, ve = j1 > j0 ? min((j1 + 3) & ~3, va + kRecCap) : va;
                int* info = rec_info[r];
                info[0] = j0;
                info[1] = j1;
                info[2] = ca;
                info[3] = ce;
                info[4] = va;
                info[5] = ve;
                const uint32_t bc = (uint32_t)(ce - ca) * 2, bv = (uint32_t)(ve - va) * 4;
                unsigned char* slot = sr + r * kRecSlotBytes;
                mbar_expect_tx(&rec_full[r], bc + bv);
                if (bc) bulk_load(slot, a.off + ca, bc, &rec_full[r]);
                if (bv) bulk_load(slot + kRecCap * 2, a.hl + va, bv, &rec_full[r]);
            }
            if (!ok) drain_ring(rec_full, kRecSlots, w);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            for (int w = 0; w < n_win; ++w) {
                const int s_a = w % kStagesA, s_b = w % kStagesB;
                const int q = w / kTcPeriod, ab = q & 1;
                const bool first = (w % kTcPeriod) == 0;
                if (!mbar_wait(&full_a[s_a], (w / kStagesA) & 1) ||
                    !mbar_wait(&full_b[s_b], (w / kStagesB) & 1) ||
                    (first && q >= 2 && !mbar_wait(&acce[ab], ((q >> 1) - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ah = smem_u32(sa + s_a * kStageA), al = ah + kPieceA;
                const uint32_t bh = smem_u32(sb + s_b * kStageB), bl = bh + kPieceB;
                const uint32_t d = tmem + ab * kAccStride;
#pragma unroll
                for (int kk = 0; kk < kTcK / 16; ++kk) {
                    const uint32_t o = 32 * kk;
                    mma_f16(d, desc_sw128(ah + o), desc_sw128(bh + o), (first && kk == 0) ? 0u : 1u);
                    mma_f16(d, desc_sw128(ah + o), desc_sw128(bl + o), 1u);
                    mma_f16(d, desc_sw128(al + o), desc_sw128(bh + o), 1u);
                }
                if (w + kStagesA < n_win) mma_commit(&empty_a[s_a]);
                if (w + kStagesB < n_win) mma_commit(&empty_b[s_b]);
                if ((w % kTcPeriod) == kTcPeriod - 1 || w == n_win - 1) mma_commit(&accf[ab]);
            }
            // every MMA issued has completed once fin completes (also after
            // an early stop: TMEM and the stages are released only then)
            mma_commit(&fin);
            if (!mbar_wait(&fin, 0, kTcDrainCycles)) ok = false;
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- builders
        const int lq = warp & 3;         // TMEM lane quarter this warp may read
        const int half = warp >> 2;      // accumulator columns [half * kColsPerThread, ...)
        float acc[kColsPerThread];
#pragma unroll
        for (int j = 0; j < kColsPerThread; ++j) acc[j] = 0.f;
        const int n_per = (n_win + kTcPeriod - 1) / kTcPeriod;
        int drained = 0;
        // add accumulator turn q into the registers and hand the accumulator back;
        // the whole warp reads TMEM or none of it does
        auto drain = [&](int q) {
            const int ab = q & 1;
            const bool got = __all_sync(0xffffffffu, mbar_wait(&accf[ab], (q >> 1) & 1));
            if (!got) return false;
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * lq) << 16) + ab * kAccStride + kColsPerThread * half;
#pragma unroll
            for (int c = 0; c < kColsPerThread / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(ta + 32 * c, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[32 * c + i] += __uint_as_float(r[i]);
            }
            tc_fence_before();
            mbar_arrive(&acce[ab]);
            return true;
        };
        for (int w = 0; w < n_win; ++w) {
            const int s = w % kStagesB, r = w % kRecSlots;
            if (w >= kStagesB && !mbar_wait(&empty_b[s], ((w / kStagesB) - 1) & 1)) ok = false;
            // turn q is complete once window (q+1)P - 1 has left its stage
            if (drained < n_per && w == (drained + 1) * kTcPeriod + kStagesB - 1) {
                if (!drain(drained)) ok = false;
                ++drained;
            }
            if (!mbar_wait(&rec_full[r], (w / kRecSlots) & 1)) ok = false;
            unsigned char* Bh = sb + s * kStageB;
            unsigned char* Bl = Bh + kPieceB;
            if (a.zero_fill && w >= kStagesB && ok) {
                // dense windows: 16-byte stores clear the whole stage
                uint4* pb = reinterpret_cast<uint4*>(Bh);
#pragma unroll 4
                for (int i = t; i < kStageB / 16; i += kTcBuilders) pb[i] = make_uint4(0, 0, 0, 0);
            }
            if (!a.zero_fill && w >= kStagesB && ok) {
                // sparse windows: clear what window w - kStagesB wrote into
                // this stage, then release its staging slot
                const int ro = (w - kStagesB) % kRecSlots;
                const int* info = rec_info[ro];
                const uint16_t* sc = reinterpret_cast<const uint16_t*>(sr + ro * kRecSlotBytes);
                const int j1 = info[1], ca = info[2], ce = info[3];
                for (int j = info[0] + t; j < j1; j += kTcBuilders) {
                    const uint32_t off = j < ce ? sc[j - ca] : a.off[j];
                    *reinterpret_cast<uint16_t*>(Bh + off) = 0;
                    *reinterpret_cast<uint16_t*>(Bl + off) = 0;
                }
                mbar_arrive(&rec_empty[ro]);
            }
            // every clear lands before this window's writes; a wait that ran
            // out anywhere stops all builders here
            if (builders_any(!ok)) {
                ok = false;
                break;
            }
            {
                const int* info = rec_info[r];
                const unsigned char* slot = sr + r * kRecSlotBytes;
                const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot);
                const uint32_t* sv = reinterpret_cast<const uint32_t*>(slot + kRecCap * 2);
                const int j1 = info[1], ca = info[2], ce = info[3], va = info[4], ve = info[5];
                for (int j = info[0] + t; j < j1; j += kTcBuilders) {
                    const uint32_t off = j < ce ? sc[j - ca] : a.off[j];
                    const uint32_t v = j < ve ? sv[j - va] : a.hl[j];
                    *reinterpret_cast<uint16_t*>(Bh + off) = (uint16_t)(v & 0xFFFFu);
                    *reinterpret_cast<uint16_t*>(Bl + off) = (uint16_t)(v >> 16);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&full_b[s]);
            if (a.zero_fill) mbar_arrive(&rec_empty[r]);   // this window's staged entries are used
        }
        while (ok && drained < n_per) {
            ok = drain(drained);
            ++drained;
        }
        // ---------------------------------------------------------------- epilogue
        const int row = 32 * lq + lane;
        const int64_t rr = r0 + row;
        if (rr < a.b) {
            // undo the two power-of-two scalings (each factor a normal float);
            // a slice of a shared tile leaves its partial sum, in tile
            // coordinates, for k_tc_split_sum
            const float ir = ok ? ldexpf(1.f, -a.row_exp[rr]) : __int_as_float(0x7fc00000);
            float* yrow = whole ? a.Y + rr * a.n_seg + s0 : a.part + ((int64_t)jt * kTcM + row) * kTcN;
            const float* bias = whole ? a.bias : nullptr;
            const int c0 = kColsPerThread * half;
#pragma unroll
            for (int j = 0; j < kColsPerThread; ++j) {
                const int64_t sg = s0 + c0 + j;
                if (sg < a.n_seg) {
                    float y = (acc[j] * ir) * __frcp_rn(pw_seg[c0 + j]);
                    if (bias) y += bias[sg];
                    yrow[c0 + j] = y;
                }
            }
        }
    }
    if (!ok) atomicExch(&abort_flag, 1);
    tc_fence_before();
    __syncthreads();
    if (abort_flag && t == 0) atomicOr(a.status, kStatLimit);
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// Y = bias + the slices' partial sums of every shared tile (tiles full ..
// tiles - 1 in raster order), added in slice order.  Blocks (shared tile,
// slice of its outputs): every output's loads are in flight at once (one
// block per tile, looping over its 24,576 outputs, left each thread ~100
// dependent rounds).
__global__ void k_tc_split_sum(const float* __restrict__ part, int full, int split, int n_mt, int n_nt,
                               int64_t rows, int64_t n_seg, const float* __restrict__ bias, float* __restrict__ Y) {
    const int tl = blockIdx.x;   // shared tile, counted from `full`
    int mt, nt;
    tc_tile_of(full + tl, n_mt, n_nt, mt, nt);
    const int64_t r0 = (int64_t)mt * kTcM, s0 = (int64_t)nt * kTcN;
    for (int i = blockIdx.y * blockDim.x + threadIdx.x; i < kTcM * kTcN; i += gridDim.y * blockDim.x) {
        const int row = i / kTcN, col = i % kTcN;
        const int64_t rr = r0 + row, sg = s0 + col;
        if (rr >= rows || sg >= n_seg) continue;
        float y = 0.f;
        for (int k = 0; k < split; ++k) y += part[((int64_t)(tl * split + k) * kTcM + row) * kTcN + col];
        Y[rr * n_seg + sg] = bias ? y + bias[sg] : y;
    }
}

// Dense operand, once per call: per row the scale exponent of its largest
// finite magnitude, and the scaled values split into fp16 hi / lo at row
// stride ks (one block per row; non-finite values are split as zeros).  The
// row's code (an inf or NaN; the count of nonzero values below 2^-3 after
// scaling) is checked against W's largest segment sum and magnitude
// (tc_needs_exact); a row that fails is listed in rows[] for the exact
// recomputation.  The row's sum of finite magnitudes and its largest one go
// into the running maxima that the segments' own check uses.
template <bool VEC>
__global__ void k_tc_split(const float* __restrict__ D, int64_t len, int64_t ks, int32_t* __restrict__ e_out,
                           __half* __restrict__ dh, __half* __restrict__ dl, int32_t* __restrict__ rows,
                           uint32_t* __restrict__ fix) {
    __shared__ float red[3][32];
    __shared__ int red_n[32];
    const int64_t r = blockIdx.x;
    const float* p = D + r * len;
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5, lane = threadIdx.x & 31;
    float m = 0.f, sum = 0.f, nf = 0.f;
    auto take = [&](float x) {
        x = fabsf(x);
        if (isfinite(x)) {
            m = fmaxf(m, x);
            sum += x;
        } else {
            nf = 1.f;
        }
    };
    if (VEC) {
        for (int64_t k = 4 * threadIdx.x; k < len; k += 4 * blockDim.x) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p + k));
            take(v.x);
            take(v.y);
            take(v.z);
            take(v.w);
        }
    } else {
        for (int64_t k = threadIdx.x; k < len; k += blockDim.x) take(p[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        nf = fmaxf(nf, __shfl_xor_sync(0xffffffffu, nf, o));
    }
    if (lane == 0) {
        red[0][w] = m;
        red[1][w] = sum;
        red[2][w] = nf;
    }
    __syncthreads();
    m = 0.f;
    sum = 0.f;
    nf = 0.f;
    for (int i = 0; i < nw; ++i) {   // every thread reduces the warp results in the same order
        m = fmaxf(m, red[0][i]);
        sum += red[1][i];
        nf = fmaxf(nf, red[2][i]);
    }
    const int e = tc_exponent(m);
    const float pw = ldexpf(1.f, e);
    const float tiny = ldexpf(0.125f, -e);
    int n_tiny = 0;
    auto scaled = [&](float x) {
        const float ax = fabsf(x);
        n_tiny += (ax > 0.f && ax < tiny) ? 1 : 0;
        return isfinite(x) ? x * pw : 0.f;
    };
    __half* oh = dh + r * ks;
    __half* ol = dl + r * ks;
    if (VEC) {
        for (int64_t k = 4 * threadIdx.x; k < len; k += 4 * blockDim.x) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p + k));
            __half h0, h1, h2, h3, l0, l1, l2, l3;
            split16(scaled(v.x), h0, l0);
            split16(scaled(v.y), h1, l1);
            split16(scaled(v.z), h2, l2);
            split16(scaled(v.w), h3, l3);
            uint2 hh, ll;
            hh.x = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            hh.y = (uint32_t)__half_as_ushort(h2) | ((uint32_t)__half_as_ushort(h3) << 16);
            ll.x = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
            ll.y = (uint32_t)__half_as_ushort(l2) | ((uint32_t)__half_as_ushort(l3) << 16);
            *reinterpret_cast<uint2*>(oh + k) = hh;
            *reinterpret_cast<uint2*>(ol + k) = ll;
        }
    } else {
        for (int64_t k = threadIdx.x; k < len; k += blockDim.x) {
            __half h, l;
            split16(scaled(p[k]), h, l);
            oh[k] = h;
            ol[k] = l;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n_tiny += __shfl_xor_sync(0xffffffffu, n_tiny, o);
    if (lane == 0) red_n[w] = n_tiny;
    __syncthreads();
    if (threadIdx.x == 0) {
        int n = 0;
        for (int i = 0; i < nw; ++i) n += red_n[i];
        e_out[r] = e;
        const int cd = (nf > 0.f ? 1 : 0) | (n << 1);
        if (tc_needs_exact(cd, e, __uint_as_float(fix[kFixSegL1]), __uint_as_float(fix[kFixSegMax])))
            rows[atomicAdd(fix + kFixRows, 1u)] = (int32_t)r;
        atomicMax(fix + kFixRowL1, __float_as_uint(sum));
        atomicMax(fix + kFixRowMax, __float_as_uint(m));
    }
}

// ------------------------------------------------------------ weight gradient
// dW_k = sum_b dY[b, r_k] X[b, c_k] on the tensor cores: the dense product
// dY^T X over one batch chunk for 128-row x 192-column blocks of W, kept
// only at each block's entries.  A = dY^T (rows of W, batch contiguous) and
// B = X^T (columns of W), both scaled per row and split into fp16 hi / lo by
// k_tc_tsplit, arrive by TMA; the accumulators take turns and are drained
// into registers as in k_tc_spmm.
//
// The CTAs are persistent, one per SM: CTA c takes the blocks c, c + grid,
// c + 2 grid, ... in raster order, and counts its windows, accumulator turns
// and barrier phases across them, so the loads and MMAs of its next block
// run while the builders drain and write out the last one.  The write-out
// needs no block-wide step: builder warp (quarter q, half h) owns the block's
// rows 32q..32q+31 (its TMEM lanes) and columns 96h..96h+95, and writes its
// sums one 32 x 32 chunk at a time into its own shared-memory scratch, from
// which its lanes send the chunk's entries to their canonical slots.  The
// weight-gradient view lists every block's entries grouped by (quarter,
// chunk) for this.
struct TcwArgs {
    int n_win;                 // batch windows in this chunk
    int n_ot, n_it;            // row blocks (of kTcM) and column blocks (of kTcN) of W
    int64_t out_f, in_f;
    const int32_t* e_row;      // [out] scale exponents of dY^T rows
    const int32_t* e_col;      // [in] scale exponents of X^T rows
    const int32_t* perm;       // weight-gradient view: canonical slot per entry
    const uint16_t* off;       // row within the quarter * 32 + column within the chunk
    const int32_t* group_ptr;  // [n_ot * n_it * kWGroups + 1] first entry of each (block, group)
    float* dW;
    int accumulate;            // add to dW (later batch chunks) instead of writing it
    int32_t* status;
};

constexpr int kWThreads = kTcBuilders + 64;       // 8 drain warps, a TMA warp, an MMA warp
constexpr int kWStage = kStageA + kStageB;        // one batch window of A and B
constexpr int kWChunks = kTcN / 32;               // 32-column chunks per block
constexpr int kWGroups = 32;                      // group slots per block: quarter * kWChunks + chunk
constexpr int kWScratch = 32 * 33;                // floats per builder warp: one chunk, rows padded
constexpr int kWUnroll = 4;                       // entries per lane whose loads are in flight together
constexpr int kWSmem = 2 * kWStage + (kTcBuilders / 32) * kWScratch * 4 + 1024;
static_assert((kTcM / 32) * kWChunks <= kWGroups, "quarters and chunks fit the group slots");
static_assert(kColsPerThread == 3 * 32, "each builder warp owns three chunks");
static_assert(kWSmem <= 227 * 1024 - 4096, "stages and scratch exceed shared memory");

__global__ void __launch_bounds__(kWThreads, 1)
    k_tc_sddmm(const __grid_constant__ CUtensorMap map_ah, const __grid_constant__ CUtensorMap map_al,
               const __grid_constant__ CUtensorMap map_bh, const __grid_constant__ CUtensorMap map_bl,
               const TcwArgs a) {
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    unsigned char* sm = tc_raw + ((1024 - (smem_u32(tc_raw) & 1023)) & 1023);
    __shared__ uint64_t full[2], empty[2], accf[2], acce[2], fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int n_win = a.n_win;
    const int n_per = (n_win + kTcPeriod - 1) / kTcPeriod;
    const int tiles = a.n_ot * a.n_it;
    const int grid = (int)gridDim.x, first = (int)blockIdx.x;
    const int mine = (tiles - first + grid - 1) / grid;   // blocks of this CTA (grid <= tiles)

    if (t == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], kTcBuilders);
        }
        mbar_init(&fin, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    bool ok = true;

    if (warp == kTmaWarp) {
        if (lane == 0) {
            int gw = 0;   // windows issued by this CTA, over all its blocks
            for (int i = 0; i < mine && ok; ++i) {
                int ot, it;
                tc_tile_of(first + i * grid, a.n_ot, a.n_it, ot, it);
                const int y0 = ot * kTcM, x0 = it * kTcN;
                for (int w = 0; w < n_win; ++w, ++gw) {
                    const int s = gw & 1;
                    if (gw >= 2 && !mbar_wait(&empty[s], ((gw >> 1) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    unsigned char* st = sm + s * kWStage;
                    mbar_expect_tx(&full[s], kWStage);
                    tma_load_2d(st, &map_ah, w * kTcK, y0, &full[s]);
                    tma_load_2d(st + kPieceA, &map_al, w * kTcK, y0, &full[s]);
                    tma_load_2d(st + kStageA, &map_bh, w * kTcK, x0, &full[s]);
                    tma_load_2d(st + kStageA + kPieceB, &map_bl, w * kTcK, x0, &full[s]);
                }
            }
            if (!ok) drain_ring(full, 2, gw);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const int total = mine * n_win;
            int gw = 0;
            for (int i = 0; i < mine && ok; ++i) {
                for (int w = 0; w < n_win; ++w, ++gw) {
                    const int s = gw & 1;
                    const int q = i * n_per + w / kTcPeriod, ab = q & 1;   // accumulator turn
                    const bool turn0 = (w % kTcPeriod) == 0;
                    if (!mbar_wait(&full[s], (gw >> 1) & 1) ||
                        (turn0 && q >= 2 && !mbar_wait(&acce[ab], ((q >> 1) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ah = smem_u32(sm + s * kWStage), al = ah + kPieceA;
                    const uint32_t bh = ah + kStageA, bl = bh + kPieceB;
                    const uint32_t d = tmem + ab * kAccStride;
#pragma unroll
                    for (int kk = 0; kk < kTcK / 16; ++kk) {
                        const uint32_t o = 32 * kk;
                        mma_f16(d, desc_sw128(ah + o), desc_sw128(bh + o), (turn0 && kk == 0) ? 0u : 1u);
                        mma_f16(d, desc_sw128(ah + o), desc_sw128(bl + o), 1u);
                        mma_f16(d, desc_sw128(al + o), desc_sw128(bh + o), 1u);
                    }
                    if (gw + 2 < total) mma_commit(&empty[s]);
                    if ((w % kTcPeriod) == kTcPeriod - 1 || w == n_win - 1) mma_commit(&accf[ab]);
                }
            }
            mma_commit(&fin);
            if (!mbar_wait(&fin, 0, kTcDrainCycles)) ok = false;
        }
        __syncwarp();
    } else {
        const int lq = warp & 3, half = warp >> 2;
        const int row = 32 * lq + lane;
        float* scr = reinterpret_cast<float*>(sm + 2 * kWStage) + warp * kWScratch;
        // false once one of this warp's waits has run out (the same in every
        // lane): from then on its entries get NaN, so none is left stale
        bool wok = true;
        for (int i = 0; i < mine; ++i) {
            int ot, it;
            tc_tile_of(first + i * grid, a.n_ot, a.n_it, ot, it);
            const int64_t o0 = (int64_t)ot * kTcM, i0 = (int64_t)it * kTcN;
            // the block's scales and entry ranges, loaded before the wait
            const float ir = ldexpf(1.f, o0 + row < a.out_f ? -a.e_row[o0 + row] : 0);
            float ic[3];
#pragma unroll
            for (int cc = 0; cc < 3; ++cc) {
                const int64_t col = i0 + 32 * (3 * half + cc) + lane;
                ic[cc] = ldexpf(1.f, col < a.in_f ? -a.e_col[col] : 0);
            }
            const int32_t* gp =
                a.group_ptr + ((int64_t)ot * a.n_it + it) * kWGroups + lq * kWChunks + 3 * half;
            int jr[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) jr[k] = gp[k];
            // kWUnroll entries per lane at a time, their loads issued together;
            // the first batch of each chunk is loaded one step early (the first
            // chunk's before the drain)
            auto load = [&](int jb, int j1, int (&o)[kWUnroll], int (&pm)[kWUnroll]) {
#pragma unroll
                for (int u = 0; u < kWUnroll; ++u) {
                    const int j = jb + 32 * u + lane;
                    o[u] = j < j1 ? (int)__ldg(a.off + j) : 0;
                    pm[u] = j < j1 ? __ldg(a.perm + j) : 0;
                }
            };
            auto send = [&](int jb, int j1, float cscale, const int (&o)[kWUnroll], const int (&pm)[kWUnroll]) {
#pragma unroll
                for (int u = 0; u < kWUnroll; ++u) {
                    const float cs = __shfl_sync(0xffffffffu, cscale, o[u] & 31);
                    if (jb + 32 * u + lane < j1) {
                        float* dst = a.dW + pm[u];
                        if (!wok) {
                            *dst = __int_as_float(0x7fc00000);
                        } else {
                            const float v = scr[o[u] + (o[u] >> 5)] * cs;
                            *dst = a.accumulate ? *dst + v : v;
                        }
                    }
                }
            };
            int o_cur[kWUnroll], p_cur[kWUnroll];
            load(jr[0], jr[1], o_cur, p_cur);
            float acc[kColsPerThread];
#pragma unroll
            for (int j = 0; j < kColsPerThread; ++j) acc[j] = 0.f;
            for (int ql = 0; ql < n_per && wok; ++ql) {
                const int q = i * n_per + ql, ab = q & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&accf[ab], (q >> 1) & 1))) {
                    wok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ta =
                    tmem + ((uint32_t)(32 * lq) << 16) + ab * kAccStride + kColsPerThread * half;
#pragma unroll
                for (int c = 0; c < kColsPerThread / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(ta + 32 * c, r);
#pragma unroll
                    for (int k = 0; k < 32; ++k) acc[32 * c + k] += __uint_as_float(r[k]);
                }
                tc_fence_before();
                mbar_arrive(&acce[ab]);
            }
#pragma unroll
            for (int cc = 0; cc < 3; ++cc) {
                if (wok) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) scr[lane * 33 + k] = acc[32 * cc + k] * ir;
                }
                __syncwarp();
                int o_nxt[kWUnroll], p_nxt[kWUnroll];
                if (cc < 2) load(jr[cc + 1], jr[cc + 2], o_nxt, p_nxt);
                const int j1 = jr[cc + 1];
                send(jr[cc], j1, ic[cc], o_cur, p_cur);
                for (int jb = jr[cc] + 32 * kWUnroll; jb < j1; jb += 32 * kWUnroll) {
                    load(jb, j1, o_cur, p_cur);
                    send(jb, j1, ic[cc], o_cur, p_cur);
                }
                __syncwarp();
                if (cc < 2) {
#pragma unroll
                    for (int u = 0; u < kWUnroll; ++u) {
                        o_cur[u] = o_nxt[u];
                        p_cur[u] = p_nxt[u];
                    }
                }
            }
        }
        ok = wok;
    }
    if (!ok) atomicExch(&abort_flag, 1);
    tc_fence_before();
    __syncthreads();
    if (abort_flag && t == 0) atomicOr(a.status, kStatLimit);
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// Per column of D [rows, n]: the scale exponent of its largest finite
// magnitude, its code's inf / NaN bit (k_tc_tsplit adds the count of values
// under the fp16 floor; see tc_needs_exact), the running maxima over columns
// of the sum of finite magnitudes and of the largest one (l1max[0], l1max[1],
// fp32 bit patterns) and, if sum is given, the column's plain sum (written,
// or added when accumulate), summed in runs of 32 rows and then pairwise so
// no fp32 chain exceeds ~45 terms; an inf or NaN propagates into that sum as
// it does in the definition.
template <bool SUM>
__global__ void __launch_bounds__(256) k_tc_colstats(const float* __restrict__ D, int64_t rows, int64_t n,
                                                     int32_t* __restrict__ e_out, int32_t* __restrict__ code,
                                                     uint32_t* __restrict__ l1max, float* __restrict__ sum,
                                                     int accumulate) {
    __shared__ float sm_max[8][32], sm_sum[8][32], sm_abs[8][32], sm_nf[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t col = (int64_t)blockIdx.x * 32 + lane;
    float m = 0.f, tot = 0.f, ab = 0.f, nf = 0.f;
    if (col < n) {
        for (int64_t g = w; g * 32 < rows; g += 8) {
            float part = 0.f;
            const int64_t r1 = min(rows, g * 32 + 32);
            for (int64_t r = g * 32; r < r1; ++r) {
                const float x = D[r * n + col];
                const float ax = fabsf(x);
                if (isfinite(ax)) {
                    m = fmaxf(m, ax);
                    ab += ax;
                } else {
                    nf = 1.f;
                }
                if (SUM) part += x;
            }
            if (SUM) tot += part;
        }
    }
    sm_max[w][lane] = m;
    sm_sum[w][lane] = tot;
    sm_abs[w][lane] = ab;
    sm_nf[w][lane] = nf;
    __syncthreads();
    if (w == 0 && col < n) {
        for (int i = 1; i < 8; ++i) {
            m = fmaxf(m, sm_max[i][lane]);
            ab += sm_abs[i][lane];
            nf = fmaxf(nf, sm_nf[i][lane]);
        }
        if (SUM) {
            const float s01 = sm_sum[0][lane] + sm_sum[1][lane], s23 = sm_sum[2][lane] + sm_sum[3][lane];
            const float s45 = sm_sum[4][lane] + sm_sum[5][lane], s67 = sm_sum[6][lane] + sm_sum[7][lane];
            const float s = (s01 + s23) + (s45 + s67);
            sum[col] = accumulate ? sum[col] + s : s;
        }
        e_out[col] = tc_exponent(m);
        code[col] = nf > 0.f ? 1 : 0;
        atomicMax(l1max, __float_as_uint(ab));
        atomicMax(l1max + 1, __float_as_uint(m));
    }
}

// Weight gradient, per batch chunk: the rows (dY columns, list value r) and
// columns (X columns, list value out + c) of W whose entries are recomputed
// exactly (tc_needs_exact against the other operand's maxima, scaled by the
// number of chunks, since each chunk adds its own floor error), each listed
// once per call however many chunks flag it.
__global__ void k_tc_dw_decide(const int32_t* __restrict__ e_row, const int32_t* __restrict__ code_row,
                               const int32_t* __restrict__ e_col, const int32_t* __restrict__ code_col,
                               int64_t out_f, int64_t in_f, float n_chunks, int32_t* __restrict__ flag,
                               int32_t* __restrict__ list, uint32_t* __restrict__ fix) {
    const float dy_l1 = __uint_as_float(fix[kFixDyL1]) * n_chunks;
    const float dy_mx = __uint_as_float(fix[kFixDyMax]) * n_chunks;
    const float x_l1 = __uint_as_float(fix[kFixXL1]) * n_chunks;
    const float x_mx = __uint_as_float(fix[kFixXMax]) * n_chunks;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < out_f + in_f;
         u += (int64_t)gridDim.x * blockDim.x) {
        const bool is_row = u < out_f;
        const int64_t i = is_row ? u : u - out_f;
        const bool need = is_row ? tc_needs_exact(code_row[i], e_row[i], x_l1, x_mx)
                                 : tc_needs_exact(code_col[i], e_col[i], dy_l1, dy_mx);
        if (need && atomicOr(flag + u, 1) == 0) list[atomicAdd(fix + kFixDwList, 1u)] = (int32_t)u;
    }
}

// out[c][r] = split(D[r][c] * 2^e[c]) for r < rows, c < n: the transposed,
// scaled fp16 pieces (row stride bs) the weight-gradient product loads
// (non-finite values are split as zeros); each column's count of nonzero
// values below 2^-3 after scaling is added into its code (2 per value).
__global__ void k_tc_tsplit(const float* __restrict__ D, int64_t rows, int64_t n, const int32_t* __restrict__ e,
                            int64_t bs, __half* __restrict__ oh, __half* __restrict__ ol,
                            int32_t* __restrict__ code) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
    const int64_t c0 = (int64_t)blockIdx.x * 32, r0 = (int64_t)blockIdx.y * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t r = r0 + ty + 8 * i, c = c0 + tx;
        tile[ty + 8 * i][tx] = (r < rows && c < n) ? D[r * n + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t c = c0 + ty + 8 * i, r = r0 + tx;
        int n_tiny = 0;
        if (c < n && r < rows) {
            __half h, l;
            const float x = tile[tx][ty + 8 * i];
            const int ex = e[c];
            const float ax = fabsf(x);
            n_tiny = (ax > 0.f && ax < ldexpf(0.125f, -ex)) ? 1 : 0;
            split16(isfinite(x) ? x * ldexpf(1.f, ex) : 0.f, h, l);
            oh[c * bs + r] = h;
            ol[c * bs + r] = l;
        }
        // the 32 lanes of this warp hold the rows of one column
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) n_tiny += __shfl_xor_sync(0xffffffffu, n_tiny, o);
        if (tx == 0 && n_tiny) atomicAdd(code + c, 2 * n_tiny);
    }
}

// ------------------------------------------------------------ per-call passes
// Per segment of W (a row, or a column through perm): the scale exponent of
// its largest finite magnitude, and bit 0 of its code (tc_needs_exact: it
// holds an inf or NaN); k_tc_values adds the count of its tiny values.  Also
// the largest sum of finite magnitudes over the segments and the largest
// magnitude, which the dense rows' own check uses.
__global__ void k_tc_seg_exp(const int32_t* __restrict__ ptr, const float* __restrict__ v,
                             const int32_t* __restrict__ perm, int64_t n_seg, int32_t* __restrict__ e,
                             int32_t* __restrict__ code, uint32_t* __restrict__ fix) {
    __shared__ float red[2][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    // the block's largest segment sum and magnitude, sent once per block: one
    // atomic per segment on the same two words serialised in the L2
    float m_run = 0.f, s_run = 0.f;
    for (int64_t sg = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; sg < n_seg;
         sg += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int k0 = ptr[sg], k1 = ptr[sg + 1];
        float m = 0.f, sum = 0.f;
        bool nf = false;
        for (int k = k0 + lane; k < k1; k += 32) {
            const float x = fabsf(perm ? v[perm[k]] : v[k]);
            if (isfinite(x)) {
                m = fmaxf(m, x);
                sum += x;
            } else {
                nf = true;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
        }
        nf = __any_sync(0xffffffffu, nf);
        if (lane == 0) {
            e[sg] = tc_exponent(m);
            code[sg] = nf ? 1 : 0;
        }
        m_run = fmaxf(m_run, m);
        s_run = fmaxf(s_run, sum);
    }
    if (lane == 0) {
        red[0][w] = s_run;
        red[1][w] = m_run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < (int)(blockDim.x >> 5); ++i) {
            s_run = fmaxf(s_run, red[0][i]);
            m_run = fmaxf(m_run, red[1][i]);
        }
        atomicMax(fix + kFixSegL1, __float_as_uint(s_run));
        atomicMax(fix + kFixSegMax, __float_as_uint(m_run));
    }
}

// Segments with a nonzero code (an inf or NaN, or tiny values) become
// candidates for the exact recomputation.
__global__ void k_tc_seg_cand(const int32_t* __restrict__ code, int64_t n_seg, int32_t* __restrict__ cand,
                              uint32_t* __restrict__ fix) {
    for (int64_t sg = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; sg < n_seg;
         sg += (int64_t)gridDim.x * blockDim.x)
        if (code[sg]) cand[atomicAdd(fix + kFixCand, 1u)] = (int32_t)sg;
}

// The values in tile order, scaled by their segment's power of two and
// split into fp16 hi | lo << 16 (seg_of: rows for W's rows, cols for its
// columns).  Each nonzero value below 2^-3 after scaling adds 2 to its
// segment's code (the tiny count of tc_needs_exact).
__global__ void k_tc_values(const float* __restrict__ v, const int32_t* __restrict__ perm_t,
                            const int32_t* __restrict__ seg_of, const int32_t* __restrict__ seg_exp, int64_t n,
                            uint32_t* __restrict__ hl, int32_t* __restrict__ code) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const int32_t k = perm_t[j];
        const float x = v[k];
        const int32_t sg = seg_of[k];
        const int ex = seg_exp[sg];   // in [-120, 120]: 2^ex and 2^(-3-ex) are normal floats
        const float ax = fabsf(x);
        if (ax > 0.f && ax < __int_as_float((124 - ex) << 23)) atomicAdd(code + sg, 2);
        __half h, l;
        // an inf or NaN flags its segment for the exact recomputation; the
        // tile holds a zero in its place
        split16(isfinite(x) ? x * __int_as_float((127 + ex) << 23) : 0.f, h, l);
        hl[j] = (uint32_t)__half_as_ushort(h) | ((uint32_t)__half_as_ushort(l) << 16);
    }
}

// ------------------------------------------------------------ view build
// Tile shapes of the three views: mode 0 tiles W's rows (kTcN segments x
// kTcK reduction indices, offsets in the swizzled fp16 tile), mode 1 its
// columns the same way, mode 2 blocks of kTcM rows x kTcN columns, each
// cut into (32-row quarter, 32-column chunk) groups (key: block * kWGroups +
// group; offset: row * 32 + column within the group).
struct TileOf {
    int mode, n_inner;   // tiles along the second coordinate
    __device__ __forceinline__ uint32_t key(int32_t r, int32_t c) const {
        if (mode == 2)
            return ((uint32_t)(r / kTcM) * (uint32_t)n_inner + (uint32_t)(c / kTcN)) * kWGroups +
                   (uint32_t)((r % kTcM) / 32 * kWChunks + (c % kTcN) / 32);
        const int32_t sg = mode ? c : r, kk = mode ? r : c;
        return (uint32_t)(sg / kTcN) * (uint32_t)n_inner + (uint32_t)(kk / kTcK);
    }
    __device__ __forceinline__ uint16_t off(int32_t r, int32_t c) const {
        if (mode == 2) return (uint16_t)((r & 31) * 32 + (c % kTcN) % 32);
        const int32_t sg = mode ? c : r, kk = mode ? r : c;
        return (uint16_t)sw128(sg % kTcN, kk % kTcK);
    }
};

// Sort keys of the entries: their tile, and with by_bank also the
// shared-memory bank their 16-bit store hits (tile * 32 + bank).
__global__ void k_tc_keys(const int32_t* __restrict__ r, const int32_t* __restrict__ c, int64_t n,
                          TileOf tile, bool by_bank, uint32_t* __restrict__ keys, uint32_t* __restrict__ vals) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t t = tile.key(r[k], c[k]);
        keys[k] = by_bank ? t * 32u + ((tile.off(r[k], c[k]) >> 2) & 31u) : t;
        vals[k] = (uint32_t)k;
    }
}

// Entries sorted by (tile, bank): the first position of every (tile, bank) run.
__global__ void k_tc_run_start(const uint32_t* __restrict__ keys, int64_t n, int32_t* __restrict__ start) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x)
        if (j == 0 || keys[j] != keys[j - 1]) start[keys[j]] = (int32_t)j;
}

// (tile, bank) -> (tile, rank within the bank, bank): sorted by this key, each
// aligned group of 32 entries of a window (one warp's store instruction) takes
// one entry from each bank while the banks last, instead of up to 32 from one.
__global__ void k_tc_rank_key(uint32_t* __restrict__ keys, int64_t n, const int32_t* __restrict__ start) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t k1 = keys[j];
        const uint32_t rank = (uint32_t)(j - start[k1]);
        keys[j] = ((k1 >> 5) * kRankSpan + rank) * 32u + (k1 & 31u);
    }
}

// From the entries sorted by tile: their canonical slots, their byte offsets
// in the swizzled fp16 tile, and the first entry of every tile (empty tiles
// included).
__global__ void k_tc_finish(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals,
                            int64_t n, int64_t n_tiles, int shift, const int32_t* __restrict__ r,
                            const int32_t* __restrict__ c, TileOf tile, int32_t* __restrict__ perm_t,
                            uint16_t* __restrict__ off, int32_t* __restrict__ tile_ptr) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j <= n;
         j += (int64_t)gridDim.x * blockDim.x) {
        if (j < n) {
            const uint32_t k = vals[j];
            perm_t[j] = (int32_t)k;
            off[j] = tile.off(r[k], c[k]);
        }
        const int64_t lo = j == 0 ? 0 : (int64_t)(keys[j - 1] >> shift) + 1;
        const int64_t hi = j == n ? n_tiles : (int64_t)(keys[j] >> shift);
        for (int64_t tt = lo; tt <= hi; ++tt) tile_ptr[tt] = (int32_t)j;
    }
}

int grid_for(int64_t n, int threads, int num_sms) {
    return (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, threads), (int64_t)num_sms * 8));
}

int bits_of(uint64_t n_values) {
    int b = 0;
    while (b < 64 && (n_values - 1) >> b) ++b;
    return b;
}

template <typename T>
bool tc_alloc(T** p, int64_t count) {
    if (cudaMalloc((void**)p, (size_t)std::max<int64_t>(count, 1) * sizeof(T)) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return false;
    }
    return true;
}

void tc_shape(const Layer* L, bool columns, int64_t* n_seg, int64_t* k_len) {
    *n_seg = columns ? L->in_f : L->out_f;
    *k_len = columns ? L->out_f : L->in_f;
}

int build_view(Layer* L, int mode, cudaStream_t s) {
    TcView& V = L->tc->view[mode];
    const int64_t n = L->nnz;
    if (mode == 2) {
        V.n_win = (int)ceil_div(L->in_f, kTcN);    // column blocks
        V.n_nt = (int)ceil_div(L->out_f, kTcM);    // row blocks
    } else {
        int64_t n_seg, k_len;
        tc_shape(L, mode == 1, &n_seg, &k_len);
        V.n_win = (int)ceil_div(k_len, kTcK);
        V.n_nt = (int)ceil_div(n_seg, kTcN);
    }
    V.n_tiles = (int64_t)V.n_win * V.n_nt;
    // sort keys: tiles, or (block, group) pairs for the weight gradient
    const int64_t n_keys = mode == 2 ? V.n_tiles * kWGroups : V.n_tiles;
    if (!V.perm_t) {
        if (!tc_alloc(&V.perm_t, n) || !tc_alloc(&V.off, n + kTcPad) || !tc_alloc(&V.tile_ptr, n_keys + 1)) {
            // all or nothing: a later call starts over
            void* ptrs[] = {V.perm_t, V.off, V.tile_ptr};
            for (void* p : ptrs)
                if (p) cudaFree(p);
            V.perm_t = nullptr;
            V.off = nullptr;
            V.tile_ptr = nullptr;
            return SNK_ERR_OOM;
        }
    }
    const TileOf tile{mode, V.n_win};
    const int T = 256;
    const int G = grid_for(n, T, L->num_sms);
    const int tile_bits = bits_of((uint64_t)n_keys);
    // the sparse-tile views also spread each window's entries over the banks
    // when the (tile, rank, bank) key fits 32 bits
    const bool by_bank = mode != 2 && tile_bits + 14 <= 32;
    if (by_bank && !L->tc->run_start) {
        int64_t most = 0;
        for (int m = 0; m < 2; ++m) {
            int64_t n_seg, k_len;
            tc_shape(L, m == 1, &n_seg, &k_len);
            most = std::max(most, ceil_div(n_seg, kTcN) * ceil_div(k_len, kTcK) * 32);
        }
        if (!tc_alloc(&L->tc->run_start, most)) return SNK_ERR_OOM;
    }
    uint32_t* ck = L->col_keys;
    uint32_t* cv = L->col_vals;
    k_tc_keys<<<G, T, 0, s>>>(L->r, L->c, n, tile, by_bank, ck, cv);
    bool flipped = false;
    int st = sort_pairs_u32(ck, cv, ck + n, cv + n, n, tile_bits + (by_bank ? 5 : 0), L->tile_hist,
                            L->tile_hist_len, s, &flipped);
    if (st != SNK_OK) return st;
    uint32_t* kk = flipped ? ck + n : ck;
    uint32_t* vv = flipped ? cv + n : cv;
    int shift = 0;
    if (by_bank) {
        k_tc_run_start<<<G, T, 0, s>>>(kk, n, L->tc->run_start);
        k_tc_rank_key<<<G, T, 0, s>>>(kk, n, L->tc->run_start);
        uint32_t* k2 = flipped ? ck : ck + n;
        uint32_t* v2 = flipped ? cv : cv + n;
        st = sort_pairs_u32(kk, vv, k2, v2, n, tile_bits + 14, L->tile_hist, L->tile_hist_len, s, &flipped);
        if (st != SNK_OK) return st;
        if (flipped) {
            kk = k2;
            vv = v2;
        }
        shift = 14;
    }
    k_tc_finish<<<grid_for(n + 1, T, L->num_sms), T, 0, s>>>(kk, vv, n, n_keys, shift, L->r, L->c, tile,
                                                             V.perm_t, V.off, V.tile_ptr);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

// Which path: SNK_LARGE_BATCH=on|off forces it (tests); otherwise the
// measured crossover with 64-row batch tiling (10000^2 and 5000^2 layers,
// forward + dX + dW): from kTcTierBatch[t] rows at density
// 1 / kTcTierDiv[t] and above, for any tier t.
//   10% (10000^2 and 5000^2): tiled at 64, tensor from 96;  5%: tiled at 64,
//   tensor from 96 (3% ahead there);  3%: tiled at 128, tensor at 192;
//   2%: tiled at 192, tensor at 256;  1%: tiled to 384, tie at 512,
//   tensor at 640.
constexpr int kTcTiers = 4;
constexpr int64_t kTcTierBatch[kTcTiers] = {96, 192, 256, 512};
constexpr int64_t kTcTierDiv[kTcTiers] = {20, 34, 50, 100};

}  // namespace

bool tc_eligible(const Layer* L, int64_t b) {
    if (L->nnz == 0) return false;
    const int64_t n_tiles = ceil_div(L->out_f, kTcN) * ceil_div(L->in_f, kTcK) +
                            ceil_div(L->in_f, kTcN) * ceil_div(L->out_f, kTcK) +
                            ceil_div(L->out_f, kTcM) * ceil_div(L->in_f, kTcN);
    if (n_tiles > INT32_MAX / 2) return false;
    // the weight-gradient view's (block, group) keys
    if (ceil_div(L->out_f, kTcM) * ceil_div(L->in_f, kTcN) * kWGroups > INT32_MAX) return false;
    const char* f = getenv("SNK_LARGE_BATCH");
    if (f && strcmp(f, "off") == 0) return false;
    if (f && strcmp(f, "on") == 0) return true;
    for (int t = 0; t < kTcTiers; ++t)
        if (b >= kTcTierBatch[t] && L->nnz * kTcTierDiv[t] >= L->out_f * L->in_f) return true;
    return false;
}

void free_tc(Layer* L) {
    if (!L->tc) return;
    TcState* T = L->tc;
    void* ptrs[] = {T->view[0].perm_t, T->view[0].off, T->view[0].tile_ptr, T->view[1].perm_t,
                    T->view[1].off, T->view[1].tile_ptr, T->view[2].perm_t, T->view[2].off,
                    T->view[2].tile_ptr, T->hl, T->seg_exp, T->col_exp, T->run_start, T->row_exp, T->dh,
                    T->dl, T->seg_code, T->col_code, T->cand, T->frows, T->dw_flag, T->dw_list, T->fix, T->part};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    delete T;
    L->tc = nullptr;
}

// Rebuild the views that exist, from a new canonical triple; the caller
// marks them current once it has advanced the topology version.
int refresh_tc_views(Layer* L, cudaStream_t s) {
    if (!L->tc) return SNK_OK;
    for (int d = 0; d < 3; ++d)
        if (L->tc->view[d].perm_t) {
            int st = build_view(L, d, s);
            if (st != SNK_OK) return st;
        }
    return SNK_OK;
}

void mark_tc_views(Layer* L) {
    if (!L->tc) return;
    for (int d = 0; d < 3; ++d)
        if (L->tc->view[d].perm_t) L->tc->view[d].version = L->topology_version;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, resolved once through the runtime.
EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &f, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        cudaGetLastError();
    }
    return fn;
}

// fp16 [rows][len] at row stride ks, loaded in 64 x 128 boxes with the
// 128-byte swizzle; reads past len or rows come back as zeros.
bool encode_map(CUtensorMap* map, __half* base, int64_t len, int64_t rows, int64_t ks, int box_rows = kTcM) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)len, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ks * sizeof(__half)};
    cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How the output tiles map to CTAs (one CTA per SM).  When the tiles fill
// at most half a wave, every tile is shared by `split` CTAs over consecutive
// ranges of windows, as many as still fit one wave (at most kTcMaxSplit).
// When they fill more than one wave, the tiles of the last, partial wave are
// shared the same way, as many as fit beside each other, so that wave ends
// sooner; the others are computed whole.  Anything else runs one CTA per
// tile: a split that needs a second wave of its own was measured slower
// (10000^2, 90%, batch 256: 297 against 257 us).
constexpr int kTcMaxSplit = 8;
struct TcGrid {
    int full, split;
};
TcGrid tc_grid(int tiles, int n_win, int num_sms) {
    auto ways = [&](int n) {
        const int sp = std::min(std::min(kTcMaxSplit, n_win), num_sms / std::max(n, 1));
        return sp >= 2 ? sp : 1;
    };
    if (2 * tiles <= num_sms) {
        const int sp = ways(tiles);
        return sp > 1 ? TcGrid{0, sp} : TcGrid{tiles, 1};
    }
    const int rem = tiles % num_sms;
    if (tiles > num_sms && rem > 0) {
        const int sp = ways(rem);
        if (sp > 1) return TcGrid{tiles - rem, sp};
    }
    return TcGrid{tiles, 1};
}

// The large-batch workspace, allocated on first use.
int ensure_tc(Layer* L) {
    if (L->tc) return SNK_OK;
    TcState* T = new TcState();
    L->tc = T;
    T->k_stride = ceil_div(std::max(L->out_f, L->in_f), 8) * 8;
    if (!tc_alloc(&T->hl, L->nnz + kTcPad) || !tc_alloc(&T->seg_exp, std::max(L->out_f, L->in_f)) ||
        !tc_alloc(&T->col_exp, L->in_f) || !tc_alloc(&T->row_exp, kTcChunk) ||
        !tc_alloc(&T->dh, kTcChunk * T->k_stride) || !tc_alloc(&T->dl, kTcChunk * T->k_stride) ||
        !tc_alloc(&T->seg_code, std::max(L->out_f, L->in_f)) || !tc_alloc(&T->col_code, L->in_f) ||
        !tc_alloc(&T->cand, std::max(L->out_f, L->in_f)) || !tc_alloc(&T->frows, kTcChunk) ||
        !tc_alloc(&T->dw_flag, L->out_f + L->in_f) || !tc_alloc(&T->dw_list, L->out_f + L->in_f) ||
        !tc_alloc(&T->fix, kFixWords)) {
        free_tc(L);
        return SNK_ERR_OOM;
    }
    // slices' partial sums: at most one wave of shared-tile slices
    T->part_len = (int64_t)L->num_sms * kTcM * kTcN;
    if (!tc_alloc(&T->part, T->part_len)) {
        free_tc(L);
        return SNK_ERR_OOM;
    }
    return SNK_OK;
}

}  // namespace

int run_tc(Layer* L, bool columns, const float* D, int64_t b, const float* bias, float* Y,
           cudaStream_t s) {
    int st0 = ensure_tc(L);
    if (st0 != SNK_OK) return st0;
    TcState* T = L->tc;
    TcView& V = T->view[columns ? 1 : 0];
    if (V.version != L->topology_version) {
        int st = build_view(L, columns ? 1 : 0, s);
        if (st != SNK_OK) return st;
        V.version = L->topology_version;
    }
    int64_t n_seg, k_len;
    tc_shape(L, columns, &n_seg, &k_len);
    const int TH = 256;
    if (cudaMemsetAsync(T->fix, 0, kFixWords * sizeof(uint32_t), s) != cudaSuccess) return SNK_ERR_CUDA;
    k_tc_seg_exp<<<grid_for(n_seg * 32, TH, L->num_sms), TH, 0, s>>>(
        columns ? L->col_ptr : L->row_ptr, L->v, columns ? L->perm : nullptr, n_seg, T->seg_exp, T->seg_code,
        T->fix);
    k_tc_values<<<grid_for(L->nnz, TH, L->num_sms), TH, 0, s>>>(L->v, V.perm_t, columns ? L->c : L->r,
                                                                T->seg_exp, L->nnz, T->hl, T->seg_code);
    k_tc_seg_cand<<<grid_for(n_seg, TH, L->num_sms), TH, 0, s>>>(T->seg_code, n_seg, T->cand, T->fix);
    if (cudaFuncSetAttribute(k_tc_spmm, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess)
        return SNK_ERR_CUDA;
    const bool vec = (k_len % 4) == 0 && ((uintptr_t)D & 15) == 0;
    // the entries of the segments, for the exact recomputation of flagged outputs
    TcSide side{columns ? L->col_ptr : L->row_ptr, columns ? L->rows_c : L->c, columns ? L->perm : nullptr,
                L->v};
    for (int64_t c0 = 0; c0 < b; c0 += kTcChunk) {
        const int bc = (int)std::min<int64_t>(kTcChunk, b - c0);
        const float* Dc = D + c0 * k_len;
        if (c0 > 0 && cudaMemsetAsync(T->fix + kFixRows, 0, sizeof(uint32_t), s) != cudaSuccess)
            return SNK_ERR_CUDA;
        if (vec)
            k_tc_split<true><<<bc, TH, 0, s>>>(Dc, k_len, T->k_stride, T->row_exp, T->dh, T->dl, T->frows,
                                               T->fix);
        else
            k_tc_split<false><<<bc, TH, 0, s>>>(Dc, k_len, T->k_stride, T->row_exp, T->dh, T->dl, T->frows,
                                                T->fix);
        CUtensorMap mh, ml;
        if (!encode_map(&mh, T->dh, k_len, bc, T->k_stride) || !encode_map(&ml, T->dl, k_len, bc, T->k_stride))
            return SNK_ERR_CUDA;
        TcArgs a;
        a.b = bc;
        a.K_len = k_len;
        a.row_exp = T->row_exp;
        a.off = V.off;
        a.hl = T->hl;
        // dense windows are cleared whole, sparse ones entry by entry
        a.zero_fill = L->nnz >= kZeroFillEntries * V.n_tiles;
        a.tile_ptr = V.tile_ptr;
        a.seg_exp = T->seg_exp;
        a.n_seg = n_seg;
        a.n_win = V.n_win;
        a.n_nt = V.n_nt;
        a.n_mt = (int)ceil_div(bc, kTcM);
        a.bias = bias;
        a.Y = Y + c0 * n_seg;
        a.status = L->status;
        const int tiles = a.n_mt * a.n_nt;
        const TcGrid g = tc_grid(tiles, a.n_win, L->num_sms);
        a.full = g.full;
        a.split = g.split;
        a.part = T->part;
        const int shared = tiles - g.full;   // tiles whose slices leave partial sums
        if ((int64_t)shared * g.split * kTcM * kTcN > T->part_len) {
            a.full = tiles;
            a.split = 1;
        }
        k_tc_spmm<<<a.full + (tiles - a.full) * a.split, kTcThreads, kTcSmem, s>>>(mh, ml, a);
        if (a.full < tiles)
            k_tc_split_sum<<<dim3((unsigned)(tiles - a.full), kTcM * kTcN / 256), 256, 0, s>>>(
                T->part, a.full, a.split, a.n_mt, a.n_nt, bc, n_seg, bias, Y + c0 * n_seg);
        // dense rows of this chunk that the split cannot carry: every output
        // of theirs again, per stored entry
        int st = launch_exact_rows(side, n_seg, Dc, k_len, bias, Y + c0 * n_seg, T->frows,
                                   T->fix + kFixRows, L->num_sms, s);
        if (st != SNK_OK) return st;
    }
    // segments of W that the split cannot carry, for every dense row
    return launch_exact_segs(side, n_seg, D, k_len, b, bias, Y, T->cand, T->fix + kFixCand, T->seg_exp,
                             T->seg_code, T->fix + kFixRowL1, L->num_sms, s);
}

int run_tc_sddmm(Layer* L, const float* X, const float* dY, int64_t b, float* dW, float* db,
                 cudaStream_t s) {
    int st = ensure_tc(L);
    if (st != SNK_OK) return st;
    TcState* T = L->tc;
    TcView& V = T->view[2];
    if (V.version != L->topology_version) {
        st = build_view(L, 2, s);
        if (st != SNK_OK) return st;
        V.version = L->topology_version;
    }
    if (cudaFuncSetAttribute(k_tc_sddmm, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem) != cudaSuccess)
        return SNK_ERR_CUDA;
    const int64_t out_f = L->out_f, in_f = L->in_f;
    if (cudaMemsetAsync(T->fix, 0, kFixWords * sizeof(uint32_t), s) != cudaSuccess ||
        cudaMemsetAsync(T->dw_flag, 0, (out_f + in_f) * sizeof(int32_t), s) != cudaSuccess)
        return SNK_ERR_CUDA;
    // batch rows per chunk: the transposed pieces of dY and X share the workspace
    const int64_t cap = (kTcChunk * T->k_stride) / (out_f + in_f);
    const int64_t chunk = std::max<int64_t>(kTcK, cap / kTcK * kTcK);
    for (int64_t c0 = 0; c0 < b; c0 += chunk) {
        const int64_t bc = std::min<int64_t>(chunk, b - c0);
        const int64_t bs = ceil_div(bc, 8) * 8;
        const float* dYc = dY + c0 * out_f;
        const float* Xc = X + c0 * in_f;
        const int acc = c0 > 0;
        if (c0 > 0 && cudaMemsetAsync(T->fix + kFixDyL1, 0, 4 * sizeof(uint32_t), s) != cudaSuccess)
            return SNK_ERR_CUDA;
        if (db)
            k_tc_colstats<true><<<(unsigned)ceil_div(out_f, 32), 256, 0, s>>>(
                dYc, bc, out_f, T->seg_exp, T->seg_code, T->fix + kFixDyL1, db, acc);
        else
            k_tc_colstats<false><<<(unsigned)ceil_div(out_f, 32), 256, 0, s>>>(
                dYc, bc, out_f, T->seg_exp, T->seg_code, T->fix + kFixDyL1, nullptr, 0);
        k_tc_colstats<false><<<(unsigned)ceil_div(in_f, 32), 256, 0, s>>>(Xc, bc, in_f, T->col_exp, T->col_code,
                                                                          T->fix + kFixXL1, nullptr, 0);
        __half* ah = T->dh;
        __half* al = T->dl;
        __half* bh = T->dh + out_f * bs;
        __half* bl = T->dl + out_f * bs;
        const dim3 tb(32, 8);
        k_tc_tsplit<<<dim3((unsigned)ceil_div(out_f, 32), (unsigned)ceil_div(bc, 32)), tb, 0, s>>>(
            dYc, bc, out_f, T->seg_exp, bs, ah, al, T->seg_code);
        k_tc_tsplit<<<dim3((unsigned)ceil_div(in_f, 32), (unsigned)ceil_div(bc, 32)), tb, 0, s>>>(
            Xc, bc, in_f, T->col_exp, bs, bh, bl, T->col_code);
        k_tc_dw_decide<<<grid_for(out_f + in_f, 256, L->num_sms), 256, 0, s>>>(
            T->seg_exp, T->seg_code, T->col_exp, T->col_code, out_f, in_f, (float)ceil_div(b, chunk),
            T->dw_flag, T->dw_list, T->fix);
        CUtensorMap mah, mal, mbh, mbl;
        if (!encode_map(&mah, ah, bc, out_f, bs, kTcM) || !encode_map(&mal, al, bc, out_f, bs, kTcM) ||
            !encode_map(&mbh, bh, bc, in_f, bs, kTcN) || !encode_map(&mbl, bl, bc, in_f, bs, kTcN))
            return SNK_ERR_CUDA;
        TcwArgs a;
        a.n_win = (int)ceil_div(bc, kTcK);
        a.n_ot = V.n_nt;
        a.n_it = V.n_win;
        a.out_f = out_f;
        a.in_f = in_f;
        a.e_row = T->seg_exp;
        a.e_col = T->col_exp;
        a.perm = V.perm_t;
        a.off = V.off;
        a.group_ptr = V.tile_ptr;
        a.dW = dW;
        a.accumulate = acc;
        a.status = L->status;
        // persistent: one CTA per SM, each taking every grid-th block
        const int grid = (int)std::min<int64_t>((int64_t)a.n_ot * a.n_it, L->num_sms);
        k_tc_sddmm<<<grid, kWThreads, kWSmem, s>>>(mah, mal, mbh, mbl, a);
    }
    if (cudaGetLastError() != cudaSuccess) return SNK_ERR_CUDA;
    // rows and columns of W flagged by any chunk: their entries again, over the whole batch
    return launch_exact_dw(L, X, dY, b, dW, T->dw_list, T->fix + kFixDwList, s);
}

}  // namespace snk
