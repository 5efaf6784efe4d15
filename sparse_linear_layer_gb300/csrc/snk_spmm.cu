// Forward SpMM  Y = X W^T + bias   and transposed SpMM  dX = dY W.
//
//   "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
//     GPU", Fig. 1 (the forward pass computed on the COO triple; only live
//     connections cost memory and FLOPs).
//   "Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
//     sec. 6.1 (for each live entry scale the matching input row and add it
//     to the output row), sec. 7.1 (dL/dX is another SpMM through W^T),
//     sec. 7.2 (W^T read through a permutation map built once per topology;
//     per call only the values are gathered).
//
// One kernel serves both products.  The stored entries of one matrix side
// are walked in segment order: rows of W (canonical order, forward) or
// columns of W (the column-sorted view, transposed product, with the value
// fetched through perm).  Each output segment o receives
//     Y[beta, o] = bias[o] + sum_{k in seg(o)} w_k * X[beta, idx_k].
//
// GB300 design
//  * Load balance: one block per SM owns an equal share of the entries,
//    with its boundaries moved to the nearest segment boundary (unless that
//    segment is longer than half a share), and its warps split the share
//    into equal chunks (merge path), so skewed segments cost nothing.
//    Segments cut between warps are added in shared memory after one block
//    barrier, in warp order.  Only a segment cut between blocks (a very long
//    one) goes through global memory: each block stores its partial, the
//    last block to arrive (an arrival counter per segment) adds them in
//    block order and resets the counter.  No result depends on timing.
//  * The dense operand is staged once per block in shared memory transposed,
//    [idx][BP], so one 128-bit shared load serves 4 batch columns of one
//    entry; when it does not fit, a transposed copy in global memory is read
//    through the read-only path instead.
//  * Values and indices stream with 128-bit evict-first loads.
//  * A warp splits into GPW groups of LPE lanes; a group owns one entry at a
//    time and its lanes split the BP batch columns.  Each lane accumulates
//    its own partial sums (at least 32 per output for BP <= 4), reduced at the
//    segment end with __shfl_xor_sync.
#include "snk_device.cuh"

namespace snk {

struct SpmmArgs {
    const float* val;        // stored values, canonical order
    const int32_t* perm;     // column-order -> canonical slot (transposed product) or null
    const int32_t* idx;      // operand index per stored entry (col, or row in column order)
    const uint16_t* idx16;   // the same as 16-bit, zero padded (shared-memory path)
    const int32_t* seg_ptr;  // [n_seg+1]
    const int4* cdesc;       // [n_blocks * kWarpsPerBlock] (k0, k1, first seg, end seg)
    const BlockDesc* bdesc;  // [n_blocks]
    const int32_t* bnd;      // [n_blocks+1] first entry of each block
    int64_t nnz;
    int64_t n_seg;           // output length per batch row
    int64_t n_src;           // operand length per batch row
    int b;                   // batch columns of this tile (<= BP)
    int n_blocks;
    const float* X;          // [b, n_src] row-major
    const float* xt;         // [n_src][BP] transposed copy (global-memory path)
    const float* bias;       // [n_seg] or null
    float* Y;                // [b, n_seg] row-major
    float* part;             // [n_blocks][2][BP] cross-block partial sums
    int32_t* cnt;            // [n_seg] arrival counters
    // column sweep of the transposed product (k_sweep only)
    const int4* sw_blk;      // per block: two records
    const int2* sw_col;      // per block and column: (first virtual lane, lanes)
    const int4* sw_lane;     // per virtual lane: (first quad, quad stride, first entry, end entry)
    float* sw_gpart;         // partials of virtual lanes beyond the block's threads
    const int* sw_split;     // [boundary][lane] resume quad of each lane at each table boundary
    int64_t sw_nlane;        // lanes per boundary in sw_split
    int sw_rows;             // operand rows staged per phase (a multiple of 4)
    int sw_phases;           // phases of this launch
    int sw_stride;           // table boundaries per phase of this launch
};

// A segment cut by a chunk boundary, whose partial sum this warp stored in
// its shared-memory slot (0: the segment entered the chunk from before,
// 1: it starts in the chunk and leaves it).
struct Pending {
    int r;
    uint32_t rs, re;
};

// Shared memory: [transposed operand (shared-memory path)][partials
// [warps][2][BP]][segment ids [warps][2]].
template <bool GATHER>
struct SpmmShape {
    static constexpr int kNT = GATHER ? kThreadsDx : kThreads;
    static constexpr int kW = kNT / kWarp;
};
template <int BP, bool GATHER>
__host__ __device__ constexpr size_t spmm_slot_bytes() {
    return (size_t)SpmmShape<GATHER>::kW * 2 * BP * sizeof(float) +
           (size_t)SpmmShape<GATHER>::kW * 2 * sizeof(int);
}
__host__ __device__ inline size_t operand_floats(int64_t n_src, int bp) {
    return ((size_t)n_src * bp + 3) & ~(size_t)3;
}

// Finish one output segment: reduce the per-lane partial sums across the
// warp's groups; write the result, or, for a segment cut by a chunk boundary,
// store this warp's partial in its shared slot.
template <int BP>
__device__ __forceinline__ void finish_segment(const SpmmArgs& a, float (&acc)[Tile<BP>::VEC],
                                               int r, uint32_t rs, uint32_t re, uint32_t k0,
                                               uint32_t k1, float bo, int lane, int sub,
                                               float* my_slots, Pending (&pend)[2]) {
    using TL = Tile<BP>;
    constexpr int VEC = TL::VEC, LPE = TL::LPE;
#pragma unroll
    for (int o = LPE; o < kWarp; o <<= 1) {
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
    }
    if (rs >= k0 && re <= k1) {
        if (lane < LPE) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const int beta = TL::beta(sub, j);
                if (beta < a.b) a.Y[(int64_t)beta * a.n_seg + r] = acc[j] + bo;
            }
        }
    } else {
        const int slot = (rs < k0) ? 0 : 1;
        if (lane < LPE) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) my_slots[slot * BP + sub * VEC + j] = acc[j];
        }
        pend[slot] = Pending{r, rs, re};
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
}

// A segment cut between blocks: store this block's partial, count the
// arrival, and let the last arriving block add the partials of the non-empty
// blocks first..last in block order (the first block's is in its slot 1).
template <int BP>
__device__ __noinline__ void cross_block(const SpmmArgs& a, int r, int slot,
                                         const float (&sum)[Tile<BP>::VEC], int first, int last,
                                         int n_contrib, int lane, int sub) {
    using TL = Tile<BP>;
    constexpr int VEC = TL::VEC, LPE = TL::LPE;
    if (lane < LPE) {
        float* my = a.part + ((int64_t)blockIdx.x * 2 + slot) * BP + sub * VEC;
#pragma unroll
        for (int j = 0; j < VEC; ++j) my[j] = sum[j];
    }
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomicAdd(a.cnt + r, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != n_contrib - 1) return;
    __threadfence();
    if (lane < LPE) {
        float tot[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) tot[j] = 0.f;
        for (int c = first; c <= last; ++c) {
            if (__ldg(a.bnd + c + 1) == __ldg(a.bnd + c)) continue;
            const float* pp = a.part + ((int64_t)c * 2 + (c == first ? 1 : 0)) * BP + sub * VEC;
#pragma unroll
            for (int j = 0; j < VEC; ++j) tot[j] += __ldcg(pp + j);
        }
        const float bo = a.bias ? __ldg(a.bias + r) : 0.f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const int beta = TL::beta(sub, j);
            if (beta < a.b) a.Y[(int64_t)beta * a.n_seg + r] = tot[j] + bo;
        }
    }
    if (lane == 0) a.cnt[r] = 0;
}

// After the block barrier: the warp where a cut segment starts adds the
// partials of the following warps that continue it (warp order) and writes
// the result, unless the segment leaves the block; warp 0 does the same for
// the segment that entered the block from before.  Segments that cross a
// block boundary continue in cross_block.
template <int BP, int W>
__device__ __forceinline__ void block_combine(const SpmmArgs& a, const float* sp, const int* srow,
                                              const Pending (&pend)[2], int warp, int lane,
                                              int sub) {
    using TL = Tile<BP>;
    constexpr int VEC = TL::VEC, LPE = TL::LPE;
    if (pend[1].r < 0 && !(warp == 0 && pend[0].r >= 0)) return;
    const BlockDesc bd = a.bdesc[blockIdx.x];
#pragma unroll
    for (int which = 1; which >= 0; --which) {
        const int slot = which;
        if (slot == 0 && warp != 0) continue;
        const int r = pend[slot].r;
        if (r < 0) continue;
        float sum[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            sum[j] = lane < LPE ? sp[(warp * 2 + slot) * BP + sub * VEC + j] : 0.f;
        for (int w2 = warp + 1; w2 < W && srow[w2 * 2] == r; ++w2) {
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (lane < LPE) sum[j] += sp[(w2 * 2) * BP + sub * VEC + j];
        }
        const bool ends_here = pend[slot].re <= (uint32_t)bd.k1;
        if (slot == 1) {
            if (ends_here) {
                if (lane < LPE) {
                    const float bo = a.bias ? __ldg(a.bias + r) : 0.f;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const int beta = TL::beta(sub, j);
                        if (beta < a.b) a.Y[(int64_t)beta * a.n_seg + r] = sum[j] + bo;
                    }
                }
            } else {
                cross_block<BP>(a, r, 1, sum, blockIdx.x, bd.tail_last, bd.n_tail, lane, sub);
            }
        } else {
            if (ends_here)
                cross_block<BP>(a, r, 0, sum, bd.head_first, blockIdx.x, bd.n_head, lane, sub);
            else
                cross_block<BP>(a, r, 0, sum, bd.head_first, bd.tail_last,
                                bd.n_head + bd.n_tail - 1, lane, sub);
        }
    }
}

// One warp per chunk.  The chunk's entries [k0, k1) are streamed as a flat
// sequence of blocks of 4*GPW entries from the multiple of 4 at or below k0
// (each group of LPE lanes owns 4 consecutive entries of a block).  Blocks
// sit in D+1 register slots: while block j is consumed, blocks j+1 .. j+D
// are in flight (and, for the transposed product, the values of blocks
// j+1 .. j+G are being gathered).  The loop over slots is unrolled so every slot index
// is a compile-time constant.  A block inside one segment is consumed
// without masks; a block that straddles segment or chunk boundaries is
// consumed once per segment it touches, with masks.
template <int BP, bool GATHER, bool SMEM, bool I16 = SMEM && SNK_IDX16>
__global__ void __launch_bounds__(SpmmShape<GATHER>::kNT, 1) k_spmm(const SpmmArgs a) {
    constexpr int NT = SpmmShape<GATHER>::kNT;
    constexpr int W = SpmmShape<GATHER>::kW;
    using TL = Tile<BP>;
    constexpr int VEC = TL::VEC, LPE = TL::LPE, GPW = TL::GPW;
    constexpr uint32_t BLK = 4 * GPW;
    constexpr int D = GATHER ? (BP == 16 ? SNK_PIPE_DX16 : SNK_PIPE_DX) : (BP == 1 ? SNK_PIPE_FWD_NARROW : SNK_PIPE_FWD);
    constexpr int NS = D + 1;
    // blocks whose values are gathered ahead of the consumed one (the
    // permutation of a block arrives NS - G blocks before its gather)
    constexpr int G = GATHER ? (SNK_GATHER_LEAD < D ? SNK_GATHER_LEAD : D) : 0;
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);
    float* sp = xs + (SMEM ? operand_floats(a.n_src, BP) : 0);
    int* srow = reinterpret_cast<int*>(sp + W * 2 * BP);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int grp = lane / LPE;
    const int sub = lane % LPE;
    const uint32_t nnz = (uint32_t)a.nnz;
    const int4 cd = a.cdesc[blockIdx.x * W + warp];
    const uint32_t k0 = (uint32_t)cd.x, k1 = (uint32_t)cd.y;
    const uint32_t base_first = k0 & ~3u;
    float* my_slots = sp + warp * 2 * BP;

    IdxBlk<I16> ib[NS];
    float wb[NS][4];
    int pb[NS][4];
    auto issue = [&](int s, uint32_t blk0) {
        const uint32_t base = blk0 + 4 * grp;
        if constexpr (I16) ib[s].load(a.idx16, base);
        else ib[s].load(a.idx, base, nnz);
        if constexpr (GATHER) padded4(a.perm, base, pb[s]);
        else stream4(a.val, base, nnz, wb[s]);
    };
    // The value gather hits L1 when another entry of the same row (in the
    // block's column range) brought its sector in, so it goes through L1;
    // except with a 4-column operand in shared memory (160 KB at out =
    // 10000), where the L1 left is small and caching the gathered sectors
    // only in L2 is faster (measured: 56 against 60 us at 10000^2, 90%).
    constexpr bool kGatherL2Only = SMEM && BP == 4;
    auto gather = [&](int s, uint32_t blk0) {
        const uint32_t base = blk0 + 4 * grp;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            wb[s][j] = (base + j < k1) ? (kGatherL2Only ? __ldcg(a.val + pb[s][j]) : __ldg(a.val + pb[s][j])) : 0.f;
    };

    // Everything that only depends on the chunk is requested before the
    // operand staging: the first blocks of the stream and the first window of
    // segment starts (and biases).
    if (k0 < k1) {
#pragma unroll
        for (int s = 0; s < NS; ++s)
            if (base_first + s * BLK < k1) issue(s, base_first + s * BLK);
    }
    SegWindow win{cd.z, cd.w - cd.z, 0, 0u, 0.f};
    if (win.nrows > 0) win.load(0, lane, a.seg_ptr, a.bias);
    if constexpr (SMEM) stage_transposed<BP>(xs, a.X, a.n_src, a.b, a.n_src, threadIdx.x, NT);
    __syncthreads();
    const float* xsrc = SMEM ? xs : a.xt;

    Pending pend[2] = {Pending{-1, 0u, 0u}, Pending{-1, 0u, 0u}};
    if (win.nrows > 0) {
        if constexpr (GATHER) {
#pragma unroll
            for (int s = 0; s < G; ++s)
                if (k0 < k1 && base_first + s * BLK < k1) gather(s, base_first + s * BLK);
        }
        const int r_begin = win.r_begin;
        int i = 0;
        uint32_t rs = win.bnd(0, lane, a.seg_ptr, a.bias), re = win.bnd(1, lane, a.seg_ptr, a.bias);
        float acc[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[j] = 0.f;

        auto consume = [&](int s, uint32_t blk0) {
            const uint32_t base = blk0 + 4 * grp;
            if (rs <= blk0 && k0 <= blk0 && blk0 + BLK < re && blk0 + BLK <= k1) {
                // interior block: every entry belongs to the current segment,
                // which continues past the block
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x[VEC];
                    const float* px = xsrc + ib[s].get(j) * BP;
                    if constexpr (SMEM) TL::load(px, sub, x);
                    else TL::ldg(px, sub, x);
#pragma unroll
                    for (int t = 0; t < VEC; ++t) acc[t] = fmaf(wb[s][j], x[t], acc[t]);
                }
                return;
            }
            const uint32_t blk_end = min(blk0 + BLK, k1);
            while (true) {
                const uint32_t lo_k = max(max(rs, k0), blk0), hi_k = min(re, blk_end);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t k = base + j;
                    if (k >= lo_k && k < hi_k) {
                        float x[VEC];
                        const float* px = xsrc + ib[s].get(j) * BP;
                        if constexpr (SMEM) TL::load(px, sub, x);
                        else TL::ldg(px, sub, x);
#pragma unroll
                        for (int t = 0; t < VEC; ++t) acc[t] = fmaf(wb[s][j], x[t], acc[t]);
                    }
                }
                if (min(re, k1) > blk_end) break;  // segment continues in the next block
                finish_segment<BP>(a, acc, r_begin + i, rs, re, k0, k1, win.bias_of(i), lane, sub,
                                   my_slots, pend);
                if (++i >= win.nrows) break;
                rs = re;
                re = win.bnd(i + 1, lane, a.seg_ptr, a.bias);
                if (rs >= blk_end) break;
            }
        };

        if (k0 < k1) {
            for (uint32_t base0 = base_first; base0 < k1; base0 += NS * BLK) {
#pragma unroll
                for (int s = 0; s < NS; ++s) {
                    const uint32_t blk0 = base0 + s * BLK;
                    if (blk0 < k1) {
                        if constexpr (GATHER) {
                            if (blk0 + G * BLK < k1) gather((s + G) % NS, blk0 + G * BLK);
                        }
                        consume(s, blk0);
                        if (blk0 + NS * BLK < k1) issue(s, blk0 + NS * BLK);
                    }
                }
            }
        }
        // segments that start at the end of the chunk (empty here)
        while (i < win.nrows) {
            finish_segment<BP>(a, acc, r_begin + i, rs, re, k0, k1, win.bias_of(i), lane, sub,
                               my_slots, pend);
            if (++i >= win.nrows) break;
            rs = re;
            re = win.bnd(i + 1, lane, a.seg_ptr, a.bias);
        }
    }
    if (lane == 0) {
        srow[warp * 2 + 0] = pend[0].r;
        srow[warp * 2 + 1] = pend[1].r;
    }
    __syncthreads();
    block_combine<BP, W>(a, sp, srow, pend, warp, lane, sub);
}

// ---------------------------------------------------------------------------
// Column sweep of the transposed product (batch tile BP <= 4, operand in
// shared memory).  (An 8-column version measured no faster than the chunk
// walk at 10000^2, 90%, and slower at 95% and 99%: two 128-bit operand loads
// per entry and twice the row phases.)  Every column of the block has its
// own lanes (snk_sweep.cu builds the tables, and orders the entries within
// quads so that the rows 8 lanes load together spread over the banks); lane j
// of a column with n lanes takes the column's
// aligned quads j, j + n, j + 2n, ... and masks the entries outside the
// column's range in this block.  Rows rise along a column, so all lanes move
// down the rows together, and the values they gather for nearby rows share
// sectors in L1.
//
// Row phases: the operand is staged a band of rows at a time, so that L1
// keeps room for the gathered values (at batch 4 the whole operand would take
// 160 KB of an SM's 256 KB at out = 10000).  The tables cut the rows into P
// equal phases (P a power of two, about SNK_SWEEP_PHASE_KB of shared memory
// each at a 4-column tile) and hold, for every lane and cut, the quad where
// the lane crosses it; a 1-column tile merges phases in pairs.  A phase
// takes the entries whose rows it holds, up to that quad (inclusive when the
// quad straddles the cut), and the next phase resumes there, so a lane's
// loop bound is known before it starts.
//
// A lane keeps two accumulators (even and odd positions of the quad) and
// folds them into its partial sums every 8 quads and at the end of each
// phase, so no running sum takes more than 16 terms.  The column's result
// adds its lanes' partials in lane order, 32 at a time; the column cut by the
// block's first (or last) boundary goes through the same cross-block
// protocol as the chunk walk, so results are deterministic and launches of
// either kernel mix.

// Index loads of the sweep bypass L1 allocation, leaving L1 to the values.
__device__ __forceinline__ int4 sw_ld4(const int4* p) {
    int4 r;
    asm volatile("ld.global.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 sw_ld2(const uint2* p) {
    uint2 r;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// The walk of one virtual lane, resumable across row phases: between phases
// it keeps only its next quad and its partial sums.  (Priming a phase before
// its operand rows are staged, to overlap the first loads with the staging,
// measured no faster: the pipeline registers then live across the staging.)
template <int BP>
struct SweepLane {
    static constexpr int NS = SNK_SWEEP_NS;   // quads in flight
    uint32_t u;          // next quad
    uint32_t st, s, e;   // quad stride; the column's entry range in the block
    uint32_t qe;         // quad bound of the current phase
    float outer[BP];     // partial sums
    int pp[NS][4];       // canonical slots of quads in flight
    uint32_t rr[NS][2];  // their rows, two 16-bit rows per word
    float ww[NS][4];     // their gathered values

    __device__ __forceinline__ void init(const int4 ln) {
        u = (uint32_t)ln.x;
        st = (uint32_t)ln.y;
        s = (uint32_t)ln.z;
        e = (uint32_t)ln.w;
#pragma unroll
        for (int t = 0; t < BP; ++t) outer[t] = 0.f;
    }
    __device__ __forceinline__ int row_of(int sl, int j) const {
        const uint32_t w2 = rr[sl][j >> 1];
        return (int)((j & 1) ? (w2 >> 16) : (w2 & 0xffffu));
    }
    __device__ __forceinline__ void issue(const SpmmArgs& a, int sl, uint32_t q) {
        const int4 p4 = sw_ld4(reinterpret_cast<const int4*>(a.perm) + q);
        const uint2 r4 = sw_ld2(reinterpret_cast<const uint2*>(a.idx16) + q);
        pp[sl][0] = p4.x;
        pp[sl][1] = p4.y;
        pp[sl][2] = p4.z;
        pp[sl][3] = p4.w;
        rr[sl][0] = r4.x;
        rr[sl][1] = r4.y;
    }
    __device__ __forceinline__ void gather(const SpmmArgs& a, int sl, uint32_t q) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t k = 4 * q + j;
            ww[sl][j] = (k >= s && k < e) ? __ldg(a.val + pp[sl][j]) : 0.f;
        }
    }

    // Start the phase that ends before quad qend: index loads of its first
    // NS - 1 quads, the values of the first.
    __device__ __forceinline__ void prime(const SpmmArgs& a, uint32_t qend) {
        qe = min((e + 3) >> 2, qend);
        if (u >= qe) return;
#pragma unroll
        for (int k = 0; k < NS - 1; ++k)
            if (u + k * st < qe) issue(a, k, u + k * st);
        gather(a, 0, u);
    }

    // The primed phase: quads from u up to qe, entries with rows in
    // [r0, r1) (xs holds those operand rows, or with GX the operand is read
    // from X).  Quads stream NS - 1 ahead; their values are gathered one
    // ahead.  Two accumulators (even and odd positions of the quad) fold into
    // the partial sums every 8 quads and at the end of the phase, so no
    // running sum takes more than 16 terms.
    template <bool GX = false>
    __device__ __forceinline__ void run(const SpmmArgs& a, const float* xs, int r0, int r1) {
        float acc[2][BP];
#pragma unroll
        for (int t = 0; t < BP; ++t) acc[0][t] = acc[1][t] = 0.f;
        int since_fold = 0;
        auto fold = [&]() {
#pragma unroll
            for (int t = 0; t < BP; ++t) {
                outer[t] += acc[0][t] + acc[1][t];
                acc[0][t] = acc[1][t] = 0.f;
            }
        };
        // the quad's entries with rows in [r0, r1)
        auto consume = [&](int sl, uint32_t q) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t k = 4 * q + j;
                const int r = row_of(sl, j);
                if (k >= s && k < e) {
                    if (r >= r0 && r < r1) {
                        float x[BP];
                        if constexpr (GX) {
#pragma unroll
                            for (int t = 0; t < BP; ++t) x[t] = t < a.b ? __ldg(a.X + (int64_t)t * a.n_src + r) : 0.f;
                        } else {
                            VecF<BP>::load(xs + (r - r0) * BP, x);
                        }
#pragma unroll
                        for (int t = 0; t < BP; ++t) acc[j & 1][t] = fmaf(ww[sl][j], x[t], acc[j & 1][t]);
                    }
                }
            }
            if (++since_fold == 8) {
                since_fold = 0;
                fold();
            }
        };
        if (u >= qe) {
            u = qe;
            return;
        }
        for (uint32_t qb = u; qb < qe; qb += NS * st) {
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                const uint32_t q = qb + i * st;
                if (q < qe) {
                    if (q + (NS - 1) * st < qe) issue(a, (i + NS - 1) % NS, q + (NS - 1) * st);
                    if (q + st < qe) gather(a, (i + 1) % NS, q + st);
                    consume(i, q);
                }
            }
        }
        u = qe;
        fold();
    }
};

// Sum of the partials of virtual lanes v0 .. v0 + n - 1 (in shared memory
// below the thread count, else in global scratch), 32 at a time.
template <int BP>
__device__ __forceinline__ void sweep_sum(const float* red, const float* gred, int v0, int n, float (&sum)[BP]) {
#pragma unroll
    for (int t = 0; t < BP; ++t) sum[t] = 0.f;
    for (int k0 = 0; k0 < n; k0 += 32) {
        float u[BP];
#pragma unroll
        for (int t = 0; t < BP; ++t) u[t] = 0.f;
        const int k1 = min(n, k0 + 32);
        for (int k = k0; k < k1; ++k) {
            const int v = v0 + k;
            const float* p = v < kThreadsDx ? red + v * BP : gred + (int64_t)(v - kThreadsDx) * BP;
#pragma unroll
            for (int t = 0; t < BP; ++t) u[t] += p[t];
        }
#pragma unroll
        for (int t = 0; t < BP; ++t) sum[t] += u[t];
    }
}

// A further virtual lane of a thread (blocks with more than NT / 2 columns
// only): walked once over all rows after the phases, its operand read
// straight from X, its partial kept in global scratch.
template <int BP>
__device__ __forceinline__ void sweep_extra(const SpmmArgs& a, const int4 ln, float* g) {
    SweepLane<BP> w2;
    w2.init(ln);
    w2.prime(a, 0xffffffffu);
    w2.template run<true>(a, nullptr, 0, (int)a.n_src);
#pragma unroll
    for (int t = 0; t < BP; ++t) g[t] = w2.outer[t];
}

// Phase ph stages operand rows [ph sw_rows, (ph + 1) sw_rows); a lane
// stops where the tables say its column crosses the phase's last row.
template <int BP>
__global__ void __launch_bounds__(kThreadsDx, 1) k_sweep(const SpmmArgs a) {
    static_assert(BP <= 4, "one lane holds all BP columns of an entry");
    constexpr int NT = kThreadsDx;
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);
    SweepLane<BP> w;
    w.init(a.sw_lane[a.sw_blk[2 * blockIdx.x].w + threadIdx.x]);
    const int n_rows = (int)a.n_src;
    const int v0 = a.sw_blk[2 * blockIdx.x].w + threadIdx.x;
    for (int ph = 0; ph < a.sw_phases; ++ph) {
        const int r0 = ph * a.sw_rows, r1 = min(n_rows, r0 + a.sw_rows);
        // this lane's resume quad at row r1 (twice it, plus one when that
        // quad also holds entries below r1)
        const bool cut = ph + 1 < a.sw_phases;
        const int sp = cut ? __ldg(a.sw_split + (int64_t)((ph + 1) * a.sw_stride - 1) * a.sw_nlane + v0) : -2;
        if (ph > 0) __syncthreads();   // the previous phase's rows are read no more
        stage_transposed<BP, false>(xs, a.X + r0, a.n_src, a.b, r1 - r0, threadIdx.x, NT);
        __syncthreads();
        w.prime(a, cut ? (uint32_t)(sp >> 1) + (uint32_t)(sp & 1) : 0xffffffffu);
        w.run(a, xs, r0, r1);
        if (cut) w.u = (uint32_t)(sp >> 1);
    }
    const int4 b = a.sw_blk[2 * blockIdx.x], b2 = a.sw_blk[2 * blockIdx.x + 1];
    const int T = b.z;   // virtual lanes, a multiple of NT
    float* gred = a.sw_gpart + (int64_t)b2.y * BP;
    for (int v = threadIdx.x + NT; v < T; v += NT)
        sweep_extra<BP>(a, a.sw_lane[b.w + v], gred + (int64_t)(v - NT) * BP);
    __syncthreads();   // the operand is read no more: its space takes the partials
    float* red = xs;
#pragma unroll
    for (int t = 0; t < BP; ++t) red[threadIdx.x * BP + t] = w.outer[t];
    __syncthreads();
    const int lo = b.x, ncols = b.y - b.x;
    for (int i = threadIdx.x; i < ncols; i += NT) {
        const int c = lo + i;
        if (c == b2.z || c == b2.w) continue;
        const int2 cr = a.sw_col[b2.x + i];
        float sum[BP];
        sweep_sum<BP>(red, gred, cr.x, cr.y, sum);
#pragma unroll
        for (int t = 0; t < BP; ++t)
            if (t < a.b) a.Y[(int64_t)t * a.n_seg + c] = sum[t];
    }
    // the columns cut by the block's boundaries: warp 0 the head, warp 1 the tail
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = warp == 0 ? b2.z : (warp == 1 ? b2.w : -1);
    if (c >= 0) {
        const int2 cr = a.sw_col[b2.x + (c - lo)];
        float sum[BP];
        sweep_sum<BP>(red, gred, cr.x, cr.y, sum);
        // in the chunk walk's lane layout: lane sub < LPE holds its VEC columns
        using TL = Tile<BP>;
        const int sub = lane % TL::LPE;
        float mine[TL::VEC];
#pragma unroll
        for (int j = 0; j < TL::VEC; ++j) mine[j] = sum[TL::beta(sub, j)];
        const BlockDesc bd = a.bdesc[blockIdx.x];
        if (warp == 0) {
            if (__ldg(a.seg_ptr + c + 1) <= bd.k1)
                cross_block<BP>(a, c, 0, mine, bd.head_first, blockIdx.x, bd.n_head, lane, sub);
            else
                cross_block<BP>(a, c, 0, mine, bd.head_first, bd.tail_last, bd.n_head + bd.n_tail - 1, lane, sub);
        } else {
            cross_block<BP>(a, c, 1, mine, blockIdx.x, bd.tail_last, bd.n_tail, lane, sub);
        }
    }
}

// Transposed copy of the operand for the global-memory path.
template <int BP>
__global__ void k_transpose(const float* __restrict__ X, int64_t n, int b, float* __restrict__ xt) {
    stage_transposed<BP>(xt, X, n, b, n, blockIdx.x * blockDim.x + threadIdx.x,
                         gridDim.x * blockDim.x);
}

// Y[beta, o] = bias[o] (or 0) when W holds no entries.
__global__ void k_fill_bias(float* Y, int64_t b, int64_t n, const float* bias) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < b * n;
         i += (int64_t)gridDim.x * blockDim.x)
        Y[i] = bias ? bias[i % n] : 0.f;
}

template <typename F>
static int set_smem(F fn, size_t smem) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return SNK_ERR_CUDA;
    return SNK_OK;
}

template <int BP, bool GATHER>
static int launch_bp(Layer* L, SpmmArgs a, cudaStream_t s) {
    constexpr int NT = SpmmShape<GATHER>::kNT;
    const size_t slots = spmm_slot_bytes<BP, GATHER>();
    const size_t smem = operand_floats(a.n_src, BP) * sizeof(float) + slots;
    if constexpr (GATHER && BP <= 4) {
        // the column sweep, when the layer has its tables: the tables cut
        // the rows into P equal phases (P a power of two, ~96 KB of a
        // 4-column operand each); 4- and 2-column tiles take them all (the
        // 2-column phases then leave L1 more room: 35.0 against 36.4 us at
        // 10000^2, 90%), a 1-column tile takes P / 2 (at least one)
        SweepView v;
        if (a.idx16 && !a.bias && sweep_view(L, &v)) {
            // Phases pay for a barrier and a restart of every lane's stream;
            // with fewer than 32 entries per lane (8 quads) one phase is
            // faster when the whole operand fits (10000^2, 99%, b = 4: 18.5
            // against 20.4 us).
            const bool few = a.nnz < (int64_t)32 * a.n_blocks * kThreadsDx;
            const bool fits = operand_floats(a.n_src, BP) * sizeof(float) <= (size_t)L->max_smem;
            const int phases = (few && fits) ? 1 : (BP >= 2 ? v.phases : std::max(1, v.phases / 2));
            const int stride = v.phases / phases;
            const int64_t rows = phases == 1 ? a.n_src : std::min<int64_t>(a.n_src, (int64_t)v.rows * stride);
            const size_t smem_sw = std::max(operand_floats(rows, BP), (size_t)kThreadsDx * BP) * sizeof(float);
            if (smem_sw <= (size_t)L->max_smem) {
                a.sw_blk = v.blk;
                a.sw_col = v.col;
                a.sw_lane = v.lane;
                a.sw_split = v.split;
                a.sw_nlane = v.n_lane;
                a.sw_gpart = L->xt;
                a.sw_rows = (int)rows;
                a.sw_phases = phases;
                a.sw_stride = stride;
                a.perm = v.perm;
                a.idx16 = v.r16;
                auto fn = k_sweep<BP>;
                if (set_smem(fn, smem_sw) != SNK_OK) return SNK_ERR_CUDA;
                fn<<<a.n_blocks, kThreadsDx, smem_sw, s>>>(a);
                return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
            }
        }
    }
    if (smem <= (size_t)L->max_smem && a.idx16) {
        auto fn = k_spmm<BP, GATHER, true>;
        if (set_smem(fn, smem) != SNK_OK) return SNK_ERR_CUDA;
        fn<<<a.n_blocks, NT, smem, s>>>(a);
    } else {
        k_transpose<BP><<<L->num_sms * 4, 256, 0, s>>>(a.X, a.n_src, a.b, L->xt);
        a.xt = L->xt;
        auto fn = k_spmm<BP, GATHER, false>;
        if (set_smem(fn, slots) != SNK_OK) return SNK_ERR_CUDA;
        fn<<<a.n_blocks, NT, slots, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

template <bool GATHER>
static int launch_tile(Layer* L, const SpmmArgs& a, int bp, cudaStream_t s) {
    switch (bp) {
        case 1: return launch_bp<1, GATHER>(L, a, s);
        case 2: return launch_bp<2, GATHER>(L, a, s);
        case 4: return launch_bp<4, GATHER>(L, a, s);
        case 8: return launch_bp<8, GATHER>(L, a, s);
        case 16: return launch_bp<16, GATHER>(L, a, s);
        case 32: return launch_bp<32, GATHER>(L, a, s);
        default: return launch_bp<64, GATHER>(L, a, s);
    }
}

template <bool GATHER>
static int run_spmm(Layer* L, SpmmArgs a, int64_t b, cudaStream_t s) {
    const float* X0 = a.X;
    float* Y0 = a.Y;
    for (int64_t t0 = 0; t0 < b; t0 += kMaxBatchTile) {
        const int64_t bt = std::min<int64_t>(kMaxBatchTile, b - t0);
        a.b = (int)bt;
        a.X = X0 + t0 * a.n_src;
        a.Y = Y0 + t0 * a.n_seg;
        if (a.nnz == 0) {
            k_fill_bias<<<L->num_sms * 4, 256, 0, s>>>(a.Y, bt, a.n_seg, a.bias);
            if (cudaGetLastError() != cudaSuccess) return SNK_ERR_CUDA;
            continue;
        }
        int st = launch_tile<GATHER>(L, a, batch_tile(bt), s);
        if (st != SNK_OK) return st;
    }
    return SNK_OK;
}

// Forward SpMM on a caller's CSR (32-bit column indices) with a partition and
// scratch supplied by the caller (the allocation-free entry point).  Shared-
// memory operand path only.
template <int BP>
static int launch_csr_bp(SpmmArgs a, int max_smem, cudaStream_t s) {
    const size_t smem = operand_floats(a.n_src, BP) * sizeof(float) + spmm_slot_bytes<BP, false>();
    if (smem > (size_t)max_smem) return SNK_ERR_LIMIT;
    auto fn = k_spmm<BP, false, true, false>;
    if (set_smem(fn, smem) != SNK_OK) return SNK_ERR_CUDA;
    fn<<<a.n_blocks, kThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

size_t forward_csr_smem(int64_t in_f, int bp) {
    size_t slots = 0;
    switch (bp) {
        case 1: slots = spmm_slot_bytes<1, false>(); break;
        case 2: slots = spmm_slot_bytes<2, false>(); break;
        case 4: slots = spmm_slot_bytes<4, false>(); break;
        case 8: slots = spmm_slot_bytes<8, false>(); break;
        case 16: slots = spmm_slot_bytes<16, false>(); break;
        case 32: slots = spmm_slot_bytes<32, false>(); break;
        default: slots = spmm_slot_bytes<64, false>(); break;
    }
    return operand_floats(in_f, bp) * sizeof(float) + slots;
}

int launch_forward_csr(const float* val, const int32_t* cols, const int32_t* row_ptr,
                       const int4* cdesc, const BlockDesc* bdesc, const int32_t* bnd, int64_t nnz,
                       int64_t out_f, int64_t in_f, int n_blocks, const float* X, int64_t b,
                       const float* bias, float* Y, float* part, int32_t* cnt, int max_smem,
                       cudaStream_t s) {
    SpmmArgs a{};
    a.val = val;
    a.idx = cols;
    a.seg_ptr = row_ptr;
    a.cdesc = cdesc;
    a.bdesc = bdesc;
    a.bnd = bnd;
    a.nnz = nnz;
    a.n_seg = out_f;
    a.n_src = in_f;
    a.n_blocks = n_blocks;
    a.bias = bias;
    a.part = part;
    a.cnt = cnt;
    for (int64_t t0 = 0; t0 < b; t0 += kMaxBatchTile) {
        const int64_t bt = std::min<int64_t>(kMaxBatchTile, b - t0);
        a.b = (int)bt;
        a.X = X + t0 * in_f;
        a.Y = Y + t0 * out_f;
        int st;
        if (nnz == 0) {
            k_fill_bias<<<n_blocks * 4, 256, 0, s>>>(a.Y, bt, out_f, bias);
            st = cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
        } else {
            switch (batch_tile(bt)) {
                case 1: st = launch_csr_bp<1>(a, max_smem, s); break;
                case 2: st = launch_csr_bp<2>(a, max_smem, s); break;
                case 4: st = launch_csr_bp<4>(a, max_smem, s); break;
                case 8: st = launch_csr_bp<8>(a, max_smem, s); break;
                case 16: st = launch_csr_bp<16>(a, max_smem, s); break;
                case 32: st = launch_csr_bp<32>(a, max_smem, s); break;
                default: st = launch_csr_bp<64>(a, max_smem, s); break;
            }
        }
        if (st != SNK_OK) return st;
    }
    return SNK_OK;
}

static SpmmArgs layer_args(Layer* L, bool columns) {
    SpmmArgs a{};
    a.val = L->v;
    a.nnz = L->nnz;
    a.n_blocks = L->n_blocks;
    a.part = L->part;
    a.cnt = L->cnt;
    if (!columns) {
        a.idx = L->c;
        a.idx16 = L->c16;
        a.seg_ptr = L->row_ptr;
        a.cdesc = L->cdesc_r;
        a.bdesc = L->bdesc_r;
        a.bnd = L->bnd_r;
        a.n_seg = L->out_f;
        a.n_src = L->in_f;
    } else {
        a.perm = L->perm;
        a.idx = L->rows_c;
        a.idx16 = L->rc16;
        a.seg_ptr = L->col_ptr;
        a.cdesc = L->cdesc_c;
        a.bdesc = L->bdesc_c;
        a.bnd = L->bnd_c;
        a.n_seg = L->in_f;
        a.n_src = L->out_f;
    }
    return a;
}

int launch_forward(Layer* L, const float* X, int64_t b, const float* bias, float* Y,
                   cudaStream_t s) {
    if (tc_eligible(L, b)) return run_tc(L, false, X, b, bias, Y, s);
    SpmmArgs a = layer_args(L, false);
    a.X = X;
    a.bias = bias;
    a.Y = Y;
    return run_spmm<false>(L, a, b, s);
}

int launch_backward_input(Layer* L, const float* dY, int64_t b, float* dX, cudaStream_t s) {
    if (tc_eligible(L, b)) return run_tc(L, true, dY, b, nullptr, dX, s);
    SpmmArgs a = layer_args(L, true);
    a.X = dY;
    a.bias = nullptr;
    a.Y = dX;
    return run_spmm<true>(L, a, b, s);
}

}  // namespace snk
