// Lane tables of the column sweep (the transposed product at batch 1..4).
//
//   "Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
//     sec. 7.1 (dL/dX is another SpMM through W^T), sec. 7.2 (W^T is read
//     through a permutation built once per topology).
//
// The transposed product gathers one value per stored entry, values[perm[k]],
// and a block's column range holds, for every row of W, a few entries that
// sit next to each other in canonical order (one or two 32-byte sectors).
// When the block's threads are at unrelated rows, nearly every entry fetches
// its sector again.  The sweep gives every column of a block its own set of
// threads ("lanes"), as many as its share of the block's entries, and the
// lanes of a column stride over its entries in row order.  All columns then
// advance through the rows at the same pace, and the entries of one row are
// gathered close together in time while their sector is still in L1
// (measured at 10000^2, 90%: a gather of 36.5 us this way against 46.9 us
// with the threads in contiguous chunks).
//
// Tables (rebuilt in place with the topology; sizes fixed at the first build
// so that a captured graph stays valid):
//   blk[2c]   = (first column, end column, virtual lanes T, first lane)
//   blk[2c+1] = (first column record, first global partial, head, tail)
//   col[r]    = (first virtual lane, lanes) of each column of each block
//   lane[v]   = (first quad, quad stride, first entry, end entry)
// Block c owns the columns its warp chunks own in the merge-path partition
// (the same ownership as the chunk walk); head / tail is the column cut by
// the block's first / last boundary (or -1), whose partial sums go through
// the cross-block protocol.  With m non-empty columns and L entries, the
// block has T = NT virtual lanes (NT threads) when m <= NT / 2, else
// NT * ceil(2m / NT); column j of length l gets 1 + floor(l (T - m) / L)
// lanes, so no lane holds more than L / (T - m) <= 2 L / NT entries.
// Threads take virtual lanes v, v + NT, ...; partials of v >= NT are kept in
// the layer's transposed-operand scratch (unused on this path).
//
// Row phases: the rows are cut into P equal phases (P the least power of two,
// at most 8, that keeps a phase of a 4-column operand within
// SNK_SWEEP_PHASE_KB); for every lane and every cut at row R the tables hold
// 2 U + x, U = the lane's first quad at or after the quad holding the
// column's first entry with row >= R, x = 1 when U is that very quad (it
// straddles R).  Rows rise along a column, so the lane's quads before U lie
// wholly below R.
#include <algorithm>

#include "snk_internal.cuh"

namespace snk {

struct Sweep {
    bool enabled = false;
    bool valid = false;
    int64_t version = -1;
    int64_t cap_col = 0, cap_lane = 0;
    int4* blk = nullptr;
    int2* col = nullptr;
    int4* lane = nullptr;
    int4* tmp = nullptr;     // [2 n_blocks]: (columns, T, m, gpart lanes), (first col, end col, head, tail)
    int32_t* err = nullptr;  // [2]: capacity overrun; the total virtual lanes
    int* split = nullptr;    // [phases - 1][cap_lane] resume quads at the cuts
    int phases = 1, rows = 0;
    int32_t* perm = nullptr;  // [nnz_pad] the column view's slots, reordered within quads
    uint16_t* r16 = nullptr;  // [nnz_pad] its rows, reordered the same way
};

namespace {

constexpr int kNT = kThreadsDx;
constexpr int64_t kSweepMaxCols = int64_t(1) << 24;   // 16M columns: 128 MB of column records

// Entry range of column j inside block [b0, b1).
__device__ __forceinline__ void in_block(const int32_t* col_ptr, int64_t j, int64_t b0, int64_t b1, int64_t& s,
                                         int64_t& e) {
    s = max((int64_t)col_ptr[j], b0);
    e = min((int64_t)col_ptr[j + 1], b1);
    if (e < s) e = s;
}

// Per block: its column range (from the chunk table), the number m of
// columns with entries inside the block, T, and the head / tail columns.
__global__ void k_sw_count(const int4* __restrict__ cdesc, const int32_t* __restrict__ bnd,
                           const int32_t* __restrict__ col_ptr, int warps, int n_blocks, int4* __restrict__ tmp) {
    __shared__ int red[32];
    const int c = blockIdx.x;
    const int64_t lo = cdesc[(int64_t)c * warps].z, hi = cdesc[(int64_t)c * warps + warps - 1].w;
    const int64_t b0 = bnd[c], b1 = bnd[c + 1];
    int m = 0;
    for (int64_t j = lo + threadIdx.x; j < hi; j += blockDim.x) {
        int64_t s, e;
        in_block(col_ptr, j, b0, b1, s, e);
        m += e > s;
    }
    for (int o = 16; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
        const int T = (2 * tot <= kNT) ? kNT : kNT * (int)((2 * (int64_t)tot + kNT - 1) / kNT);
        int head = -1, tail = -1;
        if (b1 > b0 && hi > lo) {
            if ((int64_t)col_ptr[lo] < b0) head = (int)lo;
            // below the last block, hi is the first column starting at or
            // after b1, so column hi - 1 holds entry b1 - 1: the tail when it
            // continues past b1 (and is not the head itself)
            const int j = (int)hi - 1;
            if (c < n_blocks - 1 && (int64_t)col_ptr[j + 1] > b1 && j != head) tail = j;
        }
        tmp[2 * c] = make_int4((int)(hi - lo), T, tot, T - kNT);
        tmp[2 * c + 1] = make_int4((int)lo, (int)hi, head, tail);
    }
}

// Prefix sums over the blocks: one warp, each lane a contiguous run of
// blocks (n_blocks is the SM count).
__global__ void k_sw_scan(const int4* __restrict__ tmp, int n_blocks, int64_t cap_col, int64_t cap_lane,
                          int4* __restrict__ blk, int32_t* __restrict__ err) {
    const int ln = threadIdx.x;
    const int per = (n_blocks + 31) / 32;
    const int c0 = min(n_blocks, ln * per), c1 = min(n_blocks, c0 + per);
    long long rec = 0, lane = 0, gp = 0;
    for (int c = c0; c < c1; ++c) {
        const int4 t = tmp[2 * c];
        rec += t.x;
        lane += t.y;
        gp += t.w;
    }
    // exclusive prefix of the lanes' totals
    long long r2 = rec, l2 = lane, g2 = gp;
    for (int o = 1; o < 32; o <<= 1) {
        const long long a = __shfl_up_sync(0xffffffffu, r2, o), b = __shfl_up_sync(0xffffffffu, l2, o),
                        g = __shfl_up_sync(0xffffffffu, g2, o);
        if (ln >= o) {
            r2 += a;
            l2 += b;
            g2 += g;
        }
    }
    const long long rec_all = __shfl_sync(0xffffffffu, r2, 31), lane_all = __shfl_sync(0xffffffffu, l2, 31);
    rec = r2 - rec;
    lane = l2 - lane;
    gp = g2 - gp;
    for (int c = c0; c < c1; ++c) {
        const int4 t = tmp[2 * c], u = tmp[2 * c + 1];
        blk[2 * c] = make_int4(u.x, u.y, t.y, (int)lane);
        blk[2 * c + 1] = make_int4((int)rec, (int)gp, u.z, u.w);
        rec += t.x;
        lane += t.y;
        gp += t.w;
    }
    if (ln == 0) {
        if (rec_all > cap_col || lane_all > cap_lane) err[0] = 1;
        err[1] = (int32_t)min(lane_all, (long long)cap_lane);
    }
}

// Lanes per column and the lane records.  Column records first (a block-wide
// scan of the lane counts), then each column writes its lanes.
__global__ void k_sw_assign(const int4* __restrict__ tmp, const int4* __restrict__ blk,
                            const int32_t* __restrict__ bnd, const int32_t* __restrict__ col_ptr,
                            const int32_t* __restrict__ err, int2* __restrict__ col, int4* __restrict__ lane) {
    __shared__ int red[33];
    if (*err) return;
    const int c = blockIdx.x;
    const int4 t = tmp[2 * c];
    const int4 b = blk[2 * c], b2 = blk[2 * c + 1];
    const int64_t b0 = bnd[c], b1 = bnd[c + 1];
    const int64_t L = b1 - b0;
    const int lo = b.x, ncols = t.x, T = t.y, m = t.z;
    const int64_t spare = T - m;
    int carry = 0;
    for (int base = 0; base < ncols; base += blockDim.x) {
        const int i = base + threadIdx.x;
        int n = 0;
        int64_t s = 0, e = 0;
        if (i < ncols) {
            in_block(col_ptr, lo + i, b0, b1, s, e);
            if (e > s) n = 1 + (int)((e - s) * spare / L);
        }
        // block-wide exclusive scan of n
        int x = n;
        const int ln = threadIdx.x & 31, w = threadIdx.x >> 5;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (ln >= o) x += y;
        }
        if (ln == 31) red[w] = x;
        __syncthreads();
        if (threadIdx.x == 0) {
            int run = 0;
            for (int k = 0; k < (int)(blockDim.x >> 5); ++k) {
                const int v = red[k];
                red[k] = run;
                run += v;
            }
            red[32] = run;
        }
        __syncthreads();
        const int v0 = carry + red[w] + x - n;
        if (i < ncols) {
            col[b2.x + i] = make_int2(v0, n);
            for (int j = 0; j < n; ++j)
                lane[b.w + v0 + j] = make_int4((int)(s >> 2) + j, n, (int)s, (int)e);
        }
        carry += red[32];
        __syncthreads();
    }
    // virtual lanes left over: empty
    for (int v = carry + threadIdx.x; v < T; v += blockDim.x) lane[b.w + v] = make_int4(0, 1, 0, 0);
}

// Resume quads of every lane at the cuts R = rows, 2 rows, ..., (phases - 1) rows.
__global__ void k_sw_split(const int4* __restrict__ lane, const int32_t* __restrict__ err,
                           const int32_t* __restrict__ rows_c, int phases, int rows, int64_t cap_lane,
                           int* __restrict__ split) {
    if (err[0]) return;
    const int64_t n = err[1];
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n; v += (int64_t)gridDim.x * blockDim.x) {
        const int4 l = lane[v];
        const int64_t q0 = l.x, st = l.y, s = l.z, e = l.w;
        for (int p = 1; p < phases; ++p) {
            const int64_t R = (int64_t)p * rows;
            // first entry in [s, e) with row >= R
            int64_t lo = s, hi = e;
            while (lo < hi) {
                const int64_t mid = (lo + hi) >> 1;
                if ((int64_t)rows_c[mid] < R) lo = mid + 1;
                else hi = mid;
            }
            const int64_t Q = lo >> 2;
            const int64_t U = Q <= q0 ? q0 : q0 + (Q - q0 + st - 1) / st * st;
            split[(int64_t)(p - 1) * cap_lane + v] = (int)(2 * U + (U == Q ? 1 : 0));
        }
    }
}

// Order within quads.  In a 128-bit shared load of operand rows a warp is
// served 8 lanes at a time; two lanes of such a quarter that read different
// rows with the same row mod 8 (the same 4 banks, with 4-column rows) cost
// an extra pass.  The quarter's 8 lanes load their quads' entries in the
// same slot order, and the order of the 4 entries inside a quad is free (a
// lane adds them into its own sums).  So for every quarter (8 consecutive
// lanes of a block) and every step of its walk (the quads its lanes take
// side by side, phase by phase, as a 4-column tile runs them), the entries
// of each quad are put in the order that, lane after lane, adds the fewest
// repeated row groups per slot (greedy over the 24 orders; modelled 2.60 ->
// 1.96 passes per quarter with random rows).  Only quads wholly inside their
// column's range in the block and not straddling a phase cut are reordered;
// each such quad belongs to exactly one lane, so the writes do not overlap.
// The copies the sweep reads (perm, 16-bit rows) are the library's own; the
// column view returned to callers keeps its order.  Steps are independent of
// one another (the counts start afresh at each), so the kSwOrderSteps threads
// of a quarter take its steps in turn.
constexpr int kSwOrderSteps = 8;
__device__ __forceinline__ int sw_cost_add(const unsigned char (&cnt)[4][8], const int (&g)[4], const int (&o)[4]) {
    int c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) c += cnt[j][g[o[j]]];   // entries already in that slot's group
    return c;
}

__global__ void k_sw_order(const int4* __restrict__ lane, const int4* __restrict__ blk, const int* __restrict__ split,
                           int phases, int64_t cap_lane, const int32_t* __restrict__ err,
                           const int32_t* __restrict__ perm, const uint16_t* __restrict__ r16,
                           int32_t* __restrict__ perm_o, uint16_t* __restrict__ r16_o) {
    if (err[0]) return;
    const int c = blockIdx.x;
    const int quarter = threadIdx.x % (kNT / 8);   // blockDim = kNT / 8 * kSwOrderSteps
    const int step0 = threadIdx.x / (kNT / 8);
    const int4 b = blk[2 * c];
    const int lane0 = b.w + quarter * 8;
    // the 24 orders of a quad
    int orders[24][4];
    {
        int n = 0;
        for (int a0 = 0; a0 < 4; ++a0)
            for (int a1 = 0; a1 < 4; ++a1)
                for (int a2 = 0; a2 < 4; ++a2) {
                    const int a3 = 6 - a0 - a1 - a2;
                    if (a0 == a1 || a0 == a2 || a1 == a2 || a3 < 0 || a3 > 3 || a3 == a0 || a3 == a1 || a3 == a2)
                        continue;
                    orders[n][0] = a0;
                    orders[n][1] = a1;
                    orders[n][2] = a2;
                    orders[n][3] = a3;
                    ++n;
                }
    }
    int4 ln[8];
    for (int l = 0; l < 8; ++l) ln[l] = lane[lane0 + l];
    for (int p = 0; p < phases; ++p) {
        uint32_t u[8], qend[8];
        int skip[8];   // a quad of this lane that straddles a cut (left unordered)
        for (int l = 0; l < 8; ++l) {
            const uint32_t qe = ((uint32_t)ln[l].w + 3) >> 2;
            u[l] = p == 0 ? (uint32_t)ln[l].x : (uint32_t)(split[(int64_t)(p - 1) * cap_lane + lane0 + l] >> 1);
            if (p + 1 < phases) {
                const int sp = split[(int64_t)p * cap_lane + lane0 + l];
                qend[l] = min(qe, (uint32_t)(sp >> 1) + (uint32_t)(sp & 1));
                skip[l] = (sp & 1) ? (sp >> 1) : -1;
            } else {
                qend[l] = qe;
                skip[l] = -1;
            }
        }
        for (int i = step0;; i += kSwOrderSteps) {
            bool any = false;
            unsigned char cnt[4][8];
            for (int j = 0; j < 4; ++j)
                for (int g = 0; g < 8; ++g) cnt[j][g] = 0;
            // quads of this step: fixed ones first, then the free ones lane by lane
            for (int pass = 0; pass < 2; ++pass) {
                for (int l = 0; l < 8; ++l) {
                    const uint32_t st = (uint32_t)ln[l].y, s0 = (uint32_t)ln[l].z, e0 = (uint32_t)ln[l].w;
                    const uint32_t q = u[l] + (uint32_t)i * st;
                    if (q >= qend[l]) continue;
                    any = true;
                    const bool first_of_phase = p > 0 && q == u[l] && i == 0;   // may straddle the previous cut
                    const bool free_q = 4 * q >= s0 && 4 * q + 3 < e0 && (int)q != skip[l] && !first_of_phase;
                    if ((pass == 0) == free_q) continue;
                    int g[4];
                    for (int j = 0; j < 4; ++j) g[j] = r16[4 * q + j] & 7;
                    if (!free_q) {
                        for (int j = 0; j < 4; ++j) cnt[j][g[j]] += 1;
                        continue;
                    }
                    int best = 0, best_cost = 1 << 30;
                    for (int o = 0; o < 24; ++o) {
                        const int cst = sw_cost_add(cnt, g, orders[o]);
                        if (cst < best_cost) {
                            best_cost = cst;
                            best = o;
                        }
                    }
                    int pv[4];
                    uint16_t rv[4];
                    for (int j = 0; j < 4; ++j) {
                        const int src = 4 * q + orders[best][j];
                        pv[j] = perm[src];
                        rv[j] = r16[src];
                        cnt[j][g[orders[best][j]]] += 1;
                    }
                    for (int j = 0; j < 4; ++j) {
                        perm_o[4 * q + j] = pv[j];
                        r16_o[4 * q + j] = rv[j];
                    }
                }
            }
            if (!any) break;
        }
    }
}

template <typename T>
bool sw_alloc(T** p, int64_t count) {
    if (cudaMalloc((void**)p, (size_t)std::max<int64_t>(count, 1) * sizeof(T)) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return false;
    }
    return true;
}

void sw_free_arrays(Sweep* S) {
    void* ptrs[] = {S->blk, S->col, S->lane, S->tmp, S->err, S->split, S->perm, S->r16};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    S->split = nullptr;
    S->perm = nullptr;
    S->r16 = nullptr;
    S->blk = nullptr;
    S->col = nullptr;
    S->lane = nullptr;
    S->tmp = nullptr;
    S->err = nullptr;
    S->enabled = false;
    S->valid = false;
}

}  // namespace

void free_sweep(Layer* L) {
    if (!L->sweep) return;
    sw_free_arrays(L->sweep);
    delete L->sweep;
    L->sweep = nullptr;
}

// Build (or rebuild in place) the sweep tables after the column view and its
// partition.  The first build allocates them at their upper bounds: column
// records <= in + n_blocks (neighbouring blocks share at most the cut
// column), virtual lanes <= NT n_blocks + 2 min(in + n_blocks, nnz +
// n_blocks), global partials <= 2 (in + n_blocks) lanes of 4 floats in the
// transposed-operand scratch.  Layers wider than kSweepMaxCols columns get
// no tables.
// Layers without 16-bit rows (out > 65536) or entries get no tables; so does
// a layer whose scratch is too small.  A failure leaves the chunk walk in use.
int build_sweep(Layer* L, cudaStream_t s) {
    const int64_t n = L->nnz;
    const int W = kWarpsPerBlockDx;
    if (!L->sweep) {
        L->sweep = new Sweep();
        Sweep* S = L->sweep;
        if (!L->rc16 || n == 0) return SNK_OK;
        // a record per column (empty ones too): very wide layers keep the
        // chunk walk rather than gigabytes of tables
        if (L->in_f > kSweepMaxCols) return SNK_OK;
        S->cap_col = L->in_f + L->n_blocks;
        // non-empty columns per block, summed, are at most the entries (plus
        // the columns cut between blocks)
        S->cap_lane = (int64_t)kNT * L->n_blocks + 2 * std::min(S->cap_col, n + L->n_blocks);
        if (8 * S->cap_col > std::max(L->out_f, L->in_f) * kMaxBatchTile) return SNK_OK;
        if (S->cap_lane >= INT32_MAX || n >= INT32_MAX) return SNK_OK;
        // phases: the least power of two (at most 8) that keeps a phase of a
        // 4-column operand within the budget (a larger layer takes more)
        const int64_t budget_rows = std::max<int64_t>(4, (int64_t)SNK_SWEEP_PHASE_KB * 1024 / 16);
        S->phases = 1;
        while (S->phases < 8 && (int64_t)S->phases * budget_rows < L->out_f) S->phases *= 2;
        S->rows = (int)((ceil_div(L->out_f, S->phases) + 3) & ~(int64_t)3);
        if (!sw_alloc(&S->blk, 2 * (int64_t)L->n_blocks) || !sw_alloc(&S->col, S->cap_col) ||
            !sw_alloc(&S->lane, S->cap_lane) || !sw_alloc(&S->tmp, 2 * (int64_t)L->n_blocks) || !sw_alloc(&S->err, 2) ||
            !sw_alloc(&S->split, (int64_t)(S->phases - 1) * S->cap_lane) || !sw_alloc(&S->perm, L->nnz_pad) ||
            !sw_alloc(&S->r16, L->nnz_pad)) {
            sw_free_arrays(S);
            return SNK_OK;
        }
        S->enabled = true;
    }
    Sweep* S = L->sweep;
    if (!S->enabled) return SNK_OK;
    S->valid = false;
    cudaMemsetAsync(S->err, 0, 2 * sizeof(int32_t), s);
    k_sw_count<<<L->n_blocks, 256, 0, s>>>(L->cdesc_c, L->bnd_c, L->col_ptr, W, L->n_blocks, S->tmp);
    k_sw_scan<<<1, 32, 0, s>>>(S->tmp, L->n_blocks, S->cap_col, S->cap_lane, S->blk, S->err);
    k_sw_assign<<<L->n_blocks, 256, 0, s>>>(S->tmp, S->blk, L->bnd_c, L->col_ptr, S->err, S->col, S->lane);
    if (S->phases > 1)
        k_sw_split<<<(unsigned)std::min<int64_t>(ceil_div(S->cap_lane, 256), (int64_t)L->num_sms * 8), 256, 0, s>>>(
            S->lane, S->err, L->rows_c, S->phases, S->rows, S->cap_lane, S->split);
    // the sweep's own streams: the column view, then its quads reordered
    cudaMemcpyAsync(S->perm, L->perm, L->nnz_pad * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    cudaMemcpyAsync(S->r16, L->rc16, L->nnz_pad * sizeof(uint16_t), cudaMemcpyDeviceToDevice, s);
    k_sw_order<<<L->n_blocks, kNT / 8 * kSwOrderSteps, 0, s>>>(S->lane, S->blk, S->split, S->phases, S->cap_lane,
                                                               S->err, L->perm, L->rc16, S->perm, S->r16);
    int32_t err = 0;
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(&err, S->err, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SNK_ERR_CUDA;
    // a capacity overrun (ruled out by the bounds above) leaves the chunk walk
    S->valid = (err == 0);
    return SNK_OK;
}

void mark_sweep(Layer* L) {
    if (L->sweep && L->sweep->valid) L->sweep->version = L->topology_version;
}

bool sweep_view(const Layer* L, SweepView* v) {
    const Sweep* S = L->sweep;
    if (!S || !S->enabled || !S->valid || S->version != L->topology_version) return false;
    v->blk = S->blk;
    v->col = S->col;
    v->lane = S->lane;
    v->split = S->split;
    v->n_lane = S->cap_lane;
    v->perm = S->perm;
    v->r16 = S->r16;
    v->phases = S->phases;
    v->rows = S->rows;
    return true;
}

}  // namespace snk
