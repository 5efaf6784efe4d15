// Row runs over column bands: the weight gradient for batch tiles whose
// operand does not fit shared memory.
//
//   "Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
//     sec. 7.1 (dL/dW is wanted only at the live slots of W: for each one
//     the dot product of a dL/dY row with an X row).
//   "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
//     GPU", Fig. 3 (the layer at batch 1..64).
//
// At a batch tile of BP >= 8 columns the operand X^T takes in * BP * 4 bytes
// (320 KB at in = 10000, BP = 8; 2.5 MB at BP = 64), more than a block's
// shared memory, and the row-order kernel reads each entry's X row through
// L1 from a transposed copy in L2.  Here the columns are cut into nb bands
// of `width` columns that each fit shared memory; a block owns one band and
// a range of rows, copies its band of the transposed operand in once (one
// TMA bulk copy), and its warps walk the rows of the range: row r's entries
// in band k are one contiguous run of the canonical order (columns ascend
// within a row), found in a table built with the topology, so the column
// indices stream from their canonical places with 128-bit loads, the row's
// dY values sit in registers for the whole run, and every gradient is
// written in place.  No gather, no second copy of the entries.
//
// Measured at 10000^2 (us per call, L2 flushed; row-order kernel -> bands):
// 90%: b = 16 112.6 -> 95.4, b = 32 172.6 -> 121.7, b = 64 279.4 -> 211.0;
// 95%: b = 32 101.0 -> 77.9.  Short runs lose: every run costs a table
// lookup and a dY row, and a band's staging is paid even for few entries
// (99%, b = 64: 59.8 -> 91.2).  So the bands are taken only when the runs
// average at least kMinRun entries and a block's entries are at least twice
// its band's columns.  (The forward on the same runs, its band results added
// by a second kernel, was slower than the row-order kernel at b = 8, 16 and
// 64 and within 2% at 32: 90%, b = 8: 50.5 -> 55.7 us; b = 64: 155 -> 178.)
//
// Table (per batch tile 8, 16, 32, 64; built on first use, rebuilt in place
// with the topology so captured graphs stay valid):
//   run[k * out + r] = the first canonical slot of row r with column >=
//                      k * width (k = nb: the row's end);
//   cut[j]           = the first row of block j of a band (rows balanced by
//                      their entries; every band uses the same cuts).
#include <algorithm>

#include "snk_device.cuh"

namespace snk {

struct BandTable {
    bool alloc = false;   // arrays allocated (shapes fixed)
    bool failed = false;  // allocation failed: this tile keeps the row-order kernel
    bool valid = false;   // built for `version`
    int bp = 0, nb = 0, width = 0, bpb = 0;   // batch tile, bands, columns per band, blocks per band
    int64_t version = -1;
    int32_t* run = nullptr;   // [(nb + 1) * out]
    int32_t* cut = nullptr;   // [bpb + 1]
};

struct Bands {
    BandTable t[4];   // batch tiles 8, 16, 32, 64
};

namespace {

constexpr int64_t kMinRun = 40;   // entries per (band, row) run, on average

int tile_slot(int bp) { return bp <= 8 ? 0 : bp <= 16 ? 1 : bp <= 32 ? 2 : 3; }

template <typename T>
bool b_alloc(T** p, int64_t count) {
    if (cudaMalloc((void**)p, (size_t)std::max<int64_t>(count, 1) * sizeof(T)) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return false;
    }
    return true;
}

void free_table(BandTable* t) {
    void* ptrs[] = {t->run, t->cut};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    *t = BandTable{};
}

// First position in idx[lo, hi) (ascending) holding a value >= v.
__device__ __forceinline__ int64_t first_ge(const int32_t* idx, int64_t lo, int64_t hi, int64_t v) {
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)idx[mid] < v) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__global__ void k_band_runs(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col, int64_t out,
                            int nb, int width, int32_t* __restrict__ run) {
    const int64_t n = (int64_t)(nb + 1) * out;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
        const int k = (int)(t / out);
        const int64_t r = t - (int64_t)k * out;
        const int64_t lo = row_ptr[r], hi = row_ptr[r + 1];
        run[t] = (int32_t)(k == 0 ? lo : (k == nb ? hi : first_ge(col, lo, hi, (int64_t)k * width)));
    }
}

// cut[j] = the first row whose entries start at or after j * nnz / bpb.
__global__ void k_band_cuts(const int32_t* __restrict__ row_ptr, int64_t out, int64_t nnz, int bpb,
                            int32_t* __restrict__ cut) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j > bpb) return;
    if (j == 0 || j == bpb) {
        cut[j] = j == 0 ? 0 : (int32_t)out;
        return;
    }
    const int64_t t = (int64_t)j * nnz / bpb;
    cut[j] = (int32_t)first_ge(row_ptr, 0, out, t);
}

int build_table(Layer* L, BandTable* t, cudaStream_t s) {
    const int T = 256;
    const int64_t n = (int64_t)(t->nb + 1) * L->out_f;
    const unsigned g = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, T), (int64_t)L->num_sms * 8));
    k_band_runs<<<g, T, 0, s>>>(L->row_ptr, L->c, L->out_f, t->nb, t->width, t->run);
    k_band_cuts<<<(unsigned)ceil_div(t->bpb + 1, T), T, 0, s>>>(L->row_ptr, L->out_f, L->nnz, t->bpb, t->cut);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

}  // namespace

bool band_shape(const Layer* L, int bp, int* nb, int* width) {
    // the operand band and the staging barrier (static shared memory)
    const int64_t avail = (int64_t)L->max_smem - 128;
    if (bp < 8 || !L->c16 || avail <= 0) return false;
    const int64_t fit = (avail / ((int64_t)bp * 4)) & ~(int64_t)3;
    if (fit < 64) return false;
    const int64_t k = ceil_div(L->in_f, fit);
    const int64_t w = (ceil_div(L->in_f, k) + 3) & ~(int64_t)3;
    // at least two bands, and at least two blocks for each
    if (k < 2 || 2 * k > L->n_blocks) return false;
    // long enough runs, and more entries per block than its band stages
    if (L->nnz < (int64_t)kMinRun * k * L->out_f || L->nnz < (int64_t)2 * w * L->n_blocks) return false;
    *nb = (int)k;
    *width = (int)w;
    return true;
}

const BandTable* band_table(Layer* L, int bp, cudaStream_t s, int* status) {
    *status = SNK_OK;
    int nb = 0, width = 0;
    if (L->nnz == 0 || !band_shape(L, bp, &nb, &width)) return nullptr;
    if (!L->bands) L->bands = new Bands();
    BandTable* t = &L->bands->t[tile_slot(bp)];
    if (t->valid && t->version == L->topology_version) return t;
    if (t->failed) return nullptr;
    if (!t->alloc) {
        t->bp = bp;
        t->nb = nb;
        t->width = width;
        t->bpb = L->n_blocks / nb;
        if (!b_alloc(&t->run, (int64_t)(nb + 1) * L->out_f) || !b_alloc(&t->cut, t->bpb + 1)) {
            // the bands are an optimisation: without their table the call
            // runs the row-order kernel, now and later
            free_table(t);
            t->failed = true;
            return nullptr;
        }
        t->alloc = true;
    }
    t->valid = false;
    if (int st = build_table(L, t, s); st != SNK_OK) {
        *status = st;
        return nullptr;
    }
    t->valid = true;
    t->version = L->topology_version;
    return t;
}

int refresh_bands(Layer* L, cudaStream_t s) {
    if (!L->bands) return SNK_OK;
    for (auto& t : L->bands->t) {
        if (!t.alloc) continue;
        t.valid = false;
        if (int st = build_table(L, &t, s); st != SNK_OK) return st;
        t.valid = true;
    }
    return SNK_OK;
}

void mark_bands(Layer* L) {
    if (!L->bands) return;
    for (auto& t : L->bands->t)
        if (t.alloc && t.valid) t.version = L->topology_version;
}

void free_bands(Layer* L) {
    if (!L->bands) return;
    for (auto& t : L->bands->t) free_table(&t);
    delete L->bands;
    L->bands = nullptr;
}

// ---------------------------------------------------------------------------
// The kernel.

struct BandArgs {
    const uint16_t* c16;     // canonical columns, 16-bit, zero padded
    const int32_t* run;      // run table
    const int32_t* cut;      // row cuts of a band's blocks
    const float* xt;         // [in][BP] transposed operand
    int64_t out_f, in_f;
    int nb, width, bpb, b;
    const float* dY;         // [b, out] (tile)
    float* dW;               // [nnz]
    bool accumulate;         // add to dW (later batch tiles)
    const float* dY_all;     // [b_all, out] for db, or null
    int64_t b_all;
    float* db;               // [out] or null
    int32_t* status;         // device status word (a staging wait that ran out)
};

// One warp per row at a time (the rows of the block's range taken
// cyclically); the run [c0, c1) streams as blocks of 4*GPW column indices
// from the multiple of 4 at or below c0, NS blocks in flight; blocks wholly
// inside the run are consumed without masks.  The row's dY values are in
// registers for the whole run, and the next row's (and its run bounds) are
// requested while this one is walked.  Each entry's dot product is reduced
// over the LPE lanes that share it, and the 4 results of a group go out with
// one 128-bit store when the quad lies inside the run.
template <int BP>
__global__ void __launch_bounds__(kThreads, 1) k_band_dw(const BandArgs a) {
    using TL = Tile<BP>;
    constexpr int VEC = TL::VEC, LPE = TL::LPE, GPW = TL::GPW;
    constexpr uint32_t BLK = 4 * GPW;
    constexpr int NS = 3;
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);
    __shared__ uint64_t stage_bar;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = lane / LPE, sub = lane % LPE;
    const int k = blockIdx.x / a.bpb, j = blockIdx.x - k * a.bpb;
    const int r0 = __ldg(a.cut + j), r1 = __ldg(a.cut + j + 1);
    const int col0 = k * a.width;
    const int ncol = min(a.width, (int)a.in_f - col0);
    const int32_t* run_lo = a.run + (int64_t)k * a.out_f;
    const int32_t* run_hi = run_lo + a.out_f;

    if (a.db) {
        // bias gradient over the whole batch, sequential in batch order
        for (int64_t o = blockIdx.x * (int64_t)kThreads + threadIdx.x; o < a.out_f;
             o += (int64_t)gridDim.x * kThreads) {
            float sacc = 0.f;
            for (int64_t beta = 0; beta < a.b_all; ++beta) sacc += a.dY_all[beta * a.out_f + o];
            a.db[o] = sacc;
        }
    }
    auto dy_row = [&](int row, float (&d)[VEC]) {
#pragma unroll
        for (int t = 0; t < VEC; ++t) {
            const int beta = TL::beta(sub, t);
            d[t] = (row < r1 && beta < a.b) ? __ldg(a.dY + (int64_t)beta * a.out_f + row) : 0.f;
        }
    };
    // the first row's run and dY values, then the band's operand rows
    int r = r0 + warp;
    uint32_t c0 = 0, c1 = 0;
    if (r < r1) {
        c0 = (uint32_t)__ldg(run_lo + r);
        c1 = (uint32_t)__ldg(run_hi + r);
    }
    float dyr[VEC];
    dy_row(r, dyr);
    stage_band<BP>(xs, a.xt, col0, ncol, &stage_bar, a.status);
    __syncthreads();

    for (; r < r1; r += kWarpsPerBlock) {
        const int rn = r + kWarpsPerBlock;
        uint32_t n0 = 0, n1 = 0;
        if (rn < r1) {
            n0 = (uint32_t)__ldg(run_lo + rn);
            n1 = (uint32_t)__ldg(run_hi + rn);
        }
        float dyn[VEC];
        dy_row(rn, dyn);
        if (c0 < c1) {
            IdxBlk<true> ib[NS];
            const uint32_t bf = c0 & ~3u;
            auto consume = [&](int s, uint32_t blk0) {
                const uint32_t base = blk0 + 4 * grp;
                const bool interior = c0 <= blk0 && blk0 + BLK <= c1;
                float res[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t e = base + q;
                    if (interior || (e >= c0 && e < c1)) {
                        float x[VEC];
                        TL::load(xs + (ib[s].get(q) - col0) * BP, sub, x);
                        float p = 0.f;
#pragma unroll
                        for (int t = 0; t < VEC; ++t) p = fmaf(dyr[t], x[t], p);
                        res[q] = p;
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int o = 1; o < LPE; o <<= 1) res[q] += __shfl_xor_sync(0xffffffffu, res[q], o);
                if (sub == 0) {
                    if (base >= c0 && base + 3 < c1) {
                        float4 v = make_float4(res[0], res[1], res[2], res[3]);
                        float4* dst = reinterpret_cast<float4*>(a.dW + base);
                        if (a.accumulate) {
                            const float4 o4 = *dst;
                            v.x += o4.x;
                            v.y += o4.y;
                            v.z += o4.z;
                            v.w += o4.w;
                        }
                        *dst = v;
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t e = base + q;
                            if (e >= c0 && e < c1) a.dW[e] = a.accumulate ? a.dW[e] + res[q] : res[q];
                        }
                    }
                }
            };
#pragma unroll
            for (int s = 0; s < NS; ++s)
                if (bf + s * BLK < c1) ib[s].load(a.c16, bf + s * BLK + 4 * grp);
            for (uint32_t b0 = bf; b0 < c1; b0 += NS * BLK) {
#pragma unroll
                for (int s = 0; s < NS; ++s) {
                    const uint32_t blk0 = b0 + s * BLK;
                    if (blk0 < c1) {
                        consume(s, blk0);
                        if (blk0 + NS * BLK < c1) ib[s].load(a.c16, blk0 + NS * BLK + 4 * grp);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < VEC; ++t) dyr[t] = dyn[t];
        c0 = n0;
        c1 = n1;
    }
}

// The operand transposed into xt[n][BP] (zero columns beyond b).
template <int BP>
__global__ void k_band_transpose(const float* __restrict__ X, int64_t n, int b, float* __restrict__ xt) {
    stage_transposed<BP>(xt, X, n, b, n, blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x);
}

namespace {

template <int BP>
int launch_band_bp(Layer* L, BandArgs a, const BandTable* t, const float* X, cudaStream_t s) {
    k_band_transpose<BP><<<L->num_sms * 4, 256, 0, s>>>(X, L->in_f, a.b, L->xt);
    a.xt = L->xt;
    a.run = t->run;
    a.cut = t->cut;
    a.nb = t->nb;
    a.width = t->width;
    a.bpb = t->bpb;
    a.status = L->status;
    const size_t smem = (size_t)t->width * BP * sizeof(float);
    auto fn = k_band_dw<BP>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return SNK_ERR_CUDA;
    fn<<<t->nb * t->bpb, kThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

}  // namespace

int band_backward_weight(Layer* L, int bp, const float* X, const float* dY, int b, float* dW, bool accumulate,
                         const float* dY_all, int64_t b_all, float* db, cudaStream_t s, bool* done) {
    *done = false;
    int st = SNK_OK;
    const BandTable* t = band_table(L, bp, s, &st);
    if (st != SNK_OK || !t) return st;
    BandArgs a{};
    a.c16 = L->c16;
    a.out_f = L->out_f;
    a.in_f = L->in_f;
    a.b = b;
    a.dY = dY;
    a.dW = dW;
    a.accumulate = accumulate;
    a.dY_all = dY_all;
    a.b_all = b_all;
    a.db = db;
    *done = true;
    switch (t->bp) {
        case 8: return launch_band_bp<8>(L, a, t, X, s);
        case 16: return launch_band_bp<16>(L, a, t, X, s);
        case 32: return launch_band_bp<32>(L, a, t, X, s);
        default: return launch_band_bp<64>(L, a, t, X, s);
    }
}

}  // namespace snk
