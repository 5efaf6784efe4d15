// Padded-CSR view of a layer, derived from its canonical triple, with batched
// O(1) topology mutation on the GPU.
//
//   "Padded-CSR: A sparse storage format for dynamic sparse training on CPU"
//     sec. 5.1  six arrays: slot values and column indices (-1 marks a
//               padding slot), row_start, row_nnz (a row's live slots come
//               first in its region), row_capacity and a version counter;
//     sec. 5.2  row_capacity = max(1, ceil(row_nnz * (1 + padding_ratio)));
//     sec. 5.3  an insertion writes slot row_start + row_nnz and bumps the
//               counter; a full row is resized (sec. 4.3: more slots, the
//               row copied, its pointers updated);
//     sec. 8.3  compact_all, for dynamic sparse training whose per-row nnz
//               changes.
//
// Readings where the page is silent (the test oracle takes the same ones):
// padding is a whole percentage p and the capacity is computed in integers,
// max(1, (n * (100 + p) + 99) / 100); inserts come in batches: rows whose
// live count plus inserts would overflow move, in ascending row order, to
// fresh slots at the end of the used area with the capacity rule applied to
// the new count (their old slots become padding), then every insert takes the
// next slot of its row in batch order; deletes clear their slots and each
// touched row closes up in order; compact_all lays the rows out again from
// slot 0 with fresh padding and columns ascending.
//
// GB300 mapping: the slot arrays live in HBM with headroom for relocations
// (grown by reallocation when a batch needs more).  An insert batch is a
// stable radix sort of its rows (so slot order follows batch order), one
// scan over the rows that must move, a warp per moved row, and one thread per
// insert; a delete batch is a thread per delete (scan of its row's live
// slots), then a warp per touched row that closes the gaps with a ballot.
#include <algorithm>

#include "snk_internal.cuh"

namespace snk {

struct PcsrState {
    int pct = 20;
    int64_t used = 0;          // slots in use (the end of the last row region)
    int64_t alloc = 0;         // slots allocated
    int64_t version = 0;
    float* val = nullptr;      // [alloc]
    int32_t* col = nullptr;    // [alloc], -1 = padding
    int32_t* row_start = nullptr;
    int32_t* row_nnz = nullptr;
    int32_t* row_cap = nullptr;
    // scratch over rows
    int32_t* rtmp = nullptr;   // [out + 1] per-row insert counts / touched flags
    int32_t* roff = nullptr;   // [out + 1] per-row offsets (scan results)
    int32_t* rneed = nullptr;  // [out + 1] capacity a row moves to (0 = stays)
    int32_t* rmove = nullptr;  // [out + 1] offset of a moved row's new region
    int32_t* scan_tmp = nullptr;
    int64_t scan_tmp_len = 0;
    int32_t* total = nullptr;
    int32_t* status = nullptr;
    // scratch over a batch (grown on demand)
    int64_t bcap = 0;
    void* bkeys = nullptr;     // 2 * bcap uint64
    uint32_t* bvals = nullptr; // 2 * bcap
    int32_t* bslot = nullptr;  // bcap
    int32_t* hist = nullptr;
    int64_t hist_len = 0;
};

namespace {

constexpr int kBadRange = 1;
constexpr int kNotLive = 2;
constexpr int kDup = 4;

__host__ __device__ inline int32_t pcsr_capacity(int64_t n, int pct) {
    const int64_t c = (n * (100 + pct) + 99) / 100;
    return (int32_t)(c < 1 ? 1 : c);
}

unsigned grid_of(int64_t n, int num_sms) {
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, 256), (int64_t)num_sms * 8));
}

template <typename T>
bool dalloc(T** p, int64_t count) {
    if (cudaMalloc((void**)p, (size_t)std::max<int64_t>(count, 1) * sizeof(T)) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return false;
    }
    return true;
}

__global__ void k_fill_padding(float* __restrict__ val, int32_t* __restrict__ col, int64_t lo,
                               int64_t hi) {
    for (int64_t i = lo + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < hi;
         i += (int64_t)gridDim.x * blockDim.x) {
        val[i] = 0.f;
        col[i] = -1;
    }
}

// row_nnz from the CSR row pointer, and each row's capacity
__global__ void k_row_counts(const int32_t* __restrict__ row_ptr, int64_t out_f, int pct,
                             int32_t* __restrict__ row_nnz, int32_t* __restrict__ row_cap) {
    for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < out_f;
         r += (int64_t)gridDim.x * blockDim.x) {
        const int32_t n = row_ptr[r + 1] - row_ptr[r];
        row_nnz[r] = n;
        row_cap[r] = pcsr_capacity(n, pct);
    }
}

// canonical entry k of row r goes to slot row_start[r] + (k - row_ptr[r])
__global__ void k_scatter_live(const float* __restrict__ v, const int32_t* __restrict__ r,
                               const int32_t* __restrict__ c, int64_t n,
                               const int32_t* __restrict__ row_ptr,
                               const int32_t* __restrict__ row_start, float* __restrict__ val,
                               int32_t* __restrict__ col) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int32_t row = r[k];
        const int64_t s = (int64_t)row_start[row] + (k - row_ptr[row]);
        val[s] = v[k];
        col[s] = c[k];
    }
}

// ---- insert -------------------------------------------------------------
__global__ void k_ins_check(const int32_t* __restrict__ rows, const int32_t* __restrict__ cols,
                            int64_t n, int64_t out_f, int64_t in_f, int32_t* __restrict__ demand,
                            uint32_t* __restrict__ keys, uint32_t* __restrict__ idx,
                            int32_t* status) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t r = rows[i], c = cols[i];
        if (r < 0 || r >= out_f || c < 0 || c >= in_f) {
            atomicOr(status, kBadRange);
            keys[i] = 0;
        } else {
            atomicAdd(&demand[r], 1);
            keys[i] = (uint32_t)r;
        }
        idx[i] = (uint32_t)i;
    }
}

// per row: the capacity it moves to (0 if it stays)
__global__ void k_ins_need(const int32_t* __restrict__ demand, const int32_t* __restrict__ row_nnz,
                           const int32_t* __restrict__ row_cap, int64_t out_f, int pct,
                           int32_t* __restrict__ need) {
    for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < out_f;
         r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t want = (int64_t)row_nnz[r] + demand[r];
        need[r] = want > row_cap[r] ? pcsr_capacity(want, pct) : 0;
    }
}

// one warp per row that moves: copy its live slots to the new region, pad
// the rest of the region, turn the old region into padding
__global__ void k_ins_move(const int32_t* __restrict__ need, const int32_t* __restrict__ off,
                           int64_t out_f, int64_t used, int32_t* __restrict__ row_start,
                           const int32_t* __restrict__ row_nnz, int32_t* __restrict__ row_cap,
                           float* __restrict__ val, int32_t* __restrict__ col) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < out_f;
         r += nw) {
        const int32_t nc = need[r];
        if (nc == 0) continue;
        const int64_t src = row_start[r], dst = used + off[r];
        const int32_t n = row_nnz[r], oc = row_cap[r];
        for (int32_t j = lane; j < nc; j += 32) {
            val[dst + j] = j < n ? val[src + j] : 0.f;
            col[dst + j] = j < n ? col[src + j] : -1;
        }
        __syncwarp();
        for (int32_t j = lane; j < oc; j += 32) {
            val[src + j] = 0.f;
            col[src + j] = -1;
        }
        __syncwarp();
        if (lane == 0) {
            row_start[r] = (int32_t)dst;
            row_cap[r] = nc;
        }
    }
}

// sorted position j holds insert i = idx[j]; rows sorted stably, so inserts of
// one row appear in batch order; rank = j - first position of its row
__global__ void k_ins_place(const uint32_t* __restrict__ idx, int64_t n,
                            const int32_t* __restrict__ rows, const int32_t* __restrict__ cols,
                            const float* __restrict__ vals, const int32_t* __restrict__ row_off,
                            const int32_t* __restrict__ row_start,
                            const int32_t* __restrict__ row_nnz, float* __restrict__ val,
                            int32_t* __restrict__ col) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t i = idx[j];
        const int32_t r = rows[i];
        const int64_t s = (int64_t)row_start[r] + row_nnz[r] + (j - row_off[r]);
        val[s] = vals[i];
        col[s] = cols[i];
    }
}

__global__ void k_add_i32(int32_t* __restrict__ a, const int32_t* __restrict__ b, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        a[i] += b[i];
}

// ---- delete -------------------------------------------------------------
__global__ void k_del_find(const int32_t* __restrict__ rows, const int32_t* __restrict__ cols,
                           int64_t n, int64_t out_f, int64_t in_f,
                           const int32_t* __restrict__ row_start,
                           const int32_t* __restrict__ row_nnz, const int32_t* __restrict__ col,
                           int32_t* __restrict__ slot, int32_t* status) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t r = rows[i], c = cols[i];
        slot[i] = -1;
        if (r < 0 || r >= out_f || c < 0 || c >= in_f) {
            atomicOr(status, kBadRange);
            continue;
        }
        const int64_t s0 = row_start[r];
        const int32_t nl = row_nnz[r];
        for (int32_t j = 0; j < nl; ++j)
            if (col[s0 + j] == c) {
                slot[i] = (int32_t)(s0 + j);
                break;
            }
        if (slot[i] < 0) atomicOr(status, kNotLive);
    }
}

__global__ void k_del_mark(const int32_t* __restrict__ rows, const int32_t* __restrict__ slot,
                           int64_t n, int32_t* __restrict__ col, int32_t* __restrict__ touched) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        col[slot[i]] = -1;
        touched[rows[i]] = 1;
    }
}

// one warp per touched row: stable in-place compaction of its live slots
__global__ void k_del_close(const int32_t* __restrict__ touched, int64_t out_f,
                            const int32_t* __restrict__ row_start, int32_t* __restrict__ row_nnz,
                            float* __restrict__ val, int32_t* __restrict__ col) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < out_f;
         r += nw) {
        if (!touched[r]) continue;
        const int64_t s0 = row_start[r];
        const int32_t n = row_nnz[r];
        int32_t w = 0;
        for (int32_t base = 0; base < n; base += 32) {
            const int32_t j = base + lane;
            const int32_t cj = j < n ? col[s0 + j] : -1;
            const float vj = j < n ? val[s0 + j] : 0.f;
            const bool live = cj != -1;
            const unsigned m = __ballot_sync(0xffffffffu, live);
            __syncwarp();
            if (live) {
                const int32_t d = w + __popc(m & ((1u << lane) - 1u));
                col[s0 + d] = cj;
                val[s0 + d] = vj;
            }
            w += __popc(m);
            __syncwarp();
        }
        for (int32_t j = w + lane; j < n; j += 32) {
            col[s0 + j] = -1;
            val[s0 + j] = 0.f;
        }
        __syncwarp();
        if (lane == 0) row_nnz[r] = w;
    }
}

// ---- compact_all ----------------------------------------------------------
// live slot j of row r -> key (r * in + col), value bits, at off[r] + j
__global__ void k_live_keys(int64_t out_f, int64_t in_f, const int32_t* __restrict__ row_start,
                            const int32_t* __restrict__ row_nnz, const int32_t* __restrict__ off,
                            const float* __restrict__ val, const int32_t* __restrict__ col,
                            uint64_t* __restrict__ keys, uint32_t* __restrict__ bits) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < out_f;
         r += nw) {
        const int64_t s0 = row_start[r], o = off[r];
        for (int32_t j = lane; j < row_nnz[r]; j += 32) {
            keys[o + j] = (uint64_t)r * (uint64_t)in_f + (uint64_t)col[s0 + j];
            bits[o + j] = __float_as_uint(val[s0 + j]);
        }
    }
}

__global__ void k_check_sorted_unique(const uint64_t* __restrict__ keys, int64_t n, int32_t* status) {
    for (int64_t i = 1 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        if (keys[i] == keys[i - 1]) atomicOr(status, kDup);
}

// sorted entry j (row r) -> slot row_start[r] + (j - off[r])
__global__ void k_place_sorted(const uint64_t* __restrict__ keys, const uint32_t* __restrict__ bits,
                               int64_t n, int64_t in_f, const int32_t* __restrict__ off,
                               const int32_t* __restrict__ row_start, float* __restrict__ val,
                               int32_t* __restrict__ col) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t r = keys[j] / (uint64_t)in_f;
        const int64_t s = (int64_t)row_start[r] + (j - off[r]);
        val[s] = __uint_as_float(bits[j]);
        col[s] = (int32_t)(keys[j] - r * (uint64_t)in_f);
    }
}

__global__ void k_export(const uint64_t* __restrict__ keys, const uint32_t* __restrict__ bits,
                         int64_t n, int64_t in_f, float* __restrict__ v, int32_t* __restrict__ r,
                         int32_t* __restrict__ c) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t rr = keys[j] / (uint64_t)in_f;
        v[j] = __uint_as_float(bits[j]);
        r[j] = (int32_t)rr;
        c[j] = (int32_t)(keys[j] - rr * (uint64_t)in_f);
    }
}

__global__ void k_capacities(const int32_t* __restrict__ row_nnz, int64_t out_f, int pct,
                             int32_t* __restrict__ row_cap) {
    for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < out_f;
         r += (int64_t)gridDim.x * blockDim.x)
        row_cap[r] = pcsr_capacity(row_nnz[r], pct);
}

// ---- host helpers -----------------------------------------------------------
int read_i32(const int32_t* d, int32_t* h, cudaStream_t s) {
    if (cudaMemcpyAsync(h, d, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SNK_ERR_CUDA;
    return SNK_OK;
}

// Make room for `slots` slots (keeping [0, used)).
int ensure_slots(PcsrState* P, int64_t slots, cudaStream_t s) {
    if (slots <= P->alloc) return SNK_OK;
    if (slots > INT32_MAX) return SNK_ERR_LIMIT;
    const int64_t na = std::min<int64_t>(INT32_MAX, std::max<int64_t>(2 * P->alloc, slots + 1024));
    float* nv = nullptr;
    int32_t* nc = nullptr;
    if (!dalloc(&nv, na) || !dalloc(&nc, na)) {
        if (nv) cudaFree(nv);
        return SNK_ERR_OOM;
    }
    if (P->used > 0 &&
        (cudaMemcpyAsync(nv, P->val, P->used * sizeof(float), cudaMemcpyDeviceToDevice, s) !=
             cudaSuccess ||
         cudaMemcpyAsync(nc, P->col, P->used * sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
             cudaSuccess)) {
        cudaFree(nv);
        cudaFree(nc);
        return SNK_ERR_CUDA;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return SNK_ERR_CUDA;
    cudaFree(P->val);
    cudaFree(P->col);
    P->val = nv;
    P->col = nc;
    P->alloc = na;
    return SNK_OK;
}

int ensure_batch(PcsrState* P, int64_t n) {
    if (n <= P->bcap) return SNK_OK;
    cudaFree(P->bkeys);
    cudaFree(P->bvals);
    cudaFree(P->bslot);
    cudaFree(P->hist);
    P->bkeys = nullptr;
    P->bvals = nullptr;
    P->bslot = nullptr;
    P->hist = nullptr;
    P->bcap = 0;
    const int64_t cap = std::max<int64_t>(n, 1024);
    P->hist_len = topology_hist_len(cap);
    uint64_t* k = nullptr;
    if (!dalloc(&k, 2 * cap) || !dalloc(&P->bvals, 2 * cap) || !dalloc(&P->bslot, cap) ||
        !dalloc(&P->hist, P->hist_len)) {
        if (k) cudaFree(k);
        return SNK_ERR_OOM;
    }
    P->bkeys = k;
    P->bcap = cap;
    return SNK_OK;
}

int bits_for(uint64_t n_values) {
    int b = 0;
    while (b < 64 && (n_values - 1) >> b) ++b;
    return b;
}

// The live entries sorted canonically into (keys, bits) of the batch scratch
// (returned pointers); n_live via *n.  status gets kDup for a repeated position.
int sorted_live(Layer* L, PcsrState* P, uint64_t** keys_out, uint32_t** bits_out, int64_t* n,
                cudaStream_t s) {
    const int64_t out_f = L->out_f;
    int32_t live = 0;
    if (exclusive_scan_i32(P->row_nnz, P->roff, out_f, P->scan_tmp, P->scan_tmp_len, P->total, s) !=
            SNK_OK ||
        read_i32(P->total, &live, s) != SNK_OK)
        return SNK_ERR_CUDA;
    int st = ensure_batch(P, live);
    if (st != SNK_OK) return st;
    uint64_t* keys = static_cast<uint64_t*>(P->bkeys);
    k_live_keys<<<grid_of(out_f * 32, L->num_sms), 256, 0, s>>>(out_f, L->in_f, P->row_start,
                                                                P->row_nnz, P->roff, P->val, P->col,
                                                                keys, P->bvals);
    bool flipped = false;
    st = sort_pairs_u64(keys, P->bvals, keys + P->bcap, P->bvals + P->bcap, live,
                        bits_for((uint64_t)out_f * (uint64_t)L->in_f), P->hist, P->hist_len, s,
                        &flipped);
    if (st != SNK_OK) return st;
    *keys_out = flipped ? keys + P->bcap : keys;
    *bits_out = flipped ? P->bvals + P->bcap : P->bvals;
    *n = live;
    return SNK_OK;
}

// Lay the rows out again from slot 0 with fresh padding (the sorted live
// entries are in keys/bits; P->roff holds each row's offset among them).
int relayout(Layer* L, PcsrState* P, const uint64_t* keys, const uint32_t* bits, int64_t live,
             cudaStream_t s) {
    const int64_t out_f = L->out_f;
    k_capacities<<<grid_of(out_f, L->num_sms), 256, 0, s>>>(P->row_nnz, out_f, P->pct, P->row_cap);
    int32_t used = 0;
    if (exclusive_scan_i32(P->row_cap, P->row_start, out_f, P->scan_tmp, P->scan_tmp_len, P->total,
                           s) != SNK_OK ||
        read_i32(P->total, &used, s) != SNK_OK)
        return SNK_ERR_CUDA;
    // the sorted copy lives in the batch scratch, so the slot arrays can be
    // rewritten in place
    int st = ensure_slots(P, used, s);
    if (st != SNK_OK) return st;
    k_fill_padding<<<grid_of(used, L->num_sms), 256, 0, s>>>(P->val, P->col, 0, used);
    k_place_sorted<<<grid_of(live, L->num_sms), 256, 0, s>>>(keys, bits, live, L->in_f, P->roff,
                                                             P->row_start, P->val, P->col);
    P->used = used;
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

}  // namespace

void free_pcsr(Layer* L) {
    PcsrState* P = L->pcsr;
    if (!P) return;
    void* ptrs[] = {P->val, P->col, P->row_start, P->row_nnz, P->row_cap, P->rtmp, P->roff,
                    P->rneed, P->rmove, P->scan_tmp, P->total, P->status, P->bkeys, P->bvals, P->bslot, P->hist};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    delete P;
    L->pcsr = nullptr;
}

}  // namespace snk

using namespace snk;

extern "C" int snk_pcsr_build(snk_handle h, int padding_pct, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || padding_pct < 0 || padding_pct > 10000) return SNK_ERR_ARG;
    // the slot count (live entries, padding and room to move rows) must fit int32
    if ((double)L->nnz * (100.0 + padding_pct) / 100.0 * 2.0 + 4.0 * (double)L->out_f + 2048.0 >
        (double)INT32_MAX)
        return SNK_ERR_LIMIT;
    cudaStream_t s = (cudaStream_t)stream;
    free_pcsr(L);
    PcsrState* P = new PcsrState();
    L->pcsr = P;
    P->pct = padding_pct;
    const int64_t out_f = L->out_f;
    P->scan_tmp_len = scan_tmp_len(out_f + 1);
    if (!dalloc(&P->row_start, out_f) || !dalloc(&P->row_nnz, out_f) || !dalloc(&P->row_cap, out_f) ||
        !dalloc(&P->rtmp, out_f + 1) || !dalloc(&P->roff, out_f + 1) ||
        !dalloc(&P->rneed, out_f + 1) || !dalloc(&P->rmove, out_f + 1) ||
        !dalloc(&P->scan_tmp, P->scan_tmp_len) || !dalloc(&P->total, 1) || !dalloc(&P->status, 1)) {
        free_pcsr(L);
        return SNK_ERR_OOM;
    }
    k_row_counts<<<grid_of(out_f, L->num_sms), 256, 0, s>>>(L->row_ptr, out_f, P->pct, P->row_nnz,
                                                            P->row_cap);
    int32_t used = 0;
    if (exclusive_scan_i32(P->row_cap, P->row_start, out_f, P->scan_tmp, P->scan_tmp_len, P->total,
                           s) != SNK_OK ||
        read_i32(P->total, &used, s) != SNK_OK) {
        free_pcsr(L);
        return SNK_ERR_CUDA;
    }
    int st = ensure_slots(P, 2 * (int64_t)used + 1024, s);
    if (st != SNK_OK) {
        free_pcsr(L);
        return st;
    }
    k_fill_padding<<<grid_of(used, L->num_sms), 256, 0, s>>>(P->val, P->col, 0, used);
    if (L->nnz > 0)
        k_scatter_live<<<grid_of(L->nnz, L->num_sms), 256, 0, s>>>(L->v, L->r, L->c, L->nnz,
                                                                   L->row_ptr, P->row_start, P->val,
                                                                   P->col);
    P->used = used;
    P->version = 1;
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        free_pcsr(L);
        return SNK_ERR_CUDA;
    }
    return SNK_OK;
}

extern "C" int snk_pcsr_info(snk_handle h, int64_t* used_slots, int64_t* n_live,
                             int64_t* version, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || !L->pcsr) return SNK_ERR_ARG;
    PcsrState* P = L->pcsr;
    cudaStream_t s = (cudaStream_t)stream;
    if (used_slots) *used_slots = P->used;
    if (version) *version = P->version;
    if (n_live) {
        int32_t live = 0;
        if (exclusive_scan_i32(P->row_nnz, P->roff, L->out_f, P->scan_tmp, P->scan_tmp_len,
                               P->total, s) != SNK_OK ||
            read_i32(P->total, &live, s) != SNK_OK)
            return SNK_ERR_CUDA;
        *n_live = live;
    }
    return SNK_OK;
}

extern "C" int snk_pcsr_copy(snk_handle h, float* slot_values, int32_t* slot_cols,
                             int32_t* row_start, int32_t* row_nnz, int32_t* row_capacity,
                             void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || !L->pcsr) return SNK_ERR_ARG;
    PcsrState* P = L->pcsr;
    cudaStream_t s = (cudaStream_t)stream;
    const auto d2d = cudaMemcpyDeviceToDevice;
    const size_t rb = (size_t)L->out_f * sizeof(int32_t);
    if ((slot_values && cudaMemcpyAsync(slot_values, P->val, P->used * sizeof(float), d2d, s)) ||
        (slot_cols && cudaMemcpyAsync(slot_cols, P->col, P->used * sizeof(int32_t), d2d, s)) ||
        (row_start && cudaMemcpyAsync(row_start, P->row_start, rb, d2d, s)) ||
        (row_nnz && cudaMemcpyAsync(row_nnz, P->row_nnz, rb, d2d, s)) ||
        (row_capacity && cudaMemcpyAsync(row_capacity, P->row_cap, rb, d2d, s)))
        return SNK_ERR_CUDA;
    return SNK_OK;
}

extern "C" int snk_pcsr_insert(snk_handle h, int64_t n, const int32_t* rows, const int32_t* cols,
                               const float* values, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || !L->pcsr || n < 0 || n > INT32_MAX) return SNK_ERR_ARG;
    if (n == 0) return SNK_OK;
    if (!rows || !cols || !values) return SNK_ERR_ARG;
    PcsrState* P = L->pcsr;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t out_f = L->out_f;
    int st = ensure_batch(P, n);
    if (st != SNK_OK) return st;
    uint32_t* keys = reinterpret_cast<uint32_t*>(P->bkeys);  // n row keys, then their alternate
    uint32_t* keys_alt = keys + P->bcap;
    cudaMemsetAsync(P->rtmp, 0, (out_f + 1) * sizeof(int32_t), s);
    cudaMemsetAsync(P->status, 0, sizeof(int32_t), s);
    k_ins_check<<<grid_of(n, L->num_sms), 256, 0, s>>>(rows, cols, n, out_f, L->in_f, P->rtmp, keys,
                                                       P->bvals, P->status);
    int32_t bad = 0;
    if (read_i32(P->status, &bad, s) != SNK_OK) return SNK_ERR_CUDA;
    if (bad) return SNK_ERR_RANGE;
    // stable sort of the batch by row: inserts of a row keep batch order
    bool flipped = false;
    st = sort_pairs_u32(keys, P->bvals, keys_alt, P->bvals + P->bcap, n, bits_for((uint64_t)out_f),
                        P->hist, P->hist_len, s, &flipped);
    if (st != SNK_OK) return st;
    const uint32_t* idx = flipped ? P->bvals + P->bcap : P->bvals;
    // first sorted position of each row's inserts
    if (exclusive_scan_i32(P->rtmp, P->roff, out_f, P->scan_tmp, P->scan_tmp_len, P->total, s) !=
        SNK_OK)
        return SNK_ERR_CUDA;
    // rows that must move, and the offsets of their new regions
    k_ins_need<<<grid_of(out_f, L->num_sms), 256, 0, s>>>(P->rtmp, P->row_nnz, P->row_cap, out_f,
                                                          P->pct, P->rneed);
    int32_t moved = 0;
    if (exclusive_scan_i32(P->rneed, P->rmove, out_f, P->scan_tmp, P->scan_tmp_len, P->total, s) !=
            SNK_OK ||
        read_i32(P->total, &moved, s) != SNK_OK)
        return SNK_ERR_CUDA;
    if (moved > 0) {
        st = ensure_slots(P, P->used + moved, s);
        if (st != SNK_OK) return st;
        k_ins_move<<<grid_of(out_f * 32, L->num_sms), 256, 0, s>>>(P->rneed, P->rmove, out_f,
                                                                   P->used, P->row_start,
                                                                   P->row_nnz, P->row_cap, P->val,
                                                                   P->col);
        P->used += moved;
    }
    k_ins_place<<<grid_of(n, L->num_sms), 256, 0, s>>>(idx, n, rows, cols, values, P->roff,
                                                       P->row_start, P->row_nnz, P->val, P->col);
    k_add_i32<<<grid_of(out_f, L->num_sms), 256, 0, s>>>(P->row_nnz, P->rtmp, out_f);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return SNK_ERR_CUDA;
    P->version += 1;
    return SNK_OK;
}

extern "C" int snk_pcsr_delete(snk_handle h, int64_t n, const int32_t* rows, const int32_t* cols,
                               void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || !L->pcsr || n < 0 || n > INT32_MAX) return SNK_ERR_ARG;
    if (n == 0) return SNK_OK;
    if (!rows || !cols) return SNK_ERR_ARG;
    PcsrState* P = L->pcsr;
    cudaStream_t s = (cudaStream_t)stream;
    int st = ensure_batch(P, n);
    if (st != SNK_OK) return st;
    cudaMemsetAsync(P->status, 0, sizeof(int32_t), s);
    k_del_find<<<grid_of(n, L->num_sms), 256, 0, s>>>(rows, cols, n, L->out_f, L->in_f,
                                                      P->row_start, P->row_nnz, P->col, P->bslot,
                                                      P->status);
    int32_t bad = 0;
    if (read_i32(P->status, &bad, s) != SNK_OK) return SNK_ERR_CUDA;
    if (bad & kBadRange) return SNK_ERR_RANGE;
    if (bad & kNotLive) return SNK_ERR_ARG;
    cudaMemsetAsync(P->rtmp, 0, (L->out_f + 1) * sizeof(int32_t), s);
    k_del_mark<<<grid_of(n, L->num_sms), 256, 0, s>>>(rows, P->bslot, n, P->col, P->rtmp);
    k_del_close<<<grid_of(L->out_f * 32, L->num_sms), 256, 0, s>>>(P->rtmp, L->out_f, P->row_start,
                                                                   P->row_nnz, P->val, P->col);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return SNK_ERR_CUDA;
    P->version += 1;
    return SNK_OK;
}

extern "C" int snk_pcsr_compact(snk_handle h, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || !L->pcsr) return SNK_ERR_ARG;
    PcsrState* P = L->pcsr;
    cudaStream_t s = (cudaStream_t)stream;
    uint64_t* keys = nullptr;
    uint32_t* bits = nullptr;
    int64_t live = 0;
    cudaMemsetAsync(P->status, 0, sizeof(int32_t), s);
    int st = sorted_live(L, P, &keys, &bits, &live, s);
    if (st != SNK_OK) return st;
    k_check_sorted_unique<<<grid_of(live, L->num_sms), 256, 0, s>>>(keys, live, P->status);
    int32_t bad = 0;
    if (read_i32(P->status, &bad, s) != SNK_OK) return SNK_ERR_CUDA;
    if (bad) return SNK_ERR_DUP;
    st = relayout(L, P, keys, bits, live, s);
    if (st != SNK_OK) return st;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SNK_ERR_CUDA;
    P->version += 1;
    return SNK_OK;
}

extern "C" int snk_pcsr_export(snk_handle h, float* values, int32_t* rows, int32_t* cols,
                               int64_t capacity, int64_t* nnz_out, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || !L->pcsr || !nnz_out || capacity < 0) return SNK_ERR_ARG;
    PcsrState* P = L->pcsr;
    cudaStream_t s = (cudaStream_t)stream;
    uint64_t* keys = nullptr;
    uint32_t* bits = nullptr;
    int64_t live = 0;
    cudaMemsetAsync(P->status, 0, sizeof(int32_t), s);
    int st = sorted_live(L, P, &keys, &bits, &live, s);
    if (st != SNK_OK) return st;
    *nnz_out = live;
    if (live > capacity) return SNK_ERR_LIMIT;
    if (live > 0 && (!values || !rows || !cols)) return SNK_ERR_ARG;
    k_check_sorted_unique<<<grid_of(live, L->num_sms), 256, 0, s>>>(keys, live, P->status);
    int32_t bad = 0;
    if (read_i32(P->status, &bad, s) != SNK_OK) return SNK_ERR_CUDA;
    if (bad) return SNK_ERR_DUP;
    if (live > 0)
        k_export<<<grid_of(live, L->num_sms), 256, 0, s>>>(keys, bits, live, L->in_f, values, rows,
                                                           cols);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return SNK_ERR_CUDA;
    return SNK_OK;
}
