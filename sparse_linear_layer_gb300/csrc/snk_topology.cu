// Topology build: validate the COO triple, sort it into canonical (row, col)
// order, and derive the CSR row pointer, the column-sorted view (col_ptr,
// rows_c, perm) and the merge-path chunk tables.
//
//   "Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
//     sec. 3.2 (sort by row, row pointer), sec. 4.1 (CSR, columns sorted
//     within a row), sec. 7.2 (transpose = per-column count + scatter, kept
//     as a permutation map and rebuilt only when the topology changes).
//   "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
//     GPU", Table 7 (COO, CSR and CSC of the same matrix).
//
// GB300 mapping: both orders come from a stable LSD radix sort (8-bit digits,
// 4096-key tiles, warp-level ranking with __match_any_sync), which replaces
// the pages' host-side argsort.  Keys are row*in + col, so only
// ceil(log2(out*in)) bits are sorted; the column view is a stable sort of the
// canonical order by column (ceil(log2(in)) bits), which leaves rows
// ascending within a column.
#include <algorithm>

#include "snk_internal.cuh"

namespace snk {

// ------------------------------------------------------------------ scan
constexpr int kScanThreads = 512;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int x, int* sm, int* block_total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm[w] = incl;
    __syncthreads();
    if (w == 0) {
        int t = (lane < NT / 32) ? sm[lane] : 0;
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += y;
        }
        if (lane < NT / 32) sm[lane] = ti - t;
        if (lane == NT / 32 - 1) sm[NT / 32] = ti;
    }
    __syncthreads();
    int res = sm[w] + incl - x;
    if (block_total) *block_total = sm[NT / 32];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(kScanThreads) k_tile_sums(const int32_t* in, int64_t n,
                                                            int32_t* sums) {
    __shared__ int sm[kScanThreads / 32 + 1];
    int64_t base = (int64_t)blockIdx.x * kScanTile;
    int acc = 0;
    for (int i = threadIdx.x; i < kScanTile; i += kScanThreads) {
        int64_t k = base + i;
        if (k < n) acc += in[k];
    }
    int tot;
    block_exclusive_scan<kScanThreads>(acc, sm, &tot);
    if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(1024) k_scan_sums(int32_t* sums, int64_t nt, int32_t* total) {
    __shared__ int sm[1024 / 32 + 1];
    int carry = 0;
    for (int64_t base = 0; base < nt; base += 1024) {
        int64_t k = base + threadIdx.x;
        int x = (k < nt) ? sums[k] : 0;
        int tot;
        int ex = block_exclusive_scan<1024>(x, sm, &tot);
        if (k < nt) sums[k] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0 && total) *total = carry;
}

__global__ void __launch_bounds__(kScanThreads) k_tile_scan(const int32_t* in, int32_t* out,
                                                            int64_t n, const int32_t* sums) {
    __shared__ int sm[kScanThreads / 32 + 1];
    int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
    int x[kScanItems];
    int acc = 0;
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
        int64_t k = base + j;
        x[j] = (k < n) ? in[k] : 0;
        acc += x[j];
    }
    int ex = block_exclusive_scan<kScanThreads>(acc, sm, nullptr) + sums[blockIdx.x];
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
        int64_t k = base + j;
        if (k < n) out[k] = ex;
        ex += x[j];
    }
}

int64_t scan_tmp_len(int64_t n) { return std::max<int64_t>(1, ceil_div(n, kScanTile)); }

// out[i] = sum_{j<i} in[j]; in == out allowed; *total (device) = sum of all.
int exclusive_scan_i32(const int32_t* in, int32_t* out, int64_t n, int32_t* tmp, int64_t tmp_len,
                       int32_t* total, cudaStream_t s) {
    int64_t nt = ceil_div(n, kScanTile);
    if (nt > tmp_len) return SNK_ERR_ARG;
    if (n == 0) {
        if (total) cudaMemsetAsync(total, 0, sizeof(int32_t), s);
        return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
    }
    k_tile_sums<<<(unsigned)nt, kScanThreads, 0, s>>>(in, n, tmp);
    k_scan_sums<<<1, 1024, 0, s>>>(tmp, nt, total);
    k_tile_scan<<<(unsigned)nt, kScanThreads, 0, s>>>(in, out, n, tmp);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

// ------------------------------------------------------------------ radix sort
constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortRounds = 16;
constexpr int kSortTile = kSortThreads * kSortRounds;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <typename K>
__global__ void __launch_bounds__(kSortThreads) k_radix_hist(const K* __restrict__ keys, int64_t n,
                                                             int shift, int nbits,
                                                             int32_t* __restrict__ hist,
                                                             int64_t n_tiles) {
    __shared__ int h[256];
    for (int i = threadIdx.x; i < 256; i += kSortThreads) h[i] = 0;
    __syncthreads();
    const unsigned mask = (1u << nbits) - 1u;
    int64_t base = (int64_t)blockIdx.x * kSortTile;
    for (int i = threadIdx.x; i < kSortTile; i += kSortThreads) {
        int64_t k = base + i;
        if (k < n) atomicAdd(&h[(unsigned)(keys[k] >> shift) & mask], 1);
    }
    __syncthreads();
    for (int d = threadIdx.x; d < (1 << nbits); d += kSortThreads)
        hist[(int64_t)d * n_tiles + blockIdx.x] = h[d];
}

// Stable scatter of one 2^nbits-way digit pass.  Within a tile, warp w owns a
// contiguous run of kSortRounds*32 keys and walks it 32 at a time; equal
// digits in a round are ranked by lane with __match_any_sync, and a per-warp
// counter per digit carries the rank across rounds.  offs holds the
// exclusive prefix over (digit, tile) in digit-major order.
template <typename K>
__global__ void __launch_bounds__(kSortThreads) k_radix_scatter(
    const K* __restrict__ keys, const uint32_t* __restrict__ vals, K* __restrict__ keys_out,
    uint32_t* __restrict__ vals_out, int64_t n, int shift, int nbits,
    const int32_t* __restrict__ offs, int64_t n_tiles) {
    __shared__ int wcnt[kSortWarps][256];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int i = lane; i < 256; i += 32) wcnt[w][i] = 0;
    __syncwarp();
    const unsigned mask = (1u << nbits) - 1u;
    const unsigned lt = lanemask_lt();
    int64_t wbase = (int64_t)blockIdx.x * kSortTile + (int64_t)w * 32 * kSortRounds;
    K kk[kSortRounds];
    uint32_t vv[kSortRounds];
    int dig[kSortRounds];
    int rnk[kSortRounds];
#pragma unroll
    for (int i = 0; i < kSortRounds; ++i) {
        int64_t k = wbase + i * 32 + lane;
        bool ok = k < n;
        K key = ok ? keys[k] : (K)0;
        uint32_t val = ok ? vals[k] : 0u;
        int d = ok ? (int)((unsigned)(key >> shift) & mask) : -1;
        unsigned peers = __match_any_sync(0xffffffffu, d);
        int pre = ok ? wcnt[w][d] : 0;
        int r = __popc(peers & lt);
        __syncwarp();
        if (ok && r == 0) wcnt[w][d] = pre + __popc(peers);
        __syncwarp();
        kk[i] = key;
        vv[i] = val;
        dig[i] = d;
        rnk[i] = pre + r;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < 256; d += kSortThreads) {
        int run = 0;
#pragma unroll
        for (int w2 = 0; w2 < kSortWarps; ++w2) {
            int t = wcnt[w2][d];
            wcnt[w2][d] = run;
            run += t;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kSortRounds; ++i) {
        if (dig[i] >= 0) {
            int64_t pos = (int64_t)offs[(int64_t)dig[i] * n_tiles + blockIdx.x] + wcnt[w][dig[i]] +
                          rnk[i];
            keys_out[pos] = kk[i];
            vals_out[pos] = vv[i];
        }
    }
}

static int64_t sort_tiles(int64_t n) { return std::max<int64_t>(1, ceil_div(n, kSortTile)); }

// Histogram + scan scratch needed to sort n keys.
int64_t topology_hist_len(int64_t n) {
    const int64_t nt = sort_tiles(n);
    return 256 * nt + scan_tmp_len(256 * nt);
}

// Sorts (keys, vals) by the low `total_bits` bits of keys, stably.  The
// result lands in either the primary or the alternate buffers; *flipped says
// which (true = alternate).
template <typename K>
static int radix_sort_pairs(K* keys, uint32_t* vals, K* keys_alt, uint32_t* vals_alt, int64_t n,
                            int total_bits, int32_t* hist, int64_t hist_len, cudaStream_t s,
                            bool* flipped) {
    *flipped = false;
    if (n <= 1 || total_bits <= 0) return SNK_OK;
    int64_t nt = sort_tiles(n);
    if (256 * nt + scan_tmp_len(256 * nt) > hist_len) return SNK_ERR_ARG;
    int32_t* scan_tmp = hist + 256 * nt;
    K *ka = keys, *kb = keys_alt;
    uint32_t *va = vals, *vb = vals_alt;
    for (int shift = 0; shift < total_bits; shift += 8) {
        int nbits = std::min(8, total_bits - shift);
        k_radix_hist<K><<<(unsigned)nt, kSortThreads, 0, s>>>(ka, n, shift, nbits, hist, nt);
        int st = exclusive_scan_i32(hist, hist, (int64_t)(1 << nbits) * nt, scan_tmp,
                                    scan_tmp_len(256 * nt), nullptr, s);
        if (st != SNK_OK) return st;
        k_radix_scatter<K><<<(unsigned)nt, kSortThreads, 0, s>>>(ka, va, kb, vb, n, shift, nbits,
                                                                 hist, nt);
        std::swap(ka, kb);
        std::swap(va, vb);
        *flipped = !*flipped;
    }
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

int sort_pairs_u64(uint64_t* keys, uint32_t* vals, uint64_t* keys_alt, uint32_t* vals_alt, int64_t n,
                   int total_bits, int32_t* hist, int64_t hist_len, cudaStream_t s, bool* flipped) {
    return radix_sort_pairs<uint64_t>(keys, vals, keys_alt, vals_alt, n, total_bits, hist,
                                      hist_len, s, flipped);
}
int sort_pairs_u32(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt, int64_t n,
                   int total_bits, int32_t* hist, int64_t hist_len, cudaStream_t s, bool* flipped) {
    return radix_sort_pairs<uint32_t>(keys, vals, keys_alt, vals_alt, n, total_bits, hist,
                                      hist_len, s, flipped);
}

// ------------------------------------------------------------------ topology kernels
static int bits_for(uint64_t n_values) {
    // number of bits needed to represent 0 .. n_values-1
    int b = 0;
    while (b < 64 && (n_values - 1) >> b) ++b;
    return b;
}

template <typename K>
__global__ void k_make_lin(const float* __restrict__ v, const int32_t* __restrict__ r,
                           const int32_t* __restrict__ c, int64_t n, int64_t out_f, int64_t in_f,
                           K* __restrict__ keys, uint32_t* __restrict__ vals,
                           int32_t* __restrict__ status) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        int32_t rr = r[k], cc = c[k];
        bool bad = rr < 0 || rr >= out_f || cc < 0 || cc >= in_f;
        if (bad) {
            atomicOr(status, kStatRange);
            rr = 0;
            cc = 0;
        }
        keys[k] = (K)((uint64_t)rr * (uint64_t)in_f + (uint64_t)cc);
        vals[k] = __float_as_uint(v[k]);
    }
}

template <typename K>
__global__ void k_check_dup(const K* __restrict__ keys, int64_t n, int32_t* __restrict__ status) {
    for (int64_t k = 1 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        if (keys[k] == keys[k - 1]) atomicOr(status, kStatDup);
    }
}

template <typename K>
__global__ void k_unpack(const K* __restrict__ keys, const uint32_t* __restrict__ vals, int64_t n,
                         int64_t in_f, float* __restrict__ v, int32_t* __restrict__ r,
                         int32_t* __restrict__ c, uint32_t* __restrict__ col_key,
                         uint32_t* __restrict__ col_val) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        uint64_t lin = (uint64_t)keys[k];
        int32_t rr = (int32_t)(lin / (uint64_t)in_f);
        int32_t cc = (int32_t)(lin - (uint64_t)rr * (uint64_t)in_f);
        v[k] = __uint_as_float(vals[k]);
        r[k] = rr;
        c[k] = cc;
        col_key[k] = (uint32_t)cc;
        col_val[k] = (uint32_t)k;
    }
}

// ptr[j] = number of entries whose index is < j, for j in [0, n_seg], given
// the indices in ascending order.
__global__ void k_fill_ptr(const int32_t* __restrict__ idx, int64_t n, int64_t n_seg,
                           int32_t* __restrict__ ptr) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k <= n;
         k += (int64_t)gridDim.x * blockDim.x) {
        int64_t prev = (k == 0) ? -1 : (int64_t)idx[k - 1];
        int64_t cur = (k == n) ? n_seg : (int64_t)idx[k];
        for (int64_t j = prev + 1; j <= cur; ++j) ptr[j] = (int32_t)k;
    }
}

__global__ void k_fill_ptr_u32(const uint32_t* __restrict__ idx, int64_t n, int64_t n_seg,
                               int32_t* __restrict__ ptr) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k <= n;
         k += (int64_t)gridDim.x * blockDim.x) {
        int64_t prev = (k == 0) ? -1 : (int64_t)idx[k - 1];
        int64_t cur = (k == n) ? n_seg : (int64_t)idx[k];
        for (int64_t j = prev + 1; j <= cur; ++j) ptr[j] = (int32_t)k;
    }
}

__global__ void k_gather_rows(const uint32_t* __restrict__ perm_u, const int32_t* __restrict__ r,
                              int64_t n, int32_t* __restrict__ perm, int32_t* __restrict__ rows_c) {
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
         j += (int64_t)gridDim.x * blockDim.x) {
        uint32_t p = perm_u[j];
        perm[j] = (int32_t)p;
        rows_c[j] = r[p];
    }
}

// 16-bit copy of an index stream, zero-padded to n_pad entries.
__global__ void k_narrow16(const int32_t* __restrict__ src, int64_t n, int64_t n_pad,
                           uint16_t* __restrict__ dst) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n_pad;
         k += (int64_t)gridDim.x * blockDim.x)
        dst[k] = k < n ? (uint16_t)src[k] : (uint16_t)0;
}

// ---- work partition -----------------------------------------------------
__device__ __forceinline__ int64_t lower_bound_ptr(const int32_t* ptr, int64_t n, int64_t t) {
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)ptr[mid] < t) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}
// largest i with a[i] <= t (a non-decreasing, a[0] <= t)
__device__ __forceinline__ int64_t last_le(const int32_t* a, int64_t n, int64_t t) {
    int64_t lo = 0, hi = n;  // first index with a[i] > t
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)a[mid] <= t) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

// Block boundaries: the even split point c*nnz/n_blocks (rounded down to a
// multiple of 4), moved to the nearer boundary of the segment it falls in,
// unless that segment is longer than half a block's share (then it is cut).
__global__ void k_block_bounds(const int32_t* __restrict__ ptr, int64_t n_seg, int64_t nnz,
                               int n_blocks, int32_t* __restrict__ bnd) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c > n_blocks) return;
    if (c == 0 || c == n_blocks) {
        bnd[c] = c == 0 ? 0 : (int32_t)nnz;
        return;
    }
    const int64_t t = ((int64_t)c * nnz / n_blocks) & ~(int64_t)3;
    int64_t r = last_le(ptr, n_seg + 1, t);
    if (r > n_seg - 1) r = n_seg - 1;
    const int64_t lo = ptr[r], hi = ptr[r + 1];
    const int64_t share = nnz / n_blocks;
    int64_t k;
    if (hi - lo > share / 2) k = t;
    else k = (t - lo <= hi - t) ? lo : hi;
    bnd[c] = (int32_t)k;
}

// Chunk q = (block c, warp w): an equal share of the block's range, rounded
// to a multiple of 4 entries; (k0, k1, first segment touched, one past the
// last segment it owns).  A chunk owns the segments whose start lies in
// [k0, k1) (the very last chunk also owns the empty segments at the end) and
// continues the segment that runs into it, if it holds any entry.  Thread
// w = 0 of each block also fills the block descriptor.
__global__ void k_chunk_desc(const int32_t* __restrict__ ptr, int64_t n_seg,
                             const int32_t* __restrict__ bnd, int n_blocks, int warps,
                             int4* __restrict__ cdesc, BlockDesc* __restrict__ bdesc) {
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= n_blocks * warps) return;
    const int c = q / warps, w = q % warps;
    const int64_t kc = bnd[c], kn = bnd[c + 1];
    const int64_t len = kn - kc;
    const int64_t sz = len > 0 ? ((len + warps - 1) / warps + 3) / 4 * 4 : 0;
    const int64_t k0 = min(kc + w * sz, kn);
    const int64_t k1 = (w == warps - 1) ? kn : min(kc + (w + 1) * sz, kn);
    const bool last = (q == n_blocks * warps - 1);
    const int64_t lo = lower_bound_ptr(ptr, n_seg, k0);
    const int64_t hi = last ? n_seg : lower_bound_ptr(ptr, n_seg, k1);
    const int64_t first = (k1 > k0 && lo > 0 && (int64_t)ptr[lo] > k0) ? lo - 1 : lo;
    cdesc[q] = make_int4((int)k0, (int)k1, (int)first, (int)hi);
    if (w != 0) return;
    BlockDesc d;
    d.k0 = (int)kc;
    d.k1 = (int)kn;
    d.head_first = c;
    d.tail_last = c;
    d.pad0 = d.pad1 = 0;
    if (kn > kc) {
        const int64_t r = last_le(ptr, n_seg + 1, kc);
        if ((int64_t)ptr[r] < kc) d.head_first = (int)last_le(bnd, n_blocks + 1, ptr[r]);
        const int64_t r2 = last_le(ptr, n_seg + 1, kn - 1);
        if ((int64_t)ptr[r2 + 1] > kn) d.tail_last = (int)last_le(bnd, n_blocks + 1, ptr[r2 + 1] - 1);
    }
    int nh = 0, nt = 0;
    for (int x = d.head_first; x <= c; ++x) nh += bnd[x + 1] > bnd[x];
    for (int x = c; x <= d.tail_last; ++x) nt += bnd[x + 1] > bnd[x];
    d.n_head = nh;
    d.n_tail = nt;
    bdesc[c] = d;
}

int build_partition(const int32_t* ptr, int64_t n_seg, int64_t nnz, int n_blocks, int warps,
                    int32_t* bnd, int4* cdesc, BlockDesc* bdesc, cudaStream_t s) {
    const int T = 256;
    k_block_bounds<<<(unsigned)ceil_div(n_blocks + 1, T), T, 0, s>>>(ptr, n_seg, nnz, n_blocks, bnd);
    const int64_t nq = (int64_t)n_blocks * warps;
    k_chunk_desc<<<(unsigned)ceil_div(nq, T), T, 0, s>>>(ptr, n_seg, bnd, n_blocks, warps, cdesc,
                                                         bdesc);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

static unsigned grid_for(int64_t n, int threads, int num_sms) {
    int64_t g = std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, threads), (int64_t)num_sms * 8));
    return (unsigned)g;
}

int build_topology(Layer* L, cudaStream_t s, bool validate) {
    const int64_t n = L->nnz;
    const int T = 256;
    const int64_t bits_lin = bits_for((uint64_t)L->out_f * (uint64_t)L->in_f);
    cudaMemsetAsync(L->status, 0, sizeof(int32_t), s);

    if (n > 0) {
        bool flipped = false;
        int st;
        if (bits_lin <= 32) {
            uint32_t* ka = (uint32_t*)L->sort_keys;
            uint32_t* kb = ka + n;
            k_make_lin<uint32_t><<<grid_for(n, T, L->num_sms), T, 0, s>>>(
                L->v, L->r, L->c, n, L->out_f, L->in_f, ka, L->sort_vals, L->status);
            st = radix_sort_pairs<uint32_t>(ka, L->sort_vals, kb, L->sort_vals + n, n,
                                            (int)bits_lin, L->tile_hist, L->tile_hist_len, s,
                                            &flipped);
            if (st != SNK_OK) return st;
            uint32_t* ks = flipped ? kb : ka;
            uint32_t* vs = flipped ? L->sort_vals + n : L->sort_vals;
            if (validate) k_check_dup<uint32_t><<<grid_for(n, T, L->num_sms), T, 0, s>>>(ks, n, L->status);
            int32_t h_status = 0;
            cudaMemcpyAsync(&h_status, L->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
            if (cudaStreamSynchronize(s) != cudaSuccess) return SNK_ERR_CUDA;
            if (h_status & kStatRange) return SNK_ERR_RANGE;
            if (h_status & kStatDup) return SNK_ERR_DUP;
            k_unpack<uint32_t><<<grid_for(n, T, L->num_sms), T, 0, s>>>(
                ks, vs, n, L->in_f, L->v, L->r, L->c, L->col_keys, L->col_vals);
        } else {
            uint64_t* ka = (uint64_t*)L->sort_keys;
            uint64_t* kb = ka + n;
            k_make_lin<uint64_t><<<grid_for(n, T, L->num_sms), T, 0, s>>>(
                L->v, L->r, L->c, n, L->out_f, L->in_f, ka, L->sort_vals, L->status);
            st = radix_sort_pairs<uint64_t>(ka, L->sort_vals, kb, L->sort_vals + n, n,
                                            (int)bits_lin, L->tile_hist, L->tile_hist_len, s,
                                            &flipped);
            if (st != SNK_OK) return st;
            uint64_t* ks = flipped ? kb : ka;
            uint32_t* vs = flipped ? L->sort_vals + n : L->sort_vals;
            if (validate) k_check_dup<uint64_t><<<grid_for(n, T, L->num_sms), T, 0, s>>>(ks, n, L->status);
            int32_t h_status = 0;
            cudaMemcpyAsync(&h_status, L->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
            if (cudaStreamSynchronize(s) != cudaSuccess) return SNK_ERR_CUDA;
            if (h_status & kStatRange) return SNK_ERR_RANGE;
            if (h_status & kStatDup) return SNK_ERR_DUP;
            k_unpack<uint64_t><<<grid_for(n, T, L->num_sms), T, 0, s>>>(
                ks, vs, n, L->in_f, L->v, L->r, L->c, L->col_keys, L->col_vals);
        }
    }
    return build_views(L, s);
}

// The derived views of a triple that is already in canonical order, with
// col_keys / col_vals holding (column, canonical slot) of every entry.
int build_views(Layer* L, cudaStream_t s) {
    const int64_t n = L->nnz;
    const int T = 256;
    const int bits_col = bits_for((uint64_t)L->in_f);
    // CSR row pointer from the canonical rows
    k_fill_ptr<<<grid_for(n + 1, T, L->num_sms), T, 0, s>>>(L->r, n, L->out_f, L->row_ptr);

    // column view: stable sort of (col, canonical slot) by col
    if (n > 0) {
        uint32_t* ck = L->col_keys;
        uint32_t* cv = L->col_vals;
        bool flipped = false;
        int st = radix_sort_pairs<uint32_t>(ck, cv, ck + n, cv + n, n, bits_col, L->tile_hist,
                                            L->tile_hist_len, s, &flipped);
        if (st != SNK_OK) return st;
        uint32_t* cks = flipped ? ck + n : ck;
        uint32_t* cvs = flipped ? cv + n : cv;
        k_gather_rows<<<grid_for(n, T, L->num_sms), T, 0, s>>>(cvs, L->r, n, L->perm, L->rows_c);
        k_fill_ptr_u32<<<grid_for(n + 1, T, L->num_sms), T, 0, s>>>(cks, n, L->in_f, L->col_ptr);
    } else {
        k_fill_ptr<<<1, T, 0, s>>>(L->r, 0, L->in_f, L->col_ptr);
    }

    // zero padding after the library-owned streams, and their 16-bit copies
    if (L->nnz_pad > n) {
        cudaMemsetAsync(L->perm + n, 0, (L->nnz_pad - n) * sizeof(int32_t), s);
        cudaMemsetAsync(L->rows_c + n, 0, (L->nnz_pad - n) * sizeof(int32_t), s);
    }
    if (L->c16)
        k_narrow16<<<grid_for(L->nnz_pad, T, L->num_sms), T, 0, s>>>(L->c, n, L->nnz_pad, L->c16);
    if (L->rc16)
        k_narrow16<<<grid_for(L->nnz_pad, T, L->num_sms), T, 0, s>>>(L->rows_c, n, L->nnz_pad,
                                                                     L->rc16);

    if (build_partition(L->row_ptr, L->out_f, n, L->n_blocks, kWarpsPerBlock, L->bnd_r, L->cdesc_r,
                        L->bdesc_r, s) != SNK_OK ||
        build_partition(L->col_ptr, L->in_f, n, L->n_blocks, kWarpsPerBlockDx, L->bnd_c, L->cdesc_c,
                        L->bdesc_c, s) != SNK_OK)
        return SNK_ERR_CUDA;
    if (refresh_tc_views(L, s) != SNK_OK) return SNK_ERR_CUDA;
    if (int st = build_sweep(L, s); st != SNK_OK) return st;
    if (int st = refresh_bands(L, s); st != SNK_OK) return st;
    if (cudaGetLastError() != cudaSuccess) return SNK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SNK_ERR_CUDA;
    L->topology_version += 1;
    mark_tc_views(L);
    mark_sweep(L);
    mark_bands(L);
    return SNK_OK;
}

}  // namespace snk
