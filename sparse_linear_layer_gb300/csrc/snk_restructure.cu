// In-place dynamic-sparse-training restructure: magnitude prune of a fraction
// zeta, then a seeded uniform regrow of as many zero-valued entries; nnz is
// unchanged and the topology is rebuilt.
//
//   "Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
//     sec. 1.1 (prune the smallest-magnitude weights), sec. 4.3 (drop a
//     fraction of the live entries and grow the same number elsewhere),
//     sec. 8.2 (SET with drop_fraction 0.3).
//   "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
//     GPU", Fig. 1 (connections added or dropped in place).
//
// Readings where the pages are silent (the same ones the oracle takes):
//   k = floor((double)zeta * nnz); entries are ranked by (bit pattern of
//   |value|, row*in + col), and the k smallest are removed.  Regrow draws
//   p_t = floor(z_t * N / 2^64), z_t the t-th SplitMix64 output (Steele, Lea
//   & Flood, OOPSLA 2014) from state `seed`, N = out*in (Lemire's
//   multiply-shift, 2019), and accepts p_t when it is neither kept nor
//   accepted before, in draw order, until k are accepted; at most 64 k + 1024
//   draws.  New values are +0.0f.
//
// GB300 mapping
//  * Prune: MSB-first radix select of the k-th smallest key, 8 bits per pass
//    (4 passes over the magnitude bits, then the position bits of the few
//    entries that tie on magnitude), with the selection state kept on the
//    device so the passes queue without host round trips; then a stable
//    compaction (flag, scan, scatter).
//  * Regrow: rounds of B consecutive draws evaluated in parallel.  A draw
//    survives when its position is in neither the kept-or-accepted hash set
//    nor drawn earlier in the round (the smallest t per position is kept
//    with an integer atomicMin in a round-local table); survivors are ranked
//    by t with a scan and the first `need` are accepted.  This picks exactly
//    the positions the sequential definition picks, in the same order, for
//    any B.
//  * Gradient grow (the RigL variant, "grow at high-gradient locations",
//    sec. 4.3 of the Padded-CSR page): the gradient of every candidate
//    position is recomputed on the fly in each pass (one warp per row, the
//    row's kept columns marked in a shared-memory bitmap per 1024-column
//    tile) and never stored; an MSB-first radix select with 12-bit digits
//    over the 64-bit key (complement of the bits of |g|, then the position)
//    finds the k-th smallest key, stopping early when a digit bin holds
//    exactly the remaining count; a last pass collects every candidate at or
//    below it: exactly k positions, since keys are unique.
//  * Write-back: the kept entries come out of the compaction already in
//    canonical order, so only the k grown positions are radix-sorted and the
//    two lists are merged (merge path) straight into the caller's triple in
//    canonical order; only the derived views are rebuilt.
#include <algorithm>

#include "snk_internal.cuh"

namespace snk {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kEmpty = ~0ull;
constexpr int kGradTile = 1024;            // columns per bitmap tile
constexpr int kGradDigit = 12;             // digit width of the select passes
constexpr int kGradBins = 1 << kGradDigit;
constexpr int kGradWarps = 8;              // warps per block of the gradient passes
constexpr int kGradDyMax = 64;             // batch sizes whose dY row is kept in shared memory

struct SelState {
    uint32_t mag;
    uint32_t done;   // 1 once every entry of the selected magnitude is known to go
    uint64_t lin;
    int64_t krem;
};

struct RestructureWs {
    int64_t cap = 0;             // nnz the buffers were sized for
    int32_t* hist = nullptr;     // [256]
    SelState* sel = nullptr;
    int32_t* flags = nullptr;    // [2 * flag_half]: flags, then their exclusive scan
    int64_t flag_half = 0;       // max(cap, cand_cap)
    int32_t* scan_tmp = nullptr;
    int64_t scan_tmp_len = 0;
    int32_t* total = nullptr;    // device scalar
    int64_t* acc = nullptr;      // device scalars: accepted so far, boundary keys
    uint64_t* kept_lin = nullptr;
    uint32_t* kept_val = nullptr;
    uint64_t* H = nullptr;       // kept-or-accepted hash set (large matrices)
    uint64_t H_mask = 0;
    uint32_t* bits = nullptr;    // the same as a bitmap over all positions (out*in <= 2^31)
    uint64_t* R_key = nullptr;
    uint64_t* R_t = nullptr;
    uint64_t R_mask = 0;
    uint64_t* cand = nullptr;
    int64_t cand_cap = 0;
    uint64_t* new_lin = nullptr;
    int32_t* err = nullptr;
    // gradient grow
    int32_t* ghist = nullptr;    // [kGradBins]
    void* gsel = nullptr;        // GradSel
    int32_t* kept_ptr = nullptr; // [kept_ptr_len] kept entries per row
    int64_t kept_ptr_len = 0;
};

static uint64_t next_pow2(uint64_t x) {
    uint64_t p = 1;
    while (p < x) p <<= 1;
    return p;
}

void free_restructure(Layer* L) {
    RestructureWs* w = L->rws;
    if (!w) return;
    void* ptrs[] = {w->hist, w->sel, w->flags, w->scan_tmp, w->total, w->acc, w->kept_lin,
                    w->kept_val, w->H, w->bits, w->R_key, w->R_t, w->cand, w->new_lin, w->err,
                    w->ghist, w->gsel, w->kept_ptr};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    delete w;
    L->rws = nullptr;
}

static int alloc_restructure(Layer* L) {
    if (L->rws && L->rws->cap >= L->nnz) return SNK_OK;
    free_restructure(L);
    RestructureWs* w = new RestructureWs();
    L->rws = w;
    const int64_t n = std::max<int64_t>(L->nnz, 1);
    w->cap = n;
    w->cand_cap = n + n / 2 + 4096;
    const int64_t fl = std::max<int64_t>(n, w->cand_cap);
    w->flag_half = fl;
    w->scan_tmp_len = scan_tmp_len(fl);
    const uint64_t n_pos = (uint64_t)L->out_f * (uint64_t)L->in_f;
    const bool use_bits = n_pos <= (1ull << 31);
    const uint64_t hcap = use_bits ? 0 : next_pow2(2 * (uint64_t)n + 64);
    const uint64_t rcap = next_pow2(2 * (uint64_t)w->cand_cap + 64);
    w->H_mask = use_bits ? 0 : hcap - 1;
    w->R_mask = rcap - 1;
    bool ok = cudaMalloc(&w->hist, 256 * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->sel, sizeof(SelState)) == cudaSuccess &&
              cudaMalloc(&w->flags, 2 * fl * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->scan_tmp, w->scan_tmp_len * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->total, sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->acc, 2 * sizeof(int64_t)) == cudaSuccess &&
              cudaMalloc(&w->kept_lin, n * sizeof(uint64_t)) == cudaSuccess &&
              cudaMalloc(&w->kept_val, n * sizeof(uint32_t)) == cudaSuccess &&
              (use_bits ? cudaMalloc(&w->bits, (n_pos / 32 + 1) * sizeof(uint32_t))
                        : cudaMalloc(&w->H, hcap * sizeof(uint64_t))) == cudaSuccess &&
              cudaMalloc(&w->R_key, rcap * sizeof(uint64_t)) == cudaSuccess &&
              cudaMalloc(&w->R_t, rcap * sizeof(uint64_t)) == cudaSuccess &&
              cudaMalloc(&w->cand, w->cand_cap * sizeof(uint64_t)) == cudaSuccess &&
              cudaMalloc(&w->new_lin, n * sizeof(uint64_t)) == cudaSuccess &&
              cudaMalloc(&w->err, sizeof(int32_t)) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        free_restructure(L);
        return SNK_ERR_OOM;
    }
    return SNK_OK;
}

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint64_t splitmix64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Hash-table slot mixing: the 64-bit finaliser of MurmurHash3 (A. Appleby).
__device__ __forceinline__ uint64_t slot_hash(uint64_t x) {
    x ^= x >> 33;
    x *= 0xff51afd7ed558ccdull;
    x ^= x >> 33;
    x *= 0xc4ceb9fe1a85ec53ull;
    x ^= x >> 33;
    return x;
}

__device__ __forceinline__ bool set_has(const uint64_t* H, uint64_t mask, uint64_t key) {
    uint64_t i = slot_hash(key) & mask;
    for (uint64_t probes = 0; probes <= mask; ++probes, i = (i + 1) & mask) {
        uint64_t cur = H[i];
        if (cur == key) return true;
        if (cur == kEmpty) return false;
    }
    return false;
}

// Insert; returns the slot.  *err is set if the table is full (cannot happen
// at the load factors used here, but the loop is bounded regardless).
__device__ __forceinline__ uint64_t set_insert(uint64_t* H, uint64_t mask, uint64_t key,
                                               int32_t* err) {
    uint64_t i = slot_hash(key) & mask;
    for (uint64_t probes = 0; probes <= mask; ++probes, i = (i + 1) & mask) {
        unsigned long long prev = atomicCAS(reinterpret_cast<unsigned long long*>(H + i),
                                            (unsigned long long)kEmpty, (unsigned long long)key);
        if (prev == kEmpty || prev == key) return i;
    }
    atomicOr(err, kStatLimit);
    return 0;
}

__device__ __forceinline__ uint64_t table_get(const uint64_t* K, const uint64_t* V, uint64_t mask,
                                              uint64_t key) {
    uint64_t i = slot_hash(key) & mask;
    for (uint64_t probes = 0; probes <= mask; ++probes, i = (i + 1) & mask) {
        uint64_t cur = K[i];
        if (cur == key) return V[i];
        if (cur == kEmpty) return kEmpty;
    }
    return kEmpty;
}

__device__ __forceinline__ bool hi_match(uint64_t x, uint64_t y, int s) {
    return s >= 64 ? true : (x >> s) == (y >> s);
}

// ---------------------------------------------------------------- prune kernels
__global__ void k_sel_init(SelState* sel, int64_t k) {
    sel->mag = 0;
    sel->done = 0;
    sel->lin = 0;
    sel->krem = k;
}

// Histogram of the 8-bit digit at `shift` of the magnitude bits (phase 0) or
// of the position (phase 1), among the entries whose higher digits equal the
// prefix selected so far.
__global__ void k_sel_hist(const float* __restrict__ v, const int32_t* __restrict__ r,
                           const int32_t* __restrict__ c, int64_t n, int64_t in_f,
                           const SelState* __restrict__ sel, int phase, int shift,
                           int32_t* __restrict__ hist) {
    if (phase == 1 && sel->done) return;  // no tie on the magnitude to break
    __shared__ int h[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const uint32_t pmag = sel->mag;
    const uint64_t plin = sel->lin;
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        uint32_t m = __float_as_uint(v[k]) & 0x7fffffffu;
        if (phase == 0) {
            if (hi_match(m, pmag, shift + 8)) atomicAdd(&h[(m >> shift) & 255u], 1);
        } else if (m == pmag) {
            uint64_t lin = (uint64_t)r[k] * (uint64_t)in_f + (uint64_t)c[k];
            if (hi_match(lin, plin, shift + 8)) atomicAdd(&h[(lin >> shift) & 255u], 1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        if (h[i]) atomicAdd(&hist[i], h[i]);
}

__global__ void k_sel_pick(const int32_t* __restrict__ hist, SelState* sel, int phase, int shift) {
    if (threadIdx.x != 0) return;
    if (phase == 1 && sel->done) return;
    int64_t cum = 0;
    const int64_t krem = sel->krem;
    for (int d = 0; d < 256; ++d) {
        if (cum + hist[d] >= krem) {
            if (phase == 0) sel->mag |= (uint32_t)d << shift;
            else sel->lin |= (uint64_t)d << shift;
            sel->krem = krem - cum;
            // the last magnitude digit: if every entry of this magnitude goes,
            // no position is needed to break a tie (every position passes)
            if (phase == 0 && shift == 0 && hist[d] == krem - cum) {
                sel->done = 1;
                sel->lin = ~0ull;
            }
            return;
        }
        cum += hist[d];
    }
}

// keep flag = key > theta
__global__ void k_keep_flags(const float* __restrict__ v, const int32_t* __restrict__ r,
                             const int32_t* __restrict__ c, int64_t n, int64_t in_f,
                             const SelState* __restrict__ sel, int32_t* __restrict__ flags) {
    const uint32_t tm = sel->mag;
    const uint64_t tl = sel->lin;
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        uint32_t m = __float_as_uint(v[k]) & 0x7fffffffu;
        bool keep;
        if (m != tm) keep = m > tm;
        else keep = ((uint64_t)r[k] * (uint64_t)in_f + (uint64_t)c[k]) > tl;
        flags[k] = keep ? 1 : 0;
    }
}

__global__ void k_compact(const float* __restrict__ v, const int32_t* __restrict__ r,
                          const int32_t* __restrict__ c, int64_t n, int64_t in_f,
                          const int32_t* __restrict__ keep, const int32_t* __restrict__ pos,
                          uint64_t* __restrict__ kept_lin, uint32_t* __restrict__ kept_val) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        if (keep[k]) {
            int32_t p = pos[k];
            kept_lin[p] = (uint64_t)r[k] * (uint64_t)in_f + (uint64_t)c[k];
            kept_val[p] = __float_as_uint(v[k]);
        }
    }
}

// ---------------------------------------------------------------- regrow kernels
// The set of held positions (kept, then also accepted): a bitmap over all
// positions when there are at most 2^31 of them (it then sits in L2), else
// an open-addressing hash set.
struct HeldSet {
    uint64_t* H;
    uint64_t mask;
    uint32_t* bits;
    __device__ __forceinline__ bool has(uint64_t p) const {
        if (bits) return (bits[p >> 5] >> (p & 31u)) & 1u;
        return set_has(H, mask, p);
    }
    __device__ __forceinline__ void insert(uint64_t p, int32_t* err) const {
        if (bits) atomicOr(bits + (p >> 5), 1u << (p & 31u));
        else set_insert(H, mask, p, err);
    }
};

__global__ void k_set_fill(HeldSet hs, const uint64_t* __restrict__ keys, int64_t n, int32_t* err) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        hs.insert(keys[i], err);
}

__global__ void k_draw(uint64_t seed, uint64_t t0, int64_t B, uint64_t n_pos, HeldSet hs,
                       uint64_t* R_key, uint64_t* R_t, uint64_t R_mask,
                       uint64_t* __restrict__ cand, int32_t* err) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < B;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t t = t0 + (uint64_t)i;
        const uint64_t z = splitmix64_mix(seed + (t + 1ull) * kGamma);
        const uint64_t p = __umul64hi(z, n_pos);
        if (hs.has(p)) {
            cand[i] = kEmpty;
        } else {
            cand[i] = p;
            uint64_t slot = set_insert(R_key, R_mask, p, err);
            atomicMin(reinterpret_cast<unsigned long long*>(R_t + slot), (unsigned long long)t);
        }
    }
}

__global__ void k_first_flags(const uint64_t* __restrict__ cand, int64_t B, uint64_t t0,
                              const uint64_t* __restrict__ R_key, const uint64_t* __restrict__ R_t,
                              uint64_t R_mask, int32_t* __restrict__ flags) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < B;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t p = cand[i];
        flags[i] = (p != kEmpty && table_get(R_key, R_t, R_mask, p) == t0 + (uint64_t)i) ? 1 : 0;
    }
}

__global__ void k_take(const uint64_t* __restrict__ cand, const int32_t* __restrict__ surv,
                       const int32_t* __restrict__ pos, int64_t B, const int64_t* acc, int64_t k,
                       uint64_t* __restrict__ new_lin, HeldSet hs, int32_t* err) {
    const int64_t a = *acc;
    const int64_t need = k - a;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < B;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (surv[i] && pos[i] < need) {
            new_lin[a + pos[i]] = cand[i];
            hs.insert(cand[i], err);
        }
    }
}

__global__ void k_advance(int64_t* acc, const int32_t* total, int64_t k) {
    if (threadIdx.x == 0) {
        const int64_t need = k - *acc;
        *acc += (int64_t)(*total < need ? *total : need);
    }
}

// ---------------------------------------------------------------- gradient grow kernels
struct GradSel {
    uint64_t prefix;    // the selected high bits of the k-th smallest key
    int32_t level;      // how many high key bits are fixed
    int32_t exact;      // 1 when the selected bin holds exactly the remaining rank
    int64_t krem;       // rank still to find among keys with that prefix
    int64_t bin_count;  // keys in the selected bin
};

__global__ void k_grad_init(GradSel* sel, int64_t k) {
    sel->prefix = 0;
    sel->level = 0;
    sel->exact = 0;
    sel->krem = k;
}

// kept_ptr[j] = number of kept entries in rows < j, for j in [0, out]
__global__ void k_kept_row_ptr(const uint64_t* __restrict__ kept, int64_t m, int64_t in_f,
                               int64_t out_f, int32_t* __restrict__ ptr) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i <= m;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t prev = i == 0 ? -1 : (int64_t)(kept[i - 1] / (uint64_t)in_f);
        const int64_t cur = i == m ? out_f : (int64_t)(kept[i] / (uint64_t)in_f);
        for (int64_t j = prev + 1; j <= cur; ++j) ptr[j] = (int32_t)i;
    }
}

// The gradient of position (r, c): the fused multiply-add chain over the
// batch in order, g = fma(dY[b-1,r], X[b-1,c], ... fma(dY[0,r], X[0,c], 0)).
// Key: complement of the bit pattern of |g| (high 32 bits), then the position.
// dy holds dY[beta, r] for the row (shared memory when b <= kGradDyMax, else
// read from global memory with stride out_f).
__device__ __forceinline__ uint64_t grad_key(const float* __restrict__ X, const float* dy,
                                             int64_t dy_stride, int b, int64_t in_f, int64_t c,
                                             uint32_t p) {
    float g = 0.f;
    for (int beta = 0; beta < b; ++beta)
        g = __fmaf_rn(dy[beta * dy_stride], __ldg(X + beta * in_f + c), g);
    const uint32_t a = __float_as_uint(g) & 0x7fffffffu;
    return ((uint64_t)(~a) << 32) | (uint64_t)p;
}

// One pass over every candidate (a position held by no kept entry).  One
// warp per row; per 1024-column tile the row's kept columns are marked in a
// shared-memory bitmap, then lane l evaluates columns l, l+32, ...
//   COLLECT = false: histogram of the digit [shift, shift+width) of the keys
//     whose top `level` bits equal the selected prefix.
//   COLLECT = true: every key whose top `level` bits are <= the prefix is
//     selected; its position is appended to out_lin (at most cap).
//   MODE 0: histogram of the digit [shift, shift+width) of the keys whose top
//     `level` bits equal the selected prefix;
//   MODE 1: every key whose top bits are <= the prefix is selected (its
//     position appended to out_lin, at most cap);
//   MODE 2: keys whose top bits are below the prefix are selected as in
//     MODE 1, and the full keys of the selected bin (top bits equal) are
//     appended to bnd_keys (at most bcap) to be sorted.
template <int MODE>
__global__ void __launch_bounds__(kGradWarps * 32) k_grad_pass(
    const uint64_t* __restrict__ kept, const int32_t* __restrict__ kept_ptr, int64_t out_f,
    int64_t in_f, const float* __restrict__ X, const float* __restrict__ dY, int b,
    const GradSel* __restrict__ sel, int shift, int width, int32_t* __restrict__ hist,
    uint64_t* __restrict__ out_lin, int64_t* __restrict__ n_out, int64_t cap,
    uint64_t* __restrict__ bnd_keys, int64_t* __restrict__ n_bnd, int64_t bcap, int32_t* err) {
    constexpr bool COLLECT = MODE != 0;
    __shared__ int h[COLLECT ? 1 : kGradBins];
    __shared__ uint32_t bm[kGradWarps][kGradTile / 32];
    __shared__ float dys[kGradWarps][kGradDyMax];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (!COLLECT) {
        for (int i = threadIdx.x; i < (1 << width); i += blockDim.x) h[i] = 0;
        __syncthreads();
    }
    const uint64_t prefix = sel->prefix;
    const int level = sel->level;
    const uint32_t dmask = (1u << width) - 1u;
    for (int64_t r = (int64_t)blockIdx.x * kGradWarps + w; r < out_f;
         r += (int64_t)gridDim.x * kGradWarps) {
        int64_t j = kept_ptr[r];
        const int64_t j_end = kept_ptr[r + 1];
        const uint64_t row0 = (uint64_t)r * (uint64_t)in_f;
        // the row's dY values, once per row
        const bool dy_smem = b <= kGradDyMax;
        if (dy_smem)
            for (int beta = lane; beta < b; beta += 32) dys[w][beta] = __ldg(dY + beta * out_f + r);
        __syncwarp();
        const float* dy = dy_smem ? dys[w] : dY + r;
        const int64_t dy_stride = dy_smem ? 1 : out_f;
        for (int64_t c0 = 0; c0 < in_f; c0 += kGradTile) {
            const int64_t c1 = min(in_f, c0 + (int64_t)kGradTile);
            bm[w][lane] = 0u;
            __syncwarp();
            // mark the kept columns of [c0, c1): they are kept[j ..] while < row0 + c1
            while (j < j_end) {
                const int64_t jj = j + lane;
                const bool in_tile = jj < j_end && kept[jj] < row0 + (uint64_t)c1;
                if (in_tile) {
                    const uint32_t cc = (uint32_t)(kept[jj] - row0 - (uint64_t)c0);
                    atomicOr(&bm[w][cc >> 5], 1u << (cc & 31u));
                }
                const unsigned took = __ballot_sync(0xffffffffu, in_tile);
                j += __popc(took);
                if (took != 0xffffffffu) break;
            }
            __syncwarp();
            for (int t = 0; t < kGradTile / 32 && c0 + t * 32 < c1; ++t) {  // warp-uniform
                const int64_t c = c0 + t * 32 + lane;
                const bool cand = c < c1 && !((bm[w][t] >> lane) & 1u);
                uint64_t key = 0;
                if (cand) key = grad_key(X, dy, dy_stride, b, in_f, c, (uint32_t)(row0 + (uint64_t)c));
                if (!COLLECT) {
                    // lanes that hit the same bin add once, from their lowest lane
                    int bin = -1;
                    if (cand && (level == 0 || (key >> (64 - level)) == prefix))
                        bin = (int)((uint32_t)(key >> shift) & dmask);
                    const unsigned same = __match_any_sync(0xffffffffu, bin);
                    if (bin >= 0 && (same & ((1u << lane) - 1u)) == 0) atomicAdd(&h[bin], __popc(same));
                } else if (cand) {
                    const uint64_t top = key >> (64 - level);
                    if (top < prefix || (MODE == 1 && top == prefix)) {
                        const unsigned long long i =
                            atomicAdd(reinterpret_cast<unsigned long long*>(n_out), 1ull);
                        if ((int64_t)i < cap) out_lin[i] = row0 + (uint64_t)c;
                        else atomicOr(err, kStatLimit);
                    } else if (MODE == 2 && top == prefix) {
                        const unsigned long long i =
                            atomicAdd(reinterpret_cast<unsigned long long*>(n_bnd), 1ull);
                        if ((int64_t)i < bcap) bnd_keys[i] = key;
                        else atomicOr(err, kStatLimit);
                    }
                }
            }
            __syncwarp();
        }
    }
    if (!COLLECT) {
        __syncthreads();
        for (int i = threadIdx.x; i < (1 << width); i += blockDim.x)
            if (h[i]) atomicAdd(&hist[i], h[i]);
    }
}

// out[i] = position (low 32 bits) of the i-th smallest boundary key, i < n
__global__ void k_take_keys(const uint64_t* __restrict__ keys, int64_t n, uint64_t* __restrict__ out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = keys[i] & 0xffffffffull;
}

// Pick the digit bin holding the krem-th smallest key; one warp.
__global__ void k_grad_pick(const int32_t* __restrict__ hist, int width, GradSel* sel) {
    const int lane = threadIdx.x;
    const int nb = 1 << width;
    const int per = (nb + 31) / 32;
    const int lo = min(nb, lane * per), hi = min(nb, lo + per);
    int64_t mine = 0;
    for (int d = lo; d < hi; ++d) mine += hist[d];
    int64_t incl = mine;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int64_t krem = sel->krem;
    const int64_t excl = incl - mine;
    if (excl < krem && krem <= incl) {
        int64_t cum = excl;
        for (int d = lo; d < hi; ++d) {
            if (cum + hist[d] >= krem) {
                const int64_t left = krem - cum;
                sel->prefix = (sel->prefix << width) | (uint64_t)d;
                sel->level += width;
                sel->krem = left;
                sel->exact = (hist[d] == left) ? 1 : 0;
                sel->bin_count = hist[d];
                return;
            }
            cum += hist[d];
        }
    }
}

// Canonical triple from the kept entries (ascending positions, with values)
// and the grown positions (ascending, value +0.0f), by merge path: output
// tile q covers slots [q*T, (q+1)*T); the split of each tile boundary between
// the two lists is found by a binary search on the diagonal (the lists share
// no position), the block stages its pieces of both lists in shared memory,
// and each thread merges kMergePer consecutive outputs from its own split.
// Also writes the (column, slot) pairs the column view is sorted from.
constexpr int kMergeThreads = 256;
constexpr int kMergePer = 8;
constexpr int kMergeTile = kMergeThreads * kMergePer;

// number of kept entries among the first d outputs of the merge
template <typename KG>
__device__ __forceinline__ int64_t merge_split(const uint64_t* __restrict__ a, int64_t m,
                                               const KG* __restrict__ b, int64_t k, int64_t d) {
    int64_t lo = d > k ? d - k : 0, hi = d < m ? d : m;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (a[mid] < (uint64_t)b[d - mid - 1]) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__global__ void k_narrow_u32(const uint64_t* __restrict__ a, int64_t n, uint32_t* __restrict__ o) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        o[i] = (uint32_t)a[i];
}

template <typename KG>
__global__ void __launch_bounds__(kMergeThreads) k_merge_assemble(
    const uint64_t* __restrict__ kept_lin, const uint32_t* __restrict__ kept_val, int64_t m,
    const KG* __restrict__ new_lin, int64_t k, int64_t in_f, float* __restrict__ v,
    int32_t* __restrict__ r, int32_t* __restrict__ c, uint32_t* __restrict__ col_key,
    uint32_t* __restrict__ col_val) {
    __shared__ uint64_t sa[kMergeTile], sb[kMergeTile];
    __shared__ uint32_t sv[kMergeTile];
    __shared__ int64_t split[2];
    const int64_t n = m + k;
    for (int64_t t0 = (int64_t)blockIdx.x * kMergeTile; t0 < n; t0 += (int64_t)gridDim.x * kMergeTile) {
        const int64_t t1 = min(n, t0 + (int64_t)kMergeTile);
        if (threadIdx.x < 2) split[threadIdx.x] = merge_split(kept_lin, m, new_lin, k, threadIdx.x ? t1 : t0);
        __syncthreads();
        const int64_t i0 = split[0], i1 = split[1];
        const int64_t j0 = t0 - i0, j1 = t1 - i1;
        const int na = (int)(i1 - i0), nb = (int)(j1 - j0);
        for (int x = threadIdx.x; x < na; x += kMergeThreads) {
            sa[x] = kept_lin[i0 + x];
            sv[x] = kept_val[i0 + x];
        }
        for (int x = threadIdx.x; x < nb; x += kMergeThreads) sb[x] = (uint64_t)new_lin[j0 + x];
        __syncthreads();
        // this thread's outputs: [d0, d1) within the tile
        const int d0 = min(na + nb, threadIdx.x * kMergePer);
        const int d1 = min(na + nb, d0 + kMergePer);
        int lo = d0 > nb ? d0 - nb : 0, hi = d0 < na ? d0 : na;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sa[mid] < sb[d0 - mid - 1]) lo = mid + 1;
            else hi = mid;
        }
        int ia = lo, ib = d0 - lo;
        uint64_t ml[kMergePer];
        uint32_t mv[kMergePer];
#pragma unroll
        for (int q = 0; q < kMergePer; ++q) {
            if (d0 + q < d1) {
                const bool take_a = ib >= nb || (ia < na && sa[ia] < sb[ib]);
                ml[q] = take_a ? sa[ia] : sb[ib];
                mv[q] = take_a ? sv[ia] : 0u;
                if (take_a) ++ia;
                else ++ib;
            }
        }
        __syncthreads();  // every thread has read its inputs: reuse sa / sv for the output
#pragma unroll
        for (int q = 0; q < kMergePer; ++q) {
            if (d0 + q < d1) {
                sa[d0 + q] = ml[q];
                sv[d0 + q] = mv[q];
            }
        }
        __syncthreads();
        // coalesced write of the merged tile
        for (int x = threadIdx.x; x < na + nb; x += kMergeThreads) {
            const uint64_t lin = sa[x];
            const int64_t pos = t0 + x;
            const uint64_t rr = lin / (uint64_t)in_f;
            const int32_t cc = (int32_t)(lin - rr * (uint64_t)in_f);
            v[pos] = __uint_as_float(sv[x]);
            r[pos] = (int32_t)rr;
            c[pos] = cc;
            col_key[pos] = (uint32_t)cc;
            col_val[pos] = (uint32_t)pos;
        }
        __syncthreads();  // before the next tile reuses the shared arrays
    }
}

static int bits_for(uint64_t n_values) {
    int b = 0;
    while (b < 64 && (n_values - 1) >> b) ++b;
    return b;
}

static unsigned grid_of(int64_t n, int num_sms) {
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, 256), (int64_t)num_sms * 8));
}

// Prune step: the k smallest (|v| bits, lin) are removed; the kept entries
// are compacted, in canonical order, into kept_lin / kept_val.
static int prune_step(Layer* L, int64_t k, cudaStream_t s) {
    RestructureWs* w = L->rws;
    const int64_t n = L->nnz;
    const uint64_t n_pos = (uint64_t)L->out_f * (uint64_t)L->in_f;
    const unsigned G = grid_of(n, L->num_sms);
    k_sel_init<<<1, 1, 0, s>>>(w->sel, k);
    for (int shift = 24; shift >= 0; shift -= 8) {
        cudaMemsetAsync(w->hist, 0, 256 * sizeof(int32_t), s);
        k_sel_hist<<<G, 256, 0, s>>>(L->v, L->r, L->c, n, L->in_f, w->sel, 0, shift, w->hist);
        k_sel_pick<<<1, 32, 0, s>>>(w->hist, w->sel, 0, shift);
    }
    const int lin_bits = bits_for(n_pos);
    for (int shift = ((lin_bits + 7) / 8) * 8 - 8; shift >= 0; shift -= 8) {
        cudaMemsetAsync(w->hist, 0, 256 * sizeof(int32_t), s);
        k_sel_hist<<<G, 256, 0, s>>>(L->v, L->r, L->c, n, L->in_f, w->sel, 1, shift, w->hist);
        k_sel_pick<<<1, 32, 0, s>>>(w->hist, w->sel, 1, shift);
    }
    k_keep_flags<<<G, 256, 0, s>>>(L->v, L->r, L->c, n, L->in_f, w->sel, w->flags);
    int32_t* pos = w->flags + w->flag_half;
    int st = exclusive_scan_i32(w->flags, pos, n, w->scan_tmp, w->scan_tmp_len, w->total, s);
    if (st != SNK_OK) return st;
    k_compact<<<G, 256, 0, s>>>(L->v, L->r, L->c, n, L->in_f, w->flags, pos, w->kept_lin,
                                w->kept_val);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

// Uniform grow: k seeded draws accepted in draw order into new_lin.
static int grow_uniform(Layer* L, int64_t k, uint64_t seed, cudaStream_t s) {
    RestructureWs* w = L->rws;
    const int64_t m = L->nnz - k;
    const uint64_t n_pos = (uint64_t)L->out_f * (uint64_t)L->in_f;
    const HeldSet hs{w->H, w->H_mask, w->bits};
    if (w->bits) cudaMemsetAsync(w->bits, 0, (n_pos / 32 + 1) * sizeof(uint32_t), s);
    else cudaMemsetAsync(w->H, 0xFF, (w->H_mask + 1) * sizeof(uint64_t), s);
    k_set_fill<<<grid_of(m, L->num_sms), 256, 0, s>>>(hs, w->kept_lin, m, w->err);
    cudaMemsetAsync(w->acc, 0, sizeof(int64_t), s);
    const uint64_t t_max = 64ull * (uint64_t)k + 1024ull;
    uint64_t t0 = 0;
    int64_t accepted = 0;
    while (accepted < k && t0 < t_max) {
        const int64_t need = k - accepted;
        int64_t B = std::min<int64_t>(need + need / 2 + 1024, w->cand_cap);
        B = (int64_t)std::min<uint64_t>((uint64_t)B, t_max - t0);
        int32_t* surv = w->flags;
        int32_t* rank = w->flags + w->flag_half;
        // the round-local table is sized for this round's draws
        const uint64_t rm = std::min<uint64_t>(w->R_mask, next_pow2(2 * (uint64_t)B + 64) - 1);
        cudaMemsetAsync(w->R_key, 0xFF, (rm + 1) * sizeof(uint64_t), s);
        cudaMemsetAsync(w->R_t, 0xFF, (rm + 1) * sizeof(uint64_t), s);
        const unsigned GB = grid_of(B, L->num_sms);
        k_draw<<<GB, 256, 0, s>>>(seed, t0, B, n_pos, hs, w->R_key, w->R_t, rm, w->cand, w->err);
        k_first_flags<<<GB, 256, 0, s>>>(w->cand, B, t0, w->R_key, w->R_t, rm, surv);
        int st = exclusive_scan_i32(surv, rank, B, w->scan_tmp, w->scan_tmp_len, w->total, s);
        if (st != SNK_OK) return st;
        k_take<<<GB, 256, 0, s>>>(w->cand, surv, rank, B, w->acc, k, w->new_lin, hs, w->err);
        k_advance<<<1, 32, 0, s>>>(w->acc, w->total, k);
        if (cudaMemcpyAsync(&accepted, w->acc, sizeof(int64_t), cudaMemcpyDeviceToHost, s) !=
                cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return SNK_ERR_CUDA;
        t0 += (uint64_t)B;
    }
    int32_t h_err = 0;
    if (cudaMemcpyAsync(&h_err, w->err, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SNK_ERR_CUDA;
    if (h_err) return SNK_ERR_LIMIT;
    if (accepted < k) return SNK_ERR_LIMIT;
    return SNK_OK;
}

// Gradient grow: the k candidates with the smallest gradient keys into new_lin.
static int grow_gradient(Layer* L, int64_t k, const float* X, const float* dY, int64_t b,
                         cudaStream_t s) {
    RestructureWs* w = L->rws;
    const int64_t m = L->nnz - k;
    if (!w->ghist) {
        w->kept_ptr_len = L->out_f + 1;
        if (cudaMalloc(&w->ghist, kGradBins * sizeof(int32_t)) != cudaSuccess ||
            cudaMalloc(&w->gsel, sizeof(GradSel)) != cudaSuccess ||
            cudaMalloc(&w->kept_ptr, w->kept_ptr_len * sizeof(int32_t)) != cudaSuccess) {
            cudaGetLastError();
            return SNK_ERR_OOM;
        }
    }
    GradSel* sel = static_cast<GradSel*>(w->gsel);
    k_kept_row_ptr<<<grid_of(m + 1, L->num_sms), 256, 0, s>>>(w->kept_lin, m, L->in_f, L->out_f,
                                                              w->kept_ptr);
    k_grad_init<<<1, 1, 0, s>>>(sel, k);
    const unsigned G = (unsigned)std::max<int64_t>(
        1, std::min<int64_t>(ceil_div(L->out_f, kGradWarps), (int64_t)L->num_sms * 4));
    // boundary bins up to this size are sorted instead of refined by more passes
    // (the radix sort's scratch is sized for nnz keys)
    const int64_t bcap = std::min<int64_t>(L->nnz, int64_t(1) << 21);
    GradSel h{};
    bool boundary = false;
    for (int level = 0; level < 64;) {
        const int width = std::min(kGradDigit, 64 - level);
        const int shift = 64 - level - width;
        cudaMemsetAsync(w->ghist, 0, (size_t)(1 << width) * sizeof(int32_t), s);
        k_grad_pass<0><<<G, kGradWarps * 32, 0, s>>>(w->kept_lin, w->kept_ptr, L->out_f, L->in_f,
                                                    X, dY, (int)b, sel, shift, width, w->ghist,
                                                    nullptr, nullptr, 0, nullptr, nullptr, 0,
                                                    w->err);
        k_grad_pick<<<1, 32, 0, s>>>(w->ghist, width, sel);
        if (cudaMemcpyAsync(&h, sel, sizeof(GradSel), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return SNK_ERR_CUDA;
        if (h.level != level + width) return SNK_ERR_CUDA;  // rank not found: cannot happen
        level = h.level;
        if (h.exact) break;
        if (h.bin_count <= bcap && level < 64) {
            boundary = true;
            break;
        }
    }
    int64_t* n_bnd = w->acc + 1;
    cudaMemsetAsync(w->acc, 0, 2 * sizeof(int64_t), s);
    if (!boundary) {
        k_grad_pass<1><<<G, kGradWarps * 32, 0, s>>>(w->kept_lin, w->kept_ptr, L->out_f, L->in_f,
                                                    X, dY, (int)b, sel, 0, 1, nullptr, w->new_lin,
                                                    w->acc, k, nullptr, nullptr, 0, w->err);
    } else {
        // keys below the selected bin are in; the bin itself is sorted and
        // its first krem keys are in
        k_grad_pass<2><<<G, kGradWarps * 32, 0, s>>>(w->kept_lin, w->kept_ptr, L->out_f, L->in_f,
                                                    X, dY, (int)b, sel, 0, 1, nullptr, w->new_lin,
                                                    w->acc, k - h.krem, w->cand, n_bnd, bcap,
                                                    w->err);
        bool flipped = false;
        int st = sort_pairs_u64(w->cand, reinterpret_cast<uint32_t*>(w->flags), w->R_key,
                                reinterpret_cast<uint32_t*>(w->flags + w->flag_half), h.bin_count,
                                64 - h.level, L->tile_hist, L->tile_hist_len, s, &flipped);
        if (st != SNK_OK) return st;
        k_take_keys<<<grid_of(h.krem, L->num_sms), 256, 0, s>>>(flipped ? w->R_key : w->cand,
                                                                h.krem,
                                                                w->new_lin + (k - h.krem));
    }
    int64_t got[2] = {0, 0};
    int32_t h_err = 0;
    if (cudaMemcpyAsync(got, w->acc, 2 * sizeof(int64_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(&h_err, w->err, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SNK_ERR_CUDA;
    // keys are unique: exactly k are selected
    if (h_err) return SNK_ERR_CUDA;
    if (!boundary && got[0] != k) return SNK_ERR_CUDA;
    if (boundary && (got[0] != k - h.krem || got[1] != h.bin_count)) return SNK_ERR_CUDA;
    return SNK_OK;
}

// Write the new triple in canonical order: the kept entries are already in
// order, so only the k grown positions are sorted and the two lists merged;
// then the views are rebuilt.
static int assemble(Layer* L, int64_t k, cudaStream_t s) {
    RestructureWs* w = L->rws;
    const int64_t m = L->nnz - k;
    const uint64_t n_pos = (uint64_t)L->out_f * (uint64_t)L->in_f;
    const unsigned gm = (unsigned)std::max<int64_t>(
        1, std::min<int64_t>(ceil_div(L->nnz, kMergeTile), (int64_t)L->num_sms * 8));
    bool flipped = false;
    uint32_t* vals = reinterpret_cast<uint32_t*>(w->flags);
    uint32_t* vals_alt = reinterpret_cast<uint32_t*>(w->flags + w->flag_half);
    int st;
    if (n_pos <= (1ull << 32)) {
        // positions fit 32 bits: sort them as such (half the bytes moved)
        uint32_t* k32 = reinterpret_cast<uint32_t*>(w->cand);  // 2 * cand_cap words
        k_narrow_u32<<<grid_of(k, L->num_sms), 256, 0, s>>>(w->new_lin, k, k32);
        st = sort_pairs_u32(k32, vals, k32 + w->cand_cap, vals_alt, k, bits_for(n_pos),
                            L->tile_hist, L->tile_hist_len, s, &flipped);
        if (st != SNK_OK) return st;
        k_merge_assemble<uint32_t><<<gm, kMergeThreads, 0, s>>>(
            w->kept_lin, w->kept_val, m, flipped ? k32 + w->cand_cap : k32, k, L->in_f, L->v,
            L->r, L->c, L->col_keys, L->col_vals);
    } else {
        st = sort_pairs_u64(w->new_lin, vals, w->cand, vals_alt, k, bits_for(n_pos), L->tile_hist,
                            L->tile_hist_len, s, &flipped);
        if (st != SNK_OK) return st;
        k_merge_assemble<uint64_t><<<gm, kMergeThreads, 0, s>>>(
            w->kept_lin, w->kept_val, m, flipped ? w->cand : w->new_lin, k, L->in_f, L->v, L->r,
            L->c, L->col_keys, L->col_vals);
    }
    if (cudaGetLastError() != cudaSuccess) return SNK_ERR_CUDA;
    return build_views(L, s);
}

int run_prune_regrow(Layer* L, float zeta, uint64_t seed, cudaStream_t s) {
    if (!(zeta >= 0.0f && zeta < 1.0f)) return SNK_ERR_ARG;
    const int64_t n = L->nnz;
    const int64_t k = (int64_t)((double)zeta * (double)n);  // floor for non-negative values
    const uint64_t n_pos = (uint64_t)L->out_f * (uint64_t)L->in_f;
    if (n_pos - (uint64_t)(n - k) < (uint64_t)k) return SNK_ERR_NOSPACE;
    if (k == 0) return SNK_OK;
    int st = alloc_restructure(L);
    if (st != SNK_OK) return st;
    cudaMemsetAsync(L->rws->err, 0, sizeof(int32_t), s);
    if ((st = prune_step(L, k, s)) != SNK_OK) return st;
    if ((st = grow_uniform(L, k, seed, s)) != SNK_OK) return st;
    return assemble(L, k, s);
}

int run_prune_regrow_gradient(Layer* L, float zeta, const float* X, const float* dY, int64_t b,
                              cudaStream_t s) {
    if (!(zeta >= 0.0f && zeta < 1.0f)) return SNK_ERR_ARG;
    const int64_t n = L->nnz;
    const int64_t k = (int64_t)((double)zeta * (double)n);
    const uint64_t n_pos = (uint64_t)L->out_f * (uint64_t)L->in_f;
    if (n_pos > (1ull << 32)) return SNK_ERR_LIMIT;
    if (n_pos - (uint64_t)(n - k) < (uint64_t)k) return SNK_ERR_NOSPACE;
    if (k == 0) return SNK_OK;
    int st = alloc_restructure(L);
    if (st != SNK_OK) return st;
    cudaMemsetAsync(L->rws->err, 0, sizeof(int32_t), s);
    if ((st = prune_step(L, k, s)) != SNK_OK) return st;
    if ((st = grow_gradient(L, k, X, dY, b, s)) != SNK_OK) return st;
    return assemble(L, k, s);
}

}  // namespace snk
