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
//  * The kept and grown entries are written back into the caller's triple
//    and the topology build re-sorts it.
#include <algorithm>

#include "snk_internal.cuh"

namespace snk {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kEmpty = ~0ull;

struct SelState {
    uint32_t mag;
    uint32_t pad;
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
    int64_t* acc = nullptr;      // device scalar: accepted so far
    uint64_t* kept_lin = nullptr;
    uint32_t* kept_val = nullptr;
    uint64_t* H = nullptr;
    uint64_t H_mask = 0;
    uint64_t* R_key = nullptr;
    uint64_t* R_t = nullptr;
    uint64_t R_mask = 0;
    uint64_t* cand = nullptr;
    int64_t cand_cap = 0;
    uint64_t* new_lin = nullptr;
    int32_t* err = nullptr;
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
                    w->kept_val, w->H, w->R_key, w->R_t, w->cand, w->new_lin, w->err};
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
    const uint64_t hcap = next_pow2(2 * (uint64_t)n + 64);
    const uint64_t rcap = next_pow2(2 * (uint64_t)w->cand_cap + 64);
    w->H_mask = hcap - 1;
    w->R_mask = rcap - 1;
    bool ok = cudaMalloc(&w->hist, 256 * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->sel, sizeof(SelState)) == cudaSuccess &&
              cudaMalloc(&w->flags, 2 * fl * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->scan_tmp, w->scan_tmp_len * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->total, sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&w->acc, sizeof(int64_t)) == cudaSuccess &&
              cudaMalloc(&w->kept_lin, n * sizeof(uint64_t)) == cudaSuccess &&
              cudaMalloc(&w->kept_val, n * sizeof(uint32_t)) == cudaSuccess &&
              cudaMalloc(&w->H, hcap * sizeof(uint64_t)) == cudaSuccess &&
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
    sel->pad = 0;
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
    int64_t cum = 0;
    const int64_t krem = sel->krem;
    for (int d = 0; d < 256; ++d) {
        if (cum + hist[d] >= krem) {
            if (phase == 0) sel->mag |= (uint32_t)d << shift;
            else sel->lin |= (uint64_t)d << shift;
            sel->krem = krem - cum;
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
__global__ void k_set_fill(uint64_t* H, uint64_t mask, const uint64_t* __restrict__ keys, int64_t n,
                           int32_t* err) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        set_insert(H, mask, keys[i], err);
}

__global__ void k_draw(uint64_t seed, uint64_t t0, int64_t B, uint64_t n_pos,
                       const uint64_t* __restrict__ H, uint64_t H_mask, uint64_t* R_key,
                       uint64_t* R_t, uint64_t R_mask, uint64_t* __restrict__ cand, int32_t* err) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < B;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t t = t0 + (uint64_t)i;
        const uint64_t z = splitmix64_mix(seed + (t + 1ull) * kGamma);
        const uint64_t p = __umul64hi(z, n_pos);
        if (set_has(H, H_mask, p)) {
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
                       uint64_t* __restrict__ new_lin, uint64_t* H, uint64_t H_mask, int32_t* err) {
    const int64_t a = *acc;
    const int64_t need = k - a;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < B;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (surv[i] && pos[i] < need) {
            new_lin[a + pos[i]] = cand[i];
            set_insert(H, H_mask, cand[i], err);
        }
    }
}

__global__ void k_advance(int64_t* acc, const int32_t* total, int64_t k) {
    if (threadIdx.x == 0) {
        const int64_t need = k - *acc;
        *acc += (int64_t)(*total < need ? *total : need);
    }
}

__global__ void k_assemble(const uint64_t* __restrict__ kept_lin, const uint32_t* __restrict__ kept_val,
                           int64_t m, const uint64_t* __restrict__ new_lin, int64_t k, int64_t in_f,
                           float* __restrict__ v, int32_t* __restrict__ r, int32_t* __restrict__ c) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < m + k;
         i += (int64_t)gridDim.x * blockDim.x) {
        uint64_t lin;
        uint32_t val;
        if (i < m) {
            lin = kept_lin[i];
            val = kept_val[i];
        } else {
            lin = new_lin[i - m];
            val = 0u;
        }
        const uint64_t rr = lin / (uint64_t)in_f;
        v[i] = __uint_as_float(val);
        r[i] = (int32_t)rr;
        c[i] = (int32_t)(lin - rr * (uint64_t)in_f);
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

int run_prune_regrow(Layer* L, float zeta, uint64_t seed, cudaStream_t s) {
    if (!(zeta >= 0.0f && zeta < 1.0f)) return SNK_ERR_ARG;
    const int64_t n = L->nnz;
    const int64_t k = (int64_t)((double)zeta * (double)n);  // floor for non-negative values
    const uint64_t n_pos = (uint64_t)L->out_f * (uint64_t)L->in_f;
    if (n_pos - (uint64_t)(n - k) < (uint64_t)k) return SNK_ERR_NOSPACE;
    if (k == 0) return SNK_OK;
    int st = alloc_restructure(L);
    if (st != SNK_OK) return st;
    RestructureWs* w = L->rws;
    const unsigned G = grid_of(n, L->num_sms);
    cudaMemsetAsync(w->err, 0, sizeof(int32_t), s);

    // ---- prune: radix select of the k-th smallest (|v| bits, lin)
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
    st = exclusive_scan_i32(w->flags, pos, n, w->scan_tmp, w->scan_tmp_len, w->total, s);
    if (st != SNK_OK) return st;
    k_compact<<<G, 256, 0, s>>>(L->v, L->r, L->c, n, L->in_f, w->flags, pos, w->kept_lin,
                                w->kept_val);
    const int64_t m = n - k;

    // ---- regrow
    cudaMemsetAsync(w->H, 0xFF, (w->H_mask + 1) * sizeof(uint64_t), s);
    k_set_fill<<<grid_of(m, L->num_sms), 256, 0, s>>>(w->H, w->H_mask, w->kept_lin, m, w->err);
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
        cudaMemsetAsync(w->R_key, 0xFF, (w->R_mask + 1) * sizeof(uint64_t), s);
        cudaMemsetAsync(w->R_t, 0xFF, (w->R_mask + 1) * sizeof(uint64_t), s);
        const unsigned GB = grid_of(B, L->num_sms);
        k_draw<<<GB, 256, 0, s>>>(seed, t0, B, n_pos, w->H, w->H_mask, w->R_key, w->R_t, w->R_mask,
                                  w->cand, w->err);
        k_first_flags<<<GB, 256, 0, s>>>(w->cand, B, t0, w->R_key, w->R_t, w->R_mask, surv);
        st = exclusive_scan_i32(surv, rank, B, w->scan_tmp, w->scan_tmp_len, w->total, s);
        if (st != SNK_OK) return st;
        k_take<<<GB, 256, 0, s>>>(w->cand, surv, rank, B, w->acc, k, w->new_lin, w->H, w->H_mask,
                                  w->err);
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

    // ---- write back and rebuild
    k_assemble<<<G, 256, 0, s>>>(w->kept_lin, w->kept_val, m, w->new_lin, k, L->in_f, L->v, L->r,
                                 L->c);
    if (cudaGetLastError() != cudaSuccess) return SNK_ERR_CUDA;
    return build_topology(L, s, false);
}

}  // namespace snk
