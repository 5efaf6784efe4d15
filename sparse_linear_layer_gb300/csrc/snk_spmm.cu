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
//  * Load balance: the nnz stream is cut into equal chunks (merge path), 64
//    per SM, two per warp, so skewed row lengths cost nothing.  A segment cut
//    by a chunk boundary is finished by whichever of its chunks arrives last
//    (an arrival counter per segment); the partials are summed in chunk order,
//    so the result does not depend on timing.  Counters return to zero.
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
    const float* val;       // stored values, canonical order
    const int32_t* perm;    // column-order -> canonical slot (transposed product) or null
    const int32_t* idx;     // operand index per stored entry (col, or row in column order)
    const int32_t* seg_ptr; // [n_seg+1]
    const int32_t* own;     // [n_chunks+1]
    int64_t nnz;
    int64_t n_seg;          // output length per batch row
    int64_t n_src;          // operand length per batch row
    int b;                  // batch columns of this tile (<= BP)
    int chunk;
    int n_chunks;
    const float* X;         // [b, n_src] row-major
    const float* xt;        // [n_src][BP] transposed copy (global-memory path)
    const float* bias;      // [n_seg] or null
    float* Y;               // [b, n_seg] row-major
    float* part;            // [n_chunks][2][BP]
    int32_t* cnt;           // [n_seg]
};

template <int BP, bool GATHER, bool SMEM>
__global__ void __launch_bounds__(kThreads, 1) k_spmm(const SpmmArgs a) {
    using TL = Tile<BP>;
    constexpr int VEC = TL::VEC, LPE = TL::LPE, GPW = TL::GPW;
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);
    if constexpr (SMEM) {
        stage_transposed<BP>(xs, a.X, a.n_src, a.b, a.n_src, threadIdx.x, kThreads);
        __syncthreads();
    }
    const float* xsrc = SMEM ? xs : a.xt;

    const int lane = threadIdx.x & 31;
    const int grp = lane / LPE;
    const int sub = lane % LPE;
    const int n_warps = gridDim.x * kWarpsPerBlock;
    const uint32_t nnz = (uint32_t)a.nnz;
    for (int q = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); q < a.n_chunks; q += n_warps) {
        const uint32_t k0 = (uint32_t)q * (uint32_t)a.chunk;
        const uint32_t k1 = min(k0 + (uint32_t)a.chunk, nnz);
        const int lo = a.own[q];
        const int hi = a.own[q + 1];
        const int r_begin = (lo > 0 && (uint32_t)a.seg_ptr[lo] > k0) ? lo - 1 : lo;
        for (int r = r_begin; r < hi; ++r) {
            const uint32_t rs = (uint32_t)a.seg_ptr[r], re = (uint32_t)a.seg_ptr[r + 1];
            const uint32_t s = max(rs, k0), e = min(re, k1);
            float acc[VEC];
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
            // warp-uniform trip count: every group runs the same iterations
            for (uint32_t base0 = s & ~3u; base0 < e; base0 += 4 * GPW) {
                const uint32_t base = base0 + 4 * grp;
                float w[4];
                int col[4];
                stream4(a.idx, base, nnz, col);
                if constexpr (!GATHER) {
                    stream4(a.val, base, nnz, w);
                } else {
                    int pm[4];
                    stream4(a.perm, base, nnz, pm);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t k = base + j;
                        w[j] = (k >= s && k < e) ? __ldg(a.val + pm[j]) : 0.f;
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t k = base + j;
                    if (k >= s && k < e) {
                        float x[VEC];
                        const float* px = xsrc + col[j] * BP + sub * VEC;
                        if constexpr (SMEM) VecF<VEC>::load(px, x);
                        else VecF<VEC>::ldg(px, x);
#pragma unroll
                        for (int t = 0; t < VEC; ++t) acc[t] = fmaf(w[j], x[t], acc[t]);
                    }
                }
            }
#pragma unroll
            for (int o = LPE; o < kWarp; o <<= 1) {
#pragma unroll
                for (int j = 0; j < VEC; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
            }
            const float bo = a.bias ? __ldg(a.bias + r) : 0.f;
            if (rs >= k0 && re <= k1) {
                if (lane < LPE) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const int beta = sub * VEC + j;
                        if (beta < a.b) a.Y[(int64_t)beta * a.n_seg + r] = acc[j] + bo;
                    }
                }
            } else {
                // segment cut by a chunk boundary: publish this chunk's partial,
                // and let the last arriving chunk sum all of them in chunk order
                const int64_t q_first = rs / (uint32_t)a.chunk;
                const int64_t q_last = (re - 1) / (uint32_t)a.chunk;
                const int slot = (rs < k0) ? 0 : 1;
                if (lane < LPE) {
                    float* my = a.part + ((int64_t)q * 2 + slot) * BP + sub * VEC;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) my[j] = acc[j];
                }
                __threadfence();
                __syncwarp();
                int old = 0;
                if (lane == 0) old = atomicAdd(a.cnt + r, 1);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old == (int)(q_last - q_first)) {
                    __threadfence();
                    if (lane < LPE) {
                        float sum[VEC];
#pragma unroll
                        for (int j = 0; j < VEC; ++j) sum[j] = 0.f;
                        for (int64_t qq = q_first; qq <= q_last; ++qq) {
                            const float* pp =
                                a.part + (qq * 2 + (qq == q_first ? 1 : 0)) * BP + sub * VEC;
#pragma unroll
                            for (int j = 0; j < VEC; ++j) sum[j] += __ldcg(pp + j);
                        }
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            const int beta = sub * VEC + j;
                            if (beta < a.b) a.Y[(int64_t)beta * a.n_seg + r] = sum[j] + bo;
                        }
                    }
                    if (lane == 0) a.cnt[r] = 0;
                }
            }
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

template <int BP, bool GATHER>
static int launch_bp(Layer* L, SpmmArgs a, cudaStream_t s) {
    const size_t smem = (size_t)a.n_src * BP * sizeof(float);
    const int grid = (int)std::min<int64_t>(L->num_sms, ceil_div(a.n_chunks, kWarpsPerBlock));
    if (smem <= (size_t)L->max_smem) {
        auto fn = k_spmm<BP, GATHER, true>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
            return SNK_ERR_CUDA;
        fn<<<grid, kThreads, smem, s>>>(a);
    } else {
        k_transpose<BP><<<L->num_sms * 4, 256, 0, s>>>(a.X, a.n_src, a.b, L->xt);
        a.xt = L->xt;
        k_spmm<BP, GATHER, false><<<grid, kThreads, 0, s>>>(a);
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

int launch_forward(Layer* L, const float* X, int64_t b, const float* bias, float* Y,
                   cudaStream_t s) {
    SpmmArgs a{};
    a.val = L->v;
    a.perm = nullptr;
    a.idx = L->c;
    a.seg_ptr = L->row_ptr;
    a.own = L->own_r;
    a.nnz = L->nnz;
    a.n_seg = L->out_f;
    a.n_src = L->in_f;
    a.chunk = L->chunk;
    a.n_chunks = L->n_chunks;
    a.X = X;
    a.bias = bias;
    a.Y = Y;
    a.part = L->part;
    a.cnt = L->cnt;
    return run_spmm<false>(L, a, b, s);
}

int launch_backward_input(Layer* L, const float* dY, int64_t b, float* dX, cudaStream_t s) {
    SpmmArgs a{};
    a.val = L->v;
    a.perm = L->perm;
    a.idx = L->rows_c;
    a.seg_ptr = L->col_ptr;
    a.own = L->own_c;
    a.nnz = L->nnz;
    a.n_seg = L->in_f;
    a.n_src = L->out_f;
    a.chunk = L->chunk;
    a.n_chunks = L->n_chunks;
    a.X = dY;
    a.bias = nullptr;
    a.Y = dX;
    a.part = L->part;
    a.cnt = L->cnt;
    return run_spmm<true>(L, a, b, s);
}

}  // namespace snk
