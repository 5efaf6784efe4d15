// Weight gradient on the support (SDDMM) and the bias gradient.
//
//   "Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
//     sec. 7.1: dL/dW is wanted only at the live slots of W; for each live
//     slot at (i, c) it is the dot product of the dL/dY row i with the X
//     row c, so the dense M x K gradient is never formed.
//   "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
//     GPU", Fig. 1: the backward pass as a sparse outer product over supp(W).
//
//     dW_k  = sum_beta dY[beta, r_k] * X[beta, c_k]     (canonical order)
//     db[o] = sum_beta dY[beta, o]
//
// GB300 design: the same merge-path chunks and lane layout as the SpMM
// kernel, walking the canonical order.  The row index comes from the row
// pointer (no rows[] stream), the dY values of a row sit in registers for
// the whole row, X is staged transposed in shared memory, and the output is
// written with 128-bit stores in the order it is read, so the only HBM
// streams are cols (read) and dW (write).  No entry depends on another, so no
// chunk ever waits for another.
#include "snk_device.cuh"

namespace snk {

struct SddmmArgs {
    const int32_t* col;     // canonical column indices
    const uint16_t* col16;  // the same as 16-bit, zero padded (shared-memory path)
    const int32_t* row_ptr; // [out+1]
    const int4* cdesc;      // [n_blocks * kWarpsPerBlock] (k0, k1, first row, end row)
    int64_t nnz, out_f, in_f;
    int b;                  // batch columns of this tile
    int n_blocks;
    const float* X;         // [b, in] (tile)
    const float* xt;        // [in][BP] (global path)
    const float* dY;        // [b, out] (tile)
    float* dW;              // [nnz]
    bool accumulate;        // add to dW (later batch tiles)
    const float* dY_all;    // [b_all, out] for db, or null
    int64_t b_all;
    float* db;              // [out] or null
};

template <int BP>
__device__ __forceinline__ void load_dy_row(const SddmmArgs& a, int r, int sub,
                                            float (&d)[Tile<BP>::VEC]) {
    constexpr int VEC = Tile<BP>::VEC;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        const int beta = Tile<BP>::beta(sub, j);
        d[j] = beta < a.b ? __ldg(a.dY + (int64_t)beta * a.out_f + r) : 0.f;
    }
}

// One warp per chunk; the chunk's column indices stream as flat blocks of
// 4*GPW entries held in D+1 register slots (D blocks in flight while one is
// consumed; the slot loop is unrolled so slot indices are constants).  The dY
// values of the current row are in registers and the next row's are
// requested one row ahead.
template <int BP, bool SMEM>
__global__ void __launch_bounds__(kThreads, 1) k_sddmm(const SddmmArgs a) {
    constexpr bool I16 = SMEM && SNK_IDX16;
    using TL = Tile<BP>;
    constexpr int VEC = TL::VEC, LPE = TL::LPE, GPW = TL::GPW;
    constexpr uint32_t BLK = 4 * GPW;
    constexpr int D = BP <= 2 ? SNK_PIPE_DW_NARROW : ((BP == 4 || SMEM) ? SNK_PIPE_DW : SNK_PIPE_DW_WIDE);
    constexpr int NS = D + 1;
    extern __shared__ float4 smem4[];
    float* xs = reinterpret_cast<float*>(smem4);

    const int lane = threadIdx.x & 31;
    const int grp = lane / LPE;
    const int sub = lane % LPE;
    const uint32_t nnz = (uint32_t)a.nnz;
    const int4 cd = a.cdesc[blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)];
    const uint32_t k0 = (uint32_t)cd.x, k1 = (uint32_t)cd.y;
    const uint32_t base_first = k0 & ~3u;
    IdxBlk<I16> ib[NS];
    auto issue = [&](int s, uint32_t blk0) {
        const uint32_t base = blk0 + 4 * grp;
        if constexpr (I16) ib[s].load(a.col16, base);
        else ib[s].load(a.col, base, nnz);
    };
    SegWindow win{cd.z, cd.w - cd.z, 0, 0u, 0.f};
    if (k0 < k1) {
#pragma unroll
        for (int s = 0; s < NS; ++s)
            if (base_first + s * BLK < k1) issue(s, base_first + s * BLK);
        win.load(0, lane, a.row_ptr, nullptr);
    }
    if (a.db) {
        // bias gradient over the whole batch, sequential in batch order
        for (int64_t o = blockIdx.x * (int64_t)kThreads + threadIdx.x; o < a.out_f;
             o += (int64_t)gridDim.x * kThreads) {
            float sacc = 0.f;
            for (int64_t beta = 0; beta < a.b_all; ++beta) sacc += a.dY_all[beta * a.out_f + o];
            a.db[o] = sacc;
        }
    }
    if constexpr (SMEM) {
        stage_transposed<BP>(xs, a.X, a.in_f, a.b, a.in_f, threadIdx.x, kThreads);
        __syncthreads();
    }
    if (k0 >= k1) return;  // no entries in this chunk (rows without entries need no output)
    const float* xsrc = SMEM ? xs : a.xt;

    const int r_begin = win.r_begin;
    int i = 0;
    uint32_t rs = win.bnd(0, lane, a.row_ptr, nullptr), re = win.bnd(1, lane, a.row_ptr, nullptr);
    float dyr[VEC], dyn[VEC];
    load_dy_row<BP>(a, r_begin, sub, dyr);
#pragma unroll
    for (int j = 0; j < VEC; ++j) dyn[j] = 0.f;
    if (win.nrows > 1) load_dy_row<BP>(a, r_begin + 1, sub, dyn);

    auto consume = [&](int s, uint32_t blk0) {
        const uint32_t base = blk0 + 4 * grp;
        const uint32_t blk_end = min(blk0 + BLK, k1);
        float res[4] = {0.f, 0.f, 0.f, 0.f};
        const bool interior = rs <= blk0 && k0 <= blk0 && blk0 + BLK < re && blk0 + BLK <= k1;
        while (true) {
            if (interior) {
                // every entry of the block belongs to the current row, which
                // continues past the block
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x[VEC];
                    const float* px = xsrc + ib[s].get(j) * BP;
                    if constexpr (SMEM) TL::load(px, sub, x);
                    else TL::ldg(px, sub, x);
                    float p = 0.f;
#pragma unroll
                    for (int t = 0; t < VEC; ++t) p = fmaf(dyr[t], x[t], p);
#pragma unroll
                    for (int o = 1; o < LPE; o <<= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
                    res[j] = p;
                }
                break;
            }
            const uint32_t lo_k = max(max(rs, k0), blk0), hi_k = min(re, blk_end);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t k = base + j;
                const bool ok = k >= lo_k && k < hi_k;
                float x[VEC];
                const float* px = xsrc + (ok ? ib[s].get(j) : 0) * BP;
                if constexpr (SMEM) TL::load(px, sub, x);
                else TL::ldg(px, sub, x);
                float p = 0.f;
#pragma unroll
                for (int t = 0; t < VEC; ++t) p = fmaf(dyr[t], x[t], p);
#pragma unroll
                for (int o = 1; o < LPE; o <<= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
                if (ok) res[j] = p;
            }
            if (min(re, k1) > blk_end) break;  // row continues in the next block
            if (++i >= win.nrows) break;
            rs = re;
            re = win.bnd(i + 1, lane, a.row_ptr, nullptr);
#pragma unroll
            for (int j = 0; j < VEC; ++j) dyr[j] = dyn[j];
            if (i + 1 < win.nrows) load_dy_row<BP>(a, r_begin + i + 1, sub, dyn);
            if (rs >= blk_end) break;
        }
        if (sub == 0) {
            if (base >= k0 && base + 3 < k1) {
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
                for (int j = 0; j < 4; ++j) {
                    const uint32_t k = base + j;
                    if (k >= k0 && k < k1) a.dW[k] = a.accumulate ? a.dW[k] + res[j] : res[j];
                }
            }
        }
    };

    for (uint32_t base0 = base_first; base0 < k1; base0 += NS * BLK) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const uint32_t blk0 = base0 + s * BLK;
            if (blk0 < k1) {
                consume(s, blk0);
                if (blk0 + NS * BLK < k1) issue(s, blk0 + NS * BLK);
            }
        }
    }
}

template <int BP>
__global__ void k_transpose_x(const float* __restrict__ X, int64_t n, int b, float* __restrict__ xt) {
    stage_transposed<BP>(xt, X, n, b, n, blockIdx.x * blockDim.x + threadIdx.x,
                         gridDim.x * blockDim.x);
}

__global__ void k_bias_grad_only(const float* __restrict__ dY, int64_t b, int64_t n,
                                 float* __restrict__ db) {
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < n;
         o += (int64_t)gridDim.x * blockDim.x) {
        float sacc = 0.f;
        for (int64_t beta = 0; beta < b; ++beta) sacc += dY[beta * n + o];
        db[o] = sacc;
    }
}

template <int BP>
static int launch_bp(Layer* L, SddmmArgs a, cudaStream_t s) {
    const size_t smem = (size_t)a.in_f * BP * sizeof(float);
    const int grid = a.n_blocks;
    if constexpr (BP >= 8 && SNK_BANDS) {
        // an operand too wide for shared memory: row runs over column bands
        if (smem > (size_t)L->max_smem) {
            bool done = false;
            const int st = band_backward_weight(L, BP, a.X, a.dY, a.b, a.dW, a.accumulate, a.dY_all, a.b_all,
                                                a.db, s, &done);
            if (st != SNK_OK || done) return st;
        }
    }
    if (smem <= (size_t)L->max_smem && a.col16) {
        auto fn = k_sddmm<BP, true>;
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
            return SNK_ERR_CUDA;
        fn<<<grid, kThreads, smem, s>>>(a);
    } else {
        k_transpose_x<BP><<<L->num_sms * 4, 256, 0, s>>>(a.X, a.in_f, a.b, L->xt);
        a.xt = L->xt;
        k_sddmm<BP, false><<<grid, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

int launch_backward_weight(Layer* L, const float* X, const float* dY, int64_t b, float* dW,
                           float* db, cudaStream_t s) {
    if (L->nnz == 0) {
        if (db) {
            k_bias_grad_only<<<L->num_sms * 4, 256, 0, s>>>(dY, b, L->out_f, db);
            if (cudaGetLastError() != cudaSuccess) return SNK_ERR_CUDA;
        }
        return SNK_OK;
    }
    if (tc_eligible(L, b)) return run_tc_sddmm(L, X, dY, b, dW, db, s);
    SddmmArgs a{};
    a.col = L->c;
    a.col16 = L->c16;
    a.row_ptr = L->row_ptr;
    a.cdesc = L->cdesc_r;
    a.nnz = L->nnz;
    a.out_f = L->out_f;
    a.in_f = L->in_f;
    a.n_blocks = L->n_blocks;
    a.dW = dW;
    a.b_all = b;
    a.dY_all = dY;
    for (int64_t t0 = 0; t0 < b; t0 += kMaxBatchTile) {
        const int64_t bt = std::min<int64_t>(kMaxBatchTile, b - t0);
        a.b = (int)bt;
        a.X = X + t0 * L->in_f;
        a.dY = dY + t0 * L->out_f;
        a.accumulate = t0 > 0;
        a.db = (t0 == 0) ? db : nullptr;
        int st;
        switch (batch_tile(bt)) {
            case 1: st = launch_bp<1>(L, a, s); break;
            case 2: st = launch_bp<2>(L, a, s); break;
            case 4: st = launch_bp<4>(L, a, s); break;
            case 8: st = launch_bp<8>(L, a, s); break;
            case 16: st = launch_bp<16>(L, a, s); break;
            case 32: st = launch_bp<32>(L, a, s); break;
            default: st = launch_bp<64>(L, a, s); break;
        }
        if (st != SNK_OK) return st;
    }
    return SNK_OK;
}

}  // namespace snk
