// Exact recomputation, on the CUDA cores, of the large-batch outputs that the
// tensor-core path cannot deliver within the layer's tolerance.
//
// The tensor path ("Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural
// Networks on GPU", appendix Table 13's batch-4096 regime) multiplies
// densified tiles of W with the dense operand after splitting both into
// scaled fp16 pieces.  Two kinds of input defeat that representation:
//   * an inf or NaN: a densified tile also multiplies the stored zeros, so it
//     would spread NaN over a whole output row or column, where the layer's
//     definition (a sum over the stored entries only) gives NaN or +-inf only
//     at the outputs an entry actually reaches;
//   * a row (or segment) whose values span more than about 2^16: its smallest
//     nonzero values fall under fp16's normal range after scaling, so they are
//     held only to an absolute floor, which can exceed 1e-5 * A + 1e-6.
// The pre-passes of the tensor path flag such dense rows and segments of W;
// the kernels here then recompute every output they reach from the
// definition, per stored entry, exactly like the batch-tiled path would:
// fp32 products summed as 32 lane-strided partial sums and a shuffle tree,
// so inf and NaN propagate per entry and the error bound of the batch-tiled
// kernels holds.  An output reached from both a flagged row and a flagged
// segment is computed twice by the same routine, so both writes carry the
// same bits.
#include "snk_internal.cuh"

namespace snk {
namespace {

// Warp-wide sum of val(j) * d[idx[j]] over the entries [j0, j1) of one
// segment: lane l takes entries j0 + l, j0 + l + 32, ...; the 32 partial sums
// are added by a shuffle tree (every lane gets the result).
__device__ __forceinline__ float seg_dot(const TcSide& sd, int64_t j0, int64_t j1,
                                         const float* __restrict__ d, int lane) {
    float acc = 0.f;
    for (int64_t j = j0 + lane; j < j1; j += 32) {
        const float w = sd.perm ? __ldg(sd.val + __ldg(sd.perm + j)) : __ldg(sd.val + j);
        acc = fmaf(w, __ldg(d + __ldg(sd.idx + j)), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// Flagged dense rows: Y[rows[i], o] for every segment o, one warp per
// (row, segment) item, consecutive warps on consecutive segments of a row.
__global__ void __launch_bounds__(256) k_exact_rows(const TcSide sd, int64_t n_seg,
                                                    const float* __restrict__ D, int64_t K,
                                                    const float* __restrict__ bias,
                                                    float* __restrict__ Y,
                                                    const int32_t* __restrict__ rows,
                                                    const uint32_t* __restrict__ n_rows) {
    const int lane = threadIdx.x & 31;
    const int64_t items = (int64_t)*n_rows * n_seg;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t it = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items;
         it += warps) {
        const int64_t beta = rows[it / n_seg];
        const int64_t o = it % n_seg;
        const float y = seg_dot(sd, sd.ptr[o], sd.ptr[o + 1], D + beta * K, lane);
        if (lane == 0) Y[beta * n_seg + o] = y + (bias ? bias[o] : 0.f);
    }
}

// Candidate segments (those holding a non-finite value or values under the
// fp16 floor): each block takes candidates in turn, confirms the flag against
// the dense rows' largest L1 norm and magnitude, and its warps recompute the
// segment's output for every dense row.
__global__ void __launch_bounds__(256) k_exact_segs(const TcSide sd, int64_t n_seg,
                                                    const float* __restrict__ D, int64_t K,
                                                    int64_t b, const float* __restrict__ bias,
                                                    float* __restrict__ Y,
                                                    const int32_t* __restrict__ cand,
                                                    const uint32_t* __restrict__ n_cand,
                                                    const int32_t* __restrict__ seg_exp,
                                                    const int32_t* __restrict__ seg_code,
                                                    const uint32_t* __restrict__ other) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const uint32_t nc = *n_cand;
    const float l1 = __uint_as_float(other[0]), mx = __uint_as_float(other[1]);
    for (uint32_t c = blockIdx.x; c < nc; c += gridDim.x) {
        const int64_t o = cand[c];
        if (!tc_needs_exact(seg_code[o], seg_exp[o], l1, mx)) continue;
        const int64_t j0 = sd.ptr[o], j1 = sd.ptr[o + 1];
        const float bo = bias ? bias[o] : 0.f;
        for (int64_t beta = warp; beta < b; beta += nw) {
            const float y = seg_dot(sd, j0, j1, D + beta * K, lane);
            if (lane == 0) Y[beta * n_seg + o] = y + bo;
        }
    }
}

// dW_k = sum_beta dY[beta, r_k] X[beta, c_k] over the whole batch, one warp
// per entry, lane l taking beta = l, l + 32, ...; for every entry of the
// listed rows of W (list values below out) and columns (out + column).
__global__ void __launch_bounds__(256) k_exact_dw(const int32_t* __restrict__ row_ptr,
                                                  const int32_t* __restrict__ cols,
                                                  const int32_t* __restrict__ col_ptr,
                                                  const int32_t* __restrict__ rows_c,
                                                  const int32_t* __restrict__ perm,
                                                  const float* __restrict__ X,
                                                  const float* __restrict__ dY, int64_t b,
                                                  int64_t out_f, int64_t in_f,
                                                  float* __restrict__ dW,
                                                  const int32_t* __restrict__ list,
                                                  const uint32_t* __restrict__ n_list) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const uint32_t n = *n_list;
    for (uint32_t u = blockIdx.x; u < n; u += gridDim.x) {
        const int64_t item = list[u];
        const bool is_row = item < out_f;
        const int64_t j0 = is_row ? row_ptr[item] : col_ptr[item - out_f];
        const int64_t j1 = is_row ? row_ptr[item + 1] : col_ptr[item - out_f + 1];
        for (int64_t j = j0 + warp; j < j1; j += nw) {
            const int64_t k = is_row ? j : perm[j];
            const int64_t r = is_row ? item : rows_c[j];
            const int64_t c = is_row ? cols[j] : item - out_f;
            float acc = 0.f;
            for (int64_t beta = lane; beta < b; beta += 32)
                acc = fmaf(__ldg(dY + beta * out_f + r), __ldg(X + beta * in_f + c), acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) dW[k] = acc;
        }
    }
}

}  // namespace

int launch_exact_rows(const TcSide& sd, int64_t n_seg, const float* D, int64_t K,
                      const float* bias, float* Y, const int32_t* rows, const uint32_t* n_rows,
                      int num_sms, cudaStream_t s) {
    k_exact_rows<<<num_sms * 4, 256, 0, s>>>(sd, n_seg, D, K, bias, Y, rows, n_rows);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

int launch_exact_segs(const TcSide& sd, int64_t n_seg, const float* D, int64_t K, int64_t b,
                      const float* bias, float* Y, const int32_t* cand, const uint32_t* n_cand,
                      const int32_t* seg_exp, const int32_t* seg_code, const uint32_t* other,
                      int num_sms, cudaStream_t s) {
    k_exact_segs<<<num_sms * 2, 256, 0, s>>>(sd, n_seg, D, K, b, bias, Y, cand, n_cand, seg_exp,
                                             seg_code, other);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

int launch_exact_dw(const Layer* L, const float* X, const float* dY, int64_t b, float* dW,
                    const int32_t* list, const uint32_t* n_list, cudaStream_t s) {
    k_exact_dw<<<L->num_sms * 2, 256, 0, s>>>(L->row_ptr, L->c, L->col_ptr, L->rows_c, L->perm,
                                              X, dY, b, L->out_f, L->in_f, dW, list, n_list);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

}  // namespace snk
