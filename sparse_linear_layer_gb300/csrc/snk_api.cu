// C-ABI entry points of libsnk: argument checks, workspace ownership, and
// dispatch to the kernels.  See include/snk.h for the contract of each call.
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "snk_internal.cuh"

namespace snk {

// Host-side fault injection for tests: SNK_FAULT=alloc makes workspace
// allocation fail, SNK_FAULT=launch makes the product calls fail before they
// queue work.  Nothing here touches the GPU.
static bool fault(const char* what) {
    const char* f = getenv("SNK_FAULT");
    return f && strcmp(f, what) == 0;
}

static bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

static void free_layer(Layer* L) {
    if (!L) return;
    free_restructure(L);
    free_pcsr(L);
    free_tc(L);
    free_sweep(L);
    free_bands(L);
    void* ptrs[] = {L->row_ptr, L->col_ptr, L->rows_c, L->perm, L->c16, L->rc16, L->bnd_r, L->bnd_c, L->cdesc_r, L->cdesc_c,
                    L->bdesc_r, L->bdesc_c,
                    L->part, L->cnt, L->xt, L->status, L->sort_keys, L->sort_vals,
                    L->col_keys, L->col_vals, L->tile_hist};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    delete L;
}

template <typename T>
static bool dmalloc(T** p, int64_t count) {
    if (fault("alloc")) return false;
    size_t bytes = (size_t)std::max<int64_t>(count, 1) * sizeof(T);
    if (cudaMalloc((void**)p, bytes) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return false;
    }
    return true;
}

}  // namespace snk

using namespace snk;

extern "C" {

const char* snk_status_string(int status) {
    switch (status) {
        case SNK_OK: return "ok";
        case SNK_ERR_ARG: return "invalid argument (shape, null or misaligned pointer, zeta)";
        case SNK_ERR_DUP: return "duplicate (row, col) position in the triple";
        case SNK_ERR_RANGE: return "row or column index outside the matrix";
        case SNK_ERR_CUDA: return "CUDA error";
        case SNK_ERR_OOM: return "out of device memory for the workspace";
        case SNK_ERR_NOSPACE: return "fewer free positions than entries to regrow";
        case SNK_ERR_LIMIT: return "limit reached (regrow draws, or the fixed scratch size)";
        default: return "unknown status";
    }
}

int snk_create(snk_handle* handle, int64_t out_f, int64_t in_f, int64_t nnz, float* values,
               int32_t* rows, int32_t* cols, void* stream) {
    if (!handle) return SNK_ERR_ARG;
    if (out_f < 1 || in_f < 1 || out_f > INT32_MAX || in_f > INT32_MAX) return SNK_ERR_ARG;
    if (out_f > INT64_MAX / in_f) return SNK_ERR_ARG;
    if (nnz < 0 || nnz > INT32_MAX || nnz > out_f * in_f) return SNK_ERR_ARG;
    if (nnz > 0 && (!values || !rows || !cols)) return SNK_ERR_ARG;
    if (!aligned(values, 16) || !aligned(rows, 16) || !aligned(cols, 16)) return SNK_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;

    Layer* L = new Layer();
    L->out_f = out_f;
    L->in_f = in_f;
    L->nnz = nnz;
    L->v = values;
    L->r = rows;
    L->c = cols;
    if (cudaGetDevice(&L->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&L->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, L->device) !=
            cudaSuccess) {
        cudaGetLastError();
        delete L;
        return SNK_ERR_CUDA;
    }
    // one block per SM, one chunk per warp
    L->n_blocks = L->num_sms;
    L->n_chunks = L->n_blocks * std::max(kWarpsPerBlock, kWarpsPerBlockDx);
    const int64_t n_max = std::max(out_f, in_f);
    const bool wide = (uint64_t)out_f * (uint64_t)in_f > (1ull << 32);
    L->tile_hist_len = topology_hist_len(nnz);
    L->nnz_pad = ceil_div(nnz, 4) * 4 + kStreamPad;

    bool ok = dmalloc(&L->row_ptr, out_f + 1) && dmalloc(&L->col_ptr, in_f + 1) &&
              dmalloc(&L->rows_c, L->nnz_pad) && dmalloc(&L->perm, L->nnz_pad) &&
              (in_f > 65536 || dmalloc(&L->c16, L->nnz_pad)) &&
              (out_f > 65536 || dmalloc(&L->rc16, L->nnz_pad)) &&
              dmalloc(&L->bnd_r, (int64_t)L->n_blocks + 1) &&
              dmalloc(&L->bnd_c, (int64_t)L->n_blocks + 1) &&
              dmalloc(&L->cdesc_r, (int64_t)L->n_chunks) &&
              dmalloc(&L->cdesc_c, (int64_t)L->n_chunks) &&
              dmalloc(&L->bdesc_r, (int64_t)L->n_blocks) &&
              dmalloc(&L->bdesc_c, (int64_t)L->n_blocks) &&
              dmalloc(&L->part, (int64_t)L->n_blocks * 2 * kMaxBatchTile) &&
              dmalloc(&L->cnt, n_max) && dmalloc(&L->xt, n_max * kMaxBatchTile) &&
              dmalloc(&L->status, 1) &&
              dmalloc((char**)&L->sort_keys, 2 * nnz * (wide ? 8 : 4)) &&
              dmalloc(&L->sort_vals, 2 * nnz) && dmalloc(&L->col_keys, 2 * nnz) &&
              dmalloc(&L->col_vals, 2 * nnz) && dmalloc(&L->tile_hist, L->tile_hist_len);
    if (!ok) {
        free_layer(L);
        return SNK_ERR_OOM;
    }
    if (cudaMemsetAsync(L->cnt, 0, n_max * sizeof(int32_t), s) != cudaSuccess) {
        free_layer(L);
        return SNK_ERR_CUDA;
    }
    int st = build_topology(L, s, true);
    if (st != SNK_OK) {
        cudaStreamSynchronize(s);
        cudaGetLastError();
        free_layer(L);
        return st;
    }
    *handle = reinterpret_cast<snk_handle>(L);
    return SNK_OK;
}

int snk_forward(snk_handle h, const float* X, int64_t batch, const float* bias, float* Y,
                void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || batch < 0) return SNK_ERR_ARG;
    if (batch == 0) return SNK_OK;
    if (!X || !Y || !aligned(X, 4) || !aligned(Y, 4) || !aligned(bias, 4)) return SNK_ERR_ARG;
    if (fault("launch")) return SNK_ERR_CUDA;
    return launch_forward(L, X, batch, bias, Y, (cudaStream_t)stream);
}

int snk_backward_input(snk_handle h, const float* dY, int64_t batch, float* dX, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || batch < 0) return SNK_ERR_ARG;
    if (batch == 0) return SNK_OK;
    if (!dY || !dX || !aligned(dY, 4) || !aligned(dX, 4)) return SNK_ERR_ARG;
    if (fault("launch")) return SNK_ERR_CUDA;
    return launch_backward_input(L, dY, batch, dX, (cudaStream_t)stream);
}

int snk_backward_weight(snk_handle h, const float* X, const float* dY, int64_t batch, float* dW,
                        float* db, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || batch < 0) return SNK_ERR_ARG;
    if (batch == 0) return SNK_OK;
    if (!X || !dY || (!dW && L->nnz > 0)) return SNK_ERR_ARG;
    if (!aligned(X, 4) || !aligned(dY, 4) || !aligned(dW, 16) || !aligned(db, 4))
        return SNK_ERR_ARG;
    if (fault("launch")) return SNK_ERR_CUDA;
    return launch_backward_weight(L, X, dY, batch, dW, db, (cudaStream_t)stream);
}

int snk_prune_regrow(snk_handle h, float zeta, uint64_t seed, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L) return SNK_ERR_ARG;
    if (!(zeta >= 0.0f && zeta < 1.0f)) return SNK_ERR_ARG;
    if (fault("launch")) return SNK_ERR_CUDA;
    return run_prune_regrow(L, zeta, seed, (cudaStream_t)stream);
}

int snk_prune_regrow_gradient(snk_handle h, float zeta, const float* X, const float* dY,
                              int64_t batch, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L || batch < 1 || !X || !dY || !aligned(X, 4) || !aligned(dY, 4)) return SNK_ERR_ARG;
    if (!(zeta >= 0.0f && zeta < 1.0f)) return SNK_ERR_ARG;
    if (batch > INT32_MAX) return SNK_ERR_ARG;
    if (fault("launch")) return SNK_ERR_CUDA;
    return run_prune_regrow_gradient(L, zeta, X, dY, batch, (cudaStream_t)stream);
}

int snk_destroy(snk_handle h) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L) return SNK_OK;
    int dev = 0;
    cudaGetDevice(&dev);
    const int own = L->device;
    if (dev != own) cudaSetDevice(own);
    cudaDeviceSynchronize();
    free_layer(L);
    if (dev != own) cudaSetDevice(dev);
    return cudaGetLastError() == cudaSuccess ? SNK_OK : SNK_ERR_CUDA;
}

int snk_check(snk_handle h, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L) return SNK_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t word = 0;
    if (cudaMemcpyAsync(&word, L->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return SNK_ERR_CUDA;
    }
    if (!(word & kStatLimit)) return SNK_OK;
    if (cudaMemsetAsync(L->status, 0, sizeof(int32_t), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return SNK_ERR_CUDA;
    }
    return SNK_ERR_LIMIT;
}

int snk_get_shape(snk_handle h, int64_t* out_features, int64_t* in_features, int64_t* nnz,
                  int64_t* topology_version) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L) return SNK_ERR_ARG;
    if (out_features) *out_features = L->out_f;
    if (in_features) *in_features = L->in_f;
    if (nnz) *nnz = L->nnz;
    if (topology_version) *topology_version = L->topology_version;
    return SNK_OK;
}

int snk_copy_topology(snk_handle h, int32_t* row_ptr, int32_t* col_ptr, int32_t* rows_c,
                      int32_t* perm, void* stream) {
    Layer* L = reinterpret_cast<Layer*>(h);
    if (!L) return SNK_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const cudaMemcpyKind d2d = cudaMemcpyDeviceToDevice;
    if (row_ptr &&
        cudaMemcpyAsync(row_ptr, L->row_ptr, (L->out_f + 1) * sizeof(int32_t), d2d, s) != cudaSuccess)
        return SNK_ERR_CUDA;
    if (col_ptr &&
        cudaMemcpyAsync(col_ptr, L->col_ptr, (L->in_f + 1) * sizeof(int32_t), d2d, s) != cudaSuccess)
        return SNK_ERR_CUDA;
    if (L->nnz > 0) {
        if (rows_c &&
            cudaMemcpyAsync(rows_c, L->rows_c, L->nnz * sizeof(int32_t), d2d, s) != cudaSuccess)
            return SNK_ERR_CUDA;
        if (perm && cudaMemcpyAsync(perm, L->perm, L->nnz * sizeof(int32_t), d2d, s) != cudaSuccess)
            return SNK_ERR_CUDA;
    }
    return SNK_OK;
}

}  // extern "C"
