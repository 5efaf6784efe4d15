// Internal declarations of libsnk (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "snk.h"

namespace snk {

constexpr int kWarp = 32;
// Tuning parameters (compile-time; the defaults are the measured best on
// GB300 for 10000x10000 layers at batch 1..64).
#ifndef SNK_THREADS
#define SNK_THREADS 768    // SpMM / SDDMM block size; one block per SM
#endif
#ifndef SNK_PIPE_FWD
#define SNK_PIPE_FWD 2     // stream blocks in flight ahead of the consumed one (forward)
#endif
#ifndef SNK_PIPE_DX
#define SNK_PIPE_DX 1      // the same for the transposed product
#endif
#ifndef SNK_PIPE_DW
#define SNK_PIPE_DW 4      // the same for the weight gradient
#endif
#ifndef SNK_IDX16
#define SNK_IDX16 1        // read 16-bit index copies on the shared-memory path
#endif

constexpr int kThreads = SNK_THREADS;
constexpr int kWarpsPerBlock = kThreads / kWarp;
constexpr int kChunksPerSm = kWarpsPerBlock;   // merge-path chunks per SM (one per warp)
constexpr int kMaxBatchTile = 64;    // batch columns handled by one launch
constexpr int kStreamPad = 128;      // zero entries after library-owned streams

// Device status word bits.
constexpr int kStatRange = 1;
constexpr int kStatDup = 2;
constexpr int kStatLimit = 4;

struct RestructureWs;

// Library-owned state behind an snk_handle.
struct Layer {
    int64_t out_f = 0, in_f = 0, nnz = 0;
    float* v = nullptr;       // caller-owned, canonical order
    int32_t* r = nullptr;     // caller-owned
    int32_t* c = nullptr;     // caller-owned

    int device = 0;
    int num_sms = 0;
    int max_smem = 0;         // opt-in dynamic shared memory per block (bytes)
    int64_t topology_version = 0;

    // topology (rebuilt at create and after each restructure)
    int32_t* row_ptr = nullptr;   // [out+1]
    int32_t* col_ptr = nullptr;   // [in+1]
    int32_t* rows_c = nullptr;    // [nnz_pad] row of the j-th entry in column order
    int32_t* perm = nullptr;      // [nnz_pad] canonical slot of the j-th entry in column order
    // 16-bit copies of the index streams (when the dimension allows), read by
    // the shared-memory kernels; padded with zeros so blocks never test the end
    uint16_t* c16 = nullptr;      // [nnz_pad] canonical columns, if in <= 65536
    uint16_t* rc16 = nullptr;     // [nnz_pad] rows in column order, if out <= 65536
    int64_t nnz_pad = 0;          // round_up(nnz, 4) + kStreamPad

    // merge-path chunking of the canonical (row) and column orders
    int32_t chunk = 0;            // nnz per chunk
    int32_t n_chunks = 0;         // ceil(nnz / chunk)
    int2* desc_r = nullptr;       // [n_chunks] (first row touched by chunk q, end of its rows)
    int2* desc_c = nullptr;       // [n_chunks] the same for columns

    // scratch of the SpMM kernels
    float* part = nullptr;        // [n_chunks * 2 * kMaxBatchTile] split-segment partials
    int32_t* cnt = nullptr;       // [max(out,in)] arrival counters, all zero between calls
    float* xt = nullptr;          // [max(out,in) * kMaxBatchTile] transposed operand

    int32_t* status = nullptr;    // device status word

    // sort workspace (topology build)
    void* sort_keys = nullptr;    // 2 * nnz uint64
    uint32_t* sort_vals = nullptr;// 2 * nnz
    uint32_t* col_keys = nullptr; // 2 * nnz (column sort)
    uint32_t* col_vals = nullptr; // 2 * nnz
    int32_t* tile_hist = nullptr; // radix histograms
    int64_t tile_hist_len = 0;

    RestructureWs* rws = nullptr; // allocated on first prune_regrow
};

// ---- small helpers -------------------------------------------------------
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int batch_tile(int64_t b) {
    int bp = 1;
    while (bp < b) bp <<= 1;
    return bp;
}

// ---- topology (snk_topology.cu) -----------------------------------------
// Sort + validate + write back the canonical triple + CSR + CSC + chunk tables.
// Returns an SNK_* status; synchronises `s`.
int build_topology(Layer* L, cudaStream_t s, bool validate);

// Radix helpers reused by the restructure code.
int exclusive_scan_i32(const int32_t* in, int32_t* out, int64_t n, int32_t* tmp, int64_t tmp_len,
                       int32_t* total, cudaStream_t s);
int64_t scan_tmp_len(int64_t n);

// ---- kernels launched by the API ----------------------------------------
int launch_forward(Layer* L, const float* X, int64_t b, const float* bias, float* Y,
                   cudaStream_t s);
int launch_backward_input(Layer* L, const float* dY, int64_t b, float* dX, cudaStream_t s);
int launch_backward_weight(Layer* L, const float* X, const float* dY, int64_t b, float* dW,
                           float* db, cudaStream_t s);
int run_prune_regrow(Layer* L, float zeta, uint64_t seed, cudaStream_t s);
int launch_chunk_desc(const int32_t* ptr, int64_t n_seg, int32_t chunk, int32_t n_chunks,
                      int2* desc, int num_sms, cudaStream_t s);
int launch_forward_csr(const float* val, const int32_t* cols, const int32_t* row_ptr,
                       const int2* desc, int64_t nnz, int64_t out_f, int64_t in_f, int chunk,
                       int n_chunks, const float* X, int64_t b, const float* bias, float* Y,
                       float* part, int32_t* cnt, int num_sms, int max_smem, cudaStream_t s);
void free_restructure(Layer* L);

}  // namespace snk
