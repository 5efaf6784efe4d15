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
#ifndef SNK_PIPE_FWD_NARROW
#define SNK_PIPE_FWD_NARROW 3  // the same for 1-column tiles (less work per entry)
#endif
#ifndef SNK_PIPE_DX
#define SNK_PIPE_DX 1      // the same for the transposed product
#endif
#ifndef SNK_PIPE_DX16
#define SNK_PIPE_DX16 2    // the same at a 16-column tile (8 entries per warp step:
                           // 10000^2, 90%, b = 16: 109.6 -> 99.8 us; 1 or 3 elsewhere lose)
#endif
#ifndef SNK_GATHER_LEAD
#define SNK_GATHER_LEAD 1  // transposed product: blocks whose values are gathered ahead
#endif
#ifndef SNK_THREADS_DX
#define SNK_THREADS_DX SNK_THREADS  // block size of the transposed product
#endif
#ifndef SNK_PIPE_DW
#define SNK_PIPE_DW 4      // the same for the weight gradient
#endif
#ifndef SNK_PIPE_DW_NARROW
#define SNK_PIPE_DW_NARROW 6   // the same for tiles of 1 or 2 batch columns
#endif
#ifndef SNK_PIPE_DW_WIDE
#define SNK_PIPE_DW_WIDE 2     // the same for tiles of 8+ columns read from the transposed
                               // copy in global memory (99%, b = 64: 62.5 -> 57.2 us)
#endif
// (10000^2, b = 1: forward 19.4 -> 18.9 us at 90%; dW b = 1 / 2 at 90%
// 22.5 / 23.4 -> 21.3 / 22.6 us, at 95% b = 2 16.4 -> 15.2; the forward at
// b = 2 and the 99% layer do not gain.)
#ifndef SNK_IDX16
#define SNK_IDX16 1        // read 16-bit index copies on the shared-memory path
#endif
#ifndef SNK_SWEEP_PHASE_KB
#define SNK_SWEEP_PHASE_KB 96  // column sweep: shared memory per phase at a 4-column tile
#endif
#ifndef SNK_SWEEP_NS
#define SNK_SWEEP_NS 3     // column sweep: quads in flight per lane
#endif
#ifndef SNK_BANDS
#define SNK_BANDS 1        // dW: row runs over column bands for wide operands at batch tiles >= 8
#endif

constexpr int kThreads = SNK_THREADS;
constexpr int kWarpsPerBlock = kThreads / kWarp;
constexpr int kThreadsDx = SNK_THREADS_DX;
constexpr int kWarpsPerBlockDx = kThreadsDx / kWarp;
constexpr int kChunksPerSm = kWarpsPerBlock;   // merge-path chunks per SM (one per warp)
constexpr int kMaxBatchTile = 64;    // batch columns handled by one launch
constexpr int kStreamPad = 128;      // zero entries after library-owned streams

// Device status word bits.
constexpr int kStatRange = 1;
constexpr int kStatDup = 2;
constexpr int kStatLimit = 4;

struct RestructureWs;
struct PcsrState;
struct TcState;
struct Sweep;
struct Bands;

// Per block: its entry range [k0, k1), and for the segment that enters the
// block from before (head) and the one that leaves it (tail) the first and
// last block holding entries of that segment, with the number of non-empty
// blocks from there to this block (head) and from this block to there (tail).
struct BlockDesc {
    int k0, k1;
    int head_first, tail_last;
    int n_head, n_tail;
    int pad0, pad1;
};

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

    // work partition of the canonical (row) and column orders: one block per
    // SM owns a range of entries aligned to segment boundaries, split into one
    // chunk per warp
    int32_t n_blocks = 0;         // blocks (= SMs)
    int32_t n_chunks = 0;         // n_blocks * (warps per block of the larger kernel)
    int32_t* bnd_r = nullptr;     // [n_blocks+1] first entry of each block (rows)
    int32_t* bnd_c = nullptr;     // [n_blocks+1] the same (columns)
    int4* cdesc_r = nullptr;      // [n_chunks] (k0, k1, first segment touched, one past last)
    int4* cdesc_c = nullptr;      // [n_chunks]
    BlockDesc* bdesc_r = nullptr; // [n_blocks] segments cut by block boundaries
    BlockDesc* bdesc_c = nullptr; // [n_blocks]

    // scratch of the SpMM kernels
    float* part = nullptr;        // [n_blocks * 2 * kMaxBatchTile] cross-block partial sums
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
    PcsrState* pcsr = nullptr;    // Padded-CSR view, built on request
    TcState* tc = nullptr;        // tile-ordered views of the large-batch path, built on first use
    Sweep* sweep = nullptr;       // lane tables of the column sweep (snk_sweep.cu)
    Bands* bands = nullptr;       // dW's row-run tables over column bands (snk_band.cu), built on first use
};

void free_pcsr(Layer* L);

// ---- column sweep of the transposed product (snk_sweep.cu) ---------------
// Every column of a block gets its own lanes, as many as its share of the
// block's entries; see snk_sweep.cu for the tables' layout.
struct SweepView {
    const int4* blk;    // [2 n_blocks] (first col, end col, virtual lanes, first lane), (first col record, first global partial, head, tail)
    const int2* col;    // per block and column: (first virtual lane, lanes)
    const int4* lane;   // per virtual lane: (first quad, quad stride, first entry, end entry)
    const int* split;   // [phases - 1][n_lane]: 2 * resume quad (+1 if that quad straddles the row)
    int64_t n_lane;
    int phases;         // row phases of the tables (a power of two, at most 8)
    int rows;           // rows per phase (a multiple of 4)
    const int32_t* perm;   // the column view's slots and 16-bit rows, reordered within quads
    const uint16_t* r16;
};
int build_sweep(Layer* L, cudaStream_t s);
void mark_sweep(Layer* L);
void free_sweep(Layer* L);
bool sweep_view(const Layer* L, SweepView* v);

// ---- row runs over column bands (snk_band.cu) ------------------------------
// dW for a batch tile of bp >= 8 columns whose operand does not fit shared
// memory: each block stages one band of the transposed operand and walks the
// runs of its rows in that band.  *done says whether the layer took this path
// (false: no bands for it; the caller goes on).
int band_backward_weight(Layer* L, int bp, const float* X, const float* dY, int b, float* dW, bool accumulate,
                         const float* dY_all, int64_t b_all, float* db, cudaStream_t s, bool* done);
// The band count and width for a batch tile of bp columns; false when the
// layer takes no bands (operand fits, runs too short, or too few entries).
bool band_shape(const Layer* L, int bp, int* nb, int* width);
int refresh_bands(Layer* L, cudaStream_t s);
void mark_bands(Layer* L);
void free_bands(Layer* L);

// ---- large-batch path on the tensor cores (snk_tc.cu) ---------------------
bool tc_eligible(const Layer* L, int64_t b);
// Y[b, n_seg] = D[b, K] times the rows (columns = false) or the columns of W,
// + bias.  Allocates and builds the tile-ordered view on first use.
int run_tc(Layer* L, bool columns, const float* D, int64_t b, const float* bias, float* Y,
           cudaStream_t s);
// dW on the entries of W (and db = column sums of dY) for a large batch.
int run_tc_sddmm(Layer* L, const float* X, const float* dY, int64_t b, float* dW, float* db,
                 cudaStream_t s);
int refresh_tc_views(Layer* L, cudaStream_t s);

// The tensor path's fp16 split holds a value x of a row scaled by 2^e to
// within 2^-22 |x| while |x| 2^e >= 2^-3, and to an absolute 2^-25 * 2^-e
// below that (fp16's subnormal spacing).  Per row (or segment of W) the
// pre-passes record a code: bit 0 = it holds an inf or NaN, the bits above =
// how many nonzero values it holds below 2^-3 after scaling ("tiny").  The
// tiny values can add at most 2^-25 * 2^-e times the sum of the magnitudes
// they meet on the other side, which is at most the largest L1 norm there,
// and at most their count times the largest magnitude there.  The outputs are
// recomputed exactly on the CUDA cores when bit 0 is set, or when that bound
// exceeds kTcFloorBudget (a quarter of the 1e-6 absolute term of the
// tolerance; the other side gets another quarter).
constexpr float kTcFloorBudget = 2.5e-7f;
__device__ __forceinline__ bool tc_needs_exact(int code, int e, float other_l1, float other_max) {
    if (code & 1) return true;
    const int n = code >> 1;
    if (n == 0) return false;
    return ldexpf(fminf(other_l1, (float)n * other_max), -25 - e) > kTcFloorBudget;
}
// One side of W for the exact recomputation: segment o holds entries
// [ptr[o], ptr[o+1]) with operand index idx[j] and value val[perm[j]] (or
// val[j] when perm is null).
struct TcSide {
    const int32_t* ptr;
    const int32_t* idx;
    const int32_t* perm;
    const float* val;
};
// snk_tc_exact.cu: Y[rows[i], o] for every segment o (rows relative to D and
// Y), for i < *n_rows.
int launch_exact_rows(const TcSide& sd, int64_t n_seg, const float* D, int64_t K,
                      const float* bias, float* Y, const int32_t* rows, const uint32_t* n_rows,
                      int num_sms, cudaStream_t s);
// Y[beta, o] for every beta < b and every candidate segment o that
// tc_needs_exact confirms against other[0] (largest L1 norm of the dense rows)
// and other[1] (their largest magnitude), both fp32 bit patterns.
int launch_exact_segs(const TcSide& sd, int64_t n_seg, const float* D, int64_t K, int64_t b,
                      const float* bias, float* Y, const int32_t* cand, const uint32_t* n_cand,
                      const int32_t* seg_exp, const int32_t* seg_code, const uint32_t* other,
                      int num_sms, cudaStream_t s);
// dW for every entry of the listed rows (values below out) and columns
// (out + column) of W, over the whole batch.
int launch_exact_dw(const Layer* L, const float* X, const float* dY, int64_t b, float* dW,
                    const int32_t* list, const uint32_t* n_list, cudaStream_t s);
void mark_tc_views(Layer* L);
void free_tc(Layer* L);

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
// The rest of the build for a triple already in canonical order whose
// col_keys / col_vals hold (column, slot) of every entry.
int build_views(Layer* L, cudaStream_t s);

// Radix helpers reused by the restructure code.
int exclusive_scan_i32(const int32_t* in, int32_t* out, int64_t n, int32_t* tmp, int64_t tmp_len,
                       int32_t* total, cudaStream_t s);
int64_t scan_tmp_len(int64_t n);
int64_t topology_hist_len(int64_t n);
// Stable LSD radix sort of (key, value) pairs by the low total_bits of the
// key; the result is in the alternate buffers when *flipped.
int sort_pairs_u64(uint64_t* keys, uint32_t* vals, uint64_t* keys_alt, uint32_t* vals_alt, int64_t n,
                   int total_bits, int32_t* hist, int64_t hist_len, cudaStream_t s, bool* flipped);
int sort_pairs_u32(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt, int64_t n,
                   int total_bits, int32_t* hist, int64_t hist_len, cudaStream_t s, bool* flipped);

// ---- kernels launched by the API ----------------------------------------
int launch_forward(Layer* L, const float* X, int64_t b, const float* bias, float* Y,
                   cudaStream_t s);
int launch_backward_input(Layer* L, const float* dY, int64_t b, float* dX, cudaStream_t s);
int launch_backward_weight(Layer* L, const float* X, const float* dY, int64_t b, float* dW,
                           float* db, cudaStream_t s);
int run_prune_regrow(Layer* L, float zeta, uint64_t seed, cudaStream_t s);
int run_prune_regrow_gradient(Layer* L, float zeta, const float* X, const float* dY, int64_t b,
                              cudaStream_t s);
// Partition nnz entries with segment pointer ptr[n_seg+1] over n_blocks
// blocks of kWarpsPerBlock chunks (block boundaries on segment boundaries
// except inside segments longer than half a block's share).
int build_partition(const int32_t* ptr, int64_t n_seg, int64_t nnz, int n_blocks, int warps,
                    int32_t* bnd, int4* cdesc, BlockDesc* bdesc, cudaStream_t s);
int launch_forward_csr(const float* val, const int32_t* cols, const int32_t* row_ptr,
                       const int4* cdesc, const BlockDesc* bdesc, const int32_t* bnd, int64_t nnz,
                       int64_t out_f, int64_t in_f, int n_blocks, const float* X, int64_t b,
                       const float* bias, float* Y, float* part, int32_t* cnt, int max_smem,
                       cudaStream_t s);
// Shared memory one block of the forward product on a caller's CSR takes for
// an operand of in_f columns and a batch tile of bp columns.
size_t forward_csr_smem(int64_t in_f, int bp);
void free_restructure(Layer* L);

}  // namespace snk
