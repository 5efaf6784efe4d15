/*
 * snk.h - C ABI of libsnk, a truly sparse linear layer for NVIDIA GB300
 * (sm_103a).
 *
 * The weight W (out x in) exists only as its non-zeros, a COO triple
 * (values, rows, cols) in device memory.  The library computes
 *   forward            Y  = X W^T + b                      (SpMM)
 *   backward_input     dX = dY W                           (transposed SpMM)
 *   backward_weight    dW_k = sum_beta dY[beta,r_k] X[beta,c_k], db = 1^T dY
 *                      (the weight gradient on supp(W) only: an SDDMM)
 *   prune_regrow       magnitude prune of a fraction zeta, then a seeded
 *                      uniform regrow of as many new zero-valued entries
 *                      (nnz unchanged); prune_regrow_gradient grows at the
 *                      largest-|gradient| positions instead
 * with hand-written CUDA kernels.  The caller owns every buffer it passes;
 * the library owns only the workspace behind the handle.
 *
 * Sources (page titles; sections, figures and tables as printed there):
 *   [SNACK] "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural
 *           Networks on GPU"
 *   [PCSR]  "Padded-CSR: A sparse storage format for dynamic sparse training
 *           on CPU"
 *
 * Common conventions
 *   - Matrices are row-major fp32: X is [batch, in], Y and dY are
 *     [batch, out], dX is [batch, in] (the nn.Linear layout of [PCSR]
 *     sec. 2.2; [PCSR] sec. 6.1 writes the same product features-major).
 *   - Every pointer argument is a DEVICE pointer on the current CUDA device,
 *     to contiguous memory.  values/rows/cols and dW must be 16-byte
 *     aligned; X, Y, dY, dX, bias and db 4-byte aligned.  Violations return
 *     SNK_ERR_ARG before any work is queued.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous on that stream unless said otherwise.
 *   - Outputs are overwritten, never accumulated into.  batch == 0 is a
 *     no-op that returns SNK_OK.
 *   - A handle is used by one stream at a time; calls on one handle that
 *     overlap on the GPU race on its workspace.
 *   - snk_forward, snk_backward_input and snk_backward_weight only enqueue
 *     kernels (no allocation, no host synchronisation), and their kernels
 *     leave the handle's scratch as they found it.  They may therefore be
 *     captured into a CUDA graph (the inference-latency mode); a replay gives
 *     the same bits as a direct call.  A graph stays valid across
 *     snk_prune_regrow (nnz and the workspace addresses do not change) and
 *     becomes invalid at snk_destroy.  The exceptions are the first call
 *     of each product on the large-batch path (below), and the first
 *     snk_backward_weight at each batch tile of 8, 16, 32 or 64 columns that
 *     runs on column bands (an X too wide for shared memory, in <= 65536,
 *     and runs of 40 entries or more on average): each allocates its
 *     workspace and builds its table, so capture after one such call.  The
 *     band tables, like the large-batch views, are rebuilt in place by
 *     snk_prune_regrow.
 *   - Nothing crosses the ABI as an exception; every entry point returns a
 *     status code (snk_status_string gives its text).
 *   - Limits: 1 <= out, in <= 2^31 - 1; 0 <= nnz <= min(out*in, 2^31 - 1);
 *     out*in < 2^63.
 *   - Numerics: fp32 products accumulated in fp32 with at least 32 partial
 *     sums per output reduced by a tree (dX at batch <= 4: each lane of an
 *     output column keeps two running sums, folds them into its partial every
 *     16 terms, and the column adds its lanes' partials 32 at a time), so that
 *     each output y satisfies |y - exact| <= 1e-5 * A + 1e-6 with A the sum
 *     of |terms| (+|bias|).  The order of every sum is fixed by the topology:
 *     repeated calls give the same bits.
 *
 * Large batches ([SNACK] appendix Table 13 trains at batch 4096)
 *   - From batch 96 when at least 5% of W is stored, from batch 192 when at
 *     least 1/34 (2.9%) is, from batch 256 when at least 2% is, and from
 *     batch 512 when at least 1% is, the three product calls run on the
 *     tensor cores instead of 64-row batch tiling.  W is
 *     densified tile by tile in shared memory (never in device memory) and
 *     multiplied with the dense operand.  The environment variable
 *     SNK_LARGE_BATCH=on|off forces the choice for every batch size.
 *   - Numerics: the same contract as above, for every input.  Every operand
 *     row is scaled by a power of two and split into two fp16 pieces.  The
 *     three products hi*hi, hi*lo and lo*hi carry about 22 bits.  The tensor
 *     core's fp32 accumulation truncates, so it is never chained over more
 *     than 8 windows of 64 terms (96 MMA steps); the partial results are
 *     added in fp32 with round-to-nearest.  The error stays inside the bound
 *     above even when every term has the same sign (about 4e-6 * A then).
 *   - Inputs the split cannot carry are found by the per-call passes and
 *     their outputs recomputed per stored entry on the CUDA cores (fp32, 32
 *     partial sums and a tree, as in the batch-tiled kernels): a row of X
 *     (dY) or a row / column of W holding an inf or NaN (a densified tile
 *     would otherwise spread NaN over a whole output row or column, where the
 *     definition gives NaN or +-inf only at the outputs an entry reaches), and
 *     a row or segment whose values span more than about 2^16 when the fp16
 *     floor of its small values could reach a quarter of the 1e-6 term.
 *     Ordinary data (values within a few orders of magnitude of each other)
 *     triggers neither; each call then costs three more small launches.
 *   - Memory, allocated on the first such call and kept until snk_destroy:
 *     about 22 bytes per stored entry (three tile-ordered views of 6 bytes
 *     and a 4-byte fp16 value pair), plus 32 KB per row or column of the
 *     larger dimension (fp16 pieces of 8192 dense rows; larger batches run
 *     in chunks of that size).  An allocation failure returns SNK_ERR_OOM.
 */
#ifndef SNK_H
#define SNK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SNK_OK 0          /* success                                          */
#define SNK_ERR_ARG 1     /* bad shape, null or misaligned pointer, bad zeta   */
#define SNK_ERR_DUP 2     /* the triple holds the same (row, col) twice        */
#define SNK_ERR_RANGE 3   /* a row or column index lies outside the matrix     */
#define SNK_ERR_CUDA 4    /* a CUDA call or kernel launch failed               */
#define SNK_ERR_OOM 5     /* workspace allocation failed                       */
#define SNK_ERR_NOSPACE 6 /* fewer free positions than entries to regrow       */
#define SNK_ERR_LIMIT 7   /* a limit was reached: regrow draws (64 k + 1024),  */
                          /* or the fixed scratch of the allocation-free call */

typedef struct snk_layer* snk_handle;

/*
 * snk_create - bind a layer to a caller-owned COO triple and build its
 * topology.
 *   [SNACK] Fig. 1: the weight is stored on the GPU as the COO triple over its
 *   non-zeros only.  [PCSR] sec. 3.2 / 4.1: entries sorted by row, then by
 *   column within a row, with a row pointer.  [SNACK] Table 7 and [PCSR]
 *   sec. 7.2: the column-sorted (CSC) view and the permutation map that
 *   gathers values into column order, built once per topology.
 *
 * handle   out: the new handle (unchanged on error).
 * out_features, in_features: W is out_features x in_features.
 * nnz      number of stored entries.
 * values, rows, cols: device arrays of nnz fp32 / int32 / int32 in any order.
 *          They are sorted IN PLACE into canonical order (by row, then
 *          column) and BORROWED for the life of the handle: the caller keeps
 *          them allocated, may update `values` between calls (e.g. an SGD
 *          step), and must not modify `rows` or `cols`.
 * stream   queue for the build.  The call synchronises the stream before it
 *          returns, so that device-detected errors can be reported.
 * Device memory taken by the handle: about 52 bytes per stored entry (index
 *          views, 16-bit copies, sort scratch) plus about 264 bytes per row or
 *          column of the larger dimension (pointers, arrival counters, and the
 *          transposed operand copy of the global-memory path, 64 batch columns
 *          wide); the first snk_prune_regrow adds its own workspace (about 100
 *          bytes per entry, plus a bitmap of out * in bits when that is at
 *          most 2^31 bits).
 * Errors:  SNK_ERR_ARG, SNK_ERR_RANGE (an index outside the matrix),
 *          SNK_ERR_DUP (a repeated position), SNK_ERR_OOM, SNK_ERR_CUDA.  On
 *          SNK_ERR_RANGE / SNK_ERR_DUP the caller's arrays are left as given.
 */
int snk_create(snk_handle* handle, int64_t out_features, int64_t in_features, int64_t nnz,
               float* values, int32_t* rows, int32_t* cols, void* stream);

/*
 * snk_forward - Y = X W^T + bias over supp(W) only.
 *   [SNACK] Fig. 1 (the forward pass computed directly on the triple);
 *   [PCSR] sec. 6.1 (for each live entry, scale the matching input and add
 *   it to the output row).
 * X     [batch, in] input.   bias  [out] or NULL (then no bias term).
 * Y     [batch, out] output; a row of W with no entries yields bias (or 0).
 * Errors: SNK_ERR_ARG, SNK_ERR_CUDA.
 */
int snk_forward(snk_handle handle, const float* X, int64_t batch, const float* bias, float* Y,
                void* stream);

/*
 * snk_backward_input - dX = dY W (the transposed SpMM).
 *   [PCSR] sec. 7.1 (dL/dX = W^T dL/dY in its features-major form, another
 *   SpMM) and sec. 7.2 (the transpose is read through the column-sorted view
 *   and the permutation built at create / restructure time; only the values
 *   are gathered per call).
 * dY    [batch, out] upstream gradient.
 * dX    [batch, in] output; a column of W with no entries yields 0.
 * Errors: SNK_ERR_ARG, SNK_ERR_CUDA.
 */
int snk_backward_input(snk_handle handle, const float* dY, int64_t batch, float* dX,
                       void* stream);

/*
 * snk_backward_weight - the weight gradient at live entries only (SDDMM),
 * and optionally the bias gradient.
 *   [PCSR] sec. 7.1 (dL/dW only at live slots: a dot product of the dL/dY row
 *   with the X row for each live entry); [SNACK] Fig. 1 (the backward pass as
 *   a sparse outer product over supp(W)).  db = sum over the batch of dY, the
 *   plain gradient of the bias (not on the pages).
 * X, dY as above.
 * dW    [nnz] output in canonical order: dW[k] belongs to (rows[k], cols[k]).
 * db    [out] output or NULL.
 * Errors: SNK_ERR_ARG, SNK_ERR_CUDA.
 */
int snk_backward_weight(snk_handle handle, const float* X, const float* dY, int64_t batch,
                        float* dW, float* db, void* stream);

/*
 * snk_prune_regrow - one dynamic-sparse-training restructure, nnz fixed.
 *   [PCSR] sec. 4.3 (drop a fraction of the live entries, grow the same
 *   number elsewhere), sec. 1.1 (prune by smallest magnitude), sec. 8.2 (SET
 *   with a drop fraction); [SNACK] Fig. 1 (connections added or dropped in
 *   place).  The pages give no order of ties and no generator; this library
 *   fixes them as follows.
 *   Prune: k = floor((double)zeta * nnz) entries with the smallest keys
 *     (bit pattern of |value|, row*in + col) are removed.
 *   Regrow: positions p_t = floor(z_t * out*in / 2^64), z_t the t-th output
 *     (t = 0, 1, ...) of SplitMix64 started at state `seed`, are accepted in
 *     draw order when not held by a kept entry nor accepted before, until k
 *     are accepted.  New entries get value +0.0f.  A position pruned in this
 *     call may be drawn again.
 *   The whole triple is then re-emitted in canonical order into the caller's
 *   values/rows/cols, and the topology is rebuilt.
 * zeta  in [0, 1).   seed  any 64-bit value.
 * The call synchronises the stream (it reads device counts back).
 * Errors: SNK_ERR_ARG (zeta outside [0,1)), SNK_ERR_NOSPACE (fewer than k
 *   free positions, found before any work), SNK_ERR_LIMIT (fewer than k
 *   positions accepted after 64 k + 1024 draws), SNK_ERR_OOM, SNK_ERR_CUDA.
 *   On every error the caller's arrays and the topology are left unchanged.
 */
int snk_prune_regrow(snk_handle handle, float zeta, uint64_t seed, void* stream);

/*
 * snk_prune_regrow_gradient - one RigL-style restructure, nnz fixed: the same
 * magnitude prune as snk_prune_regrow, then growth at the positions with the
 * largest gradient magnitude instead of random ones.
 *   [PCSR] sec. 4.3 (the typical dynamic-sparse-training update, e.g. RigL:
 *   drop a fraction of the live entries, grow as many "at high-gradient
 *   locations"); [SNACK] Tables 8-9 (RigL trained with the truly sparse
 *   layer).  The pages fix no arithmetic or tie order; this library fixes:
 *   Gradient of position (r, c): g = sum over beta of dY[beta, r] * X[beta, c],
 *     evaluated in fp32 as the fused multiply-add chain
 *     g = fma(dY[b-1,r], X[b-1,c], ... fma(dY[0,r], X[0,c], 0.0f)).
 *   Candidates: every position not held by a kept entry (a position pruned in
 *     this call is a candidate, as in snk_prune_regrow).
 *   Grown: the k candidates with the largest bit pattern of |g| (NaN above
 *     every number), ties going to the smaller r*in + c.  New values +0.0f.
 *   The whole triple is then re-emitted in canonical order and the topology
 *   rebuilt.  No out x in array is ever stored.
 * X [batch, in], dY [batch, out]: the batch whose gradient ranks the
 *   candidates (device, row-major fp32, 4-byte aligned); batch >= 1.
 * zeta in [0, 1).  Limits: out * in <= 2^32.
 * The call synchronises the stream (it reads device counts back).
 * Errors: SNK_ERR_ARG, SNK_ERR_NOSPACE, SNK_ERR_LIMIT (out * in > 2^32),
 *   SNK_ERR_OOM, SNK_ERR_CUDA.  On every error the caller's arrays and the
 *   topology are left unchanged.
 */
int snk_prune_regrow_gradient(snk_handle handle, float zeta, const float* X, const float* dY,
                              int64_t batch, void* stream);

/*
 * Padded-CSR view ([PCSR] sec. 5), for dynamic sparse training whose per-row
 * counts change.  A library-owned copy of the layer in the six arrays of
 * [PCSR] sec. 5.1: slot values and column indices (column -1 marks a padding
 * slot, value 0), row_start, row_nnz (a row's live slots come first in its
 * region), row_capacity, and a version counter.  The view is taken from the
 * handle's triple by snk_pcsr_build and is independent of it afterwards:
 * mutations of the view reach a layer through snk_pcsr_export (a canonical
 * triple for a new handle), and restructures of the handle do not reach the
 * view.  Readings fixed by this library where the page is silent:
 *   - padding is a whole percentage p: capacity(n) = max(1, ceil(n*(100+p)/100))
 *     in integers ([PCSR] sec. 5.2's 0.2 is p = 20);
 *   - an insert batch first moves every row whose live count plus inserts
 *     exceeds its capacity, in ascending row order, to fresh slots at the end
 *     of the used slot area with capacity(live + inserts); the old slots become
 *     padding ([PCSR] sec. 4.3's resize); then each insert takes the next slot
 *     of its row in batch order ([PCSR] sec. 5.3: O(1) per insert);
 *   - a delete batch clears the slots and each touched row closes up, its
 *     remaining live entries keeping their order;
 *   - compact ([PCSR] sec. 8.3's compact_all) lays all rows out again from
 *     slot 0, row by row, capacity(live) each, columns ascending.
 *   - the version starts at 1 and goes up by one per applied insert batch,
 *     delete batch and compact.
 * Slot indices are int32: at most 2^31 - 1 slots.  All pointers are device
 * pointers; calls synchronise the stream (they read counts back).
 */

/* Build (or rebuild) the view from the handle's current triple, padding p %
 * (0 <= p <= 10000).  Errors: SNK_ERR_ARG, SNK_ERR_OOM, SNK_ERR_LIMIT, SNK_ERR_CUDA. */
int snk_pcsr_build(snk_handle handle, int padding_pct, void* stream);

/* Slots in use (the end of the last row region), live entries and version;
 * any output may be NULL.  Errors: SNK_ERR_ARG (no view), SNK_ERR_CUDA. */
int snk_pcsr_info(snk_handle handle, int64_t* used_slots, int64_t* n_live, int64_t* version,
                  void* stream);

/* Copy the view out: slot_values / slot_cols [used_slots], row_start, row_nnz,
 * row_capacity [out]; any may be NULL.  Asynchronous. */
int snk_pcsr_copy(snk_handle handle, float* slot_values, int32_t* slot_cols, int32_t* row_start,
                  int32_t* row_nnz, int32_t* row_capacity, void* stream);

/* Insert n entries (rows[i], cols[i], values[i]).  The positions must not be
 * live (a repeat is reported by snk_pcsr_compact / snk_pcsr_export as
 * SNK_ERR_DUP).  Errors: SNK_ERR_ARG, SNK_ERR_RANGE (an index outside the
 * matrix; nothing changed), SNK_ERR_OOM, SNK_ERR_LIMIT, SNK_ERR_CUDA. */
int snk_pcsr_insert(snk_handle handle, int64_t n, const int32_t* rows, const int32_t* cols,
                    const float* values, void* stream);

/* Delete the n live entries at (rows[i], cols[i]).  Errors: SNK_ERR_RANGE (an
 * index outside the matrix), SNK_ERR_ARG (a position that is not live); on
 * either nothing changed. */
int snk_pcsr_delete(snk_handle handle, int64_t n, const int32_t* rows, const int32_t* cols,
                    void* stream);

/* compact_all: lay the view out again from slot 0 with fresh padding and
 * columns ascending.  Errors: SNK_ERR_DUP (a position held twice; nothing
 * changed), SNK_ERR_OOM, SNK_ERR_CUDA. */
int snk_pcsr_compact(snk_handle handle, void* stream);

/* Write the live entries as a canonical COO triple (row-major, columns
 * ascending) into values / rows / cols of the given capacity; *nnz_out gets
 * the count (also when it exceeds capacity, which returns SNK_ERR_LIMIT and
 * writes nothing).  The triple can be bound to a new handle with snk_create.
 * Errors: SNK_ERR_ARG, SNK_ERR_LIMIT, SNK_ERR_DUP, SNK_ERR_CUDA. */
int snk_pcsr_export(snk_handle handle, float* values, int32_t* rows, int32_t* cols,
                    int64_t capacity, int64_t* nnz_out, void* stream);

/*
 * snk_destroy - free the library-owned workspace (never the caller's arrays).
 * NULL is accepted.  Waits for work queued on the handle's device.
 */
int snk_destroy(snk_handle handle);

/* Text of a status code (static storage). */
const char* snk_status_string(int status);

/*
 * snk_check - report a stopped product kernel.  The tensor-core kernels of
 * the large-batch path (above) bound every wait of their pipeline (about two
 * seconds).  A wait that runs out stops that kernel: it waits for the copies
 * and tensor-core operations it has already issued, writes NaN to every
 * output it owns (Y or dX entries, or the dW entries of its blocks of W:
 * a weight-gradient warp whose wait ran out writes NaN to its share of the
 * CTA's current block and of every later one), and
 * records the event in the handle's device status word.  The product calls
 * are asynchronous and cannot return that record themselves; this call
 * synchronises `stream`, reads the word and clears it.  No page has a
 * counterpart; it is part of the library's failure handling.
 * Returns SNK_ERR_LIMIT if such a stop happened since the last snk_check
 * (or since snk_create), SNK_OK if not; SNK_ERR_ARG, SNK_ERR_CUDA.
 */
int snk_check(snk_handle handle, void* stream);

/*
 * snk_get_shape - sizes and the topology version of a handle.  The version
 * starts at 1 and grows by one at each restructure that changes the support
 * ([PCSR] sec. 5.1, the topology_version counter).  Any output may be NULL.
 */
int snk_get_shape(snk_handle handle, int64_t* out_features, int64_t* in_features, int64_t* nnz,
                  int64_t* topology_version);

/*
 * snk_copy_topology - copy the derived index arrays to caller device buffers
 * (any may be NULL): row_ptr [out+1], col_ptr [in+1], rows_c [nnz] (row of the
 * j-th entry in column order) and perm [nnz] (its canonical slot, so values
 * in column order are values[perm]).  [SNACK] Table 7; [PCSR] sec. 7.2.
 * Asynchronous on `stream`.
 */
int snk_copy_topology(snk_handle handle, int32_t* row_ptr, int32_t* col_ptr, int32_t* rows_c,
                      int32_t* perm, void* stream);

/*
 * snk_forward_csr_noalloc - the forward product Y = X W^T + bias for callers
 * that cannot let the library allocate device memory.  The pages have no
 * counterpart to this entry point.
 *
 * Who needs it: a program whose device memory is owned entirely by its own
 * arena, or whose hot path must never reach cudaMalloc/cudaFree (they
 * synchronise the device and can stall other streams, and an allocation
 * failure there cannot be handled).  Such a caller cannot use snk_create,
 * which allocates the layer's workspace; this call takes the matrix as a
 * ready CSR and allocates nothing.
 *
 * Arguments (device pointers on the current device):
 *   row_ptr [out+1]  CSR row pointer (row_ptr[0] = 0, non-decreasing,
 *                    row_ptr[out] = nnz), 4-byte aligned;
 *   cols [nnz], values [nnz]  column index and value of each entry, rows
 *                    stored one after another, 16-byte aligned;
 *   X [batch, in], bias [out] or NULL, Y [batch, out]  as for snk_forward.
 * The CSR is not validated: indices must lie in range (snk_create is the
 * validating path).
 * Scratch: a fixed array inside the library image (2,574,352 bytes per GPU,
 * held for the life of the process).  Limits: out <= 524,288, at most 512
 * SMs, and the operand, in * (batch rounded up to a power of two, at most
 * 64) * 4 bytes, together with the kernel's per-warp partial sums (about
 * 12.5 KB at a batch of 64) must fit one block's shared memory; larger
 * requests return SNK_ERR_LIMIT before any work is queued.  Every call shares the scratch and starts by clearing
 * the part it needs; calls whose kernels overlap on the GPU (other streams or
 * threads) race on it and must be serialised by the caller.
 * The first call on a device looks the scratch address up (once per device,
 * with that device current); make that first call before any stream
 * capture.
 * Errors: SNK_ERR_ARG, SNK_ERR_LIMIT, SNK_ERR_CUDA.  Asynchronous on stream.
 */
int snk_forward_csr_noalloc(int64_t out_features, int64_t in_features, int64_t nnz,
                            const int32_t* row_ptr, const int32_t* cols, const float* values,
                            const float* X, int64_t batch, const float* bias, float* Y,
                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SNK_H */
