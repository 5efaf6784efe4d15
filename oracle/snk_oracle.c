/*
 * snk_oracle.c - plain CPU oracle for the truly sparse linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * cpu_baseline / reference leg of the benchmark load this code.  The CUDA
 * library never does, and the two share no source, header, table or helper.
 *
 * What it computes, and where the pages define it:
 *   [SNACK] "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural
 *           Networks on GPU" - Fig. 1 (the weight kept only as the COO triple
 *           (values, rows, cols); forward on the triple; backward as a sparse
 *           outer product over supp(W); connections added or dropped in place),
 *           Table 7 (COO, CSR and CSC of one small matrix).
 *   [PCSR]  "Padded-CSR: A sparse storage format for dynamic sparse training
 *           on CPU" - sec. 3.1/3.2/4.1 (COO, row pointer, CSR), sec. 4.3 (a DST
 *           update drops a fraction of live entries and grows as many new
 *           ones elsewhere), sec. 6.1 (what the SpMM computes), sec. 7.1 (the
 *           two gradients; dL/dW only at live slots), sec. 7.2 (transpose via a
 *           per-column count and a scatter, with a permutation map).
 *
 * Orientation: W is out x in, X is [b, in], Y and dY are [b, out], all
 * row-major, the nn.Linear convention ([PCSR] sec. 2.2).  [PCSR] sec. 6.1 writes
 * the same product features-major (Y = W @ X); the arithmetic is identical.
 *
 * Precision: every sum is accumulated in double, one term at a time, in the
 * order of the triple as given.  There is no blocking, fusion or reordering.
 * Next to each output the oracle also accumulates the magnitude sum
 * A = sum |term| (plus |bias|), which fixes the fp32 tolerance of a faster
 * implementation: |y - y_oracle| <= 1e-5 * A + 1e-6.
 *
 * Procedural parts (canonical order, prune, regrow) follow the steps in the
 * order the pages give them; where the pages leave a step open the plainest
 * reading is taken and named at the function.
 *
 * The gradient grow ([PCSR] sec. 4.3, RigL: grow "at high-gradient
 * locations") ranks positions by an fp32 value, so here, where floating point
 * decides which integers are chosen, the oracle takes the decision in the
 * same precision as the library: each gradient is the fp32 fused
 * multiply-add chain over the batch in order (C99 fmaf, correctly rounded).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Multi-core build.  Built with -fopenmp, the three products split their    */
/* OUTPUTS among threads, in the spirit of [PCSR] sec. 6.3's static split of */
/* rows over cores: each thread owns a contiguous block of output rows       */
/* (forward) or columns (input gradient), walks the whole triple in the      */
/* given order and skips entries whose output it does not own; the weight    */
/* gradient's entries are independent and are split statically.  Every      */
/* output therefore receives the same terms in the same order as in the      */
/* single-threaded build, so both builds give identical bits.  Without      */
/* OpenMP there is one block holding every output.                          */
/* ------------------------------------------------------------------------ */
static void orc_my_block(int64_t n, int64_t* lo, int64_t* hi) {
#ifdef _OPENMP
    const int64_t nt = omp_get_num_threads(), t = omp_get_thread_num();
    *lo = n * t / nt;
    *hi = n * (t + 1) / nt;
#else
    *lo = 0;
    *hi = n;
#endif
}

/* Threads the products use (1 in the single-threaded build). */
int orc_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

enum {
    ORC_OK = 0,
    ORC_ERR_ARG = 1,
    ORC_ERR_DUP = 2,
    ORC_ERR_RANGE = 3,
    ORC_ERR_OOM = 5,
    ORC_ERR_NOSPACE = 6,
    ORC_ERR_LIMIT = 7
};

/* ------------------------------------------------------------------------ */
/* Canonical order: sort by (row, col), i.e. by lin = row * in + col.        */
/* [PCSR] sec. 3.2 ("sort the entries by row") and sec. 4.1 (values stored    */
/* row by row, sorted by column within each row).  Duplicates and indices    */
/* outside the matrix are rejected: the pages never store either.           */
/* ------------------------------------------------------------------------ */

typedef struct {
    uint64_t lin;
    float v;
} orc_entry;

static int orc_cmp_entry(const void* a, const void* b) {
    const orc_entry* x = (const orc_entry*)a;
    const orc_entry* y = (const orc_entry*)b;
    return (x->lin > y->lin) - (x->lin < y->lin);
}

/*
 * Sort the triple in place into canonical order and, when the output arrays
 * are given, build
 *   row_ptr[out+1]  CSR row pointer ([PCSR] sec. 3.2, 4.1),
 *   col_ptr[in+1]   CSC column pointer ([SNACK] Table 7 "CSC ... indptr"),
 *   rows_c[nnz]     row of the j-th entry in column order ([SNACK] Table 7),
 *   perm[nnz]       canonical slot of the j-th entry in column order, so that
 *                   values-in-column-order = values[perm] ([PCSR] sec. 7.2).
 * The column order is a count per column followed by a scatter that walks the
 * canonical order, which is the two-pass transpose of [PCSR] sec. 7.2; being
 * a stable scatter it leaves rows ascending within each column.
 * Returns ORC_ERR_RANGE / ORC_ERR_DUP without touching the arrays.
 */
int orc_canonicalize(int64_t out_f, int64_t in_f, int64_t nnz,
                     float* v, int32_t* r, int32_t* c,
                     int32_t* row_ptr, int32_t* col_ptr,
                     int32_t* rows_c, int32_t* perm) {
    if (out_f <= 0 || in_f <= 0 || nnz < 0) return ORC_ERR_ARG;
    for (int64_t k = 0; k < nnz; ++k) {
        if (r[k] < 0 || (int64_t)r[k] >= out_f || c[k] < 0 || (int64_t)c[k] >= in_f)
            return ORC_ERR_RANGE;
    }
    orc_entry* e = (orc_entry*)malloc(sizeof(orc_entry) * (size_t)(nnz > 0 ? nnz : 1));
    if (!e) return ORC_ERR_OOM;
    for (int64_t k = 0; k < nnz; ++k) {
        e[k].lin = (uint64_t)r[k] * (uint64_t)in_f + (uint64_t)c[k];
        e[k].v = v[k];
    }
    qsort(e, (size_t)nnz, sizeof(orc_entry), orc_cmp_entry);
    for (int64_t k = 1; k < nnz; ++k) {
        if (e[k].lin == e[k - 1].lin) {
            free(e);
            return ORC_ERR_DUP;
        }
    }
    for (int64_t k = 0; k < nnz; ++k) {
        v[k] = e[k].v;
        r[k] = (int32_t)(e[k].lin / (uint64_t)in_f);
        c[k] = (int32_t)(e[k].lin % (uint64_t)in_f);
    }
    free(e);

    if (row_ptr) {
        for (int64_t i = 0; i <= out_f; ++i) row_ptr[i] = 0;
        for (int64_t k = 0; k < nnz; ++k) row_ptr[r[k] + 1] += 1;
        for (int64_t i = 0; i < out_f; ++i) row_ptr[i + 1] += row_ptr[i];
    }
    if (col_ptr) {
        for (int64_t j = 0; j <= in_f; ++j) col_ptr[j] = 0;
        for (int64_t k = 0; k < nnz; ++k) col_ptr[c[k] + 1] += 1;
        for (int64_t j = 0; j < in_f; ++j) col_ptr[j + 1] += col_ptr[j];
        if (rows_c || perm) {
            int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)in_f);
            if (!next) return ORC_ERR_OOM;
            for (int64_t j = 0; j < in_f; ++j) next[j] = col_ptr[j];
            for (int64_t k = 0; k < nnz; ++k) {
                int32_t pos = next[c[k]]++;
                if (perm) perm[pos] = (int32_t)k;
                if (rows_c) rows_c[pos] = r[k];
            }
            free(next);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* S2 forward:  Y[beta, o] = bias[o] + sum_{k: r_k = o} v_k * X[beta, c_k]  */
/* [SNACK] Fig. 1 (forward on the COO triple); [PCSR] sec. 6.1 (for each live */
/* entry, scale the matching row of X by the value and add it to the output  */
/* row).  The loop walks the triple as given; empty rows keep the bias.      */
/* ------------------------------------------------------------------------ */
void orc_forward(int64_t out_f, int64_t in_f, int64_t nnz,
                 const float* v, const int32_t* r, const int32_t* c,
                 const float* X, int64_t b, const float* bias,
                 double* Y, double* A) {
    for (int64_t beta = 0; beta < b; ++beta) {
        for (int64_t o = 0; o < out_f; ++o) {
            double bo = bias ? (double)bias[o] : 0.0;
            Y[beta * out_f + o] = bo;
            if (A) A[beta * out_f + o] = fabs(bo);
        }
    }
#pragma omp parallel
    {
        int64_t o0, o1;
        orc_my_block(out_f, &o0, &o1);
        for (int64_t k = 0; k < nnz; ++k) {
            if (r[k] < o0 || r[k] >= o1) continue;
            double w = (double)v[k];
            for (int64_t beta = 0; beta < b; ++beta) {
                double x = (double)X[beta * in_f + c[k]];
                Y[beta * out_f + r[k]] += w * x;
                if (A) A[beta * out_f + r[k]] += fabs(w * x);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* S3 input gradient:  dX = dY . (W (.) M),  dX[beta, i] =                    */
/*   sum_{k: c_k = i} v_k * dY[beta, r_k].                                   */
/* [PCSR] sec. 7.1 (dL/dX = W^T dL/dY, another SpMM).  Empty columns give 0.  */
/* ------------------------------------------------------------------------ */
void orc_backward_input(int64_t out_f, int64_t in_f, int64_t nnz,
                        const float* v, const int32_t* r, const int32_t* c,
                        const float* dY, int64_t b, double* dX, double* A) {
    for (int64_t q = 0; q < b * in_f; ++q) {
        dX[q] = 0.0;
        if (A) A[q] = 0.0;
    }
#pragma omp parallel
    {
        int64_t i0, i1;
        orc_my_block(in_f, &i0, &i1);
        for (int64_t k = 0; k < nnz; ++k) {
            if (c[k] < i0 || c[k] >= i1) continue;
            double w = (double)v[k];
            for (int64_t beta = 0; beta < b; ++beta) {
                double g = (double)dY[beta * out_f + r[k]];
                dX[beta * in_f + c[k]] += w * g;
                if (A) A[beta * in_f + c[k]] += fabs(w * g);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* S4 weight gradient on the support only:                                   */
/*   dW_k = sum_beta dY[beta, r_k] * X[beta, c_k]        (one per live entry) */
/*   db[o] = sum_beta dY[beta, o]                                            */
/* [PCSR] sec. 7.1 (dL/dW computed only at live slots, a dot product of the   */
/* dL/dY row with the X row); [SNACK] Fig. 1 (sparse outer product over       */
/* supp(W)).  The bias gradient is not on the pages; it is the plain          */
/* gradient of Y = X W^T + b with respect to b.                              */
/* ------------------------------------------------------------------------ */
void orc_backward_weight(int64_t out_f, int64_t in_f, int64_t nnz,
                         const int32_t* r, const int32_t* c,
                         const float* X, const float* dY, int64_t b,
                         double* dW, double* A_dW, double* db, double* A_db) {
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < nnz; ++k) {
        double s = 0.0, a = 0.0;
        for (int64_t beta = 0; beta < b; ++beta) {
            double t = (double)dY[beta * out_f + r[k]] * (double)X[beta * in_f + c[k]];
            s += t;
            a += fabs(t);
        }
        dW[k] = s;
        if (A_dW) A_dW[k] = a;
    }
    if (db) {
        for (int64_t o = 0; o < out_f; ++o) {
            double s = 0.0, a = 0.0;
            for (int64_t beta = 0; beta < b; ++beta) {
                double t = (double)dY[beta * out_f + o];
                s += t;
                a += fabs(t);
            }
            db[o] = s;
            if (A_db) A_db[o] = a;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* S5 magnitude prune.                                                       */
/* [PCSR] sec. 1.1 (prune the smallest-magnitude weights) and sec. 4.3 (drop  */
/* a fraction of the live entries); [PCSR] sec. 8.2 (drop_fraction).          */
/* Readings where the pages are silent:                                      */
/*   - the count is k = floor(zeta * nnz), computed in double;               */
/*   - the order is by (|v| as its IEEE-754 bit pattern, lin), ascending, so */
/*     equal magnitudes are broken by position, -0.0 and +0.0 tie, and a NaN */
/*     ranks above +inf;                                                     */
/*   - the k smallest keys are removed.                                      */
/* ------------------------------------------------------------------------ */
int64_t orc_prune_count(float zeta, int64_t nnz) {
    return (int64_t)floor((double)zeta * (double)nnz);
}

static uint32_t orc_abs_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u & 0x7fffffffu;
}

typedef struct {
    uint32_t mag;
    uint64_t lin;
    int64_t slot;
} orc_key;

static int orc_cmp_key(const void* a, const void* b) {
    const orc_key* x = (const orc_key*)a;
    const orc_key* y = (const orc_key*)b;
    if (x->mag != y->mag) return (x->mag > y->mag) - (x->mag < y->mag);
    return (x->lin > y->lin) - (x->lin < y->lin);
}

/* removed[k] = 1 for each of the k entries with the smallest keys. */
int orc_prune(int64_t out_f, int64_t in_f, int64_t nnz,
              const float* v, const int32_t* r, const int32_t* c,
              float zeta, uint8_t* removed, int64_t* k_out) {
    (void)out_f;
    if (!(zeta >= 0.0f && zeta < 1.0f)) return ORC_ERR_ARG;
    int64_t k = orc_prune_count(zeta, nnz);
    orc_key* keys = (orc_key*)malloc(sizeof(orc_key) * (size_t)(nnz > 0 ? nnz : 1));
    if (!keys) return ORC_ERR_OOM;
    for (int64_t i = 0; i < nnz; ++i) {
        keys[i].mag = orc_abs_bits(v[i]);
        keys[i].lin = (uint64_t)r[i] * (uint64_t)in_f + (uint64_t)c[i];
        keys[i].slot = i;
        removed[i] = 0;
    }
    qsort(keys, (size_t)nnz, sizeof(orc_key), orc_cmp_key);
    for (int64_t i = 0; i < k; ++i) removed[keys[i].slot] = 1;
    free(keys);
    if (k_out) *k_out = k;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* S6 seeded uniform regrow.                                                 */
/* [PCSR] sec. 4.3 (grow the same number of new entries elsewhere) and the    */
/* SET usage of sec. 8.2; [SNACK] Fig. 1 (connections added in place).        */
/* The pages give no generator.  Reading taken: draw t = 0, 1, 2, ...        */
/*   z_t = SplitMix64 output for state seed + (t+1) * 0x9E3779B97F4A7C15    */
/*         (Steele, Lea & Flood, "Fast splittable pseudorandom number         */
/*         generators", OOPSLA 2014; the mixing constants of its published   */
/*         reference form),                                                 */
/*   p_t = floor(z_t * N / 2^64), N = out * in (Lemire, "Fast random integer */
/*         generation in an interval", ACM TOMACS 2019, multiply-shift),      */
/* accept p_t when it is neither in the kept support nor already accepted,   */
/* stop at k accepted, and fail after 64 * k + 1024 draws.  New values are   */
/* +0.0f.  Positions pruned in the same step are eligible again.             */
/* ------------------------------------------------------------------------ */
#define ORC_GOLDEN_GAMMA 0x9E3779B97F4A7C15ull

uint64_t orc_splitmix64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* The n-th output (n = 0, 1, ...) of a SplitMix64 generator whose state
 * starts at `state`: the state is advanced by the golden gamma, then mixed. */
uint64_t orc_splitmix64_nth(uint64_t state, uint64_t n) {
    return orc_splitmix64_mix(state + (n + 1) * ORC_GOLDEN_GAMMA);
}

uint64_t orc_mulhi64(uint64_t a, uint64_t b) {
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    return (uint64_t)(p >> 64);
}

uint64_t orc_candidate(uint64_t seed, uint64_t t, uint64_t n_positions) {
    return orc_mulhi64(orc_splitmix64_nth(seed, t), n_positions);
}

/* A plain open-addressing set of positions (membership only). */
typedef struct {
    uint64_t* slot;
    uint64_t mask;
} orc_set;

#define ORC_EMPTY UINT64_MAX

static int orc_set_init(orc_set* s, int64_t n) {
    uint64_t cap = 16;
    while (cap < (uint64_t)(2 * n + 16)) cap <<= 1;
    s->slot = (uint64_t*)malloc(sizeof(uint64_t) * cap);
    if (!s->slot) return ORC_ERR_OOM;
    for (uint64_t i = 0; i < cap; ++i) s->slot[i] = ORC_EMPTY;
    s->mask = cap - 1;
    return ORC_OK;
}

static uint64_t orc_set_home(const orc_set* s, uint64_t key) {
    return (key * ORC_GOLDEN_GAMMA >> 17) & s->mask;
}

static int orc_set_has(const orc_set* s, uint64_t key) {
    for (uint64_t i = orc_set_home(s, key);; i = (i + 1) & s->mask) {
        if (s->slot[i] == key) return 1;
        if (s->slot[i] == ORC_EMPTY) return 0;
    }
}

static void orc_set_add(orc_set* s, uint64_t key) {
    for (uint64_t i = orc_set_home(s, key);; i = (i + 1) & s->mask) {
        if (s->slot[i] == key) return;
        if (s->slot[i] == ORC_EMPTY) {
            s->slot[i] = key;
            return;
        }
    }
}

/* new_lin[0..k) receives the accepted positions in the order drawn;
 * *draws_out (if given) the number of draws used. */
int orc_regrow(int64_t out_f, int64_t in_f, int64_t n_kept,
               const int32_t* r_kept, const int32_t* c_kept,
               int64_t k, uint64_t seed, int64_t* new_lin, int64_t* draws_out) {
    uint64_t n_pos = (uint64_t)out_f * (uint64_t)in_f;
    if ((uint64_t)n_kept + (uint64_t)k > n_pos) return ORC_ERR_NOSPACE;
    orc_set s;
    if (orc_set_init(&s, n_kept + k) != ORC_OK) return ORC_ERR_OOM;
    for (int64_t i = 0; i < n_kept; ++i)
        orc_set_add(&s, (uint64_t)r_kept[i] * (uint64_t)in_f + (uint64_t)c_kept[i]);
    uint64_t t_max = 64ull * (uint64_t)k + 1024ull;
    int64_t got = 0;
    uint64_t t = 0;
    for (; t < t_max && got < k; ++t) {
        uint64_t p = orc_candidate(seed, t, n_pos);
        if (orc_set_has(&s, p)) continue;
        orc_set_add(&s, p);
        new_lin[got++] = (int64_t)p;
    }
    free(s.slot);
    if (draws_out) *draws_out = (int64_t)t;
    return got == k ? ORC_OK : ORC_ERR_LIMIT;
}

/* ------------------------------------------------------------------------ */
/* Gradient grow (RigL, [PCSR] sec. 4.3: "grow ... new entries at            */
/* high-gradient locations").  The gradient of the loss with respect to the   */
/* weight at (r, c) is sum_beta dY[beta, r] * X[beta, c] ([PCSR] sec. 7.1,    */
/* evaluated at every position instead of only the live ones).  It is taken   */
/* as the fp32 chain g = fmaf(dY[b-1,r], X[b-1,c], ... fmaf(dY[0,r], X[0,c],  */
/* 0)).  Readings: the candidates are the positions held by no kept entry;    */
/* larger bits(|g|) first (NaN above every number), ties to the smaller       */
/* position.  new_lin receives the k chosen positions in ascending order.     */
/* ------------------------------------------------------------------------ */
float orc_grad_at(int64_t out_f, int64_t in_f, const float* X, const float* dY, int64_t b,
                  int64_t row, int64_t col) {
    float g = 0.0f;
    for (int64_t beta = 0; beta < b; ++beta)
        g = fmaf(dY[beta * out_f + row], X[beta * in_f + col], g);
    return g;
}

/* The ranking key: ascending key = descending bits(|g|), then ascending lin. */
uint64_t orc_grad_key(float g, uint64_t lin) {
    return ((uint64_t)(~orc_abs_bits(g)) << 32) | (lin & 0xffffffffull);
}

static int orc_cmp_u64(const void* a, const void* b) {
    uint64_t x = *(const uint64_t*)a, y = *(const uint64_t*)b;
    return (x > y) - (x < y);
}

int orc_grow_gradient(int64_t out_f, int64_t in_f, int64_t n_kept, const int32_t* r_kept,
                      const int32_t* c_kept, const float* X, const float* dY, int64_t b,
                      int64_t k, int64_t* new_lin) {
    uint64_t n_pos = (uint64_t)out_f * (uint64_t)in_f;
    if (n_pos > (1ull << 32)) return ORC_ERR_LIMIT;
    if ((uint64_t)n_kept + (uint64_t)k > n_pos) return ORC_ERR_NOSPACE;
    uint8_t* held = (uint8_t*)calloc((size_t)n_pos, 1);
    uint64_t* keys = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(n_pos - (uint64_t)n_kept + 1));
    if (!held || !keys) {
        free(held);
        free(keys);
        return ORC_ERR_OOM;
    }
    for (int64_t i = 0; i < n_kept; ++i)
        held[(uint64_t)r_kept[i] * (uint64_t)in_f + (uint64_t)c_kept[i]] = 1;
    size_t n_cand = 0;
    for (uint64_t p = 0; p < n_pos; ++p) {
        if (held[p]) continue;
        int64_t row = (int64_t)(p / (uint64_t)in_f), col = (int64_t)(p % (uint64_t)in_f);
        keys[n_cand++] = orc_grad_key(orc_grad_at(out_f, in_f, X, dY, b, row, col), p);
    }
    qsort(keys, n_cand, sizeof(uint64_t), orc_cmp_u64);
    for (int64_t j = 0; j < k; ++j) new_lin[j] = (int64_t)(keys[j] & 0xffffffffull);
    qsort(new_lin, (size_t)k, sizeof(int64_t), orc_cmp_u64);
    free(held);
    free(keys);
    return ORC_OK;
}

/* The ranking keys of the given positions. */
void orc_grad_keys(int64_t out_f, int64_t in_f, const float* X, const float* dY, int64_t b,
                   const int64_t* lin, int64_t n, uint64_t* keys) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t row = lin[i] / in_f, col = lin[i] % in_f;
        keys[i] = orc_grad_key(orc_grad_at(out_f, in_f, X, dY, b, row, col), (uint64_t)lin[i]);
    }
}

/* Number of candidates (positions not held by the kept set) whose key is
 * below `theta`: the exact rank of a key among all candidates, for checking
 * a selection on layers too large to sort. */
int64_t orc_grad_count_below(int64_t out_f, int64_t in_f, int64_t n_kept, const int32_t* r_kept,
                             const int32_t* c_kept, const float* X, const float* dY, int64_t b,
                             uint64_t theta) {
    uint64_t n_pos = (uint64_t)out_f * (uint64_t)in_f;
    uint8_t* held = (uint8_t*)calloc((size_t)n_pos, 1);
    if (!held) return -1;
    for (int64_t i = 0; i < n_kept; ++i)
        held[(uint64_t)r_kept[i] * (uint64_t)in_f + (uint64_t)c_kept[i]] = 1;
    int64_t below = 0;
    for (uint64_t p = 0; p < n_pos; ++p) {
        if (held[p]) continue;
        int64_t row = (int64_t)(p / (uint64_t)in_f), col = (int64_t)(p % (uint64_t)in_f);
        below += orc_grad_key(orc_grad_at(out_f, in_f, X, dY, b, row, col), p) < theta;
    }
    free(held);
    return below;
}

/* ------------------------------------------------------------------------ */
/* S5 + S6 together, in place, nnz unchanged: prune k, regrow k at value     */
/* +0.0f, then re-emit the whole triple in canonical order.  On any error    */
/* the arrays are left as they were.                                         */
/* ------------------------------------------------------------------------ */
int orc_prune_regrow(int64_t out_f, int64_t in_f, int64_t nnz,
                     float* v, int32_t* r, int32_t* c,
                     float zeta, uint64_t seed) {
    if (out_f <= 0 || in_f <= 0 || nnz < 0) return ORC_ERR_ARG;
    if (!(zeta >= 0.0f && zeta < 1.0f)) return ORC_ERR_ARG;
    int64_t k = orc_prune_count(zeta, nnz);
    uint64_t n_pos = (uint64_t)out_f * (uint64_t)in_f;
    if (n_pos - (uint64_t)(nnz - k) < (uint64_t)k) return ORC_ERR_NOSPACE;
    if (k == 0) return ORC_OK;

    size_t n = (size_t)nnz;
    uint8_t* removed = (uint8_t*)malloc(n);
    float* v2 = (float*)malloc(sizeof(float) * n);
    int32_t* r2 = (int32_t*)malloc(sizeof(int32_t) * n);
    int32_t* c2 = (int32_t*)malloc(sizeof(int32_t) * n);
    int64_t* grown = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
    int rc = ORC_ERR_OOM;
    if (!removed || !v2 || !r2 || !c2 || !grown) goto done;

    rc = orc_prune(out_f, in_f, nnz, v, r, c, zeta, removed, NULL);
    if (rc != ORC_OK) goto done;
    int64_t m = 0;
    for (int64_t i = 0; i < nnz; ++i) {
        if (removed[i]) continue;
        v2[m] = v[i];
        r2[m] = r[i];
        c2[m] = c[i];
        ++m;
    }
    rc = orc_regrow(out_f, in_f, m, r2, c2, k, seed, grown, NULL);
    if (rc != ORC_OK) goto done;
    for (int64_t j = 0; j < k; ++j) {
        v2[m + j] = 0.0f;
        r2[m + j] = (int32_t)((uint64_t)grown[j] / (uint64_t)in_f);
        c2[m + j] = (int32_t)((uint64_t)grown[j] % (uint64_t)in_f);
    }
    rc = orc_canonicalize(out_f, in_f, nnz, v2, r2, c2, NULL, NULL, NULL, NULL);
    if (rc != ORC_OK) goto done;
    memcpy(v, v2, sizeof(float) * n);
    memcpy(r, r2, sizeof(int32_t) * n);
    memcpy(c, c2, sizeof(int32_t) * n);
done:
    free(removed);
    free(v2);
    free(r2);
    free(c2);
    free(grown);
    return rc;
}

/* The RigL restructure: the same prune as orc_prune_regrow, then the
 * gradient grow instead of the seeded one, then canonical re-emission. */
int orc_prune_regrow_gradient(int64_t out_f, int64_t in_f, int64_t nnz,
                              float* v, int32_t* r, int32_t* c, float zeta,
                              const float* X, const float* dY, int64_t b) {
    if (out_f <= 0 || in_f <= 0 || nnz < 0 || b < 1) return ORC_ERR_ARG;
    if (!(zeta >= 0.0f && zeta < 1.0f)) return ORC_ERR_ARG;
    int64_t k = orc_prune_count(zeta, nnz);
    uint64_t n_pos = (uint64_t)out_f * (uint64_t)in_f;
    if (n_pos > (1ull << 32)) return ORC_ERR_LIMIT;
    if (n_pos - (uint64_t)(nnz - k) < (uint64_t)k) return ORC_ERR_NOSPACE;
    if (k == 0) return ORC_OK;

    size_t n = (size_t)nnz;
    uint8_t* removed = (uint8_t*)malloc(n);
    float* v2 = (float*)malloc(sizeof(float) * n);
    int32_t* r2 = (int32_t*)malloc(sizeof(int32_t) * n);
    int32_t* c2 = (int32_t*)malloc(sizeof(int32_t) * n);
    int64_t* grown = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
    int rc = ORC_ERR_OOM;
    if (!removed || !v2 || !r2 || !c2 || !grown) goto done;

    rc = orc_prune(out_f, in_f, nnz, v, r, c, zeta, removed, NULL);
    if (rc != ORC_OK) goto done;
    int64_t m = 0;
    for (int64_t i = 0; i < nnz; ++i) {
        if (removed[i]) continue;
        v2[m] = v[i];
        r2[m] = r[i];
        c2[m] = c[i];
        ++m;
    }
    rc = orc_grow_gradient(out_f, in_f, m, r2, c2, X, dY, b, k, grown);
    if (rc != ORC_OK) goto done;
    for (int64_t j = 0; j < k; ++j) {
        v2[m + j] = 0.0f;
        r2[m + j] = (int32_t)((uint64_t)grown[j] / (uint64_t)in_f);
        c2[m + j] = (int32_t)((uint64_t)grown[j] % (uint64_t)in_f);
    }
    rc = orc_canonicalize(out_f, in_f, nnz, v2, r2, c2, NULL, NULL, NULL, NULL);
    if (rc != ORC_OK) goto done;
    memcpy(v, v2, sizeof(float) * n);
    memcpy(r, r2, sizeof(int32_t) * n);
    memcpy(c, c2, sizeof(int32_t) * n);
done:
    free(removed);
    free(v2);
    free(r2);
    free(c2);
    free(grown);
    return rc;
}
