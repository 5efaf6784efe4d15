"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle against something it does not compute itself:
values the pages print for a worked example, a dense closed form evaluated
by numpy, finite differences of the forward map, the adjoint identity,
brute force on tiny inputs, published generator outputs, or special cases
whose answer does not depend on the random draws.

Pages:
  [SNACK] "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU"
  [PCSR]  "Padded-CSR: A sparse storage format for dynamic sparse training on CPU"
"""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import synth
from tests.conftest import load_golden


def dense_of(out_f, in_f, v, r, c):
    W = np.zeros((out_f, in_f), np.float64)
    W[np.asarray(r), np.asarray(c)] = np.asarray(v, np.float64)
    return W


def tiny_layer(out_f, in_f, nnz, seed, std=1.0):
    r, c = synth.uniform_support(out_f, in_f, nnz, seed)
    v = synth.normal(nnz, std, seed + 100)
    return v, r, c


# ---------------------------------------------------------------- worked examples

def test_forward_matches_pcsr_worked_example():
    """[PCSR] sec. 6.1: Y = [[23,28],[5,10],[23,28]] (features-major)."""
    g = load_golden("pcsr_spmm_worked_example.json")
    X = np.array(g["x_batch_major"], np.float32)
    np.testing.assert_array_equal(X, np.array(g["x_page_features_major"], np.float32).T)
    Y, A = oracle.forward(g["out"], g["in"], g["values"], g["rows"], g["cols"], X)
    np.testing.assert_array_equal(Y, np.array(g["y_batch_major"], np.float64))
    np.testing.assert_array_equal(Y.T, np.array(g["y_page_features_major"], np.float64))
    # all products are positive, so the magnitude sum equals the result
    np.testing.assert_array_equal(A, Y)


def test_forward_worked_example_any_triple_order():
    g = load_golden("pcsr_spmm_worked_example.json")
    X = np.array(g["x_batch_major"], np.float32)
    order = [4, 2, 0, 3, 1]
    v = np.array(g["values"])[order]
    r = np.array(g["rows"])[order]
    c = np.array(g["cols"])[order]
    Y, _ = oracle.forward(g["out"], g["in"], v, r, c, X)
    np.testing.assert_array_equal(Y, np.array(g["y_batch_major"], np.float64))


def test_canonical_csr_matches_pcsr_toy():
    """[PCSR] sec. 3.2 / 4.1: the 4x6 toy sorts to rows [0,2,2,3,3], cols
    [2,0,4,1,5], values [3,2,5,7,4] with row_ptr [0,1,1,3,5]."""
    g = load_golden("pcsr_toy_4x6.json")
    W = np.array(g["dense"], np.float64)
    r, c = np.nonzero(W)
    np.testing.assert_array_equal(r, g["rows"])
    np.testing.assert_array_equal(c, g["cols"])
    shuffle = np.array([3, 0, 4, 2, 1])
    out = oracle.canonicalize(g["out"], g["in"], np.array(g["values"], np.float32)[shuffle],
                              np.array(g["rows"])[shuffle], np.array(g["cols"])[shuffle])
    np.testing.assert_array_equal(out["rows"], g["rows"])
    np.testing.assert_array_equal(out["cols"], g["cols"])
    np.testing.assert_array_equal(out["values"], g["values"])
    np.testing.assert_array_equal(out["row_ptr"], g["row_ptr"])


def test_canonical_order_reproduces_pcsr_insert_example():
    """[PCSR] sec. 4.2: after adding (2,2,6) the CSR reads values
    [3,2,6,5,7,4], cols [2,0,2,4,1,5], row_ptr [0,1,1,4,6]."""
    g = load_golden("pcsr_toy_4x6.json")
    ins = g["csr_insert_example"]
    rr, cc, vv = ins["insert"]
    v = np.array(g["values"] + [vv], np.float32)
    r = np.array(g["rows"] + [rr])
    c = np.array(g["cols"] + [cc])
    out = oracle.canonicalize(g["out"], g["in"], v, r, c)
    np.testing.assert_array_equal(out["values"], ins["values_after"])
    np.testing.assert_array_equal(out["cols"], ins["col_indices_after"])
    np.testing.assert_array_equal(out["row_ptr"], ins["row_ptr_after"])


def test_csc_and_perm_match_snack_table7():
    """[SNACK] Table 7: CSR indptr [0,1,2,3] cols [2,0,1]; CSC data [4,5,3],
    rows [1,2,0], indptr [0,1,2,3]."""
    g = load_golden("snack_table7_formats.json")
    coo = g["coo"]
    out = oracle.canonicalize(g["out"], g["in"], coo["data"], coo["row"], coo["col"])
    np.testing.assert_array_equal(out["row_ptr"], g["csr"]["indptr"])
    np.testing.assert_array_equal(out["cols"], g["csr"]["col"])
    np.testing.assert_array_equal(out["values"], g["csr"]["data"])
    np.testing.assert_array_equal(out["col_ptr"], g["csc"]["indptr"])
    np.testing.assert_array_equal(out["rows_c"], g["csc"]["row"])
    np.testing.assert_array_equal(out["values"][out["perm"]], g["csc"]["data"])


def test_csc_matches_scipy_style_transpose_brute_force():
    """CSC built by the oracle equals the column-major order found by brute
    force: sort (col, row) pairs with numpy lexsort."""
    out_f, in_f = 37, 29
    v, r, c = tiny_layer(out_f, in_f, 300, 5)
    o = oracle.canonicalize(out_f, in_f, v, r, c)
    order = np.lexsort((o["rows"], o["cols"]))
    np.testing.assert_array_equal(o["perm"], order)
    np.testing.assert_array_equal(o["rows_c"], o["rows"][order])
    np.testing.assert_array_equal(o["col_ptr"],
                                  np.concatenate([[0], np.cumsum(np.bincount(o["cols"], minlength=in_f))]))
    lin = o["rows"].astype(np.int64) * in_f + o["cols"]
    assert np.all(np.diff(lin) > 0)


def test_canonicalize_rejects_duplicates_and_range():
    with pytest.raises(oracle.OracleError) as e:
        oracle.canonicalize(4, 4, [1, 2], [1, 1], [2, 2])
    assert e.value.status == oracle.ORC_ERR_DUP
    with pytest.raises(oracle.OracleError) as e:
        oracle.canonicalize(4, 4, [1], [4], [0])
    assert e.value.status == oracle.ORC_ERR_RANGE
    with pytest.raises(oracle.OracleError) as e:
        oracle.canonicalize(4, 4, [1], [0], [-1])
    assert e.value.status == oracle.ORC_ERR_RANGE


# ---------------------------------------------------------------- closed forms

SHAPES = [(1, 1, 1), (5, 7, 9), (16, 3, 20), (3, 16, 20), (33, 31, 100), (64, 64, 400)]


@pytest.mark.parametrize("out_f,in_f,nnz", SHAPES)
@pytest.mark.parametrize("b", [1, 3, 8])
def test_three_products_match_dense_closed_form(out_f, in_f, nnz, b):
    """Y = X (W.M)^T + bias, dX = dY (W.M), dW = (dY^T X) restricted to M,
    db = 1^T dY, each evaluated densely by numpy in fp64."""
    v, r, c = tiny_layer(out_f, in_f, nnz, out_f * 1000 + in_f)
    X = synth.normal((b, in_f), 1.0, 7)
    dY = synth.normal((b, out_f), 1.0, 8)
    bias = synth.normal(out_f, 1.0, 9)
    W = dense_of(out_f, in_f, v, r, c)
    Xd, dYd = X.astype(np.float64), dY.astype(np.float64)

    Y, A = oracle.forward(out_f, in_f, v, r, c, X, bias)
    np.testing.assert_allclose(Y, Xd @ W.T + bias.astype(np.float64), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(A, np.abs(Xd) @ np.abs(W).T + np.abs(bias), rtol=1e-12, atol=1e-12)

    dX, Ax = oracle.backward_input(out_f, in_f, v, r, c, dY)
    np.testing.assert_allclose(dX, dYd @ W, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Ax, np.abs(dYd) @ np.abs(W), rtol=1e-12, atol=1e-12)

    dW, Aw, db, Adb = oracle.backward_weight(out_f, in_f, r, c, X, dY)
    G = dYd.T @ Xd
    np.testing.assert_allclose(dW, G[r, c], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Aw, (np.abs(dYd).T @ np.abs(Xd))[r, c], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, dYd.sum(0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Adb, np.abs(dYd).sum(0), rtol=1e-12, atol=1e-12)
    # supp(dW) = supp(W): scattering dW back gives the dense gradient masked by M
    dWd = np.zeros_like(W)
    dWd[r, c] = dW
    M = dense_of(out_f, in_f, np.ones(nnz), r, c)
    np.testing.assert_allclose(dWd, G * M, rtol=1e-12, atol=1e-12)


def test_empty_rows_columns_and_no_bias():
    out_f, in_f = 6, 5
    r = np.array([1, 1, 4], np.int32)
    c = np.array([0, 3, 3], np.int32)
    v = np.array([2.0, -1.0, 0.5], np.float32)
    X = np.arange(10, dtype=np.float32).reshape(2, 5)
    Y, _ = oracle.forward(out_f, in_f, v, r, c, X)
    exp = np.zeros((2, 6))
    exp[:, 1] = 2 * X[:, 0] - X[:, 3]
    exp[:, 4] = 0.5 * X[:, 3]
    np.testing.assert_array_equal(Y, exp)
    dX, _ = oracle.backward_input(out_f, in_f, v, r, c, np.ones((2, 6), np.float32))
    np.testing.assert_array_equal(dX[:, [1, 2, 4]], 0.0)
    np.testing.assert_array_equal(dX[:, 0], 2.0)
    np.testing.assert_array_equal(dX[:, 3], -0.5)


def test_no_nonzeros():
    X = np.ones((2, 3), np.float32)
    bias = np.array([1, 2], np.float32)
    Y, A = oracle.forward(2, 3, [], [], [], X, bias)
    np.testing.assert_array_equal(Y, [[1, 2], [1, 2]])
    dX, _ = oracle.backward_input(2, 3, [], [], [], np.ones((2, 2), np.float32))
    np.testing.assert_array_equal(dX, 0.0)
    dW, _, db, _ = oracle.backward_weight(2, 3, [], [], X, np.ones((2, 2), np.float32))
    assert dW.shape == (0,)
    np.testing.assert_array_equal(db, [2, 2])


def test_permutation_matrix_forward_is_an_exact_copy():
    """One weight of 1.0 per row: Y is a permuted copy of X, bit for bit."""
    n = 50
    p = synth.rng(3).permutation(n)
    X = synth.normal((4, n), 1.0, 4)
    Y, _ = oracle.forward(n, n, np.ones(n, np.float32), np.arange(n), p, X)
    np.testing.assert_array_equal(Y, X[:, p].astype(np.float64))


# ---------------------------------------------------------------- finite differences

def dyadic(shape, seed, scale_bits=6):
    """Small dyadic rationals: products and short sums are exact in fp64, and
    x +- h stays exact in fp32, so a central difference of the bilinear map
    returns the gradient exactly."""
    g = synth.rng(seed)
    return (g.integers(-64, 65, size=shape) / float(1 << scale_bits)).astype(np.float32)


def test_central_differences_give_both_gradients():
    out_f, in_f, nnz, b = 7, 9, 25, 3
    r, c = synth.uniform_support(out_f, in_f, nnz, 11)
    v = dyadic(nnz, 12)
    X = dyadic((b, in_f), 13)
    G = dyadic((b, out_f), 14)
    h = np.float32(0.25)

    def loss(vv, XX):
        Y, _ = oracle.forward(out_f, in_f, vv, r, c, XX)
        return float(np.sum(Y * G.astype(np.float64)))

    dX, _ = oracle.backward_input(out_f, in_f, v, r, c, G)
    for beta in range(b):
        for i in range(in_f):
            Xp, Xm = X.copy(), X.copy()
            Xp[beta, i] += h
            Xm[beta, i] -= h
            fd = (loss(v, Xp) - loss(v, Xm)) / (2 * float(h))
            assert fd == dX[beta, i]

    dW, _, _, _ = oracle.backward_weight(out_f, in_f, r, c, X, G)
    for k in range(nnz):
        vp, vm = v.copy(), v.copy()
        vp[k] += h
        vm[k] -= h
        fd = (loss(vp, X) - loss(vm, X)) / (2 * float(h))
        assert fd == dW[k]


def test_adjoint_identity():
    """<X W^T, G> = <X, G W> for the same sparse W."""
    out_f, in_f = 40, 30
    v, r, c = tiny_layer(out_f, in_f, 200, 21)
    X = synth.normal((5, in_f), 1.0, 22)
    G = synth.normal((5, out_f), 1.0, 23)
    Y, _ = oracle.forward(out_f, in_f, v, r, c, X)
    dX, _ = oracle.backward_input(out_f, in_f, v, r, c, G)
    lhs = float(np.sum(Y * G.astype(np.float64)))
    rhs = float(np.sum(X.astype(np.float64) * dX))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


# ---------------------------------------------------------------- prune

def brute_force_prune(v, r, c, in_f, zeta):
    k = int(np.floor(np.float64(np.float32(zeta)) * len(v)))
    mag = np.asarray(v, np.float32).view(np.uint32) & np.uint32(0x7FFFFFFF)
    keys = sorted(range(len(v)), key=lambda i: (int(mag[i]), int(r[i]) * in_f + int(c[i])))
    removed = np.zeros(len(v), bool)
    removed[keys[:k]] = True
    return removed, k


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("zeta", [0.0, 0.1, 0.3, 0.5, 0.99])
def test_prune_matches_brute_force(seed, zeta):
    out_f, in_f, nnz = 9, 11, 60
    v, r, c = tiny_layer(out_f, in_f, nnz, seed)
    g = synth.rng(seed + 50)
    # plant ties, signed zeros and repeated magnitudes of both signs
    v[g.choice(nnz, 10, replace=False)] = 0.0
    v[g.choice(nnz, 5, replace=False)] = -0.0
    v[g.choice(nnz, 6, replace=False)] = 0.5
    v[g.choice(nnz, 6, replace=False)] = -0.5
    removed, k = oracle.prune(out_f, in_f, v, r, c, zeta)
    exp, k_exp = brute_force_prune(v, r, c, in_f, zeta)
    assert k == k_exp == oracle.prune_count(zeta, nnz)
    np.testing.assert_array_equal(removed, exp)


def test_prune_invariants_and_special_values():
    v = np.array([np.inf, 1.0, -2.0, np.nan, -0.0, 0.0, 3.0, -np.inf], np.float32)
    r = np.arange(8, dtype=np.int32)
    c = np.zeros(8, np.int32)
    removed, k = oracle.prune(8, 1, v, r, c, 0.75)
    assert k == 6
    # NaN ranks above +-inf; -0.0 and +0.0 tie and are split by position
    np.testing.assert_array_equal(np.nonzero(~removed)[0], [3, 7])
    mag = v.view(np.uint32) & 0x7FFFFFFF
    keys = [(int(mag[i]), i) for i in range(8)]
    assert max(keys[i] for i in range(8) if removed[i]) < min(keys[i] for i in range(8) if not removed[i])


def test_prune_count_rounding():
    assert oracle.prune_count(0.3, 10_000_000) == 3_000_000
    assert oracle.prune_count(0.3, 10) == 3
    assert oracle.prune_count(0.5, 7) == 3
    assert oracle.prune_count(0.0, 12345) == 0


# ---------------------------------------------------------------- regrow

def test_splitmix64_published_outputs():
    g = load_golden("splitmix64_reference.json")
    for seq in g["sequences"]:
        outs = seq.get("outputs") or [int(h, 16) for h in seq["outputs_hex"]]
        for n, want in enumerate(outs):
            assert oracle.splitmix64_nth(seq["state"], n) == want


def test_multiply_shift_range_reduction_closed_forms():
    M = 2**64 - 1
    for n_pos in [1, 2, 3, 100, 10**8, 2**40 + 7, 2**63]:
        assert oracle.mulhi64(0, n_pos) == 0
        assert oracle.mulhi64(M, n_pos) == n_pos - 1
        assert oracle.mulhi64(2**63, n_pos) == n_pos // 2
    assert oracle.mulhi64(M, M) == M - 1
    for z in [1, 12345, 2**40, M]:
        assert oracle.mulhi64(z, 1) == 0
        assert oracle.mulhi64(z, 2**32) == z >> 32


def test_regrow_first_draw_is_the_first_candidate():
    for seed in [0, 1, 0x5E7, 2**63 + 5]:
        new, draws = oracle.regrow(16, 16, [], [], 1, seed)
        assert draws == 1
        assert new[0] == oracle.mulhi64(oracle.splitmix64_nth(seed, 0), 256)


def test_regrow_fills_the_whole_complement():
    """When exactly k positions are free the result is the complement of the
    kept set, whatever the draws."""
    out_f, in_f = 6, 7
    N = out_f * in_f
    kept = synth.rng(1).choice(N, 30, replace=False)
    new, _ = oracle.regrow(out_f, in_f, kept // in_f, kept % in_f, N - 30, 99)
    assert sorted(new.tolist()) == sorted(set(range(N)) - set(kept.tolist()))
    new, _ = oracle.regrow(out_f, in_f, [], [], N, 7)
    assert sorted(new.tolist()) == list(range(N))


def test_regrow_invariants():
    out_f, in_f = 20, 30
    N = out_f * in_f
    kept = synth.rng(2).choice(N, 200, replace=False)
    new, draws = oracle.regrow(out_f, in_f, kept // in_f, kept % in_f, 150, 1234)
    assert len(new) == 150 and len(set(new.tolist())) == 150
    assert not (set(new.tolist()) & set(kept.tolist()))
    assert new.min() >= 0 and new.max() < N
    assert draws >= 150
    # replaying the candidates: every accepted position is the first occurrence
    # of a free position among the draws, in draw order
    seen, acc = set(kept.tolist()), []
    for t in range(draws):
        p = oracle.candidate(1234, t, N)
        if p not in seen:
            seen.add(p)
            acc.append(p)
    assert acc == new.tolist()


def test_regrow_no_space():
    with pytest.raises(oracle.OracleError) as e:
        oracle.regrow(2, 2, [0, 0, 1], [0, 1, 0], 2, 1)
    assert e.value.status == oracle.ORC_ERR_NOSPACE


def test_regrow_first_candidate_is_roughly_uniform():
    """Sanity check of the generator (not parity): first draws over a 16x16
    layer, chi-square over 256 cells with 25600 seeds."""
    counts = np.zeros(256)
    for seed in range(25600):
        counts[oracle.candidate(seed, 0, 256)] += 1
    chi2 = float(((counts - 100.0) ** 2 / 100.0).sum())
    assert chi2 < 360  # 255 dof; p ~ 1e-5


def test_prune_regrow_keeps_nnz_and_order():
    lay = synth.make_layer(30, 40, 80, 1.0, 5, 6)
    v, r, c = oracle.prune_regrow(30, 40, lay.values, lay.rows, lay.cols, 0.3, 77)
    nnz = lay.nnz
    assert len(v) == nnz
    lin = r.astype(np.int64) * 40 + c
    assert np.all(np.diff(lin) > 0)
    removed, k = oracle.prune(30, 40, lay.values, lay.rows, lay.cols, 0.3)
    before = {int(a) * 40 + int(b): float(x) for a, b, x in zip(lay.rows, lay.cols, lay.values)}
    kept = {p: x for (p, x), rm in zip(before.items(), removed) if not rm}
    after = dict(zip(lin.tolist(), v.tolist()))
    for p, x in kept.items():
        assert after[p] == x
    grown = set(after) - set(kept)
    assert len(grown) == k
    assert all(after[p] == 0.0 and np.signbit(np.float32(after[p])) == False for p in grown)


def test_prune_regrow_zero_fraction_is_identity():
    lay = synth.make_layer(10, 10, 50, 1.0, 1, 2)
    can = oracle.canonicalize(10, 10, lay.values, lay.rows, lay.cols)
    v, r, c = oracle.prune_regrow(10, 10, can["values"], can["rows"], can["cols"], 0.0, 5)
    np.testing.assert_array_equal(v, can["values"])
    np.testing.assert_array_equal(r, can["rows"])


# ---------------------------------------------------------------- gradient grow (RigL)
# [PCSR] sec. 4.3: a DST update drops a fraction of the live entries and grows
# as many "at high-gradient locations".  The gradient at (r, c) is
# sum_beta dY[beta, r] X[beta, c] ([PCSR] sec. 7.1 evaluated off the support).

def _numpy_topk(keys_by_pos, k):
    """Positions sorted by (larger |g| first, smaller position first)."""
    pos = np.array(sorted(keys_by_pos, key=lambda p: (-keys_by_pos[p], p)), np.int64)
    return np.sort(pos[:k])


def test_grad_at_single_product_is_the_rounded_product():
    # b = 1: fmaf(a, b, 0) is the product rounded once, which is what an fp32
    # multiply gives
    gen = synth.rng(91)
    X = gen.standard_normal((1, 17)).astype(np.float32)
    dY = gen.standard_normal((1, 11)).astype(np.float32)
    for r in range(11):
        for c in range(17):
            assert np.float32(oracle.grad_at(11, 17, X, dY, r, c)) == dY[0, r] * X[0, c]


def test_grow_gradient_batch1_matches_numpy_ranking():
    gen = synth.rng(92)
    out_f, in_f = 23, 31
    X = gen.standard_normal((1, in_f)).astype(np.float32)
    dY = gen.standard_normal((1, out_f)).astype(np.float32)
    kept = set(gen.choice(out_f * in_f, 200, replace=False).tolist())
    kr = np.array([p // in_f for p in sorted(kept)], np.int32)
    kc = np.array([p % in_f for p in sorted(kept)], np.int32)
    g = dY[0][:, None] * X[0][None, :]                      # exact fp32 products
    mag = np.abs(g).view(np.uint32).astype(np.int64)
    cand = {p: int(mag.flat[p]) for p in range(out_f * in_f) if p not in kept}
    for k in (1, 10, 57, len(cand)):
        np.testing.assert_array_equal(oracle.grow_gradient(out_f, in_f, kr, kc, X, dY, k),
                                      _numpy_topk(cand, k))


def test_grow_gradient_exact_integer_sums():
    # small integers: every product and partial sum is exact in fp32, so the
    # gradient is the integer dY^T X whatever the order
    gen = synth.rng(93)
    out_f, in_f, b = 13, 19, 3
    X = gen.integers(-5, 6, (b, in_f)).astype(np.float32)
    dY = gen.integers(-5, 6, (b, out_f)).astype(np.float32)
    G = dY.astype(np.int64).T @ X.astype(np.int64)
    kept = set(gen.choice(out_f * in_f, 60, replace=False).tolist())
    kr = np.array([p // in_f for p in sorted(kept)], np.int32)
    kc = np.array([p % in_f for p in sorted(kept)], np.int32)
    cand = {p: abs(int(G.flat[p])) for p in range(out_f * in_f) if p not in kept}
    for k in (5, 40, 100):
        np.testing.assert_array_equal(oracle.grow_gradient(out_f, in_f, kr, kc, X, dY, k),
                                      _numpy_topk(cand, k))


def test_grow_gradient_ties_go_to_smaller_positions():
    # every gradient has the same magnitude: the grown set is the k smallest
    # free positions
    out_f, in_f = 8, 9
    X = np.ones((2, in_f), np.float32)
    dY = np.full((2, out_f), 0.5, np.float32)
    dY[:, ::2] *= -1
    kr = np.array([0, 0, 3], np.int32)
    kc = np.array([0, 5, 2], np.int32)
    free = [p for p in range(out_f * in_f) if p not in (0, 5, 3 * in_f + 2)]
    np.testing.assert_array_equal(oracle.grow_gradient(out_f, in_f, kr, kc, X, dY, 7), free[:7])


def test_grow_gradient_nan_ranks_first_and_zero_last():
    out_f, in_f = 4, 5
    X = np.array([[1, 2, 0, 3, 1]], np.float32)
    dY = np.array([[1, 1, 1, 1]], np.float32)
    X[0, 4] = np.nan
    kr = np.zeros(0, np.int32)
    kc = np.zeros(0, np.int32)
    # column 4 is NaN in every row (4 positions), then |g| = 3 (column 3)
    got = oracle.grow_gradient(out_f, in_f, kr, kc, X, dY, 6)
    np.testing.assert_array_equal(got, sorted([4, 9, 14, 19, 3, 8]))
    # the zero column comes last of all
    allp = oracle.grow_gradient(out_f, in_f, kr, kc, X, dY, 20)
    np.testing.assert_array_equal(allp, np.arange(20))
    last = oracle.grow_gradient(out_f, in_f, kr, kc, X, dY, 16)
    assert set(range(20)) - set(last.tolist()) == {2, 7, 12, 17}


def test_grow_gradient_count_below_is_the_rank():
    gen = synth.rng(94)
    out_f, in_f = 20, 24
    X = gen.standard_normal((3, in_f)).astype(np.float32)
    dY = gen.standard_normal((3, out_f)).astype(np.float32)
    kept = np.sort(gen.choice(out_f * in_f, 100, replace=False))
    kr, kc = (kept // in_f).astype(np.int32), (kept % in_f).astype(np.int32)
    k = 50
    grown = oracle.grow_gradient(out_f, in_f, kr, kc, X, dY, k)
    keys = [oracle.grad_key(oracle.grad_at(out_f, in_f, X, dY, p // in_f, p % in_f), p)
            for p in grown]
    theta = max(keys)
    assert oracle.grad_count_below(out_f, in_f, kr, kc, X, dY, theta) == k - 1
    assert oracle.grad_count_below(out_f, in_f, kr, kc, X, dY, theta + 1) == k


def test_prune_regrow_gradient_regrows_a_pruned_position():
    # the smallest-magnitude entry sits where the gradient is largest: it is
    # pruned and grown back at value +0.0 (the post-prune complement reading)
    out_f, in_f = 5, 6
    r = np.array([0, 1, 2, 3, 4], np.int32)
    c = np.array([0, 1, 2, 3, 4], np.int32)
    v = np.array([1e-3, 2.0, 3.0, 4.0, 5.0], np.float32)
    X = np.zeros((1, in_f), np.float32)
    dY = np.zeros((1, out_f), np.float32)
    X[0, 0], dY[0, 0] = 10.0, 10.0      # |g(0, 0)| = 100, every other g is 0
    v2, r2, c2 = oracle.prune_regrow_gradient(out_f, in_f, v, r, c, 0.2, X, dY)
    np.testing.assert_array_equal(r2, r)
    np.testing.assert_array_equal(c2, c)
    assert v2[0] == 0.0 and not np.signbit(v2[0])
    np.testing.assert_array_equal(v2[1:], v[1:])


def test_prune_regrow_gradient_invariants():
    lay = synth.make_layer(30, 40, 80, 1.0, 5, 6)
    X = synth.normal((4, 40), 1.0, 7)
    dY = synth.normal((4, 30), 1.0, 8)
    v, r, c = oracle.prune_regrow_gradient(30, 40, lay.values, lay.rows, lay.cols, 0.3, X, dY)
    lin = r.astype(np.int64) * 40 + c
    assert len(v) == lay.nnz and np.all(np.diff(lin) > 0)
    removed, k = oracle.prune(30, 40, lay.values, lay.rows, lay.cols, 0.3)
    kept_lin = sorted(int(a) * 40 + int(b) for a, b, rm in zip(lay.rows, lay.cols, removed) if not rm)
    kl = np.array(kept_lin, np.int64)
    grown = oracle.grow_gradient(30, 40, (kl // 40).astype(np.int32), (kl % 40).astype(np.int32),
                                 X, dY, k)
    assert set(lin.tolist()) == set(kept_lin) | set(grown.tolist())
    assert len(set(kept_lin) & set(grown.tolist())) == 0


def test_openmp_build_gives_the_same_bits():
    """The OpenMP build of the oracle (the benchmark's all-core CPU baseline)
    splits outputs among threads but adds each output's terms in the same
    order, so it must return exactly the single-threaded results, also on a
    triple in random order and with empty rows."""
    if not oracle.openmp_available():
        pytest.skip("gcc without OpenMP")
    lay = synth.make_layer(333, 257, 80, 0.05, 71, 72)
    X = synth.normal((5, 257), 1.0, 73)
    dY = synth.normal((5, 333), 1.0, 74)
    bias = synth.normal(333, 0.1, 75)
    v, r, c = lay.values, lay.rows, lay.cols
    for a, b_ in zip(oracle.forward(333, 257, v, r, c, X, bias),
                     oracle.forward(333, 257, v, r, c, X, bias, omp=True)):
        assert np.array_equal(a, b_)
    for a, b_ in zip(oracle.backward_input(333, 257, v, r, c, dY),
                     oracle.backward_input(333, 257, v, r, c, dY, omp=True)):
        assert np.array_equal(a, b_)
    for a, b_ in zip(oracle.backward_weight(333, 257, r, c, X, dY),
                     oracle.backward_weight(333, 257, r, c, X, dY, omp=True)):
        assert np.array_equal(a, b_)
    assert oracle.threads(omp=False) == 1
