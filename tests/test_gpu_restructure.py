"""GPU prune/regrow against the oracle: the whole triple must be bit-identical
after each restructure, given the same values and seed.

Pages: "Padded-CSR: A sparse storage format for dynamic sparse training on
CPU" (sec. 1.1, 4.3, 8.2); "Beyond Masked Sparsity: SNACK Enables Truly
Sparse Neural Networks on GPU" (Fig. 1).
"""
import os

import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import binding, synth
from tests.gpu_util import dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def restructure_and_compare(torch, g, out_f, in_f, zeta, seed):
    v0, r0, c0 = host(g.values), host(g.rows), host(g.cols)
    ver = g.topology_version
    g.prune_regrow(zeta, seed)
    ve, re_, ce = oracle.prune_regrow(out_f, in_f, v0, r0, c0, zeta, seed)
    np.testing.assert_array_equal(host(g.rows), re_)
    np.testing.assert_array_equal(host(g.cols), ce)
    np.testing.assert_array_equal(host(g.values).view(np.uint32), ve.view(np.uint32))
    k = oracle.prune_count(zeta, len(v0))
    assert g.topology_version == ver + (1 if k > 0 else 0)
    t = g.topology()
    can = oracle.canonicalize(out_f, in_f, ve, re_, ce)
    for key in ("row_ptr", "col_ptr", "rows_c", "perm"):
        np.testing.assert_array_equal(host(t[key]), can[key], err_msg=key)


@pytest.mark.parametrize("out_f,in_f,sp,zeta,seed", [
    (16, 16, 50, 0.3, 1),
    (500, 500, 95, 0.3, 0x5E7),
    (129, 77, 90, 0.5, 7),
    (1000, 1000, 90, 0.3, 2**64 - 3),
    (3072, 768, 90, 0.3, 9),
    (10, 10, 10, 0.9, 3),        # dense-ish: few free positions, many collisions
])
def test_prune_regrow_bit_exact(torch, out_f, in_f, sp, zeta, seed):
    lay = synth.make_layer(out_f, in_f, sp, 0.05, 5, 6)
    g = make_gpu_layer(torch, lay)
    restructure_and_compare(torch, g, out_f, in_f, zeta, seed)
    g.close()


@pytest.mark.parametrize("out_f,in_f,nnz", [
    (70_000, 70_000, 60_000),     # 4.9e9 positions: hash set for held positions, 64-bit sort
    (40_000, 60_000, 50_000),     # 2.4e9 positions: hash set, 32-bit sort of grown positions
])
def test_prune_regrow_large_position_space(torch, out_f, in_f, nnz):
    """Layers with more than 2^31 positions take the hash-set path for held
    positions (and above 2^32 the 64-bit sort of the grown ones)."""
    r, c = synth.uniform_support(out_f, in_f, nnz, 61)
    lay = synth.Layer(out_f, in_f, synth.normal(nnz, 0.05, 62), r, c)
    g = make_gpu_layer(torch, lay)
    for i in range(2):
        restructure_and_compare(torch, g, out_f, in_f, 0.3, 0x5E7 + i)
    g.close()


def test_ties_zeros_and_signed_zero(torch):
    out_f, in_f = 60, 70
    lay = synth.make_layer(out_f, in_f, 80, 1.0, 8, 9)
    v = lay.values
    gen = synth.rng(10)
    v[gen.choice(len(v), 200, replace=False)] = 0.0
    v[gen.choice(len(v), 50, replace=False)] = -0.0
    v[gen.choice(len(v), 80, replace=False)] = 0.25
    v[gen.choice(len(v), 80, replace=False)] = -0.25
    g = make_gpu_layer(torch, lay)
    for i in range(3):
        restructure_and_compare(torch, g, out_f, in_f, 0.3, 100 + i)
    g.close()


def test_full_fraction_edge_and_exactly_full_complement(torch):
    # 4x4 with 12 entries, zeta = 0.99 -> prune 11, 5 free slots after prune... 4 + 11
    lay = synth.make_layer(4, 4, 25, 1.0, 1, 2)
    g = make_gpu_layer(torch, lay)
    restructure_and_compare(torch, g, 4, 4, 0.99, 5)
    g.close()
    # full matrix: nothing is free but the pruned positions themselves
    n = 36
    r, c = np.divmod(np.arange(n, dtype=np.int32), 6)
    lay = synth.Layer(6, 6, synth.normal(n, 1.0, 3), r.astype(np.int32), c.astype(np.int32))
    g = make_gpu_layer(torch, lay)
    restructure_and_compare(torch, g, 6, 6, 0.5, 11)
    g.close()


def test_zero_fraction_is_a_no_op(torch):
    lay = synth.make_layer(100, 100, 90, 0.05, 3, 4)
    g = make_gpu_layer(torch, lay)
    before = host(g.rows).copy(), host(g.values).copy()
    g.prune_regrow(0.0, 1)
    assert g.topology_version == 1
    np.testing.assert_array_equal(host(g.rows), before[0])
    np.testing.assert_array_equal(host(g.values), before[1])
    g.close()


def test_errors_leave_the_layer_unchanged(torch):
    lay = synth.make_layer(50, 40, 90, 0.05, 3, 4)
    g = make_gpu_layer(torch, lay)
    snap = host(g.rows).copy(), host(g.cols).copy()
    for bad in (-0.1, 1.0, float("nan")):
        with pytest.raises(binding.SnkError) as e:
            g.prune_regrow(bad, 1)
        assert e.value.status == binding.SNK_ERR_ARG
    np.testing.assert_array_equal(host(g.rows), snap[0])
    g.close()


def test_no_space_is_reported_before_work(torch):
    # all positions held: pruning frees k, so the regrow always fits; a layer
    # with out*in - (nnz - k) < k cannot be built with nnz <= out*in, so the
    # check is exercised through the oracle's identical rule on a tiny case
    with pytest.raises(oracle.OracleError) as e:
        oracle.regrow(2, 2, [0, 0, 1], [0, 1, 0], 2, 1)
    assert e.value.status == oracle.ORC_ERR_NOSPACE


def test_host_fault_injection_allocation(torch):
    lay = synth.make_layer(30, 30, 90, 0.05, 3, 4)
    v, r, c = dev(lay.values, torch), dev(lay.rows, torch), dev(lay.cols, torch)
    os.environ["SNK_FAULT"] = "alloc"
    try:
        with pytest.raises(binding.SnkError) as e:
            binding.snk_create(30, 30, v, r, c)
        assert e.value.status == binding.SNK_ERR_OOM
    finally:
        del os.environ["SNK_FAULT"]
    g = binding.SparseLinear(30, 30, v, r, c)
    os.environ["SNK_FAULT"] = "launch"
    try:
        with pytest.raises(binding.SnkError) as e:
            g.forward(dev(synth.normal((2, 30), 1.0, 5), torch))
        assert e.value.status == binding.SNK_ERR_CUDA
    finally:
        del os.environ["SNK_FAULT"]
    g.close()


def test_set_training_stepwise_and_resume(torch):
    """A SET run (SGD steps on an MSE loss, restructure every 10 steps): each
    restructure is compared with the oracle on the GPU's current state, and a
    run restarted from a checkpoint of the triple reaches the same topology."""
    out_f, in_f, b = 1000, 800, 4
    lay = synth.make_layer(out_f, in_f, 90, 0.01, 31, 32)
    X = dev(synth.normal((b, in_f), 1.0, 33), torch)
    T = dev(synth.normal((b, out_f), 1.0, 34), torch)

    def run(g, steps, start=0, snapshot_at=None):
        snap = None
        for step in range(start, steps):
            Y = g.forward(X)
            dY = (2.0 / (b * out_f)) * (Y - T)
            dW = g.backward_weight(X, dY)
            g.values.sub_(0.01 * dW)
            if (step + 1) % 10 == 0:
                restructure_and_compare(torch, g, out_f, in_f, 0.3, 0x5E7 + (step + 1) // 10)
            if snapshot_at is not None and step + 1 == snapshot_at:
                snap = (g.values.clone(), g.rows.clone(), g.cols.clone())
        return snap

    g = make_gpu_layer(torch, lay)
    snap = run(g, 30, snapshot_at=15)
    final = host(g.rows).copy(), host(g.cols).copy(), host(g.values).copy()
    g.close()
    g2 = binding.SparseLinear(out_f, in_f, *snap)
    run(g2, 30, start=15)
    np.testing.assert_array_equal(host(g2.rows), final[0])
    np.testing.assert_array_equal(host(g2.cols), final[1])
    np.testing.assert_array_equal(host(g2.values), final[2])
    g2.close()


def test_full_size_restructure(torch):
    """10000 x 10000 at 90% (10,000,000 entries), zeta = 0.3: 3,000,000 pruned
    and regrown, bit-exact against the oracle."""
    lay = synth.make_layer(10_000, 10_000, 90, 0.01, 31, 32)
    g = make_gpu_layer(torch, lay)
    restructure_and_compare(torch, g, 10_000, 10_000, 0.3, 0x5E7 + 1)
    g.close()


# ---------------------------------------------------------------- gradient grow (RigL)

def gradient_restructure_and_compare(torch, g, out_f, in_f, zeta, X, dY):
    v0, r0, c0 = host(g.values), host(g.rows), host(g.cols)
    ver = g.topology_version
    g.prune_regrow_gradient(zeta, dev(X, torch), dev(dY, torch))
    ve, re_, ce = oracle.prune_regrow_gradient(out_f, in_f, v0, r0, c0, zeta, X, dY)
    np.testing.assert_array_equal(host(g.rows), re_)
    np.testing.assert_array_equal(host(g.cols), ce)
    np.testing.assert_array_equal(host(g.values).view(np.uint32), ve.view(np.uint32))
    k = oracle.prune_count(zeta, len(v0))
    assert g.topology_version == ver + (1 if k > 0 else 0)
    t = g.topology()
    can = oracle.canonicalize(out_f, in_f, ve, re_, ce)
    for key in ("row_ptr", "col_ptr", "rows_c", "perm"):
        np.testing.assert_array_equal(host(t[key]), can[key], err_msg=key)


@pytest.mark.parametrize("out_f,in_f,sp,zeta,b,zipf", [
    (16, 16, 50, 0.3, 1, None),
    (500, 500, 95, 0.3, 4, None),
    (129, 77, 90, 0.5, 3, None),
    (1000, 700, 90, 0.3, 16, None),
    (768, 3072, 90, 0.3, 4, 1.2),     # GPT-2 MLP shape, Zipf rows
    (3072, 768, 99, 0.5, 2, 1.2),
    (10, 10, 10, 0.9, 2, None),       # nearly full: the whole complement is grown
    (200, 300, 90, 0.3, 70, None),    # batch above 64: dY rows read from global memory
    (400, 250, 95, 0.4, 1, None),     # batch 1: the gradient is one rounded product
])
def test_prune_regrow_gradient_bit_exact(torch, out_f, in_f, sp, zeta, b, zipf):
    lay = synth.make_layer(out_f, in_f, sp, 0.05, 5, 6, zipf_s=zipf)
    X = synth.normal((b, in_f), 1.0, 7)
    dY = synth.normal((b, out_f), 1.0, 8)
    g = make_gpu_layer(torch, lay)
    gradient_restructure_and_compare(torch, g, out_f, in_f, zeta, X, dY)
    g.close()


def test_prune_regrow_gradient_massive_ties(torch):
    """Most gradients are exactly zero (X is zero outside 3 columns) and many
    others repeat: the selection has to go down to the position bits."""
    out_f, in_f, b = 300, 200, 2
    lay = synth.make_layer(out_f, in_f, 90, 0.05, 11, 12)
    X = np.zeros((b, in_f), np.float32)
    X[:, [3, 77, 150]] = np.array([[1.0, -2.0, 0.5], [0.25, 1.0, -0.5]], np.float32)
    dY = np.ones((b, out_f), np.float32)
    dY[:, ::3] = -1.0
    g = make_gpu_layer(torch, lay)
    for i in range(2):
        gradient_restructure_and_compare(torch, g, out_f, in_f, 0.3, X, dY)
    g.close()


def test_prune_regrow_gradient_nan_and_errors(torch):
    out_f, in_f = 40, 50
    lay = synth.make_layer(out_f, in_f, 80, 0.05, 13, 14)
    g = make_gpu_layer(torch, lay)
    X = synth.normal((2, in_f), 1.0, 15)
    X[1, 7] = np.nan
    dY = synth.normal((2, out_f), 1.0, 16)
    gradient_restructure_and_compare(torch, g, out_f, in_f, 0.25, X, dY)
    snap = host(g.rows).copy(), host(g.cols).copy(), host(g.values).copy()
    Xd, dYd = dev(X, torch), dev(dY, torch)
    for zeta in (-0.1, 1.0):
        with pytest.raises(binding.SnkError) as e:
            g.prune_regrow_gradient(zeta, Xd, dYd)
        assert e.value.status == binding.SNK_ERR_ARG
    with pytest.raises(binding.SnkError) as e:
        binding.snk_prune_regrow_gradient(g.handle, 0.3, Xd, dYd, batch=0)
    assert e.value.status == binding.SNK_ERR_ARG
    with pytest.raises(binding.SnkError) as e:
        binding.snk_prune_regrow_gradient(g.handle, 0.3, 0, dYd, batch=2)
    assert e.value.status == binding.SNK_ERR_ARG
    before = g.topology_version
    g.prune_regrow_gradient(0.0, Xd, dYd)      # k = 0: nothing happens
    assert g.topology_version == before
    np.testing.assert_array_equal(host(g.rows), snap[0])
    np.testing.assert_array_equal(host(g.cols), snap[1])
    np.testing.assert_array_equal(host(g.values), snap[2])
    g.close()


def test_rigl_training_stepwise(torch):
    """A RigL run: SGD steps on an MSE loss, and every 10 steps a restructure
    that grows where the current batch's gradient is largest; each restructure
    is compared with the oracle on the GPU's current state."""
    out_f, in_f, b = 800, 600, 4
    lay = synth.make_layer(out_f, in_f, 90, 0.01, 41, 42)
    X = synth.normal((b, in_f), 1.0, 43)
    T = dev(synth.normal((b, out_f), 1.0, 44), torch)
    Xd = dev(X, torch)
    g = make_gpu_layer(torch, lay)
    for step in range(30):
        Y = g.forward(Xd)
        dY = (2.0 / (b * out_f)) * (Y - T)
        g.values.sub_(0.01 * g.backward_weight(Xd, dY))
        if (step + 1) % 10 == 0:
            gradient_restructure_and_compare(torch, g, out_f, in_f, 0.3, X, host(dY))
    g.close()


def test_full_size_gradient_restructure(torch):
    """10000 x 10000 at 90%, zeta = 0.3, batch 4: 3,000,000 entries pruned and
    grown at the largest gradients among 93,000,000 candidates.  Too large to
    sort on the host, so the grown set is checked through its threshold theta
    (the largest grown key): every kept entry survives with its value, k new
    zero-valued positions were grown, and exactly k - 1 candidates have a key
    below theta (the oracle's plain count over all positions).  Keys are
    unique, so this pins the set exactly."""
    out_f = in_f = 10_000
    lay = synth.make_layer(out_f, in_f, 90, 0.01, 31, 32)
    X = synth.normal((4, in_f), 1.0, 33)
    dY = synth.normal((4, out_f), 1.0, 34)
    g = make_gpu_layer(torch, lay)
    v0, r0, c0 = host(g.values), host(g.rows), host(g.cols)
    g.prune_regrow_gradient(0.3, dev(X, torch), dev(dY, torch))
    removed, k = oracle.prune(out_f, in_f, v0, r0, c0, 0.3)
    keep = removed == 0
    kr, kc, kv = r0[keep], c0[keep], v0[keep]
    lin0 = kr.astype(np.int64) * in_f + kc
    r1, c1, v1 = host(g.rows), host(g.cols), host(g.values)
    lin1 = r1.astype(np.int64) * in_f + c1
    assert len(lin1) == len(v0) and np.all(np.diff(lin1) > 0)
    held = np.isin(lin1, lin0)
    assert int(held.sum()) == len(lin0)
    np.testing.assert_array_equal(v1[held].view(np.uint32), kv.view(np.uint32))
    grown = lin1[~held]
    assert len(grown) == k and np.all(v1[~held].view(np.uint32) == 0)
    theta = int(oracle.grad_keys(out_f, in_f, X, dY, grown).max())
    assert oracle.grad_count_below(out_f, in_f, kr, kc, X, dY, theta) == k - 1
    g.close()
