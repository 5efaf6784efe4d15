"""GPU parity: every product call through the C ABI against the CPU oracle.

Topology output is compared bit for bit; fp32 products element by element
within |gpu - oracle| <= 1e-5 * A + 1e-6.  Cases span several merge-path
chunks and ragged tails, empty rows and columns, skewed (Zipf) rows, batch
sizes that are not powers of two, both operand paths (shared memory and the
global transposed copy) and the full 10000 x 10000 layers in the launch
configuration the benchmark times.

Pages: "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
GPU" (Fig. 1, Table 7); "Padded-CSR: A sparse storage format for dynamic
sparse training on CPU" (sec. 3-4, 6.1, 7.1, 7.2).
"""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import binding, synth
from tests.conftest import load_golden
from tests.gpu_util import assert_within, dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def check_all_products(torch, lay, b, bias=True, seed=7):
    X = synth.normal((b, lay.in_f), 1.0, seed)
    dY = synth.normal((b, lay.out_f), 1.0, seed + 1)
    bb = synth.normal(lay.out_f, 1.0, seed + 2) if bias else None
    g = make_gpu_layer(torch, lay)
    can = oracle.canonicalize(lay.out_f, lay.in_f, lay.values, lay.rows, lay.cols)
    np.testing.assert_array_equal(host(g.values), can["values"])
    np.testing.assert_array_equal(host(g.rows), can["rows"])
    np.testing.assert_array_equal(host(g.cols), can["cols"])
    v, r, c = can["values"], can["rows"], can["cols"]
    Xd, dYd = dev(X, torch), dev(dY, torch)
    Y = g.forward(Xd, None if bb is None else dev(bb, torch))
    dX = g.backward_input(dYd)
    dW, db = g.backward_weight(Xd, dYd, with_bias=True)
    torch.cuda.synchronize()
    Yr, Ay = oracle.forward(lay.out_f, lay.in_f, v, r, c, X, bb)
    dXr, Ax = oracle.backward_input(lay.out_f, lay.in_f, v, r, c, dY)
    dWr, Aw, dbr, Ab = oracle.backward_weight(lay.out_f, lay.in_f, r, c, X, dY)
    assert_within(host(Y), Yr, Ay, "forward")
    assert_within(host(dX), dXr, Ax, "backward_input")
    assert_within(host(dW), dWr, Aw, "backward_weight")
    assert_within(host(db), dbr, Ab, "bias grad")
    g.close()


# ---------------------------------------------------------------- pages' examples

def test_worked_example_is_exact(torch):
    gold = load_golden("pcsr_spmm_worked_example.json")
    g = binding.SparseLinear(gold["out"], gold["in"],
                             dev(np.array(gold["values"], np.float32), torch),
                             dev(np.array(gold["rows"], np.int32), torch),
                             dev(np.array(gold["cols"], np.int32), torch))
    Y = g.forward(dev(np.array(gold["x_batch_major"], np.float32), torch))
    np.testing.assert_array_equal(host(Y), np.array(gold["y_batch_major"], np.float32))
    g.close()


@pytest.mark.parametrize("name", ["pcsr_toy_4x6.json", "snack_table7_formats.json"])
def test_topology_of_printed_examples(torch, name):
    gold = load_golden(name)
    if "coo" in gold:
        v, r, c = gold["coo"]["data"], gold["coo"]["row"], gold["coo"]["col"]
    else:
        v, r, c = gold["values"], gold["rows"], gold["cols"]
    order = np.arange(len(v))[::-1]
    v = np.array(v, np.float32)[order]
    r = np.array(r, np.int32)[order]
    c = np.array(c, np.int32)[order]
    g = binding.SparseLinear(gold["out"], gold["in"], dev(v, torch), dev(r, torch), dev(c, torch))
    t = g.topology()
    can = oracle.canonicalize(gold["out"], gold["in"], v, r, c)
    for key in ("row_ptr", "col_ptr", "rows_c", "perm"):
        np.testing.assert_array_equal(host(t[key]), can[key], err_msg=key)
    if "csc" in gold:
        np.testing.assert_array_equal(host(t["col_ptr"]), gold["csc"]["indptr"])
        np.testing.assert_array_equal(host(t["rows_c"]), gold["csc"]["row"])
        np.testing.assert_array_equal(host(g.values)[host(t["perm"])], gold["csc"]["data"])
    else:
        np.testing.assert_array_equal(host(t["row_ptr"]), gold["row_ptr"])
    g.close()


# ---------------------------------------------------------------- topology

@pytest.mark.parametrize("out_f,in_f,nnz", [
    (1, 1, 1), (7, 5, 35), (500, 500, 12_500), (1000, 37, 20_000), (37, 1000, 20_000),
    (3000, 3000, 90_001), (70_000, 70_000, 50_000),   # last one: out*in > 2^32 (64-bit keys)
])
def test_topology_bit_exact(torch, out_f, in_f, nnz):
    lay = synth.Layer(out_f, in_f, synth.normal(nnz, 1.0, 4),
                      *synth.uniform_support(out_f, in_f, nnz, 3))
    g = make_gpu_layer(torch, lay)
    t = g.topology()
    can = oracle.canonicalize(out_f, in_f, lay.values, lay.rows, lay.cols)
    np.testing.assert_array_equal(host(g.rows), can["rows"])
    np.testing.assert_array_equal(host(g.cols), can["cols"])
    np.testing.assert_array_equal(host(g.values), can["values"])
    for key in ("row_ptr", "col_ptr", "rows_c", "perm"):
        np.testing.assert_array_equal(host(t[key]), can[key], err_msg=key)
    assert g.topology_version == 1
    g.close()


def test_create_rejects_duplicates_and_range_and_leaves_arrays(torch):
    r = np.array([0, 1, 1, 2], np.int32)
    c = np.array([0, 2, 2, 1], np.int32)
    v = np.array([1, 2, 3, 4], np.float32)
    rd, cd, vd = dev(r, torch), dev(c, torch), dev(v, torch)
    with pytest.raises(binding.SnkError) as e:
        binding.snk_create(3, 3, vd, rd, cd)
    assert e.value.status == binding.SNK_ERR_DUP
    np.testing.assert_array_equal(host(rd), r)
    np.testing.assert_array_equal(host(vd), v)
    c2 = dev(np.array([0, 2, 3, 1], np.int32), torch)
    with pytest.raises(binding.SnkError) as e:
        binding.snk_create(3, 3, vd, rd, c2)
    assert e.value.status == binding.SNK_ERR_RANGE
    r3 = dev(np.array([0, -1, 1, 2], np.int32), torch)
    with pytest.raises(binding.SnkError) as e:
        binding.snk_create(3, 3, vd, r3, dev(np.array([0, 0, 1, 1], np.int32), torch))
    assert e.value.status == binding.SNK_ERR_RANGE


# ---------------------------------------------------------------- products

SMALL = [
    # (out, in, sparsity %, zipf s or None)
    (500, 500, 95, None),      # 500^2 at 95%: 12,500 entries
    (64, 64, 50, None),
    (129, 77, 90, None),       # ragged everything
    (1000, 300, 99, None),     # many empty rows
    (300, 1000, 99, None),     # many empty columns
    (768, 3072, 90, 1.2),      # GPT-2 MLP down-projection shape, Zipf rows
    (3072, 768, 90, 1.2),      # up-projection shape, dense rows capped at 768
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:3])) + ("z" if s[3] else ""))
@pytest.mark.parametrize("b", [1, 2, 3, 4, 5, 8, 16, 31, 32, 64, 65])
def test_products_match_oracle(torch, shape, b):
    out_f, in_f, sp, zs = shape
    std = 0.05 if zs is None else (1.0 / (in_f * (100 - sp) / 100)) ** 0.5
    lay = synth.make_layer(out_f, in_f, sp, std, 11, 12, zipf_s=zs)
    check_all_products(torch, lay, b)


def test_single_dense_row_and_dense_column(torch):
    """Row 7 holds every column and column 3 every row: one segment far longer
    than a merge-path chunk on each side."""
    out_f, in_f = 40, 5000
    others = np.array([o for o in range(out_f) if o != 7], np.int32)
    rows = np.concatenate([np.full(in_f, 7, np.int32), others])
    cols = np.concatenate([np.arange(in_f, dtype=np.int32), np.full(len(others), 3, np.int32)])
    order = synth.rng(6).permutation(len(rows))
    lay = synth.Layer(out_f, in_f, synth.normal(len(rows), 1.0, 5), rows[order], cols[order])
    for b in (1, 4, 33):
        check_all_products(torch, lay, b)


def test_operand_larger_than_shared_memory(torch):
    """in * BP * 4 bytes exceeds shared memory: every operand row is read from
    a transposed copy in global memory (L1-cached read-only loads).
      in = 60,000 at b = 1, 4, 8; out = 20,000 (the dX operand) at b = 16, 64;
      in = 70,000 and out = 70,000, which have no 16-bit index copy, at b = 1, 4."""
    lay = synth.make_layer(50, 60_000, 99, 0.05, 21, 22)
    for b in (1, 4, 8):
        check_all_products(torch, lay, b)
    lay = synth.make_layer(20_000, 64, 90, 0.05, 23, 24)
    for b in (16, 64):
        check_all_products(torch, lay, b)
    lay = synth.make_layer(40, 70_000, 99.5, 0.05, 25, 26)
    for b in (1, 4):
        check_all_products(torch, lay, b)
    # out = 70,000: the transposed product has no 16-bit row copy either
    lay = synth.make_layer(70_000, 40, 99.5, 0.05, 27, 28)
    for b in (1, 4):
        check_all_products(torch, lay, b)


@pytest.mark.parametrize("in_f", [16_384, 28_000, 56_000])
def test_sixteen_bit_columns_of_wide_layers(torch, in_f):
    """The 16-bit column copy with its top bits in use (columns up to 55,999,
    above 32,767 from 32,768 on): b = 1 stages every width here in shared
    memory and takes the 16-bit path; b = 2 does so up to 28,000 columns and
    reads 56,000 from global memory."""
    lay = synth.make_layer(600, in_f, 98, 0.05, 61, 62)
    assert lay.cols.max() == in_f - 1
    for b in (1, 2):
        check_all_products(torch, lay, b)


def test_no_entries(torch):
    lay = synth.Layer(6, 9, np.zeros(0, np.float32), np.zeros(0, np.int32), np.zeros(0, np.int32))
    check_all_products(torch, lay, 3)


def test_permutation_matrix_is_bit_exact(torch):
    n = 4099
    p = synth.rng(3).permutation(n).astype(np.int32)
    lay = synth.Layer(n, n, np.ones(n, np.float32), np.arange(n, dtype=np.int32), p)
    g = make_gpu_layer(torch, lay)
    X = synth.normal((5, n), 1.0, 4)
    Y = host(g.forward(dev(X, torch)))
    np.testing.assert_array_equal(Y, X[:, p])
    dX = host(g.backward_input(dev(Y, torch)))
    np.testing.assert_array_equal(dX, X)
    g.close()


def test_repeat_calls_are_bit_identical_and_follow_value_updates(torch):
    """Arrival counters reset themselves; the column view gathers live values,
    so updating values in place is reflected (refresh equals rebuild)."""
    lay = synth.make_layer(2000, 1500, 90, 0.05, 31, 32)
    g = make_gpu_layer(torch, lay)
    X = dev(synth.normal((4, 1500), 1.0, 33), torch)
    dY = dev(synth.normal((4, 2000), 1.0, 34), torch)
    Y1, dX1, dW1 = g.forward(X), g.backward_input(dY), g.backward_weight(X, dY)
    Y2, dX2, dW2 = g.forward(X), g.backward_input(dY), g.backward_weight(X, dY)
    assert torch.equal(Y1, Y2) and torch.equal(dX1, dX2) and torch.equal(dW1, dW2)
    g.values.mul_(-0.5).add_(0.01)   # an SGD-like in-place update
    Y3, dX3 = g.forward(X), g.backward_input(dY)
    fresh = binding.SparseLinear(2000, 1500, g.values.clone(), g.rows.clone(), g.cols.clone())
    assert torch.equal(Y3, fresh.forward(X))
    assert torch.equal(dX3, fresh.backward_input(dY))
    fresh.close()
    g.close()


def test_non_default_stream(torch):
    lay = synth.make_layer(800, 600, 90, 0.05, 41, 42)
    g = make_gpu_layer(torch, lay)
    X = dev(synth.normal((8, 600), 1.0, 43), torch)
    ref = g.forward(X)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        Y = torch.empty_like(ref)
        binding.snk_forward(g.handle, X, None, Y, stream=s)
    s.synchronize()
    assert torch.equal(Y, ref)
    g.close()


# ---------------------------------------------------------------- full size

@pytest.mark.parametrize("sp,b", [(90, 4), (90, 1), (90, 64), (99, 4), (95, 16)])
def test_full_size_10000(torch, sp, b):
    """10000 x 10000 layers from the benchmark workload, every output element
    compared with the oracle."""
    lay = synth.make_layer(10_000, 10_000, sp, 0.01, 21, 22)
    check_all_products(torch, lay, b, bias=False, seed=23)


@pytest.mark.parametrize("sp", [80, 99])
def test_full_size_5000(torch, sp):
    lay = synth.make_layer(5000, 5000, sp, 0.01, 11, 12)
    check_all_products(torch, lay, 2, bias=False, seed=13)


@pytest.mark.parametrize("out_f,in_f,sp,b", [
    (12500, 10000, 90, 1),   # [SNACK] Table 10 layer, batch 1
    (12500, 10000, 99, 1),
    (2500, 10000, 90, 2),    # [SNACK] Fig. 5 layer
    (7500, 10000, 95, 4),    # [SNACK] Fig. 7 layer
    (5000, 5000, 95, 1),     # [SNACK] Table 6 (GAMLP-shaped) layer, batch 1
])
def test_full_size_rectangular(torch, out_f, in_f, sp, b):
    """The non-square layers of the pages' latency tables and figures, every
    output element compared with the oracle."""
    lay = synth.make_layer(out_f, in_f, sp, 0.01, 71, 72)
    check_all_products(torch, lay, b, bias=True, seed=73)
