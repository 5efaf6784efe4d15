"""The column sweep of the transposed product (batch 1..4).

dX = dY W at a batch tile of at most 4 columns walks every column of a block
with its own lanes (as many as its share of the block's entries), so that all
columns advance through the rows together.  These cases check it against the
oracle element by element within |gpu - oracle| <= 1e-5 * A + 1e-6, on the
shapes that exercise each part of its tables:
  - the benchmark layers at every batch 1..4 (ragged 3 included);
  - more non-empty columns per block than half its threads, so threads take
    several virtual lanes and keep partials in global scratch;
  - a column cut between blocks, and one column spanning about 90 blocks, so
    that a block's head and tail are the same column;
  - operand rows staged in phases (2 to 8 of them), lanes resuming at the
    quad where their column crosses each cut;
  - empty columns, and non-finite values in dY and W;
  - repeat calls (bit-identical) and restructures.

Pages: "Padded-CSR: A sparse storage format for dynamic sparse training on
CPU" (sec. 7.1: dL/dX is another SpMM through W^T; sec. 7.2: W^T read
through a permutation built once per topology).
"""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import synth
from tests.gpu_util import assert_within, dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _check_dx(torch, g, lay, dY_h):
    dY = dev(dY_h, torch)
    dX = g.backward_input(dY)
    dX2 = g.backward_input(dY)
    torch.cuda.synchronize()
    assert torch.equal(dX, dX2) or np.array_equal(host(dX), host(dX2), equal_nan=True), "repeat call differs"
    v, r, c = host(g.values), host(g.rows), host(g.cols)
    ref, A = oracle.backward_input(lay.out_f, lay.in_f, v, r, c, dY_h)
    assert_within(host(dX), ref, A, f"dX b={dY_h.shape[0]}")


def _with_dense_column(out_f, in_f, sp, col, seed):
    """Uniform support plus column `col` holding every row."""
    lay = synth.make_layer(out_f, in_f, sp, 0.05, seed, seed + 1)
    keep = lay.cols != col
    rows = np.concatenate([lay.rows[keep], np.arange(out_f, dtype=np.int32)])
    cols = np.concatenate([lay.cols[keep], np.full(out_f, col, np.int32)])
    vals = np.concatenate([lay.values[keep], synth.normal(out_f, 0.05, seed + 2)])
    return synth.Layer(out_f, in_f, vals, rows, cols)


@pytest.mark.parametrize("sp", [90, 95, 99])
def test_benchmark_layers_every_small_batch(torch, sp):
    lay = synth.make_layer(10_000, 10_000, sp, 0.01, 91, 92)
    g = make_gpu_layer(torch, lay)
    for b in (1, 2, 3, 4):
        _check_dx(torch, g, lay, synth.normal((b, 10_000), 1.0, 93 + b))
    g.close()


def test_many_columns_per_block(torch):
    """120,000 columns of about 20 entries: ~790 per block, more than half the
    block's 768 threads, so every thread takes three virtual lanes."""
    lay = synth.make_layer(2_000, 120_000, 99, 0.05, 101, 102)
    g = make_gpu_layer(torch, lay)
    for b in (1, 4):
        _check_dx(torch, g, lay, synth.normal((b, 2_000), 1.0, 103 + b))
    g.close()


def test_column_cut_between_blocks(torch):
    lay = _with_dense_column(10_000, 3_000, 90, 5, 111)
    g = make_gpu_layer(torch, lay)
    for b in (1, 3, 4):
        _check_dx(torch, g, lay, synth.normal((b, 10_000), 1.0, 114 + b))
    g.close()


def test_column_spanning_many_blocks(torch):
    """A 40,000-entry column among 64 columns (65,600 entries): it spans about
    90 blocks, each of whose head and tail it is.  Its operand does not fit
    shared memory from b = 2 on: 4 row phases at b = 2, 8 at b = 4."""
    lay = _with_dense_column(40_000, 64, 99, 17, 121)
    g = make_gpu_layer(torch, lay)
    for b in (1, 2, 4):
        _check_dx(torch, g, lay, synth.normal((b, 40_000), 1.0, 124 + b))
    g.close()


def test_row_phases_on_a_tall_layer(torch):
    """30,000 x 3,000 at 90%: 8 row phases at b = 4 and 3, 4 at b = 2, 2 at
    b = 1, with every lane resuming where its column crosses each cut."""
    lay = synth.make_layer(30_000, 3_000, 90, 0.05, 161, 162)
    g = make_gpu_layer(torch, lay)
    for b in (1, 2, 3, 4):
        _check_dx(torch, g, lay, synth.normal((b, 30_000), 1.0, 163 + b))
    g.close()


def test_empty_columns_and_ragged_shapes(torch):
    for (out_f, in_f, sp) in ((300, 1_000, 99), (129, 77, 90), (4_097, 2_051, 97)):
        lay = synth.make_layer(out_f, in_f, sp, 0.05, 131, 132)
        g = make_gpu_layer(torch, lay)
        for b in (1, 2, 3, 4):
            _check_dx(torch, g, lay, synth.normal((b, out_f), 1.0, 133 + b))
        g.close()


def test_non_finite_values(torch):
    """NaN and +-inf reach exactly the outputs whose terms hold them."""
    lay = synth.make_layer(6_000, 4_000, 90, 0.05, 141, 142)
    vals = lay.values.copy()
    vals[17] = np.inf
    vals[5_000] = np.nan
    lay = synth.Layer(lay.out_f, lay.in_f, vals, lay.rows, lay.cols)
    g = make_gpu_layer(torch, lay)
    dY = synth.normal((4, 6_000), 1.0, 143)
    dY[1, 7] = np.nan
    dY[2, 100] = -np.inf
    dY[3, 2_000] = np.inf
    _check_dx(torch, g, lay, dY)
    g.close()


def test_restructure_keeps_the_sweep_current(torch):
    lay = synth.make_layer(6_000, 4_000, 90, 0.05, 151, 152)
    g = make_gpu_layer(torch, lay)
    _check_dx(torch, g, lay, synth.normal((4, 6_000), 1.0, 153))
    for k in range(3):
        g.prune_regrow(0.3, 0xC0 + k)
        g.values.add_(0.01)
        _check_dx(torch, g, lay, synth.normal((k + 1, 6_000), 1.0, 154 + k))
    g.close()
