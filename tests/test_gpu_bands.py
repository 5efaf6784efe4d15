"""Row runs over column bands: dW at batch tiles whose operand does not fit
shared memory (8 or more batch columns of a wide operand).

Each block stages one band of the transposed operand's rows (a TMA bulk
copy) and its warps walk, row by row, the run of each row's entries in that
band (contiguous in canonical order), writing every gradient in place.  The
layer takes the bands when its runs average at least 40 entries and a
block's entries are at least twice its band's columns; the other cases keep
the row-order kernel.  Every case compares forward, dX, dW and db with the
oracle element by element within |gpu - oracle| <= 1e-5 * A + 1e-6:
  - the benchmark layer at b = 8, 32 (2 and 6 bands) and 95% at b = 8, 64;
    99% at b = 8 stays on the row-order kernel (too few entries per block);
  - the GPT-2-shaped layers with Zipf rows at b = 64 (4 bands on the
    down-projection, in = 3072; the up-projection's 768 columns fit);
  - ragged shapes and batch sizes (the last band narrower, b = 13, 33, and
    130 over three batch tiles on the batch-tiled path, dW accumulated
    across tiles of both kinds);
  - empty bands, and a single dense row;
  - repeat calls (bit-identical), a restructure (the tables rebuilt in place)
    and a CUDA-graph replay.

Pages: "Padded-CSR: A sparse storage format for dynamic sparse training on
CPU" (sec. 7.1); "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural
Networks on GPU" (Fig. 3: the layer at batch 1..64).
"""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import binding, synth
from tests.gpu_util import assert_within, dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _products(torch, g, X_h, dY_h, bias_h):
    Y = g.forward(dev(X_h, torch), None if bias_h is None else dev(bias_h, torch))
    dX = g.backward_input(dev(dY_h, torch))
    dW, db = g.backward_weight(dev(X_h, torch), dev(dY_h, torch), with_bias=True)
    torch.cuda.synchronize()
    return host(Y), host(dX), host(dW), host(db)


def _check(torch, g, lay, b, seed, bias=True, repeat=True):
    X = synth.normal((b, lay.in_f), 1.0, seed)
    dY = synth.normal((b, lay.out_f), 1.0, seed + 1)
    bb = synth.normal(lay.out_f, 1.0, seed + 2) if bias else None
    Y, dX, dW, db = _products(torch, g, X, dY, bb)
    if repeat:
        Y2, dX2, dW2, db2 = _products(torch, g, X, dY, bb)
        for p, q, what in ((Y, Y2, "forward"), (dX, dX2, "dX"), (dW, dW2, "dW")):
            assert np.array_equal(p, q, equal_nan=True), f"{what}: repeat call differs"
    v, r, c = host(g.values), host(g.rows), host(g.cols)
    Yr, Ay = oracle.forward(lay.out_f, lay.in_f, v, r, c, X, bb)
    dXr, Ax = oracle.backward_input(lay.out_f, lay.in_f, v, r, c, dY)
    dWr, Aw, dbr, Ab = oracle.backward_weight(lay.out_f, lay.in_f, r, c, X, dY)
    assert_within(Y, Yr, Ay, f"forward b={b}")
    assert_within(dX, dXr, Ax, f"dX b={b}")
    assert_within(dW, dWr, Aw, f"dW b={b}")
    assert_within(db, dbr, Ab, f"db b={b}")


@pytest.mark.parametrize("sp,b", [(90, 8), (90, 32), (95, 8), (95, 64), (99, 8)])
def test_benchmark_layer(torch, sp, b):
    lay = synth.make_layer(10_000, 10_000, sp, 0.01, 21, 22)
    g = make_gpu_layer(torch, lay)
    _check(torch, g, lay, b, 31)
    g.close()


@pytest.mark.parametrize("out_f,in_f", [(3072, 768), (768, 3072)])
def test_gpt2_mlp_layers_zipf_rows(torch, out_f, in_f):
    """3072 operand columns at b = 64 take 4 bands (768 KB) on the
    down-projection (in = 3072); the up-projection's 768 fit shared memory."""
    std = (1.0 / (in_f * 0.1)) ** 0.5
    lay = synth.make_layer(out_f, in_f, 90, std, 41, 42, zipf_s=1.2)
    g = make_gpu_layer(torch, lay)
    _check(torch, g, lay, 64, 43)
    g.close()


@pytest.mark.parametrize("b", [13, 33, 130])
def test_ragged_bands_and_batches(torch, monkeypatch, b):
    """9001 columns: the last band narrower than the others; b = 130 runs
    three batch tiles (64 and 64 on bands, then 2 on the row-order kernel),
    dW accumulated across them (the tensor path is switched off)."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "off")
    lay = synth.make_layer(1_500, 9_001, 90, 0.05, 51, 52)
    g = make_gpu_layer(torch, lay)
    _check(torch, g, lay, b, 53, repeat=(b != 130))
    g.close()


def test_empty_bands_and_dense_row(torch):
    """Columns from 6,000 on hold no entry (the last of 3 bands at b = 16 and
    the last 3 of 10 at b = 64 are empty) and row 5 holds every column below
    6,000 (one run far longer than the others in each non-empty band)."""
    out_f, in_f = 4_000, 9_000
    lay = synth.make_layer(out_f, 6_000, 90, 0.05, 61, 62)
    keep = lay.rows != 5
    rows = np.concatenate([lay.rows[keep], np.full(6_000, 5, np.int32)])
    cols = np.concatenate([lay.cols[keep], np.arange(6_000, dtype=np.int32)])
    vals = np.concatenate([lay.values[keep], synth.normal(6_000, 0.05, 63)])
    lay = synth.Layer(out_f, in_f, vals, rows, cols)
    g = make_gpu_layer(torch, lay)
    for b in (16, 64):
        _check(torch, g, lay, b, 64 + b)
    g.close()


def test_restructure_rebuilds_the_tables(torch):
    lay = synth.make_layer(3_000, 9_000, 95, 0.05, 71, 72)
    g = make_gpu_layer(torch, lay)
    _check(torch, g, lay, 16, 73, repeat=False)
    for k in range(2):
        g.prune_regrow(0.3, 0xB0 + k)
        g.values.add_(0.01)
        _check(torch, g, lay, 16, 74 + k, repeat=False)
    g.close()


def test_graph_replay_matches_direct_calls(torch):
    """After one direct call has built the tables, captured forward / dX / dW
    calls replay to the same bits as direct calls, before and after a
    restructure (the tables are rebuilt in place)."""
    lay = synth.make_layer(3_000, 9_000, 95, 0.05, 81, 82)
    g = make_gpu_layer(torch, lay)
    b = 16
    X = dev(synth.normal((b, lay.in_f), 1.0, 83), torch)
    dY = dev(synth.normal((b, lay.out_f), 1.0, 84), torch)
    outs = [torch.empty((b, lay.out_f), device="cuda"), torch.empty((b, lay.in_f), device="cuda"),
            torch.empty(lay.nnz, device="cuda")]
    direct = [torch.empty_like(t) for t in outs]

    def step(Y, dX, dW):
        binding.snk_forward(g.handle, X, None, Y)
        binding.snk_backward_input(g.handle, dY, dX)
        binding.snk_backward_weight(g.handle, X, dY, dW, None)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(*outs)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(*outs)
    torch.cuda.synchronize()
    for rnd in range(2):
        for t in outs:
            t.zero_()
        graph.replay()
        step(*direct)
        torch.cuda.synchronize()
        for p, q, what in zip(outs, direct, ("forward", "dX", "dW")):
            assert torch.equal(p, q), f"{what}: replay differs from the direct call ({rnd})"
        g.prune_regrow(0.3, 0xC1 + rnd)
    g.close()
