"""Large-batch products on the tensor cores (forward, dX and dW / db) against
the oracle.

"Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU",
appendix Table 13, trains the layer at batch 4096.  The library runs such
batches by densifying tiles of W in shared memory and multiplying them on the
tensor cores with an fp16 hi/lo split of both operands.  The cases here:
- force that path (SNK_LARGE_BATCH=on) on small shapes that span several tiles
  and leave ragged tails in every dimension, including reduction lengths that
  are not a multiple of 4 (scalar operand loads) and a batch of one row;
- take it by default (batch >= 256) on the 10000 x 10000 layer of the
  benchmark, checking rows at the edges of the 128-row batch tiles;
- use inputs that are all positive, where a long chain in the tensor core's
  truncating fp32 accumulator would drift outside the tolerance;
- rebuild the tile-ordered views after a restructure, and replay a CUDA graph;
- feed inf and NaN, and rows or segments whose values span 1e8, which the
  fp16 split cannot carry: those outputs are recomputed per stored entry.
Every element is compared with |gpu - oracle| <= 1e-5 * A + 1e-6 (and the same
NaN or infinity where the oracle has one).
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


def _check(torch, lay, X, dY, bias, rows=None, weight=True):
    """forward (with bias), dX and dW / db through the library vs the
    oracle; rows limits the forward and dX comparison to those batch rows
    (dW and db always reduce over the whole batch)."""
    g = make_gpu_layer(torch, lay)
    can = oracle.canonicalize(lay.out_f, lay.in_f, lay.values, lay.rows, lay.cols)
    v, r, c = can["values"], can["rows"], can["cols"]
    Xd, dYd = dev(X, torch), dev(dY, torch)
    Y = g.forward(Xd, None if bias is None else dev(bias, torch))
    dX = g.backward_input(dYd)
    if weight:
        dW, db = g.backward_weight(Xd, dYd, with_bias=True)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    Yr, Ay = oracle.forward(lay.out_f, lay.in_f, v, r, c, X[sel], bias)
    dXr, Ax = oracle.backward_input(lay.out_f, lay.in_f, v, r, c, dY[sel])
    assert_within(host(Y)[sel], Yr, Ay, "forward")
    assert_within(host(dX)[sel], dXr, Ax, "backward_input")
    if weight:
        dWr, Aw, dbr, Ab = oracle.backward_weight(lay.out_f, lay.in_f, r, c, X, dY)
        assert_within(host(dW), dWr, Aw, "backward_weight")
        assert_within(host(db), dbr, Ab, "bias grad")
    g.close()


@pytest.mark.parametrize("out_f,in_f,sp,b", [
    (300, 200, 90, 130),      # 2 x 2 batch tiles, ragged segment and window tails
    (1000, 700, 95, 257),     # 3 batch tiles, last one a single row
    (513, 1030, 50, 1),       # one batch row
    (260, 203, 80, 129),      # forward reduction length 203: scalar operand loads
    (203, 260, 80, 129),      # the same for dX
    (64, 64, 0, 200),         # fully dense W
    (450, 390, 90, 4500),     # weight gradient over two batch chunks (4416 + 84 rows)
    (1000, 700, 99, 300),     # sparse windows: stages cleared entry by entry, not by bulk copy
    (2000, 1500, 90, 2560),   # more output tiles than SMs (152): the last partial wave's
                              # tiles shared 2 ways (forward, 220 tiles) and 8 ways (dX, 160)
    (1000, 700, 90, 8192),    # forward: 384 tiles, two full waves and 80 tiles one per CTA
    (192, 4000, 90, 128),     # forward: one tile of 63 windows shared 8 ways
])
def test_forced_small_shapes(torch, monkeypatch, out_f, in_f, sp, b):
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    lay = synth.make_layer(out_f, in_f, sp, 0.05, 81, 82)
    X = synth.normal((b, in_f), 1.0, 83)
    dY = synth.normal((b, out_f), 1.0, 84)
    bias = synth.normal(out_f, 0.1, 85)
    _check(torch, lay, X, dY, bias)


def test_default_dispatch_full_size(torch, monkeypatch):
    """10000 x 10000 at 90%, batch 512: the path the library picks by itself."""
    monkeypatch.delenv("SNK_LARGE_BATCH", raising=False)
    lay = synth.make_layer(10_000, 10_000, 90, 0.01, 21, 22)
    b = 512
    X = synth.normal((b, 10_000), 1.0, 86)
    dY = synth.normal((b, 10_000), 1.0, 87)
    rows = np.array([0, 1, 127, 128, 255, 256, 383, 384, 510, 511])
    _check(torch, lay, X, dY, None, rows, weight=False)


def test_default_dispatch_weight_gradient(torch, monkeypatch):
    """dW and db at 5000 x 5000, 90%, batch 1024 (every entry of W)."""
    monkeypatch.delenv("SNK_LARGE_BATCH", raising=False)
    lay = synth.make_layer(5000, 5000, 90, 0.01, 11, 12)
    b = 1024
    X = synth.normal((b, 5000), 1.0, 101)
    dY = synth.normal((b, 5000), 1.0, 102)
    g = make_gpu_layer(torch, lay)
    can = oracle.canonicalize(lay.out_f, lay.in_f, lay.values, lay.rows, lay.cols)
    dW, db = g.backward_weight(dev(X, torch), dev(dY, torch), with_bias=True)
    torch.cuda.synchronize()
    dWr, Aw, dbr, Ab = oracle.backward_weight(5000, 5000, can["rows"], can["cols"], X, dY)
    assert_within(host(dW), dWr, Aw, "backward_weight")
    assert_within(host(db), dbr, Ab, "bias grad")
    g.close()


@pytest.mark.parametrize("b", [95, 96])
def test_first_tier_boundary(torch, monkeypatch, b):
    """2000 x 1500 at 90% (10% stored): 95 rows run batch-tiled, 96 on the
    tensor cores (the first tier); both meet the contract."""
    monkeypatch.delenv("SNK_LARGE_BATCH", raising=False)
    lay = synth.make_layer(2000, 1500, 90, 0.05, 161, 162)
    X = synth.normal((b, 1500), 1.0, 163)
    dY = synth.normal((b, 2000), 1.0, 164)
    bias = synth.normal(2000, 0.1, 165)
    _check(torch, lay, X, dY, bias)


@pytest.mark.parametrize("b", [1300, 4300])
def test_weight_gradient_blocks_per_cta(torch, monkeypatch, b):
    """dW and db at 3000 x 2900, 90%: 24 x 16 = 384 blocks of W, two or
    three per CTA of the persistent kernel.  b = 1300 gives 21 batch windows
    (the last one ragged), so three accumulator turns per block and an odd
    number of turns per CTA; b = 4300 runs two batch chunks (4160 + 140
    rows), the second adding to the first.  A repeat call gives the same
    bits."""
    monkeypatch.delenv("SNK_LARGE_BATCH", raising=False)
    lay = synth.make_layer(3000, 2900, 90, 0.02, 151, 152)
    X = synth.normal((b, 2900), 1.0, 153)
    dY = synth.normal((b, 3000), 1.0, 154)
    g = make_gpu_layer(torch, lay)
    can = oracle.canonicalize(lay.out_f, lay.in_f, lay.values, lay.rows, lay.cols)
    Xd, dYd = dev(X, torch), dev(dY, torch)
    dW, db = g.backward_weight(Xd, dYd, with_bias=True)
    dW2, _ = g.backward_weight(Xd, dYd, with_bias=True)
    torch.cuda.synchronize()
    assert torch.equal(dW, dW2), "repeat call differs"
    dWr, Aw, dbr, Ab = oracle.backward_weight(3000, 2900, can["rows"], can["cols"], X, dY)
    assert_within(host(dW), dWr, Aw, "backward_weight")
    assert_within(host(db), dbr, Ab, "bias grad")
    g.close()


@pytest.mark.parametrize("out_f,in_f", [(300, 10_000), (10_000, 300)])
def test_all_positive_long_reduction(torch, monkeypatch, out_f, in_f):
    """Sign-coherent sums over 10000 terms: every rounding error of a
    truncating accumulator has the same sign, so only short accumulation
    chains stay within 1e-5 * A."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    lay = synth.make_layer(out_f, in_f, 50, 1.0, 88, 89)
    lay.values = np.abs(lay.values).astype(np.float32) + np.float32(0.01)
    b = 130
    X = np.abs(synth.normal((b, in_f), 1.0, 90)).astype(np.float32)
    dY = np.abs(synth.normal((b, out_f), 1.0, 91)).astype(np.float32)
    _check(torch, lay, X, dY, None)


def test_views_follow_restructure(torch, monkeypatch):
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    lay = synth.make_layer(700, 900, 90, 0.05, 92, 93)
    g = make_gpu_layer(torch, lay)
    b = 140
    X = synth.normal((b, 900), 1.0, 94)
    dY = synth.normal((b, 700), 1.0, 95)
    Xd, dYd = dev(X, torch), dev(dY, torch)
    for step in range(3):
        if step:
            g.prune_regrow(0.3, 0x5E7 + step)
            g.values.copy_(dev(synth.normal(g.nnz, 0.05, 96 + step), torch))
        Y = g.forward(Xd)
        dX = g.backward_input(dYd)
        dW = g.backward_weight(Xd, dYd)
        torch.cuda.synchronize()
        v, r, c = host(g.values), host(g.rows), host(g.cols)
        Yr, Ay = oracle.forward(700, 900, v, r, c, X, None)
        dXr, Ax = oracle.backward_input(700, 900, v, r, c, dY)
        dWr, Aw, _, _ = oracle.backward_weight(700, 900, r, c, X, dY)
        assert_within(host(Y), Yr, Ay, f"forward after {step} restructures")
        assert_within(host(dX), dXr, Ax, f"backward_input after {step} restructures")
        assert_within(host(dW), dWr, Aw, f"backward_weight after {step} restructures")
    g.close()


def test_graph_replay_matches_direct(torch, monkeypatch):
    """After a first call has built the views, forward, dX and dW only
    enqueue kernels: a captured step replays to the direct result bit for
    bit, also after a restructure rebuilt the views in place."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    from sparse_linear_layer_gb300 import binding
    lay = synth.make_layer(600, 500, 90, 0.05, 97, 98)
    g = make_gpu_layer(torch, lay)
    b = 300
    X = dev(synth.normal((b, 500), 1.0, 99), torch)
    dY = dev(synth.normal((b, 600), 1.0, 100), torch)
    Y = torch.empty((b, 600), device="cuda")
    dX = torch.empty((b, 500), device="cuda")
    dW = torch.empty(g.nnz, device="cuda")
    db = torch.empty(600, device="cuda")

    def step():
        binding.snk_forward(g.handle, X, None, Y)
        binding.snk_backward_input(g.handle, dY, dX)
        binding.snk_backward_weight(g.handle, X, dY, dW, db)

    step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for phase in range(2):
        if phase:
            g.prune_regrow(0.3, 0x5E7)
            g.values.add_(0.01)
            torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got = [t_.clone() for t_ in (Y, dX, dW, db)]
        step()
        torch.cuda.synchronize()
        for name, a_, b_ in zip(("Y", "dX", "dW", "db"), got, (Y, dX, dW, db)):
            assert torch.equal(a_, b_), f"phase {phase}: replayed {name} differs"
    g.close()


def _split_repr(a, axis):
    """Host emulation of the tensor path's operand split: each row (axis=1)
    or column (axis=0) scaled by the power of two that brings its largest
    finite magnitude into [2^13, 2^14), written as fp16 hi + fp16 lo, and
    scaled back.  Used only to show that an input defeats the split."""
    a = np.asarray(a, np.float32)
    mag = np.where(np.isfinite(a), np.abs(a), 0).astype(np.float64)
    m = mag.max(axis=axis, keepdims=True)
    ex = np.where(m > 0, 14 - np.frexp(np.where(m > 0, m, 1.0))[1], 0)
    s = np.ldexp(a.astype(np.float64), ex)
    hi = s.astype(np.float16).astype(np.float64)
    lo = (s - hi).astype(np.float16).astype(np.float64)
    return np.ldexp(hi + lo, -ex)


def _violates(gpu_like, ref, A):
    err = np.abs(np.asarray(gpu_like, np.float64) - ref)
    return bool((err > 1e-5 * A + 1e-6).any())


def test_non_finite_inputs_follow_the_definition(torch, monkeypatch):
    """inf and NaN in X, dY and W: the outputs match the oracle entry by
    entry (NaN where it has NaN, the same infinity where it has one, within
    the tolerance elsewhere), although a densified tile multiplies the stored
    zeros too: the rows and segments holding them are recomputed per entry."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    out_f, in_f, b = 300, 200, 130
    lay = synth.make_layer(out_f, in_f, 90, 0.05, 103, 104)
    can = oracle.canonicalize(out_f, in_f, lay.values, lay.rows, lay.cols)
    v, r, c = can["values"].copy(), can["rows"], can["cols"]
    X = synth.normal((b, in_f), 1.0, 105)
    dY = synth.normal((b, out_f), 1.0, 106)
    # a row whose two stored columns meet +inf and -inf (NaN there), a NaN,
    # an inf that meets a stored zero (NaN), and infinities in the tail tile
    k0 = int(can["row_ptr"][40])
    ca, cb = int(c[k0]), int(c[k0 + 1])
    v[k0], v[k0 + 1] = 0.5, 0.5
    X[3, ca], X[3, cb] = np.inf, -np.inf
    X[7, 11] = np.nan
    kz = int(can["row_ptr"][90])
    v[kz] = 0.0
    X[64, int(c[kz])] = np.inf
    X[129, 0] = -np.inf
    dY[5, 17] = np.nan
    dY[128, 299] = np.inf
    dY[70, r[k0]] = -np.inf
    # non-finite values in W: each poisons one segment of either side
    v[int(can["row_ptr"][150])] = np.inf
    v[int(can["row_ptr"][151])] = np.nan
    v[int(can["row_ptr"][299])] = -np.inf
    bias = synth.normal(out_f, 0.1, 107)
    lay2 = synth.Layer(out_f, in_f, v, r, c)
    _check(torch, lay2, X, dY, bias)


def test_wide_range_dense_rows(torch, monkeypatch):
    """Rows of X and dY holding one value near 1e8 among N(0, 1) values: after
    scaling, the small values fall under fp16's normal range.  The emulated
    split alone misses the tolerance; the library recomputes those rows."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    out_f, in_f, b = 300, 200, 130
    lay = synth.make_layer(out_f, in_f, 90, 0.05, 111, 112)
    can = oracle.canonicalize(out_f, in_f, lay.values, lay.rows, lay.cols)
    X = synth.normal((b, in_f), 1.0, 113)
    dY = synth.normal((b, out_f), 1.0, 114)
    X[5, 17] = 1.0e8
    X[100, 3] = -3.0e7
    dY[9, 250] = 1.0e8
    Yr, Ay = oracle.forward(out_f, in_f, can["values"], can["rows"], can["cols"], X, None)
    Ye, _ = oracle.forward(out_f, in_f, can["values"], can["rows"], can["cols"],
                           _split_repr(X, 1).astype(np.float32), None)
    assert _violates(Ye, Yr, Ay), "the case must defeat the plain split"
    dXr, Ax = oracle.backward_input(out_f, in_f, can["values"], can["rows"], can["cols"], dY)
    dXe, _ = oracle.backward_input(out_f, in_f, can["values"], can["rows"], can["cols"],
                                   _split_repr(dY, 1).astype(np.float32))
    assert _violates(dXe, dXr, Ax), "the case must defeat the plain split"
    _check(torch, lay, X, dY, None)


def test_wide_range_segments_of_w(torch, monkeypatch):
    """A row and a column of W each holding one value near 1e8 among
    N(0, 0.05^2) values, with the operand zero where that value would make
    the tolerance loose: the emulated split of W alone misses it; the library
    recomputes those segments for every batch row."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    out_f, in_f, b = 300, 200, 130
    lay = synth.make_layer(out_f, in_f, 90, 0.05, 121, 122)
    can = oracle.canonicalize(out_f, in_f, lay.values, lay.rows, lay.cols)
    v, r, c = can["values"].copy(), can["rows"], can["cols"]
    k_big = int(can["row_ptr"][33])        # forward: row 33 of W
    v[k_big] = 1.0e8
    c_big = int(c[k_big])
    col_idx = np.nonzero(c == 77)[0]       # dX: column 77 of W
    k_col = int(col_idx[0])
    v[k_col] = -1.0e8
    r_col = int(r[k_col])
    X = synth.normal((b, in_f), 1.0, 123)
    dY = synth.normal((b, out_f), 1.0, 124)
    X[::2, c_big] = 0.0                    # half the rows do not meet the big value
    dY[::2, r_col] = 0.0
    Yr, Ay = oracle.forward(out_f, in_f, v, r, c, X, None)
    We = np.empty_like(v)
    for o in range(out_f):
        lo_, hi_ = int(can["row_ptr"][o]), int(can["row_ptr"][o + 1])
        if hi_ > lo_:
            We[lo_:hi_] = _split_repr(v[lo_:hi_][None, :], 1)[0]
    Ye, _ = oracle.forward(out_f, in_f, We.astype(np.float32), r, c, X, None)
    assert _violates(Ye, Yr, Ay), "the case must defeat the plain split"
    _check(torch, synth.Layer(out_f, in_f, v, r, c), X, dY, None)


def test_wide_range_weight_gradient_columns(torch, monkeypatch):
    """dW when a column of dY and a column of X hold one value near 1e8 among
    N(0, 1) values (with zeros where it would make the tolerance loose): the
    rows and columns of W they feed are recomputed over the whole batch."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    out_f, in_f, b = 300, 200, 130
    lay = synth.make_layer(out_f, in_f, 90, 0.05, 131, 132)
    X = synth.normal((b, in_f), 1.0, 133)
    dY = synth.normal((b, out_f), 1.0, 134)
    dY[4, 21] = 1.0e8
    X[4, :] = 0.0                          # the big dY value meets no X value
    X[9, 150] = -1.0e8
    dY[9, :] = 0.0
    can = oracle.canonicalize(out_f, in_f, lay.values, lay.rows, lay.cols)
    dWr, Aw, _, _ = oracle.backward_weight(out_f, in_f, can["rows"], can["cols"], X, dY)
    dWe, _, _, _ = oracle.backward_weight(out_f, in_f, can["rows"], can["cols"],
                                          _split_repr(X, 0).astype(np.float32),
                                          _split_repr(dY, 0).astype(np.float32))
    assert _violates(dWe, dWr, Aw), "the case must defeat the plain split"
    _check(torch, lay, X, dY, None)


def test_batch_chunks_and_empty_segments(torch, monkeypatch):
    """A batch over the 8192-row chunk of the dense workspace (two launch
    sequences for forward and dX; two batch chunks of 4672 rows for dW), on
    a layer whose many empty rows and columns leave whole tiles without
    entries (outputs = bias or 0)."""
    monkeypatch.setenv("SNK_LARGE_BATCH", "on")
    lay = synth.make_layer(400, 300, 80, 0.05, 106, 107, zipf_s=1.2)
    # empty every third row and every fifth column, and all of rows 192-383
    # (one whole segment tile) and columns 64-127 (one whole window)
    keep = ((lay.rows % 3) != 0) & ((lay.cols % 5) != 0)
    keep &= ~((lay.rows >= 192) & (lay.rows < 384)) & ~((lay.cols >= 64) & (lay.cols < 128))
    lay.values, lay.rows, lay.cols = lay.values[keep], lay.rows[keep], lay.cols[keep]
    assert (np.bincount(lay.rows, minlength=400) == 0).sum() > 250
    b = 8300
    X = synth.normal((b, 300), 1.0, 108)
    dY = synth.normal((b, 400), 1.0, 109)
    bias = synth.normal(400, 0.1, 110)
    _check(torch, lay, X, dY, bias)

