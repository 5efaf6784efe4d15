"""The torch.nn front end (sparse_linear_layer_gb300/module.py): autograd
through the library's kernels against the oracle, and a SET training loop
whose restructures match the oracle on the module's own state.

Pages: "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
GPU" (a drop-in nn.Linear replacement, Fig. 1); "Padded-CSR: A sparse storage
format for dynamic sparse training on CPU", sec. 8.2 (SparseLinear / SET /
step())."""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import synth
from tests.gpu_util import assert_within, dev, host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("lead", [(2, 3), (4, 80)])
def test_autograd_matches_oracle(torch, lead):
    """(2, 3): 6 rows, the batch-tiled kernels; (4, 80): 320 rows, which the
    library runs on the tensor cores."""
    from sparse_linear_layer_gb300.module import SparseLinear
    out_f, in_f = 300, 200
    rows = lead[0] * lead[1]
    lay = synth.make_layer(out_f, in_f, 90, 0.1, 81, 82)
    m = SparseLinear.from_triple(in_f, out_f, dev(lay.values, torch), dev(lay.rows, torch),
                                 dev(lay.cols, torch), bias=True)
    with torch.no_grad():
        m.bias.copy_(dev(synth.normal(out_f, 0.1, 83), torch))
    x = dev(synth.normal((*lead, in_f), 1.0, 84), torch).requires_grad_(True)
    G = dev(synth.normal((*lead, out_f), 1.0, 85), torch)
    y = m(x)
    assert y.shape == (*lead, out_f)
    (y * G).sum().backward()
    can = oracle.canonicalize(out_f, in_f, lay.values, lay.rows, lay.cols)
    v, r, c = can["values"], can["rows"], can["cols"]
    X2 = host(x.detach()).reshape(rows, in_f)
    G2 = host(G).reshape(rows, out_f)
    yr, ay = oracle.forward(out_f, in_f, v, r, c, X2, host(m.bias.detach()))
    assert_within(host(y.detach()).reshape(rows, out_f), yr, ay, "forward")
    dxr, ax = oracle.backward_input(out_f, in_f, v, r, c, G2)
    assert_within(host(x.grad).reshape(rows, in_f), dxr, ax, "input grad")
    dwr, aw, dbr, ab = oracle.backward_weight(out_f, in_f, r, c, X2, G2)
    assert_within(host(m.values.grad), dwr, aw, "values grad")
    assert_within(host(m.bias.grad), dbr, ab, "bias grad")
    np.testing.assert_array_equal(host(m.rows), r)
    m.close()


def test_set_training_loop_restructures_like_the_oracle(torch):
    from sparse_linear_layer_gb300.module import SET, SparseLinear
    torch.manual_seed(0)
    in_f, out_f, b = 400, 300, 8
    m = SparseLinear(in_f, out_f, 0.9, bias=True, seed=91)
    assert m.nnz == synth.nnz_for(out_f, in_f, 90)
    opt = torch.optim.SGD(m.parameters(), lr=0.05)
    algo = SET([m], zeta=0.3, every=5, seed0=0x5E7)
    X = dev(synth.normal((b, in_f), 1.0, 92), torch)
    T = dev(synth.normal((b, out_f), 1.0, 93), torch)
    losses = []
    for step in range(15):
        opt.zero_grad()
        loss = ((m(X) - T) ** 2).mean()
        loss.backward()
        opt.step()
        losses.append(float(loss.detach()))
        v0, r0, c0 = host(m.values.detach()), host(m.rows), host(m.cols)
        if algo.step():
            seed = 0x5E7 + algo.restructures
            ve, re_, ce = oracle.prune_regrow(out_f, in_f, v0, r0, c0, 0.3, seed)
            np.testing.assert_array_equal(host(m.rows), re_)
            np.testing.assert_array_equal(host(m.cols), ce)
            np.testing.assert_array_equal(host(m.values.detach()).view(np.uint32),
                                          ve.view(np.uint32))
    assert algo.restructures == 3 and m.topology_version == 4
    assert losses[-1] < losses[0]
    m.close()


def test_rigl_step_through_the_module(torch):
    from sparse_linear_layer_gb300.module import SparseLinear
    in_f, out_f, b = 200, 150, 4
    m = SparseLinear(in_f, out_f, 0.8, bias=False, seed=95)
    X = dev(synth.normal((b, in_f), 1.0, 96), torch)
    G = dev(synth.normal((b, out_f), 1.0, 97), torch)
    v0, r0, c0 = host(m.values.detach()), host(m.rows), host(m.cols)
    m.prune_regrow_gradient(0.25, X, G)
    ve, re_, ce = oracle.prune_regrow_gradient(out_f, in_f, v0, r0, c0, 0.25, host(X), host(G))
    np.testing.assert_array_equal(host(m.rows), re_)
    np.testing.assert_array_equal(host(m.cols), ce)
    np.testing.assert_array_equal(host(m.values.detach()).view(np.uint32), ve.view(np.uint32))
    m.close()
