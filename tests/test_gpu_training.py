"""Training runs at the benchmark layer's full size, checked step by step.

"Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU",
Fig. 3 / Table 3: the 10000 x 10000 layer trained for 100 SGD iterations at
batch 4 (90 / 95 / 99 % sparsity); "Padded-CSR: A sparse storage format for
dynamic sparse training on CPU", sec. 8.2: SET with drop fraction 0.3.

A step is forward (with bias), the MSE gradient dY = 2 (Y - T) / (b * out)
against a fixed random target (computed by torch on the GPU: harness glue,
not part of the layer), dX, dW and db, then values -= lr * dW and
bias -= lr * db with lr = 0.01.  fp32 trajectories drift apart from an fp64
one, so each check feeds the GPU's current state (values, bias, the dY it
used) to the oracle: every 10th step, Y, dX, dW and db are compared element
by element within 1e-5 * A + 1e-6.  In the SET run, prune_regrow(0.3,
0x5E7 + i) follows every 10th step and the whole triple and its derived
views must equal the oracle's bit for bit.
"""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import synth
from tests.gpu_util import assert_within, dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu

LR = 0.01


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _check_step(g, out_f, in_f, X_h, bias, dY, Y, dX, dW, db, what):
    v, r, c = host(g.values), host(g.rows), host(g.cols)
    b_h, dY_h = host(bias), host(dY)
    Yr, Ay = oracle.forward(out_f, in_f, v, r, c, X_h, b_h)
    assert_within(host(Y), Yr, Ay, f"{what}: forward")
    dXr, Ax = oracle.backward_input(out_f, in_f, v, r, c, dY_h)
    assert_within(host(dX), dXr, Ax, f"{what}: backward_input")
    dWr, Aw, dbr, Ab = oracle.backward_weight(out_f, in_f, r, c, X_h, dY_h)
    assert_within(host(dW), dWr, Aw, f"{what}: backward_weight")
    assert_within(host(db), dbr, Ab, f"{what}: bias grad")


def _train(torch, sparsity, b, steps, seeds, check_every=10, set_every=None, set_seed=0x5E7):
    out_f = in_f = 10_000
    s_sup, s_val, s_x, s_t = seeds
    lay = synth.make_layer(out_f, in_f, sparsity, 0.01, s_sup, s_val)
    g = make_gpu_layer(torch, lay)
    X_h = synth.normal((b, in_f), 1.0, s_x)
    X = dev(X_h, torch)
    T = dev(synth.normal((b, out_f), 1.0, s_t), torch)
    bias = torch.zeros(out_f, device="cuda")
    restructures = 0
    losses = []
    for step in range(steps):
        Y = g.forward(X, bias)
        dY = (2.0 / (b * out_f)) * (Y - T)
        dX = g.backward_input(dY)
        dW, db = g.backward_weight(X, dY, with_bias=True)
        losses.append(float(((Y - T) ** 2).mean()))
        if step % check_every == 0 or step == steps - 1:
            torch.cuda.synchronize()
            _check_step(g, out_f, in_f, X_h, bias, dY, Y, dX, dW, db, f"step {step}")
        g.values.sub_(LR * dW)
        bias.sub_(LR * db)
        if set_every and (step + 1) % set_every == 0:
            torch.cuda.synchronize()
            v0, r0, c0 = host(g.values), host(g.rows), host(g.cols)
            ver = g.topology_version
            seed = set_seed + restructures
            g.prune_regrow(0.3, seed)
            ve, re_, ce = oracle.prune_regrow(out_f, in_f, v0, r0, c0, 0.3, seed)
            np.testing.assert_array_equal(host(g.rows), re_, err_msg=f"rows after step {step}")
            np.testing.assert_array_equal(host(g.cols), ce, err_msg=f"cols after step {step}")
            np.testing.assert_array_equal(host(g.values).view(np.uint32), ve.view(np.uint32),
                                          err_msg=f"values after step {step}")
            assert g.topology_version == ver + 1
            t = g.topology()
            can = oracle.canonicalize(out_f, in_f, ve, re_, ce)
            for key in ("row_ptr", "col_ptr", "rows_c", "perm"):
                np.testing.assert_array_equal(host(t[key]), can[key], err_msg=f"{key} after step {step}")
            restructures += 1
    g.close()
    return losses, restructures


def test_sgd_100_steps_full_size(torch):
    """10000 x 10000 at 90 %, batch 4, 100 SGD steps: every 10th step (and
    the last) matches the oracle on the GPU's current state, and the loss
    goes down."""
    losses, _ = _train(torch, 90, 4, 100, (21, 22, 23, 24))
    assert losses[-1] < losses[0]


@pytest.mark.parametrize("sparsity,b", [(95, 16), (99, 64)])
def test_sgd_other_sparsities_and_batches(torch, sparsity, b):
    """The same run at the other sparsities of the sweep, with batches that
    take the global-memory operand path: 30 steps, checked every 10th."""
    losses, _ = _train(torch, sparsity, b, 30, (21, 22, 23, 24))
    assert losses[-1] < losses[0]


def test_set_training_100_steps_full_size(torch):
    """10000 x 10000 at 90 %, batch 4, 100 SGD steps with a SET restructure
    (drop 0.3 of the smallest magnitudes, regrow as many seeded positions at
    zero) after every 10th step: each of the 10 restructures equals the
    oracle's bit for bit, and the products stay within the tolerance."""
    _, n = _train(torch, 90, 4, 100, (31, 32, 33, 34), set_every=10)
    assert n == 10
