"""CUDA-graph capture of the layer's calls (inference-latency mode and a
captured training step).

snk_forward, snk_backward_input and snk_backward_weight only enqueue kernels
on the caller's stream: no allocation, no synchronisation, and the handle's
scratch (cross-block partials, arrival counters) is returned to its initial
state by the kernels themselves.  So a captured call replays to the same
result as a direct one, bit for bit, and a graph captured before a
restructure stays valid after it (the topology arrays keep their addresses,
nnz is fixed).  Shapes: the 5000 x 5000 GAMLP-shaped layer of [SNACK] Table 6
and the 12500 x 10000 layer of [SNACK] Table 10, batch 1."""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import synth
from tests.gpu_util import assert_within, dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _capture(torch, fn):
    """Warm fn up on a side stream, then capture one call of it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("out_f,in_f,sp", [(5000, 5000, 90), (5000, 5000, 99), (12500, 10000, 90)])
def test_forward_graph_replay_is_bit_identical(torch, out_f, in_f, sp):
    from sparse_linear_layer_gb300 import binding
    lay = synth.make_layer(out_f, in_f, sp, 0.01, 61, 62)
    g = make_gpu_layer(torch, lay)
    X = dev(synth.normal((1, in_f), 1.0, 63), torch)
    bias = dev(synth.normal((out_f,), 0.1, 64), torch)
    Y = torch.empty((1, out_f), device="cuda")
    graph = _capture(torch, lambda: binding.snk_forward(g.handle, X, bias, Y))
    Y_direct = torch.empty_like(Y)
    for step in range(3):
        X.copy_(dev(synth.normal((1, in_f), 1.0, 70 + step), torch))
        graph.replay()
        binding.snk_forward(g.handle, X, bias, Y_direct)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y_direct), f"replay {step} differs from the direct call"
    # and the replayed result is the product itself
    ref, A = oracle.forward(lay.out_f, lay.in_f, lay.values, lay.rows, lay.cols,
                            host(X).astype(np.float32), host(bias).astype(np.float32))
    assert_within(host(Y), ref, A, "graph forward")
    g.close()


def test_training_step_graph_survives_restructure(torch):
    """forward + dX + dW/db captured once; replays match direct calls before
    and after prune_regrow rewrote the topology in place."""
    from sparse_linear_layer_gb300 import binding
    lay = synth.make_layer(3072, 768, 90, 0.05, 64, 65)
    g = make_gpu_layer(torch, lay)
    b = 4
    X = dev(synth.normal((b, 768), 1.0, 66), torch)
    dY = dev(synth.normal((b, 3072), 1.0, 67), torch)
    Y = torch.empty((b, 3072), device="cuda")
    dX = torch.empty((b, 768), device="cuda")
    dW = torch.empty(g.nnz, device="cuda")
    db = torch.empty(3072, device="cuda")

    def step():
        binding.snk_forward(g.handle, X, None, Y)
        binding.snk_backward_input(g.handle, dY, dX)
        binding.snk_backward_weight(g.handle, X, dY, dW, db)

    graph = _capture(torch, step)
    for phase in range(2):
        if phase == 1:
            g.prune_regrow(0.3, 0x5E7)
            g.values.add_(0.01)  # new entries get non-zero values too
            torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (Y, dX, dW, db)]
        step()
        torch.cuda.synchronize()
        for name, a, b_ in zip(("Y", "dX", "dW", "db"), got, (Y, dX, dW, db)):
            assert torch.equal(a, b_), f"phase {phase}: replayed {name} differs"
    assert g.topology_version == 2
    g.close()
