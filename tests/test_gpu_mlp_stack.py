"""The GPT-2-small MLP stack: 12 blocks of [sparse 768 -> 3072 (W 3072 x 768),
GELU, sparse 3072 -> 768], Zipf(1.2) row degrees, forward through all 24
layers and backward from a random upstream gradient, every layer checked
against the oracle on the GPU's own inputs to that layer (fp32 activations
drift between implementations, so the comparison is stepwise).  GELU and its
derivative are torch's (outside the library).  Pages: "Beyond Masked
Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU", Tables 4-5 (the
GPT-2 rows; the synthetic stack stands in for the model)."""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import synth
from tests.gpu_util import assert_within, dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("sp,b", [(90, 1), (90, 64), (99, 16)])
def test_mlp_stack_forward_backward(torch, sp, b):
    blocks = 12
    layers, lays = [], []
    for i in range(2 * blocks):
        out_f, in_f = (3072, 768) if i % 2 == 0 else (768, 3072)
        density = (100 - sp) / 100
        lay = synth.make_layer(out_f, in_f, sp, (1.0 / (in_f * density)) ** 0.5, 41 + 2 * i,
                               42 + 2 * i, zipf_s=1.2)
        lays.append(lay)
        layers.append(make_gpu_layer(torch, lay))
    cans = [oracle.canonicalize(l.out_f, l.in_f, l.values, l.rows, l.cols) for l in lays]
    x = dev(synth.normal((b, 768), 1.0, 43), torch)
    inputs, pre = [], []
    for i, g in enumerate(layers):
        inputs.append(x)
        y = g.forward(x)
        c = cans[i]
        yr, ay = oracle.forward(g.out_features, g.in_features, c["values"], c["rows"], c["cols"],
                                host(x), None)
        assert_within(host(y), yr, ay, f"forward layer {i}")
        if i % 2 == 0:
            pre.append(y)
            x = torch.nn.functional.gelu(y)
        else:
            x = y
    dy = dev(synth.normal((b, 768), 1.0, 44), torch)
    for i in reversed(range(len(layers))):
        g, c = layers[i], cans[i]
        dx = g.backward_input(dy)
        dw = g.backward_weight(inputs[i], dy)
        dxr, ax = oracle.backward_input(g.out_features, g.in_features, c["values"], c["rows"],
                                        c["cols"], host(dy))
        dwr, aw, _, _ = oracle.backward_weight(g.out_features, g.in_features, c["rows"], c["cols"],
                                               host(inputs[i]), host(dy))
        assert_within(host(dx), dxr, ax, f"dX layer {i}")
        assert_within(host(dw), dwr, aw, f"dW layer {i}")
        if i % 2 == 1:
            # through the GELU of the block's first layer
            yv = pre[i // 2].detach().requires_grad_(True)
            act = torch.nn.functional.gelu(yv)
            (gy,) = torch.autograd.grad(act, yv, dx)
            dy = gy.detach()
        else:
            dy = dx
    for g in layers:
        g.close()
