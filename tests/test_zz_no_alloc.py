"""The allocation-free forward entry point, called through the C ABI, must
give what the regular forward entry point gives, on two calls in a row.

It serves callers that cannot let the library allocate device memory (an
application that owns all device memory through its own arena, or a hot
path where cudaMalloc/cudaFree must not run).  Its scratch is a fixed array
inside the library that every call reuses, so the second call also checks
that state left by the first call does not leak into the result.  This file
is collected last on purpose.
"""
import numpy as np
import pytest

import oracle
from sparse_linear_layer_gb300 import binding, synth
from tests.gpu_util import assert_within, dev, host, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("out_f,in_f,sp,zipf,b", [
    (3000, 2000, 90, None, 4),     # several chunks, rows cut by chunk boundaries
    (768, 3072, 90, 1.2, 3),       # skewed rows, a batch that is not a power of two
    (10_000, 10_000, 99, None, 1),
])
def test_noalloc_forward_matches_regular_forward_twice(torch, out_f, in_f, sp, zipf, b):
    std = 0.05 if zipf is None else (1.0 / (in_f * (100 - sp) / 100)) ** 0.5
    lay = synth.make_layer(out_f, in_f, sp, std, 51, 52, zipf_s=zipf)
    g = binding.SparseLinear(out_f, in_f, dev(lay.values, torch), dev(lay.rows, torch),
                             dev(lay.cols, torch))
    row_ptr = g.topology()["row_ptr"]
    bias = dev(synth.normal(out_f, 1.0, 53), torch)
    for call in range(2):
        X_h = synth.normal((b, in_f), 1.0, 54 + call)
        X = dev(X_h, torch)
        Y_ref = g.forward(X, bias)
        Y = torch.full((b, out_f), float("nan"), device="cuda")
        binding.snk_forward_csr_noalloc(out_f, in_f, row_ptr, g.cols, g.values, X, bias, Y)
        torch.cuda.synchronize()
        _, A = oracle.forward(out_f, in_f, host(g.values), host(g.rows), host(g.cols), X_h,
                              host(bias))
        assert_within(host(Y), host(Y_ref).astype(np.float64), A, f"call {call}")
    g.close()


def test_noalloc_rejects_oversize_requests(torch):
    big_out = (1 << 19) + 1
    row_ptr = torch.zeros(big_out + 1, dtype=torch.int32, device="cuda")
    X = torch.zeros(1, 8, device="cuda")
    Y = torch.zeros(1, big_out, device="cuda")
    with pytest.raises(binding.SnkError) as e:
        binding.snk_forward_csr_noalloc(big_out, 8, row_ptr, None, torch.zeros(0, device="cuda"),
                                        X, None, Y)
    assert e.value.status == binding.SNK_ERR_LIMIT
    # an operand too wide for shared memory is refused as well
    wide = 1 << 20
    row_ptr = torch.zeros(5, dtype=torch.int32, device="cuda")
    X = torch.zeros(1, wide, device="cuda")
    Y = torch.zeros(1, 4, device="cuda")
    with pytest.raises(binding.SnkError) as e:
        binding.snk_forward_csr_noalloc(4, wide, row_ptr, None, torch.zeros(0, device="cuda"), X,
                                        None, Y)
    assert e.value.status == binding.SNK_ERR_LIMIT
