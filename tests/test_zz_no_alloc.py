"""The allocation-free forward entry point, called through the C ABI, checked
against the oracle on two calls in a row.

It serves callers that cannot let the library allocate device memory (an
application that owns all device memory through its own arena, or a hot
path where cudaMalloc/cudaFree must not run).  Its scratch is a fixed array
inside the library that every call reuses: partial sums of rows cut between
blocks and their arrival counters.  So each case runs twice, the batches
cross 64-row tiles (one launch per tile, all sharing the scratch), one layer
has a dense row spread over most blocks beside sparse rows (the cross-block
path that uses the scratch), and a call with more output rows runs before a
smaller one, so that anything left behind would show.  Every output is
compared with the oracle's fp64 result within 1e-5 * A + 1e-6.  This file is
collected last on purpose.
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


def _csr(torch, lay):
    """Canonical CSR of a synthetic layer on the device (oracle order)."""
    can = oracle.canonicalize(lay.out_f, lay.in_f, lay.values, lay.rows, lay.cols)
    return can, (dev(can["row_ptr"], torch), dev(can["cols"], torch), dev(can["values"], torch))


def _call_and_check(torch, lay, can, csr, b, seed, what):
    out_f, in_f = lay.out_f, lay.in_f
    row_ptr, cols, vals = csr
    bias_h = synth.normal(out_f, 1.0, seed)
    X_h = synth.normal((b, in_f), 1.0, seed + 1)
    Y = torch.full((b, out_f), float("nan"), device="cuda")
    binding.snk_forward_csr_noalloc(out_f, in_f, row_ptr, cols, vals, dev(X_h, torch),
                                    dev(bias_h, torch), Y)
    torch.cuda.synchronize()
    Yr, A = oracle.forward(out_f, in_f, can["values"], can["rows"], can["cols"], X_h, bias_h)
    assert_within(host(Y), Yr, A, what)


def _dense_row_layer(out_f, in_f, dense_row, seed):
    """A layer whose row `dense_row` holds every column, the others one entry
    each on average: the dense row is longer than many blocks' shares."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = [np.full(in_f, dense_row, np.int32)]
    cols = [np.arange(in_f, dtype=np.int32)]
    for r in range(out_f):
        if r == dense_row:
            continue
        k = int(rng.integers(0, 3))
        rows.append(np.full(k, r, np.int32))
        cols.append(np.sort(rng.choice(in_f, size=k, replace=False)).astype(np.int32))
    rows, cols = np.concatenate(rows), np.concatenate(cols)
    vals = rng.normal(0.0, 0.05, rows.size).astype(np.float32)
    return synth.Layer(out_f, in_f, vals, rows, cols)


@pytest.mark.parametrize("out_f,in_f,sp,zipf,b", [
    (3000, 2000, 90, None, 4),     # several chunks, rows cut by chunk boundaries
    (768, 3072, 90, 1.2, 3),       # skewed rows, a batch that is not a power of two
    (10_000, 10_000, 99, None, 1),
    (3000, 700, 95, None, 130),    # three batch tiles (64 + 64 + 2 rows) on one scratch
])
def test_noalloc_forward_matches_oracle_twice(torch, out_f, in_f, sp, zipf, b):
    std = 0.05 if zipf is None else (1.0 / (in_f * (100 - sp) / 100)) ** 0.5
    lay = synth.make_layer(out_f, in_f, sp, std, 51, 52, zipf_s=zipf)
    can, csr = _csr(torch, lay)
    for call in range(2):
        _call_and_check(torch, lay, can, csr, b, 53 + 2 * call, f"call {call}")


def test_noalloc_dense_row_after_larger_layer(torch):
    """A dense row cut across many blocks goes through the scratch's partial
    sums and counters.  A first call with more output rows (and its dense row
    further down) leaves its state in the scratch; the smaller layer's two
    calls that follow, at batch 4 and across batch tiles at batch 70, must
    still match the oracle."""
    big = _dense_row_layer(20_000, 9000, 15_000, 61)
    can_b, csr_b = _csr(torch, big)
    _call_and_check(torch, big, can_b, csr_b, 4, 62, "larger layer")
    small = _dense_row_layer(4000, 700, 5, 63)
    counts = np.bincount(small.rows, minlength=small.out_f)
    # the dense row is longer than ten blocks' shares of the entries
    assert counts[5] > 10 * small.nnz / 152
    can_s, csr_s = _csr(torch, small)
    for call, b in enumerate((4, 4, 70)):
        _call_and_check(torch, small, can_s, csr_s, b, 64 + 2 * call, f"small layer call {call}")


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


def test_noalloc_refuses_operand_plus_slots_over_shared_memory(torch):
    """At batch 64 an operand that alone fits one block's shared memory but
    not together with the kernel's partial-sum slots is refused before any
    work is queued (Y keeps its contents)."""
    max_smem = torch.cuda.get_device_properties(0).shared_memory_per_block_optin
    in_f = max_smem // (64 * 4)           # operand alone fits
    assert in_f * 64 * 4 <= max_smem
    row_ptr = torch.zeros(5, dtype=torch.int32, device="cuda")
    X = torch.zeros(64, in_f, device="cuda")
    Y = torch.full((64, 4), 7.0, device="cuda")
    with pytest.raises(binding.SnkError) as e:
        binding.snk_forward_csr_noalloc(4, in_f, row_ptr, None, torch.zeros(0, device="cuda"), X,
                                        None, Y)
    assert e.value.status == binding.SNK_ERR_LIMIT
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())
