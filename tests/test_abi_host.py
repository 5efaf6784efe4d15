"""The C-ABI library builds, loads, exports every declared entry point, and
rejects bad arguments on the host before touching the GPU.  No compute calls
run here; on a machine without a GPU the product path must fail loudly."""
import ctypes

import pytest

from sparse_linear_layer_gb300 import binding, build

ARG = binding.SNK_ERR_ARG


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def test_every_declared_symbol_is_exported(L):
    names = binding.declared_symbols()
    assert {"snk_create", "snk_forward", "snk_backward_input", "snk_backward_weight",
            "snk_prune_regrow", "snk_destroy", "snk_status_string", "snk_get_shape",
            "snk_copy_topology", "snk_check", "snk_forward_csr_noalloc"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for st in range(8):
        assert len(binding.snk_status_string(st)) >= 2
    assert binding.snk_status_string(99) == "unknown status"


def test_create_rejects_bad_arguments_on_host(L):
    h = ctypes.c_void_p()
    P = ctypes.byref(h)
    good = 0x1000
    assert L.snk_create(None, 4, 4, 1, good, good, good, None) == ARG
    assert L.snk_create(P, 0, 4, 1, good, good, good, None) == ARG
    assert L.snk_create(P, 4, -1, 1, good, good, good, None) == ARG
    assert L.snk_create(P, 2**31, 4, 1, good, good, good, None) == ARG
    assert L.snk_create(P, 4, 4, 17, good, good, good, None) == ARG      # nnz > out*in
    assert L.snk_create(P, 4, 4, -1, good, good, good, None) == ARG
    assert L.snk_create(P, 4, 4, 2, None, good, good, None) == ARG       # null with nnz > 0
    assert L.snk_create(P, 4, 4, 2, good + 4, good, good, None) == ARG   # misaligned values
    assert L.snk_create(P, 4, 4, 2, good, good + 8, good, None) == ARG   # misaligned rows
    assert h.value is None


def test_calls_on_null_handle_are_rejected(L):
    assert L.snk_forward(None, 0x1000, 1, None, 0x1000, None) == ARG
    assert L.snk_backward_input(None, 0x1000, 1, 0x1000, None) == ARG
    assert L.snk_backward_weight(None, 0x1000, 0x1000, 1, 0x1000, None, None) == ARG
    assert L.snk_prune_regrow(None, ctypes.c_float(0.3), 1, None) == ARG
    assert L.snk_get_shape(None, None, None, None, None) == ARG
    assert L.snk_copy_topology(None, None, None, None, None, None) == ARG
    assert L.snk_destroy(None) == binding.SNK_OK


def test_no_gpu_means_a_loud_cuda_error(L):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = L.snk_create(ctypes.byref(h), 4, 4, 0, None, None, None, None)
    assert st == binding.SNK_ERR_CUDA
    assert h.value is None
