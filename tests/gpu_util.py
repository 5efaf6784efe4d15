"""Helpers for the GPU parity tests: build/load the library, move seeded
inputs to the device, and compare against the oracle within the fp32
tolerance |gpu - oracle| <= 1e-5 * A + 1e-6 (A = sum of |terms| + |bias|)."""
import numpy as np
import pytest

RTOL_A = 1e-5
ATOL = 1e-6


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_linear_layer_gb300 import build
    build.build()
    return torch


def dev(a, torch, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_within(gpu, ref, A, what=""):
    """Element-wise parity: where the oracle's result is finite, the GPU's is
    finite and within 1e-5 * A + 1e-6 of it; where it is NaN or +-inf, the
    GPU's is NaN or the same infinity."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    with np.errstate(invalid="ignore"):
        err = np.abs(gpu - ref)
    bound = RTOL_A * A + ATOL
    ok = np.where(fin, err <= bound,
                  np.where(np.isnan(ref), np.isnan(gpu), gpu == ref))
    bad = ~ok
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)}: "
            f"gpu={gpu[tuple(i)]!r} oracle={ref[tuple(i)]!r} A={A[tuple(i)]!r}")


def make_gpu_layer(torch, lay):
    """Copy a synth.Layer to the device and create the library handle."""
    from sparse_linear_layer_gb300 import binding
    v = dev(lay.values, torch)
    r = dev(lay.rows, torch)
    c = dev(lay.cols, torch)
    return binding.SparseLinear(lay.out_f, lay.in_f, v, r, c)
