"""The seeded input generators: sizes and structure of the pages' workloads."""
import numpy as np
import pytest

from sparse_linear_layer_gb300 import synth


@pytest.mark.parametrize("out_f,in_f,s,nnz", [
    (500, 500, 95, 12_500),
    (5000, 5000, 80, 5_000_000), (5000, 5000, 90, 2_500_000),
    (5000, 5000, 95, 1_250_000), (5000, 5000, 99, 250_000),
    (10000, 10000, 90, 10_000_000), (10000, 10000, 95, 5_000_000), (10000, 10000, 99, 1_000_000),
    (3072, 768, 90, 235_930), (3072, 768, 99, 23_593),
])
def test_nnz_for(out_f, in_f, s, nnz):
    assert synth.nnz_for(out_f, in_f, s) == nnz


def test_uniform_support_is_distinct_and_seeded():
    r, c = synth.uniform_support(300, 200, 6000, 1)
    lin = r.astype(np.int64) * 200 + c
    assert len(np.unique(lin)) == 6000
    assert r.min() >= 0 and r.max() < 300 and c.min() >= 0 and c.max() < 200
    r2, c2 = synth.uniform_support(300, 200, 6000, 1)
    np.testing.assert_array_equal(r, r2)
    np.testing.assert_array_equal(c, c2)
    assert np.any(np.diff(lin) < 0)  # returned unsorted


@pytest.mark.parametrize("out_f,in_f,sp", [(3072, 768, 90), (768, 3072, 90), (768, 3072, 99)])
def test_zipf_degrees(out_f, in_f, sp):
    nnz = synth.nnz_for(out_f, in_f, sp)
    deg = synth.zipf_row_degrees(out_f, in_f, nnz, 1.2, 41)
    assert deg.sum() == nnz
    assert deg.max() <= in_f and deg.min() >= 0
    srt = np.sort(deg)[::-1]
    # heavy head: the top row is far above the mean, and some rows are capped
    # or nearly so when the budget allows
    assert srt[0] > 5 * nnz / out_f


def test_zipf_support_matches_degrees():
    r, c = synth.zipf_support(768, 3072, 23_593, 1.2, 41)
    deg = synth.zipf_row_degrees(768, 3072, 23_593, 1.2, 41)
    np.testing.assert_array_equal(np.bincount(r, minlength=768), deg)
    lin = r.astype(np.int64) * 3072 + c
    assert len(np.unique(lin)) == len(lin)
