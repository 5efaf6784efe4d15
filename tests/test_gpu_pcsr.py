"""GPU Padded-CSR view against the reference state machine (oracle/pcsr.py):
every array of the view must be identical after each batch.

Page: "Padded-CSR: A sparse storage format for dynamic sparse training on
CPU", sec. 5.1-5.3 (format, capacity rule, worked example), sec. 4.3 (row
resize), sec. 8.3 (compact_all)."""
import numpy as np
import pytest

import oracle
from oracle import pcsr
from sparse_linear_layer_gb300 import binding, synth
from tests.conftest import load_golden
from tests.gpu_util import assert_within, dev, host, make_gpu_layer, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def assert_same_view(g, ref):
    v = g.pcsr()
    assert v["version"] == ref.version
    assert v["n_live"] == sum(ref.row_nnz)
    np.testing.assert_array_equal(host(v["row_start"]), ref.row_start)
    np.testing.assert_array_equal(host(v["row_nnz"]), ref.row_nnz)
    np.testing.assert_array_equal(host(v["row_capacity"]), ref.row_capacity)
    np.testing.assert_array_equal(host(v["slot_cols"]), ref.slot_cols)
    np.testing.assert_array_equal(host(v["slot_values"]).view(np.uint32),
                                  np.asarray(ref.slot_values, np.float32).view(np.uint32))


def test_worked_example(torch):
    gd = load_golden("pcsr_padded_worked_example.json")
    lay = synth.Layer(4, 6, np.array(gd["values"], np.float32), np.array(gd["rows"], np.int32),
                      np.array(gd["cols"], np.int32))
    g = make_gpu_layer(torch, lay)
    binding.snk_pcsr_build(g.handle, gd["padding_pct"])
    v = g.pcsr()
    np.testing.assert_array_equal(host(v["slot_cols"]), gd["slot_cols"])
    np.testing.assert_array_equal(host(v["slot_values"]), gd["slot_values"])
    np.testing.assert_array_equal(host(v["row_start"]), gd["row_start"])
    np.testing.assert_array_equal(host(v["row_capacity"]), gd["row_capacity"])
    r, c, val = gd["insert"]
    binding.snk_pcsr_insert(g.handle, dev(np.array([r], np.int32), torch),
                            dev(np.array([c], np.int32), torch),
                            dev(np.array([val], np.float32), torch))
    v = g.pcsr()
    a = gd["after_insert"]
    np.testing.assert_array_equal(host(v["slot_cols"]), a["slot_cols"])
    np.testing.assert_array_equal(host(v["slot_values"]), a["slot_values"])
    np.testing.assert_array_equal(host(v["row_nnz"]), a["row_nnz"])
    assert v["version"] == 2
    g.close()


def _batches(torch, g, ref, gen, steps, max_ins, max_del, compact_every):
    out_f, in_f = ref.out_f, ref.in_f
    for step in range(steps):
        rows, cols, _ = ref.live_triple()
        live = set(zip(rows, cols))
        n_ins = int(gen.integers(1, max_ins))
        cand = gen.integers(0, out_f * in_f, 4 * n_ins)
        ins, seen = [], set()
        for p in cand.tolist():
            key = divmod(p, in_f)
            if key not in live and key not in seen:
                seen.add(key)
                ins.append(key)
            if len(ins) == n_ins:
                break
        # skew: a quarter of the inserts go to three rows, so rows overflow
        for j in range(len(ins) // 4):
            rr = int(gen.choice([0, out_f // 2, out_f - 1]))
            cc = int(gen.integers(0, in_f))
            if (rr, cc) not in live and (rr, cc) not in seen:
                seen.add((rr, cc))
                ins[j] = (rr, cc)
        ins = list(dict.fromkeys(ins))
        vals = gen.standard_normal(len(ins)).astype(np.float32)
        ir = np.array([a for a, _ in ins], np.int32)
        ic = np.array([b for _, b in ins], np.int32)
        binding.snk_pcsr_insert(g.handle, dev(ir, torch), dev(ic, torch), dev(vals, torch))
        ref.insert(ir, ic, vals.tolist())
        assert_same_view(g, ref)
        rows, cols, _ = ref.live_triple()
        live = list(zip(rows, cols))
        k = min(len(live), int(gen.integers(0, max_del)))
        dels = [live[i] for i in gen.choice(len(live), k, replace=False)]
        if dels:
            dr = np.array([a for a, _ in dels], np.int32)
            dc = np.array([b for _, b in dels], np.int32)
            binding.snk_pcsr_delete(g.handle, dev(dr, torch), dev(dc, torch))
            ref.delete(dr, dc)
            assert_same_view(g, ref)
        if compact_every and step % compact_every == compact_every - 1:
            binding.snk_pcsr_compact(g.handle)
            ref.compact_all()
            assert_same_view(g, ref)


@pytest.mark.parametrize("out_f,in_f,sp,pct,zipf", [
    (60, 45, 90, 20, None),
    (300, 200, 95, 20, None),
    (257, 311, 80, 0, None),       # no padding: every insert moves its row
    (768, 3072, 99, 20, 1.2),      # GPT-2 MLP shape, Zipf rows
])
def test_random_batches_match_reference(torch, out_f, in_f, sp, pct, zipf):
    lay = synth.make_layer(out_f, in_f, sp, 1.0, 21, 22, zipf_s=zipf)
    g = make_gpu_layer(torch, lay)
    binding.snk_pcsr_build(g.handle, pct)
    ref = pcsr.PaddedCSR(out_f, in_f, lay.rows, lay.cols, lay.values, pct)
    assert_same_view(g, ref)
    _batches(torch, g, ref, synth.rng(23), 8, 400, 300, 3)
    g.close()


def test_export_feeds_a_new_layer(torch):
    """Adaptive density: the view's live entries, after inserts and deletes,
    become a new layer whose products match the oracle on the same triple."""
    out_f, in_f = 500, 400
    lay = synth.make_layer(out_f, in_f, 90, 0.05, 31, 32)
    g = make_gpu_layer(torch, lay)
    binding.snk_pcsr_build(g.handle, 20)
    ref = pcsr.PaddedCSR(out_f, in_f, lay.rows, lay.cols, lay.values, 20)
    _batches(torch, g, ref, synth.rng(33), 4, 3000, 1000, 0)
    rows, cols, vals = ref.live_triple()
    n = len(rows)
    v2 = torch.empty(n + 10, device="cuda")
    r2 = torch.empty(n + 10, dtype=torch.int32, device="cuda")
    c2 = torch.empty(n + 10, dtype=torch.int32, device="cuda")
    got = binding.snk_pcsr_export(g.handle, v2, r2, c2)
    assert got == n
    np.testing.assert_array_equal(host(r2[:n]), rows)
    np.testing.assert_array_equal(host(c2[:n]), cols)
    np.testing.assert_array_equal(host(v2[:n]), np.asarray(vals, np.float32))
    g2 = binding.SparseLinear(out_f, in_f, v2[:n].clone(), r2[:n].clone(), c2[:n].clone())
    X = synth.normal((3, in_f), 1.0, 34)
    Y = g2.forward(dev(X, torch))
    Yr, Ay = oracle.forward(out_f, in_f, np.asarray(vals, np.float32), np.asarray(rows, np.int32),
                            np.asarray(cols, np.int32), X, None)
    assert_within(host(Y), Yr, Ay, "forward of the exported layer")
    small = torch.empty(1, device="cuda")
    with pytest.raises(binding.SnkError) as e:
        binding.snk_pcsr_export(g.handle, small, small.int(), small.int())
    assert e.value.status == binding.SNK_ERR_LIMIT
    g2.close()
    g.close()


def test_errors_leave_the_view_unchanged(torch):
    out_f, in_f = 40, 30
    lay = synth.make_layer(out_f, in_f, 80, 1.0, 41, 42)
    g = make_gpu_layer(torch, lay)
    binding.snk_pcsr_build(g.handle, 20)
    ref = pcsr.PaddedCSR(out_f, in_f, lay.rows, lay.cols, lay.values, 20)
    i32 = lambda a: dev(np.array(a, np.int32), torch)
    with pytest.raises(binding.SnkError) as e:
        binding.snk_pcsr_insert(g.handle, i32([1, out_f]), i32([0, 0]),
                                dev(np.ones(2, np.float32), torch))
    assert e.value.status == binding.SNK_ERR_RANGE
    rows, cols, _ = ref.live_triple()
    free_c = next(c for c in range(in_f) if (rows[0], c) not in set(zip(rows, cols)))
    with pytest.raises(binding.SnkError) as e:
        binding.snk_pcsr_delete(g.handle, i32([rows[0], rows[0]]), i32([cols[0], free_c]))
    assert e.value.status == binding.SNK_ERR_ARG
    assert_same_view(g, ref)
    # a position inserted twice is caught by compact, which then changes nothing
    binding.snk_pcsr_insert(g.handle, i32([rows[0]]), i32([cols[0]]),
                            dev(np.ones(1, np.float32), torch))
    ref.insert([rows[0]], [cols[0]], [1.0])
    with pytest.raises(binding.SnkError) as e:
        binding.snk_pcsr_compact(g.handle)
    assert e.value.status == binding.SNK_ERR_DUP
    assert_same_view(g, ref)
    g.close()
