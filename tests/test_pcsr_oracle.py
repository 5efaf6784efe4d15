"""Pins for the Padded-CSR reference state machine (oracle/pcsr.py), from
"Padded-CSR: A sparse storage format for dynamic sparse training on CPU",
sec. 5.2 (capacity rule and its printed examples) and sec. 5.3 (the encoding
of the 4x6 matrix and the insertion of (2, 2, 6), arrays printed on the page),
plus a plain set model of the live entries under random batches."""
import numpy as np
import pytest

from oracle import pcsr
from sparse_linear_layer_gb300 import synth
from tests.conftest import load_golden


def test_capacity_rule_examples():
    g = load_golden("pcsr_padded_worked_example.json")["capacity_examples"]
    assert [pcsr.capacity(n, 20) for n in g["row_nnz"]] == g["capacity"]


def test_worked_example_encoding_and_insert():
    g = load_golden("pcsr_padded_worked_example.json")
    p = pcsr.PaddedCSR(g["out"], g["in"], g["rows"], g["cols"], g["values"], g["padding_pct"])
    assert p.row_nnz == g["row_nnz"]
    assert p.row_capacity == g["row_capacity"]
    assert p.row_start == g["row_start"]
    assert p.used == g["total_capacity"]
    assert p.slot_values == g["slot_values"]
    assert p.slot_cols == g["slot_cols"]
    r, c, v = g["insert"]
    p.insert([r], [c], [v])
    a = g["after_insert"]
    for key in ("row_nnz", "row_capacity", "row_start", "slot_values", "slot_cols"):
        assert getattr(p, key) == a[key], key
    assert p.version == 2


def test_full_row_moves_to_the_end():
    # row 1 (capacity 1, empty) gets 2 entries: it moves to slots 9..11 with
    # capacity ceil(2 * 1.2) = 3; its old slot 2 stays padding
    g = load_golden("pcsr_padded_worked_example.json")
    p = pcsr.PaddedCSR(4, 6, g["rows"], g["cols"], g["values"], 20)
    p.insert([1, 1], [5, 0], [8.0, 9.0])
    assert p.row_start[1] == 9 and p.row_capacity[1] == 3 and p.row_nnz[1] == 2
    assert p.slot_cols[9:12] == [5, 0, -1] and p.slot_values[9:12] == [8.0, 9.0, 0.0]
    assert p.slot_cols[2] == -1 and p.used == 12


def test_delete_closes_the_row():
    g = load_golden("pcsr_padded_worked_example.json")
    p = pcsr.PaddedCSR(4, 6, g["rows"], g["cols"], g["values"], 20)
    p.delete([2], [0])
    assert p.row_nnz[2] == 1
    assert p.slot_cols[3:6] == [4, -1, -1] and p.slot_values[3:6] == [5.0, 0.0, 0.0]
    with pytest.raises(KeyError):
        p.delete([0, 3], [2, 0])      # (3, 0) is not live: nothing changes
    assert p.row_nnz == [1, 0, 1, 2] and p.slot_cols[0] == 2


def test_random_batches_match_a_set_model():
    out_f, in_f = 37, 23
    lay = synth.make_layer(out_f, in_f, 85, 1.0, 1, 2)
    p = pcsr.PaddedCSR(out_f, in_f, lay.rows, lay.cols, lay.values, 20)
    model = {(int(r), int(c)): float(v) for r, c, v in zip(lay.rows, lay.cols, lay.values)}
    gen = synth.rng(3)
    for step in range(30):
        free = [(r, c) for r in range(out_f) for c in range(in_f) if (r, c) not in model]
        ins = [free[i] for i in gen.choice(len(free), int(gen.integers(0, 40)), replace=False)]
        vals = gen.standard_normal(len(ins)).astype(np.float32).tolist()
        p.insert([a for a, _ in ins], [b for _, b in ins], vals)
        model.update({k: float(np.float32(v)) for k, v in zip(ins, vals)})
        live = sorted(model)
        dels = [live[i] for i in gen.choice(len(live), int(gen.integers(0, 30)), replace=False)]
        p.delete([a for a, _ in dels], [b for _, b in dels])
        for k in dels:
            del model[k]
        if step % 7 == 6:
            p.compact_all()
        rows, cols, vals2 = p.live_triple()
        assert list(zip(rows, cols)) == sorted(model)
        assert vals2 == [model[k] for k in sorted(model)]
        for r in range(out_f):
            s, n, cap = p.row_start[r], p.row_nnz[r], p.row_capacity[r]
            assert n <= cap and all(x != -1 for x in p.slot_cols[s:s + n])
            assert all(x == -1 for x in p.slot_cols[s + n:s + cap])
