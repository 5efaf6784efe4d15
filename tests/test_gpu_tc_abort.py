"""A tensor-core kernel whose bounded wait runs out reports it and leaves no
stale output.

The large-batch kernels bound every wait of their pipeline.  A build with the
limit set to zero cycles (SNK_TC_WAIT_CYCLES=0) makes the first wait that is
not already satisfied give up, so CTAs stop early through the same path
a real stall would take: it waits (with the separate drain limit) for the
copies and MMAs it has issued, writes NaN to the outputs it owns and records
the stop in the status word.  The test runs that build in a child process on
the large-batch path and checks that
  - snk_check reports SNK_ERR_LIMIT once, then SNK_OK;
  - every element of Y, dX and dW is NaN (its CTA stopped) or matches the
    oracle, none keeps the value it held before the call, and some are NaN;
    db, which another kernel computes, matches the oracle;
  - the context still works: a batch-tiled forward afterwards matches the
    oracle.
No GPU fault is involved: every wait is bounded and every issued copy is
waited for before a CTA exits.
"""
import json
import os
import subprocess
import sys

import pytest

from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, ROOT)
import numpy as np
import torch
import oracle
from sparse_linear_layer_gb300 import binding, synth
binding.LIB_PATH = VARIANT
dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
out_f, in_f, b = 300, 200, 130
lay = synth.make_layer(out_f, in_f, 90, 0.05, 141, 142)
g = binding.SparseLinear(out_f, in_f, dev(lay.values), dev(lay.rows), dev(lay.cols))
X_h = synth.normal((b, in_f), 1.0, 143)
dY_h = synth.normal((b, out_f), 1.0, 144)
X, dY = dev(X_h), dev(dY_h)
res = {}
os.environ["SNK_LARGE_BATCH"] = "on"
SENT = 777.0   # what a stale output would still hold
Y = torch.full((b, out_f), SENT, device="cuda")
dX = torch.full((b, in_f), SENT, device="cuda")
dW = torch.full((g.nnz,), SENT, device="cuda")
db = torch.full((out_f,), SENT, device="cuda")
binding.snk_forward(g.handle, X, None, Y)
binding.snk_backward_input(g.handle, dY, dX)
binding.snk_backward_weight(g.handle, X, dY, dW, db)
try:
    binding.snk_check(g.handle)
    res["first_check"] = 0
except binding.SnkError as e:
    res["first_check"] = e.status
try:
    binding.snk_check(g.handle)
    res["second_check"] = 0
except binding.SnkError as e:
    res["second_check"] = e.status
v, r, c = (t.cpu().numpy() for t in (g.values, g.rows, g.cols))
Yr, Ay = oracle.forward(out_f, in_f, v, r, c, X_h, None)
dXr, Ax = oracle.backward_input(out_f, in_f, v, r, c, dY_h)
dWr, Aw, dbr, Ab = oracle.backward_weight(out_f, in_f, r, c, X_h, dY_h)
res["nan_count"] = 0
for name, got, ref, A in (("Y", Y, Yr, Ay), ("dX", dX, dXr, Ax), ("dW", dW, dWr, Aw)):
    a = got.cpu().numpy().astype(np.float64)
    nan = np.isnan(a)
    res["nan_count"] += int(nan.sum())
    # every output is NaN (its CTA stopped) or correct: none keeps the sentinel
    res[name + "_nan_or_correct"] = bool((nan | (np.abs(a - ref) <= 1e-5 * A + 1e-6)).all())
res["db_ok"] = bool((np.abs(db.cpu().numpy().astype(np.float64) - dbr) <= 1e-5 * Ab + 1e-6).all())
os.environ["SNK_LARGE_BATCH"] = "off"
Y4 = g.forward(X[:4])
torch.cuda.synchronize()
Yr, Ay = oracle.forward(out_f, in_f, v, r, c, X_h[:4], None)
res["tiled_ok"] = bool((np.abs(Y4.cpu().numpy().astype(np.float64) - Yr) <= 1e-5 * Ay + 1e-6).all())
g.close()
print("RESULT " + json.dumps(res))
"""


def test_wait_limit_is_reported_and_outputs_are_nan():
    need_gpu()
    from sparse_linear_layer_gb300 import binding, build
    variant = os.path.join(build.PKG, "_build", "waitlimit", "libsnk.so")
    build.build(extra_flags=["-DSNK_TC_WAIT_CYCLES=0"], out=variant)
    code = CHILD.replace("ROOT", repr(ROOT)).replace("VARIANT", repr(variant))
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("RESULT ")]
    assert p.returncode == 0 and lines, p.stdout[-2000:] + p.stderr[-4000:]
    res = json.loads(lines[-1][len("RESULT "):])
    assert res["first_check"] == binding.SNK_ERR_LIMIT, res
    assert res["second_check"] == 0, res
    # at least one CTA stopped; the outputs of a CTA that did are NaN, the
    # rest correct, and nothing keeps the value it held before the call
    assert res["nan_count"] > 0, res
    assert res["Y_nan_or_correct"] and res["dX_nan_or_correct"] and res["dW_nan_or_correct"], res
    assert res["db_ok"], res
    assert res["tiled_ok"], res
