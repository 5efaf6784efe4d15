"""Benchmark of the truly sparse linear layer on GB300.

Workload (default): W 10000 x 10000 at 90% unstructured sparsity
(nnz = 10,000,000, support uniform without replacement), fp32, batch 4: the
layer of the SNACK page's Table 3 / Fig. 3 ("Beyond Masked Sparsity: SNACK
Enables Truly Sparse Neural Networks on GPU").  One step = one pass of the hot
path over one batch: forward SpMM (with bias), transposed SpMM (dX) and the
weight gradient on the support (dW, with db).  The restructure
(prune_regrow) runs at its own cadence and is timed separately
(``restructure`` key).

Metric: microseconds per call and achieved HBM GB/s for forward / dX / dW.
``value`` = the contract bytes of the step's three kernels / their summed
device time, over all ranks (GB/s).  The contract bytes per call are the
layer's formula: nnz*12 + b*(in+out)*4 for forward and dX, plus nnz*4 (the
gradient written) for dW.  L2 is flushed (a 512 MB write) before every
kernel, outside the timed interval; each kernel is bracketed by CUDA events
on the stream it is launched on.  ``sweep`` repeats the three calls over
b = 1..64 at 90 / 95 / 99 % sparsity.

The minimal bytes each kernel must move with the index width it reads (i: 2
bytes for the 16-bit copies of the shared-memory operand path, else 4) are
reported beside them (``frac_minimal``):
  forward  nnz*(4+i) (values, cols) + (out+1)*4 (row_ptr) + b*in*4 (X) + b*out*4 (Y) + out*4 (bias)
  dX       nnz*(i+4+4) (rows in column order, perm, values) + (in+1)*4 + b*out*4 + b*in*4
  dW       nnz*(i+4) (cols read, dW written) + (out+1)*4 + b*(in+out)*4 (X, dY) + out*4 (db)

--impl reference runs the CPU oracle (the plain fp64 reference) on the host
cores instead, each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (% of roofline) for fwd/dX/dW at b=1–64"
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--out", type=int, default=10000)
    p.add_argument("--inp", type=int, default=10000)
    p.add_argument("--sparsity", type=float, default=90)
    p.add_argument("--batch", type=int, default=4)
    p.add_argument("--zipf", type=float, default=None, metavar="S",
                   help="power-law (Zipf, exponent S) row degrees instead of a uniform support "
                        "(the GPT-2-shaped MLP layers use S = 1.2)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-restructure", action="store_true")
    p.add_argument("--only", choices=["fwd", "dx", "dw"], default=None,
                   help="time a single operation (profiling runs)")
    p.add_argument("--flush-mb", type=int, default=512,
                   help="L2 flush buffer written before every kernel (0 = no flush)")
    p.add_argument("--sweep", default=None, metavar="FILE",
                   help="instead of the single line, write one JSON object per "
                        "(sparsity, batch) of the 10000x10000 sweep to FILE")
    p.add_argument("--latency", default=None, metavar="FILE",
                   help="instead of the single line, write one JSON object per layer of the "
                        "batch-1 inference-latency set (forward only; cold, warm and "
                        "CUDA-graph replay) to FILE")
    p.add_argument("--large-batch", default=None, metavar="FILE",
                   help="instead of the single line, write one JSON object per (layer, batch) "
                        "of the large-batch set (tensor-core path against 64-row batch "
                        "tiling) to FILE")
    p.add_argument("--no-large-batch", action="store_true",
                   help="leave the large-batch measurement out of the single line")
    p.add_argument("--no-sweep", action="store_true",
                   help="leave the b = 1..64 x 90/95/99 %% sweep out of the single line")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_ms(ms, device=None):
    """Max over ranks of a per-rank elapsed time (timing plumbing only; the
    layer itself exchanges nothing between ranks)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world, bytes_per_step, steps, max_ms):
    """Whole-job GB/s: every rank moved bytes_per_step per step; the job took
    the slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


def index_bytes(n_src, b, max_smem=232448):
    """Bytes per index the kernels stream: 16-bit copies on the shared-memory
    operand path (which implies n_src <= 65536), 32-bit otherwise."""
    bt = min(b, 64)
    bp = 1
    while bp < bt:
        bp <<= 1
    return 2 if (n_src * bp * 4 <= max_smem and n_src <= 65536) else 4


def op_bytes(out_f, in_f, nnz, b, max_smem=232448):
    """Algorithmic bytes per launch (what each kernel must move at least, with
    the index width it actually reads) and the contract formula bytes."""
    ic = index_bytes(in_f, b, max_smem)    # column indices (forward, dW)
    ir = index_bytes(out_f, b, max_smem)   # row indices in column order (dX)
    alg = {
        "fwd": nnz * (4 + ic) + (out_f + 1) * 4 + b * in_f * 4 + b * out_f * 4 + out_f * 4,
        "dx": nnz * (ir + 4 + 4) + (in_f + 1) * 4 + b * out_f * 4 + b * in_f * 4,
        "dw": nnz * (ic + 4) + (out_f + 1) * 4 + b * (in_f + out_f) * 4 + out_f * 4,
    }
    formula = {
        "fwd": nnz * 12 + b * (in_f + out_f) * 4,
        "dx": nnz * 12 + b * (in_f + out_f) * 4,
        "dw": nnz * 16 + b * (in_f + out_f) * 4,
    }
    return alg, formula


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The source files that define each profiled kernel (its own file, the
# device helpers it includes and the shared header with the tuning knobs).
KERNEL_SOURCES = {
    "k_spmm_fwd": ["snk_spmm.cu", "snk_device.cuh", "snk_internal.cuh"],
    "k_spmm_dx": ["snk_spmm.cu", "snk_device.cuh", "snk_internal.cuh"],
    "k_sweep_dx": ["snk_spmm.cu", "snk_sweep.cu", "snk_device.cuh", "snk_internal.cuh"],
    "k_sddmm": ["snk_sddmm.cu", "snk_device.cuh", "snk_internal.cuh"],
    "k_band_dw": ["snk_band.cu", "snk_device.cuh", "snk_internal.cuh"],
    "k_tc_spmm": ["snk_tc.cu", "snk_internal.cuh"],
    "k_tc_sddmm": ["snk_tc.cu", "snk_internal.cuh"],
}


def _code_only(text):
    """Source text without comments and blank space, so that editing a
    comment does not detach committed measurements from a kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest(kernel_tag=None):
    """Digest of the code a kernel is built from (all of csrc when the tag
    is not listed); comments do not count."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_linear_layer_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel_tag) or sorted(n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh")))
    for name in names:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel_tag, workload):
    """DRAM bytes per launch from the committed ncu summary of that kernel on
    that workload (profiles/traffic.json: kernel -> workload -> entry), if it
    was taken on the current sources of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(kernel_tag, {}).get(workload)
    if not e or e.get("source_digest") != kernel_source_digest(kernel_tag):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- reference arm
def oracle_step_sample(lay, X, dY, rows_lo, rows_hi):
    """One bounded oracle step: forward, dX and dW restricted to the entries of
    rows [rows_lo, rows_hi) of the canonical triple."""
    import oracle
    o = oracle
    sel = slice(int(lay["row_ptr"][rows_lo]), int(lay["row_ptr"][rows_hi]))
    v, r, c = lay["values"][sel], lay["rows"][sel], lay["cols"][sel]
    o.forward(lay["out"], lay["in"], v, r, c, X, None)
    o.backward_input(lay["out"], lay["in"], v, r, c, dY)
    o.backward_weight(lay["out"], lay["in"], r, c, X, dY)
    return int(sel.stop - sel.start)


def run_reference(args, workload, rank, world):
    if rank != 0:
        return
    import numpy as np

    import oracle
    from sparse_linear_layer_gb300 import synth
    oracle.build()
    lay0 = synth.make_layer(args.out, args.inp, args.sparsity, 0.01, 21, 22, zipf_s=args.zipf)
    can = oracle.canonicalize(args.out, args.inp, lay0.values, lay0.rows, lay0.cols)
    can["out"], can["in"] = args.out, args.inp
    b = args.batch
    X = synth.normal((b, args.inp), 1.0, 23)
    dY = synth.normal((b, args.out), 1.0, 24)
    rows_per_step = max(1, args.out // 100)
    for i in range(args.warmup):
        lo = (i * rows_per_step) % args.out
        oracle_step_sample(can, X, dY, lo, min(args.out, lo + rows_per_step))
    t0 = time.perf_counter()
    nnz_done = 0
    for i in range(args.steps):
        lo = (i * rows_per_step) % args.out
        nnz_done += oracle_step_sample(can, X, dY, lo, min(args.out, lo + rows_per_step))
    dt = time.perf_counter() - t0
    # bytes of the sampled work: entries scale the triple terms; the dense
    # operands are counted for the rows touched
    _, formula = op_bytes(args.out, args.inp, lay0.nnz, b)
    total_bytes = sum(formula.values()) * (nnz_done / lay0.nnz if lay0.nnz else 0.0)
    value = total_bytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step: forward + dX + dW of the oracle over the entries of "
                                   f"{rows_per_step} consecutive rows of W (about 1% of the layer), "
                                   f"batch {b}; rows advance each step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- our arm
# The library's dispatch rule for the tensor-core path (batches of 256 rows
# and more at density 1% and above, 128 and more at 5% and above) and the
# launches that path makes per call: per-call passes plus the product kernels
# of each batch chunk.
TC_CHUNK = 8192
# (first batch, density divisor) of the tensor path's tiers: from that many
# rows at density 1 / divisor and above
TC_TIERS = ((96, 20), (192, 34), (256, 50), (512, 100))
TC_SMS, TC_N = 152, 192


def tc_path(out_f, in_f, nnz, b):
    mode = os.environ.get("SNK_LARGE_BATCH")
    if nnz == 0 or mode == "off":
        return False
    return mode == "on" or any(b >= tb and nnz * div >= out_f * in_f for tb, div in TC_TIERS)


def dx_kernel(out_f, in_f, b, num_sms=152):
    """The kernel the library runs for dX on the batch-tiled path: the column
    sweep for tiles of up to 4 columns when the rows have 16-bit copies (out
    <= 65536) and its lane tables fit the layer's scratch, else the chunk
    walk."""
    if b <= 4 and out_f <= 65536 and 8 * (in_f + num_sms) <= max(out_f, in_f) * 64:
        return "k_sweep_dx"
    return "k_spmm_dx"


def tc_launches(op, out_f, in_f, b):
    """Kernels per call on the tensor-core path: per batch chunk the column
    passes, the flag decision, the transposes and the product, plus the exact
    recomputation of flagged entries (dW); the segment scale pass, the value
    pass and the candidate list, per chunk the split, the product and the
    exact recomputation of flagged rows, plus that of flagged segments
    (forward, dX)."""
    if op == "dw":
        k_stride = (max(out_f, in_f) + 7) // 8 * 8
        chunk = max(64, (TC_CHUNK * k_stride) // (out_f + in_f) // 64 * 64)
        return 6 * ((b + chunk - 1) // chunk) + 1
    n_seg = in_f if op == "dx" else out_f
    n_win = ((out_f if op == "dx" else in_f) + 63) // 64
    n_nt = (n_seg + TC_N - 1) // TC_N
    n = 4
    for c0 in range(0, b, TC_CHUNK):
        n_mt = (min(TC_CHUNK, b - c0) + 127) // 128
        n += 4 if tc_shares_tiles(n_mt * n_nt, n_win) else 3   # split pass, product, (partial sum), exact rows
    return n


def tc_shares_tiles(tiles, n_win, sms=TC_SMS):
    """Whether the tensor forward / dX shares output tiles between CTAs (and
    so adds the partial-sum kernel): all tiles when they fill at most half a
    wave, the last partial wave's when they fill more than one, whenever at
    least 2 ways fit (at most 8, at most one per window)."""
    def ways(n):
        return min(8, n_win, sms // max(n, 1))
    if 2 * tiles <= sms:
        return ways(tiles) >= 2
    rem = tiles % sms
    return tiles > sms and rem > 0 and ways(rem) >= 2


def launches_per_op(n_src, b, max_smem):
    launches = 0
    for t0 in range(0, b, 64):
        bt = min(64, b - t0)
        bp = 1
        while bp < bt:
            bp <<= 1
        launches += 1 if n_src * bp * 4 <= max_smem else 2
    return launches


def time_cpu_baseline(lay, X, dY, budget_s=12.0, max_steps=25, omp=False):
    """Full oracle steps (forward, dX, dW) of the layer until the budget is
    spent; omp runs the OpenMP build of the same source on every core this
    process may use."""
    import oracle
    oracle.build()
    can = oracle.canonicalize(lay.out_f, lay.in_f, lay.values, lay.rows, lay.cols)
    v, r, c = can["values"], can["rows"], can["cols"]
    steps = 0
    t0 = time.perf_counter()
    while steps < max_steps and (time.perf_counter() - t0) < budget_s:
        oracle.forward(lay.out_f, lay.in_f, v, r, c, X, None, omp=omp)
        oracle.backward_input(lay.out_f, lay.in_f, v, r, c, dY, omp=omp)
        oracle.backward_weight(lay.out_f, lay.in_f, r, c, X, dY, omp=omp)
        steps += 1
    return steps, time.perf_counter() - t0


class L2Flush:
    """Evicts the layer's data from L2 between timed kernels: writes a buffer
    larger than L2, then reads a second one so that the written lines are
    written back before the next kernel starts (no dirty lines are left for
    the timed kernel to evict)."""

    def __init__(self, torch, dev, mb):
        n = mb * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n // 2, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.sink.copy_(self.r.sum())


def time_ops(binding, g, X, dY, bias, Y, dX, dW, db, flush, stream, steps, warmup, only=None):
    """Per-op device times (ms) over `steps` steps, each kernel bracketed by
    CUDA events on its stream, L2 flushed before every kernel (untimed)."""
    import torch
    sh = stream.cuda_stream
    ops = [("fwd", lambda: binding.snk_forward(g.handle, X, bias, Y, sh)),
           ("dx", lambda: binding.snk_backward_input(g.handle, dY, dX, sh)),
           ("dw", lambda: binding.snk_backward_weight(g.handle, X, dY, dW, db, sh))]
    if only:
        ops = [o for o in ops if o[0] == only]
    for _ in range(warmup):
        for _, f in ops:
            if flush is not None:
                flush.zero_()
            f()
    torch.cuda.synchronize()
    ev = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps)] for name, _ in ops}
    for i in range(steps):
        for name, f in ops:
            if flush is not None:
                flush.zero_()
            e0, e1 = ev[name][i]
            e0.record(stream)
            f()
            e1.record(stream)
    torch.cuda.synchronize()
    return {name: [e0.elapsed_time(e1) for e0, e1 in ev[name]] for name, _ in ops}


def gather_reference(torch, g, flush, stream, dx_us, dx_tag):
    """The transposed product reads values[perm] in random order: one 4-byte
    value per stored entry, each from its own 32-byte sector.  That gather
    alone, timed here as torch's index_select over the same permutation (a
    library kernel used only as a yardstick, like the copy kernel behind the
    HBM peak), bounds dX from below; 'frac' is gather time / dX time."""
    perm = g.topology()["perm"].long()
    out = torch.empty_like(g.values)
    ts = []
    for i in range(13):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        torch.index_select(g.values, 0, perm, out=out)
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            ts.append(e0.elapsed_time(e1) * 1e3)
    t = statistics.mean(ts)
    return {"bound": "random value gather (L1 sector lookups)", "kernel": dx_tag,
            "reference": "torch.index_select(values, 0, perm), same 10M-entry permutation, "
                         "L2 flushed, CUDA events",
            "gather_us": t, "dx_us": dx_us, "frac": t / dx_us}


def summarize(per_op_ms, alg, formula, peak):
    """Per op: event-timed µs, and GB/s and fraction of the HBM peak on the
    contract (formula) bytes, with the minimal-bytes figures beside them."""
    out = {}
    for n, v in per_op_ms.items():
        mean_us = sum(v) / len(v) * 1e3
        srt = sorted(v)
        out[n] = {"us_median": statistics.median(v) * 1e3, "us_mean": mean_us,
                  "us_p10": srt[len(v) // 10] * 1e3, "us_p90": srt[(9 * len(v)) // 10] * 1e3,
                  "gbs": formula[n] / (mean_us * 1e-6) / 1e9,
                  "frac": formula[n] / (mean_us * 1e-6) / 1e9 / peak,
                  "minimal_gbs": alg[n] / (mean_us * 1e-6) / 1e9,
                  "frac_minimal": alg[n] / (mean_us * 1e-6) / 1e9 / peak}
    return out


def make_device_layer(torch, binding, synth, dev, out_f, in_f, sparsity, b, zipf_s=None):
    import numpy as np
    lay = synth.make_layer(out_f, in_f, sparsity, 0.01, 21, 22, zipf_s=zipf_s)
    X_h = synth.normal((b, in_f), 1.0, 23)
    dY_h = synth.normal((b, out_f), 1.0, 24)
    bias_h = synth.normal(out_f, 0.1, 25)
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    g = binding.SparseLinear(out_f, in_f, td(lay.values), td(lay.rows), td(lay.cols))
    return lay, g, X_h, dY_h, td(X_h), td(dY_h), td(bias_h)


SWEEP_SPARSITY = (90, 95, 99)
SWEEP_BATCHES = (1, 2, 4, 8, 16, 32, 64)


def sweep_points(torch, binding, synth, dev, out_f, in_f, flush, stream, steps, warmup,
                 layers=None):
    """The metric's range: forward, dX and dW at b = 1..64 on the layer at
    90 / 95 / 99 % sparsity, each call event-timed after an L2 flush.  Per
    point: mean µs and the fraction of the HBM peak on the contract bytes.
    layers maps a sparsity to an existing (synth layer, handle) to reuse."""
    peak, _ = measured_peaks()
    max_smem = torch.cuda.get_device_properties(dev).shared_memory_per_block_optin
    pts = []
    for sp in SWEEP_SPARSITY:
        own = not (layers and sp in layers)
        if own:
            lay, g, _, _, _, _, _ = make_device_layer(torch, binding, synth, dev, out_f, in_f, sp, 1)
        else:
            lay, g = layers[sp]
        bias = torch.zeros(out_f, device=dev)
        for b in SWEEP_BATCHES:
            X = torch.randn(b, in_f, device=dev)
            dY = torch.randn(b, out_f, device=dev)
            Y = torch.empty(b, out_f, device=dev)
            dX = torch.empty(b, in_f, device=dev)
            dW = torch.empty(lay.nnz, device=dev)
            db = torch.empty(out_f, device=dev)
            ms = time_ops(binding, g, X, dY, bias, Y, dX, dW, db, flush, stream, steps, warmup)
            alg, formula = op_bytes(out_f, in_f, lay.nnz, b, max_smem)
            summ = summarize(ms, alg, formula, peak)
            pts.append({"sparsity_pct": sp, "batch": b,
                        "us": {n: round(v["us_mean"], 2) for n, v in summ.items()},
                        "frac": {n: round(v["frac"], 4) for n, v in summ.items()}})
        if own:
            g.close()
    return pts


def run_sweep(args, dev):
    import torch

    from sparse_linear_layer_gb300 import binding, synth
    peak, peak_kind = measured_peaks()
    flush = L2Flush(torch, dev, args.flush_mb) if args.flush_mb else None
    stream = torch.cuda.current_stream(dev)
    with open(args.sweep, "w") as fo:
        for sp in (90, 95, 99):
            lay, g, _, _, _, _, bias = make_device_layer(torch, binding, synth, dev, args.out,
                                                         args.inp, sp, 1)
            for b in (1, 2, 4, 8, 16, 32, 64):
                X = torch.randn(b, args.inp, device=dev)
                dY = torch.randn(b, args.out, device=dev)
                Y = torch.empty(b, args.out, device=dev)
                dX = torch.empty(b, args.inp, device=dev)
                dW = torch.empty(lay.nnz, device=dev)
                db = torch.empty(args.out, device=dev)
                ms = time_ops(binding, g, X, dY, bias, Y, dX, dW, db, flush, stream,
                              args.steps, args.warmup)
                alg, formula = op_bytes(args.out, args.inp, lay.nnz, b,
                                        torch.cuda.get_device_properties(dev).shared_memory_per_block_optin)
                row = {"out": args.out, "in": args.inp, "sparsity_pct": sp, "nnz": lay.nnz,
                       "batch": b, "peak_gbs": peak, "peak_kind": peak_kind,
                       "ops": summarize(ms, alg, formula, peak)}
                fo.write(json.dumps(row) + "\n")
                fo.flush()
            g.close()


# Batch-1 forward layers of the pages' latency tables: the GAMLP-shaped 5000 x 5000
# layer ([SNACK] Table 6, latency in ms) and the 12500 x 10000 layer ([SNACK]
# Table 10, CUDA time in us), with the pages' own numbers (other hardware).
LATENCY_SET = [
    (5000, 5000, 90, {"source": "[SNACK] Table 6", "inference_latency_ms": 0.25}),
    (5000, 5000, 95, {"source": "[SNACK] Table 6", "inference_latency_ms": 0.21}),
    (5000, 5000, 99, {"source": "[SNACK] Table 6", "inference_latency_ms": 0.21}),
    (12500, 10000, 90, {"source": "[SNACK] Table 10", "cuda_us": 163.1}),
    (12500, 10000, 95, {"source": "[SNACK] Table 10", "cuda_us": 83.0}),
    (12500, 10000, 99, None),
    (2500, 10000, 90, None),
    (7500, 10000, 90, None),
]


def run_latency(args, dev):
    """Forward latency at batch 1: one call after an L2 flush (cold,
    event-timed); back-to-back direct calls and back-to-back replays of a CUDA
    graph holding one forward call (warm: the layer stays in L2, as in
    repeated inference; device time per call); one call at a time, issue
    to completion on the host clock, direct and as a graph replay; and one
    cold training step (forward, dX, dW + db), event-timed."""
    import torch

    from sparse_linear_layer_gb300 import binding, synth
    flush = L2Flush(torch, dev, args.flush_mb) if args.flush_mb else None
    stream = torch.cuda.current_stream(dev)
    n = max(args.steps, 20)
    with open(args.latency, "w") as fo:
        for out_f, in_f, sp, pages in LATENCY_SET:
            lay, g, _, _, _, _, bias = make_device_layer(torch, binding, synth, dev, out_f, in_f,
                                                         sp, 1)
            X = torch.randn(1, in_f, device=dev)
            Y = torch.empty(1, out_f, device=dev)
            fwd = lambda: binding.snk_forward(g.handle, X, bias, Y, stream.cuda_stream)
            for _ in range(args.warmup):
                fwd()
            torch.cuda.synchronize()
            # cold
            cold = []
            for _ in range(n):
                if flush is not None:
                    flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fwd()
                e1.record(stream)
                e1.synchronize()
                cold.append(e0.elapsed_time(e1) * 1e3)
            # warm, direct calls back to back
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(n):
                fwd()
            e1.record(stream)
            e1.synchronize()
            warm = e0.elapsed_time(e1) * 1e3 / n
            # warm, graph replays
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                binding.snk_forward(g.handle, X, bias, Y, side.cuda_stream)
            stream.wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                binding.snk_forward(g.handle, X, bias, Y)
            torch.cuda.synchronize()
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(torch.cuda.current_stream(dev))
            for _ in range(n):
                graph.replay()
            e1.record(torch.cuda.current_stream(dev))
            e1.synchronize()
            replay = e0.elapsed_time(e1) * 1e3 / n
            # one training step (forward, dX, dW + db) after an L2 flush, for
            # the pages whose time may cover more than the forward
            dY = torch.randn(1, out_f, device=dev)
            dX = torch.empty(1, in_f, device=dev)
            dW = torch.empty(lay.nnz, device=dev)
            db = torch.empty(out_f, device=dev)
            step_cold = []
            for _ in range(n):
                if flush is not None:
                    flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fwd()
                binding.snk_backward_input(g.handle, dY, dX, stream.cuda_stream)
                binding.snk_backward_weight(g.handle, X, dY, dW, db, stream.cuda_stream)
                e1.record(stream)
                e1.synchronize()
                step_cold.append(e0.elapsed_time(e1) * 1e3)
            # one call at a time, host wall clock from issue to completion
            sync = {}
            for name, call in (("direct", fwd), ("graph", graph.replay)):
                ts = []
                for _ in range(n):
                    t0 = time.perf_counter()
                    call()
                    torch.cuda.current_stream(dev).synchronize()
                    ts.append((time.perf_counter() - t0) * 1e6)
                sync[name] = statistics.median(ts)
            row = {"out": out_f, "in": in_f, "sparsity_pct": sp, "nnz": lay.nnz, "batch": 1,
                   "op": "forward", "calls": n,
                   "us_cold_mean": statistics.mean(cold), "us_cold_median": statistics.median(cold),
                   "us_warm_direct": warm, "us_warm_graph_replay": replay,
                   "us_wall_sync_direct_median": sync["direct"],
                   "us_wall_sync_graph_median": sync["graph"],
                   "us_step_fwd_dx_dw_cold_mean": statistics.mean(step_cold),
                   "pages": pages}
            fo.write(json.dumps(row) + "\n")
            fo.flush()
            del graph
            g.close()


# Large-batch set: the GAMLP-scale batches of [SNACK] appendix Table 13
# (batch 4096) on the benchmark's 10000 x 10000 layers and the 5000 x 5000
# GAMLP-shaped one, batches 256 .. 4096.
LARGE_BATCH_SET = [(10000, 10000, 90), (10000, 10000, 99), (5000, 5000, 90)]
LARGE_BATCHES = [256, 1024, 4096]


def measure_large_batch(torch, binding, g, lay, b, dev, flush, reps, tiled_reps):
    """Device µs of forward, dX and dW at batch b on the tensor-core path
    (SNK_LARGE_BATCH=on, so that a batch below the layer's tier is measured
    on that path too) and on 64-row batch tiling (SNK_LARGE_BATCH=off), L2
    flushed before every call.  The tensor roofline counts what the path
    executes: three fp16 products (hi*hi, hi*lo, lo*hi) of the densified
    tiles, 6 * b * out * in flops per call, against the measured bf16 dense
    peak (kind::f16 runs at the bf16 rate)."""
    out_f, in_f = lay.out_f, lay.in_f
    X = torch.randn(b, in_f, device=dev)
    dY = torch.randn(b, out_f, device=dev)
    Y = torch.empty(b, out_f, device=dev)
    dX = torch.empty(b, in_f, device=dev)
    dW = torch.empty(lay.nnz, device=dev)
    db = torch.empty(out_f, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    ops = {"fwd": lambda: binding.snk_forward(g.handle, X, None, Y, sh),
           "dx": lambda: binding.snk_backward_input(g.handle, dY, dX, sh),
           "dw": lambda: binding.snk_backward_weight(g.handle, X, dY, dW, db, sh)}

    def timed(f, n):
        f()   # builds the tile-ordered views on first use
        ts = []
        for _ in range(n):
            if flush is not None:
                flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.mean(ts)

    saved = os.environ.pop("SNK_LARGE_BATCH", None)
    try:
        os.environ["SNK_LARGE_BATCH"] = "on"
        tc = {n: timed(f, reps) for n, f in ops.items()}
        tiled = {}
        if tiled_reps:
            os.environ["SNK_LARGE_BATCH"] = "off"
            tiled = {n: timed(f, tiled_reps) for n, f in ops.items()}
    finally:
        os.environ.pop("SNK_LARGE_BATCH", None)
        if saved is not None:
            os.environ["SNK_LARGE_BATCH"] = saved
    peak = measured_peak_tflops()
    dense = 6.0 * b * out_f * in_f
    useful = 2.0 * b * lay.nnz
    res = {"out": out_f, "in": in_f, "nnz": lay.nnz, "batch": b, "us_tensor_path": tc,
           "us_batch_tiled": tiled or None,
           "speedup_vs_batch_tiled": {n: tiled[n] / tc[n] for n in tiled} if tiled else None,
           "dense_equiv_tflops": {n: dense / tc[n] / 1e6 for n in tc},
           "useful_tflops": {n: useful / tc[n] / 1e6 for n in tc}}
    dom = max(tc, key=lambda n: tc[n])
    res["roofline"] = {"bound": "tensor", "op": dom,
                       "kernel": "k_tc_sddmm" if dom == "dw" else "k_tc_spmm",
                       "achieved": dense / tc[dom] / 1e6, "peak": peak[0], "unit": "TFLOP/s",
                       "frac": dense / tc[dom] / 1e6 / peak[0], "peak_kind": peak[1],
                       "flops_per_launch": dense,
                       "note": "whole call (per-call passes included) / mean event time"}
    del X, dY, Y, dX, dW, db
    return res


def measured_peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "bf16_tflops, of measured (MEASURED_PEAKS.json, burst)"
    except Exception:
        return 1900.0, "bf16 dense, of fallback"


def run_large_batch(args, dev):
    import torch

    from sparse_linear_layer_gb300 import binding, synth
    flush = L2Flush(torch, dev, args.flush_mb) if args.flush_mb else None
    with open(args.large_batch, "w") as fo:
        for out_f, in_f, sp in LARGE_BATCH_SET:
            lay, g, _, _, _, _, _ = make_device_layer(torch, binding, synth, dev, out_f, in_f, sp, 1)
            for b in LARGE_BATCHES:
                row = measure_large_batch(torch, binding, g, lay, b, dev, flush, reps=5,
                                          tiled_reps=1 if b >= 1024 else 3)
                row["sparsity_pct"] = sp
                fo.write(json.dumps(row) + "\n")
                fo.flush()
            g.close()


def run_ours(args, workload, rank, world, local):
    import numpy as np
    import torch

    from sparse_linear_layer_gb300 import binding, build, synth
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.sweep:
        run_sweep(args, dev)
        return
    if args.latency:
        run_latency(args, dev)
        return
    if args.large_batch:
        run_large_batch(args, dev)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    out_f, in_f, b = args.out, args.inp, args.batch
    lay, g, X_h, dY_h, X, dY, bias = make_device_layer(torch, binding, synth, dev, out_f, in_f,
                                                       args.sparsity, b, args.zipf)
    nnz = lay.nnz
    Y = torch.empty((b, out_f), device=dev)
    dX = torch.empty((b, in_f), device=dev)
    dW = torch.empty(nnz, device=dev)
    db = torch.empty(out_f, device=dev)
    flush = L2Flush(torch, dev, args.flush_mb) if args.flush_mb else None
    stream = torch.cuda.current_stream(dev)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    try:
        smi_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        smi_id = str(local)
    with ClockSampler(smi_id) as clk:
        wall0 = time.perf_counter()
        per_op_ms = time_ops(binding, g, X, dY, bias, Y, dX, dW, db, flush, stream, args.steps,
                             args.warmup, args.only)
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    total_ms = reduce_max_ms(sum(sum(v) for v in per_op_ms.values()), dev)
    max_smem = torch.cuda.get_device_properties(dev).shared_memory_per_block_optin
    alg, formula = op_bytes(out_f, in_f, nnz, b, max_smem)
    step_bytes = sum(formula[n] for n in per_op_ms)
    value = aggregate_gbs(world, step_bytes, args.steps, total_ms)
    peak, peak_kind = measured_peaks()
    per_op = summarize(per_op_ms, alg, formula, peak)
    # mean, not median: the event timer ticks in steps of about 2 us on this GPU
    us = {n: v["us_mean"] for n, v in per_op.items()}
    dom = max(per_op, key=lambda n: per_op[n]["us_mean"])
    if tc_path(out_f, in_f, nnz, b):
        # large batch: the tensor-core path, bound by the tensor pipe
        tpeak, tkind = measured_peak_tflops()
        flops = 6.0 * b * out_f * in_f
        ach = flops / (per_op[dom]["us_mean"] * 1e-6) / 1e12
        roofline = {
            "bound": "tensor", "kernel": "k_tc_sddmm" if dom == "dw" else "k_tc_spmm", "op": dom,
            "achieved": ach, "peak": tpeak, "peak_kind": tkind, "unit": "TFLOP/s", "frac": ach / tpeak,
            "traffic": committed_traffic("k_tc_sddmm" if dom == "dw" else "k_tc_spmm", workload["workload"]),
            "flops_per_launch": flops, "per_op": per_op,
            "note": "6*b*out*in fp16 flops: three products of the densified tiles",
        }
    else:
        kernel_tags = {"fwd": "k_spmm_fwd", "dx": dx_kernel(out_f, in_f, b), "dw": "k_sddmm"}
        roofline = {
            "bound": "hbm", "kernel": kernel_tags[dom], "op": dom, "achieved": per_op[dom]["gbs"],
            "peak": peak, "peak_kind": f"hbm_gbs, {peak_kind}", "unit": "GB/s",
            "frac": per_op[dom]["frac"], "frac_formula": per_op[dom]["frac"],
            "frac_minimal": per_op[dom]["frac_minimal"],
            "traffic": committed_traffic(kernel_tags[dom], workload["workload"]),
            "algorithmic_bytes_per_launch": formula[dom], "minimal_bytes_per_launch": alg[dom],
            "bytes_note": "achieved/frac use the contract bytes (nnz*12 + b*(in+out)*4, + nnz*4 "
                          "for dW); frac_minimal uses the bytes the kernel must move with the "
                          "index width it reads",
            "per_op": per_op,
        }
        if not args.only and lay.nnz > 0:
            roofline["onchip"] = gather_reference(torch, g, flush, stream, per_op["dx"]["us_mean"],
                                                  dx_kernel(out_f, in_f, b))

    # ---- end to end through the C ABI with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e and args.only is None:
        sh = stream.cuda_stream
        Xp = torch.from_numpy(X_h).pin_memory()
        dYp = torch.from_numpy(dY_h).pin_memory()
        Yp = torch.empty((b, out_f)).pin_memory()
        dXp = torch.empty((b, in_f)).pin_memory()
        n_e2e = max(10, args.steps // 2)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_e2e)]
        # copies run on their own stream so that they overlap the kernels that
        # do not need them: dY arrives during the forward, Y leaves during dX
        # and dW, dX leaves during dW; the step ends when both streams are done
        cs = torch.cuda.Stream(dev)
        ev = {k: torch.cuda.Event() for k in ("t0", "x", "dy", "y", "dx")}
        for i in range(n_e2e + 3):
            if flush is not None:
                flush.zero_()
            t0 = evs[i - 3][0] if i >= 3 else ev["t0"]
            t0.record(stream)
            cs.wait_event(t0)
            with torch.cuda.stream(cs):
                X.copy_(Xp, non_blocking=True)
                ev["x"].record(cs)
                dY.copy_(dYp, non_blocking=True)
                ev["dy"].record(cs)
            stream.wait_event(ev["x"])
            binding.snk_forward(g.handle, X, bias, Y, sh)
            ev["y"].record(stream)
            stream.wait_event(ev["dy"])
            binding.snk_backward_input(g.handle, dY, dX, sh)
            ev["dx"].record(stream)
            binding.snk_backward_weight(g.handle, X, dY, dW, db, sh)
            cs.wait_event(ev["y"])
            with torch.cuda.stream(cs):
                Yp.copy_(Y, non_blocking=True)
                cs.wait_event(ev["dx"])
                dXp.copy_(dX, non_blocking=True)
            stream.wait_stream(cs)
            if i >= 3:
                evs[i - 3][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max_ms(sum(a0.elapsed_time(z) for a0, z in evs), dev)
        e2e = {"value": aggregate_gbs(world, step_bytes, n_e2e, e2e_ms), "unit": "GB/s",
               "h2d_bytes_per_step": (X_h.nbytes + dY_h.nbytes),
               "d2h_bytes_per_step": b * (out_f + in_f) * 4,
               "ms_per_step": e2e_ms / n_e2e,
               "note": "pinned host X, dY copied in; Y, dX copied out, on a copy stream that "
                       "overlaps the kernels not waiting for them; dW stays on the device for "
                       "the optimizer; L2 flushed before each step only"}

    # ---- the metric's range: b = 1..64 at 90 / 95 / 99 % (the step's layer is reused)
    sweep = None
    if rank == 0 and world == 1 and args.only is None and (out_f, in_f) == (10000, 10000) \
            and b <= 64 and not args.no_sweep:
        reuse = {int(args.sparsity): (lay, g)} if float(args.sparsity).is_integer() else None
        sweep = {"layer": f"{out_f}x{in_f}", "steps": 20, "warmup": 3,
                 "unit": "us per call (mean) and fraction of the HBM peak on the contract bytes",
                 "points": sweep_points(torch, binding, synth, dev, out_f, in_f, flush, stream, 20, 3,
                                        reuse)}

    # ---- restructure (SET cadence work), timed separately
    restructure = None
    if rank == 0 and not args.no_restructure:
        torch.cuda.synchronize()
        ts = []
        for i in range(3):
            t0 = time.perf_counter()
            g.prune_regrow(0.3, 0x5E7 + i)
            torch.cuda.synchronize()
            ts.append((time.perf_counter() - t0) * 1e6)
        tg = []
        for i in range(3):
            t0 = time.perf_counter()
            g.prune_regrow_gradient(0.3, X, dY)
            torch.cuda.synchronize()
            tg.append((time.perf_counter() - t0) * 1e6)
        restructure = {"op": "prune_regrow", "zeta": 0.3,
                       "us_median_host_timed": statistics.median(ts),
                       "gradient_grow_us_median_host_timed": statistics.median(tg),
                       "note": "synchronous calls (they read device counts back); wall-clock µs; "
                               "the gradient variant ranks all out*in - kept candidates by the "
                               "batch's |dY^T X|"}

    large = None
    if rank == 0 and world == 1 and not args.no_large_batch and args.only is None and nnz > 0:
        large = measure_large_batch(torch, binding, g, lay, 4096, dev, flush, reps=5, tiled_reps=1)
        large["workload"] = f"{out_f}x{in_f}, {args.sparsity:g}% sparse, batch 4096 ([SNACK] Table 13 batch)"

    if tc_path(out_f, in_f, nnz, b):
        per_op_launch = {n: tc_launches(n, out_f, in_f, b) for n in ("fwd", "dx", "dw")}
    else:
        per_op_launch = {"fwd": launches_per_op(in_f, b, max_smem),
                         "dx": launches_per_op(out_f, b, max_smem),
                         "dw": launches_per_op(in_f, b, max_smem)}
    launches = args.steps * sum(per_op_launch[n] for n in per_op_ms)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        steps_c, dt_c = time_cpu_baseline(lay, X_h, dY_h)
        cpu = {"value": sum(formula.values()) * steps_c / dt_c / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{steps_c} full steps (forward + dX + dW, fp64 accumulation) of the same "
                         f"{out_f}x{in_f} layer, batch {b}, single-threaded"}
        import oracle
        if oracle.openmp_available():
            cores = len(os.sched_getaffinity(0))
            os.environ["OMP_NUM_THREADS"] = str(cores)
            os.environ.setdefault("OMP_PROC_BIND", "false")
            steps_o, dt_o = time_cpu_baseline(lay, X_h, dY_h, budget_s=8.0, omp=True)
            cpu["openmp"] = {
                "value": sum(formula.values()) * steps_o / dt_o / 1e9, "unit": "GB/s",
                "cores": oracle.threads(omp=True), "affinity_cores": cores, "kind": "oracle",
                "sample": f"{steps_o} full steps of the same layer and batch, the oracle's "
                          f"source built with OpenMP: outputs split statically over the cores "
                          f"(rows for the forward, columns for dX, entries for dW), the same "
                          f"bits as the single-threaded build"}
        else:
            cpu["openmp"] = None

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": workload,
            "us_per_call": us, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clk.summary(), "restructure": restructure,
            "large_batch": large, "sweep": sweep,
            "library": {"path": os.path.relpath(binding.LIB_PATH, ROOT),
                        "source_digest": kernel_source_digest()},
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    g.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    nnz = None
    try:
        from sparse_linear_layer_gb300 import synth
        nnz = synth.nnz_for(args.out, args.inp, args.sparsity)
    except Exception:
        pass
    zipf = "" if args.zipf is None else f"_zipf{args.zipf:g}"
    support = ("uniform random sparsity" if args.zipf is None
               else f"sparsity with Zipf (s = {args.zipf:g}) row degrees")
    workload = {
        "workload": f"layer{args.out}x{args.inp}_s{args.sparsity:g}{zipf}_b{args.batch}",
        "description": f"W {args.out}x{args.inp}, {args.sparsity:g}% {support}, fp32, "
                       f"batch {args.batch}; step = forward (bias) + backward_input + "
                       f"backward_weight (db)",
        "out": args.out, "in": args.inp, "sparsity_pct": args.sparsity, "nnz": nnz,
        "batch": args.batch,
        "l2": (f"flushed before every kernel, untimed: a {args.flush_mb} MB write, then a "
               f"{args.flush_mb // 2} MB read so no dirty lines remain"
               if args.flush_mb else "not flushed"),
        "parallelism": f"replicas x{world}",
    }
    if args.impl == "reference":
        run_reference(args, workload, rank, world)
    else:
        run_ours(args, workload, rank, world, local)


if __name__ == "__main__":
    main()
