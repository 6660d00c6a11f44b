"""Layout autotuning for librs (ResServe Sec. 5.1 "Layout Autotuning", Fig. 3).

The paper selects a kernel layout per (M, N, K) by measuring the candidates.
This script does that for librs's launch tactics -- K-split count, in-GEMM
quantization of the bf16 input, MMA width and the weight ring depth of split
plans (see rs_set_tactic in include/rs.h) -- on the GPU it runs on, and
writes the winners as the C table that librs compiles in
(csrc/rs_tactics_gb300.inc), keyed by the GPU's SM count.

Each candidate runs through the public entry points (rs_linear_w4a4 /
rs_linear_compensated with a bf16 input), captured `steps` calls at a time in a
CUDA graph whose calls rotate over copies of the quantized weight larger than
twice the L2 cache, and is timed with CUDA events (median of the replays).  A
shape keeps the analytic plan unless a candidate beats it by more than
`--margin`; either way the table records the chosen tactic for every tuned
(shape, M), so that a call of M rows resolves to the entry of its own
tuned row count and not to a larger one.

    python -m block_scaled_quantized_gb300.tune            # full table (a few minutes)
    python -m block_scaled_quantized_gb300.tune --quick    # a handful of shapes, printed only
    python -m block_scaled_quantized_gb300.tune --from-log LOG   # table from an earlier run's --log
    python -m block_scaled_quantized_gb300.tune --min-rows 64    # re-tune the cases of at least 64
                                                                 # activation rows, keep the other rows
"""
from __future__ import annotations

import argparse
import math
import os
import re
import statistics
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(HERE))

import torch  # noqa: E402

from block_scaled_quantized_gb300 import build, rs, workloads  # noqa: E402

NVFP4, MXFP4 = 0, 1
SMALL_MS = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512)


def tuning_set(quick: bool):
    """(fmt, N, K, Ms) of the shapes the library is tuned for: the 22
    projection shapes of the paper's kernel evaluation, the attention
    projection, MLP and gauss-outlier shapes, the MXFP4 sweep shape, and the
    prefill shape."""
    if quick:
        return [(NVFP4, 4096, 4096, (1, 8, 64)), (NVFP4, 8192, 1024, (8,)), (MXFP4, 27648, 5120, (64, 128))]
    shapes = [(NVFP4, N, K, SMALL_MS) for N, K in workloads.PROJECTION_SHAPES]
    shapes += [(NVFP4, 2048, 2048, SMALL_MS), (NVFP4, 28672, 4096, SMALL_MS[:7]), (NVFP4, 4096, 14336, SMALL_MS[:7]),
               (MXFP4, 27648, 5120, SMALL_MS[:8]), (NVFP4, 8192, 8192, (2048, 4096))]
    seen, out = set(), []
    for s in shapes:
        if (s[0], s[1], s[2]) not in seen:
            seen.add((s[0], s[1], s[2]))
            out.append(s)
    return out


def natural_bn(rows: int) -> int:
    for b in (16, 32, 64, 128):
        if rows <= b:
            return b
    return 256


def candidates(M: int, K: int, compensated: bool):
    rows = 2 * M if compensated else M
    b0 = natural_bn(rows)
    bns = [b for b in (b0, 2 * b0, 4 * b0) if b <= 256] if rows <= 64 else [b for b in (b0, 2 * b0) if b <= 256]
    chunks = (K + 255) // 256
    for bn in bns:
        for splits in range(1, min(8, chunks) + 1):
            for fused in ((2, 1, 0) if bn <= 32 else (0,)):
                for deep in ((0, 1) if splits > 1 else (0,)):
                    yield splits, fused, bn, deep


class Shape:
    """Quantized weight copies (rotated so that every call streams from HBM),
    one bf16 input and output per M."""

    def __init__(self, fmt, N, K, seed=11):
        dev = torch.device("cuda")
        self.fmt, self.N, self.K = fmt, N, K
        w = workloads.make_w("proj_shapes", N=N, K=K, seed=seed).to(dev)
        self.aw = torch.empty(1, dtype=torch.float32, device=dev)
        if fmt == NVFP4:
            rs.rs_compute_tensor_scale(w, self.aw)
        wq = torch.empty(rs.rs_weight_bytes(fmt, N, K), dtype=torch.uint8, device=dev)
        rs.rs_quantize_weight(fmt, w, self.aw if fmt == NVFP4 else None, wq)
        del w
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(2, math.ceil(2 * l2 / wq.numel()) + 1)
        self.wqs = [wq] + [wq.clone() for _ in range(n - 1)]

    def inputs(self, M, seed=12):
        dev = torch.device("cuda")
        x = workloads.make_x("proj_shapes", M, K=self.K, seed=seed).to(dev)
        ax = torch.empty(1, dtype=torch.float32, device=dev)
        if self.fmt == NVFP4:
            rs.rs_compute_tensor_scale(x, ax)
        y = torch.empty((M, self.N), dtype=torch.bfloat16, device=dev)
        return x, ax, y


def time_calls(shape: Shape, M: int, compensated: bool, inp, steps: int, reps: int) -> float:
    x, ax, y = inp
    nv = shape.fmt == NVFP4
    ws = rs.empty_workspace(shape.fmt, M, shape.N, shape.K, compensated)
    fn = rs.rs_linear_compensated if compensated else rs.rs_linear_w4a4

    def call(i):
        fn(shape.fmt, M, shape.N, shape.K, x=x, alpha_x=ax if nv else None, wq=shape.wqs[i % len(shape.wqs)],
           alpha_w=shape.aw if nv else None, y=y, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(2):
            call(i)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                call(i)
    torch.cuda.synchronize()
    g.replay()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0 / steps)
    del g
    if rs.rs_get_device_error() != 0:
        raise RuntimeError("device error word set while timing a candidate")
    return statistics.median(times)


def plan_key(fmt, compensated, M, N, K, sms):
    p = rs.rs_plan_linear(fmt, compensated, M, N, K, sms)
    return tuple(v for k, v in p.items() if k != "tuned")


def analytic_tactic(fmt, compensated, M, N, K, sms):
    """(splits, fused, bn, deep) of the analytic plan (host only)."""
    rs.rs_reset_tactics(False)
    p = rs.rs_plan_linear(fmt, compensated, M, N, K, sms)
    return p["splits"], p["fused"], p["bn"], 0


def tune_one(shape: Shape, M: int, compensated: bool, sms: int, margin: float):
    """Tactic for one (shape, M, compensated): ((splits, fused, bn, deep), its us,
    analytic us, plans timed, whether the analytic plan was kept)."""
    fmt, N, K = shape.fmt, shape.N, shape.K
    steps = 32 if M <= 512 else 8
    reps = 5 if M <= 512 else 3
    inp = shape.inputs(M)
    rs.rs_reset_tactics(False)
    base_key = plan_key(fmt, compensated, M, N, K, sms)
    base_us = time_calls(shape, M, compensated, inp, steps, reps)
    seen = {base_key: base_us}
    best, best_us = None, base_us
    for splits, fused, bn, deep in candidates(M, K, compensated):
        rs.rs_reset_tactics(False)
        rs.rs_set_tactic(fmt, compensated, M, N, K, sms, splits, fused, bn, deep)
        p = rs.rs_plan_linear(fmt, compensated, M, N, K, sms)
        if not p["tuned"]:
            continue  # the tactic's plan does not fit
        key = plan_key(fmt, compensated, M, N, K, sms)
        if key in seen:
            continue
        us = time_calls(shape, M, compensated, inp, steps, reps)
        seen[key] = us
        if us < best_us:
            best, best_us = (splits, p["fused"], p["bn"], deep), us
    kept = best is None or best_us > base_us * (1.0 - margin)
    if kept:
        best, best_us = analytic_tactic(fmt, compensated, M, N, K, sms), base_us
    rs.rs_reset_tactics(False)
    return best, best_us, base_us, len(seen), kept


def write_table(path: str, sms: int, rows: list):
    lines = ["// Measured launch tactics for GB300 (%d SMs): {fmt, compensated, M, N, K," % sms,
             "// SMs, splits, fused, bn, deep}, each with the measured us per call of the",
             "// tactic and of the analytic plan.  Written by block_scaled_quantized_gb300/tune.py.",
             "{0, 1, 0, 0, 0, 0, 0, 0, 0, 0},  // placeholder row (M = 0 never matches)"]
    for (fmt, comp, M, N, K, t, us, base, kept) in rows:
        note = "analytic plan" if kept else "analytic plan %.3f us" % base
        lines.append("{%d, %d, %d, %d, %d, %d, %d, %d, %d, %d},  // %.3f us (%s)"
                     % (fmt, comp, M, N, K, sms, t[0], t[1], t[2], t[3], us, note))
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


LOG_LINE = re.compile(r"fmt=(\d) comp=(\d) M=(\d+) N=(\d+) K=(\d+) sms=(\d+): analytic ([\d.]+) us, "
                      r"best ([\d.]+) us \((\d+), (\d), (\d+)(?:, (\d))?\)( analytic)?")


TABLE_LINE = re.compile(r"\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\},  "
                        r"// ([\d.]+) us \(analytic plan(?: ([\d.]+) us)?\)")


def rows_from_table(path):
    """The rows of a table written by write_table (placeholder row excluded)."""
    rows, sms = [], None
    for line in open(path):
        m = TABLE_LINE.match(line)
        if not m or int(m.group(3)) == 0:
            continue
        fmt, comp, M, N, K, sms, sp, fu, bn, deep = (int(v) for v in m.groups()[:10])
        us = float(m.group(11))
        kept = m.group(12) is None
        base = us if kept else float(m.group(12))
        rows.append((fmt, comp, M, N, K, (sp, fu, bn, deep), us, base, kept))
    return sms, rows


def rows_from_log(path):
    rows, sms = [], None
    for line in open(path):
        m = LOG_LINE.match(line)
        if not m:
            continue
        fmt, comp, M, N, K, sms = (int(v) for v in m.groups()[:6])
        base, us = float(m.group(7)), float(m.group(8))
        t = tuple(int(v) for v in m.groups()[8:11]) + (int(m.group(12) or 0),)
        rows.append((fmt, comp, M, N, K, t, us, base, m.group(13) is not None))
    return sms, rows


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--quick", action="store_true", help="a few shapes; print, do not write the table")
    ap.add_argument("--margin", type=float, default=0.01,
                    help="keep the analytic plan unless a tactic is faster by more than this fraction")
    ap.add_argument("--out", default=os.path.join(HERE, "csrc", "rs_tactics_gb300.inc"))
    ap.add_argument("--log", default=None, help="also write one line per tuned case to this file")
    ap.add_argument("--from-log", default=None, help="write the table from an earlier run's --log (no GPU)")
    ap.add_argument("--min-rows", type=int, default=0,
                    help="tune only the cases with at least this many activation rows (2M compensated, M "
                         "plain) and keep the table's other rows")
    a = ap.parse_args(argv)
    build.build()
    if a.from_log:
        sms, rows = rows_from_log(a.from_log)
        write_table(a.out, sms, rows)
        print(f"wrote {a.out}: {len(rows)} tactics")
        return
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    t0 = time.time()
    rows, log = [], []
    kept_rows = {}
    if a.min_rows > 0 and os.path.exists(a.out):
        _, old = rows_from_table(a.out)
        kept_rows = {r[:5]: r for r in old}
    for fmt, N, K, Ms in tuning_set(a.quick):
        shape = None
        for M in Ms:
            for comp in (False, True):
                key = (fmt, int(comp), M, N, K)
                if (2 * M if comp else M) < a.min_rows and key in kept_rows:
                    rows.append(kept_rows[key])
                    continue
                if shape is None:
                    shape = Shape(fmt, N, K)
                t, us, base, n, kept = tune_one(shape, M, comp, sms, a.margin)
                line = (f"fmt={fmt} comp={int(comp)} M={M} N={N} K={K} sms={sms}: analytic {base:.3f} us, "
                        f"best {us:.3f} us ({t[0]}, {t[1]}, {t[2]}, {t[3]}){' analytic' if kept else ''} over {n} plans")
                print(line, flush=True)
                log.append(line)
                rows.append((fmt, int(comp), M, N, K, t, us, base, kept))
        del shape
        torch.cuda.empty_cache()
    rs.rs_reset_tactics(True)
    print(f"{len(rows)} tactics in {time.time() - t0:.0f} s", flush=True)
    if a.log:
        with open(a.log, "w") as f:
            f.write("\n".join(log) + "\n")
    if not a.quick:
        write_table(a.out, sms, rows)
        print("wrote", a.out)


if __name__ == "__main__":
    main()
