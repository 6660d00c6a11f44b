"""Benchmark of the residue-compensated FP4 linear layer on GB300.

One step = one residue-compensated NVFP4 linear call (online activation +
residue quantization, block-scaled tcgen05 GEMM with on-chip Fold, bf16
output) for the attention-projection workload: M=8 tokens, K=N=4096,
X = Student-t(nu=4) x per-channel LogNormal(0,1), W ~ N(0, 0.02^2), seed 0.
The weight operand is rotated over enough copies that every step reads it
from HBM (working set > 2x L2).  K steps are captured in one CUDA graph; the
graph is replayed several times, each replay timed with CUDA events between
synchronizations, and `value` is the median microseconds per step.

Extra keys: the paper's protocol (a 200-call graph, median of five replays,
also as the median over three fresh processes) and the latency of one call
on its own; config 1 (M=1, K=N=2048); the M in
{1,2,4,8} sweep of compensated vs W4A4 latency and HBM roofline fraction;
the MLP pair, the MXFP4 sweep, the prefill TFLOP/s, the 22 projection shapes,
the on-chip Fold ablation and ResAttn decode attention; the roofline of the dominant kernel; the CPU
oracle on all host cores and on one (and on a sample of the prefill rows);
an end-to-end number through host buffers; the SM clocks sampled during the
timed region.

--impl reference times the CPU oracle (the plain C reference) on the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "compensated FP4 linear µs & % HBM roofline at M=1–8 vs W4A4; TFLOP/s at M≥2048"
WORKLOAD = "nvfp4_compensated_linear_attn_proj_M8_K4096_N4096"

# DRAM bytes per launch of the dominant kernel from an ncu capture, keyed by
# the hash of the kernel sources it was taken on (null once they change).
TRAFFIC = {"sources_sha": "3c9985b531553ff8", "bytes_per_launch": 9596928}


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    for name in ("rs_gemm.cu", "rs_device.cuh", "rs_quant_core.cuh"):
        with open(os.path.join(ROOT, "block_scaled_quantized_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ------------------------------------------------------------ clock sampling --

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (200 ms)."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- GPU arm --

class Linear:
    """One prepared linear layer (weights quantized on the GPU, rotated copies)."""

    def __init__(self, torch, rs, workloads, fmt, recipe, M, compensated, copies_for_l2=True,
                 out_dtype=None, seed=None, N=None, K=None, w=None):
        self.torch, self.rs = torch, rs
        dev = torch.device("cuda")
        self.fmt, self.M, self.compensated = fmt, M, compensated
        x = workloads.make_x(recipe, M, K=K, seed=seed)
        if w is None:
            w = workloads.make_w(recipe, N=N, K=K, seed=seed)
        self.N, self.K = w.shape
        self.x_host = x
        self.x = x.to(dev)
        wg = w.to(dev)
        self.ax = torch.empty(1, dtype=torch.float32, device=dev)
        self.aw = torch.empty(1, dtype=torch.float32, device=dev)
        if fmt == rs.NVFP4:
            rs.rs_compute_tensor_scale(self.x, self.ax)   # calibrated activation scale
            rs.rs_compute_tensor_scale(wg, self.aw)
        wq = torch.empty(rs.rs_weight_bytes(fmt, self.N, self.K), dtype=torch.uint8, device=dev)
        rs.rs_quantize_weight(fmt, wg, self.aw if fmt == rs.NVFP4 else None, wq)
        del wg
        self.wq_bytes = wq.numel()
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(2, math.ceil(2 * l2 / self.wq_bytes) + 1) if copies_for_l2 else 1
        self.wqs = [wq] + [wq.clone() for _ in range(n - 1)]
        self.y = torch.empty((M, self.N), dtype=out_dtype or torch.bfloat16, device=dev)
        self.ws = rs.empty_workspace(fmt, M, self.N, self.K, compensated)
        rows = 2 * M if compensated else M
        self.xq = torch.empty(rs.rs_act_bytes(fmt, rows, self.K), dtype=torch.uint8, device=dev)
        quant = rs.rs_quantize_residue if compensated else rs.rs_quantize_fp4
        quant(fmt, self.x, self.ax if fmt == rs.NVFP4 else None, self.xq)
        torch.cuda.synchronize()

    def alphas(self):
        nv = self.fmt == self.rs.NVFP4
        return (self.ax if nv else None), (self.aw if nv else None)

    def call(self, i: int, prequantized: bool = False, x=None, y=None, own_scale: bool = False):
        rs = self.rs
        ax, aw = self.alphas()
        if own_scale:
            ax = None  # the call finds the activation tensor scale itself
        fn = rs.rs_linear_compensated if self.compensated else rs.rs_linear_w4a4
        wq = self.wqs[i % len(self.wqs)]
        y = self.y if y is None else y
        if prequantized:
            key = "xq_paired" if self.compensated else "xq"
            fn(self.fmt, self.M, self.N, self.K, alpha_x=ax, wq=wq, alpha_w=aw, y=y, workspace=self.ws,
               **{key: self.xq})
        else:
            fn(self.fmt, self.M, self.N, self.K, x=self.x if x is None else x, alpha_x=ax, wq=wq, alpha_w=aw,
               y=y, workspace=self.ws)

    def fused(self) -> bool:
        """librs quantizes inside the GEMM (one launch) when the activation
        tile has at most 32 rows (2M for compensated, M for W4A4)."""
        return (2 * self.M if self.compensated else self.M) <= 32

    def launches_per_call(self) -> int:
        return 1 if self.fused() else 2

    def call_bytes(self) -> int:
        return self.algo_bytes(self.fused())

    def algo_bytes(self, fused_quant: bool) -> int:
        """HBM bytes the call must move: weight codes + scales, X, Y, and,
        for the two-kernel path, the activation operand written and read."""
        bs = 16 if self.fmt == self.rs.NVFP4 else 32
        w = self.N * self.K // 2 + self.N * self.K // bs
        rows = 2 * self.M if self.compensated else self.M
        act = rows * (self.K // 2 + self.K // bs)
        xbytes = self.M * self.K * 2
        ybytes = self.M * self.N * self.y.element_size()
        return w + xbytes + ybytes + (0 if fused_quant else 2 * act)

    def gemm_bytes(self) -> int:
        """HBM bytes of the GEMM kernel alone: weights, activation operand, Y."""
        bs = 16 if self.fmt == self.rs.NVFP4 else 32
        rows = 2 * self.M if self.compensated else self.M
        return (self.N * self.K // 2 + self.N * self.K // bs + rows * (self.K // 2 + self.K // bs)
                + self.M * self.N * self.y.element_size())

    def flops(self) -> tuple[int, int]:
        useful = 2 * self.M * self.N * self.K
        return useful, (2 * useful if self.compensated else useful)


class KextLinear:
    """A prefill linear layer with selective compensation (K-Ext): channels
    chosen per group of 8 from a calibration score (mean |x| over calibration
    rows of the same recipe), extended weight [W | W[:, S]] quantized once."""

    def __init__(self, torch, rs, workloads, recipe, M, k, seed=None):
        self.torch, self.rs = torch, rs
        dev = torch.device("cuda")
        self.fmt, self.M, self.k = rs.NVFP4, M, k
        x = workloads.make_x(recipe, M, seed=seed)
        w = workloads.make_w(recipe, seed=seed)
        self.N, self.K = w.shape
        self.x = x.to(dev)
        calib = workloads.make_x(recipe, 256, seed=(seed or 0) + 7919).to(dev)
        score = torch.empty(self.K, dtype=torch.float32, device=dev)
        rs.rs_channel_mean_abs(calib, score)
        self.mask = torch.from_numpy(rs.rs_kext_select(score.cpu().numpy(), k)).to(dev)
        wg = w.to(dev)
        self.ax = torch.empty(1, dtype=torch.float32, device=dev)
        self.aw = torch.empty(1, dtype=torch.float32, device=dev)
        rs.rs_compute_tensor_scale(self.x, self.ax)
        rs.rs_compute_tensor_scale(wg, self.aw)
        self.wq = torch.empty(rs.rs_kext_weight_bytes(self.fmt, self.N, self.K, k), dtype=torch.uint8, device=dev)
        rs.rs_quantize_weight_kext(self.fmt, wg, k, self.aw, self.mask, self.wq)
        del wg
        self.y = torch.empty((M, self.N), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(rs.rs_kext_workspace_bytes(self.fmt, M, self.N, self.K, k), dtype=torch.uint8,
                              device=dev)
        torch.cuda.synchronize()

    def call(self, i: int):
        self.rs.rs_linear_kext(self.fmt, self.M, self.N, self.K, self.k, x=self.x, alpha_x=self.ax, mask=self.mask,
                               wq=self.wq, alpha_w=self.aw, y=self.y, workspace=self.ws)

    def launches_per_call(self) -> int:
        return 2

    def flops(self) -> tuple[int, int]:
        useful = 2 * self.M * self.N * self.K
        return useful, useful + useful * self.k // 8


def nmse_vs_bf16(torch, x, w, y) -> float:
    """Normalised squared error of y against the fp32 product of the bf16
    operands (an accuracy figure beside the timing, not a parity check)."""
    ref = x.float() @ w.float().t()
    return float(((y.float() - ref) ** 2).sum() / (ref ** 2).sum())


def shape_sweep(torch, rs, workloads, hbm, Ms=(8,)) -> list:
    """Compensated and W4A4 NVFP4 over the 22 projection shapes (N, K) the
    paper times one by one (Fig. 18 / 19): us per call and HBM fraction."""
    rows = []
    for N, K in workloads.PROJECTION_SHAPES:
        w = workloads.make_w("proj_shapes", N=N, K=K)
        for M in Ms:
            row = {"N": N, "K": K, "M": M}
            for comp in (False, True):
                lin = Linear(torch, rs, workloads, rs.NVFP4, "proj_shapes", M, comp, N=N, K=K, w=w)
                us, _ = graph_time_us(torch, lin.call, 30, reps=3)
                key = "comp" if comp else "w4a4"
                row[f"{key}_us"] = round(us, 3)
                row[f"{key}_hbm_frac"] = round(lin.call_bytes() / (us * 1e-6) / 1e9 / hbm, 4)
                del lin
            row["comp_over_w4a4"] = round(row["comp_us"] / row["w4a4_us"], 4)
            rows.append(row)
        del w
        torch.cuda.empty_cache()
    return rows


def capture(torch, fn_step, steps: int):
    """A CUDA graph of `steps` calls (after three eager warm-up calls)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            fn_step(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                fn_step(i)
    torch.cuda.synchronize()
    return g


def replay_us(torch, g, steps: int, reps: int, world: int = 1) -> list[float]:
    """us per call of each of `reps` replays of a graph of `steps` calls, each
    replay bracketed by a barrier (several ranks) and a synchronize."""
    times = []
    for _ in range(reps):
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0 / steps)
    return times


def isolated_call_us(torch, lin, reps: int = 60) -> dict:
    """Latency of one call with no kernel of ours in flight before it: one
    call per CUDA graph (one graph per weight copy, so each call reads its
    weights from HBM), launched behind a sleep kernel so that the host launch
    is hidden, CUDA events right around it."""
    graphs = [capture(torch, lambda i, c=c: lin.call(c), 1) for c in range(len(lin.wqs))]
    times = []
    for r in range(reps):
        g = graphs[r % len(graphs)]
        torch.cuda._sleep(40000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0)
    return {"us": round(statistics.median(times), 3), "min_us": round(min(times), 3), "calls": reps}


def fold_ablation(torch, rs, workloads, hbm, Ms=(1, 2, 4, 8, 16, 32, 64)) -> list:
    """On-chip Fold against writing the expanded Z and folding in a separate
    kernel (Sec. 5.1, Fig. 6b), compensated NVFP4, K = N = 4096: both start
    from the standalone paired quantizer; the unfused path runs the plain
    GEMM over the 2M paired rows with fp32 output, then rs_fold_pairs."""
    rows = []
    for M in Ms:
        lin = Linear(torch, rs, workloads, rs.NVFP4, "attn_proj_k4096", M, True)
        z = torch.empty((2 * M, lin.N), dtype=torch.float32, device="cuda")

        def quant(i):
            rs.rs_quantize_residue(rs.NVFP4, lin.x, lin.ax, lin.xq)

        def onchip(i):
            quant(i)
            rs.rs_linear_compensated(rs.NVFP4, M, lin.N, lin.K, xq_paired=lin.xq, alpha_x=lin.ax,
                                     wq=lin.wqs[i % len(lin.wqs)], alpha_w=lin.aw, y=lin.y, workspace=lin.ws)

        def separate(i):
            quant(i)
            rs.rs_linear_w4a4(rs.NVFP4, 2 * M, lin.N, lin.K, xq=lin.xq, alpha_x=lin.ax,
                              wq=lin.wqs[i % len(lin.wqs)], alpha_w=lin.aw, y=z, workspace=lin.ws)
            rs.rs_fold_pairs(M, lin.N, z, lin.y)

        a, _ = graph_time_us(torch, onchip, 100)
        b, _ = graph_time_us(torch, separate, 100)
        c, _ = graph_time_us(torch, lin.call, 100)
        rows.append({"M": M, "onchip_fold_us": round(a, 3), "separate_fold_us": round(b, 3),
                     "separate_over_onchip": round(b / a, 4), "one_launch_us": round(c, 3)})
        del lin, z
    return rows


RESATTN_CASES = [
    # (B, Hq, Hkv, D, tokens per sequence): head sizes 128 / 256, 4 to 8 query heads per KV head
    (1, 32, 8, 128, 32768), (8, 32, 8, 128, 8192), (32, 32, 8, 128, 2048), (1, 32, 4, 128, 131072),
    (4, 48, 8, 256, 16384), (16, 64, 8, 128, 4096),
]


class ResAttnCase:
    """One ResAttn decode workload: synthetic paged NVFP4 caches (random
    codes, E4M3 scales in [2^-2, 2^2], every sequence full length, a shuffled
    block table), rotated over enough copies that each step reads its cache
    from HBM.  Algorithmic bytes: K and V of every cached token and KV head,
    2 (D/2 + D/16) bytes (144 B at D = 128), plus Q and O."""

    def __init__(self, torch, rs, B, Hq, Hkv, D, L, gen):
        self.rs = rs
        self.B, self.Hq, self.Hkv, self.D, self.L = B, Hq, Hkv, D, L
        pages = (L + 31) // 32
        page_bytes = 32 * (D // 2 + D // 16)
        cache_bytes = B * pages * Hkv * page_bytes
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        self.copies = max(2, math.ceil(2 * l2 / (2 * cache_bytes)) + 1)
        self.caches = []
        for _ in range(self.copies):
            kv = []
            for _ in range(2):
                c = torch.randint(0, 256, (B * pages, Hkv, page_bytes), dtype=torch.uint8, device="cuda",
                                  generator=gen)
                sc = torch.randint(0x28, 0x49, (B * pages, Hkv, 32 * (D // 16)), dtype=torch.uint8, device="cuda",
                                   generator=gen)
                c[:, :, 32 * (D // 2):] = sc
                kv.append(c)
            self.caches.append(kv)
        self.table = torch.randperm(B * pages, device="cuda", generator=gen).to(torch.int32).reshape(B, pages)
        self.lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
        self.q = (torch.randn((B, Hq, D), device="cuda", generator=gen)).to(torch.bfloat16)
        self.aq = torch.empty(1, dtype=torch.float32, device="cuda")
        rs.rs_compute_tensor_scale(self.q, self.aq)
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        self.ws = torch.empty(rs.rs_resattn_workspace_bytes(B, Hq, Hkv, D, L), dtype=torch.uint8, device="cuda")
        self.algo_bytes = 2 * B * L * Hkv * (D // 2 + D // 16) + 2 * B * Hq * D * 2

    def step(self, i):
        k, v = self.caches[i % self.copies]
        self.rs.rs_resattn_decode(self.q, self.aq, k, v, self.table, self.lens, self.L, self.out, self.ws, self.Hkv)


def resattn_leg(torch, rs, hbm) -> list:
    """ResAttn decode steps (ResAttnCase) timed in CUDA graphs."""
    rows = []
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    for B, Hq, Hkv, D, L in RESATTN_CASES:
        case = ResAttnCase(torch, rs, B, Hq, Hkv, D, L, gen)
        us, _ = graph_time_us(torch, case.step, 30)
        algo = case.algo_bytes
        rows.append({"B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "tokens": L, "us": round(us, 2),
                     "achieved_gbs": round(algo / (us * 1e-6) / 1e9, 1),
                     "hbm_frac": round(algo / (us * 1e-6) / 1e9 / hbm, 4), "kv_bytes_per_token_head": 2 * (D // 2 + D // 16)})
        del case
        torch.cuda.empty_cache()
    assert rs.rs_get_device_error() == 0
    return rows


def graph_time_us(torch, fn_step, steps: int, reps: int = 5, warm: int = 3) -> tuple[float, list[float]]:
    """Capture `steps` calls in a CUDA graph; return median us per call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            fn_step(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                fn_step(i)
    torch.cuda.synchronize()
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0 / steps)
    return statistics.median(times), times


PROFILE_CASES = {
    # name: (format, recipe, M, compensated)
    "prefill_w4a4": (0, "prefill_k8192", 4096, False),
    "prefill_comp": (0, "prefill_k8192", 4096, True),
    "mlp_gate_up": (0, "mlp_gate_up", 8, True),
    "mlp_down": (0, "mlp_down", 8, True),
    "mx_m1": (1, "mx_k5120_n27648", 1, True),
    "prefill_kext1": (0, "prefill_k8192", 4096, "kext1"),
    "prefill_w4a4_pair": (0, "prefill_k8192", 4096, False, "pair"),
    # ResAttn decode: (B, Hq, Hkv, D, tokens per sequence)
    "resattn_b8_l8192": ("resattn", (8, 32, 8, 128, 8192)),
}


def run_profile_case(args) -> dict:
    """One workload's linear calls, graph-replayed (for profiler runs: ncu
    captures the launches; the printed time is not a bench value)."""
    import torch
    from block_scaled_quantized_gb300 import build, rs, workloads
    build.build()
    case = PROFILE_CASES[args.profile_case]
    if case[0] == "resattn":
        gen = torch.Generator(device="cuda")
        gen.manual_seed(0)
        att = ResAttnCase(torch, rs, *case[1], gen)
        us, _ = graph_time_us(torch, att.step, args.steps, reps=1, warm=args.warmup)
        assert rs.rs_get_device_error() == 0
        return {"profile_case": args.profile_case, "us_per_call": round(us, 3), "launches_per_call": 2}
    fmt, recipe, M, comp = case[:4]
    rs.rs_debug_pair_gemm(len(case) > 4 and case[4] == "pair")
    if comp == "kext1":
        lin = KextLinear(torch, rs, workloads, recipe, M, 1)
    else:
        lin = Linear(torch, rs, workloads, fmt, recipe, M, comp, copies_for_l2=M <= 128)
    us, _ = graph_time_us(torch, lin.call, args.steps, reps=1, warm=args.warmup)
    assert rs.rs_get_device_error() == 0
    return {"profile_case": args.profile_case, "us_per_call": round(us, 3), "launches_per_call": lin.launches_per_call()}


def processes_protocol(n: int) -> dict:
    """The headline's 200-call graph timed in n fresh processes, one after
    the other (each: median of five replays); their median."""
    vals = []
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--headline-only", "--steps", "200", "--warmup", "5",
           "--soak-s", "0", "--replays", "5"]
    for _ in range(n):
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=180, cwd=ROOT)
        if r.returncode != 0:
            return {"error": f"process exited {r.returncode}", "us": vals}
        vals.append(json.loads(r.stdout.strip().splitlines()[-1])["value"])
    return {"processes": n, "graph_calls": 200, "us": vals, "median_us": round(statistics.median(vals), 3)}


def max_over_ranks(value: float, world: int, device: str) -> float:
    """The slowest rank's value (the job's time), via an all-reduce over the
    initialised process group; the value itself with one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_gpu(args) -> dict:
    import torch
    import torch.distributed as dist
    from block_scaled_quantized_gb300 import build, rs, workloads

    build.build()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    peaks = load_peaks()
    num_sms = torch.cuda.get_device_properties(local).multi_processor_count

    # ---------------- headline: compensated, M=8, K=N=4096, NVFP4
    main = Linear(torch, rs, workloads, rs.NVFP4, "attn_proj_k4096", 8, True)
    K_steps, W = args.steps, args.warmup
    g = capture(torch, main.call, K_steps)
    for _ in range(W):
        g.replay()
    torch.cuda.synchronize()
    # soak (untimed replays) so that the clock samples see the GPU under load
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + args.soak_s
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize()
    # the timed region: `replays` replays of the K-step graph, each bracketed
    # by a barrier and a synchronize; the step time is their median
    reps = replay_us(torch, g, K_steps, max(5, args.replays), world)
    clocks = sampler.stop()
    us_local = statistics.median(reps)
    if args.headline_only:
        out = {"metric": METRIC, "value": round(us_local, 3), "unit": "us", "n_gpus": world,
               "steps": K_steps, "warmup": W, "headline_only": True, "clocks": clocks}
        return out if rank == 0 else None
    us_per_step = max_over_ranks(us_local, world, "cuda")
    hbm = peaks["hbm_gbs"]
    # the paper's protocol (App. C.1): CUDA-graph replay of >= 200 calls,
    # median of five replays; and one call on its own
    g200 = capture(torch, main.call, 200)
    protocol = {"graph_calls": 200, "replays": 5, "us": round(statistics.median(replay_us(torch, g200, 200, 5)), 3)}
    del g200
    # ... and the median over independent processes (App. C.1 takes medians
    # over at least three): the same 200-call measurement in fresh processes
    if world == 1 and args.processes > 0:
        protocol["processes"] = processes_protocol(args.processes)
    sampler2 = ClockSampler(local)
    sampler2.start()
    isolated = isolated_call_us(torch, main)
    isolated["clocks"] = sampler2.stop()

    # ---------------- dominant kernel alone: the GEMM on a pre-quantized operand
    # The headline step is one launch of the fused quantize+GEMM+Fold kernel,
    # so its average launch duration is the timed region over K steps.
    assert main.launches_per_call() == 1
    head_gbs = main.call_bytes() / (us_per_step * 1e-6) / 1e9
    traffic = TRAFFIC["bytes_per_launch"] if TRAFFIC["sources_sha"] == kernel_sources_sha() else None
    # For reference: the GEMM alone on a pre-quantized operand.
    gemm_us, _ = graph_time_us(torch, lambda i: main.call(i, prequantized=True), K_steps)
    gemm_gbs = main.gemm_bytes() / (gemm_us * 1e-6) / 1e9

    # the headline call finding its own activation tensor scale (no alpha_x)
    own_us, _ = graph_time_us(torch, lambda i: main.call(i, own_scale=True), K_steps)
    extra_own = {"us": round(own_us, 3), "over_given_scale": round(own_us / us_per_step, 4)}

    # ---------------- config 1: NVFP4, M = 1, K = N = 2048 (compensated and W4A4)
    cfg1 = {}
    for comp in (False, True):
        lin = Linear(torch, rs, workloads, rs.NVFP4, "gauss_outlier_k2048", 1, comp)
        us, _ = graph_time_us(torch, lin.call, 200)
        key = "comp" if comp else "w4a4"
        cfg1[f"{key}_us"] = round(us, 3)
        cfg1[f"{key}_hbm_frac"] = round(lin.call_bytes() / (us * 1e-6) / 1e9 / hbm, 4)
        del lin
    cfg1["comp_over_w4a4"] = round(cfg1["comp_us"] / cfg1["w4a4_us"], 4)

    # ---------------- sweep M = 1, 2, 4, 8 compensated vs W4A4
    sweep = []
    for M in (1, 2, 4, 8):
        row = {"M": M}
        for comp in (False, True):
            lin = main if (M == 8 and comp) else Linear(torch, rs, workloads, rs.NVFP4, "attn_proj_k4096", M, comp)
            us, _ = graph_time_us(torch, lin.call, 100)
            key = "comp" if comp else "w4a4"
            row[f"{key}_us"] = round(us, 3)
            row[f"{key}_hbm_frac"] = round(lin.call_bytes() / (us * 1e-6) / 1e9 / hbm, 4)
        row["comp_over_w4a4"] = round(row["comp_us"] / row["w4a4_us"], 4)
        sweep.append(row)

    extra = {}
    if not args.quick:
        # MLP pair (gate/up fused then down), M=8, compensated
        mlp = {}
        tot = 0.0
        for recipe in ("mlp_gate_up", "mlp_down"):
            lin = Linear(torch, rs, workloads, rs.NVFP4, recipe, 8, True)
            us, _ = graph_time_us(torch, lin.call, 50)
            mlp[recipe] = {"us": round(us, 3), "hbm_frac": round(lin.call_bytes() / (us * 1e-6) / 1e9 / hbm, 4)}
            tot += us
            del lin
        mlp["sum_us"] = round(tot, 3)
        extra["mlp_pair_m8"] = mlp
        # MXFP4 sweep
        mx = []
        for M in (1, 4, 8, 16, 32, 64, 128):
            row = {"M": M}
            for comp in (False, True):
                lin = Linear(torch, rs, workloads, rs.MXFP4, "mx_k5120_n27648", M, comp)
                us, _ = graph_time_us(torch, lin.call, 30)
                key = "comp" if comp else "plain"
                row[f"{key}_us"] = round(us, 3)
                row[f"{key}_hbm_frac"] = round(lin.call_bytes() / (us * 1e-6) / 1e9 / hbm, 4)
                del lin
            row["comp_over_plain"] = round(row["comp_us"] / row["plain_us"], 4)
            mx.append(row)
        extra["mxfp4_k5120_n27648"] = mx
        # the paper's 22 projection shapes at M = 8 (M in {1, 8, 64, 512} with --shapes)
        extra["projection_shapes_nvfp4"] = shape_sweep(torch, rs, workloads, hbm,
                                                       Ms=(1, 8, 64, 512) if args.shapes else (8,))
        # prefill M=4096, K=N=8192
        pre = {}
        w_pre = workloads.make_w("prefill_k8192").to(torch.device("cuda"))
        variants = [("w4a4", False, 0), ("comp", True, 0), ("kext1", None, 1), ("kext2", None, 2)]
        for key, comp, k in variants:
            if k:
                lin = KextLinear(torch, rs, workloads, "prefill_k8192", 4096, k)
            else:
                lin = Linear(torch, rs, workloads, rs.NVFP4, "prefill_k8192", 4096, comp, copies_for_l2=False)
            us, _ = graph_time_us(torch, lin.call, 10, reps=3)
            useful, executed = lin.flops()
            pre[f"{key}_us"] = round(us, 2)
            if not k:
                # the GEMM alone on the quantized operand: the default kernel, and the
                # paired-CTA kernel (cta_group::2, 256 x 256 per pair) for comparison
                g1, _ = graph_time_us(torch, lambda i: lin.call(i, prequantized=True), 10, reps=3)
                rs.rs_debug_pair_gemm(True)
                try:
                    g2, _ = graph_time_us(torch, lambda i: lin.call(i, prequantized=True), 10, reps=3)
                finally:
                    rs.rs_debug_pair_gemm(False)
                pre[f"{key}_gemm_only_us"] = round(g1, 2)
                pre[f"{key}_gemm_only_frac"] = round(executed / (g1 * 1e-6) / 1e12 / (peaks["bf16_tflops"] * 6), 4)
                pre[f"{key}_pair_cta_gemm_only_us"] = round(g2, 2)
            pre[f"{key}_useful_tflops"] = round(useful / (us * 1e-6) / 1e12, 1)
            pre[f"{key}_executed_tflops"] = round(executed / (us * 1e-6) / 1e12, 1)
            lin.call(0)
            torch.cuda.synchronize()
            pre[f"{key}_nmse_vs_bf16"] = float(f"{nmse_vs_bf16(torch, lin.x, w_pre, lin.y):.4e}")
            del lin
        del w_pre
        pre["kext_rho"] = {"kext1": 0.125, "kext2": 0.25}
        # FP4 dense peak: the measured bf16 peak x the nominal FP4/bf16 ratio (13.5 / 2.25)
        fp4_peak = peaks["bf16_tflops"] * 13.5 / 2.25
        pre["fp4_peak_tflops"] = round(fp4_peak, 1)
        pre["fp4_peak_source"] = f"{peaks['source']} bf16 x 6"
        pre["w4a4_frac"] = round(pre["w4a4_executed_tflops"] / fp4_peak, 4)
        pre["comp_frac"] = round(pre["comp_executed_tflops"] / fp4_peak, 4)
        for key in ("kext1", "kext2"):
            pre[f"{key}_frac"] = round(pre[f"{key}_executed_tflops"] / fp4_peak, 4)
        extra["prefill_M4096_K8192_N8192"] = pre
        torch.cuda.empty_cache()
        extra["fold_ablation_k4096_n4096"] = fold_ablation(torch, rs, workloads, hbm)
        extra["resattn_decode"] = resattn_leg(torch, rs, hbm)

    # ---------------- end to end through host buffers (pinned), public API
    xh = main.x_host.pin_memory()
    yh = torch.empty((main.M, main.N), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(main.x)

    def e2e_step(i):
        xd.copy_(xh, non_blocking=True)
        main.call(i, x=xd)
        yh.copy_(main.y, non_blocking=True)

    e2e_us, _ = graph_time_us(torch, e2e_step, K_steps)

    out = {
        "metric": METRIC,
        "value": round(us_per_step, 3),
        "unit": "us",
        "n_gpus": world,
        "steps": K_steps,
        "warmup": W,
        "ms_per_step": round(us_per_step / 1000.0, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e4m3 block scale) with fp32 accumulation, bf16 out",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 8, "K": 4096, "N": 4096, "format": "nvfp4",
                   "compensated": True, "global_batch": 8, "weight_copies": len(main.wqs),
                   "l2_policy": "weights rotated over copies > 2x L2 (inputs larger than L2)",
                   "parallelism": f"replicas{world}",
                   "timing": f"cuda-graph of K calls, median of {max(5, args.replays)} replays, cuda events"},
        "replays_us": [round(t, 3) for t in reps],
        "protocol_graph200": protocol,
        "isolated_call": isolated,
        "config1_nvfp4_m1_k2048_n2048": cfg1,
        "sweep_attn_proj_k4096": sweep,
        "headline_own_tensor_scale": extra_own,
        **extra,
        "roofline": {"bound": "hbm",
                     "kernel": "gemm_kernel<nvfp4, bn=16, fused> (quantizing prologue + tcgen05 GEMM + Fold)",
                     "achieved": round(head_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(head_gbs / hbm, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": main.call_bytes(), "launch_us": round(us_per_step, 3),
                     "peak_source": peaks["source"]},
        "gemm_only_prequantized": {"achieved": round(gemm_gbs, 1), "unit": "GB/s", "frac": round(gemm_gbs / hbm, 4),
                     "algorithmic_bytes_per_launch": main.gemm_bytes(), "launch_us": round(gemm_us, 3),
                     "peak_source": peaks["source"]},
        "e2e": {"value": round(e2e_us, 3), "unit": "us",
                "h2d_bytes_per_step": main.M * main.K * 2, "d2h_bytes_per_step": main.M * main.N * 2},
        "gpu_launches": main.launches_per_call() * K_steps,
        "clocks": clocks,
        "num_sms": num_sms,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        if not args.quick:
            out["cpu_oracle_prefill_sample"] = cpu_prefill_sample()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return out if rank == 0 else None


# --------------------------------------------------------------- CPU oracle --

def _oracle_headline_inputs():
    import oracle
    from block_scaled_quantized_gb300 import workloads
    oracle.build()
    x = workloads.make_x("attn_proj_k4096", 8)
    w = workloads.make_w("attn_proj_k4096")
    xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
    aw = oracle.tensor_scale(wb)
    cw, sw, _ = oracle.quantize(0, wb, aw)          # offline weight quantization: untimed
    ax = oracle.tensor_scale(xb)                    # calibrated activation scale: untimed
    return xb, ax, cw, sw, aw


def _time_oracle_calls(args, budget_s: float, max_calls: int) -> list:
    import oracle
    times = []
    t_end = time.time() + budget_s
    while True:
        t0 = time.perf_counter()
        oracle.linear(0, True, *args)
        times.append(time.perf_counter() - t0)
        if time.time() > t_end or len(times) >= max_calls:
            break
    return times


def cpu_baseline(budget_s: float) -> dict:
    """The oracle (plain C, double GEMM) on the same workload, one compensated
    linear call at M=8, K=N=4096: on all host cores (OpenMP over the output
    elements; `value`, `cores`) and single-threaded, ~budget_s in total."""
    import oracle
    inputs = _oracle_headline_inputs()
    cores = os.cpu_count() or 1
    oracle.set_threads(1)
    single = _time_oracle_calls(inputs, budget_s / 2, 30)
    oracle.set_threads(cores)
    multi = _time_oracle_calls(inputs, budget_s / 2, 200)
    oracle.set_threads(1)
    return {"value": round(statistics.median(multi) * 1e6, 1), "unit": "us", "cores": cores, "kind": "oracle",
            "single_thread_us": round(statistics.median(single) * 1e6, 1),
            "sample": f"full workload step (M=8, K=N=4096 compensated NVFP4): median of {len(multi)} calls "
                      f"on {cores} threads, {len(single)} calls on one thread"}


def cpu_prefill_sample(rows: int = 256) -> dict:
    """The oracle on a seeded sample of the prefill workload (M = 4096,
    K = N = 8192, compensated): `rows` token rows x all N, on all cores; the
    time of the whole call is that x 4096 / rows (labelled as extrapolated)."""
    import numpy as np
    import oracle
    from block_scaled_quantized_gb300 import workloads
    oracle.build()
    cores = os.cpu_count() or 1
    x = workloads.make_x("prefill_k8192", 4096)
    pick = np.sort(np.random.default_rng(5).choice(4096, rows, replace=False))
    xb = workloads.bf16_bits(x)[pick]
    wb = workloads.bf16_bits(workloads.make_w("prefill_k8192"))
    oracle.set_threads(cores)
    aw = oracle.tensor_scale(wb)
    cw, sw, _ = oracle.quantize(0, wb, aw)
    ax = oracle.tensor_scale(workloads.bf16_bits(x))
    t0 = time.perf_counter()
    oracle.linear(0, True, xb, ax, cw, sw, aw)
    dt = time.perf_counter() - t0
    oracle.set_threads(1)
    return {"rows": rows, "N": 8192, "K": 8192, "seconds": round(dt, 3), "cores": cores,
            "extrapolated_full_call_s": round(dt * 4096 / rows, 2), "kind": "oracle",
            "sample": f"{rows} seeded token rows of 4096 x all 8192 channels, compensated NVFP4"}


def run_reference(args) -> dict | None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    base = cpu_baseline(max(5.0, min(60.0, args.cpu_seconds)))
    steps = max(1, min(args.steps, 5))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": base["value"],
        "unit": "us",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(base["value"] / 1000.0, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 quantizer, f64 GEMM",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 8, "K": 4096, "N": 4096, "format": "nvfp4", "compensated": True},
        "cpu_baseline": base,
        "e2e": {"value": base["value"], "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline and M sweep only")
    ap.add_argument("--shapes", action="store_true",
                    help="projection-shape sweep at M in {1, 8, 64, 512} (default: M = 8)")
    ap.add_argument("--soak-s", type=float, default=1.5)
    ap.add_argument("--replays", type=int, default=7, help="timed replays of the K-step graph (median; at least 5)")
    ap.add_argument("--processes", type=int, default=3,
                    help="fresh processes for the 200-call protocol figure (0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the headline step only (for profiler runs; no sweeps, no baselines)")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES),
                    help="run one other workload's calls only (for profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.profile_case:
        out = run_profile_case(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
