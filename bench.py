"""Benchmark of the FP8 NT GEMM library on its headline workload.

Workload (one step): the dense sweep m in {64, 128, 4096} x (n, k) in
{(2112,7168), (24576,1536), (7168,16384), (4096,7168), (7168,2048)}: fifteen
FP8 E4M3 NT GEMMs with 1x128 (LHS) and 128x128 (RHS) FP32 scales and BF16
output, inputs made from seeded N(0,1) values (scale = amax/448).  Every
problem rotates over identical copies of its inputs and output that together
exceed twice the L2 cache, so no launch finds its inputs in L2; the K launches
of a problem run back to back between one pair of CUDA events.

Printed: one JSON line on rank 0 with the metric (TFLOP/s over valid FLOPs),
per-shape TFLOP/s and GB/s, the roofline of the dominant kernel, the
end-to-end figure (host buffers, copies inside the timed region), the clocks
seen during the timed region and the CPU oracle as a reported baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs the same sweep on its own GPU (independent
problems, weak scaling); the value is the total work over the slowest rank.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "FP8 GEMM TFLOPS (valid FLOPs) & HBM GB/s, % of GB300 roofline, 1 GPU"
UNIT = "TFLOP/s"
WORKLOAD = ("dense sweep: m in {64,128,4096} x (n,k) in {(2112,7168),(24576,1536),(7168,16384),"
            "(4096,7168),(7168,2048)}, FP8 E4M3 NT, 1x128/128x128 FP32 scales (amax/448), BF16 out")
ROTATE_BYTES = 272 << 20  # > 2 x the 129 MB L2 of a GB300
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor-core ratio (4.5 / 2.25 PFLOP/s)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def sweep_problems():
    """Host problems of the sweep: one seeded m=4096 problem per (n,k); the
    m = 64 and m = 128 problems are its leading rows."""
    probs = {}
    for i, (n, k) in enumerate(wl.DENSE_SWEEP_NK):
        probs[(n, k)] = wl.dense(max(wl.DENSE_SWEEP_M), n, k, seed=wl.seed_for(1, i))
    shapes = [(m, n, k) for m in wl.DENSE_SWEEP_M for (n, k) in wl.DENSE_SWEEP_NK]
    return probs, shapes


def kernel_name(block_n, split, pair=0, swap=0, defer=0):
    if pair:
        if defer:
            return "fg::fp8_gemm_pair_kernel<dense,4,8,deferred stores> (256x256 tiles on CTA pairs)"
        return "fg::fp8_gemm_pair_kernel<dense,5,8> (256x256 tiles on CTA pairs)"
    if swap:
        return f"fg::fp8_gemm_swap_kernel<{block_n},dense,{'splitk' if split > 1 else 'persistent'}>"
    stages = 4 if block_n == 256 else 6
    return f"fg::fp8_gemm_kernel<{block_n},{stages},dense,{'splitk' if split > 1 else 'persistent'}>"


def plan_of(fg, m, n, k):
    """(block_n, split_k, cta_pair, swap_ab, deferred_stores) of a dense call."""
    return tuple(fg.fg_query_plan(0, m, 1, n, k))


def kernel_sources_digest():
    """Digest of the CUDA sources with comments removed and white space
    collapsed: DRAM traffic figures are only used when they were captured on
    kernels built from the same code."""
    import hashlib
    import re
    h = hashlib.sha1()
    d = os.path.join(ROOT, "moe_grouped_gemm_nt_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            text = fh.read()
        # drop comments (string literals in these sources hold no comment markers)
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"\s+", " ", text)
        h.update(f.encode() + text.encode())
    return h.hexdigest()[:16]


def load_traffic():
    """{(m, n, k): DRAM bytes per launch} from profiles/dram_traffic.txt lines
    '<digest> <m> <n> <k> <read+write bytes>' of the current sources (n = 0:
    the activation quantizer on [m][k])."""
    out = {}
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return out
    dig = kernel_sources_digest()
    for line in open(path):
        f = line.split()
        if len(f) == 5 and not line.startswith("#") and f[0] == dig:
            out[(int(f[1]), int(f[2]), int(f[3]))] = float(f[4])
    return out


def bench_config(ws):
    """The `config` object of the JSON line: the same for both arms, so that the
    reference arm (the CPU oracle) is read as a run of the same workload."""
    return {"workload": WORKLOAD, "problems_per_step": len(wl.DENSE_SWEEP_M) * len(wl.DENSE_SWEEP_NK),
            "l2": ("inputs larger than L2: each problem rotates over identical copies of its "
                   "inputs and output totalling >= 272 MiB (> 2 x L2)"),
            "timing": ("CUDA events on the launching stream around K back-to-back steps; a step "
                       "launches every problem once, grouped by kernel instantiation with an event "
                       "at each group boundary (per-kernel device time); the per-problem table comes "
                       "from K launches of each problem captured in a CUDA graph and replayed after "
                       "the timed steps"),
            "parallelism": f"replica x{ws} (independent problems per GPU)"}


def problem_bytes(m, n, k):
    kb, nb = (k + 127) // 128, (n + 127) // 128
    return m * k + n * k + m * kb * 4 + nb * kb * 4 + m * n * 2


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        rows = []
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) >= 9:
                    rows.append([x.strip() for x in r])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------ distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    """Largest value of x over all ranks (timing only; no data-path exchange)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ CPU oracle

_ORACLE_CALIB = {}


def oracle_sample_rate(probs, shapes, seconds: float, seed: int = 0):
    """Time the CPU oracle (as it stands) on a bounded sample of the sweep:
    the same number of random output elements of every problem, sized for
    about `seconds` of work.  Returns (TFLOP/s of valid work, cores, sample text)."""
    import oracle

    rng = np.random.default_rng(seed)

    def run(per_shape):
        flops = 0.0
        t0 = time.perf_counter()
        for (m, n, k) in shapes:
            p = probs[(n, k)]
            rows = rng.integers(0, m, per_shape)
            cols = rng.integers(0, n, per_shape)
            oracle.gemm_fp8_nt_at(p.A[:m], 0, p.sA[:m], p.B, 0, p.sB, rows, cols)
            flops += 2.0 * k * per_shape
        return flops, time.perf_counter() - t0

    # calibration (once per process): grow the sample until the fixed cost of
    # a call (thread start-up, Python) no longer dominates, then scale to `seconds`
    if "s_per_elem" not in _ORACLE_CALIB:
        per, (f0, t0) = 256, run(256)
        while t0 < 0.5 and per < (1 << 20):
            per *= 4
            f0, t0 = run(per)
        _ORACLE_CALIB["s_per_elem"] = t0 / per
    per = int(max(64, min(1 << 22, seconds / max(_ORACLE_CALIB["s_per_elem"], 1e-12))))
    f, t = run(per)
    sample = (f"{per} random output elements of each of the {len(shapes)} sweep problems "
              f"({f / 2e9:.1f} G MAC, {t:.1f} s)")
    return f / t / 1e12, oracle.num_threads(), sample


# ------------------------------------------------------------------ arms

def graph_us(torch, launch, n_launch):
    """Device time per launch of `n_launch` calls `launch(r, stream)` captured in
    one CUDA graph on a side stream, replayed once to warm up and once between
    CUDA events.  The calls allocate nothing and never synchronize, so they
    capture as they are; replay removes the host's per-call cost (about 8 us
    through the Python binding), which the small problems would otherwise
    expose."""
    gs = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        for r in range(n_launch):
            launch(r, gs)
    with torch.cuda.stream(gs):
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(gs)
        g.replay()
        e1.record(gs)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n_launch
    del g
    return us


def quantize_bytes(rows, k, x_bytes=2):
    """Algorithmic HBM bytes of one per-token quantization: X (BF16, or FP32
    with x_bytes = 4) read once, FP8 A and one FP32 scale per row and 128-wide
    K block written once."""
    return rows * k * x_bytes + rows * k + rows * ((k + 127) // 128) * 4


def measure_quantize(fg, torch, dev, stream, hbm_peak, peak_src, reps=20, traffic_tab=None, f32_input=False):
    """Per-token FP8 quantization of the sweep's m = 4096 activations
    (BF16 [4096][k], or FP32 with f32_input, k in the sweep), each shape
    rotating over copies of X, A and sA larger than twice L2; `reps`
    back-to-back launches between CUDA events on the launching stream, after a
    warm-up."""
    ks = sorted({k for (_, k) in wl.DENSE_SWEEP_NK})
    rows_out, tot_b, tot_s = [], 0.0, 0.0
    xdt = torch.float32 if f32_input else torch.bfloat16
    for k in ks:
        m = max(wl.DENSE_SWEEP_M)
        x = torch.from_numpy(wl.activations((m, k), seed=wl.seed_for(1, 50 + k % 97))).to(xdt).to(dev)
        nb = quantize_bytes(m, k, 4 if f32_input else 2)
        ncopy = max(2, -(-ROTATE_BYTES // nb))
        copies = [(x.clone(), torch.empty((m, k), dtype=torch.float8_e4m3fn, device=dev),
                   torch.empty(((k + 127) // 128, fg.fg_scales_a_ld(m)), dtype=torch.float32, device=dev))
                  for _ in range(ncopy)]
        del x
        for X, A, sA in copies[:3]:
            fg.fg_quantize_fp8_per_token(X, A, sA, stream=stream)
        us = graph_us(torch, lambda r, st: fg.fg_quantize_fp8_per_token(*copies[r % ncopy], stream=st), reps)
        rows_out.append({"m": m, "k": k, "us": round(us, 2), "gbs": round(nb / (us * 1e-6) / 1e9, 1),
                         "algorithmic_bytes": nb,
                         "traffic": None if f32_input else (traffic_tab or {}).get((m, 0, k))})
        tot_b += nb
        tot_s += us * 1e-6
        del copies
    st, _ = fg.fg_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the quantization runs")
    ach = tot_b / tot_s / 1e9
    known = [r["traffic"] for r in rows_out]
    traffic = sum(known) / len(known) if all(v is not None for v in known) else None
    return {"kernel": "fg::quantize_per_token_kernel<E4M3, " + ("FP32" if f32_input else "BF16") + " input>",
            "algorithmic_bytes_per_launch": tot_b / len(rows_out),
            "workload": (("FP32" if f32_input else "BF16") +
                         " activations [4096][k] -> FP8 E4M3 A + MN-major 1x128 FP32 scales, k in the sweep"),
            "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(ach / hbm_peak, 3), "traffic": traffic,
                         "peak_source": f"{peak_src}: hbm copy"},
            "timing": (f"{reps} launches per shape captured in a CUDA graph and replayed between CUDA events, "
                       "rotating over copies >= 272 MiB (> 2 x L2), after the GEMM steps"),
            "shapes": rows_out}


def measure_other_configs(fg, torch, dev, stream, fp8_peak, hbm_peak, peak_src, reps=10):
    """Throughput of the other workloads (the parity tests cover their results):
    contiguous G in {4, 8} x 8192 rows per group, masked G in {1, 2, 4, 16} with
    capacity 256 and seeded uniform counts, and the large square problems
    (8192^3, k = 8192 + 384, E5M2 B).  Operands are drawn on the device from a
    seeded generator (N(0,1) x 64 clipped to the E4M3 range: the timing does not
    depend on the values); scales uniform in [0.5, 1.5], log-uniform in
    [2^-8, 2^8] for the square problems.  Each problem rotates over copies of
    its inputs and output larger than twice L2, `reps` back-to-back launches
    between CUDA events."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed_for(5))

    def f8(shape, dt=torch.float8_e4m3fn):
        lim = 448.0 if dt == torch.float8_e4m3fn else 57344.0
        return (torch.randn(shape, device=dev, generator=gen) * 64).clamp(-lim, lim).to(dt)

    def unif(shape):
        return torch.rand(shape, device=dev, generator=gen) + 0.5

    def logu(shape):
        return torch.exp2(torch.rand(shape, device=dev, generator=gen) * 16 - 8)

    def timed(fn, copies):
        for c in copies[:2]:
            fn(*c, stream=stream)
        return graph_us(torch, lambda r, st: fn(*copies[r % len(copies)], stream=st), reps)

    def row(name, us, flops, byts):
        return {"problem": name, "us": round(us, 2), "tflops": round(flops / us / 1e6, 1),
                "gbs": round(byts / us / 1e3, 1), "frac_fp8_peak": round(flops / us / 1e6 / fp8_peak, 3),
                "frac_hbm_peak": round(byts / us / 1e3 / hbm_peak, 3)}

    out = {"contiguous": [], "masked": [], "large_dense": []}
    for (G, n, k) in wl.contiguous_shapes():
        M = G * wl.CONTIGUOUS_ROWS_PER_GROUP
        kb, nb = (k + 127) // 128, (n + 127) // 128
        byts = M * k + G * n * k + M * n * 2
        nc = max(2, -(-ROTATE_BYTES // byts))
        mi = torch.arange(G, device=dev, dtype=torch.int32).repeat_interleave(wl.CONTIGUOUS_ROWS_PER_GROUP)
        copies = [(f8((M, k)), unif((kb, M)), f8((G, n, k)), unif((G, nb, kb)),
                   torch.empty((M, n), dtype=torch.bfloat16, device=dev), mi) for _ in range(nc)]
        us = timed(fg.fg_grouped_gemm_fp8_contiguous, copies)
        out["contiguous"].append(row(f"G={G} M={M} n={n} k={k}", us, 2.0 * M * n * k, byts))
        del copies
    for (G, n, k) in wl.masked_shapes():
        Mc = wl.MASKED_M_CAP
        kb, nb = (k + 127) // 128, (n + 127) // 128
        rng = wl.rng_for(wl.seed_for(3, wl.masked_shapes().index((G, n, k))))
        counts = rng.integers(0, Mc, size=G, endpoint=True).astype(np.int32)
        valid, used = int(counts.sum()), int((counts > 0).sum())
        byts = valid * k + used * n * k + valid * n * 2
        full = G * Mc * k + G * n * k + G * Mc * n * 2
        nc = max(2, -(-ROTATE_BYTES // full))
        mm = torch.from_numpy(counts).to(dev)
        copies = [(f8((G, Mc, k)), unif((G, kb, Mc)), f8((G, n, k)), unif((G, nb, kb)),
                   torch.empty((G, Mc, n), dtype=torch.bfloat16, device=dev), mm) for _ in range(nc)]
        us = timed(fg.fg_grouped_gemm_fp8_masked, copies)
        r = row(f"G={G} M_cap={Mc} n={n} k={k} valid_rows={valid}", us, 2.0 * valid * n * k, byts)
        out["masked"].append(r)
        del copies
    for (m, n, k, bfmt) in wl.large_dense_shapes():
        kb, nb = (k + 127) // 128, (n + 127) // 128
        bdt = torch.float8_e4m3fn if bfmt == wl.E4M3 else torch.float8_e5m2
        byts = m * k + n * k + m * n * 2
        nc = max(2, -(-ROTATE_BYTES // byts))
        copies = [(f8((m, k)), logu((kb, m)), f8((n, k), bdt), logu((nb, kb)),
                   torch.empty((m, n), dtype=torch.bfloat16, device=dev)) for _ in range(nc)]
        us = timed(fg.fg_gemm_fp8_nt, copies)
        out["large_dense"].append(row(f"{m}x{n}x{k} B={'E5M2' if bfmt else 'E4M3'}", us, 2.0 * m * n * k, byts))
        del copies
    # K-grouped (the weight gradient of the contiguous workload): G segments of
    # 8192 tokens, and 32 short segments of 512 tokens; D [G][M][N] in BF16
    out["k_grouped"] = []
    for (G, M, N, tok) in wl.k_grouped_shapes() + wl.k_grouped_short_shapes():
        K = G * tok
        kb, nb = (K + 127) // 128, (N + 127) // 128
        byts = M * K + N * K + G * M * N * 2
        nc = max(2, -(-ROTATE_BYTES // byts))
        ks = torch.full((G,), tok, dtype=torch.int32, device=dev)
        copies = [(f8((M, K)), unif((kb, M)), f8((N, K)), unif((nb, kb)),
                   torch.empty((G, M, N), dtype=torch.bfloat16, device=dev), ks) for _ in range(nc)]
        us = timed(fg.fg_k_grouped_gemm_fp8_nt, copies)
        out["k_grouped"].append(row(f"G={G} M={M} N={N} K={K} ({tok} tokens per group)", us, 2.0 * M * N * K, byts))
        del copies
    st, det = fg.fg_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {det:#x} after the other workloads")
    out["timing"] = (f"{reps} launches per problem in a CUDA graph, replayed between CUDA events, rotating "
                     "copies >= 272 MiB, after the GEMM steps; masked GB/s and TFLOP/s count valid rows only")
    out["peak_source"] = peak_src
    return out


def run_reference(args, ws, rank):
    if rank != 0:
        return
    probs, shapes = sweep_problems()
    per_step = max(0.5, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample_rate(probs, shapes, per_step / 4)
    rates, times = [], []
    cores, sample = 0, ""
    for _ in range(args.steps):
        t0 = time.perf_counter()
        r, cores, sample = oracle_sample_rate(probs, shapes, per_step)
        times.append(time.perf_counter() - t0)
        rates.append(r)
    value = float(np.median(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(times)) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
        "data": "synthetic (seeded N(0,1), quantized to E4M3)",
        "config": bench_config(ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample + "; host cores, no GPU involved (L2 rotation does not apply)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, ws, rank, local):
    import torch

    import moe_grouped_gemm_nt_gb300 as fg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.shapes:
        # a subset (for profiling): only the problems asked for are generated
        shapes = [tuple(int(x) for x in s.split(",")) for s in args.shapes.split(";")]
        probs = {}
        for (m, n, k) in shapes:
            idx = wl.DENSE_SWEEP_NK.index((n, k)) if (n, k) in wl.DENSE_SWEEP_NK else 99
            if (n, k) not in probs or probs[(n, k)].m < m:
                probs[(n, k)] = wl.dense(m, n, k, seed=wl.seed_for(1, idx))
    else:
        probs, shapes = sweep_problems()

    # device copies (inputs resident in HBM before timing)
    dv = {}
    for (n, k), p in probs.items():
        A = torch.from_numpy(p.A).view(torch.float8_e4m3fn).to(dev)
        B = torch.from_numpy(p.B).view(torch.float8_e4m3fn).to(dev)
        sA_rm = torch.from_numpy(p.sA).to(dev)
        sB = torch.from_numpy(p.sB).to(dev)
        dv[(n, k)] = (A, sA_rm, B, sB)
    # Each problem rotates over identical copies of its inputs and output whose
    # total size is at least twice the L2 cache, so no launch finds its inputs
    # in L2; launches of one problem run back to back between one pair of
    # CUDA events (single-launch event intervals are too coarse for the
    # microsecond-scale small-m launches).
    items = []
    for (m, n, k) in shapes:
        A, sA_rm, B, sB = dv[(n, k)]
        sA = fg.fg_scales_a_to_mn_major(sA_rm[:m].contiguous())
        nbytes = problem_bytes(m, n, k)
        ncopy = max(2, -(-ROTATE_BYTES // nbytes))
        copies = [(A[:m].clone(), sA.clone(), B.clone(), sB.clone(),
                   torch.empty((m, n), dtype=torch.bfloat16, device=dev)) for _ in range(ncopy)]
        items.append((m, n, k, copies))
    del dv
    stream = torch.cuda.current_stream()

    def run_problem(i, reps, start=0):
        copies = items[i][3]
        for r in range(reps):
            A, sA, B, sB, D = copies[(start + r) % len(copies)]
            fg.fg_gemm_fp8_nt(A, sA, B, sB, D, stream=stream)

    for i in range(len(items)):  # warm-up: W passes over every problem
        run_problem(i, args.warmup * len(items[i][3]))
    torch.cuda.synchronize()
    st, det = fg.fg_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {det:#x} after warm-up")

    # A step launches every problem once.  The problems are ordered by the
    # kernel instantiation the library's plan picks, so that one event at each
    # group boundary gives every kernel's device time inside the timed region.
    groups = {}
    for i, (m, n, k, _) in enumerate(items):
        groups.setdefault(kernel_name(*plan_of(fg, m, n, k)), []).append(i)
    group_names = list(groups)
    group_items = [groups[g] for g in group_names]

    def one_step(s):
        for idxs in group_items:
            yield
            for i in idxs:
                copies = items[i][3]
                A, sA, B, sB, D = copies[s % len(copies)]
                fg.fg_gemm_fp8_nt(A, sA, B, sB, D, stream=stream)
        yield

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(group_items) + 1)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for s in range(args.steps):  # K steps, back to back
        for g, _ in enumerate(one_step(s)):
            ev[s][g].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    wall = time.perf_counter() - w0
    clock_info = clocks.stop() if rank == 0 else None
    st, det = fg.fg_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {det:#x} after the timed steps")

    total_ms = ev[0][0].elapsed_time(ev[-1][-1])
    kernel_ms = [sum(ev[s][g].elapsed_time(ev[s][g + 1]) for s in range(args.steps)) / args.steps
                 for g in range(len(group_items))]
    step_ms = max_over_ranks(total_ms / args.steps, ws)
    flops_step = sum(2.0 * m * n * k for (m, n, k, *_) in items)
    bytes_step = sum(problem_bytes(m, n, k) for (m, n, k, *_) in items)
    value = ws * flops_step / (step_ms * 1e-3) / 1e12

    # Per-problem times, for the table and for the bandwidth-bound summary:
    # measured after the timed steps, each problem launched K times back to back.
    per_shape_ms = np.zeros(len(items))
    for i in range(len(items)):
        cps = items[i][3]
        per_shape_ms[i] = graph_us(torch, lambda r, st: fg.fg_gemm_fp8_nt(*cps[r % len(cps)], stream=st),
                                   args.steps) * 1e-3

    # FP32-output calls on the tensor-bound problems (m = 4096): same inputs and
    # copies, an FP32 D per copy, K launches back to back per problem
    f32out = None
    if not args.no_f32out:
        f32_rows, f_tot, t_tot = [], 0.0, 0.0
        for i, (m, n, k, copies) in enumerate(items):
            if m != max(wl.DENSE_SWEEP_M):
                continue
            d32 = [torch.empty((m, n), dtype=torch.float32, device=dev) for _ in copies]
            for r in range(len(copies)):  # warm-up
                A, sA, B, sB, _ = copies[r]
                fg.fg_gemm_fp8_nt_f32out(A, sA, B, sB, d32[r], stream=stream)
            torch.cuda.synchronize()

            def f32_launch(r, st, copies=copies, d32=d32):
                A, sA, B, sB, _ = copies[r % len(copies)]
                fg.fg_gemm_fp8_nt_f32out(A, sA, B, sB, d32[r % len(copies)], stream=st)

            us = graph_us(torch, f32_launch, args.steps)
            f = 2.0 * m * n * k
            f32_rows.append({"m": m, "n": n, "k": k, "us": round(us, 2), "tflops": round(f / us / 1e6, 1),
                             "time_vs_bf16_out": round(us / (per_shape_ms[i] * 1e3), 3)})
            f_tot += f
            t_tot += us
            del d32
        st, det = fg.fg_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} detail {det:#x} after the FP32-output runs")
        f32out = {"call": "fg_gemm_fp8_nt_f32out", "tflops_over_shapes": round(f_tot / t_tot / 1e6, 1),
                  "timing": "K launches per problem in a CUDA graph, replayed between events; same copies",
                  "shapes": f32_rows}

    peaks, peak_src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    hbm_peak = peaks["hbm_gbs"]
    shape_rows = []
    med = per_shape_ms
    for i, (m, n, k, *_) in enumerate(items):
        t = med[i] * 1e-3
        f, b = 2.0 * m * n * k, problem_bytes(m, n, k)
        t_roof = max(f / (fp8_peak * 1e12), b / (hbm_peak * 1e9))
        shape_rows.append({"m": m, "n": n, "k": k, "us": round(med[i] * 1e3, 2),
                           "tflops": round(f / t / 1e12, 1), "gbs": round(b / t / 1e9, 1),
                           "frac_fp8_peak": round(f / t / 1e12 / fp8_peak, 3),
                           "frac_hbm_peak": round(b / t / 1e9 / hbm_peak, 3),
                           "roofline_over_time": round(t_roof / t, 3)})
    for r in shape_rows:
        pl = plan_of(fg, r["m"], r["n"], r["k"])
        r["plan"] = {"block_n": pl[0], "split_k": pl[1], "cta_pair": pl[2], "swap_ab": pl[3], "deferred_stores": pl[4]}
        r["kernel"] = kernel_name(*pl)
    traffic_tab = load_traffic()
    ridge = fp8_peak * 1e12 / (hbm_peak * 1e9)

    def roof(g):
        name, idxs = group_names[g], group_items[g]
        rows = [shape_rows[i] for i in idxs]
        tt = kernel_ms[g] * 1e-3  # this kernel's device time per step, from the timed steps
        flops = sum(2.0 * r["m"] * r["n"] * r["k"] for r in rows)
        byts = sum(problem_bytes(r["m"], r["n"], r["k"]) for r in rows)
        known = [traffic_tab.get((r["m"], r["n"], r["k"])) for r in rows]
        traffic = (sum(known) / len(known)) if known and all(v is not None for v in known) else None
        common = {"kernel": name, "launch_shapes": [(r["m"], r["n"], r["k"]) for r in rows],
                  "launches_per_step": len(rows), "us_per_step": round(kernel_ms[g] * 1e3, 2),
                  "algorithmic_bytes_per_launch": byts / len(rows)}
        if flops / byts >= ridge:
            ach = flops / tt / 1e12
            return {"bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                    "frac": round(ach / fp8_peak, 3), "traffic": traffic, **common,
                    "peak_source": f"{peak_src}: bf16 burst {peaks['bf16_tflops']} x {FP8_PER_BF16} "
                                   "(nominal FP8/BF16 ratio)"}
        ach = byts / tt / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(ach / hbm_peak, 3), "traffic": traffic, **common,
                "peak_source": f"{peak_src}: hbm copy"}

    by_time = sorted(range(len(group_items)), key=lambda g: -kernel_ms[g])
    roofline = roof(by_time[0])
    others = [roof(g) for g in by_time[1:]]
    hbm_rows = [r for r in shape_rows if 2.0 * r["m"] * r["n"] * r["k"] / problem_bytes(r["m"], r["n"], r["k"]) < ridge]
    roofline_hbm = None
    if hbm_rows:
        tt = sum(r["us"] for r in hbm_rows) * 1e-6
        ach = sum(problem_bytes(r["m"], r["n"], r["k"]) for r in hbm_rows) / tt / 1e9
        roofline_hbm = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                        "frac": round(ach / hbm_peak, 3), "shapes": "all bandwidth-bound problems of the step",
                        "timing": "per-problem CUDA-graph replays after the timed steps",
                        "peak_source": f"{peak_src}: hbm copy"}

    others_cfg = None
    if not args.no_other_configs:
        others_cfg = measure_other_configs(fg, torch, dev, stream, fp8_peak, hbm_peak, peak_src)

    quant = None
    if not args.no_quantize:
        quant = measure_quantize(fg, torch, dev, stream, hbm_peak, peak_src, traffic_tab=traffic_tab)
        quant["f32_input"] = measure_quantize(fg, torch, dev, stream, hbm_peak, peak_src, f32_input=True)

    # ------------------------------------------------ end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        # Each problem's inputs (A, row-major sA, B, sB) packed into one pinned
        # host buffer and one device buffer at 256-byte aligned offsets, so a
        # step copies each problem's inputs with one host->device copy (the
        # fixed cost of a copy is paid once per problem, not once per tensor).
        def packed(parts):
            offs, off = [], 0
            for a in parts:
                offs.append(off)
                off += -(-a.nbytes // 256) * 256
            hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
            hv = hbuf.numpy()
            for a, o in zip(parts, offs):
                hv[o:o + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
            dbuf = torch.empty(off, dtype=torch.uint8, device=dev)
            views = [dbuf[o:o + a.nbytes].view(torch.float32 if a.dtype == np.float32 else torch.uint8).view(a.shape)
                     for a, o in zip(parts, offs)]
            return hbuf, dbuf, views

        host = []
        for (m, n, k, copies) in items:
            A, sA, B, sB, D = copies[0]
            p = probs[(n, k)]
            hbuf, dbuf, (dA, dsA_rm, dB, dsB) = packed([p.A[:m], p.sA[:m], p.B, p.sB])
            hD = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
            dsA = torch.empty(sA.shape, dtype=torch.float32, device=dev)
            host.append((m, n, k, hbuf, dbuf, hD, dA, dsA_rm, dsA, dB, dsB, D))
        h2d = sum(h[3].numel() for h in host)
        d2h = sum(h[5].numel() * 2 for h in host)

        # Three streams: host->device copies, compute, device->host copies.  The
        # copies of problem i+1 and the read-back of problem i overlap the GEMM
        # of problem i; a step's copies into a problem's buffers wait for the
        # previous step's GEMM of that problem, and its GEMM for the previous
        # read-back of its output.  (A second host->device stream measured no
        # faster: the copies already run at the link's rate.)
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in host]
        ev_gemm = [torch.cuda.Event() for _ in host]
        ev_out = [torch.cuda.Event() for _ in host]

        def e2e_step():
            for i, (m, n, k, hbuf, dbuf, hD, dA, dsA_rm, dsA, dB, dsB, D) in enumerate(host):
                with torch.cuda.stream(s_in):
                    s_in.wait_event(ev_gemm[i])
                    dbuf.copy_(hbuf, non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                stream.wait_event(ev_out[i])
                fg.fg_scales_a_to_mn_major(dsA_rm, dsA, stream=stream)
                fg.fg_gemm_fp8_nt(dA, dsA, dB, dsB, D, a_fmt=0, b_fmt=0, stream=stream)
                ev_gemm[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_gemm[i])
                    hD.copy_(D, non_blocking=True)
                    ev_out[i].record(s_out)

        for _ in range(max(1, min(args.warmup, 3))):
            e2e_step()
        torch.cuda.synchronize()
        k_e2e = max(1, min(args.steps, 50))
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for _ in range(k_e2e):
            e2e_step()
        stream.wait_event(ev_out[-1])  # the last read-back of the last step
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / k_e2e, ws)
        e2e = {"value": round(ws * flops_step / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 3),
               "steps": k_e2e,
               "streams": ("h2d copies (one per problem: its inputs packed in one pinned buffer), compute, d2h copies; "
                           "pipelined across the step's problems")}
        # the values read back are the GEMMs' outputs
        for (m, n, k, hbuf, dbuf, hD, dA, dsA_rm, dsA, dB, dsB, D) in host[:: max(1, len(host) // 4)]:
            if not torch.equal(hD.view(torch.int16), D.cpu().view(torch.int16)):
                raise RuntimeError(f"end-to-end read-back of {m}x{n}x{k} differs from the device result")
        st, det = fg.fg_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} after the end-to-end steps")

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, cores, sample = oracle_sample_rate(probs, shapes, seconds=args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
            "data": "synthetic (seeded N(0,1), quantized to E4M3 per 1x128 / 128x128 group)",
            "config": dict(bench_config(ws), problems_per_step=len(items)),
            "hbm_gbs": round(ws * bytes_step / (step_ms * 1e-3) / 1e9, 1),
            "wall_ms_per_step": round(wall / args.steps * 1e3, 3),
            "roofline": roofline, "roofline_other_kernels": others, "roofline_hbm": roofline_hbm,
            "shapes": shape_rows, "clocks": clock_info, "e2e": e2e,
            "gpu_launches": len(items) * args.steps, "cpu_baseline": cpu,
            "quantize_per_token": quant, "f32_output": f32out, "other_workloads": others_cfg,
        }
        print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--shapes", default="", help="restrict to 'm,n,k;m,n,k' (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quantize", action="store_true", help="skip the activation-quantization figures")
    ap.add_argument("--no-f32out", action="store_true", help="skip the FP32-output figures")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the contiguous, masked and large-square throughput figures")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours" and not args.shapes:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
