#!/usr/bin/env python
"""Benchmark of the block-scaled MoE GEMM hot path on GB300.

Headline workload (one step = one pass of the hot path over one batch):
  dense NVFP4 W4A4 GEMM, M=4096 N=12288 K=5120: quantise A (BF16 -> NVFP4 with
  its per-tensor global scale), quantise B (same), block-scaled GEMM with
  alpha = 1/(g_A g_B), BF16 out.  value = 2 M N K / step time, in TFLOP/s.
  Inputs are resident in HBM; L2 is flushed (256 MiB written, then another
  256 MiB read, so no dirty lines remain) before every timed step, outside the
  timed interval.

Extra keys report, on one GPU, each kernel of the other workloads (dense MXFP8
256^3 latency, grouped-contiguous MXFP8 + SwiGLU requant, grouped-masked NVFP4,
BF16 grouped GEMM + dSwiGLU, and the quantiser's GB/s) against its roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hq|reference]

--impl reference times the CPU oracle (the only other implementation of this
path) on a bounded sample of the same workload.  Under torchrun each rank runs
an independent replica (the path has no exchange step); the time is the
maximum over ranks and value sums the work of all ranks.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense tensor-core ratios to BF16 (2.25 PFLOP/s): FP8 x2, FP4 x6
RATIO = {"bf16": 1.0, "fp8": 2.0, "fp4": 6.0}
GEMM_EVENT_EVERY = 8  # timed steps per sampled GEMM duration in the headline loop
SECTIONS = ("dense_mxfp8_256", "quant_nvfp4", "moe_contig", "moe_masked", "dswiglu", "dense_mxfp4",
            "permute", "mma_rate", "host_link")


GEMM_PROFILE = os.path.join(ROOT, "profiles", "bs_gemm_2sm_kernel_dense_nvfp4_4096x12288x5120.md")
GEMM_SOURCES = ("hq_gemm_bs.cu", "hq_ptx.cuh", "hq_sched.cuh", "hq_internal.h")


def profiled_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, or None when
    the kernel's sources changed after the counters were taken."""
    import hashlib
    import re
    if not os.path.exists(GEMM_PROFILE):
        return None
    text = open(GEMM_PROFILE).read()
    mb = re.search(r"dram_bytes_per_launch \| (\d+)", text)
    mh = re.search(r"source_sha256_16: ([0-9a-f]{16})", text)
    if not (mb and mh):
        return None
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "fp4_grouped_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return int(mb.group(1)) if h.hexdigest()[:16] == mh.group(1) else None


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK, "fallback"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="hq", choices=["hq", "reference"])
    p.add_argument("--main-only", action="store_true", help="skip the per-workload extras")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", choices=list(SECTIONS), default=None,
                   help="run only one per-workload section (for profiling) and print its numbers")
    return p.parse_args()


# --------------------------------------------------------------------------- distributed


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "hq" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- clocks


class Clocks:
    """nvidia-smi sampling (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return []
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [s.strip() for s in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- helpers


class L2Flush:
    """Evicts L2 before a timed launch: writes one 256 MiB buffer, then reads
    another, so the timed kernel starts with a cold cache holding only clean
    lines (no write-backs of the flush itself land inside the timed region)."""

    def __init__(self, device, mib=256):
        n = mib * (1 << 20) // 4
        self.buf = torch.empty(n, dtype=torch.int32, device=device)
        self.buf2 = torch.ones(n, dtype=torch.int32, device=device)
        self.sink = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        self.buf.add_(1)
        torch.sum(self.buf2, dim=0, out=self.sink)


def time_kernel(fn, iters, flush=None, warmup=3):
    """Average device time (s) of fn() over iters launches, L2 flushed before each."""
    for _ in range(warmup):
        fn()
    st = torch.cuda.current_stream()
    evs = []
    for _ in range(iters):
        if flush:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        evs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / iters / 1e3


def oracle_cpu_baseline(budget_s=10.0, ms=64, ns=512):
    """The CPU oracle on a bounded sample of the headline workload."""
    from oracle import gemm as ogemm, quant as oquant
    gen = torch.Generator().manual_seed(2)
    k = 5120
    a = torch.randn(ms, k, generator=gen).to(torch.bfloat16).float().numpy()
    b = (torch.randn(ns, k, generator=gen) * 0.02).to(torch.bfloat16).float().numpy()
    flops, t0, reps = 0.0, time.time(), 0
    while True:
        qa, sa = oquant.quantize(a, "nvfp4", 37.0)
        qb, sb = oquant.quantize(b, "nvfp4", 1.0e4)
        ogemm.dense(oquant.dequantize(qa, sa, "nvfp4"), oquant.dequantize(qb, sb, "nvfp4"), alpha=[1e-6])
        flops += 2.0 * ms * ns * k
        reps += 1
        if time.time() - t0 >= budget_s:
            break
    dt = time.time() - t0
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        threads = len(os.sched_getaffinity(0))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": int(threads), "kind": "oracle",
            "sample": f"{reps} x (quantise A[{ms},{k}] and B[{ns},{k}] to NVFP4, dequantise, "
                      f"float64 GEMM) in {dt:.1f} s, from the {4096}x{12288}x{5120} workload"}


def _oracle_quant_chunk(job):
    """One process's share of the all-cores quantiser baseline: quantise a
    seeded [rows, k] BF16-valued block `reps` times; returns elapsed seconds."""
    rows, k, seed, mode, reps = job
    from oracle import quant as oquant
    x = torch.randn(rows, k, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16).float().numpy()
    t0 = time.time()
    for _ in range(reps):
        oquant.quantize(x, mode, 37.0 if mode == "nvfp4" else None)
    return time.time() - t0


def oracle_kernel_baselines(budget_s=2.0):
    """The CPU oracle per kernel of the path, each on a bounded sample:
    the quantiser single-threaded and on all cores (a process pool), and each
    GEMM workload's dequantise-then-float64 GEMM on all cores (numpy's BLAS
    threads).  Values in the unit of the matching GPU line."""
    import multiprocessing as mp
    from oracle import gemm as ogemm, glu, quant as oquant
    cores = len(os.sched_getaffinity(0))
    res = {}
    # quantiser, NVFP4 rows of the headline A (k = 5120), single thread
    rows, k = 64, 5120
    x = torch.randn(rows, k, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).float().numpy()
    n_rep, t0 = 0, time.time()
    while time.time() - t0 < budget_s:
        oquant.quantize(x, "nvfp4", 37.0)
        n_rep += 1
    dt = time.time() - t0
    byts = rows * k * 2 + rows * k // 2 + rows * k // 16
    res["quant_nvfp4_single_thread"] = {"gbs": n_rep * byts / dt / 1e9, "cores": 1,
                                        "sample": f"{n_rep} x [{rows},{k}] in {dt:.1f} s"}
    # the same on all cores: one process per core, each its own rows
    reps = max(1, int(n_rep / dt * budget_s / 2))
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pool.map(_oracle_quant_chunk, [(8, k, i, "nvfp4", 1) for i in range(cores)])  # start-up
        t0 = time.time()
        pool.map(_oracle_quant_chunk, [(rows, k, i, "nvfp4", reps) for i in range(cores)])
        dt = time.time() - t0
    res["quant_nvfp4_all_cores"] = {"gbs": cores * reps * byts / dt / 1e9, "cores": cores,
                                    "sample": f"{cores} processes x {reps} x [{rows},{k}] in {dt:.1f} s"}

    def gemm(name, m, n, k, mode, std_b):
        a = torch.randn(m, k, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).float().numpy()
        b = (torch.randn(n, k, generator=torch.Generator().manual_seed(4)) * std_b).to(torch.bfloat16).float().numpy()
        if mode == "bf16":
            ad, bd = a.astype(np.float64), b.astype(np.float64)
        else:
            g = 37.0 if mode == "nvfp4" else None
            ad = oquant.dequantize(*oquant.quantize(a, mode, g), mode)
            bd = oquant.dequantize(*oquant.quantize(b, mode, g), mode)
        reps, t0 = 0, time.time()
        while time.time() - t0 < budget_s:
            if mode == "bf16":   # the dSwiGLU backward: R, then the closed form on C
                R, _, _ = glu.grouped_R(ad, bd[None], [m], [1.0])
                c = np.ones((m, 2 * n))
                glu.dswiglu_epilogue(R, c, np.ones(m), np.ones(m))
            else:
                ogemm.dense(ad, bd)
            reps += 1
        dt = time.time() - t0
        res[name] = {"tflops": reps * 2.0 * m * n * k / dt / 1e12, "cores": cores,
                     "sample": f"{reps} x [{m}x{n}x{k}] ({mode} operands dequantised, float64) in {dt:.1f} s"}
    gemm("dense_nvfp4_gemm", 64, 512, 5120, "nvfp4", 0.02)
    gemm("moe_contig_mxfp8_gemm", 64, 512, 4096, "mxfp8", 0.02)
    gemm("moe_masked_nvfp4_gemm", 64, 512, 7168, "nvfp4", 0.02)
    gemm("dswiglu_bwd_bf16_gemm", 64, 256, 2048, "bf16", 0.02)
    return res


# --------------------------------------------------------------------------- reference arm


def run_reference(args, ws, rank):
    if rank != 0:
        return
    cfg_name = "dense_nvfp4_4096x12288x5120"
    for _ in range(max(args.warmup, 0)):
        oracle_cpu_baseline(budget_s=0.0, ms=16, ns=256)
    vals = []
    for _ in range(args.steps):
        r = oracle_cpu_baseline(budget_s=0.0, ms=16, ns=256)
        vals.append(r["value"])
    base = dict(r) if args.steps else oracle_cpu_baseline(budget_s=0.0, ms=16, ns=256)
    v = statistics.median(vals) if vals else base["value"]
    base["value"] = v
    base["sample"] = f"per step: {base['sample']}"
    line = {"metric": "block-scaled GEMM TFLOP/s (hot-path step: quantise A and B, GEMM)",
            "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": {"workload": cfg_name, "sample": base["sample"]},
            "cpu_baseline": base,
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- workloads


def headline(hq, dev, args, ws, peaks, pk_src):
    cfg = synth.dense_nvfp4(device=dev)
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    flops = 2.0 * m * n * k
    ga = torch.tensor([cfg["g_a"]], dtype=torch.float32, device=dev)
    gb = torch.tensor([cfg["g_b"]], dtype=torch.float32, device=dev)
    alpha = torch.tensor([cfg["alpha"]], dtype=torch.float32, device=dev)
    qa = torch.empty(m, k // 2, dtype=torch.uint8, device=dev)
    qb = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
    sfa = torch.empty(hq.sf_bytes(m, k, "nvfp4"), dtype=torch.uint8, device=dev)
    sfb = torch.empty(hq.sf_bytes(n, k, "nvfp4"), dtype=torch.uint8, device=dev)
    out = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
    a, b = cfg["a"], cfg["b"]
    st = torch.cuda.current_stream()

    # A and B are quantised concurrently (B on a side stream): the small A
    # launch's ramp and tail overlap B's
    side = torch.cuda.Stream(device=dev)

    def step(gemm_events=None):
        side.wait_stream(st)
        with torch.cuda.stream(side):
            hq.hq_quant(b, "nvfp4", global_scale=gb, q_out=qb, sf_out=sfb)
        hq.hq_quant(a, "nvfp4", global_scale=ga, q_out=qa, sf_out=sfa)
        st.wait_stream(side)
        if gemm_events:
            gemm_events[0].record(st)
        hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "nvfp4", alpha=alpha, out=out)
        if gemm_events:
            gemm_events[1].record(st)

    flush = L2Flush(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    # the GEMM's own events go into every GEMM_EVENT_EVERY-th timed step only:
    # an event recorded between the cross-stream wait and the GEMM launch adds
    # about 4 us to the step it sits in
    steps, gemms = [], []
    for i in range(args.steps):
        flush()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g = None
        if i % GEMM_EVENT_EVERY == 0:
            g = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            gemms.append(g)
        s0.record(st)
        step(g)
        s1.record(st)
        steps.append((s0, s1))
    torch.cuda.synchronize()
    barrier(ws)
    rows = clocks.stop()
    if len(rows) < 3:  # timed region shorter than the sampling period: continue the same step
        clocks.start()
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
        rows += clocks.stop()
    total = sum(a.elapsed_time(b) for a, b in steps) / 1e3
    gemm_avg = sum(a.elapsed_time(b) for a, b in gemms) / len(gemms) / 1e3
    total_max = max_over_ranks(total, ws, dev)
    value = ws * args.steps * flops / total_max / 1e12
    peak_fp4 = peaks["bf16_tflops"] * RATIO["fp4"]
    achieved = flops / gemm_avg / 1e12
    # the tensor pipe's own FP4 rate, measured here after the timed region
    # (the library's issue-rate probe: back-to-back kind::mxf4nvf4 MMAs of
    # M = 256, N = 256 on CTA pairs), at the SM clock sampled while timing
    clk = Clocks.summarize(rows)
    mma = hq.probe_mma_rate("nvfp4", pair=True)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    bench_mhz = clk["sm_mhz"] or mma["sm_mhz"]
    peak_mma = mma["flop_per_clk_sm"] * sms * bench_mhz * 1e6 / 1e12

    # end to end through the public API from pinned host buffers, as a
    # serving loop runs it: every step copies its own A and B from the host,
    # quantises them, runs the GEMM and copies its result back; uploads,
    # compute and the download run on three streams with double-buffered
    # device inputs and outputs, so step i's download overlaps step i + 1's
    # uploads (the host link is full duplex) and A's quantisation overlaps
    # B's upload.  Reported: steady-state time per step.
    a_h = a.cpu().pin_memory()
    b_h = b.cpu().pin_memory()
    out_h = torch.empty(m, n, dtype=torch.bfloat16).pin_memory()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    a_d = [torch.empty_like(a) for _ in range(2)]
    b_d = [torch.empty_like(b) for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    quant_done, down_done = [None, None], [None, None]

    def e2e_step(i):
        j = i % 2
        ea, eb, eg = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.stream(up):
            if quant_done[j] is not None:
                up.wait_event(quant_done[j])        # step i - 2 has read these buffers
            a_d[j].copy_(a_h, non_blocking=True)
            ea.record(up)
            b_d[j].copy_(b_h, non_blocking=True)
            eb.record(up)
        st.wait_event(ea)
        hq.hq_quant(a_d[j], "nvfp4", global_scale=ga, q_out=qa, sf_out=sfa)
        st.wait_event(eb)
        hq.hq_quant(b_d[j], "nvfp4", global_scale=gb, q_out=qb, sf_out=sfb)
        quant_done[j] = torch.cuda.Event()
        quant_done[j].record(st)
        if down_done[j] is not None:
            st.wait_event(down_done[j])              # step i - 2's result has left
        hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "nvfp4", alpha=alpha, out=outs[j])
        eg.record(st)
        with torch.cuda.stream(down):
            down.wait_event(eg)
            out_h.copy_(outs[j], non_blocking=True)
            down_done[j] = torch.cuda.Event()
            down_done[j].record(down)

    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(up)
    for i in range(2, 2 + e2e_steps):
        e2e_step(i)
    t1.record(down)
    torch.cuda.synchronize()
    e2e_t = t0.elapsed_time(t1) / e2e_steps / 1e3
    e2e_t = max_over_ranks(e2e_t, ws, dev)
    h2d = (a.numel() + b.numel()) * 2
    d2h = out.numel() * 2
    return {
        "value": value, "ms_per_step": total_max / args.steps * 1e3,
        "config": {"workload": cfg["name"], "M": m, "N": n, "K": k, "mode": "nvfp4",
                   "step": "hq_quant(A) || hq_quant(B) on two streams, then hq_gemm_dense",
                   "l2": "flushed before every timed step (256 MiB written, then 256 MiB read)",
                   "gemm_timing": f"CUDA events around the GEMM in every {GEMM_EVENT_EVERY}th timed step "
                                  f"({len(gemms)} of {args.steps})",
                   "inputs": "A ~ N(0,1), B ~ N(0,0.02) BF16, seeded; g = 2688/amax per tensor",
                   "e2e": "per step: upload A and B from pinned host memory, quantise, GEMM, download the "
                          "result; uploads / compute / download on three streams, steady-state time per "
                          "step (step i's download overlaps step i + 1's uploads)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_fp4, "unit": "TFLOP/s",
                     "frac": achieved / peak_fp4, "traffic": profiled_traffic(),
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "kernel": "bs_gemm_2sm_kernel<NVFP4,4,GEMM,384> (cluster pair, 256x384 tiles)",
                     "peak_source": f"{pk_src} bf16 burst {peaks['bf16_tflops']} x 6 (nominal FP4/BF16)",
                     "frac_measured_mma": achieved / peak_mma, "peak_measured_mma": peak_mma,
                     "measured_mma": {"kind": "mxf4nvf4.block_scale.scale_vec::4X, cta_group::2, 256x256x64",
                                      "cycles_per_mma": mma["cycles_per_mma"],
                                      "flop_per_clk_sm": mma["flop_per_clk_sm"], "sms": sms,
                                      "sm_mhz": bench_mhz,
                                      "note": "peak = FLOP/clk/SM x SMs x median SM clock of the timed region"}},
        "e2e": {"value": ws * flops / e2e_t / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "gemm_ms": gemm_avg * 1e3,
    }


class Extras:
    """Kernel-level numbers for the other workloads (one GPU), one method each."""

    NAMES = SECTIONS

    def __init__(self, hq, dev, peaks):
        self.hq, self.dev = hq, dev
        self.flush = L2Flush(dev)
        self.hbm = peaks["hbm_gbs"]
        self.p_fp8 = peaks["bf16_tflops"] * RATIO["fp8"]
        self.p_fp4 = peaks["bf16_tflops"] * RATIO["fp4"]
        self.p_bf16 = peaks["bf16_tflops"]

    def run(self, names):
        res = {}
        for name in names:
            res.update(getattr(self, name)())
            torch.cuda.empty_cache()
        return res

    def dense_mxfp8_256(self):
        hq, dev = self.hq, self.dev
        c1 = synth.dense_small(device=dev)
        qa, sfa = hq.hq_quant(c1["a"], "mxfp8")
        qb, sfb = hq.hq_quant(c1["b"], "mxfp8")
        out1 = torch.empty(256, 256, dtype=torch.bfloat16, device=dev)
        t = time_kernel(lambda: hq.hq_gemm_dense(qa, sfa, qb, sfb, 256, 256, 256, "mxfp8", out=out1), 200)
        calls = 1000  # back-to-back calls captured in one graph
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(calls):
                hq.hq_gemm_dense(qa, sfa, qb, sfb, 256, 256, 256, "mxfp8", out=out1)
        g.replay()
        torch.cuda.synchronize()
        tg = time_kernel(lambda: g.replay(), 10) / calls
        # the same graph with programmatic dependent launch: each call's
        # prologue (barriers, TMEM, tensor-map prefetch) overlaps the previous
        # call's tail, its first read waits for that call to finish
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp):
            for _ in range(calls):
                hq.hq_gemm_dense(qa, sfa, qb, sfb, 256, 256, 256, "mxfp8", out=out1, use_pdl=True)
        gp.replay()
        torch.cuda.synchronize()
        tgp = time_kernel(lambda: gp.replay(), 10) / calls
        return {"dense_mxfp8_256": {"us_per_call": t * 1e6, "us_per_call_graph": tg * 1e6,
                                    "us_per_call_graph_pdl": tgp * 1e6, "graph_calls": calls,
                                    "tflops": 2 * 256 ** 3 / t / 1e12}}

    def quant_nvfp4(self):
        hq, dev = self.hq, self.dev
        res = {}
        c2 = synth.dense_nvfp4(device=dev)
        for name, x in (("A", c2["a"]), ("B", c2["b"])):
            m, k = x.shape
            q = torch.empty(m, k // 2, dtype=torch.uint8, device=dev)
            sf = torch.empty(hq.sf_bytes(m, k, "nvfp4"), dtype=torch.uint8, device=dev)
            gsc = torch.tensor([1.0], device=dev)
            t = time_kernel(lambda: hq.hq_quant(x, "nvfp4", global_scale=gsc, q_out=q, sf_out=sf), 20, self.flush)
            byts = 2 * m * k + m * k // 2 + sf.numel()
            # the floor this launch size allows under the same timing: a plain
            # streaming pass over the same input with the same output ratio
            t_floor = time_kernel(lambda: hq.probe_stream(x, q), 20, self.flush)
            res[f"quant_nvfp4_{name}_{m}x{k}"] = {"us": t * 1e6, "gbs": byts / t / 1e9,
                                                  "frac_hbm": byts / t / 1e9 / self.hbm,
                                                  "stream_floor_us": t_floor * 1e6,
                                                  "frac_of_stream_floor": t_floor / t}
        res["empty_launch_us"] = time_kernel(lambda: hq.probe_stream(None, None), 20, self.flush) * 1e6
        return res

    def dense_mxfp4(self):
        """MXFP4 (w4a4-mxfp4, UE8M0 per 32, no alpha) on the headline shapes, and
        its quantiser from a float16 copy of A."""
        hq, dev = self.hq, self.dev
        c2 = synth.dense_nvfp4(device=dev)
        m, n, k = c2["m"], c2["n"], c2["k"]
        qa, sfa = hq.hq_quant(c2["a"], "mxfp4")
        qb, sfb = hq.hq_quant(c2["b"], "mxfp4")
        out = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        t = time_kernel(lambda: hq.hq_gemm_dense(qa, sfa, qb, sfb, m, n, k, "mxfp4", out=out), 20, self.flush)
        fl = 2.0 * m * n * k
        res = {"dense_mxfp4_4096x12288x5120": {"us": t * 1e6, "tflops": fl / t / 1e12,
                                                "frac_fp4": fl / t / 1e12 / self.p_fp4}}
        a16 = c2["a"].to(torch.float16)
        t = time_kernel(lambda: hq.hq_quant(a16, "mxfp4", q_out=qa, sf_out=sfa), 20, self.flush)
        byts = 2 * m * k + m * k // 2 + sfa.numel()
        res["quant_mxfp4_A_fp16_4096x5120"] = {"us": t * 1e6, "gbs": byts / t / 1e9,
                                               "frac_hbm": byts / t / 1e9 / self.hbm}
        return res

    def permute(self):
        """Routing permute of 8192 FP8 tokens (hidden 7168, top-8 of 32 experts,
        uniform routing, per-32 scales in direct mode) into the masked layout."""
        hq, dev = self.hq, self.dev
        T, hidden, topk, E = 8192, 7168, 8, 32
        cap = 4096                                   # twice the mean load per expert
        g = torch.Generator(device=dev).manual_seed(6)
        x = torch.randint(0, 256, (T, hidden), generator=g, device=dev, dtype=torch.uint8)
        sc = torch.randint(0, 256, (T, hidden // 32), generator=g, device=dev, dtype=torch.uint8)
        ids = torch.argsort(torch.rand(T, E, generator=g, device=dev), dim=1)[:, :topk].contiguous()
        xf = x.view(torch.float8_e4m3fn)
        px = torch.empty(E * cap, hidden, dtype=torch.float8_e4m3fn, device=dev)
        osf = torch.empty(E * cap * hidden // 32, dtype=torch.uint8, device=dev)
        imap = torch.empty(T, topk, dtype=torch.int32, device=dev)
        tn = torch.empty(E, dtype=torch.int32, device=dev)
        ws = torch.empty(hq.hq_prefill_permute_workspace_size(T, E), dtype=torch.uint8, device=dev)
        fn = lambda: hq.hq_prefill_permute(xf, sc, ids, E, cap, permute_x=px, out_scale=osf,  # noqa: E731
                                           indice_map=imap, token_nums=tn, workspace=ws)
        t = time_kernel(fn, 20, self.flush)
        # algorithmic bytes: each token's row and scales read once, written
        # once per routed slot; ids read, map written
        byts = T * (hidden + hidden // 32) + T * topk * (hidden + hidden // 32) + T * topk * (8 + 4)
        return {"permute_fp8_T8192_top8_E32_h7168": {"us": t * 1e6, "gbs": byts / t / 1e9,
                                                     "frac_hbm": byts / t / 1e9 / self.hbm}}

    def moe_contig(self):
        hq, dev = self.hq, self.dev
        res = {}
        c3 = synth.moe_contig(device=dev)
        M, n, k, L = c3["m"], c3["n"], c3["k"], c3["L"]
        qa, sfa = hq.hq_quant(c3["a"], "mxfp8")
        qb, sfb = hq.hq_quant(c3["b"].view(L * n, k), "mxfp8")
        t = time_kernel(lambda: hq.hq_quant(c3["a"], "mxfp8", q_out=qa, sf_out=sfa), 10, self.flush)
        byts = 3 * M * k + sfa.numel()
        res["quant_mxfp8_A_17408x4096"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_hbm": byts / t / 1e9 / self.hbm}
        bw = c3["b"].view(L * n, k)
        t = time_kernel(lambda: hq.hq_quant(bw, "mxfp8", q_out=qb, sf_out=sfb), 10, self.flush)
        byts = 3 * L * n * k + sfb.numel()
        res["quant_mxfp8_W_24576x4096"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_hbm": byts / t / 1e9 / self.hbm}
        off = torch.from_numpy(c3["padded_offsets"]).to(dev)
        out3 = torch.empty(M, n, dtype=torch.bfloat16, device=dev)
        qbv = qb.view(L, n, k)
        t = time_kernel(lambda: hq.hq_gemm_grouped_contig(qa, sfa, qbv, sfb, off, M, n, k, "mxfp8", out=out3),
                        20, self.flush)
        fl = 2.0 * M * n * k
        res["moe_contig_mxfp8_L8"] = {"us": t * 1e6, "tflops": fl / t / 1e12, "frac_fp8": fl / t / 1e12 / self.p_fp8,
                                     "tflops_routed_rows": 2.0 * 16384 * n * k / t / 1e12}
        H = n // 2
        qs = torch.empty(M, H, dtype=torch.uint8, device=dev)
        sfs = torch.empty(M * hq.swiglu_kb_dim(H, "mxfp8"), dtype=torch.uint8, device=dev)
        t = time_kernel(lambda: hq.hq_swiglu_quant(out3, "mxfp8", q_out=qs, sf_out=sfs), 20, self.flush)
        byts = M * n * 2 + M * H + sfs.numel()
        t_floor = time_kernel(lambda: hq.probe_stream(out3, qs), 20, self.flush)  # same bytes, plain stream
        res["swiglu_quant_mxfp8_17408x3072"] = {"us": t * 1e6, "gbs": byts / t / 1e9,
                                                "frac_hbm": byts / t / 1e9 / self.hbm,
                                                "stream_floor_us": t_floor * 1e6,
                                                "frac_of_stream_floor": t_floor / t}
        # the same up-proj with SwiGLU + MXFP8 requantisation in the GEMM's
        # epilogue (one launch instead of GEMM + separate pass)
        t = time_kernel(lambda: hq.hq_gemm_grouped_contig_swiglu_quant(qa, sfa, qbv, sfb, off, M, H, k, "mxfp8",
                                                                       "mxfp8", q_out=qs, sf_out=sfs),
                        20, self.flush)
        res["moe_contig_mxfp8_L8_fused_swiglu_quant"] = {
            "us": t * 1e6, "tflops": fl / t / 1e12, "frac_fp8": fl / t / 1e12 / self.p_fp8,
            "unfused_us": res["moe_contig_mxfp8_L8"]["us"] + res["swiglu_quant_mxfp8_17408x3072"]["us"]}
        return res

    def moe_masked(self):
        hq, dev = self.hq, self.dev
        res = {}
        c4 = synth.moe_masked(device=dev)
        E, max_m, n, k = c4["E"], c4["max_m"], c4["n"], c4["k"]
        qa, sfa = hq.hq_quant(c4["a"], "nvfp4")
        qb, sfb = hq.hq_quant(c4["b"].view(E * n, k), "nvfp4")
        mm = torch.from_numpy(c4["masked_m"]).to(dev)
        out4 = torch.empty(E * max_m, n, dtype=torch.bfloat16, device=dev)
        qbv = qb.view(E, n, k // 2)
        t = time_kernel(lambda: hq.hq_gemm_grouped_masked(qa, sfa, qbv, sfb, mm, max_m, n, k, "nvfp4",
                                                          alpha=c4["alpha"], out=out4), 20, self.flush)
        valid = int(c4["masked_m"].sum())
        tiles = int(sum(-(-int(c) // 128) for c in c4["masked_m"]))
        fl = 2.0 * valid * n * k
        byts = E * n * k // 2 + sfb.numel() + tiles * 128 * (k // 2 + k // 16) + valid * n * 2
        res["moe_masked_nvfp4_E32"] = {"us": t * 1e6, "tflops": fl / t / 1e12, "frac_fp4": fl / t / 1e12 / self.p_fp4,
                                      "gbs": byts / t / 1e9, "frac_hbm": byts / t / 1e9 / self.hbm}
        # the hot-path step on this workload: quantise the activations' valid
        # rows (masked_m[e] of each expert's max_m, BF16 -> NVFP4) and run the
        # masked GEMM against the resident NVFP4 expert weights
        a4 = c4["a"]

        def step():
            hq.hq_quant_masked(a4, mm, max_m, "nvfp4", q_out=qa, sf_out=sfa)
            hq.hq_gemm_grouped_masked(qa, sfa, qbv, sfb, mm, max_m, n, k, "nvfp4", alpha=c4["alpha"], out=out4)
        t_step = time_kernel(step, 20, self.flush)
        t_qa = time_kernel(lambda: hq.hq_quant_masked(a4, mm, max_m, "nvfp4", q_out=qa, sf_out=sfa), 20, self.flush)
        t_qa_all = time_kernel(lambda: hq.hq_quant(a4, "nvfp4", q_out=qa, sf_out=sfa), 20, self.flush)
        # end to end through the public API, as a serving loop runs it: every
        # step uploads the valid activation rows (masked_m[e] rows of each
        # expert's block) from pinned host memory, quantises them, runs the
        # GEMM and downloads the valid output rows; uploads, compute and
        # downloads on three streams with double-buffered device buffers, so
        # step i's download overlaps step i + 1's upload; steady state
        a_h = a4.cpu().pin_memory()
        out_h = torch.empty(E * max_m, n, dtype=torch.bfloat16).pin_memory()
        a_dev = [torch.empty_like(a4) for _ in range(2)]
        outs = [torch.empty_like(out4) for _ in range(2)]
        spans = [(e * max_m, int(c)) for e, c in enumerate(c4["masked_m"]) if int(c) > 0]
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        cst = torch.cuda.current_stream()
        quant_done, down_done = [None, None], [None, None]

        def e2e(i):
            j = i % 2
            ea, eg = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(up):
                if quant_done[j] is not None:
                    up.wait_event(quant_done[j])       # step i - 2 has read this buffer
                for r0, c in spans:
                    a_dev[j][r0:r0 + c].copy_(a_h[r0:r0 + c], non_blocking=True)
                ea.record(up)
            cst.wait_event(ea)
            hq.hq_quant_masked(a_dev[j], mm, max_m, "nvfp4", q_out=qa, sf_out=sfa)
            quant_done[j] = torch.cuda.Event()
            quant_done[j].record(cst)
            if down_done[j] is not None:
                cst.wait_event(down_done[j])            # step i - 2's rows have left
            hq.hq_gemm_grouped_masked(qa, sfa, qbv, sfb, mm, max_m, n, k, "nvfp4", alpha=c4["alpha"],
                                      out=outs[j])
            eg.record(cst)
            with torch.cuda.stream(down):
                down.wait_event(eg)
                for r0, c in spans:
                    out_h[r0:r0 + c].copy_(outs[j][r0:r0 + c], non_blocking=True)
                down_done[j] = torch.cuda.Event()
                down_done[j].record(down)
        for i in range(3):
            e2e(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        e0.record(up)
        for i in range(3, 3 + reps):
            e2e(i)
        e1.record(down)
        torch.cuda.synchronize()
        t_e2e = e0.elapsed_time(e1) / reps / 1e3
        res["moe_masked_nvfp4_E32_step"] = {
            "step": "hq_quant_masked(A's valid rows -> NVFP4), then hq_gemm_grouped_masked", "us": t_step * 1e6,
            "quant_us": t_qa * 1e6, "quant_all_rows_us": t_qa_all * 1e6, "tflops": fl / t_step / 1e12,
            "launches": 2,
            "e2e": {"us": t_e2e * 1e6, "tflops": fl / t_e2e / 1e12, "h2d_bytes_per_step": valid * k * 2,
                    "d2h_bytes_per_step": valid * n * 2,
                    "note": "weights resident; valid activation rows up and valid output rows down (one copy per "
                            "expert each way), uploads / compute / downloads on three streams"}}
        t = time_kernel(lambda: hq.hq_quant(c4["b"].view(E * n, k), "nvfp4", q_out=qb, sf_out=sfb), 5, self.flush)
        byts = 2 * E * n * k + E * n * k // 2 + sfb.numel()
        res["quant_nvfp4_W_131072x7168"] = {"us": t * 1e6, "gbs": byts / t / 1e9,
                                            "frac_hbm": byts / t / 1e9 / self.hbm}
        return res

    def host_link(self):
        """Copy rates between pinned host memory and the device (cudaMemcpyAsync
        through torch) at the headline step's sizes: A and B up (167.8 MB), the
        output down (100.7 MB); each direction alone and both at once on two
        streams.  No host pointer reaches a kernel."""
        dev = self.dev
        up_n, down_n = (4096 + 12288) * 5120, 4096 * 12288   # BF16 elements
        h_up = torch.empty(up_n, dtype=torch.bfloat16).pin_memory()
        d_up = torch.empty(up_n, dtype=torch.bfloat16, device=dev)
        h_down = torch.empty(down_n, dtype=torch.bfloat16).pin_memory()
        d_down = torch.empty(down_n, dtype=torch.bfloat16, device=dev)
        s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def timed(fn, reps=10):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            t0 = time.time()
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
            return (time.time() - t0) / reps

        def up():
            with torch.cuda.stream(s_up):
                d_up.copy_(h_up, non_blocking=True)

        def down():
            with torch.cuda.stream(s_down):
                h_down.copy_(d_down, non_blocking=True)

        def both():
            up()
            down()
        t_up, t_down, t_both = timed(up), timed(down), timed(both)
        ub, db = up_n * 2, down_n * 2
        return {"host_link": {"h2d_gbs": ub / t_up / 1e9, "d2h_gbs": db / t_down / 1e9,
                              "both_directions_gbs": (ub + db) / t_both / 1e9,
                              "h2d_bytes": ub, "d2h_bytes": db,
                              # a step that moves these bytes cannot beat the
                              # time of the two copies running together
                              "e2e_bound_tflops": 2.0 * 4096 * 12288 * 5120 / t_both / 1e12}}

    def mma_rate(self):
        """Issue rate of back-to-back tcgen05.mma per kind (the library's probe,
        M = 128 per SM, N = 256, one wave), single SM and CTA pairs."""
        res = {}
        for kind in ("bf16", "mxfp8", "nvfp4", "mxfp4"):
            for pair in (False, True):
                r = self.hq.probe_mma_rate(kind, pair=pair)
                res[f"{kind}_{'pair' if pair else 'single'}"] = {
                    "cycles_per_mma": r["cycles_per_mma"], "flop_per_clk_sm": r["flop_per_clk_sm"],
                    "sm_mhz": r["sm_mhz"], "ctas": r["ctas"]}
        return {"mma_rate": res}

    def dswiglu(self):
        hq, dev = self.hq, self.dev
        c5 = synth.dswiglu_bwd(device=dev)
        M, n, k, L = c5["m"], c5["n"], c5["k"], c5["L"]
        off = torch.from_numpy(c5["padded_offsets"]).to(dev)
        dprob = torch.zeros(M, device=dev)
        dbias = torch.zeros(L, 2 * n, dtype=torch.bfloat16, device=dev)
        d_row = torch.empty(M, 2 * n, dtype=torch.bfloat16, device=dev)
        ws_t = torch.empty(hq.hq_gemm_dswiglu_workspace_size(L, n), dtype=torch.uint8, device=dev)
        t = time_kernel(lambda: hq.hq_gemm_dswiglu(c5["a"], c5["b"], c5["c"], off, c5["alpha"], c5["beta"],
                                                   c5["prob"], dprob, dbias=dbias, d_row=d_row, workspace=ws_t),
                        20, self.flush)
        fl = 2.0 * M * n * k
        byts = M * k * 2 + L * n * k * 2 + 2 * M * 2 * n * 2 + M * 8
        res = {"dswiglu_bwd_L16": {"us": t * 1e6, "tflops": fl / t / 1e12, "frac_bf16": fl / t / 1e12 / self.p_bf16,
                                   "gbs": byts / t / 1e9, "frac_hbm": byts / t / 1e9 / self.hbm}}
        t = time_kernel(lambda: hq.hq_gemm_dgeglu(c5["a"], c5["b"], c5["c"], off, c5["alpha"], c5["prob"], dprob,
                                                  dbias=dbias, d_row=d_row, workspace=ws_t), 20, self.flush)
        res["dgeglu_bwd_L16"] = {"us": t * 1e6, "tflops": fl / t / 1e12, "frac_bf16": fl / t / 1e12 / self.p_bf16,
                                 "gbs": byts / t / 1e9, "frac_hbm": byts / t / 1e9 / self.hbm}
        # discrete weights: one pointer per expert (tensor maps built on the device each call)
        b_ptrs = torch.tensor([c5["b"][e].data_ptr() for e in range(L)], dtype=torch.int64, device=dev)
        ws_d = torch.empty(hq.hq_gemm_discrete_workspace_size(L, n), dtype=torch.uint8, device=dev)
        t = time_kernel(lambda: hq.hq_gemm_dglu_discrete(c5["a"], b_ptrs, c5["c"], off, c5["alpha"], c5["prob"],
                                                         dprob, n, beta=c5["beta"], dbias=dbias, d_row=d_row,
                                                         workspace=ws_d), 20, self.flush)
        res["dswiglu_bwd_L16_discrete"] = {"us": t * 1e6, "tflops": fl / t / 1e12,
                                           "frac_bf16": fl / t / 1e12 / self.p_bf16}
        # block-scaled contract on the same shapes: MXFP8 operands, FP8 D_row + SFD_row
        qa, sfa = hq.hq_quant(c5["a"], "mxfp8")
        qb, sfb = hq.hq_quant(c5["b"].view(L * n, k), "mxfp8")
        qb = qb.view(L, n, k)
        d8 = torch.empty(M, 2 * n, dtype=torch.uint8, device=dev)
        sfd = torch.empty(hq.sf_bytes(M, 2 * n, "mxfp8"), dtype=torch.uint8, device=dev)
        t = time_kernel(lambda: hq.hq_gemm_dglu_bs(qa, sfa, qb, sfb, c5["c"], off, c5["alpha"], c5["prob"], dprob,
                                                   k, "mxfp8", beta=c5["beta"], dbias=dbias, d_row=d8,
                                                   fp8_out=True, sfd_row=sfd, workspace=ws_t), 20, self.flush)
        byts8 = M * k + L * n * k + M * 2 * n * 2 + M * 2 * n + sfd.numel() + M * 8
        res["dswiglu_bwd_mxfp8_fp8out_L16"] = {"us": t * 1e6, "tflops": fl / t / 1e12,
                                               "frac_fp8": fl / t / 1e12 / self.p_fp8,
                                               "gbs": byts8 / t / 1e9, "frac_hbm": byts8 / t / 1e9 / self.hbm}
        return res


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    import __graft_entry__
    __graft_entry__.build()
    import fp4_grouped_gemm_gb300 as hq
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    peaks, pk_src = load_peaks()
    if args.only:
        print(json.dumps({"only": args.only, "workloads": Extras(hq, dev, peaks).run([args.only])}), flush=True)
        return
    h = headline(hq, dev, args, ws, peaks, pk_src)
    line = {"metric": "block-scaled GEMM TFLOP/s (hot-path step: quantise A and B, GEMM)",
            "value": h["value"], "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": h["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e2m1 (fp32 accumulate)",
            "data": "synthetic", "config": h["config"], "roofline": h["roofline"], "e2e": h["e2e"],
            "gpu_launches": h["gpu_launches"], "clocks": h["clocks"], "gemm_ms": h["gemm_ms"]}
    if rank == 0 and ws == 1 and not args.main_only:
        line["workloads"] = Extras(hq, dev, peaks).run(Extras.NAMES)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_cpu_baseline()
        line["cpu_baseline"]["per_kernel"] = oracle_kernel_baselines()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
