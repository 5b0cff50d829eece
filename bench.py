"""Benchmark of the sparse x dense hot path on GB300.

Default workload: power-law CSR SpMV, M = K = 4,194,304, Zipf(2.1) row
lengths clipped to [1, 200000] and rescaled to mean 16 (nnz ~ 67.1M), y =
A x + 0.5 y -- the configuration the headline metric is quoted on.  One step
is one SpMV call through the C ABI: the binned main launch plus the long-row
fix-up launch.  Format conversion and planning are timed once, separately.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload power-law|power-law-coo|power-law-sell|uniform|dual|spmm32|spmm128|spmm32-bf16|spmm128-bf16|
                                spmm32-f16|spmm128-f16|spmm32-power-law|bsr|bsr-skewed|wcsr|
                                wcsr-skewed]

Prints one JSON line.  Under torchrun each rank runs an independent replica of
the workload (the products shard by rows with no exchange; "weak" scaling);
rank 0 prints.  --impl reference times the CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SpMV/SpMM GFLOP/s (2·nnz·N) and achieved HBM GB/s as % of GB300 peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DATASHEET_HBM_GBS = 7900.0       # GB300 HBM3e, nominal
DATASHEET_BF16_TFLOPS = 2250.0   # GB300 dense bf16 tensor rate, nominal


# ---------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sustained=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(*names):
    h = hashlib.sha1()
    for n in names:
        h.update(open(os.path.join(ROOT, "csr_bsr_spmv_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:12]


def env_info(dev) -> dict:
    """The run's environment: GPU, SM count, compute capability, CUDA runtime, driver, torch, host cores."""
    import torch
    prop = torch.cuda.get_device_properties(dev)
    drv = None
    try:
        drv = subprocess.run(["nvidia-smi", f"--id={dev.index}", "--query-gpu=driver_version", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        pass
    return {"gpu": prop.name, "sms": prop.multi_processor_count, "cc": f"{prop.major}.{prop.minor}",
            "cuda_runtime": torch.version.cuda, "driver": drv, "torch": torch.__version__,
            "host_cores": os.cpu_count()}


def traffic_from_profile(workload, src_hash):
    """DRAM read+write bytes of the step's dominant kernel from the committed ncu
    capture for this workload, or None when the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("source_hash") != src_hash:
        return None
    return d.get("dram_bytes_per_launch")


def slowest_rank_ms(ms: float, device) -> float:
    """Max of the per-rank step times over the process group (the job is as
    slow as its slowest replica); the identity without a group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job GFLOP/s: every replica's work over the slowest replica's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------- workloads

def make_workload(name: str, rows: int = 0):
    """Host arrays of the workload; `rows` shrinks the power-law case (profiling)."""
    import synth

    if name in ("power-law", "power-law-coo", "power-law-sell"):
        c = synth.power_law_rows(M=rows) if rows else synth.power_law_rows()
        if name == "power-law-coo":
            c["name"] += " as row-sorted COO"
        if name == "power-law-sell":
            c["name"] += " as SELL-C-sigma (C 32)"
    elif name == "uniform":
        c = synth.uniform_short_rows()
    elif name == "dual":
        c = synth.banded_pair()
    elif name in ("spmm32", "spmm128"):
        c = synth.clustered_spmm(N=int(name[4:]))
    elif name in ("spmm32-bf16", "spmm128-bf16"):
        c = synth.clustered_spmm(N=int(name[4:-5]))
        c["val_bf16"] = synth.to_bf16_bits(c["val"])
        c["B_bf16"] = synth.to_bf16_bits(c["B"]).reshape(c["B"].shape)
        c["name"] += " (bf16 A values and B, fp32 accumulation)"
    elif name == "spmm32-power-law":  # skewed rows: the planned SpMM (long rows split)
        c = synth.power_law_rows()
        c["N"] = 32
        c["B"] = synth.uniform(8, synth.T_B, c["K"] * 32).reshape(c["K"], 32)
        c["name"] += " SpMM N=32 (planned: long rows split)"
    elif name in ("spmm32-f16", "spmm128-f16"):
        c = synth.clustered_spmm(N=int(name[4:-4]))
        c["B_f16"] = c["B"].astype(np.float16)
        c["name"] += " (fp16 A values and B, fp32 accumulation)"
    elif name == "bsr":
        c = synth.block_sparse()
    elif name == "bsr-skewed":  # every 16th block-row 8x longer: the planned call splits it
        c = synth.block_sparse_skewed()
    elif name == "wcsr":
        c = synth.window_pool()
    elif name == "wcsr-skewed":  # every 16th window ~6.5x wider: the planned call splits it
        c = synth.window_pool_skewed()
    else:
        raise SystemExit(f"unknown workload {name}")
    c["workload"] = name
    return c


def accounting(c):
    """(flops, algorithmic bytes) of one step, by the compulsory-traffic rules."""
    M, K, nnz = c["M"], c["K"], c["row"].size
    w = c["workload"]
    if w in ("power-law", "uniform", "power-law-sell"):  # SELL: the CSR definition's bytes (padding is overhead)
        ybytes = 8 * M if c["beta"] != 0 else 4 * M
        return 2 * nnz, 8 * nnz + 4 * (M + 1) + 4 * K + ybytes
    if w == "power-law-coo":  # row index per entry instead of row offsets
        ybytes = 8 * M if c["beta"] != 0 else 4 * M
        return 2 * nnz, 12 * nnz + 4 * K + ybytes
    if w == "dual":
        # u = A v - a u (reads v, reads+writes u); v = A^T u - b v (reads u, reads+writes v)
        b1 = 8 * nnz + 4 * (M + 1) + 4 * K + 8 * M
        b2 = 8 * nnz + 4 * (K + 1) + 4 * M + 8 * K
        return 4 * nnz, b1 + b2
    if w.startswith("spmm") and w.endswith("f16"):  # bf16 or fp16 values and B
        N = c["N"]
        return 2 * nnz * N, 6 * nnz + 4 * (M + 1) + 2 * K * N + 4 * M * N
    if w.startswith("spmm"):
        N = c["N"]
        return 2 * nnz * N, 8 * nnz + 4 * (M + 1) + 4 * K * N + 4 * M * N
    if w.startswith("wcsr"):  # flops of the stored chunks (what the tensor cores execute); bytes of the WCSR arrays
        nch, N = c["nchunks"], c["N"]
        return 2 * nch * 4096 * N, 2 * nch * 4096 + 4 * 64 * nch + 4 * (M // 64 + 1) + 2 * K * N + 4 * M * N
    if w.startswith("bsr"):
        bs, N = c["bs"], c["N"]
        nb = c["bcols"].size if "bcols" in c else c["row"].size // (bs * bs)  # dense blocks
        return 2 * nb * bs * bs * N, 2 * nb * bs * bs + 4 * nb + 4 * (M // bs + 1) + 2 * K * N + 4 * M * N
    raise ValueError(w)


# ---------------------------------------------------------------- our arm

def synth_bits(val):
    import synth

    return synth.to_bf16_bits(val).view(np.int16)


def run_ours(args, rank, world, workload=None, cpu_seconds=None):
    import torch

    from csr_bsr_spmv_gb300 import spx

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    c = make_workload(workload or args.workload, args.rows if workload in (None, args.workload) else 0)
    flops, abytes = accounting(c) if not c["workload"].startswith("wcsr") else (None, None)  # wcsr: after its build
    M, K = c["M"], c["K"]
    w = c["workload"]
    stream = torch.cuda.Stream(device=dev)
    timings = {}

    t0 = time.perf_counter()
    if w in ("bsr", "bsr-skewed", "wcsr", "wcsr-skewed"):
        rp, col, val = spx.spx_build_csr(M, K, c["row"], c["col"], c["val_bf16"])
    elif w == "power-law-coo":
        rp = col = val = None  # the generator's triplets are already sorted by row
    else:
        rp, col, val = spx.spx_build_csr(M, K, c["row"], c["col"], c["val"])
    timings["build_csr_ms"] = 1e3 * (time.perf_counter() - t0)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 256 MB > L2
    run = None
    prep = None
    h2d = d2h = 0
    e2e_run = None
    hostio = None

    def device_timing(key, fn):  # conversion on the GPU, second of two runs (the first warms the allocator)
        for _ in range(2):
            torch.cuda.synchronize(dev)
            t1 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            timings[key] = 1e3 * (time.perf_counter() - t1)

    if w in ("power-law", "uniform"):
        A = spx.Csr(M, K, to_dev(rp), to_dev(col), to_dev(val))
        dr, dc, dv = to_dev(c["row"]), to_dev(c["col"]), to_dev(c["val"])
        device_timing("build_csr_device_ms", lambda: spx.spx_build_csr(M, K, dr, dc, dv, stream=stream))
        device_timing("row_stats_device_ms", lambda: spx.spx_row_stats(M, A.row_ptr))
        del dr, dc, dv
        x = to_dev(c["x"])
        y = to_dev(c["y"])
        opts = args.plan_opts
        if args.tune:
            t0 = time.perf_counter()
            opts, tune_ms, _ = spx.spx_plan_autotune(A, rp, x, stream=stream)
            timings["tune_ms"] = 1e3 * (time.perf_counter() - t0)
        t0 = time.perf_counter()
        plan = spx.spx_plan_csr(M, K, A.nnz, rp, opts=opts, device=dev, stream=stream)
        timings["plan_ms"] = 1e3 * (time.perf_counter() - t0)
        device_timing("plan_device_ms", lambda: spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts=opts, stream=stream))
        alpha, beta = c["alpha"], c["beta"]
        src = source_hash("spx_spmv.cu", "spx_gather.cuh", "spx_carveout.cuh")

        def run():
            spx.spx_spmv_csr(plan, A, x, y, alpha, beta, stream=stream)

        xh = torch.from_numpy(c["x"]).pin_memory()
        yh = torch.from_numpy(c["y"]).pin_memory()
        yo = torch.empty_like(yh).pin_memory()
        h2d = xh.numel() * 4 + (yh.numel() * 4 if beta != 0 else 0)
        d2h = yo.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                x.copy_(xh, non_blocking=True)
                if beta != 0:
                    y.copy_(yh, non_blocking=True)
                spx.spx_spmv_csr(plan, A, x, y, alpha, beta, stream=stream)
                yo.copy_(y, non_blocking=True)

        # the host-buffer C call: every step uploads x (and y) and downloads y, pipelined against the products
        hostio = (plan, A, xh.view(1, -1), yh, alpha, beta)

        info = dict(plan.info)
        extra = {"plan": {k: info[k] for k in ("tasks", "long_rows", "cta_rows", "split_rows", "thread_groups",
                                                "lane_groups", "segmented_groups")},
                 "plan_opts": plan.opts, "row_stats": plan.stats}
    elif w == "power-law-sell":
        x = to_dev(c["x"])
        y = to_dev(c["y"])
        alpha, beta = c["alpha"], c["beta"]
        t0 = time.perf_counter()
        S = spx.Sell(M, K, rp, col, val, opts=args.plan_opts, device=dev, stream=stream)
        timings["build_sell_ms"] = 1e3 * (time.perf_counter() - t0)
        dr, dc, dv = to_dev(rp), to_dev(col), to_dev(val)
        device_timing("build_sell_device_ms", lambda: spx.Sell(M, K, dr, dc, dv, opts=args.plan_opts,
                                                                upload=False).close())
        del dr, dc, dv
        src = source_hash("spx_sell.cu", "spx_gather.cuh", "spx_carveout.cuh")

        def run():
            spx.spx_spmv_sell(S, x, y, alpha, beta, stream=stream)

        xh = torch.from_numpy(c["x"]).pin_memory()
        yh = torch.from_numpy(c["y"]).pin_memory()
        yo = torch.empty_like(yh).pin_memory()
        h2d = xh.numel() * 4 + (yh.numel() * 4 if beta != 0 else 0)
        d2h = yo.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                x.copy_(xh, non_blocking=True)
                if beta != 0:
                    y.copy_(yh, non_blocking=True)
                spx.spx_spmv_sell(S, x, y, alpha, beta, stream=stream)
                yo.copy_(y, non_blocking=True)

        extra = {"sell": dict(S.info), "sell_opts": S.opts}
    elif w == "power-law-coo":
        crow, ccol, cval = to_dev(c["row"]), to_dev(c["col"]), to_dev(c["val"])
        x = to_dev(c["x"])
        y = to_dev(c["y"])
        alpha, beta = c["alpha"], c["beta"]
        scratch = torch.empty(max(1, spx.spx_spmv_coo_scratch_bytes(c["row"].size) // 4), device=dev)
        src = source_hash("spx_coo.cu", "spx_gather.cuh", "spx_carveout.cuh")

        def run():
            spx.spx_spmv_coo(M, K, crow, ccol, cval, x, y, alpha, beta, stream=stream, scratch=scratch)

        xh = torch.from_numpy(c["x"]).pin_memory()
        yh = torch.from_numpy(c["y"]).pin_memory()
        yo = torch.empty_like(yh).pin_memory()
        h2d = xh.numel() * 4 + (yh.numel() * 4 if beta != 0 else 0)
        d2h = yo.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                x.copy_(xh, non_blocking=True)
                if beta != 0:
                    y.copy_(yh, non_blocking=True)
                spx.spx_spmv_coo(M, K, crow, ccol, cval, x, y, alpha, beta, stream=stream, scratch=scratch)
                yo.copy_(y, non_blocking=True)

        extra = {"chunks": -(-int(c["row"].size) // 2048)}
    elif w == "dual":
        A = spx.Csr(M, K, to_dev(rp), to_dev(col), to_dev(val))
        t0 = time.perf_counter()
        trp, tc, tv = spx.spx_transpose_csr(M, K, rp, col, val)
        timings["transpose_ms"] = 1e3 * (time.perf_counter() - t0)
        device_timing("transpose_device_ms", lambda: spx.spx_transpose_csr(M, K, A.row_ptr, A.col, A.val, stream=stream))
        At = spx.Csr(K, M, to_dev(trp), to_dev(tc), to_dev(tv))
        oA = oAt = args.plan_opts
        if args.tune:
            t1 = time.perf_counter()
            oA, _, _ = spx.spx_plan_autotune(A, rp, to_dev(c["v0"]), stream=stream)
            oAt, _, _ = spx.spx_plan_autotune(At, trp, to_dev(c["u0"]), stream=stream)
            timings["tune_ms"] = 1e3 * (time.perf_counter() - t1)
        t0 = time.perf_counter()
        pA = spx.spx_plan_csr(M, K, A.nnz, rp, opts=oA, device=dev, stream=stream)
        pAt = spx.spx_plan_csr(K, M, A.nnz, trp, opts=oAt, device=dev, stream=stream)
        timings["plan_ms"] = 1e3 * (time.perf_counter() - t0)
        u = to_dev(c["u0"])
        v = to_dev(c["v0"])
        a, b = float(c["alphas"][0]), float(c["betas"][0])
        src = source_hash("spx_spmv.cu", "spx_gather.cuh", "spx_carveout.cuh")

        u0, v0 = u.clone(), v.clone()

        def prep():  # every step starts from (u0, v0); untimed
            u.copy_(u0)
            v.copy_(v0)

        def run():
            spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, -a, 1.0, -b, stream=stream)

        uh = torch.from_numpy(c["u0"]).pin_memory()
        vh = torch.from_numpy(c["v0"]).pin_memory()
        uo, vo = torch.empty_like(uh).pin_memory(), torch.empty_like(vh).pin_memory()
        h2d = (uh.numel() + vh.numel()) * 4
        d2h = h2d

        def e2e_run():
            with torch.cuda.stream(stream):
                u.copy_(uh, non_blocking=True)
                v.copy_(vh, non_blocking=True)
                spx.spx_spmv_csr_dual(pA, pAt, A, At, v, u, 1.0, -a, 1.0, -b, stream=stream)
                uo.copy_(u, non_blocking=True)
                vo.copy_(v, non_blocking=True)

        extra = {"plan_A": dict(pA.info), "plan_At": dict(pAt.info), "plan_opts_A": pA.opts, "plan_opts_At": pAt.opts}
    elif w.startswith("spmm") and w.endswith("bf16"):
        A = spx.Csr(M, K, to_dev(rp), to_dev(col), to_dev(synth_bits(val)))
        B = to_dev(c["B_bf16"].view(np.int16))
        C = torch.empty(M, c["N"], device=dev)
        src = source_hash("spx_spmm.cu")

        def run():
            spx.spx_spmm_csr_bf16(A, B, C, 1.0, 0.0, stream=stream)

        Bh = torch.from_numpy(c["B_bf16"].view(np.int16)).pin_memory()
        Co = torch.empty(M, c["N"]).pin_memory()
        h2d, d2h = Bh.numel() * 2, Co.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                B.copy_(Bh, non_blocking=True)
                spx.spx_spmm_csr_bf16(A, B, C, 1.0, 0.0, stream=stream)
                Co.copy_(C, non_blocking=True)

        extra = {"variant": "bf16 storage, fp32 accumulation"}
    elif w.startswith("spmm") and w.endswith("-f16"):
        A = spx.Csr(M, K, to_dev(rp), to_dev(col), to_dev(val.astype(np.float16).view(np.int16)))
        B = to_dev(c["B_f16"].view(np.int16))
        C = torch.empty(M, c["N"], device=dev)
        src = source_hash("spx_spmm.cu")

        def run():
            spx.spx_spmm_csr_f16(A, B, C, 1.0, 0.0, stream=stream)

        Bh = torch.from_numpy(c["B_f16"].view(np.int16)).pin_memory()
        Co = torch.empty(M, c["N"]).pin_memory()
        h2d, d2h = Bh.numel() * 2, Co.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                B.copy_(Bh, non_blocking=True)
                spx.spx_spmm_csr_f16(A, B, C, 1.0, 0.0, stream=stream)
                Co.copy_(C, non_blocking=True)

        extra = {"variant": "fp16 storage, fp32 accumulation"}
    elif w == "spmm32-power-law":
        A = spx.Csr(M, K, to_dev(rp), to_dev(col), to_dev(val))
        B = to_dev(c["B"])
        C = torch.empty(M, c["N"], device=dev)
        # plan options that suit SpMM: rows past 64 nonzeros get whole CTAs, past 2048 segments
        popts = args.plan_opts or {"block_nnz": 1024, "lanes_div": 0, "pack_max": 64, "cta_max": 2048, "seg_nnz": 2048}
        t0 = time.perf_counter()
        plan = spx.spx_plan_csr(M, K, A.nnz, A.row_ptr, opts=popts, stream=stream)
        timings["plan_device_ms"] = 1e3 * (time.perf_counter() - t0)
        sc = torch.empty(max(1, plan.info["slots"] * c["N"]), device=dev)
        src = source_hash("spx_spmm.cu")

        def run():
            spx.spx_spmm_csr_planned(plan, A, B, C, 1.0, 0.0, stream=stream, scratch=sc)

        Bh = torch.from_numpy(c["B"]).pin_memory()
        Co = torch.empty(M, c["N"]).pin_memory()
        h2d, d2h = Bh.numel() * 4, Co.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                B.copy_(Bh, non_blocking=True)
                spx.spx_spmm_csr_planned(plan, A, B, C, 1.0, 0.0, stream=stream, scratch=sc)
                Co.copy_(C, non_blocking=True)

        extra = {"plan": dict(plan.info), "plan_opts": plan.opts}
    elif w.startswith("spmm"):
        A = spx.Csr(M, K, to_dev(rp), to_dev(col), to_dev(val))
        B = to_dev(c["B"])
        C = torch.empty(M, c["N"], device=dev)
        src = source_hash("spx_spmm.cu")

        def run():
            spx.spx_spmm_csr(A, B, C, 1.0, 0.0, stream=stream, col_tile=args.col_tile)

        Bh = torch.from_numpy(c["B"]).pin_memory()
        Co = torch.empty(M, c["N"]).pin_memory()
        h2d, d2h = Bh.numel() * 4, Co.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                B.copy_(Bh, non_blocking=True)
                spx.spx_spmm_csr(A, B, C, 1.0, 0.0, stream=stream, col_tile=args.col_tile)
                Co.copy_(C, non_blocking=True)

        extra = {"variant": spx.spx_spmm_csr_variant(B, C)}
    elif w.startswith("wcsr"):
        t0 = time.perf_counter()
        wp, wc, wv, fill = spx.spx_build_wcsr(M, K, rp, col, val)
        timings["build_wcsr_ms"] = 1e3 * (time.perf_counter() - t0)
        dr, dc, dv = to_dev(rp), to_dev(col), to_dev(val.view(np.int16))
        device_timing("build_wcsr_device_ms", lambda: spx.spx_build_wcsr(M, K, dr, dc, dv, stream=stream))
        del dr, dc, dv
        c["nchunks"] = int(wc.size // 64)
        flops, abytes = accounting(c)
        d_wp, d_wc = to_dev(wp), to_dev(wc)
        d_wv = to_dev(wv.reshape(-1).view(np.int16))
        Bm = to_dev(c["B_bf16"].view(np.int16))
        C = torch.empty(M, c["N"], device=dev)
        src = source_hash("spx_wcsr.cu", "spx_tc.cuh")

        wplan = spx.WcsrPlan(M, c["nchunks"], d_wp, stream=stream) if w == "wcsr-skewed" else None
        wscratch = (torch.empty(max(4, spx._lib().spx_spmm_wcsr_planned_scratch_bytes(wplan.handle, c["N"]) // 4),
                                device=dev) if wplan else None)

        def wcsr_call():
            if wplan is None:
                spx.spx_spmm_wcsr(M, K, d_wp, d_wc, d_wv, Bm, C, stream=stream)
            else:
                spx.spx_spmm_wcsr_planned(wplan, M, K, d_wp, d_wc, d_wv, Bm, C, stream=stream, scratch=wscratch)

        def run():
            wcsr_call()

        Bh = torch.from_numpy(c["B_bf16"].view(np.int16)).pin_memory()
        Co = torch.empty(M, c["N"]).pin_memory()
        h2d, d2h = Bh.numel() * 2, Co.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                Bm.copy_(Bh, non_blocking=True)
                wcsr_call()
                Co.copy_(C, non_blocking=True)

        extra = {"fill_ratio": fill, "nchunks": c["nchunks"], "useful_flops": 2 * int(c["row"].size) * c["N"],
                 "useful_gflops": None}
        if wplan is not None:  # the same product without the task split, for comparison (untimed by the step)
            extra["task_split"] = dict(wplan.info)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ts = []
            for _ in range(5):
                with torch.cuda.stream(stream):
                    ev0.record(stream)
                    spx.spx_spmm_wcsr(M, K, d_wp, d_wc, d_wv, Bm, C, stream=stream)
                    ev1.record(stream)
                ev1.synchronize()
                ts.append(ev0.elapsed_time(ev1))
            extra["unsplit_ms"] = round(sorted(ts)[2], 5)
    else:  # bsr
        t0 = time.perf_counter()
        brp, bcol, bval, fill = spx.spx_build_bsr(M, K, rp, col, val, c["bs"], c["bs"])
        timings["build_bsr_ms"] = 1e3 * (time.perf_counter() - t0)
        dr, dc, dv = to_dev(rp), to_dev(col), to_dev(val.view(np.int16))
        device_timing("build_bsr_device_ms", lambda: spx.spx_build_bsr(M, K, dr, dc, dv, c["bs"], c["bs"],
                                                                        stream=stream))
        del dr, dc, dv
        d_brp, d_bcol = to_dev(brp), to_dev(bcol)
        d_bval = to_dev(bval.view(np.int16))
        Bm = to_dev(c["B_bf16"].view(np.int16))
        C = torch.empty(M, c["N"], device=dev)
        src = source_hash("spx_bsr.cu", "spx_tc.cuh")

        bplan = spx.BsrPlan(M, int(bcol.size), d_brp, stream=stream) if w == "bsr-skewed" else None
        bscratch = (torch.empty(max(4, spx._lib().spx_spmm_bsr_planned_scratch_bytes(bplan.handle, c["N"]) // 4),
                                device=dev) if bplan else None)

        def bsr_call():
            if bplan is None:
                spx.spx_spmm_bsr(M, K, c["bs"], c["bs"], d_brp, d_bcol, d_bval, Bm, C, stream=stream)
            else:
                spx.spx_spmm_bsr_planned(bplan, M, K, c["bs"], c["bs"], d_brp, d_bcol, d_bval, Bm, C, stream=stream,
                                         scratch=bscratch)

        def run():
            bsr_call()

        Bh = torch.from_numpy(c["B_bf16"].view(np.int16)).pin_memory()
        Co = torch.empty(M, c["N"]).pin_memory()
        h2d, d2h = Bh.numel() * 2, Co.numel() * 4

        def e2e_run():
            with torch.cuda.stream(stream):
                Bm.copy_(Bh, non_blocking=True)
                bsr_call()
                Co.copy_(C, non_blocking=True)

        extra = {"fill_ratio": fill, "nnzb": int(bcol.size)}
        if bplan is not None:  # the same product without the task split, for comparison (untimed by the step)
            extra["task_split"] = dict(bplan.info)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ts = []
            for _ in range(5):
                with torch.cuda.stream(stream):
                    ev0.record(stream)
                    spx.spx_spmm_bsr(M, K, c["bs"], c["bs"], d_brp, d_bcol, d_bval, Bm, C, stream=stream)
                    ev1.record(stream)
                ev1.synchronize()
                ts.append(ev0.elapsed_time(ev1))
            extra["unsplit_ms"] = round(sorted(ts)[2], 5)

    # ---------------- timing: warmup, then K steps with an L2 flush between steps
    def flush_l2():
        with torch.cuda.stream(stream):
            if prep is not None:
                prep()
            flush.fill_(1.0)

    def hold_stream(steps):
        # A spin kernel keeps the stream busy while the host enqueues the steps that follow, so that
        # a start event never waits on the host's next launch: the events then time device work only
        # (for a call of a few microseconds the host's enqueue would otherwise show up in the step)
        spin = getattr(torch.cuda, "_sleep", None)
        if spin is not None:
            with torch.cuda.stream(stream):
                spin(int(4e6 + 6e5 * steps))  # SM cycles: about 2 ms + 0.3 ms per step at 2 GHz

    for _ in range(args.warmup):
        flush_l2()
        run()
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches0 = spx.launch_count()
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        hold_stream(len(ev))
        for s, e in ev:
            flush_l2()
            s.record(stream)
            run()
            e.record(stream)
        torch.cuda.synchronize(dev)
    launches = spx.launch_count() - launches0
    times = [s.elapsed_time(e) for s, e in ev]
    ms = sum(times) / len(times)
    if world > 1:
        import torch.distributed as dist
        ms = slowest_rank_ms(ms, dev)
        dist.barrier()
    torch.cuda.synchronize(dev)
    assert spx.spx_last_device_error(stream) == 0, "device error word set during the timed region"

    # ---------------- warm steps: the same calls back to back with no L2 flush (reported beside the flushed number)
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    run()
    hold_stream(len(wev))
    for s, e in wev:
        s.record(stream)
        run()
        e.record(stream)
    torch.cuda.synchronize(dev)
    wtimes = [s.elapsed_time(e) for s, e in wev]
    extra["warm"] = {"ms_per_step_median": round(statistics.median(wtimes), 5),
                     "ms_per_step_min": round(min(wtimes), 5),
                     "how": "the same steps back to back without the L2 flush (rank-local, CUDA events)"}

    # ---------------- launch-bound SpMV: the per-call time inside one CUDA graph of many calls
    if w == "uniform":
        calls = 200
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            run()  # warm the library's per-device set-up outside the capture
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(calls):
                    run()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        extra["graph_us_per_call"] = round(g0.elapsed_time(g1) * 1e3 / (5 * calls), 3)
        extra["graph_note"] = (f"{calls} calls captured in one CUDA graph, replayed 5 times, no L2 flush between calls "
                               "(the matrix and vectors, 0.33 MB, stay in L2): the launch-bound cost per call")
        # the same two timings of the smallest kernel there is (one 4-byte store): the floor that launching
        # and event-timing one kernel put under any call
        tiny = torch.zeros(1, device=dev)
        with torch.cuda.stream(stream):
            tiny.fill_(1.0)
        torch.cuda.synchronize(dev)
        te = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        hold_stream(len(te))
        for s_, e_ in te:
            s_.record(stream)
            with torch.cuda.stream(stream):
                tiny.fill_(1.0)
            e_.record(stream)
        torch.cuda.synchronize(dev)
        tgraph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(tgraph, stream=stream):
                for _ in range(calls):
                    tiny.fill_(1.0)
        tgraph.replay()
        torch.cuda.synchronize(dev)
        g0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(5):
                tgraph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        extra["launch_floor"] = {
            "us_per_call_median": round(statistics.median(s_.elapsed_time(e_) for s_, e_ in te) * 1e3, 3),
            "graph_us_per_call": round(g0.elapsed_time(g1) * 1e3 / (5 * calls), 3),
            "what": "a one-element fill timed the same two ways: the launch + event floor under any single call"}

    # ---------------- the stream + gather floor of the same matrix (SpMV workloads)
    gather_floor = None
    # (workloads with uniformly random columns: there the x gathers have no locality, so no kernel
    # over these arrays can beat the probe; banded columns give the group kernel a locality the
    # grid-stride probe does not have)
    if w in ("power-law", "uniform") and not args.no_floor:
        probes = [(A, x)]
        part = torch.empty(spx._lib().spx_gather_probe_blocks(), device=dev)

        def probe():
            for Am, xv in probes:
                spx.spx_gather_probe(Am, xv, part, stream=stream)

        for _ in range(args.warmup):
            flush_l2()
            probe()
        torch.cuda.synchronize(dev)
        pe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        hold_stream(len(pe))
        for s_, e_ in pe:
            flush_l2()
            s_.record(stream)
            probe()
            e_.record(stream)
        torch.cuda.synchronize(dev)
        pms = sum(s_.elapsed_time(e_) for s_, e_ in pe) / len(pe)
        gather_floor = {"probe_ms": round(pms, 5), "kernel_over_floor": round(ms / pms, 3),
                        "gathers_per_s": round(c["row"].size / (pms * 1e-3), 1),
                        "what": "spx_gather_probe on the same col/val/x: stream them and gather x once per nonzero, "
                                "no row work -- the floor of any SpMV over uniformly random columns; "
                                "kernel_over_floor = step time / probe time"}

    # ---------------- end to end through the public call with pinned host buffers
    e2e = None
    if e2e_run is not None and not args.no_e2e:
        for _ in range(2):
            e2e_run()
        torch.cuda.synchronize(dev)
        es = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(max(3, args.steps // 2))]
        for s, e in es:
            flush_l2()
            s.record(stream)
            e2e_run()
            e.record(stream)
        torch.cuda.synchronize(dev)
        ems = sum(s.elapsed_time(e) for s, e in es) / len(es)
        e2e = {"value": round(world * flops / (ems * 1e-3) / 1e9, 3), "unit": "GFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ems, 4),
               "how": "per step, one after another: pinned H2D copies, the device call, the D2H copy"}
        if hostio is not None:
            hp, hA, hx, hy0, ha, hb = hostio
            nb = max(3, args.steps)
            yb = torch.empty(nb, hy0.numel()).pin_memory()
            work = torch.empty(max(1, spx._lib().spx_spmv_csr_hostio_work_bytes(hA.M, hA.K) // 4), device=dev)
            for rep in range(2):  # the first run warms the pipeline's streams and events
                yb.copy_(hy0.expand(nb, -1))
                torch.cuda.synchronize(dev)
                s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s_.record(stream)
                spx.spx_spmv_csr_hostio(hp, hA, hx, yb, ha, hb, work=work, stream=stream)
                e_.record(stream)
                torch.cuda.synchronize(dev)
            pms = s_.elapsed_time(e_) / nb
            e2e_serial = e2e
            e2e = {"value": round(world * flops / (pms * 1e-3) / 1e9, 3), "unit": "GFLOP/s",
                   "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(pms, 4),
                   "how": f"spx_spmv_csr_hostio over {nb} steps from pinned host buffers: each step uploads x and y "
                          "and downloads y; copies on two streams overlap the neighbouring steps' products",
                   "serial": e2e_serial}

    pk = peaks()
    gflops = job_throughput(flops, world, ms)
    if w.startswith("wcsr"):
        extra["useful_gflops"] = round(extra["useful_flops"] / (ms * 1e-3) / 1e9, 1)
    if w in ("bsr", "bsr-skewed", "wcsr", "wcsr-skewed"):
        ach = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16"], 4), "peak_source": pk["src"] + " (bf16 dense, burst)"}
    else:
        ach = abytes / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(ach / pk["hbm"], 4), "peak_source": pk["src"] + " (HBM copy)"}
    tr = traffic_from_profile(w, src)
    roof["traffic"] = tr
    # the same achieved figure against the other denominators: the datasheet figures (HBM3e 7.9 TB/s,
    # 2.25 PFLOP/s dense bf16) and, for the tensor-core kernels, the sustained measured bf16 rate; the
    # ncu DRAM traffic per step over the step time, against the measured and datasheet HBM rates
    if roof["bound"] == "tensor":
        roof["vs_other_peaks"] = {"bf16_sustained_tflops": pk["bf16_sustained"],
                                  "frac_of_sustained": round(ach / pk["bf16_sustained"], 4) if pk["bf16_sustained"] else None,
                                  "bf16_datasheet_tflops": DATASHEET_BF16_TFLOPS,
                                  "frac_of_datasheet": round(ach / DATASHEET_BF16_TFLOPS, 4)}
    else:
        roof["vs_other_peaks"] = {"hbm_datasheet_gbs": DATASHEET_HBM_GBS,
                                  "frac_of_datasheet": round(ach / DATASHEET_HBM_GBS, 4)}
    if tr:
        tgbs = tr / (ms * 1e-3) / 1e9
        roof["vs_other_peaks"].update({"traffic_gbs": round(tgbs, 1), "traffic_frac_of_measured": round(tgbs / pk["hbm"], 4),
                                       "traffic_frac_of_datasheet": round(tgbs / DATASHEET_HBM_GBS, 4)})
    if gather_floor is not None:
        roof["gather_floor"] = gather_floor
    roof["algorithmic_bytes"] = int(abytes)
    roof["timed"] = ("whole step (all launches of the call), CUDA events on the launching stream; a spin kernel "
                  "holds the stream while the host enqueues the steps")

    line = {
        "metric": METRIC, "value": round(gflops, 3), "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16->f32" if (w in ("bsr", "bsr-skewed", "wcsr", "wcsr-skewed") or w.endswith("bf16"))
        else "f16->f32" if w.endswith("-f16") else "f32",
        "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": c["name"], "M": M, "K": K, "nnz": int(c["row"].size),
                   "N": c.get("N", 1), "l2": "flushed between steps (256 MB write); inputs also exceed L2",
                   "parallelism": f"replicas x{world}"},
        "hbm_gbs": round(abytes / (ms * 1e-3) / 1e9, 1), "roofline": roof, "e2e": e2e, "gpu_launches": int(launches),
        "conversion": {k: round(v, 2) for k, v in timings.items()}, "detail": extra, "env": env_info(dev),
        "step_ms_min": round(min(times), 5), "step_ms_median": round(statistics.median(times), 5),
    }
    line["clocks"] = clk.summary()
    if rank == 0 and world == 1 and not args.no_cpu and cpu_seconds != 0:
        line["cpu_baseline"] = cpu_baseline(c, budget_s=cpu_seconds or args.cpu_seconds)
    return line


# ---------------------------------------------------------------- CPU oracle

def row_major_csr(c, val):
    """The generator emits COO sorted by (row, col); its CSR row offsets are the
    first position of each row (no builder involved)."""
    rp = np.searchsorted(c["row"], np.arange(c["M"] + 1), side="left").astype(np.int32)
    return rp, c["col"], val


def cpu_step_fn(c, threads=1):
    """One bounded sample of the workload run by the oracle; returns (fn, flops, sample).
    threads > 1 runs the oracle's all-core build (OpenMP over rows; the same sums)."""
    import oracle

    w = c["workload"]
    M, K = c["M"], c["K"]
    t = dict(threads=threads)
    if w.startswith("wcsr"):
        import synth
        rp, col, val = row_major_csr(c, synth.bf16_bits_to_f32(c["val_bf16"]))
        rows = np.arange(0, M, 64 if threads == 1 else 4, dtype=np.int32)  # rows spread over every window
        Bf = synth.bf16_bits_to_f32(c["B_bf16"]).reshape(K, c["N"])
        fl = 2 * int(np.diff(rp)[rows].sum()) * c["N"]
        return (lambda: oracle.spmm(M, rp, col, val, Bf, rows=rows, **t)), fl, \
            f"{rows.size} output rows (every {M // rows.size}th) of the {M}x{K} product, nonzero flops"
    if w.startswith("bsr"):
        rp, col, val = row_major_csr(c, c["val_bf16"])
        if "_oracle_bsr" not in c:  # built once per workload (set-up, not timed)
            c["_oracle_bsr"] = oracle.build_bsr(M, K, rp, col, val, c["bs"], c["bs"])
        brp, bcol, bval, _ = c["_oracle_bsr"]
        rows = np.arange(0, M, 64 if threads == 1 else 4, dtype=np.int32)  # rows spread over every block-row
        nb = np.diff(brp)[rows // c["bs"]]
        fl = 2 * int(nb.sum()) * c["bs"] * c["N"]
        return (lambda: oracle.bsr_spmm(M, K, c["bs"], c["bs"], brp, bcol, bval, c["B_bf16"], rows=rows, **t)), fl, \
            f"{rows.size} output rows (every {M // rows.size}th) of the {M}x{K} BSR product, stored-block flops"
    if w == "power-law-coo":
        return (lambda: oracle.spmv_coo(M, K, c["row"], c["col"], c["val"], c["x"], c["alpha"], c["beta"],
                                        c["y"])), 2 * int(c["row"].size), "the full matrix, one COO SpMV (one core)"
    rp, col, val = row_major_csr(c, c["val"])
    if w in ("power-law", "uniform", "power-law-sell"):
        return (lambda: oracle.spmv(M, rp, col, val, c["x"], c["alpha"], c["beta"], c["y"], **t)), \
            2 * int(rp[-1]), "the full matrix, one SpMV"
    if w == "dual":
        if "_oracle_t" not in c:  # built once per workload (set-up, not timed)
            c["_oracle_t"] = oracle.transpose(M, K, rp, col, val)
        trp, tc, tv = c["_oracle_t"]

        def f():
            u1, _ = oracle.spmv(M, rp, col, val, c["v0"], 1.0, -float(c["alphas"][0]), c["u0"], **t)
            oracle.spmv(K, trp, tc, tv, u1.astype(np.float32), 1.0, -float(c["betas"][0]), c["v0"], **t)
        return f, 4 * int(rp[-1]), "the full operator pair, one iteration"
    N = c["N"]
    if w.endswith("bf16"):
        import synth
        val = synth.bf16_bits_to_f32(c["val_bf16"])
        c = dict(c, B=synth.bf16_bits_to_f32(c["B_bf16"]).reshape(c["B"].shape))
    elif w.endswith("-f16"):
        val = val.astype(np.float16).astype(np.float64)
        c = dict(c, B=c["B_f16"].astype(np.float64))
    rows = np.arange(0, M, 16 if threads == 1 else 2, dtype=np.int32)
    fl = 2 * int(np.diff(rp)[rows].sum()) * N
    return (lambda: oracle.spmm(M, rp, col, val, c["B"], rows=rows, **t)), fl, f"every {M // rows.size}th row ({rows.size} rows)"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _time_sample(fn, budget_s, max_reps=100000):
    fn()  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= max_reps:
            return n, el


def cpu_baseline(c, budget_s=12.0):
    """The oracle on the host cores: one core (the oracle as it stands), and its all-core build
    (OpenMP over rows on every core this process may use)."""
    fn, fl, sample = cpu_step_fn(c)
    n, el = _time_sample(fn, budget_s)
    out = {"value": round(n * fl / el / 1e9, 4), "unit": "GFLOP/s", "cores": 1, "kind": "oracle",
           "sample": f"{sample}, repeated {n}x ({el:.1f} s, fp64, single thread)"}
    cores = host_cores()
    if c["workload"] != "power-law-coo" and cores > 1:
        try:
            import oracle
            used = oracle.omp_threads(cores)
            fn, fl, sample = cpu_step_fn(c, threads=cores)
            n, el = _time_sample(fn, budget_s)
            out["all_cores"] = {"value": round(n * fl / el / 1e9, 4), "unit": "GFLOP/s", "cores": used,
                                "kind": "oracle (OpenMP build, rows over threads)",
                                "sample": f"{sample}, repeated {n}x ({el:.1f} s, fp64, {used} threads)"}
        except Exception as e:  # no OpenMP runtime on this host
            out["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    c = make_workload(args.workload, args.rows)
    fn, fl, sample = cpu_step_fn(c)
    for _ in range(args.warmup):
        fn()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    ms = 1e3 * sum(ts) / len(ts)
    val = fl / (ms * 1e-3) / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded SplitMix64)",
            "config": {"workload": c["name"], "M": c["M"], "K": c["K"], "nnz": int(c["row"].size),
                       "N": c.get("N", 1)},
            "cpu_baseline": {"value": round(val, 4), "unit": "GFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": f"{sample} per step (fp64, single thread)"},
            "e2e": {"value": round(val, 4), "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# The five configured workloads besides the headline (uniform 4096^2 SpMV, the dual pair, the clustered SpMM
# at N = 32 and 128, the block-sparse BSR SpMM) and the NEXT rows (SELL-C-sigma and COO SpMV on the power-law
# matrix, the bf16 CSR SpMM, the WCSR SpMM).  The oracle is timed beside the five configured workloads.
DEFAULT_CONFIGS = ("uniform", "dual", "spmm32", "spmm128", "bsr", "power-law-sell", "power-law-coo", "spmm32-bf16",
                   "wcsr")
CPU_CONFIGS = ("uniform", "dual", "spmm32", "spmm128", "bsr")


def config_summary(sub: dict) -> dict:
    """The figures of one configuration's run that the headline line carries for it."""
    keep = ("value", "unit", "ms_per_step", "step_ms_min", "step_ms_median", "dtype", "config", "hbm_gbs", "roofline",
            "e2e", "gpu_launches", "clocks", "cpu_baseline", "conversion")
    out = {k: sub[k] for k in keep if k in sub}
    det = sub.get("detail", {})
    for k in ("graph_us_per_call", "graph_note", "launch_floor", "warm", "fill_ratio", "nnzb", "nchunks", "useful_gflops",
              "variant"):
        if k in det:
            out[k] = det[k]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="power-law",
                    choices=["power-law", "power-law-coo", "power-law-sell", "uniform", "dual", "spmm32", "spmm128", "spmm32-f16",
                             "spmm128-f16", "spmm32-power-law", "spmm32-bf16",
                             "spmm128-bf16", "bsr", "bsr-skewed", "wcsr", "wcsr-skewed"])
    ap.add_argument("--tune", action="store_true", help="choose the SpMV plan options by spx_plan_autotune")
    ap.add_argument("--no-floor", action="store_true", help="skip timing the stream + gather floor probe")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--configs", default=",".join(DEFAULT_CONFIGS),
                    help="other workloads measured in the same run, reported under detail.configs ('' for none)")
    ap.add_argument("--config-cpu-seconds", type=float, default=4.0,
                    help="CPU oracle time per variant for each of those configurations")
    ap.add_argument("--rows", type=int, default=0, help="smaller power-law matrix (profiling only)")
    ap.add_argument("--plan", default="", help="plan options, e.g. block_nnz=4096,lanes_div=4")
    ap.add_argument("--col-tile", type=int, default=None, help="SpMM column tile (default: automatic)")
    args = ap.parse_args()
    args.plan_opts = {k: int(v) for k, v in (kv.split("=") for kv in args.plan.split(",") if kv)} or None
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world)
        configs = [w for w in args.configs.split(",") if w and w != args.workload]
        if configs:
            import torch
            line["detail"]["configs"] = {}
            for w in configs:  # the other workloads, measured the same way in the same run
                torch.cuda.empty_cache()
                t0 = time.perf_counter()
                try:
                    sub = run_ours(args, rank, world, workload=w,
                                   cpu_seconds=args.config_cpu_seconds if w in CPU_CONFIGS else 0)
                    line["detail"]["configs"][w] = config_summary(sub)
                except Exception as e:  # one configuration failing must not lose the others
                    line["detail"]["configs"][w] = {"error": f"{type(e).__name__}: {e}"}
                print(f"bench: {w} done in {time.perf_counter() - t0:.1f} s", file=sys.stderr, flush=True)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
