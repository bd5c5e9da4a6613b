#!/usr/bin/env python
"""Benchmark: Ozaki Scheme II emulated DGEMM on GB300 (one process per GPU).

One step = one pass of the whole Scheme II path (exponents -> residue split ->
per-modulus exact GEMM -> CRT + rounding) over m = n = k = 16384 with s = 14 moduli
on HPL-like phi = 0.5 inputs, through the library's C ABI with the inputs resident
in HBM.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the plain restatement of the method in
``oracle/``) on the host cores, on a bounded sample of the same workload.
Multi-GPU: the path does not shard; N ranks run N independent replicas and the
value is the total over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "emulated FP64 TFLOPS at 16384³ (s=14) and % of INT8 tensor-core roofline"
UNIT = "TFLOPS"
M = N = K = 16384
S = 14
PHI = 0.5
SEED = 0
PAGES_GH200_TFLOPS = 80.2  # the pages' Scheme II figure at 16384^3, s=14 (GH200): context
KERNELS_PER_STEP = 5       # rowexp(A), split(A), one-pass exponents + split(B), residue GEMM, CRT
# Figures the pages quote at 16384^3, each with its hardware: context only, not targets.
PAGES_FIGURES = {
    "GH200, Ozaki Scheme II, s=14": 80.2,
    "B200, NVIDIA's emulated-FP64 peak specification (tensor-core emulation)": 150.0,
    "RTX PRO 6000 Blackwell, OzII-FP4 (compute phase)": 17.31,
    "RTX PRO 6000 Blackwell, GEMMul8-INT8 (compute phase)": 40.94,
    "RTX PRO 6000 Blackwell, cuBLAS FP64": 1.85,
    "unit": "TFLOPS",
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, tag: str = ""):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"ozaki_bench_clocks{tag}_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ DRAM traffic of the GEMM
GEMM_SOURCES = ["fp64_gemm_emulation_gb300/csrc/oz_gemm.cu", "fp64_gemm_emulation_gb300/csrc/oz_device.cuh",
                "fp64_gemm_emulation_gb300/csrc/oz_internal.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "residue_gemm_16384_s14_traffic.json")


def gemm_source_digest() -> str:
    import hashlib

    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_traffic_bytes():
    """dram__bytes_read.sum + dram__bytes_write.sum of one residue-GEMM launch at this
    workload, from the committed ncu capture; None if the kernel sources changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != gemm_source_digest():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks (the slowest rank decides the job time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, flops_per_step: float, steps: int, job_ms: float) -> float:
    """Whole-job throughput in TFLOPS: the work of all ranks over the slowest rank's time."""
    return world * flops_per_step * steps / (job_ms * 1e-3) / 1e12


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ host link
def host_link_gbs(h_in, h_out, device) -> dict:
    """Pinned host<->device copy bandwidth of this machine (context for the e2e figure)."""
    import torch

    a, b = h_in.reshape(-1), h_out.reshape(-1)
    d = torch.empty(max(a.numel(), b.numel()), dtype=a.dtype, device=device)
    out = {}
    for name, copy, nbytes in (("h2d", lambda: d[: a.numel()].copy_(a, non_blocking=True), a.numel() * a.element_size()),
                               ("d2h", lambda: b.copy_(d[: b.numel()], non_blocking=True), b.numel() * b.element_size())):
        copy()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        copy()
        e1.record()
        torch.cuda.synchronize(device)
        out[name] = nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del d
    return out


# ------------------------------------------------------------------ reference arm (CPU oracle)
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from fp64_gemm_emulation_gb300.inputs import hpl_like
    from oracle import ozaki2 as O

    ms, ns = 128, 128  # sample: a 128 x 128 block of C with the full k = 16384
    A, B = hpl_like(ms, ns, K, phi=PHI, seed=SEED)
    times = []
    for it in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        O.ozaki2_dgemm(A, B, S, keep=False)
        if it >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = 2.0 * ms * ns * K * len(times) / total / 1e12
    cores = os.cpu_count()
    sample = f"oracle ozaki2_dgemm on a {ms}x{ns}x{K} block (s={S}, phi={PHI}); float64 BLAS matmul per modulus"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"ozaki2_dgemm m=n=k={M} s={S} phi={PHI} (sampled {ms}x{ns}x{K} block)",
                   "m": M, "n": N, "k": K, "moduli": S, "phi": PHI, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def cpu_baseline_measure():
    from fp64_gemm_emulation_gb300.inputs import hpl_like
    from oracle import ozaki2 as O

    ms, ns = 640, 640
    A, B = hpl_like(ms, ns, K, phi=PHI, seed=SEED)
    t0 = time.perf_counter()
    O.ozaki2_dgemm(A, B, S, keep=False)
    dt = time.perf_counter() - t0
    out = {"value": 2.0 * ms * ns * K / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"one oracle ozaki2_dgemm on a {ms}x{ns}x{K} block of the workload (s={S}, phi={PHI}), "
                     f"{dt:.1f} s; numpy float64 BLAS for the per-modulus products, Python integers for the CRT"}
    # the same oracle on one core (BLAS threads pinned to one before numpy loads), smaller block
    code = ("import time,sys; sys.path.insert(0, %r)\n"
            "from fp64_gemm_emulation_gb300.inputs import hpl_like\nfrom oracle import ozaki2 as O\n"
            "A, B = hpl_like(256, 256, %d, phi=%r, seed=%d)\nt0 = time.perf_counter()\n"
            "O.ozaki2_dgemm(A, B, %d, keep=False)\nprint(time.perf_counter() - t0)\n") % (ROOT, K, PHI, SEED, S)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        dt1 = float(r.stdout.strip().splitlines()[-1])
        out["one_core"] = {"value": 2.0 * 256 * 256 * K / dt1 / 1e12, "unit": UNIT, "cores": 1,
                           "sample": f"256x256x{K} block, {dt1:.1f} s"}
    except (subprocess.SubprocessError, ValueError, IndexError) as ex:
        out["one_core"] = f"unavailable: {ex}"[:120]
    return out


# ------------------------------------------------------------------ CPU-oracle timing protocol
# The oracle on the host cores, as a stated baseline (never a target): complete runs where
# it finishes (256^3 and 4096^3), and at the larger configurations the exponents and the
# residue planes of both operands in full (O(N^2) work) plus the exact products, CRT and
# rounding on 64 seeded 64 x 64 output tiles, extrapolated linearly by the tile fraction.
ORACLE_FULL = [(256, 256, 256, 14, 0.5), (4096, 4096, 4096, 14, 0.5)]
ORACLE_SAMPLED = [(8192, 8192, 8192, 14, 1.0), (16384, 16384, 16384, 14, 0.5), (2048, 2048, 262144, 14, 0.5)]


def _oracle_full(m, n, k, s, phi):
    from fp64_gemm_emulation_gb300.inputs import hpl_like
    from oracle import ozaki2 as O

    A, B = hpl_like(m, n, k, phi=phi, seed=SEED)
    t0 = time.perf_counter()
    O.ozaki2_dgemm(A, B, s, keep=False)
    return time.perf_counter() - t0


def _plane_block(args):
    from oracle import ozaki2 as O

    X, dd, moduli = args
    return O.residue_planes(O.scaled_trunc_matrix(X, dd), moduli)


def _oracle_sampled(m, n, k, s, phi, workers, tiles=64, tile=64):
    import multiprocessing as mp

    from fp64_gemm_emulation_gb300.inputs import hpl_like
    from oracle import ozaki2 as O

    A, B = hpl_like(m, n, k, phi=phi, seed=SEED)
    Bt = B.T
    with mp.get_context("spawn").Pool(workers) as pool:
        t0 = time.perf_counter()
        cc = O.crt_constants(O.greedy_moduli(s))
        kA = O.choose_k(cc.M, k)
        EA, EB = O.row_exponents(A), O.row_exponents(Bt)
        d, e = O.scale_exponents(EA, kA), O.scale_exponents(EB, kA)
        blk = max(1, min((1 << 22) // k, -(-max(m, n) // (4 * workers))))  # <= 4 Mi elements, >= 4 blocks a process
        Ares = np.empty((s, m, k), dtype=np.int8)
        Bres = np.empty((s, n, k), dtype=np.int8)
        for X, dd, P, rows in ((A, d, Ares, m), (Bt, e, Bres, n)):
            starts = list(range(0, rows, blk))
            jobs = ((np.ascontiguousarray(X[r0:r0 + blk]), dd[r0:r0 + blk], cc.moduli) for r0 in starts)
            for r0, planes in zip(starts, pool.imap(_plane_block, jobs)):
                P[:, r0:r0 + planes.shape[1]] = planes
        t_planes = time.perf_counter() - t0
    rng = np.random.default_rng(SEED)
    t1 = time.perf_counter()
    for _ in range(tiles):
        i0 = int(rng.integers(0, m // tile)) * tile
        j0 = int(rng.integers(0, n // tile)) * tile
        Cres = O.residue_products(Ares[:, i0:i0 + tile], np.transpose(Bres[:, j0:j0 + tile], (0, 2, 1)), cc.moduli)
        O.unscale(O.crt_reconstruct(Cres, cc), d[i0:i0 + tile], e[j0:j0 + tile])
    t_tiles = time.perf_counter() - t1
    return t_planes, t_tiles, t_planes + t_tiles * (m * n) / (tiles * tile * tile)


def oracle_protocol_entry(kind, m, n, k, s, phi, workers=1):
    if kind == "full":
        dt = _oracle_full(m, n, k, s, phi)
        return {"workload": f"{m}x{n}x{k} s={s} phi={phi}", "seconds": dt, "measured": "complete run",
                "tflops": 2.0 * m * n * k / dt / 1e12}
    t_planes, t_tiles, total = _oracle_sampled(m, n, k, s, phi, workers)
    return {"workload": f"{m}x{n}x{k} s={s} phi={phi}", "seconds": total,
            "measured": f"extrapolated: exponents + residue planes in full ({workers} processes) {t_planes:.1f} s, "
                        f"products + CRT + rounding on 64 seeded 64x64 tiles {t_tiles:.1f} s, "
                        f"scaled by the tile fraction",
            "tflops": 2.0 * m * n * k / total / 1e12}


def run_oracle_protocol(one_core: bool):
    """One JSON line per configuration.  All host cores: BLAS threads for the products and
    one process per core for the element-wise plane work of the sampled configurations.
    One core: one BLAS thread, the complete runs only."""
    cores = 1 if one_core else os.cpu_count()
    plan = [("full", c) for c in ORACLE_FULL] + ([] if one_core else [("sampled", c) for c in ORACLE_SAMPLED])
    for kind, (m, n, k, s, phi) in plan:
        out = oracle_protocol_entry(kind, m, n, k, s, phi, workers=cores)
        out.update({"kind": "oracle", "cores": cores, "unit": UNIT})
        print(json.dumps(out), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import torch

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from fp64_gemm_emulation_gb300 import ozaki as oz
    from fp64_gemm_emulation_gb300.inputs import hpl_like

    peaks, peak_src = load_peaks()
    lib = oz._lib
    A_np, B_np = hpl_like(M, N, K, phi=PHI, seed=SEED)
    dA = torch.from_numpy(A_np.T.copy()).to(device).t()
    dB = torch.from_numpy(B_np.T.copy()).to(device).t()
    dC = torch.empty((N, M), dtype=torch.float64, device=device).t()
    mp, np_, kp = oz.ozaki2_plane_dims(M, N, K)
    rowexp = torch.empty(M, dtype=torch.int32, device=device)
    colexp = torch.empty(N, dtype=torch.int32, device=device)
    Ap = torch.empty((S, mp, kp), dtype=torch.int16, device=device)
    Bp = torch.empty((S, np_, kp), dtype=torch.int16, device=device)
    Cr = torch.empty((S, np_, mp), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    ptr = lambda t: t.data_ptr()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        # steps a1 + a2 (ozaki2_scale_split: B's one-pass exponents and split, then A's exponent
        # pass and split), the GEMM, the CRT
        rc = lib.ozaki2_scale_split(M, N, K, ptr(dA), M, ptr(dB), K, S, ptr(rowexp), ptr(colexp), ptr(Ap), ptr(Bp),
                                    sh)
        if ev:
            ev[1].record(stream)
            ev[2].record(stream)
        rc |= lib.ozaki2_residue_gemm(M, N, K, S, ptr(Ap), ptr(Bp), ptr(Cr), sh)
        if ev:
            ev[3].record(stream)
        rc |= lib.ozaki2_crt(M, N, K, S, ptr(Cr), ptr(rowexp), ptr(colexp), ptr(dC), M, sh)
        if ev:
            ev[4].record(stream)
        if rc:
            raise RuntimeError(f"ozaki call failed: {rc}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    clk = clocks.stop()
    status = oz.ozaki_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    elapsed_ms = start.elapsed_time(end)
    phase_ms = np.zeros(4)
    for e in evs:
        for p in range(4):
            phase_ms[p] += e[p].elapsed_time(e[p + 1])
    phase_ms /= args.steps
    job_ms = reduce_max(elapsed_ms, world, device)
    flops = 2.0 * M * N * K
    value = job_value(world, flops, args.steps, job_ms)

    # ---- roofline of the dominant kernel (the residue GEMM), per launch
    gemm_ms = phase_ms[2]
    int_ops = S * 2.0 * M * N * K
    peak_t = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    achieved = int_ops / (gemm_ms * 1e-3) / 1e12
    traffic = gemm_traffic_bytes()
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                "frac": achieved / peak_t, "traffic": traffic,
                "kernel": "oz::residue_gemm_kernel (s x 2mnk exact integer products on tcgen05 BF16)",
                "peak_source": f"{peak_src} bf16 dense, sustained (kernel timed inside a long step)"}
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    split_bytes = 8.0 * (M * K + K * N) + 2.0 * S * (mp * kp + np_ * kp)
    phases = {
        "scale_split_ms": phase_ms[0], "gemm_ms": phase_ms[2], "crt_ms": phase_ms[3],
        "phase_note": "scale_split = steps a1 + a2 (ozaki2_scale_split); its HBM fraction counts one read of "
                      "A and B and the planes written",
        "scale_split_hbm_frac": split_bytes / (phase_ms[0] * 1e-3) / 1e9 / hbm,
        "crt_hbm_frac": (S * 1.0 * mp * np_ + 8.0 * M * N) / (phase_ms[3] * 1e-3) / 1e9 / hbm,
        "non_gemm_share": float((phase_ms.sum() - phase_ms[2]) / phase_ms.sum()),
        "gemm_frac_of_b200_int8_spec_4500": achieved / 4500.0,
    }

    # ---- the range-estimation variants ([Ozaki II, §9]) on the same workload
    variants = {}
    if not args.no_variants:
        for name, sc in (("fast", oz.OZ_SCALE_FAST), ("accu", oz.OZ_SCALE_ACCU)):
            nb = oz.ozaki2_exponents_workspace_bytes(M, N, K, sc)
            ews = torch.empty(max(nb, 1), dtype=torch.uint8, device=device)

            def vstep(ev=None):
                if ev:
                    ev[0].record(stream)
                rc = lib.ozaki2_exponents_ex(M, N, K, ptr(dA), M, ptr(dB), K, S, sc, ptr(rowexp), ptr(colexp),
                                             ptr(ews), nb, sh)
                if ev:
                    ev[1].record(stream)
                rc |= lib.ozaki2_split_ex(M, N, K, ptr(dA), M, ptr(dB), K, S, sc, ptr(rowexp), ptr(colexp), ptr(Ap),
                                          ptr(Bp), sh)
                rc |= lib.ozaki2_residue_gemm(M, N, K, S, ptr(Ap), ptr(Bp), ptr(Cr), sh)
                rc |= lib.ozaki2_crt_ex(M, N, K, S, sc, ptr(Cr), ptr(rowexp), ptr(colexp), ptr(dC), M, sh)
                if ev:
                    ev[2].record(stream)
                if rc:
                    raise RuntimeError(f"ozaki {name} call failed: {rc}")

            vstep()
            vev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(3)]
            for e in vev:
                vstep(e)
            torch.cuda.synchronize(device)
            step_ms = float(np.mean([e[0].elapsed_time(e[2]) for e in vev]))
            variants[name] = {"ms_per_step": step_ms, "value": flops / (step_ms * 1e-3) / 1e12, "unit": UNIT,
                              "exponents_ms": float(np.mean([e[0].elapsed_time(e[1]) for e in vev])), "steps": 3}
            del ews

    # ---- the secondary path on its own workload: Scheme I, m = n = k = 4096, 7 slices
    scheme1 = {}
    if not args.no_variants:
        m1 = 4096
        A1, B1 = hpl_like(m1, m1, m1, phi=PHI, seed=SEED)
        dA1 = torch.from_numpy(A1.T.copy()).to(device).t()
        dB1 = torch.from_numpy(B1.T.copy()).to(device).t()
        dC1 = torch.empty((m1, m1), dtype=torch.float64, device=device).t()
        for name in ("rn", "ef", "hybrid"):
            v = oz.OZAKI1_VARIANTS[name]
            ws1 = torch.empty(oz.ozaki1_workspace_bytes_ex(m1, m1, m1, 7, v), dtype=torch.uint8, device=device)

            def s1():
                rc = lib.ozaki1_dgemm_ex_ws(m1, m1, m1, ptr(dA1), m1, ptr(dB1), m1, ptr(dC1), m1, 7, v, ptr(ws1),
                                            ws1.numel(), sh)
                if rc:
                    raise RuntimeError(f"ozaki1 {name} call failed: {rc}")

            s1()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                s1()
            e1.record(stream)
            torch.cuda.synchronize(device)
            ms = e0.elapsed_time(e1) / 5
            scheme1[name] = {"ms_per_call": ms, "value": 2.0 * m1**3 / (ms * 1e-3) / 1e12, "unit": UNIT}
            del ws1
        scheme1["workload"] = "ozaki1_dgemm_ex m=n=k=4096, 7 slices, phi=0.5 (seed 0), 5 calls each"
        del dA1, dB1, dC1

    # ---- end to end through the C ABI with pinned HOST buffers
    hA = torch.from_numpy(A_np.T.copy()).pin_memory()   # column-major A as a (k, m) row-major block
    hB = torch.from_numpy(B_np.T.copy()).pin_memory()
    hC = torch.empty((N, M), dtype=torch.float64).pin_memory()
    e2e_steps = args.steps
    for _ in range(args.warmup):  # the same W warm-up steps as the device-resident loop
        oz.ozaki2_dgemm_host_ptr(M, N, K, hA.data_ptr(), M, hB.data_ptr(), K, hC.data_ptr(), M, S)
    e2e_clocks = ClockSampler(local, "_e2e")
    e2e_clocks.start()
    time.sleep(0.3)
    barrier(world)
    call_ms = []
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        t1 = time.perf_counter()
        oz.ozaki2_dgemm_host_ptr(M, N, K, hA.data_ptr(), M, hB.data_ptr(), K, hC.data_ptr(), M, S)
        call_ms.append(1e3 * (time.perf_counter() - t1))
    e2e_s = reduce_max(time.perf_counter() - t0, world, device)
    barrier(world)
    e2e_clk = e2e_clocks.stop()
    e2e = {"value": world * flops * e2e_steps / e2e_s / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": 8 * (M * K + K * N), "d2h_bytes_per_step": 8 * M * N,
           "api": "ozaki2_dgemm_host (pinned host A, B, C; copies inside the timed region)",
           "steps": e2e_steps,
           "call_ms": {"min": min(call_ms), "median": statistics.median(call_ms), "max": max(call_ms)},
           "clocks": e2e_clk,
           "host_link_gbs": host_link_gbs(hA, hC, device)}

    # ---- context: native FP64 GEMM (cuBLAS through torch) on the same GPU, one call
    context = {}
    if rank == 0 and not args.no_context:
        x = dA.contiguous()
        y = dB.contiguous()
        torch.matmul(x[:2048, :2048], y[:2048, :2048])
        torch.cuda.synchronize(device)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        torch.matmul(x, y)
        s1.record(stream)
        torch.cuda.synchronize(device)
        context["cublas_dgemm_tflops"] = flops / (s0.elapsed_time(s1) * 1e-3) / 1e12
        del x, y
        # cuBLAS INT8 and BF16 GEMMs at 8192^3: the tensor rates an INT8 residue product could
        # use on this GPU against the bf16 path the library uses
        n8 = 8192
        ai = torch.randint(-128, 128, (n8, n8), dtype=torch.int8, device=device)
        bi = torch.randint(-128, 128, (n8, n8), dtype=torch.int8, device=device).t().contiguous().t()
        ab = ai.to(torch.bfloat16)
        bb = bi.to(torch.bfloat16)
        for name, fn in (("cublas_int8_gemm_tops_8192", lambda: torch._int_mm(ai, bi)),
                         ("cublas_bf16_gemm_tflops_8192", lambda: torch.matmul(ab, bb))):
            try:
                fn()
                torch.cuda.synchronize(device)
                s0.record(stream)
                for _ in range(5):
                    fn()
                s1.record(stream)
                torch.cuda.synchronize(device)
                context[name] = 5 * 2.0 * n8**3 / (s0.elapsed_time(s1) * 1e-3) / 1e12
            except RuntimeError as ex:  # an INT8 GEMM the installed cuBLAS lacks
                context[name] = f"unavailable: {ex}"[:120]
        context["cuda"] = torch.version.cuda
        if isinstance(context.get("cublas_int8_gemm_tops_8192"), float):
            # exact INT8-residue products per second of the residue GEMM against cuBLAS's INT8 GEMM
            context["residue_gemm_vs_cublas_int8"] = achieved / context["cublas_int8_gemm_tops_8192"]
        del ai, bi, ab, bb

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": job_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": value / PAGES_GH200_TFLOPS, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"ozaki2_dgemm m=n=k={M} s={S} phi={PHI} (HPL-like, seed {SEED})",
                       "m": M, "n": N, "k": K, "moduli": S, "phi": PHI,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "no flush: inputs (2 GiB each) and planes are far larger than L2"},
            "roofline": roofline, "phases": phases, "e2e": e2e, "scaling_variants": variants,
            "scheme1_4096": scheme1,
            "cpu_baseline": cpu_baseline_measure() if not args.no_cpu_baseline else None,
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clk, "context": context,
            "tensor_path": "residues in bf16 on tcgen05 CTA pairs, exact FP32 accumulation in TMEM over "
                           "chunks of 1024 k, each chunk reduced mod m_t into register residues",
            "vs_baseline_ref": "pages' GH200 Scheme II figure, 80.2 TFLOPS (other hardware)",
            "pages_figures": PAGES_FIGURES,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--oracle-protocol", action="store_true",
                    help="time the CPU oracle at the workload configurations (full or sampled) and exit")
    ap.add_argument("--one-core", action="store_true", help="with --oracle-protocol: one BLAS thread")
    args = ap.parse_args()
    if args.oracle_protocol:
        if args.one_core:
            for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
                if os.environ.get(v) != "1":  # the BLAS reads these when numpy loads: start afresh
                    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
                    return subprocess.run([sys.executable] + sys.argv, env=env).returncode
        return run_oracle_protocol(args.one_core)
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
