"""Run the Scheme II path on one problem size (for profiling and quick timing).

    python -m fp64_gemm_emulation_gb300.run_case --m 4096 --n 4096 --k 4096 --moduli 14 --reps 3

Runs the steps (exponents and split, as one ``ozaki2_scale_split`` call in the uniform
scaling; residue GEMM; CRT) through the C ABI on HPL-like inputs resident on the GPU,
``--reps`` times, and prints per-step CUDA-event times of the last repetition.
"""
from __future__ import annotations

import argparse

import numpy as np


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--m", type=int, default=4096)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--moduli", type=int, default=14)
    ap.add_argument("--phi", type=float, default=0.5)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--scheme", type=int, choices=[1, 2], default=2)
    ap.add_argument("--slices", type=int, default=7)
    ap.add_argument("--scaling", choices=["uniform", "fast", "accu"], default="uniform")
    ap.add_argument("--variant", choices=["rn", "ef", "hybrid"], default="rn", help="Scheme I split/accumulation")
    ap.add_argument("--graph", action="store_true", help="also time the whole call captured in a CUDA graph")
    a = ap.parse_args()
    if a.scheme == 1:
        return run_scheme1(a)

    import torch

    from fp64_gemm_emulation_gb300 import ozaki as oz
    from fp64_gemm_emulation_gb300.inputs import hpl_like

    m, n, k, s = a.m, a.n, a.k, a.moduli
    A, B = hpl_like(m, n, k, phi=a.phi, seed=0)
    dA = torch.from_numpy(A.T.copy()).cuda().t()
    dB = torch.from_numpy(B.T.copy()).cuda().t()
    dC = torch.empty((n, m), dtype=torch.float64, device="cuda").t()
    mp, np_, kp = oz.ozaki2_plane_dims(m, n, k)
    rowexp = torch.empty(m, dtype=torch.int32, device="cuda")
    colexp = torch.empty(n, dtype=torch.int32, device="cuda")
    Ap = torch.empty((s, mp, kp), dtype=torch.int16, device="cuda")
    Bp = torch.empty((s, np_, kp), dtype=torch.int16, device="cuda")
    Cr = torch.empty((s, np_, mp), dtype=torch.uint8, device="cuda")
    sc = oz.SCALINGS[a.scaling]
    nb = oz.ozaki2_exponents_workspace_bytes(m, n, k, sc)
    ews = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    lib, st = oz._lib, torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for _ in range(a.reps):
        ev[0].record()
        if sc == oz.OZ_SCALE_UNIFORM:  # steps a1 + a2 together (timed as "split"; "exponents" is 0)
            rc = 0
            ev[1].record()
            rc |= lib.ozaki2_scale_split(m, n, k, p(dA), m, p(dB), k, s, p(rowexp), p(colexp), p(Ap), p(Bp), st)
        else:
            rc = lib.ozaki2_exponents_ex(m, n, k, p(dA), m, p(dB), k, s, sc, p(rowexp), p(colexp), p(ews), nb, st)
            ev[1].record()
            rc |= lib.ozaki2_split_ex(m, n, k, p(dA), m, p(dB), k, s, sc, p(rowexp), p(colexp), p(Ap), p(Bp), st)
        ev[2].record()
        rc |= lib.ozaki2_residue_gemm(m, n, k, s, p(Ap), p(Bp), p(Cr), st)
        ev[3].record()
        rc |= lib.ozaki2_crt_ex(m, n, k, s, sc, p(Cr), p(rowexp), p(colexp), p(dC), m, st)
        ev[4].record()
        if rc:
            raise SystemExit(f"ozaki call failed: {rc}")
    torch.cuda.synchronize()
    status = oz.ozaki_get_device_status()
    t = [ev[i].elapsed_time(ev[i + 1]) for i in range(4)]
    if sc == oz.OZ_SCALE_UNIFORM:  # steps a1 + a2 ran as one call
        names, t = ["scale_split", "residue_gemm", "crt"], [t[0] + t[1], t[2], t[3]]
    else:
        names = ["exponents", "split", "residue_gemm", "crt"]
    tg = t[names.index("residue_gemm")]
    print(f"{m}x{n}x{k} s={s} {a.scaling}: " + ", ".join(f"{nm} {x:.3f} ms" for nm, x in zip(names, t))
          + f"; gemm {s * 2.0 * m * n * k / (tg * 1e-3) / 1e12:.1f} TFLOP/s; status {status}")
    if status:
        raise SystemExit(1)
    if a.graph:
        time_graph(oz, dA, dB, s, a.scaling, m, n, k)
    return np.float64(sum(t))


def time_graph(oz, dA, dB, s, scaling, m, n, k, reps=50):
    """Mean time of the whole Scheme II call per launch: eager vs replayed from a CUDA graph."""
    import torch

    C = torch.empty((n, m), dtype=torch.float64, device="cuda").t()
    ws = torch.empty(oz.ozaki2_workspace_bytes_ex(m, n, k, s, scaling), dtype=torch.uint8, device="cuda")
    oz.ozaki2_dgemm_ex_ws(dA, dB, s, scaling, ws, C=C)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        oz.ozaki2_dgemm_ex_ws(dA, dB, s, scaling, ws, C=C)
    out = {}
    for name, fn in (("eager", lambda: oz.ozaki2_dgemm_ex_ws(dA, dB, s, scaling, ws, C=C)), ("graph", g.replay)):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / reps
    print(f"{m}x{n}x{k} s={s} {scaling}: whole call eager {out['eager'] * 1e3:.1f} us, "
          f"CUDA graph {out['graph'] * 1e3:.1f} us per call ({2.0 * m * n * k / (out['graph'] * 1e-3) / 1e12:.2f} TFLOPS)")


def run_scheme1(a):
    """Scheme I: RN split, the s(s+1)/2 exact slice products, fixed-order FP64 sum."""
    import torch

    from fp64_gemm_emulation_gb300 import ozaki as oz
    from fp64_gemm_emulation_gb300.inputs import hpl_like

    m, n, k, s = a.m, a.n, a.k, a.slices
    v = oz.OZAKI1_VARIANTS[a.variant]
    A, B = hpl_like(m, n, k, phi=a.phi, seed=0)
    dA = torch.from_numpy(A.T.copy()).cuda().t()
    dB = torch.from_numpy(B.T.copy()).cuda().t()
    dC = torch.empty((n, m), dtype=torch.float64, device="cuda").t()
    mp, np_, kp = oz.ozaki2_plane_dims(m, n, k)
    npairs = s * (s + 1) // 2
    nbatch = oz.ozaki1_num_batches(s, k, v)
    Ap = torch.empty((s, mp, kp), dtype=torch.int16, device="cuda")
    Bp = torch.empty((s, np_, kp), dtype=torch.int16, device="cuda")
    Ae = torch.empty((s, m), dtype=torch.int32, device="cuda")
    Be = torch.empty((s, n), dtype=torch.int32, device="cuda")
    P = torch.empty((npairs, np_, mp), dtype=torch.int32, device="cuda")
    nb = oz.ozaki1_split_scratch_bytes_ex(m, n, k, v)
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    lib, st = oz._lib, torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(a.reps):
        ev[0].record()
        rc = lib.ozaki1_split_ex(m, n, k, p(dA), m, p(dB), k, s, v, p(Ap), p(Bp), p(Ae), p(Be), p(scratch), nb, st)
        ev[1].record()
        rc |= lib.ozaki1_slice_gemm_ex(m, n, k, s, v, p(Ap), p(Bp), p(P), st)
        ev[2].record()
        rc |= lib.ozaki1_accumulate_ex(m, n, k, s, v, p(P), p(Ae), p(Be), p(dC), m, st)
        ev[3].record()
        if rc:
            raise SystemExit(f"ozaki1 call failed: {rc}")
    torch.cuda.synchronize()
    status = oz.ozaki_get_device_status()
    t = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    print(f"scheme I {a.variant} {m}x{n}x{k} s={s} ({npairs} products, {nbatch} FP64 terms): split {t[0]:.3f} ms, slice_gemm {t[1]:.3f} ms, "
          f"accumulate {t[2]:.3f} ms; gemm {npairs * 2.0 * m * n * k / (t[1] * 1e-3) / 1e12:.1f} TFLOP/s; "
          f"emulated {2.0 * m * n * k / (sum(t) * 1e-3) / 1e12:.1f} TFLOPS; status {status}")
    if status:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
