#!/usr/bin/env python3
"""Throughput of the Roe finite-volume shallow-water step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload pulses8192|hills2048|dam128|interface2048|tri1024|tri1024_1l|
                                flood2048]
                    [--precision 32|64] [--entropy-fix]

One "step" is one explicit time step of the IR-Roe scheme over the whole
domain: edge fluxes with the bathymetry source, per-cell accumulation, the
global CFL dt reduced on the device, and the update of the state (one layer
with pollutant: one fused kernel launch; two layers on a grid: flux pass and
update; triangles: edge, gather and update kernels).  The default workload
is the 8192 x 8192 fp32 grid of seeded Gaussian hills and surface pulses with
small random velocities (2.4 GB of state per step, far beyond the 129 MB L2).

Prints one JSON line on rank 0.  ``value`` is cell-updates per second over all
ranks (Mcell-updates/s), timed with CUDA events on the stream the kernels run
on, inputs resident in HBM.  ``e2e`` is the same metric through the C ABI with
host buffers (pinned): every step uploads the state, steps once and reads the
state back.  ``roofline`` is that of the dominant kernel (the largest share
of device time, per-kernel CUDA events through swe_set_timing): algorithmic
bytes per launch against the measured HBM copy bandwidth, or algorithmic
flops against the FP32/FP64 pipe peak where the kernel is arithmetic-bound.  ``cpu_baseline`` times the fp64 CPU oracle on a bounded sample of
the same workload on one host core.

Several GPUs run independent replicas (the step has no exchange that would
shard across GPUs here): weak scaling, max time over ranks.
``--impl reference`` times the oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "cell-updates/s (Mcell-steps/s) of the Roe FV step; achieved HBM GB/s vs peak"
UNIT = "Mcell-updates/s"
BYTES_PER_CELL = {32: 36, 64: 72}   # h, qx, qy, hC, H read; h, qx, qy, hC written
# Floating-point operations of one two-layer edge flux, counted from its
# formulas (an add or a multiply 1, an FMA 2; square roots, reciprocals and
# reciprocal square roots not counted): 93 outside the root iterations and
# P^- d (Roe averages 30, rc 2, safe starts and tolerance 13, inner-pair set-up
# 24, fluctuation 16, 2 u_k 2, results 6), 28 per outer Newton iteration
# (two roots x 14), 28 per inner one, and 30 per wave of P^- d =
# sum_k w_k alpha_k K_k.  Only the waves with l_k < 0 (w_k != 0) are needed;
# on these workloads every edge is subcritical in both wave families
# (l1 < l2 < 0 < l3 < l4), so 2 waves.  The outer iteration stops once every
# edge of the warp has converged: on the interface dam break and the triangle
# workload it takes 2.01 iterations per edge in fp32 and 3.01 in fp64
# (counted on the GPU with an instrumented build); the inner one runs 2.
# In fp64 each reciprocal is a hardware seed refined by two Newton steps of
# two FMAs each (8 flops, counted): per edge 2 for the Roe velocities, 2 per
# outer and 2 per inner iteration, 1 for 1/c1^2 and 1 per wave; in fp32 they
# are single MUFU instructions (not counted).
FLOPS_EDGE_2L_BASE, FLOPS_PER_WAVE_2L, WAVES_2L = 93, 30, 2
RCP_FLOPS_FP64 = 8
RCP_PER_EDGE_2L_FP64 = 2 + 2 * 3.01 + 2 * 2 + 1 + WAVES_2L
FLOPS_PER_EDGE_2L = {
    32: FLOPS_EDGE_2L_BASE + FLOPS_PER_WAVE_2L * WAVES_2L + 28 * 2.01 + 28 * 2,
    64: FLOPS_EDGE_2L_BASE + FLOPS_PER_WAVE_2L * WAVES_2L + 28 * 3.01 + 28 * 2
        + RCP_FLOPS_FP64 * RCP_PER_EDGE_2L_FP64}
# Per cell-update on a grid: two edges (each edge once; the tiles' halo
# recomputation not counted) plus 25 for the per-cell quantities and the
# residual sums.
FLOPS_PER_CELL_2L = {p: 2 * FLOPS_PER_EDGE_2L[p] + 25 for p in (32, 64)}
# The ALU peaks are measured in every run by libswe's FMA probe
# (swe_probe_fma_rate: independent FFMA / packed FFMA2 / DFMA chains over a
# full wave, CUDA events); these data-sheet figures are used only if the
# probe fails: 152 SMs x 128 FP32 lanes x 2 flops x 2.07 GHz, and the part's
# nominal 1.25 TFLOP/s FP64.
ALU_PEAK_FALLBACK_TFLOPS = {32: 152 * 128 * 2 * 2.07e9 / 1e12, 64: 1.25}
DTYPE_NAME = {32: "f32", 64: "f64"}
CSRC = os.path.join(ROOT, "finite_volume_shallow_gb300", "csrc")
# kernel -> (sources whose concatenation's hash keys its traffic record,
# traffic record); see source_hash()
KERNEL_SOURCES = {
    "cart1_step_kernel": (("swe_cart1.cu", "swe_internal.h"), "cart1_step_traffic.txt"),
    # (swe_fastmath.cuh is used by the fp64 kernels only, which have no
    # traffic record)
    "cart2_march_kernel<plain>": (("swe_cart2.cu", "swe_roe2.cuh", "swe_internal.h"),
                                  "cart2_march_traffic.txt"),
    "cart2_march_kernel<fused>": (("swe_cart2.cu", "swe_roe2.cuh", "swe_internal.h"),
                                  "cart2_march_traffic.txt"),
    "cart2_update_kernel": (("swe_cart2.cu", "swe_roe2.cuh", "swe_internal.h"),
                            "cart2_march_traffic.txt"),
    "wd_speed_kernel": (("swe_wetdry.cu", "swe_internal.h"), "wetdry_traffic.txt"),
    "wd_tile_kernel": (("swe_wetdry.cu", "swe_internal.h"), "wetdry_traffic.txt"),
    "mesh_tile_kernel": (("swe_mesh.cu", "swe_roe2.cuh", "swe_internal.h"), "mesh_traffic.txt"),
    "mesh_update_kernel": (("swe_mesh.cu", "swe_roe2.cuh", "swe_internal.h"),
                           "mesh_traffic.txt"),
}


def source_hash(files):
    """First 16 hex digits of the sha256 of the listed csrc files, concatenated."""
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(CSRC, f), "rb").read())
    return h.hexdigest()[:16]
# Triangle meshes, two layers, per edge: floating-point operations of the
# flux part of the tile kernel, counted from its formulas: the Roe flux above
# (2.0 outer iterations per edge in fp32, 3.0 in fp64 on the triangle
# workload) plus 79 for the rotations into and out of the edge frame, the
# fluctuation terms and the edge-length scaling; one layer 88.  Each edge is
# counted once (the second evaluation of an edge shared by two tiles is not
# counted).  Per cell the tile kernel adds 3 nf + 3 for the sums of its three
# edges, the division by the area and the wave-speed sum.  In fp32 the
# one-layer tile kernel is modelled by its bytes instead: its arithmetic is
# light.
FLOPS_PER_EDGE_MESH = {(2, 32): FLOPS_EDGE_2L_BASE + FLOPS_PER_WAVE_2L * WAVES_2L
                       + 28 * 2.0 + 28 * 2 + 79,
                       (2, 64): FLOPS_EDGE_2L_BASE + FLOPS_PER_WAVE_2L * WAVES_2L
                       + 28 * 3.0 + 28 * 2 + 79
                       + RCP_FLOPS_FP64 * (2 + 2 * 3.0 + 2 * 2 + 1 + WAVES_2L),
                       (1, 64): 88 + RCP_FLOPS_FP64 * 2}
# One layer on a grid: floating-point operations per cell-update of the
# fused step, counted from its formulas (FMA = 2; the 10 reciprocals and
# reciprocal square roots per cell not counted): 36 per edge flux pair in the
# Roe head, 10 in its tail, 18 for the per-cell quantities, 40 for the next
# step's wave speeds, 34 for accumulation, update and checks -> 200 per two
# cells; in fp64 the 4 reciprocals per cell are Newton-refined (8 flops each,
# counted; the 6 reciprocal square roots are CUDA's rsqrt, not counted).
# The fp32 step is bound by HBM; the fp64 one by GB300's FP64 pipe.
FLOPS_PER_CELL_1L = 100 + 4 * RCP_FLOPS_FP64

DESCR = {
    "pulses8192": "8192x8192 Cartesian, dx=10 m, 128 seeded Gaussian hills, 16 surface pulses, "
                  "|u|<=0.1 m/s, pollutant per 16x16 block, reflective walls",
    "hills2048": "2048x2048 Cartesian, dx=10 m, 8 seeded Gaussian hills, 3 surface bumps, "
                 "q=0, pollutant per 16x16 block, reflective walls",
    "dam128": "128x128 Cartesian, dx=1 m, circular dam break, flat bottom, reflective walls",
    "interface2048": "two layers, 2048x2048 Cartesian, dx=10 m, flat bottom 10 m, interface "
                     "dam break h1=6/4 m at x=L/2, r=0.98, at rest, reflective walls",
    "tri1024": "two layers on 1024x1024 unit squares split into 2,097,152 triangles, interior "
               "vertices jittered by +-0.2, cells shuffled then put in Hilbert order, r=0.98, "
               "8 Gaussian hills, 0.5 m interface bump, at rest, reflective walls",
    "flood2048": "one layer with pollutant and wet/dry fronts, 2048x2048 Cartesian, dx=10 m, "
                 "bed rising 4 m across x plus 64 seeded Gaussian hills (amplitude "
                 "U[0.5,2.5] m), lake at rest at level 0 (about half the domain dry), a disc "
                 "of radius 2048 m raised by 2 m at the centre flooding dry land, "
                 "h_dry=1e-2 m, Harten-Hyman entropy fix, reflective walls",
    "tri1024_1l": "one layer with pollutant on 1024x1024 unit squares split into 2,097,152 "
                  "triangles, interior vertices jittered by +-0.2, cells shuffled then "
                  "put in Hilbert order, 6 Gaussian hills under a 2 m deep surface, 4 surface pulses "
                  "of 0.5 m, |u|<=0.1 m/s per component, pollutant per 4x4 block of squares, "
                  "reflective walls",
}


def kernel_model(kernel, precision, nl, n_cells, n_edges):
    """(bound, algorithmic amount per launch, unit) of one kernel: bytes that
    must cross HBM at least once, or floating-point operations."""
    e = 4 if precision == 32 else 8
    nf = 6 if nl == 2 else 4
    if kernel == "cart1_step_kernel":
        if precision == 64:
            return "alu", FLOPS_PER_CELL_1L * n_cells, "flop"
        return "hbm", BYTES_PER_CELL[precision] * n_cells, "B"
    if kernel == "cart2_march_kernel<plain>":
        return "alu", FLOPS_PER_CELL_2L[precision] * n_cells, "flop"
    if kernel == "cart2_march_kernel<fused>":   # + the fused update, 6 FMAs per cell
        return "alu", (FLOPS_PER_CELL_2L[precision] + 12) * n_cells, "flop"
    if kernel == "cart2_update_kernel":
        return "hbm", 3 * 6 * e * n_cells, "B"
    if kernel == "mesh_tile_kernel" and nl == 1 and precision == 32:
        # light arithmetic: the state and H of every cell read once, its
        # slot references (8 B), 1/|V| and R written; per edge its two cell
        # indices (4 B) and normal and length, once
        return "hbm", ((nf + 1) * e + nf * e + e + 8) * n_cells + (4 + 3 * e) * n_edges, "B"
    if kernel == "mesh_tile_kernel":
        return "alu", (FLOPS_PER_EDGE_MESH[(nl, precision)] * n_edges
                       + (3 * nf + 3) * n_cells), "flop"
    if kernel == "mesh_update_kernel":
        return "hbm", 3 * nf * e * n_cells, "B"
    # wet/dry on a grid: each field crosses HBM once per pass
    if kernel == "wd_speed_kernel":   # h, qx, qy, H read
        return "hbm", 4 * e * n_cells, "B"
    if kernel == "wd_tile_kernel":    # h, qx, qy, hC, H read; h, qx, qy, hC written
        return "hbm", 9 * e * n_cells, "B"
    raise KeyError(kernel)


def measure_alu_peaks(S, stream=None, target_ms=100.0):
    """FMA throughput of this GPU, measured now by libswe's probe: FP32 (the
    faster of scalar and packed-pair FMAs) and FP64, in TFLOP/s."""
    out = {}
    try:
        ffma, _ = S.swe_probe_fma_rate(S.PROBE_FFMA, target_ms, stream)
        ffma2, _ = S.swe_probe_fma_rate(S.PROBE_FFMA2, target_ms, stream)
        dfma, _ = S.swe_probe_fma_rate(S.PROBE_DFMA, target_ms, stream)
        out = {32: max(ffma, ffma2) / 1e12, 64: dfma / 1e12, "ffma_tflops": ffma / 1e12,
               "ffma2_tflops": ffma2 / 1e12, "dfma_tflops": dfma / 1e12,
               "source": "measured in this run (swe_probe_fma_rate, CUDA events)"}
    except Exception as e:  # reported, never silent
        out = {32: ALU_PEAK_FALLBACK_TFLOPS[32], 64: ALU_PEAK_FALLBACK_TFLOPS[64],
               "source": f"fallback (data sheet): probe failed: {e}"}
    return out


def host_cpu_info():
    """What the oracle's baseline ran on: the host's core count and model."""
    info = {"os_cpu_count": os.cpu_count()}
    try:
        info["nproc"] = int(subprocess.run(["nproc"], capture_output=True, text=True,
                                           timeout=10).stdout.strip())
    except Exception:
        info["nproc"] = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() in ("Model name", "Architecture", "Vendor ID"):
                info[k.strip().lower().replace(" ", "_")] = v.strip()
    except Exception:
        pass
    return info


def state_fields(I, d):
    """The conserved fields of a workload dict (one or two layers)."""
    return I.fields2_of(d) if d.get("n_layers") == 2 else I.fields_of(d)


def oracle_run(O, d, nx, rows, H, W, nsteps):
    if d.get("n_layers") == 2:
        return O.grid_run2(nx, rows, d["dx"], d["dy"], H, W, d["g"], d["r"], d["cfl"], nsteps)
    return O.grid_run1(nx, rows, d["dx"], d["dy"], H, W, d["g"], d["cfl"], nsteps)


def n_cells_of(d):
    return d["n_cells"] if d.get("mesh") else d["nx"] * d["ny"]


class Sample:
    """A bounded sample of a workload for the CPU oracle: the first rows of a
    grid, or the triangles with the lowest centroids of a mesh (as a walled
    domain of their own), with their initial values."""

    def __init__(self, I, d, cells):
        import numpy as np
        self.d = d
        fields = state_fields(I, d)
        if d.get("mesh"):
            cy = I.tri_centroids(d["xy"], d["tri"])[:, 1]
            sel = np.sort(np.argsort(cy, kind="stable")[:max(1, min(cells, d["n_cells"]))])
            tri = d["tri"][sel]
            used, inv = np.unique(tri, return_inverse=True)
            self.xy = np.ascontiguousarray(d["xy"][used])
            self.tri = np.ascontiguousarray(inv.reshape(-1, 3).astype(np.int32))
            self.cells = len(sel)
            self.H = d["H"][sel]
            self.W = [f[sel] for f in fields]
            self.what = (f"the {self.cells} triangles of lowest centroid of the "
                         f"{d['n_cells']}-triangle mesh as a walled mesh")
        else:
            nx = d["nx"]
            rows = int(max(1, min(d["ny"], cells // nx)))
            sl = slice(0, rows * nx)
            self.rows, self.cells = rows, rows * nx
            self.H = d["H"][sl]
            self.W = [f[sl] for f in fields]
            self.what = (f"rows 0..{rows - 1} of the {d['nx']}x{d['ny']} initial state as a "
                         f"walled {nx}x{rows} grid")

    def run(self, O, nsteps, W=None):
        with O.entropy_fix(self.d.get("entropy_fix", 0)), \
                O.wet_dry(self.d.get("h_dry", 0.0), on=bool(self.d.get("wet_dry", 0))):
            return self._run(O, nsteps, W)

    def _run(self, O, nsteps, W=None):
        d = self.d
        W = self.W if W is None else W
        if d.get("mesh"):
            m = getattr(self, "_mesh", None) or O.tri_mesh(self.xy, self.tri)
            self._mesh = m
            if d.get("n_layers") == 2:
                return O.run2(m, self.H, W, d["g"], d["r"], d["cfl"], nsteps)
            Wf, dts, st, _ = O.run1(m, self.H, W, d["g"], d["cfl"], nsteps)
            return Wf, dts, st
        return oracle_run(O, d, d["nx"], self.rows, self.H, W, nsteps)


def calibrate(O, I, d, cal_cells):
    """Seconds per cell-update of the oracle on this workload."""
    smp = Sample(I, d, cal_cells)
    smp.run(O, 1)   # builds the sample mesh
    t0 = time.perf_counter()
    smp.run(O, 1)
    return (time.perf_counter() - t0) / smp.cells


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="pulses8192", choices=sorted(DESCR))
    p.add_argument("--precision", type=int, choices=[32, 64], default=None)
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--nx", type=int, default=None, help="reduced grid (same recipe)")
    p.add_argument("--ny", type=int, default=None)
    p.add_argument("--entropy-fix", action="store_true",
                   help="the Harten-Hyman entropy fix of the flux")
    p.add_argument("--no-clocks", action="store_true",
                   help="skip the nvidia-smi clock window (profiling runs)")
    a = p.parse_args()
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    if a.steps < 1:
        p.error("--steps must be at least 1")
    return a


def workload_of(I, args):
    d = I.make_workload(args.workload, nx=args.nx, ny=args.ny)
    if args.entropy_fix:
        d["entropy_fix"] = 1
    return d


def workload_name(args, d, precision):
    s = f"{args.workload}: {DESCR[args.workload]}, fp{precision}"
    if d.get("entropy_fix") and args.workload != "flood2048":
        s += ", Harten-Hyman entropy fix"
    return s


def max_over_ranks(x, world):
    """Maximum of a per-rank float over all ranks (the slowest replica sets the
    whole job's time); identity on one rank.  Works with the NCCL process
    group of the GPU runs and with a gloo group on CPU."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, cells_per_rank, steps, seconds):
    """Cell-updates per second of all ranks together (Mcell-updates/s): every
    replica advances its own copy of the workload by `steps` steps."""
    return world * cells_per_rank * steps / seconds / 1e6


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def traffic_per_launch(kernel, precision, workload):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or
    None when the kernel's source changed since it was captured."""
    try:
        srcs, rec = KERNEL_SOURCES[kernel]
        src_hash = source_hash(srcs)
        vals = {}
        for line in open(os.path.join(ROOT, "profiles", rec)):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("source_sha256_16") != src_hash:
            return None
        key = f"bytes_per_launch_{kernel}_{workload}_f{precision}"
        if key not in vals and kernel == "cart1_step_kernel":
            key = f"bytes_per_launch_{workload}_f{precision}"
        return float(vals[key]) if key in vals else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="swe_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        return rows

    @staticmethod
    def summarise(rows, t_marks):
        # rows carry no timestamps; all samples lie in the busy window that
        # brackets the timed steps
        if not rows or isinstance(rows, dict):
            return rows if isinstance(rows, dict) else {"sm_mhz": None, "sm_max_mhz": None,
                                                        "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_median": statistics.median(pw) if pw else None}


def physical_gpu(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


def cpu_baseline(d, budget_s=12.0):
    """The oracle (fp64, one thread) on a bounded sample of the workload."""
    import oracle as O
    from finite_volume_shallow_gb300 import inputs as I

    per_cell = calibrate(O, I, d, 64 * (d.get("nx") or 1024) if not d.get("mesh") else 65536)
    cells = int(max(512, min(n_cells_of(d), budget_s / 4 / per_cell)))
    smp = Sample(I, d, cells)
    steps = max(1, int(budget_s / (per_cell * smp.cells)))
    smp.run(O, 1)
    t0 = time.perf_counter()
    _, dts, st = smp.run(O, steps)
    el = time.perf_counter() - t0
    return {"value": smp.cells * steps / el / 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{smp.what}, {steps} steps, fp64, single thread, {el:.1f} s",
            "cores_note": "cores = threads the oracle used; host lists the box's cores",
            "host": host_cpu_info()}


def run_reference(args, rank, world):
    """Reference arm: the fp64 CPU oracle, timed on the host cores, on a
    bounded sample of the workload per step."""
    if rank != 0:
        return 0
    import oracle as O
    from finite_volume_shallow_gb300 import inputs as I

    d = workload_of(I, args)
    precision = args.precision or d["precision"]
    per_cell = calibrate(O, I, d, 16 * (d.get("nx") or 1024) if not d.get("mesh") else 16384)
    budget = 150.0
    cells = int(max(256, min(n_cells_of(d), budget / ((args.steps + args.warmup) * per_cell))))
    smp = Sample(I, d, cells)
    W, _, st = smp.run(O, args.warmup)
    t0 = time.perf_counter()
    W, _, st = smp.run(O, args.steps, W)
    el = time.perf_counter() - t0
    value = smp.cells * args.steps / el / 1e6
    sample = f"each step: one oracle step over {smp.what} (fp64, single thread)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(args, d, precision),
                   "cells": n_cells_of(d), "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_cpu_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "status": st,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np
    import torch

    from finite_volume_shallow_gb300 import inputs as I
    from finite_volume_shallow_gb300 import swe as S

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    S.load()
    d = workload_of(I, args)
    precision = args.precision or d["precision"]
    npdt = np.float32 if precision == 32 else np.float64
    tdt = torch.float32 if precision == 32 else torch.float64
    n = n_cells_of(d)
    two = d.get("n_layers") == 2
    nl = 2 if two else 1
    fields = [f.astype(npdt) for f in state_fields(I, d)]
    stream = torch.cuda.Stream()
    if d.get("mesh"):
        st = S.swe_create_mesh(d["xy"], d["tri"], d["H"].astype(npdt), fields,
                               precision=precision, g=d["g"], cfl=d["cfl"],
                               stream=stream.cuda_stream, n_layers=nl,
                               pollutant=0 if two else 1, r=d.get("r", 0.0), reorder=1,
                               entropy_fix=d.get("entropy_fix", 0))
    else:
        st = S.swe_create_grid(d["nx"], d["ny"], d["dx"], d["dy"], d["H"].astype(npdt), fields,
                               precision=precision, g=d["g"], cfl=d["cfl"],
                               stream=stream.cuda_stream, n_layers=nl,
                               pollutant=0 if two else 1, r=d.get("r", 0.0),
                               entropy_fix=d.get("entropy_fix", 0),
                               wet_dry=d.get("wet_dry", 0), h_dry=d.get("h_dry", 0.0))
    info = S.swe_get_info(st)

    # warm-up (also gives a step-time estimate for the busy window below)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    S.swe_run(st, args.warmup)
    torch.cuda.synchronize()
    est = (time.perf_counter() - w0) / args.warmup

    # timed region, inside a busy window sampled by nvidia-smi: about 0.5 s of
    # the same steps runs untimed right before it so the clock record covers
    # the kernel even when the timed region is shorter than the sampling period
    sampler = ClockSampler(physical_gpu(local))
    if not args.no_clocks:
        sampler.start()
        pre = int(min(5000, 0.5 / max(est, 1e-6)))
        S.swe_run(st, pre)
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    S.swe_run(st, args.steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    # the same K steps again with CUDA events between the kernels of every
    # step (swe_set_timing, on the kernels' stream): each kernel's average
    # launch duration for the roofline.  Kept out of `value`, which the
    # extra event records would slow by about 1 %.
    S.swe_set_timing(st, True)
    S.swe_run(st, args.steps)
    ktimes = S.swe_get_timing(st)
    S.swe_set_timing(st, False)
    torch.cuda.synchronize()
    if args.no_clocks:
        clocks = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled (--no-clocks)"]}
    else:
        clocks = ClockSampler.summarise(sampler.stop(), None)

    ms_max = max_over_ranks(ms, world)
    ms_per_step = ms_max / args.steps
    value = whole_job_rate(world, n, args.steps, ms_max / 1e3)

    # end to end through the C ABI with pinned host buffers
    ke = max(3, min(args.e2e_steps, args.steps))
    host = [torch.from_numpy(f).pin_memory() for f in S.swe_get_state(st)[0]]
    S.swe_set_state(st, host, 0.0)
    S.swe_step(st, d["cfl"])
    S.swe_get_state(st, out=host)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(ke):
        S.swe_set_state(st, host, 0.0)
        S.swe_step(st, d["cfl"])
        S.swe_get_state(st, out=host)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world)
    esz = 4 if precision == 32 else 8
    nf = len(fields)
    e2e = {"value": whole_job_rate(world, n, ke, e2e_s), "unit": UNIT, "steps": ke,
           "h2d_bytes_per_step": nf * n * esz + 8, "d2h_bytes_per_step": nf * n * esz + 8 + 8 + 4,
           "api": "swe_set_state + swe_step + swe_get_state, pinned host buffers"}
    S.swe_destroy(st)

    peak, peak_kind = load_peaks()
    ktimes = {k: v for k, v in ktimes.items() if v[0] > 0}
    # the FMA probe runs only when a kernel of this workload is bound by
    # arithmetic (it would otherwise only add launches to a profile)
    if any(kernel_model(k, precision, nl, n, info["n_edges"])[0] == "alu" for k in ktimes):
        alu = measure_alu_peaks(S, stream.cuda_stream)
    else:
        alu = {"source": "not measured: every kernel of this workload is bound by HBM"}
    kernels = {}
    for name, (launches, kms) in ktimes.items():
        bound, amount, unit = kernel_model(name, precision, nl, n, info["n_edges"])
        avg = kms / max(launches, 1)
        rate = amount / (avg / 1e3)
        if unit == "B":
            kernels[name] = {"bound": "hbm", "achieved": rate / 1e9, "peak": peak, "unit": "GB/s",
                             "frac": rate / 1e9 / peak, "peak_source": peak_kind,
                             "algorithmic_bytes_per_launch": amount}
        else:
            pk = alu[precision]
            kernels[name] = {"bound": "alu", "achieved": rate / 1e12, "peak": pk,
                             "unit": "TFLOP/s", "frac": rate / 1e12 / pk,
                             "peak_source": alu["source"],
                             "algorithmic_flops_per_launch": amount}
        kernels[name].update({"kernel": name, "launches": launches, "ms_per_launch": avg,
                              "timing": "CUDA events between the kernels of each of K "
                                        "further steps, right after the timed region",
                              "share": kms / max(sum(v[1] for v in ktimes.values()), 1e-30),
                              "traffic": traffic_per_launch(
                                  name, precision,
                                  args.workload + ("_efix" if d.get("entropy_fix") else ""))})
    dominant = max(ktimes, key=lambda k: ktimes[k][1])
    roof = dict(kernels[dominant])
    # the whole step against HBM when every kernel of it is bound by HBM: the
    # algorithmic bytes of all its kernels over the measured step time (the
    # per-kernel times come from a run with events between the kernels,
    # which stops consecutive launches overlapping)
    if len(kernels) > 1 and all(v["bound"] == "hbm" for v in kernels.values()):
        step_bytes = sum(v["algorithmic_bytes_per_launch"] * v["launches"] for v in kernels.values()) \
            / max(ktimes[dominant][0], 1)
        achieved = step_bytes / (ms_per_step / 1e3) / 1e9
        roof["step"] = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak, "algorithmic_bytes_per_step": step_bytes,
                        "timing": "ms_per_step of the timed region"}
    roof["other_kernels"] = {k: {kk: v[kk] for kk in ("bound", "achieved", "unit", "frac",
                                                      "ms_per_launch", "share")}
                             for k, v in kernels.items() if k != dominant}

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(d)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_NAME[precision], "data": "synthetic",
            "config": {"workload": workload_name(args, d, precision)
                                   + (f", reduced to {args.nx or d.get('nx')}x"
                                      f"{args.ny or d.get('ny')}" if args.nx or args.ny
                                      else ""),
                       "cells": n, "edges": info["n_edges"], "nx": d.get("nx"),
                       "ny": d.get("ny"), "parallelism": "replicas",
                       "l2": "inputs larger than L2 (no flush needed)"
                             if info["device_bytes"] > 129e6 else "inputs fit in L2 (no flush)",
                       "device_bytes": info["device_bytes"],
                       "launch": ({"tiles": info["bands"], "blocks": info["segments"],
                                   "warps_per_block": info["warps_per_block"]}
                                  if d.get("mesh") else
                                  {"bands": info["bands"], "segments": info["segments"],
                                   "warps_per_block": info["warps_per_block"]})},
            "e2e": e2e, "roofline": roof, "cpu_baseline": base, "clocks": clocks,
            "alu_peaks": {k: v for k, v in alu.items() if isinstance(k, str)},
            "gpu_launches": sum(v[0] for v in ktimes.values()),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
