#!/usr/bin/env python3
"""Benchmark of the GB300 field sweeps.

One step is one pass of every sweep on the hot path, each on its seeded
synthetic workload, all inputs resident in HBM:
  * diffusion, 8192 x 8192, alpha 0.1, 200 steps, FP32 and FP64 (interior
    uniform [0,1), zero edges)        -- the headline workload;
  * WENO pack x, y, z: 8 fields of 201^3 cells + 3 ghost layers (207^3);
  * flux difference x, y, z: nv 8 on 201^3 cells;
  * the 2D multi-variable sequence on 4800 x 1200 cells, nv 7, ghost 2:
    pack x, pack y, flux x, flux y, repeated 100 times.

``value`` is achieved HBM GB/s: the step's compulsory bytes (one read of every
input element and one write of every output element per sweep) over the
step's device time, summed over all ranks.  Every working set exceeds the
129 MB L2, so no flush is needed between iterations.

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]``;
under torchrun each rank runs the whole workload on its own GPU (independent
replicas, weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

from finite_volume_field_gb300 import inputs  # noqa: E402

METRIC = "achieved HBM GB/s and Gcell-var/s per sweep, % of GB300 HBM roofline"
WORKLOAD = ("2D 5-point diffusion 8192x8192, alpha 0.1, 200 steps, FP32 and FP64 "
            "(plus one pass of each other hot-path sweep: WENO pack x/y/z nv=8 207^3, "
            "flux difference x/y/z nv=8 201^3, 4800x1200 nv=7 pack+flux sequence x100)")
FALLBACK_HBM_GBS = 6800.0
FP64_NOMINAL_TFLOPS = 1.25   # nominal FP64 rate of the part (FMA = 2 flops): context only
# Algorithmic FP64 flops per output element of the FP64 arithmetic sweeps.
FP64_FLOPS = {"diffuse_fp64": 7, "rhs_x": 2, "rhs_y": 2, "rhs_z": 2}
# FP64-unit instructions per element as built: the diffusion update has 6
# (3 sums, the fused s - 4c, the multiply, the add), and the neighbour sum
# runs on the integer pipes (the few cells whose operands the fixed-point sum
# declines, next to the zero edges, add about 0.1); the flux difference has a
# subtraction and a multiplication, and the multiplication of three variables
# in four runs on the integer pipes.
FP64_INSTR = {"diffuse_fp64": 3, "rhs_x": 1.25, "rhs_y": 1.25, "rhs_z": 1.25}

# ---------------------------------------------------------------------------
# Workload definition (sizes, compulsory bytes, cell-var counts)
# ---------------------------------------------------------------------------

DIFF_N, DIFF_STEPS = 8192, 200
PACK_EXT, PACK_G, PACK_NV = (201, 201, 201), 3, 8
RHS_EXT, RHS_NV = (201, 201, 201), 8
SEQ_EXT, SEQ_G, SEQ_NV, SEQ_REPS = (4800, 1200, 1), 2, 7, 100


def _prod(t):
    p = 1
    for x in t:
        p *= int(x)
    return p


def pack_extents(ext, g, d):
    N = inputs.stored_extents(ext, g)
    return [(N[0], ext[1], ext[2]), (N[1], ext[0], ext[2]), (N[2], ext[1], ext[0])][d]


def pack_bytes(ext, g, nv, d):
    return 16 * _prod(pack_extents(ext, g, d)) * nv


def rhs_bytes(ext, nv, d):
    f = list(ext)
    f[d] += 1
    return 8 * (_prod(f) * nv + _prod(ext) * nv + ext[d])


def rows():
    """Per sweep: compulsory bytes, cell-var updates and launches per step."""
    r = {}
    cells = (DIFF_N - 2) ** 2
    for name, p in (("diffuse_fp32", 4), ("diffuse_fp64", 8)):
        r[name] = dict(bytes=DIFF_STEPS * 2 * DIFF_N * DIFF_N * p, cellvars=DIFF_STEPS * cells,
                       launches=DIFF_STEPS, per_launch_bytes=2 * DIFF_N * DIFF_N * p,
                       per_launch_cells=cells)
    for d, ax in enumerate("xyz"):
        b = pack_bytes(PACK_EXT, PACK_G, PACK_NV, d)
        cv = _prod(pack_extents(PACK_EXT, PACK_G, d)) * PACK_NV
        r[f"pack_{ax}"] = dict(bytes=b, cellvars=cv, launches=1, per_launch_bytes=b,
                               per_launch_cells=cv)
    for d, ax in enumerate("xyz"):
        b = rhs_bytes(RHS_EXT, RHS_NV, d)
        cv = _prod(RHS_EXT) * RHS_NV
        r[f"rhs_{ax}"] = dict(bytes=b, cellvars=cv, launches=1, per_launch_bytes=b,
                              per_launch_cells=cv)
    b = (pack_bytes(SEQ_EXT, SEQ_G, SEQ_NV, 0) + pack_bytes(SEQ_EXT, SEQ_G, SEQ_NV, 1)
         + rhs_bytes(SEQ_EXT, SEQ_NV, 0) + rhs_bytes(SEQ_EXT, SEQ_NV, 1))
    cv = (_prod(pack_extents(SEQ_EXT, SEQ_G, 0)) + _prod(pack_extents(SEQ_EXT, SEQ_G, 1))
          + 2 * _prod(SEQ_EXT)) * SEQ_NV
    r["seq2d"] = dict(bytes=SEQ_REPS * b, cellvars=SEQ_REPS * cv, launches=4 * SEQ_REPS,
                      per_launch_bytes=b / 4, per_launch_cells=cv / 4)
    return r


# ---------------------------------------------------------------------------
# Host inputs (seeded; shared recipe with the tests)
# ---------------------------------------------------------------------------

def host_inputs():
    s2, s3, s4, s5 = (inputs.config_seed(k) for k in (2, 3, 4, 5))
    h = {}
    h["u32"] = inputs.diffusion_field(DIFF_N, DIFF_N, np.float32, seed=s2, stream=0)
    h["u64"] = inputs.diffusion_field(DIFF_N, DIFF_N, np.float64, seed=s2, stream=1)
    h["pack_fields"] = inputs.normal_fields(s3, PACK_NV, PACK_EXT, PACK_G)
    h["rhs_flux"] = [inputs.face_fluxes(s4, RHS_NV, RHS_EXT, d) for d in range(3)]
    h["rhs_invd"] = [inputs.inverse_spacing(s4, RHS_EXT[d], stream=200 + d) for d in range(3)]
    h["seq_fields"] = inputs.multivar_fields_2d(s5, SEQ_EXT, SEQ_G)
    h["seq_flux"] = [inputs.face_fluxes(s5, SEQ_NV, SEQ_EXT, d) for d in range(2)]
    h["seq_invd"] = [inputs.inverse_spacing(s5, SEQ_EXT[d], stream=200 + d) for d in range(2)]
    return h


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------

class Sweeps:
    """Device buffers of one rank and the enqueueing of one step."""

    def __init__(self, torch, host, device, stream):
        self.t = torch
        self.dev = device
        self.stream = stream
        f64 = torch.float64
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
        self.inputs = {}   # name -> device tensor that a host->device copy refills
        self.outputs = {}  # name -> device tensor read back after a step
        self.u32, self.u64 = d(host["u32"]), d(host["u64"])
        self.v32, self.v64 = torch.zeros_like(self.u32), torch.zeros_like(self.u64)
        self.inputs.update(u32=self.u32, u64=self.u64)
        self.outputs.update(u32=self.u32, u64=self.u64)   # 200 steps: result back in u
        self.pack_fields = [d(f) for f in host["pack_fields"]]
        for i, f in enumerate(self.pack_fields):
            self.inputs[f"pack_field{i}"] = f
        self.pack_out = []
        for k in range(3):
            o = torch.empty(_prod(pack_extents(PACK_EXT, PACK_G, k)) * PACK_NV, dtype=f64,
                            device=device)
            self.pack_out.append(o)
            self.outputs[f"pack_out{k}"] = o
        self.rhs_flux = [d(f) for f in host["rhs_flux"]]
        self.rhs_invd = [d(w) for w in host["rhs_invd"]]
        self.rhs_out = [torch.empty(_prod(RHS_EXT) * RHS_NV, dtype=f64, device=device)
                        for _ in range(3)]
        for k in range(3):
            self.inputs[f"rhs_flux{k}"] = self.rhs_flux[k]
            self.inputs[f"rhs_invd{k}"] = self.rhs_invd[k]
            self.outputs[f"rhs_out{k}"] = self.rhs_out[k]
        self.seq_fields = [d(f) for f in host["seq_fields"]]
        self.seq_flux = [d(f) for f in host["seq_flux"]]
        self.seq_invd = [d(w) for w in host["seq_invd"]]
        self.seq_px = torch.empty(_prod(pack_extents(SEQ_EXT, SEQ_G, 0)) * SEQ_NV, dtype=f64,
                                  device=device)
        self.seq_py = torch.empty(_prod(pack_extents(SEQ_EXT, SEQ_G, 1)) * SEQ_NV, dtype=f64,
                                  device=device)
        self.seq_rx = torch.empty(_prod(SEQ_EXT) * SEQ_NV, dtype=f64, device=device)
        self.seq_ry = torch.empty_like(self.seq_rx)
        for i, f in enumerate(self.seq_fields):
            self.inputs[f"seq_field{i}"] = f
        for k in range(2):
            self.inputs[f"seq_flux{k}"] = self.seq_flux[k]
            self.inputs[f"seq_invd{k}"] = self.seq_invd[k]
        self.outputs.update(seq_px=self.seq_px, seq_py=self.seq_py, seq_rx=self.seq_rx,
                            seq_ry=self.seq_ry)
        self.seq_graph = None         # CUDA graph of the 2D sequence (capture_seq_graph)
        self.seq_graph_launches = 0   # library kernels in that graph
        self.graph_launches = 0       # kernels launched by graph replays so far

    def capture_seq_graph(self):
        """Capture the 2D multi-variable sequence (100 repetitions of pack x,
        pack y, flux x, flux y) into a CUDA graph, once, through the same
        library calls; later steps replay it.  Returns the launches in it."""
        from finite_volume_field_gb300 import api
        self.stages()                 # defines self._seq_launch
        g = self.t.cuda.CUDAGraph()
        n0 = api.launch_count()
        with self.t.cuda.graph(g, stream=self.stream, capture_error_mode="relaxed"):
            self._seq_launch(self.t.cuda.current_stream())
        self.seq_graph_launches = api.launch_count() - n0
        self.seq_graph = g
        return self.seq_graph_launches

    def stages(self):
        """The step as an ordered list of (name, input keys, output keys,
        enqueue(stream, mark)) -- the unit of the end-to-end pipeline."""
        from finite_volume_field_gb300 import api

        def diff32(s, mark):
            mark("diffuse_fp32", 0)
            api.diffuse2d_step(self.u32, self.v32, DIFF_N, DIFF_N, 0.1, DIFF_STEPS, api.FVF_FP32, s)
            mark("diffuse_fp32", 1)

        def diff64(s, mark):
            mark("diffuse_fp64", 0)
            api.diffuse2d_step(self.u64, self.v64, DIFF_N, DIFF_N, 0.1, DIFF_STEPS, api.FVF_FP64, s)
            mark("diffuse_fp64", 1)

        def pack(s, mark):
            for k, ax in enumerate("xyz"):
                mark(f"pack_{ax}", 0)
                api.weno_pack(self.pack_fields, PACK_NV, PACK_EXT, PACK_G, k, self.pack_out[k], s)
                mark(f"pack_{ax}", 1)

        def rhs(s, mark):
            for k, ax in enumerate("xyz"):
                mark(f"rhs_{ax}", 0)
                api.advect_rhs(self.rhs_flux[k], self.rhs_invd[k], RHS_NV, RHS_EXT, k,
                               self.rhs_out[k], s)
                mark(f"rhs_{ax}", 1)

        def seq_launch(s):
            for _ in range(SEQ_REPS):
                api.weno_pack(self.seq_fields, SEQ_NV, SEQ_EXT, SEQ_G, 0, self.seq_px, s)
                api.weno_pack(self.seq_fields, SEQ_NV, SEQ_EXT, SEQ_G, 1, self.seq_py, s)
                api.advect_rhs(self.seq_flux[0], self.seq_invd[0], SEQ_NV, SEQ_EXT, 0, self.seq_rx,
                               s)
                api.advect_rhs(self.seq_flux[1], self.seq_invd[1], SEQ_NV, SEQ_EXT, 1, self.seq_ry,
                               s)

        def seq(s, mark):
            mark("seq2d", 0)
            if self.seq_graph is not None:
                # the 400 launches of the sequence as one CUDA graph (captured
                # once from the same calls); replayed on the current stream
                with self.t.cuda.stream(s):
                    self.seq_graph.replay()
                self.graph_launches += self.seq_graph_launches
            else:
                seq_launch(s)
            mark("seq2d", 1)

        self._seq_launch = seq_launch

        keys_in, keys_out = list(self.inputs), list(self.outputs)
        pick = lambda keys, pre: [k for k in keys if k.startswith(pre)]  # noqa: E731
        return [
            ("diffuse_fp32", ["u32"], ["u32"], diff32),
            ("diffuse_fp64", ["u64"], ["u64"], diff64),
            ("pack", pick(keys_in, "pack_"), pick(keys_out, "pack_"), pack),
            ("rhs", pick(keys_in, "rhs_"), pick(keys_out, "rhs_"), rhs),
            ("seq2d", pick(keys_in, "seq_"), pick(keys_out, "seq_"), seq),
        ]

    def step(self, ev=None, hook=None):
        """Enqueue one step on self.stream; ev maps row name -> (start, end)
        CUDA events recorded around that row; hook(name, 0/1) is called at
        the same points."""
        s = self.stream

        def mark(name, which):
            if ev is not None:
                ev[name][which].record(s)
            if hook is not None:
                hook(name, which)

        for _, _, _, enqueue in self.stages():
            enqueue(s, mark)


def e2e_pipeline(torch, sets, pinned_in, pinned_out, streams, steps):
    """End-to-end steps through the public API with host buffers: each
    stage's inputs are copied from pinned host memory on the copy-in stream,
    the stage runs on the compute stream once its inputs have arrived, and its
    outputs are copied back on the copy-out stream once it has finished.
    Consecutive steps alternate between two device buffer sets, so a stage's
    copy-in for the next step never overwrites buffers still being read; a
    set is refilled only after its previous outputs have been copied out.
    Returns the device time of the whole run in ms (events: first copy-in
    to last copy-out)."""
    cin, comp, cout = streams
    nothing = lambda name, which: None  # noqa: E731
    freed = [dict(), dict()]   # set -> stage -> event after its outputs left
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cin)
    for k in range(steps):
        sw = sets[k % 2]
        for name, ins, outs, enqueue in sw.stages():
            if name in freed[k % 2]:
                cin.wait_event(freed[k % 2][name])
            with torch.cuda.stream(cin):
                for key in ins:
                    sw.inputs[key].copy_(pinned_in[key], non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(cin)
            comp.wait_event(arrived)
            enqueue(comp, nothing)
            done = torch.cuda.Event()
            done.record(comp)
            cout.wait_event(done)
            with torch.cuda.stream(cout):
                for key in outs:
                    pinned_out[key].copy_(sw.outputs[key], non_blocking=True)
            left = torch.cuda.Event()
            left.record(cout)
            freed[k % 2][name] = left
    cout.wait_stream(cin)
    cout.wait_stream(comp)
    e1.record(cout)
    e1.synchronize()
    return e0.elapsed_time(e1)


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.lines.append(line.strip())

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch, device_index):
    try:
        u = torch.cuda.get_device_properties(device_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else f"GPU-{s}"
    except Exception:
        return None


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text()), "measured"
        except ValueError:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def ncu_traffic(kernel: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if
    the summary was taken on the kernel source as it is now (else None)."""
    p = ROOT / "profiles" / "ncu_traffic.txt"
    if not p.exists():
        return None
    src_hash = source_hash(kernel)
    for line in p.read_text().splitlines():
        m = re.match(r"^(\S+)\s+(\d+)\s+(\S+)", line.strip())
        if m and m.group(1) == kernel and m.group(3) == src_hash:
            return int(m.group(2))
    return None


# Source files whose code a benchmark row's kernels are built from.
ROW_SOURCES = {
    "diffuse_fp64": ("diffuse2d.cu", "fp64_emu.cuh", "fvf_internal.cuh"),
    "diffuse_fp32": ("diffuse2d.cu", "fp64_emu.cuh", "fvf_internal.cuh"),
    "pack_x": ("weno_pack.cu", "fvf_internal.cuh"),
    "pack_y": ("weno_pack.cu", "fvf_internal.cuh"),
    "pack_z": ("weno_pack.cu", "fvf_internal.cuh"),
    "rhs_x": ("advect_rhs.cu", "fp64_emu.cuh", "fvf_internal.cuh"),
    "rhs_y": ("advect_rhs.cu", "fp64_emu.cuh", "fvf_internal.cuh"),
    "rhs_z": ("advect_rhs.cu", "fp64_emu.cuh", "fvf_internal.cuh"),
}


def source_hash(row: str | None = None):
    """Hash of the kernel sources of a benchmark row (all of csrc/ for None):
    a committed ncu traffic figure is used only while it matches."""
    names = ROW_SOURCES.get(row) if row else None
    h = hashlib.sha256()
    for f in sorted((ROOT / "finite_volume_field_gb300" / "csrc").glob("*")):
        if f.suffix in (".cu", ".cuh", ".h") and (names is None or f.name in names):
            h.update(f.name.encode())
            h.update(f.read_bytes())
    return h.hexdigest()[:12]


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------

def oracle_sample(host, diffusion_steps=160, passes=10):
    """Time the CPU oracle, as it stands, on a bounded sample of the step:
    ``diffusion_steps`` of each precision on the full 8192^2 grid (OpenMP over
    rows, all host threads), then ``passes`` passes of pack x/y/z and flux
    x/y/z and ``passes`` repetitions of the 2D sequence (single-threaded
    loops).  Returns (bytes, cellvars, seconds, threads)."""
    import oracle
    threads = oracle.max_threads()
    tot_b = tot_cv = tot_s = 0.0
    for key, p in (("u32", 4), ("u64", 8)):
        t0 = time.perf_counter()
        oracle.diffuse2d(host[key], diffusion_steps, nthreads=threads)
        tot_s += time.perf_counter() - t0
        tot_b += diffusion_steps * 2 * DIFF_N * DIFF_N * p
        tot_cv += diffusion_steps * (DIFF_N - 2) ** 2
    r = rows()["seq2d"]
    for _ in range(passes):
        for k in range(3):
            t0 = time.perf_counter()
            oracle.weno_pack(host["pack_fields"], PACK_EXT, PACK_G, k)
            oracle.advect_rhs(host["rhs_flux"][k], host["rhs_invd"][k], RHS_NV, RHS_EXT, k)
            tot_s += time.perf_counter() - t0
            tot_b += pack_bytes(PACK_EXT, PACK_G, PACK_NV, k) + rhs_bytes(RHS_EXT, RHS_NV, k)
            tot_cv += (_prod(pack_extents(PACK_EXT, PACK_G, k)) * PACK_NV
                       + _prod(RHS_EXT) * RHS_NV)
        t0 = time.perf_counter()
        oracle.multivar_sweep_2d(host["seq_fields"], host["seq_flux"][0], host["seq_flux"][1],
                                 host["seq_invd"][0], host["seq_invd"][1], SEQ_NV, SEQ_EXT, SEQ_G)
        tot_s += time.perf_counter() - t0
        tot_b += r["bytes"] / SEQ_REPS
        tot_cv += r["cellvars"] / SEQ_REPS
    return tot_b, tot_cv, tot_s, threads


def oracle_single_thread(host, steps=2):
    """The oracle's FP64 diffusion on the full 8192^2 grid on one host thread
    (the same loops and operation order as the all-threads run), for the
    single-core figure beside the all-cores one."""
    import oracle
    t0 = time.perf_counter()
    oracle.diffuse2d(host["u64"], steps, nthreads=1)
    sec = time.perf_counter() - t0
    b = steps * 2 * DIFF_N * DIFF_N * 8
    return {"value": round(b / sec / 1e9, 3), "unit": "GB/s", "cores": 1,
            "gcell_per_s": round(steps * (DIFF_N - 2) ** 2 / sec / 1e9, 4),
            "sample": f"{steps} FP64 diffusion steps on 8192^2, one thread",
            "seconds": round(sec, 2)}


def cpu_model():
    """The host CPU's model as the kernel reports it (x86 model name, or the
    Arm implementer and part numbers), with the logical CPU count."""
    name = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "CPU part"):
            for line in info.splitlines():
                if line.startswith(key):
                    name = line.split(":", 1)[1].strip()
                    break
            if name:
                if key == "CPU part":
                    impl = [l.split(":", 1)[1].strip() for l in info.splitlines()
                            if l.startswith("CPU implementer")]
                    name = f"implementer {impl[0] if impl else '?'} part {name}"
                break
    except OSError:
        pass
    return {"model": name or platform.processor() or platform.machine(),
            "machine": platform.machine(), "logical_cpus": os.cpu_count()}


def oracle_build_flags():
    import oracle
    return " ".join(getattr(oracle, "_CFLAGS", [])) + " (+ -fopenmp where available)"


ORACLE_SAMPLE_DESC = ("160 diffusion steps per precision on 8192^2 (OpenMP over rows, all host "
                      "threads) + 10 passes of pack x/y/z (8x207^3) and flux x/y/z (8x201^3) and 10 "
                      "repetitions of the 4800x1200 sequence (single-threaded loops); "
                      "GB/s = compulsory bytes / wall time")


REF_SAMPLE_DESC = ("per step: 10 diffusion steps per precision on 8192^2 (OpenMP over rows, "
                   "all host threads) + one pass of pack x/y/z and flux x/y/z + one repetition "
                   "of the 4800x1200 sequence (single-threaded loops); warm-up steps: 4 "
                   "diffusion steps + one pass")


# ---------------------------------------------------------------------------
# Arms
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    host = host_inputs()
    for _ in range(args.warmup):
        oracle_sample(host, diffusion_steps=4, passes=1)
    samples = []
    for _ in range(args.steps):
        samples.append(oracle_sample(host, diffusion_steps=10, passes=1))
    b = sum(s[0] for s in samples)
    cv = sum(s[1] for s in samples)
    sec = sum(s[2] for s in samples)
    threads = samples[0][3]
    gbs = b / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32+f64",
        "data": "synthetic", "gcell_var_per_s": cv / sec / 1e9,
        "config": {"workload": WORKLOAD, "reference": "CPU oracle (plain C, -O2 -ffp-contract=off)",
                   "sample": REF_SAMPLE_DESC},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": REF_SAMPLE_DESC},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def time_extra_sweeps(torch, sw, stream, reps=5):
    """Rows beyond the benchmark step, each timed on its own with CUDA events
    on the launching stream (median of several timings after one warm-up
    call; calls under a millisecond are timed 8 back to back per timing):
    the accumulating flux difference and the directional flux copy back to
    the physical frame on the 8 x 201^3 flux workload's buffers, the
    conservative-variable copy alone and fused with the pack on the 8 x 207^3
    pack workload's fields, the SSPRK3 stage update (fused with the flux
    difference, alone, and unfused) on the flux workload, the FP32 pack and
    flux difference on the same workloads, the 3D 7-point
    diffusion (512^3, 20 steps, FP32 and FP64; 10 FP64 operations per interior
    cell counting 6c) and the latency of the 64 x 64 FP64 diffusion case.  Stage rows count the bytes of the fused
    form (the unfused row's extra rhs traffic is its cost) and 13 FP64
    operations per element (5 for the update alone)."""
    from finite_volume_field_gb300 import api
    peaks, _ = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    cells = _prod(RHS_EXT) * RHS_NV
    out = {}

    def timed(fn):
        # A call shorter than a millisecond is repeated back to back between
        # the events (the time per call is the total over the calls): timed
        # alone, the host-side argument checks and launch of a single call
        # would show up as idle device time inside the interval.
        fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        inner = 1 if e0.elapsed_time(e1) >= 1.0 else 8
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(inner):
                fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) / inner)
        return statistics.median(times)

    def record(name, fn, nbytes, units, flops=0):
        t = timed(fn)
        rec = {"ms": round(t, 4), "gbs": round(nbytes / (t * 1e-3) / 1e9, 1),
               "gcell_var_per_s": round(units / (t * 1e-3) / 1e9, 2),
               "frac_hbm": round(nbytes / (t * 1e-3) / 1e9 / hbm, 4)}
        if flops:
            tf = flops * units / (t * 1e-3) / 1e12
            rec.update(fp64_tflops=round(tf, 4),
                       frac_fp64_nominal=round(tf / FP64_NOMINAL_TFLOPS, 4))
        out[name] = rec

    scratch = torch.empty_like(sw.rhs_flux[1])
    for k in (1, 2):
        ax = "xyz"[k]
        faces = sw.rhs_flux[k].numel()
        record(f"rhs_add_{ax}",
               lambda k=k: api.advect_rhs_add(sw.rhs_flux[k], sw.rhs_invd[k], RHS_NV, RHS_EXT, k,
                                              sw.rhs_out[k], stream),
               8 * (faces + 2 * cells + RHS_EXT[k]), cells, 3)
        record(f"unpack_{ax}",
               lambda k=k: api.flux_unpack(sw.rhs_flux[k], RHS_NV, RHS_EXT, k, scratch, stream),
               16 * faces, faces)
    del scratch
    # conservative-variable copy: alone, fused with the pack, and the unfused
    # pair (pack then copy) for comparison
    copies = [torch.empty_like(f) for f in sw.pack_fields]
    nst = sw.pack_fields[0].numel() * PACK_NV
    record("fields_copy",
           lambda: api.fields_copy(sw.pack_fields, PACK_NV, PACK_EXT, PACK_G, copies, stream),
           16 * nst, nst)
    for k, ax in enumerate("xyz"):
        npk = _prod(pack_extents(PACK_EXT, PACK_G, k)) * PACK_NV
        record(f"pack_copy_{ax}",
               lambda k=k: api.weno_pack_copy(sw.pack_fields, PACK_NV, PACK_EXT, PACK_G, k,
                                              sw.pack_out[k], copies, stream),
               8 * (2 * nst + npk), nst)

        def unfused(k=k):
            api.weno_pack(sw.pack_fields, PACK_NV, PACK_EXT, PACK_G, k, sw.pack_out[k], stream)
            api.fields_copy(sw.pack_fields, PACK_NV, PACK_EXT, PACK_G, copies, stream)
        record(f"pack_then_copy_{ax}", unfused, 8 * (2 * nst + npk), nst)
    del copies
    # SSPRK3 stage update on the flux workload (8 x 201^3, x/y/z faces):
    # fused with the flux difference, alone (axpby on a given rhs), and the
    # unfused sequence (flux difference x, +y, +z into rhs, then axpby)
    u0 = torch.randn(cells, dtype=torch.float64, device=sw.dev)
    u = torch.randn(cells, dtype=torch.float64, device=sw.dev)
    uo = torch.empty_like(u)
    rhs = sw.rhs_out[0]
    fl, w = sw.rhs_flux, sw.rhs_invd
    face_bytes = 8 * sum(f.numel() for f in fl)
    a, b, dt = 0.75, 0.25, 1e-4
    record("ssprk3_stage_xyz",
           lambda: api.ssprk3_stage(u0, u, fl, w, RHS_NV, RHS_EXT, a, b, dt, uo, stream),
           face_bytes + 24 * cells, cells, 13)
    record("ssprk3_axpby",
           lambda: api.ssprk3_axpby(u0, u, rhs, RHS_NV, RHS_EXT, a, b, dt, uo, stream),
           32 * cells, cells, 5)

    def stage_unfused():
        api.advect_rhs(fl[0], w[0], RHS_NV, RHS_EXT, 0, rhs, stream)
        api.advect_rhs_add(fl[1], w[1], RHS_NV, RHS_EXT, 1, rhs, stream)
        api.advect_rhs_add(fl[2], w[2], RHS_NV, RHS_EXT, 2, rhs, stream)
        api.ssprk3_axpby(u0, u, rhs, RHS_NV, RHS_EXT, a, b, dt, uo, stream)
    record("ssprk3_stage_unfused_xyz", stage_unfused, face_bytes + 24 * cells, cells, 13)
    del u0, u, uo
    # FP32 pack (8 x 207^3) and FP32 flux difference (8 x 201^3)
    f32f = [f.float() for f in sw.pack_fields]
    pout = torch.empty(sw.pack_out[0].numel(), dtype=torch.float32, device=sw.dev)
    for k, ax in enumerate("xyz"):
        npk = _prod(pack_extents(PACK_EXT, PACK_G, k)) * PACK_NV
        record(f"pack_f32_{ax}",
               lambda k=k: api.weno_pack_f32(f32f, PACK_NV, PACK_EXT, PACK_G, k, pout, stream),
               8 * npk, npk)
    del f32f, pout
    r32 = torch.empty(cells, dtype=torch.float32, device=sw.dev)
    for k, ax in enumerate("xyz"):
        fl32, w32 = sw.rhs_flux[k].float(), sw.rhs_invd[k].float()
        record(f"rhs_f32_{ax}",
               lambda fl32=fl32, w32=w32, k=k: api.advect_rhs_f32(fl32, w32, RHS_NV, RHS_EXT, k,
                                                                  r32, stream),
               4 * (fl32.numel() + cells + RHS_EXT[k]), cells)
        del fl32, w32
    del r32
    # 3D 7-point diffusion, 512^3, 20 steps per call, FP32 and FP64
    n3 = 512
    cells3 = n3 ** 3
    for name, dt, code, esize, flops in (("diffuse3d_fp32", torch.float32, api.FVF_FP32, 4, 0),
                                         ("diffuse3d_fp64", torch.float64, api.FVF_FP64, 8, 10)):
        u3 = torch.rand(cells3, dtype=dt, device=sw.dev)
        v3 = torch.zeros_like(u3)
        record(name, lambda u3=u3, v3=v3, code=code: api.diffuse3d_step(
            u3, v3, n3, n3, n3, 0.1, 20, code, stream), 20 * 2 * esize * cells3,
            20 * (n3 - 2) ** 3, flops)
        del u3, v3
    # ablation: the one-thread-per-(cell, variable) mapping that the pull
    # request replaces, against the library's one-thread-per-cell kernels
    out["collapse4_vs_collapse3"] = time_ablation(torch, sw, stream, timed)
    # ablations of the 2D FP32 diffusion kernels on the 8192^2 grid: 16-byte
    # vectors (rows aligned) against one cell per thread (the same buffers one
    # element in, which the library serves with its scalar kernel), and the
    # shared-memory blocked kernel (200 steps in one call) against 200
    # single-step calls (the vector march kernel)
    n2 = DIFF_N * DIFF_N
    whole_u = torch.empty(n2 + 4, dtype=torch.float32, device=sw.dev)
    whole_v = torch.zeros_like(whole_u)
    flat = sw.u32.reshape(-1)
    whole_u.copy_(torch.cat([flat, flat[:4]]))
    t_vec = timed(lambda: api.diffuse2d_step(whole_u[:n2], whole_v[:n2], DIFF_N, DIFF_N, 0.1, 1,
                                             api.FVF_FP32, stream))
    t_sca = timed(lambda: api.diffuse2d_step(whole_u[1:n2 + 1], whole_v[1:n2 + 1], DIFF_N, DIFF_N,
                                             0.1, 1, api.FVF_FP32, stream))
    out["vector_vs_scalar_fp32_step"] = {"vector_ms": round(t_vec, 4), "scalar_ms": round(t_sca, 4),
                                         "speedup": round(t_sca / t_vec, 3)}

    def single_steps():
        for s_ in range(DIFF_STEPS):
            a, b = (whole_u[:n2], whole_v[:n2]) if s_ % 2 == 0 else (whole_v[:n2], whole_u[:n2])
            api.diffuse2d_step(a, b, DIFF_N, DIFF_N, 0.1, 1, api.FVF_FP32, stream)
    t_blk = timed(lambda: api.diffuse2d_step(whole_u[:n2], whole_v[:n2], DIFF_N, DIFF_N, 0.1,
                                             DIFF_STEPS, api.FVF_FP32, stream))
    t_one = timed(single_steps)
    out["blocked_vs_single_step_fp32_200steps"] = {"blocked_ms": round(t_blk, 3),
                                                   "single_step_ms": round(t_one, 3),
                                                   "speedup": round(t_one / t_blk, 3)}
    del whole_u, whole_v
    # FP64 diffusion of a field with mixed signs: the 8192^2 grid with
    # interior N(0,1) values, 20 steps per call, beside the same 20 steps of
    # the uniform [0,1) field the step times (the integer-pipe additions take
    # their general form on rows where signs differ)
    nrm = torch.from_numpy(inputs.diffusion_field(DIFF_N, DIFF_N, np.float64,
                                                  seed=inputs.config_seed(2), stream=2,
                                                  values="normal")).to(sw.dev)
    nrm_v = torch.zeros_like(nrm)
    uni = sw.u64.clone()
    cells2 = (DIFF_N - 2) ** 2
    for name, fld in (("diffuse_fp64_normal_20steps", nrm), ("diffuse_fp64_uniform_20steps", uni)):
        record(name, lambda fld=fld: api.diffuse2d_step(fld, nrm_v, DIFF_N, DIFF_N, 0.1, 20,
                                                         api.FVF_FP64, stream),
               20 * 2 * DIFF_N * DIFF_N * 8, 20 * cells2, FP64_FLOPS["diffuse_fp64"])
    out["diffuse_fp64_normal_20steps"]["vs_uniform"] = round(
        out["diffuse_fp64_normal_20steps"]["ms"] / out["diffuse_fp64_uniform_20steps"]["ms"], 4)
    del nrm, nrm_v, uni
    # the 64 x 64 FP64 centre-impulse case, 32 steps: a latency measurement
    # (both states live in shared memory), reported per call and per step
    u = torch.zeros(64 * 64, dtype=torch.float64, device=sw.dev)
    u[31 + 64 * 31] = 1.0
    v = torch.zeros_like(u)
    call = lambda: api.diffuse2d_step(u, v, 64, 64, 0.1, 32, api.FVF_FP64, stream)  # noqa: E731
    call()
    times = []
    for _ in range(20):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    t = statistics.median(times)
    out["diffuse_64x64_fp64_32steps"] = {"us_per_call": round(1e3 * t, 2),
                                         "us_per_step": round(1e3 * t / 32, 3)}
    return out


ABLATION_SRCS = [ROOT / "ablation" / "collapse4.cu", ROOT / "ablation" / "peaks.cu"]
ABLATION_LIB = ROOT / "ablation" / "libfvf_ablation.so"


def build_ablation(force: bool = False) -> Path:
    """Compile ablation/libfvf_ablation.so: the benchmark-only kernels -- the
    one-thread-per-(cell, variable) mapping that libfvf's kernels replace,
    and the arithmetic issue-rate probes.  Not part of libfvf and not used
    by it; built with the library's nvcc flags."""
    from finite_volume_field_gb300 import buildlib
    newest = max([p.stat().st_mtime for p in ABLATION_SRCS]
                 + [Path(buildlib.__file__).stat().st_mtime])
    if not force and ABLATION_LIB.exists() and ABLATION_LIB.stat().st_mtime >= newest:
        return ABLATION_LIB
    tmp = ABLATION_LIB.with_suffix(f".so.tmp{os.getpid()}")
    cmd = [buildlib.nvcc(), *buildlib.NVCC_FLAGS, "-shared", "-cudart", "static",
           *map(str, ABLATION_SRCS), "-o", str(tmp)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on the ablation library:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, ABLATION_LIB)
    return ABLATION_LIB


def load_ablation():
    """ablation/libfvf_ablation.so (built by build_ablation) through ctypes."""
    import ctypes
    lib = ctypes.CDLL(str(build_ablation()))
    vp, i64, cint = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.ablation_pack_x_collapse4.argtypes = [ctypes.POINTER(vp), cint, ctypes.POINTER(i64), cint,
                                              vp, vp]
    lib.ablation_rhs_x_collapse4.argtypes = [vp, vp, cint, ctypes.POINTER(i64), vp, vp]
    lib.bench_issue_rate.argtypes = [cint, cint, ctypes.POINTER(ctypes.c_double)]
    return lib


def measured_issue_rates():
    """Arithmetic issue rates of this GPU from the probes in the benchmark
    library (operations per second; an FMA counts once): the denominators of
    the FP64-bound rows."""
    import ctypes
    lib = load_ablation()
    names = {0: "fp64_add", 1: "fp64_mul", 2: "fp64_fma", 3: "fp32_fma", 4: "int32_alu"}
    out = {}
    for op, name in names.items():
        r = ctypes.c_double(0.0)
        if lib.bench_issue_rate(op, 3, ctypes.byref(r)) == 0:
            out[name] = round(r.value / 1e12, 4)
    return out   # T operations per second


def time_ablation(torch, sw, stream, timed):
    """The x pack (8 x 207^3) and the x flux difference (8 x 201^3) with the
    one-thread-per-(cell, variable) mapping (collapse 4) and with the
    library's one-thread-per-cell kernels (collapse 3): time of each and the
    ratio, and whether the two outputs agree bit for bit."""
    import ctypes
    from finite_volume_field_gb300 import api
    lib = load_ablation()
    ext = (ctypes.c_int64 * 3)(*PACK_EXT)
    table = (ctypes.c_void_p * PACK_NV)(*[f.data_ptr() for f in sw.pack_fields])
    o4 = torch.empty_like(sw.pack_out[0])
    res = {}
    t4 = timed(lambda: lib.ablation_pack_x_collapse4(table, PACK_NV, ext, PACK_G, o4.data_ptr(),
                                                     stream.cuda_stream))
    t3 = timed(lambda: api.weno_pack(sw.pack_fields, PACK_NV, PACK_EXT, PACK_G, 0, sw.pack_out[0],
                                     stream))
    torch.cuda.synchronize()
    res["pack_x"] = {"collapse4_ms": round(t4, 4), "collapse3_ms": round(t3, 4),
                     "duration_change": round(t3 / t4 - 1.0, 3),
                     "same_bits": bool(torch.equal(o4.view(torch.int64),
                                                   sw.pack_out[0].view(torch.int64)))}
    rext = (ctypes.c_int64 * 3)(*RHS_EXT)
    r4 = torch.empty_like(sw.rhs_out[0])
    t4 = timed(lambda: lib.ablation_rhs_x_collapse4(sw.rhs_flux[0].data_ptr(),
                                                    sw.rhs_invd[0].data_ptr(), RHS_NV, rext,
                                                    r4.data_ptr(), stream.cuda_stream))
    t3 = timed(lambda: api.advect_rhs(sw.rhs_flux[0], sw.rhs_invd[0], RHS_NV, RHS_EXT, 0,
                                      sw.rhs_out[0], stream))
    torch.cuda.synchronize()
    res["rhs_x"] = {"collapse4_ms": round(t4, 4), "collapse3_ms": round(t3, 4),
                    "duration_change": round(t3 / t4 - 1.0, 3),
                    "same_bits": bool(torch.equal(r4.view(torch.int64),
                                                  sw.rhs_out[0].view(torch.int64)))}
    return res


def aggregate(per_rank, world):
    """Combine per-rank measurements: device time is the max over ranks,
    throughput counts the work of every rank."""
    ms = max(r["ms_per_step"] for r in per_rank)
    e2e_ms = max(r["e2e_ms_per_step"] for r in per_rank)
    launches = sum(r["launches"] for r in per_rank)
    return ms, e2e_ms, launches


def roofline(r, name, sw, hbm, peak_kind, rates):
    """The roofline object of the dominant kernel: algorithmic bytes of one
    launch over its CUDA-event launch time, against the measured HBM copy
    rate.  For an FP64 sweep, the same launch against this GPU's measured FP64
    issue rate (the FP64-unit instructions the kernel issues per element as
    built) sits beside it in ``fp64``; ``binding`` names the larger of the
    two fractions."""
    launch_ms = sw["ms"] / r["launches"]
    achieved = r["per_launch_bytes"] / (launch_ms * 1e-3) / 1e9
    roof = {"kernel": name, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
            "traffic": ncu_traffic(name), "launch_ms": round(launch_ms, 5),
            "algorithmic_bytes_per_launch": r["per_launch_bytes"], "binding": "hbm"}
    if name in FP64_FLOPS:
        cells = r["per_launch_cells"]
        tf = FP64_FLOPS[name] * cells / (launch_ms * 1e-3) / 1e12
        fp = {"flops_per_element": FP64_FLOPS[name], "tflops": round(tf, 4),
              "instructions_per_element": FP64_INSTR[name]}
        peak_ops = rates.get("fp64_fma")
        if peak_ops:
            ops = FP64_INSTR[name] * cells / (launch_ms * 1e-3) / 1e12
            fp.update(achieved=round(ops, 4), peak=peak_ops, unit="T FP64 instructions/s",
                      frac=round(ops / peak_ops, 4),
                      peak_source="measured: FP64 FMA issue-rate probe, this run")
            if fp["frac"] > roof["frac"]:
                roof["binding"] = "fp64"
        roof["fp64"] = fp
    return roof


def blocked_traffic(ms, hbm):
    """DRAM bytes that the blocked FP32 diffusion moves for the 8192^2 x 200
    workload, from its tiling (each 8-step launch reads every 128 x 80 staged
    region and writes every 112 x 64 tile; the last step is one plain launch
    that reads and writes the grid), and that traffic's fraction of the HBM
    copy rate: beside the row's effective fraction, which counts the one-pass
    bytes of every step."""
    tiles = -(-DIFF_N // 112) * -(-DIFF_N // 64)
    n1 = DIFF_STEPS - 1
    nb = -(-n1 // 8)
    if nb % 2 != (DIFF_STEPS + 1) % 2:
        nb += 1
    b = nb * tiles * (128 * 80 + 112 * 64) * 4 + 2 * DIFF_N * DIFF_N * 4
    return {"dram_bytes_model": b, "dram_gbs_model": round(b / (ms * 1e-3) / 1e9, 1),
            "frac_hbm_dram_model": round(b / (ms * 1e-3) / 1e9 / hbm, 4),
            "note": "frac_hbm counts 8 one-pass steps per blocked launch (effective)"}


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    from finite_volume_field_gb300 import api, buildlib
    if not api.LIB_PATH.exists():
        buildlib.build()
    api.load()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    host = host_inputs()
    stream = torch.cuda.Stream(device)
    sw = Sweeps(torch, host, device, stream)
    R = rows()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(device)

    # Warm-up; the first step also counts the kernel launches of each row
    # (the library's own launch counter; blocked diffusion runs up to 8 steps
    # per launch).
    row_launches = {}

    def count(name, which):
        if which == 0:
            row_launches[name] = -api.launch_count()
        else:
            row_launches[name] += api.launch_count()

    with torch.cuda.stream(stream):
        for w in range(max(1, args.warmup)):
            sw.step(None, count if w == 0 else None)
    barrier()
    for name, n in row_launches.items():
        R[name]["per_launch_bytes"] = R[name]["bytes"] / n
        R[name]["per_launch_cells"] = R[name]["cellvars"] / n
        R[name]["launches"] = n
    if not args.no_graph:
        sw.capture_seq_graph()
        with torch.cuda.stream(stream):
            sw.step()             # one warm-up replay of the graph
        barrier()

    # One set of row events per timed step, read after the loop (no host
    # synchronisation inside the timed region).
    evs = [{name: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for name in R} for _ in range(args.steps)]
    sampler = ClockSampler(gpu_uuid(torch, local))
    sampler.start()
    time.sleep(0.5)
    barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = api.launch_count()
    graph0 = sw.graph_launches
    with torch.cuda.stream(stream):
        start.record(stream)
        for k in range(args.steps):
            sw.step(evs[k])
        end.record(stream)
    barrier()
    per_row = {name: [e[name][0].elapsed_time(e[name][1]) for e in evs] for name in R}
    # direct launches plus the kernels that graph replays launched
    launches = api.launch_count() - launches0 + sw.graph_launches - graph0
    clocks = sampler.stop()
    total_ms = start.elapsed_time(end)
    ms_per_step = total_ms / args.steps

    # End to end through the public API with host buffers: every input copied
    # in from pinned host memory and every output copied back, inside the
    # timed region, pipelined over a copy-in, a compute and a copy-out stream.
    pinned_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v.cpu())
                 for k, v in sw.inputs.items()}
    pinned_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                  for k, v in sw.outputs.items()}
    h2d = sum(t.numel() * t.element_size() for t in pinned_in.values())
    d2h = sum(t.numel() * t.element_size() for t in pinned_out.values())
    sw2 = Sweeps(torch, host, device, stream)
    streams = (torch.cuda.Stream(device), stream, torch.cuda.Stream(device))
    e2e_steps = max(2, min(args.steps, 4))
    e2e_pipeline(torch, (sw, sw2), pinned_in, pinned_out, streams, 2)   # warm-up
    barrier()
    e2e_ms = e2e_pipeline(torch, (sw, sw2), pinned_in, pinned_out, streams, e2e_steps) / e2e_steps
    barrier()
    del sw2

    extras = time_extra_sweeps(torch, sw, stream)
    rates = measured_issue_rates() if rank == 0 else {}

    mine = {"ms_per_step": ms_per_step, "e2e_ms_per_step": e2e_ms, "launches": launches}
    if world > 1:
        import torch.distributed as dist
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
    else:
        gathered = [mine]
    ms, e2e_ms, launches = aggregate(gathered, world)

    if rank == 0:
        step_bytes = sum(r["bytes"] for r in R.values())
        step_cv = sum(r["cellvars"] for r in R.values())
        value = world * step_bytes / (ms * 1e-3) / 1e9
        peaks, peak_kind = measured_peaks()
        hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
        sweeps = {}
        for name, r in R.items():
            t = statistics.median(per_row[name])
            sweeps[name] = {
                "ms": round(t, 4), "launches": r["launches"],
                # median over the timed steps, and the fastest and slowest step
                "spread_ms": [round(min(per_row[name]), 4), round(max(per_row[name]), 4)],
                "gbs": round(r["bytes"] / (t * 1e-3) / 1e9, 1),
                "gcell_var_per_s": round(r["cellvars"] / (t * 1e-3) / 1e9, 2),
                "frac_hbm": round(r["bytes"] / (t * 1e-3) / 1e9 / hbm, 4),
            }
            if name in FP64_FLOPS:
                tf = FP64_FLOPS[name] * r["cellvars"] / (t * 1e-3) / 1e12
                sweeps[name]["fp64_tflops"] = round(tf, 4)
                if rates.get("fp64_fma"):
                    ops = FP64_INSTR[name] * r["cellvars"] / (t * 1e-3) / 1e12
                    sweeps[name]["frac_fp64_issue"] = round(ops / rates["fp64_fma"], 4)
        dom = max((n for n in R if n != "seq2d"), key=lambda n: sweeps[n]["ms"])
        roof = roofline(R[dom], dom, sweeps[dom], hbm, peak_kind, rates)
        if "diffuse_fp32" in sweeps:
            sweeps["diffuse_fp32"].update(blocked_traffic(sweeps["diffuse_fp32"]["ms"], hbm))
        line = {
            "impl": "gb300", "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32+f64", "data": "synthetic",
            "gcell_var_per_s": round(world * step_cv / (ms * 1e-3) / 1e9, 3),
            "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                       "l2": "no flush: every launch's working set (>= 0.5 GB) exceeds the 129 MB L2",
                       "bytes_per_step": step_bytes, "hbm_peak_gbs": hbm,
                       "hbm_peak_source": peak_kind,
                       "seq2d": "one CUDA graph of its 400 launches per step" if not args.no_graph
                                else "400 launches per step"},
            "roofline": roof,
            "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 3), "steps": e2e_steps},
            "gpu_launches": launches,
            "clocks": clocks,
            "measured_rates_tops": rates,
            "extra_sweeps": extras,
        }
        if world == 1 and not args.no_cpu_baseline:
            b, cv, sec, threads = oracle_sample(host)
            line["cpu_baseline"] = {"value": round(b / sec / 1e9, 3), "unit": "GB/s",
                                    "cores": threads, "kind": "oracle",
                                    "sample": ORACLE_SAMPLE_DESC,
                                    "gcell_var_per_s": round(cv / sec / 1e9, 4),
                                    "seconds": round(sec, 2),
                                    "single_thread": oracle_single_thread(host),
                                    "cpu_model": cpu_model(),
                                    "oracle_build": oracle_build_flags()}
        # the per-sweep table last: a reader of the end of the line sees it
        line["sweeps"] = sweeps
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_ncu_case():
    """Each sweep kernel at its benchmark size, one buffer set on the device
    at a time (at most about 1.1 GB), for Nsight Compute captures:
    diffusion 8192^2 FP64 then FP32, pack x/y/z on 8 fields of
    207^3, the conservative-variable copy alone and fused with the pack x/y/z
    on the same fields (at most about 1.7 GB), flux difference x/y/z on
    8 x 201^3, the SSPRK3 stage fused with the x/y/z flux difference on
    8 x 201^3 (about 3.1 GB), the 3D 7-point diffusion on 512^3, one FP32
    step then three FP64 steps (at most 2.1 GB; from the second step on the
    faces are zero, as in the benchmark's 20-step calls, so a capture skips
    the first), the FP32 pack y, z, x and the FP32 flux
    difference x, and last the 64 x 64 FP64 centre impulse for 32 steps (one
    cluster launch).  The 2D FP32 diffusion runs 17 steps (two 8-step
    shared-memory launches, then one single step).  Device-generated values:
    the timing of the sweeps does not depend on them, except the FP64
    diffusion's, whose field is U[0,1) with zero edges (the benchmark's
    field) and runs 22 single steps, so that a capture can skip the first 20
    (the fixed-point neighbour sum declines more lanes on the unsmoothed
    field)."""
    import torch
    from finite_volume_field_gb300 import api, buildlib
    if not api.LIB_PATH.exists():
        buildlib.build()
    api.load()

    def free():
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    for dt, code, steps in ((torch.float64, api.FVF_FP64, 22), (torch.float32, api.FVF_FP32, 17)):
        u = torch.rand(DIFF_N, DIFF_N, dtype=dt, device="cuda")
        u[0, :] = 0
        u[-1, :] = 0
        u[:, 0] = 0
        u[:, -1] = 0
        u = u.reshape(-1)
        v = torch.zeros_like(u)
        api.diffuse2d_step(u, v, DIFF_N, DIFF_N, 0.1, steps, code)
        del u, v
        free()
    N = _prod(inputs.stored_extents(PACK_EXT, PACK_G))
    fields = [torch.randn(N, dtype=torch.float64, device="cuda") for _ in range(PACK_NV)]
    out = torch.empty(_prod(pack_extents(PACK_EXT, PACK_G, 0)) * PACK_NV, dtype=torch.float64,
                      device="cuda")
    for d in range(3):
        api.weno_pack(fields, PACK_NV, PACK_EXT, PACK_G, d, out)
    copies = [torch.empty_like(f) for f in fields]
    api.fields_copy(fields, PACK_NV, PACK_EXT, PACK_G, copies)
    for d in range(3):
        api.weno_pack_copy(fields, PACK_NV, PACK_EXT, PACK_G, d, out, copies)
    del fields, out, copies
    free()
    for d in range(3):
        fe = list(RHS_EXT)
        fe[d] += 1
        F = torch.randn(_prod(fe) * RHS_NV, dtype=torch.float64, device="cuda")
        w = torch.rand(RHS_EXT[d], dtype=torch.float64, device="cuda") + 0.5
        r = torch.empty(_prod(RHS_EXT) * RHS_NV, dtype=torch.float64, device="cuda")
        api.advect_rhs(F, w, RHS_NV, RHS_EXT, d, r)
        del F, w, r
        free()
    fl, ws = [], []
    for d in range(3):
        fe = list(RHS_EXT)
        fe[d] += 1
        fl.append(torch.randn(_prod(fe) * RHS_NV, dtype=torch.float64, device="cuda"))
        ws.append(torch.rand(RHS_EXT[d], dtype=torch.float64, device="cuda") + 0.5)
    u0 = torch.randn(_prod(RHS_EXT) * RHS_NV, dtype=torch.float64, device="cuda")
    u = torch.randn_like(u0)
    api.ssprk3_stage(u0, u, fl, ws, RHS_NV, RHS_EXT, 0.75, 0.25, 1e-4, u)
    del fl, ws, u0, u
    free()
    for dt, code, steps in ((torch.float32, api.FVF_FP32, 1), (torch.float64, api.FVF_FP64, 3)):
        u = torch.rand(512 ** 3, dtype=dt, device="cuda")
        v = torch.zeros_like(u)
        api.diffuse3d_step(u, v, 512, 512, 512, 0.1, steps, code)
        del u, v
        free()
    # FP32 pack y, z, x on 8 fields of 207^3 and the FP32 flux difference x on
    # 8 x 201^3 (at most about 0.55 GB)
    fields = [torch.randn(N, dtype=torch.float32, device="cuda") for _ in range(PACK_NV)]
    out = torch.empty(_prod(pack_extents(PACK_EXT, PACK_G, 0)) * PACK_NV, dtype=torch.float32,
                      device="cuda")
    for d in (1, 2, 0):
        api.weno_pack_f32(fields, PACK_NV, PACK_EXT, PACK_G, d, out)
    del fields, out
    free()
    fe = list(RHS_EXT)
    fe[0] += 1
    F = torch.randn(_prod(fe) * RHS_NV, dtype=torch.float32, device="cuda")
    w = torch.rand(RHS_EXT[0], dtype=torch.float32, device="cuda") + 0.5
    r = torch.empty(_prod(RHS_EXT) * RHS_NV, dtype=torch.float32, device="cuda")
    api.advect_rhs_f32(F, w, RHS_NV, RHS_EXT, 0, r)
    del F, w, r
    free()
    # the small-grid case: 64 x 64 FP64 centre impulse, 32 steps, one cluster launch
    u = torch.zeros(64 * 64, dtype=torch.float64, device="cuda")
    u[31 * 64 + 31] = 1.0
    v = torch.zeros_like(u)
    api.diffuse2d_step(u, v, 64, 64, 0.1, 32, api.FVF_FP64)
    free()
    print("ncu case done", flush=True)
    return 0


def run_ncu_ablation():
    """The x pack on 8 x 207^3 and the x flux difference on 8 x 201^3, each
    once with the library kernel (one thread per cell) then once with the
    ablation kernel (one thread per cell-variable pair), for an Nsight
    Compute comparison of instructions, DRAM bytes and duration."""
    import ctypes

    import torch
    from finite_volume_field_gb300 import api, buildlib
    if not api.LIB_PATH.exists():
        buildlib.build()
    api.load()
    lib = load_ablation()
    N = _prod(inputs.stored_extents(PACK_EXT, PACK_G))
    fields = [torch.randn(N, dtype=torch.float64, device="cuda") for _ in range(PACK_NV)]
    out = torch.empty(_prod(pack_extents(PACK_EXT, PACK_G, 0)) * PACK_NV, dtype=torch.float64,
                      device="cuda")
    api.weno_pack(fields, PACK_NV, PACK_EXT, PACK_G, 0, out)
    table = (ctypes.c_void_p * PACK_NV)(*[f.data_ptr() for f in fields])
    lib.ablation_pack_x_collapse4(table, PACK_NV, (ctypes.c_int64 * 3)(*PACK_EXT), PACK_G,
                                  out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    del fields, out
    torch.cuda.empty_cache()
    fe = list(RHS_EXT)
    fe[0] += 1
    F = torch.randn(_prod(fe) * RHS_NV, dtype=torch.float64, device="cuda")
    w = torch.rand(RHS_EXT[0], dtype=torch.float64, device="cuda") + 0.5
    r = torch.empty(_prod(RHS_EXT) * RHS_NV, dtype=torch.float64, device="cuda")
    api.advect_rhs(F, w, RHS_NV, RHS_EXT, 0, r)
    lib.ablation_rhs_x_collapse4(F.data_ptr(), w.data_ptr(), RHS_NV,
                                 (ctypes.c_int64 * 3)(*RHS_EXT), r.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    print("ncu ablation done", flush=True)
    return 0


def run_slab(args):
    """The diffusion rows of the step (8192^2, 200 steps, FP64 then FP32) on
    a grid split into j-slabs (finite_volume_field_gb300/slab.py): one slab
    per rank under torchrun, halos exchanged with torch.distributed point to
    point (NCCL); with one process, ``--slab P`` slabs on the one device,
    halos copied between them.  FP64 takes 4-row halos (an exchange every 4
    steps), FP32 8-row halos (one exchange per 8-step blocked launch).  The
    whole grid is the work for any number of ranks: strong scaling."""
    import torch
    from finite_volume_field_gb300 import api, buildlib, slab
    world, rank, local = dist_env()
    if not api.LIB_PATH.exists():
        buildlib.build()
    api.load()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    parts = world if world > 1 else max(1, args.slab)
    host = host_inputs()
    stream = torch.cuda.Stream(device)
    runs = []
    for key, code, halo in (("u64", api.FVF_FP64, 4), ("u32", api.FVF_FP32, 8)):
        u0 = host[key]
        mine = [rank] if world > 1 else list(range(parts))
        slabs = []
        for p in mine:
            rows = slab.slab_rows(DIFF_N, parts, p, halo)
            u = torch.from_numpy(u0[rows.l0:rows.l1].reshape(-1).copy()).to(device)
            slabs.append(slab.SlabDiffusion2D(u, torch.zeros_like(u), DIFF_N, DIFF_N, rows, halo,
                                              0.1, code, stream=stream))
        if world > 1:
            ex = slab.dist_exchanger(dist, rank, world, sync=stream.synchronize)
            advance = lambda n, s=slabs[0], ex=ex: s.advance(n, ex)  # noqa: E731
        else:
            lx = slab.LocalExchange(slabs)
            advance = lx.advance
        runs.append((key, advance))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(device)

    def one_step():
        with torch.cuda.stream(stream):
            for _, advance in runs:
                advance(DIFF_STEPS)
    for _ in range(max(1, args.warmup)):
        one_step()
    barrier()
    t0 = time.perf_counter()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        one_step()
    end.record(stream)
    barrier()
    ms = start.elapsed_time(end) / args.steps
    wall_ms = 1e3 * (time.perf_counter() - t0) / args.steps
    if dist is not None:
        both = [None] * world
        dist.all_gather_object(both, (ms, wall_ms))
        ms = max(b[0] for b in both)
        wall_ms = max(b[1] for b in both)
    if rank == 0:
        step_bytes = DIFF_STEPS * 2 * DIFF_N * DIFF_N * (8 + 4)
        line = {"impl": "gb300", "metric": METRIC, "value": round(step_bytes / (ms * 1e-3) / 1e9, 2),
                "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms, 4), "wall_ms_per_step": round(wall_ms, 4),
                "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
                "dtype": "f32+f64", "data": "synthetic",
                "config": {"workload": "2D 5-point diffusion 8192x8192, alpha 0.1, 200 steps, "
                                       "FP64 then FP32, in j-slabs with halo exchange",
                           "slabs": parts, "halo_rows": {"fp64": 4, "fp32": 8},
                           "exchange": "torch.distributed point to point" if world > 1
                                       else "device copies between slabs on one GPU"}}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (it is only taken at N=1 anyway)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the 2D sequence call by call instead of replaying a CUDA graph")
    ap.add_argument("--ncu-ablation", action="store_true",
                    help="run the collapse-3 / collapse-4 kernel pairs once each (for ncu)")
    ap.add_argument("--ncu-case", action="store_true",
                    help="launch each sweep kernel once at benchmark size (for ncu), no timing")
    ap.add_argument("--slab", type=int, default=0,
                    help="the diffusion rows only, decomposed into j-slabs: one per rank under "
                         "torchrun, or this many on the one GPU (strong scaling)")
    args = ap.parse_args(argv)
    if args.slab and args.impl == "gb300":
        return run_slab(args)
    if args.ncu_case:
        return run_ncu_case()
    if args.ncu_ablation:
        return run_ncu_ablation()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
