"""DRAM-cold benchmark of the quantized decode chain on GB300.

A step is one pass of the whole hot path over one synthetic decode token: the fused
RMSNorm -> q8_1 producer on the token's activation row, then the GEMV against that q8_1
activation, reading the next of several rotated weight copies so that no launch finds its
weights in L2.  The default workload is the Q8_0 4096 x 4096 m = 1 GEMV with 16 rotated copies
(285 MB, well past the 129 MB L2).

Printed (rank 0, one JSON line):
  value       whole-step throughput: algorithmic bytes of the step (GEMV weights + scales +
              activation, plus the producer's x, w, qs, d) / device time per step, inputs
              resident in HBM; K steps replayed from CUDA graphs, timed with CUDA events.
  roofline    the dominant kernel (the GEMV): algorithmic bytes per launch / average launch
              duration in a decode loop (graph of back-to-back launches over the rotated
              copies, DRAM-cold), against the measured HBM copy bandwidth; the one-launch-at-a-
              time figure is reported beside it.
  e2e         the same metric through the public API with host buffers, per step one replay of
              a CUDA graph holding those calls (the eager Python loop is reported beside it): the
              activation row is copied host->device from pinned memory, the chain runs, the
              result y is copied device->host and the host waits for it.
  cpu_baseline  the f64 oracle on the host cores on a bounded sample of the same workload.
With --impl reference the oracle itself is the timed arm (rank 0 only).
"""
from __future__ import annotations

import argparse
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

METRIC = "m=1 quantized GEMV achieved HBM GB/s (DRAM-cold) and % of GB300 peak"
FALLBACK_HBM_GBS = 6800.0

# Workloads by name: (container, out_f, in_f, m, rotated copies).  Any other name of the form
# <e4m3|blk128|q8_0>_<out_f>x<in_f>_m<m> is accepted too (copies sized to twice the L2).
WORKLOADS = {
    "q8_0_4096x4096_m1": ("q8_0", 4096, 4096, 1, 16),
    "e4m3_1024x4096_m1": ("e4m3", 1024, 4096, 1, 64),
    "blk128_17408x5120_m1": ("blk", 17408, 5120, 1, 4),
    "e4m3_17408x5120_m1": ("e4m3", 17408, 5120, 1, 4),
    "q8_0_17408x5120_m1": ("q8_0", 17408, 5120, 1, 4),
}
DEFAULT_WORKLOAD = "q8_0_4096x4096_m1"
L2_BYTES = 129 * 2 ** 20
# f32 FMA peak of the CUDA cores: 152 SMs x 128 FMA / clock x 2 FLOP x 2.07 GHz (maximum clock)
F32_FMA_TFLOPS = round(152 * 128 * 2 * 2.07e9 / 1e12, 2)


def parse_workload(name: str):
    if name in WORKLOADS:
        return WORKLOADS[name]
    try:
        kind, shape, mtag = name.split("_") if not name.startswith("q8_0") else \
            ("q8_0",) + tuple(name[len("q8_0_"):].split("_"))
        out_f, in_f = (int(v) for v in shape.split("x"))
        m = int(mtag.lstrip("m"))
    except ValueError:
        raise SystemExit(f"unknown workload {name!r}")
    kind = {"e4m3": "e4m3", "blk128": "blk", "q8_0": "q8_0"}[kind]
    wbytes = gemv_bytes(kind, out_f, in_f, m)
    copies = max(4, -(-2 * L2_BYTES // wbytes))
    return kind, out_f, in_f, m, copies


# ------------------------------------------------------------------------------------------
# Byte accounting (algorithmic bytes, outputs excluded for the GEMV per the metric)
# ------------------------------------------------------------------------------------------

def gemv_bytes(kind: str, out_f: int, in_f: int, m: int) -> int:
    act = m * (in_f + in_f // 32 * 4)
    if kind == "q8_0":
        return out_f * (in_f // 32) * 34 + act
    if kind == "blk":
        return out_f * in_f + 4 * (-(-out_f // 128)) * (-(-in_f // 128)) + act
    return out_f * in_f + 4 + act


def producer_bytes(rows: int, ncols: int) -> int:
    return rows * ncols * 4 + ncols * 4 + rows * ncols + rows * (ncols // 32) * 4


# ------------------------------------------------------------------------------------------
# Distributed plumbing (replicas only: no data-path collective)
# ------------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(elapsed_s: float, units: float, group=None):
    """Max elapsed over ranks and the sum of units over ranks (whole-job throughput)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="memq_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [c.strip() for c in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                    power.append(float(p[3]))
                except ValueError:
                    continue
                for name, flag in zip(names, p[5:9]):
                    if flag.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "power_w_max": float(max(power)) if power else None,
                "reasons": sorted(reasons)}


# Source files each committed traffic record depends on (the kernel and its building blocks).
TRAFFIC_SOURCES = {
    "gemv_traffic.json": ("memq_dev.cuh", "memq_gemv_kernels.cuh", "memq_gemv_e4m3.cu",
                          "memq_gemv_blk128.cu", "memq_gemv_q8_0.cu"),
    "mla_traffic.json": ("memq_dev.cuh", "memq_mla.cu"),
}


def sources_sha256(record: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES[record]:
        with open(os.path.join(ROOT, "quantized_decode_memq_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(workload: str, record: str = "gemv_traffic.json"):
    """DRAM bytes per launch from the committed ncu capture of this workload, or None when there
    is none or the kernel's sources changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", record)) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if sources_sha256(record) != rec.get("kernel_sources_sha256"):
        return None
    return rec.get("dram_bytes_per_launch", {}).get(workload)


def measured_peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = json.load(f).get("hbm_gbs")
        if v:
            return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------------------------
# Workload
# ------------------------------------------------------------------------------------------

class DecodeStep:
    """Producer + GEMV with rotated weight copies, all buffers preallocated on the device."""

    def __init__(self, kind, out_f, in_f, m, copies, device, seed=0x51ED0002, fused=True):
        import torch
        import quantized_decode_memq_gb300 as memq
        from quantized_decode_memq_gb300 import synth
        self.memq = memq
        self.kind, self.out_f, self.in_f, self.m, self.copies = kind, out_f, in_f, m, copies
        self.device = device
        self.fused_step = fused
        x, wn = synth.activation_rows(in_f, m)
        self.x_host = x
        self.x = torch.from_numpy(x).to(device)
        self.wn = torch.from_numpy(wn).to(device)
        self.qs = torch.empty((m, in_f), dtype=torch.int8, device=device)
        self.d = torch.empty((m, in_f // 32), dtype=torch.float32, device=device)
        self.y = torch.empty((m, out_f), dtype=torch.float32, device=device)
        if kind == "q8_0":
            wh = synth.q8_0_bytes(seed, out_f, in_f)
            aux = None
        else:
            wh = synth.e4m3_bytes(seed + 1, out_f, in_f)
            if kind == "blk":
                aux = synth.grid_log2_uniform(seed + 2, out_f, in_f)
            else:
                aux = np.array([2.0 ** -4], np.float32)
        w0 = torch.from_numpy(wh).to(device)
        self.w = [w0] + [w0.clone() for _ in range(copies - 1)]
        self.aux = None if aux is None else [torch.from_numpy(aux).to(device) for _ in range(copies)]
        torch.cuda.synchronize()
        self.gemv_bytes = gemv_bytes(kind, out_f, in_f, m)
        self.step_bytes = self.gemv_bytes + producer_bytes(m, in_f)

    def producer(self):
        self.memq.memq_rmsnorm_q8_1(self.x, self.wn, 1e-6, qs=self.qs, d=self.d, want_z=False)

    def gemv(self, i):
        c = i % self.copies
        if self.kind == "q8_0":
            self.memq.memq_gemv_q8_0(self.w[c], self.qs, self.d, y=self.y)
        elif self.kind == "blk":
            self.memq.memq_gemv_e4m3_blk128(self.w[c], self.aux[c], self.qs, self.d, y=self.y)
        else:
            self.memq.memq_gemv_e4m3(self.w[c], self.aux[c], self.qs, self.d, y=self.y)

    def fused(self, i):
        """The whole decode step in one launch (RMSNorm -> q8_1 inside the GEMV)."""
        c = i % self.copies
        memq = self.memq
        if self.kind == "q8_0":
            memq.memq_rmsnorm_q8_1_gemv_q8_0(self.x, self.wn, self.w[c], 1e-6, qs=self.qs, d=self.d,
                                             y=self.y)
        elif self.kind == "blk":
            memq.memq_rmsnorm_q8_1_gemv_e4m3_blk128(self.x, self.wn, self.w[c], self.aux[c], 1e-6,
                                                    qs=self.qs, d=self.d, y=self.y)
        else:
            memq.memq_rmsnorm_q8_1_gemv_e4m3(self.x, self.wn, self.w[c], self.aux[c], 1e-6,
                                             qs=self.qs, d=self.d, y=self.y)

    def step(self, i):
        if self.fused_step:
            self.fused(i)
        else:
            self.producer()
            self.gemv(i)


class ProducerStep:
    """The RMSNorm -> q8_1 producer alone on rows x ncols (z written, as the fused producer of
    q8_fuse_gate.rs emits it); several input copies when one does not exceed L2."""

    def __init__(self, ncols, rows, device):
        import torch
        import quantized_decode_memq_gb300 as memq
        from quantized_decode_memq_gb300 import synth
        self.memq = memq
        self.ncols, self.rows = ncols, rows
        xb = rows * ncols * 4
        self.copies = max(1, min(16, -(-2 * L2_BYTES // xb)))
        x, wn = synth.activation_rows(ncols, rows, page_streams=rows * ncols <= 200000)
        x0 = torch.from_numpy(x).to(device)
        self.x = [x0] + [x0.clone() for _ in range(self.copies - 1)]
        self.wn = torch.from_numpy(wn).to(device)
        self.z = torch.empty((rows, ncols), dtype=torch.float32, device=device)
        self.qs = torch.empty((rows, ncols), dtype=torch.int8, device=device)
        self.d = torch.empty((rows, ncols // 32), dtype=torch.float32, device=device)
        self.step_bytes = producer_bytes(rows, ncols) + rows * ncols * 4  # + z written
        self.gemv_bytes = self.step_bytes
        self.launches_per_step = 1

    def step(self, i):
        self.memq.memq_rmsnorm_q8_1(self.x[i % self.copies], self.wn, 1e-6, z=self.z, qs=self.qs,
                                    d=self.d)


class SiluStep:
    """The silu(gate) * up -> q8_1 producer on rows x ncols (z written), rotated input copies."""

    def __init__(self, ncols, rows, device):
        import torch
        import quantized_decode_memq_gb300 as memq
        from quantized_decode_memq_gb300 import synth
        self.memq = memq
        xb = 2 * rows * ncols * 4
        self.copies = max(1, min(16, -(-2 * L2_BYTES // xb)))
        g = torch.from_numpy(synth.uniform_pm4(0x7500, rows * ncols).reshape(rows, ncols)).to(device)
        u = torch.from_numpy(synth.uniform_pm4(0x7501, rows * ncols).reshape(rows, ncols)).to(device)
        self.g = [g] + [g.clone() for _ in range(self.copies - 1)]
        self.u = [u] + [u.clone() for _ in range(self.copies - 1)]
        self.z = torch.empty((rows, ncols), dtype=torch.float32, device=device)
        self.qs = torch.empty((rows, ncols), dtype=torch.int8, device=device)
        self.d = torch.empty((rows, ncols // 32), dtype=torch.float32, device=device)
        self.step_bytes = rows * ncols * (4 + 4 + 4 + 1) + rows * ncols // 32 * 4
        self.launches_per_step = 1

    def step(self, i):
        c = i % self.copies
        self.memq.memq_silu_mul_q8_1(self.g[c], self.u[c], z=self.z, qs=self.qs, d=self.d)


class RepackStep:
    """E4M3 (per-tensor or block-128) -> Q8_0 slab, rotated source copies."""

    def __init__(self, kind, out_f, in_f, device):
        import torch
        import quantized_decode_memq_gb300 as memq
        from quantized_decode_memq_gb300 import synth
        self.memq, self.kind = memq, kind
        src = out_f * in_f
        self.copies = max(2, min(16, -(-2 * L2_BYTES // src)))
        w = torch.from_numpy(synth.e4m3_bytes(0x7600, out_f, in_f)).to(device)
        self.w = [w] + [w.clone() for _ in range(self.copies - 1)]
        if kind == "blk":
            self.aux = torch.from_numpy(synth.grid_log2_uniform(0x7601, out_f, in_f)).to(device)
        else:
            self.aux = torch.tensor([2.0 ** -4], dtype=torch.float32, device=device)
        self.out = [torch.empty((out_f, in_f // 32 * 34), dtype=torch.uint8, device=device)
                    for _ in range(2)]
        self.step_bytes = src + src // 32 * 34 + self.aux.numel() * 4
        self.launches_per_step = 1

    def step(self, i):
        c = i % self.copies
        fn = (self.memq.memq_repack_e4m3_blk128_q8_0 if self.kind == "blk"
              else self.memq.memq_repack_e4m3_q8_0)
        fn(self.w[c], self.aux, out=self.out[i % 2])


class StackStep:
    """One decode token through a synthetic 48-layer stack of block-128 E4M3 GEMVs at m = 1.

    Per layer: norm(5120) -> q; G 5120->6144 and G 5120->5120 on q; norm(5120 output) -> q';
    G 5120->17408 (gate) and G 5120->17408 (up) on q'; norm(17408 up output) -> q'';
    G 17408->5120 on q''; its output feeds the next layer.  Every layer has its own copy of the
    weights and grids (15.6 GB in all), so every GEMV reads DRAM."""

    SHAPES = ((6144, 5120), (5120, 5120), (17408, 5120), (17408, 5120), (5120, 17408))

    def __init__(self, layers, device, seed=0x57AC0000, fused=False, grouped=False):
        import torch
        import quantized_decode_memq_gb300 as memq
        from quantized_decode_memq_gb300 import synth
        self.memq = memq
        self.layers = layers
        dev = device
        base_w, base_g = [], []
        for k, (o, i) in enumerate(self.SHAPES):
            base_w.append(torch.from_numpy(synth.e4m3_bytes(seed + k, o, i)).to(dev))
            base_g.append(torch.from_numpy(synth.grid_log2_uniform(seed + 16 + k, o, i)).to(dev))
        self.w = [[bw.clone() for bw in base_w] for _ in range(layers)]
        self.g = [[bg.clone() for bg in base_g] for _ in range(layers)]
        del base_w, base_g
        self.wn = [torch.from_numpy(synth.uniform_pm4(seed + 32 + k, n)).to(dev)
                   for k, n in enumerate((5120, 5120, 17408))]
        x, _ = synth.activation_rows(5120, 1)
        self.x0 = torch.from_numpy(x).to(dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.y = [torch.empty((1, o), **f32) for (o, _) in self.SHAPES]
        self.qs = [torch.empty((1, n), dtype=torch.int8, device=dev) for n in (5120, 5120, 17408)]
        self.d = [torch.empty((1, n // 32), **f32) for n in (5120, 5120, 17408)]
        self.gemv_bytes = sum(gemv_bytes("blk", o, i, 1) for (o, i) in self.SHAPES)
        self.step_bytes = layers * (self.gemv_bytes + producer_bytes(1, 5120) * 2 +
                                    producer_bytes(1, 17408))
        self.fused, self.grouped = fused, grouped
        self.launches_per_step = (5 if fused else 6 if grouped else 8) * layers
        torch.cuda.synchronize()

    def layer(self, l, x):
        m = self.memq
        w, g, y, qs, d = self.w[l], self.g[l], self.y, self.qs, self.d
        m.memq_rmsnorm_q8_1(x, self.wn[0], 1e-6, qs=qs[0], d=d[0], want_z=False)
        m.memq_gemv_e4m3_blk128(w[0], g[0], qs[0], d[0], y=y[0])
        m.memq_gemv_e4m3_blk128(w[1], g[1], qs[0], d[0], y=y[1])
        m.memq_rmsnorm_q8_1(y[1], self.wn[1], 1e-6, qs=qs[1], d=d[1], want_z=False)
        m.memq_gemv_e4m3_blk128(w[2], g[2], qs[1], d[1], y=y[2])
        m.memq_gemv_e4m3_blk128(w[3], g[3], qs[1], d[1], y=y[3])
        m.memq_rmsnorm_q8_1(y[3], self.wn[2], 1e-6, qs=qs[2], d=d[2], want_z=False)
        m.memq_gemv_e4m3_blk128(w[4], g[4], qs[2], d[2], y=y[4])
        return y[4]

    def layer_fused(self, l, x):
        """The same layer with each RMSNorm -> q8_1 fused into the GEMV that first reads it (the
        fused call publishes qs / d, which the second GEMV on the same activation reads)."""
        m = self.memq
        w, g, y, qs, d = self.w[l], self.g[l], self.y, self.qs, self.d
        m.memq_rmsnorm_q8_1_gemv_e4m3_blk128(x, self.wn[0], w[0], g[0], 1e-6, qs=qs[0], d=d[0], y=y[0])
        m.memq_gemv_e4m3_blk128(w[1], g[1], qs[0], d[0], y=y[1])
        m.memq_rmsnorm_q8_1_gemv_e4m3_blk128(y[1], self.wn[1], w[2], g[2], 1e-6, qs=qs[1], d=d[1], y=y[2])
        m.memq_gemv_e4m3_blk128(w[3], g[3], qs[1], d[1], y=y[3])
        m.memq_rmsnorm_q8_1_gemv_e4m3_blk128(y[3], self.wn[2], w[4], g[4], 1e-6, qs=qs[2], d=d[2], y=y[4])
        return y[4]

    def layer_grouped(self, l, x):
        """The same layer with the GEMVs that share an activation in one launch each (5120->6144
        with 5120->5120; gate with up): 6 launches."""
        m = self.memq
        w, g, y, qs, d = self.w[l], self.g[l], self.y, self.qs, self.d
        m.memq_rmsnorm_q8_1(x, self.wn[0], 1e-6, qs=qs[0], d=d[0], want_z=False)
        m.memq_gemv_e4m3_blk128_group(w[0:2], g[0:2], qs[0], d[0], ys=y[0:2])
        m.memq_rmsnorm_q8_1(y[1], self.wn[1], 1e-6, qs=qs[1], d=d[1], want_z=False)
        m.memq_gemv_e4m3_blk128_group(w[2:4], g[2:4], qs[1], d[1], ys=y[2:4])
        m.memq_rmsnorm_q8_1(y[3], self.wn[2], 1e-6, qs=qs[2], d=d[2], want_z=False)
        m.memq_gemv_e4m3_blk128(w[4], g[4], qs[2], d[2], y=y[4])
        return y[4]

    def step(self, i):
        x = self.x0
        for l in range(self.layers):
            if self.fused:
                x = self.layer_fused(l, x)
            elif self.grouped:
                x = self.layer_grouped(l, x)
            else:
                x = self.layer(l, x)


def capture(fn, n, stream):
    """A CUDA graph of fn(0..n-1) launched on `stream`."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(n):
            fn(i)
    return g


def run_ours(args, world, rank, local):
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from quantized_decode_memq_gb300 import build
    build.build()
    if args.workload.split("_")[0] in ("producer", "silu", "repack") or args.workload.startswith("stack"):
        return run_other(args, world, rank, local, dev)
    if args.workload == "c3":
        return run_c3(args, world, rank, local, dev)
    if args.workload.startswith("mla_"):
        return run_mla(args, world, rank, local, dev)
    kind, out_f, in_f, m, copies = parse_workload(args.workload)
    fused = args.step == "fused"
    wl = DecodeStep(kind, out_f, in_f, m, copies, dev, fused=fused)
    stream = torch.cuda.Stream(device=dev)
    if args.ncu_launches:
        # Profiling entry: one producer launch, then N GEMV launches over the rotated copies.
        with torch.cuda.stream(stream):
            wl.producer()
            for i in range(args.ncu_launches):
                wl.step(i) if fused else wl.gemv(i)
        stream.synchronize()
        assert wl.memq.memq_device_fault(stream) == 0
        print(json.dumps({"ncu_launches": args.ncu_launches, "workload": args.workload}))
        return

    # Eager warm-up of every launch shape (sets kernel attributes outside any capture).
    with torch.cuda.stream(stream):
        for i in range(copies):
            wl.step(i)
    stream.synchronize()

    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        g_full = capture(wl.step, copies, stream)
        rem = K % copies
        g_rem = capture(wl.step, rem, stream) if rem else None
    reps = K // copies

    # Warm-up: W steps (rounded up to whole graphs).
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-W // copies))):
            g_full.replay()
    stream.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    elapsed = e0.elapsed_time(e1) / 1e3
    t_max, units = aggregate(elapsed, float(K * wl.step_bytes))
    value = units / t_max / 1e9
    ms_per_step = t_max / K * 1e3

    # Roofline: the dominant kernel -- the fused decode-step kernel (whole step's bytes) or the
    # GEMV (GEMV bytes) -- one launch at a time, DRAM-cold (rotated copies).
    launch_fn = wl.fused if fused else wl.gemv
    launch_bytes = wl.step_bytes if fused else wl.gemv_bytes
    # Average launch duration of the kernel in a decode loop: a CUDA graph of back-to-back
    # launches over the rotated copies (each launch reads its own weights from DRAM), CUDA
    # events around the replays.  Also reported: one launch at a time, event-bracketed, which
    # adds the launch and teardown latency outside the kernel's execution.
    b2b_s = time_gemv_back_to_back(wl, stream, n=16 * copies, fn=launch_fn)
    achieved = launch_bytes / b2b_s / 1e9
    gemv_s = time_gemv_launches(wl, stream, n=max(64, 4 * copies), fn=launch_fn)
    peak, peak_kind = measured_peak_hbm()

    e2e = time_e2e(wl, stream, steps=min(K, args.e2e_steps), graphs=True)
    e2e_t, e2e_units = aggregate(e2e["elapsed"], float(e2e["steps"] * wl.step_bytes))
    eager = time_e2e(wl, stream, steps=min(K, args.e2e_steps))
    eager_t, eager_units = aggregate(eager["elapsed"], float(eager["steps"] * wl.step_bytes))

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8" if kind == "q8_0" else "fp8",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: RMSNorm->q8_1 ({m}x{in_f} f32) then "
                        f"{kind} GEMV out_f={out_f} in_f={in_f} m={m}",
            "step": "one fused launch (memq_rmsnorm_q8_1_gemv_*)" if fused else
                    "two launches (memq_rmsnorm_q8_1 + memq_gemv_*)",
            "weight_copies": copies,
            "rotation_bytes": copies * (wl.gemv_bytes - m * (in_f + in_f // 8)),
            "l2": "inputs larger than L2: each step reads the next of the rotated weight "
                  "copies (DRAM-cold)",
            "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
            "step_bytes": wl.step_bytes,
            "timing": "K steps replayed from CUDA graphs, CUDA events on the launch stream",
        },
        "pct_of_peak": round(100.0 * value / peak, 2),
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": args.traffic if args.traffic is not None else profiled_traffic(args.workload),
            "kernel": f"gemv_stream_kernel<{kind}, m={m}, fused={fused}>",
            "bytes_per_launch": launch_bytes,
            "launch_us": round(b2b_s * 1e6, 3),
            "launch_timing": "average period of back-to-back launches in a CUDA graph",
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                           else "fallback 6.8 TB/s",
            "isolated_launch_us": round(gemv_s * 1e6, 3),
            "isolated_gbs": round(launch_bytes / gemv_s / 1e9, 2),
        },
        "e2e": {
            "value": round(e2e_units / e2e_t / 1e9, 3),
            "unit": "GB/s",
            "h2d_bytes_per_step": e2e["h2d"],
            "d2h_bytes_per_step": e2e["d2h"],
            "steps": e2e["steps"],
            "us_per_step": round(e2e_t / e2e["steps"] * 1e6, 2),
            "mode": "per step: one replay of a CUDA graph holding the public-API calls "
                    "(H2D of x from pinned memory, producer, GEMV, D2H of y), then a host wait",
            "eager": {"value": round(eager_units / eager_t / 1e9, 3),
                      "us_per_step": round(eager_t / eager["steps"] * 1e6, 2),
                      "mode": "the same calls issued from Python every step"},
        },
        "gpu_launches": (1 if fused else 2) * K,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_c3(args, world, rank, local, dev, out_f=17408, in_f=5120, rounds=15):
    """The three containers on the same 17408 x 5120 shape at m = 1, interleaved: per arm a CUDA
    graph of back-to-back GEMV launches over its own rotated weight copies; the graphs are
    replayed in turn (E4M3, block-128, Q8_0) for `rounds` rounds, each replay timed with CUDA
    events; per arm the median launch period.  Reports the Q8_0 : E4M3 time ratio next to the
    1.0625 byte ratio."""
    import torch
    from quantized_decode_memq_gb300 import build
    build.build()
    arms = {}
    for kind in ("e4m3", "blk", "q8_0"):
        copies = max(4, -(-2 * L2_BYTES // gemv_bytes(kind, out_f, in_f, 1)))
        arms[kind] = DecodeStep(kind, out_f, in_f, 1, copies, dev, fused=False)
    stream = torch.cuda.Stream(device=dev)
    graphs, n = {}, {}
    with torch.cuda.stream(stream):
        for kind, wl in arms.items():
            wl.producer()
            for i in range(wl.copies):
                wl.gemv(i)
            n[kind] = 8 * wl.copies
            graphs[kind] = capture(wl.gemv, n[kind], stream)
            for _ in range(max(1, args.warmup // n[kind] + 1)):
                graphs[kind].replay()
    stream.synchronize()
    times = {k: [] for k in arms}
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(rounds):
        for kind in arms:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                graphs[kind].replay()
                e1.record(stream)
            stream.synchronize()
            times[kind].append(e0.elapsed_time(e1) * 1e3 / n[kind])
    clocks = sampler.stop()
    peak, peak_kind = measured_peak_hbm()
    res = {}
    for kind, wl in arms.items():
        us = float(np.median(times[kind]))
        gbs = wl.gemv_bytes / us / 1e3
        res[kind] = {"us": round(us, 3), "gb_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                     "bytes": wl.gemv_bytes, "spread_us": [round(min(times[kind]), 3),
                                                           round(max(times[kind]), 3)]}
    tot_bytes = sum(wl.gemv_bytes for wl in arms.values())
    tot_us = sum(r["us"] for r in res.values())
    line = {"metric": METRIC, "value": round(tot_bytes / tot_us / 1e3, 2), "unit": "GB/s",
            "n_gpus": world, "steps": rounds * sum(n.values()), "warmup": args.warmup,
            "ms_per_step": tot_us / 3 / 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8+int8", "data": "synthetic",
            "config": {"workload": f"c3: E4M3, block-128 and Q8_0 GEMV {out_f}x{in_f} m=1, "
                                   f"interleaved arms, rotated weight copies (DRAM-cold)",
                       "timing": "per arm: median over rounds of the launch period of a graph "
                                 "of back-to-back launches"},
            "arms": res,
            "q8_0_to_e4m3_time_ratio": round(res["q8_0"]["us"] / res["e4m3"]["us"], 4),
            "q8_0_to_blk128_time_ratio": round(res["q8_0"]["us"] / res["blk"]["us"], 4),
            "blk128_to_e4m3_time_ratio": round(res["blk"]["us"] / res["e4m3"]["us"], 4),
            "byte_ratio": round(arms["q8_0"].gemv_bytes / arms["e4m3"].gemv_bytes, 4),
            "peak": {"hbm_gbs": peak, "source": peak_kind},
            "gpu_launches": rounds * sum(n.values()), "clocks": clocks}
    if rank == 0:
        print(json.dumps(line), flush=True)


class MlaStep:
    """One MLA decode attention kernel at the geometry of mla_decode_arm_gate.rs: 64 heads,
    kv_rank 512, d_nope = d_v = 256, d_rope 0, 2048 gathered slots from a pool of kv rows."""

    def __init__(self, kernel, t, kv, device, split=0):
        import torch
        import quantized_decode_memq_gb300 as memq
        from quantized_decode_memq_gb300 import synth
        self.memq, self.kernel, self.t, self.split = memq, kernel, t, split
        nh, kvr = synth.MLA_NH, synth.MLA_KV_RANK
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
        if kernel == "step":
            # the whole attention step: absorb_q -> attn_gathered -> decompress_v, each kernel's
            # output the next one's input
            q_nope, wk = synth.mla_absorb_inputs(t)
            _, wv = synth.mla_decompress_inputs(t)
            _, _, cache, idx = synth.mla_attn_inputs(t, kv)
            self.q_nope, self.wk, self.wv = dev(q_nope), dev(wk), dev(wv)
            self.cache, self.idx = dev(cache), dev(idx)
            self.q_lat = torch.empty((t, nh, kvr), dtype=torch.float32, device=device)
            self.o_lat = torch.empty((t, nh, kvr), dtype=torch.float32, device=device)
            self.out = torch.empty((t, nh, wv.shape[1]), dtype=torch.float32, device=device)
            n_slots = idx.shape[1]
            self.step_bytes = wk.nbytes + wv.nbytes + t * n_slots * kvr * 4
            self.flops = 2 * t * (wk.size + wv.size) + t * nh * n_slots * (2 * kvr + 2 * kvr)
        elif kernel == "attn":
            q_lat, _, cache, idx = synth.mla_attn_inputs(t, kv)
            self.args = (dev(q_lat), None, dev(cache), dev(idx), synth.MLA_SCALE)
            n_slots = idx.shape[1]
            self.out = torch.empty((t, nh, kvr), dtype=torch.float32, device=device)
            # gathered rows once per query row, the queries, the indices, the output
            self.step_bytes = t * n_slots * kvr * 4 + q_lat.nbytes + idx.nbytes + self.out.numel() * 4
            self.flops = t * nh * n_slots * (2 * kvr + 2 * kvr)
        else:
            x, w = (synth.mla_absorb_inputs(t) if kernel == "absorb"
                    else synth.mla_decompress_inputs(t))
            # rotated weight copies (past twice the L2) for the back-to-back loop timing
            self.copies = max(2, -(-2 * L2_BYTES // w.nbytes))
            w0 = dev(w)
            self.w = [w0] + [w0.clone() for _ in range(self.copies - 1)]
            self.args = (dev(x), w0)
            self.out = torch.empty((t, nh, w.shape[1]), dtype=torch.float32, device=device)
            self.step_bytes = w.nbytes + x.nbytes + self.out.numel() * 4
            self.flops = 2 * t * w.size
        # L2 scrub: 256 MB READ through the SMs (a written scrub would leave L2 full of dirty
        # lines whose write-back the timed kernel would pay for)
        self.scrub = torch.ones(256 * 2 ** 20 // 4, dtype=torch.float32, device=device)
        self.scrub_out = torch.empty((), dtype=torch.float32, device=device)
        self.launches_per_step = 1

    def flush(self):
        import torch
        torch.sum(self.scrub, dim=0, out=self.scrub_out)

    def chain_part(self, k):
        """Kernel k of the whole step (0 absorb_q, 1 attn_gathered, 2 decompress_v)."""
        m = self.memq
        if k == 0:
            m.memq_mla_absorb_q(self.q_nope, self.wk, out=self.q_lat, split=self.split)
        elif k == 1:
            from quantized_decode_memq_gb300 import synth
            m.memq_mla_attn_gathered(self.q_lat, None, self.cache, self.idx, synth.MLA_SCALE,
                                     out=self.o_lat, split=self.split)
        else:
            m.memq_mla_decompress_v(self.o_lat, self.wv, out=self.out, split=self.split)

    def step(self, i):
        if self.kernel == "step":
            for k in range(3):
                self.chain_part(k)
            return
        fn = {"attn": self.memq.memq_mla_attn_gathered, "absorb": self.memq.memq_mla_absorb_q,
              "decompress": self.memq.memq_mla_decompress_v}[self.kernel]
        args = self.args if self.kernel == "attn" else (self.args[0], self.w[i % self.copies])
        fn(*args, out=self.out, split=self.split)


def run_mla(args, world, rank, local, dev):
    """mla_<absorb|decompress>_t<t> and mla_attn_t<t>_kv<kv>: each timed launch follows a 256 MB
    L2 scrub read (outside the events), as the page times its kernels from the cold L2 that the
    expert stream between two MLA layers leaves."""
    import torch
    from quantized_decode_memq_gb300 import build
    build.build()
    parts = args.workload.split("_")
    kernel, t = parts[1], int(parts[2][1:])
    kv = int(parts[3][2:]) if kernel in ("attn", "step") else 0
    wl = MlaStep(kernel, t, kv, dev, split=args.split)
    stream = torch.cuda.Stream(device=dev)
    K, W = min(args.steps, 400), min(args.warmup, 50)  # one scrub + one launch per sample
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(W):
            wl.flush()
            wl.step(i)
    stream.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    with torch.cuda.stream(stream):
        for i in range(K):
            wl.flush()
            evs[i][0].record(stream)
            wl.step(i)
            evs[i][1].record(stream)
    stream.synchronize()
    barrier()
    clocks = sampler.stop()
    per = [a.elapsed_time(b) / 1e3 for a, b in evs]
    t_launch, _ = aggregate(float(np.mean(per)), 1.0)
    if kernel in ("attn", "step"):
        achieved = wl.flops / t_launch / 1e12
        peak = F32_FMA_TFLOPS
        roof = {"bound": "alu", "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "traffic": profiled_traffic(args.workload, "mla_traffic.json"),
                "peak_kind": "derived: 152 SMs x 128 f32 FMA/clk x 2 FLOP x 2.07 GHz"}
        if kernel == "step":
            # the same kernels one at a time (each after its own scrub), for the overlap gain
            iso = []
            for k in range(3):
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(20)]
                with torch.cuda.stream(stream):
                    for a_, b_ in ev:
                        wl.flush()
                        a_.record(stream)
                        wl.chain_part(k)
                        b_.record(stream)
                stream.synchronize()
                iso.append(float(np.mean([a_.elapsed_time(b_) for a_, b_ in ev])) * 1e3)
            roof["isolated_us"] = {"absorb_q": round(iso[0], 2), "attn_gathered": round(iso[1], 2),
                                   "decompress_v": round(iso[2], 2), "sum": round(sum(iso), 2)}
            roof["traffic"] = None
    else:
        peak, peak_kind = measured_peak_hbm()
        achieved = wl.step_bytes / t_launch / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": profiled_traffic(args.workload, "mla_traffic.json"), "peak_kind": peak_kind}
        # decode-loop view: back-to-back launches over the rotated weight copies (DRAM-cold)
        loop_s = time_gemv_back_to_back(wl, stream, wl.copies, fn=wl.step)
        roof["loop_period_us"] = round(loop_s * 1e6, 3)
        roof["loop_gbs"] = round(wl.step_bytes / loop_s / 1e9, 1)
        roof["loop_frac"] = round(wl.step_bytes / loop_s / 1e9 / peak, 4)
    desc = {"absorb": f"mla_absorb_q t={t}: 64 heads x (512 x 256) f32 weights",
            "decompress": f"mla_decompress_v t={t}: 64 heads x (256 x 512) f32 weights",
            "attn": f"mla_attn_gathered t={t}: 64 heads, kv_rank 512, 2048 slots from {kv} rows",
            "step": f"MLA attention step t={t}: absorb_q -> attn_gathered (2048 slots from {kv} "
                    f"rows) -> decompress_v, back to back"}
    line = {"metric": ("MLA attention step time (L2 scrubbed before each)" if kernel == "step" else
                       "MLA decode kernel time per launch (L2 scrubbed before each)"),
            "value": round(t_launch * 1e6, 3), "unit": "us", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": t_launch * 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": desc[kernel], "split": args.split or "auto",
                       "step_bytes": wl.step_bytes, "flops": wl.flops,
                       "timing": "one launch per sample after a 256 MB scrub read, CUDA events",
                       "min_us": round(min(per) * 1e6, 3)},
            "roofline": roof, "gpu_launches": K * (3 if kernel == "step" else 1), "clocks": clocks}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if kernel == "step":
            cb = [cpu_baseline_mla(k, t, kv, min(args.cpu_seconds, 10.0) / 3)
                  for k in ("absorb", "attn", "decompress")]
            line["cpu_baseline"] = dict(cb[1], value=round(sum(c["value"] for c in cb), 1),
                                        sample="sum of the three kernels' oracle samples: " +
                                               "; ".join(c["sample"] for c in cb))
        else:
            line["cpu_baseline"] = cpu_baseline_mla(kernel, t, kv, min(args.cpu_seconds, 10.0))
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_other(args, world, rank, local, dev):
    """Producer sweep (producer_<ncols>x<rows>) and the decode stack (stack<layers>): K steps
    replayed from a CUDA graph, whole-step algorithmic bytes / device time."""
    import torch
    from quantized_decode_memq_gb300 import build
    build.build()
    if args.workload.startswith("producer_"):
        ncols, rows = (int(v) for v in args.workload[len("producer_"):].split("x"))
        wl = ProducerStep(ncols, rows, dev)
        per_graph = wl.copies
        desc = f"{args.workload}: RMSNorm->q8_1 producer, {rows} rows x {ncols} (z written)"
    elif args.workload.startswith("silu_"):
        ncols, rows = (int(v) for v in args.workload[len("silu_"):].split("x"))
        wl = SiluStep(ncols, rows, dev)
        per_graph = wl.copies
        desc = f"{args.workload}: silu(gate) * up -> q8_1 producer, {rows} rows x {ncols} (z written)"
    elif args.workload.startswith("repack_"):
        kind, shape = args.workload[len("repack_"):].split("_")
        kind = "blk" if kind == "blk128" else kind
        out_f, in_f = (int(v) for v in shape.split("x"))
        wl = RepackStep(kind, out_f, in_f, dev)
        per_graph = wl.copies
        desc = (f"{args.workload}: E4M3 ({'block-128 grid' if kind == 'blk' else 'per-tensor scale'})"
                f" -> Q8_0 slab, {out_f}x{in_f}, read 1 B + write 1.0625 B per weight")
    else:
        layers = int(args.workload[len("stack"):] or 48)
        fused, grouped = args.step == "fused", args.step == "group"
        wl = StackStep(layers, dev, fused=fused, grouped=grouped)
        per_graph = 1
        desc = (f"{args.workload}: one token through {layers} layers of block-128 E4M3 GEMVs "
                f"(5120->6144, 5120->5120, 5120->17408 x2, 17408->5120) with 3 RMSNorm->q8_1 "
                + ("fused into the GEMVs (5 launches per layer)" if fused else
                   "producers, GEMVs on one activation grouped (6 launches per layer)" if grouped
                   else "producers each (8 launches per layer)"))
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(per_graph):
            wl.step(i)
    stream.synchronize()
    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        g = capture(wl.step, per_graph, stream)
        for _ in range(max(1, -(-W // per_graph))):
            g.replay()
    stream.synchronize()
    reps = max(1, -(-K // per_graph))
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    barrier()
    clocks = sampler.stop()
    steps = reps * per_graph
    t_max, units = aggregate(e0.elapsed_time(e1) / 1e3, float(steps * wl.step_bytes))
    peak, peak_kind = measured_peak_hbm()
    value = units / t_max / 1e9
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": W, "ms_per_step": t_max / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if args.workload.split("_")[0] in ("producer", "silu") else "fp8",
            "data": "synthetic",
            "config": {"workload": desc, "step_bytes": wl.step_bytes,
                       "timing": "steps replayed from a CUDA graph, CUDA events"},
            "pct_of_peak": round(100.0 * value / peak, 2),
            "gpu_launches": wl.launches_per_step * steps, "clocks": clocks}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.workload.startswith("stack"):
        line["cpu_baseline"] = cpu_baseline_other(args.workload, min(args.cpu_seconds, 10.0))
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_gemv_launches(wl, stream, n, fn=None):
    """Mean duration of n individually bracketed launches of fn (rotated copies)."""
    import torch
    fn = fn or wl.gemv
    try:
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n)]

        def body(i):
            evs[i][0].record(stream)
            fn(i)
            evs[i][1].record(stream)
        with torch.cuda.stream(stream):
            g = capture(body, n, stream)
            for _ in range(3):
                g.replay()
        stream.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs])) / 1e3
    except TypeError:
        # No event-record graph nodes in this torch: queue each launch behind a GPU-side spin so
        # the CPU enqueue time never lands between the two events.
        res = []
        with torch.cuda.stream(stream):
            for i in range(n):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                torch.cuda._sleep(200000)
                a.record(stream)
                fn(i)
                b.record(stream)
                stream.synchronize()
                res.append(a.elapsed_time(b))
        return float(np.mean(res[3:] if len(res) > 8 else res)) / 1e3


def time_gemv_back_to_back(wl, stream, n, fn=None):
    import torch
    with torch.cuda.stream(stream):
        g = capture(fn or wl.gemv, n, stream)
        g.replay()
        stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(4):
            g.replay()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / 1e3 / (4 * n)


def time_e2e(wl, stream, steps, graphs=False):
    """Public API with host buffers: per step the H2D copy of the activation row (pinned), the
    chain, the D2H copy of y and a host wait for it.  With graphs=True each step is one replay of
    a CUDA graph that captured exactly those public-API calls (one graph per rotated weight
    copy), the way a caller removes the per-call launch overhead of a decode loop."""
    import torch
    x_pin = torch.from_numpy(wl.x_host.copy()).pin_memory()
    y_pin = torch.empty(wl.y.shape, dtype=torch.float32).pin_memory()
    h2d = x_pin.numel() * 4
    d2h = y_pin.numel() * 4

    def one(i):
        wl.x.copy_(x_pin, non_blocking=True)
        wl.step(i)
        y_pin.copy_(wl.y, non_blocking=True)

    run = one
    if graphs:
        gs = []
        with torch.cuda.stream(stream):
            for c in range(wl.copies):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                    one(c)
                gs.append(g)
        run = lambda i: gs[i % len(gs)].replay()  # noqa: E731
    with torch.cuda.stream(stream):
        for i in range(8):
            run(i)
            stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record(stream)
        for i in range(steps):
            run(i)
            stream.synchronize()
        b.record(stream)
        stream.synchronize()
        wall = time.perf_counter() - t0
    return {"elapsed": max(wall, a.elapsed_time(b) / 1e3), "steps": steps, "h2d": h2d, "d2h": d2h}


# ------------------------------------------------------------------------------------------
# The oracle on the host cores (CPU baseline and the reference arm)
# ------------------------------------------------------------------------------------------

def _oracle_inputs(kind, out_f, in_f, m, seed=0x51ED0002):
    from quantized_decode_memq_gb300 import synth
    x, wn = synth.activation_rows(in_f, m)
    if kind == "q8_0":
        return x, wn, synth.q8_0_bytes(seed, out_f, in_f), None
    w = synth.e4m3_bytes(seed + 1, out_f, in_f)
    aux = synth.grid_log2_uniform(seed + 2, out_f, in_f) if kind == "blk" else 2.0 ** -4
    return x, wn, w, aux


def _oracle_step(oracle, kind, x, wn, w, aux, in_f, rows=None):
    _, d, qs, _ = oracle.rmsnorm_q8_1(x, wn, 1e-6)
    if kind == "q8_0":
        return oracle.gemv_q8_0(w, in_f, qs, d, rows=rows)
    if kind == "blk":
        return oracle.gemv_e4m3_blk128(w, aux, qs, d, rows=rows)
    return oracle.gemv_e4m3(w, aux, qs, d, rows=rows)


def _sample_bytes(kind, nrows, in_f, m):
    """Algorithmic bytes of one oracle step that computes `nrows` output rows."""
    return gemv_bytes(kind, nrows, in_f, m) - (4 if kind == "e4m3" else 0) + producer_bytes(m, in_f)


def cpu_baseline(wl, seconds):
    import oracle
    oracle.build()
    kind, out_f, in_f, m = wl.kind, wl.out_f, wl.in_f, wl.m
    x, wn, w, aux = _oracle_inputs(kind, out_f, in_f, m)
    _oracle_step(oracle, kind, x, wn, w, aux, in_f)  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(oracle, kind, x, wn, w, aux, in_f)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 10000:
            break
    return {"value": round(n * wl.step_bytes / el / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{n} full decode steps (f64 C oracle: producer + {kind} GEMV "
                      f"{out_f}x{in_f} m={m}), {el:.1f} s wall, single thread",
            "host_cpus": os.cpu_count()}


def _time_oracle(fn, seconds):
    """Calls fn until `seconds` of wall time have passed (at least twice); seconds per call."""
    fn()  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if (el >= seconds and n >= 2) or n >= 100000:
            return el / n, n, el


def cpu_baseline_other(workload, seconds):
    """The oracle on a bounded sample of a producer / silu / repack workload, scaled to the whole
    workload's bytes (GB/s, single thread)."""
    import oracle
    from quantized_decode_memq_gb300 import synth
    oracle.build()
    head, shape = workload.split("_", 1)
    if head == "repack":
        kind, dims = shape.split("_")
        out_f, in_f = (int(v) for v in dims.split("x"))
        rows = min(out_f, 256)
        w = synth.e4m3_bytes(0x7600, rows, in_f)
        grid = kind == "blk128"
        aux = (synth.grid_log2_uniform(0x7601, rows, in_f) if grid
               else np.array([2.0 ** -4], np.float32))
        per, n, el = _time_oracle(lambda: oracle.repack_q8_0(w, aux, grid), seconds)
        total = per * out_f / rows
        nbytes = out_f * in_f + out_f * in_f // 32 * 34
        sample = f"{n} x {rows} rows of {out_f} ({el:.1f} s)"
    else:
        ncols, rows_all = (int(v) for v in shape.split("x"))
        rows = min(rows_all, 64)
        g = synth.uniform_pm4(0x7500, rows * ncols).reshape(rows, ncols)
        if head == "silu":
            u = synth.uniform_pm4(0x7501, rows * ncols).reshape(rows, ncols)
            per, n, el = _time_oracle(lambda: oracle.silu_mul_q8_1(g, u), seconds)
            nbytes = rows_all * ncols * (4 + 4 + 4 + 1) + rows_all * ncols // 32 * 4
        else:
            wn = synth.uniform_pm4(0x7502, ncols)
            per, n, el = _time_oracle(lambda: oracle.rmsnorm_q8_1(g, wn), seconds)
            nbytes = producer_bytes(rows_all, ncols) + rows_all * ncols * 4
        total = per * rows_all / rows
        sample = f"{n} x {rows} rows of {rows_all} ({el:.1f} s)"
    return {"value": round(nbytes / total / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"f64 C oracle, {sample}, scaled to the whole workload", "host_cpus": os.cpu_count()}


def cpu_baseline_mla(kernel, t, kv, seconds):
    """The oracle on a bounded sample (a few heads) of an MLA launch, scaled to all 64 heads: us
    per launch, single thread."""
    import oracle
    from quantized_decode_memq_gb300 import synth
    oracle.build()
    nh_s = 2
    if kernel == "attn":
        q_lat, _, cache, idx = synth.mla_attn_inputs(t, kv)
        q = np.ascontiguousarray(q_lat[:, :nh_s])
        fn = lambda: oracle.mla_attn_gathered(q, None, cache, idx, synth.MLA_SCALE)  # noqa: E731
    else:
        x, w = synth.mla_absorb_inputs(t) if kernel == "absorb" else synth.mla_decompress_inputs(t)
        xs, ws = np.ascontiguousarray(x[:, :nh_s]), np.ascontiguousarray(w[:nh_s])
        fn = lambda: oracle.mla_head_gemv(xs, ws)  # noqa: E731
    per, n, el = _time_oracle(fn, seconds)
    return {"value": round(per * synth.MLA_NH / nh_s * 1e6, 1), "unit": "us", "cores": 1,
            "kind": "oracle", "sample": f"f64 C oracle, {n} calls on {nh_s} of {synth.MLA_NH} heads "
                                        f"({el:.1f} s), scaled to all heads",
            "host_cpus": os.cpu_count()}


def run_reference(args, world, rank):
    """The oracle as the timed arm: every step is the producer plus a bounded row sample of the
    GEMV, sized from a calibration step so that warm-up + K steps take about a minute."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    kind, out_f, in_f, m, copies = parse_workload(args.workload)
    x, wn, w, aux = _oracle_inputs(kind, out_f, in_f, m)
    t0 = time.perf_counter()
    _oracle_step(oracle, kind, x, wn, w, aux, in_f, rows=np.arange(min(out_f, 256)))
    per_row = (time.perf_counter() - t0) / min(out_f, 256)
    budget = 60.0 / max(1, args.steps + args.warmup)
    nrows = int(max(1, min(out_f, budget / max(per_row, 1e-9))))
    rng = np.random.default_rng(7)
    samples = [np.sort(rng.choice(out_f, size=nrows, replace=False)) for _ in range(8)]
    for i in range(args.warmup):
        _oracle_step(oracle, kind, x, wn, w, aux, in_f, rows=samples[i % 8])
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_step(oracle, kind, x, wn, w, aux, in_f, rows=samples[i % 8])
    el = time.perf_counter() - t0
    v = args.steps * _sample_bytes(kind, nrows, in_f, m) / el / 1e9
    sample = (f"each step: producer 1x{in_f} + {nrows} of {out_f} GEMV rows ({kind}, m={m}), "
              f"f64 C oracle, single thread")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 5),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: f64 C oracle of the same decode step "
                               f"(producer + {kind} GEMV out_f={out_f} in_f={in_f} m={m})",
                   "sample_rows_per_step": nrows},
        "cpu_baseline": {"value": round(v, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="one of %s, or <e4m3|blk128|q8_0>_<out_f>x<in_f>_m<m>, c3, "
                         "producer_<ncols>x<rows>, silu_<ncols>x<rows>, "
                         "repack_<e4m3|blk128>_<out_f>x<in_f>, stack<layers>, "
                         "mla_<absorb|decompress>_t<t>, mla_attn_t<t>_kv<kv>, mla_step_t<t>_kv<kv>"
                         % sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=3000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per GEMV launch from an ncu capture of this kernel")
    ap.add_argument("--step", choices=["fused", "split", "group"], default="split",
                    help="decode step as one fused launch or as producer + GEMV launches; "
                         "for the stack, 'group' runs the GEMVs that share an activation as one "
                         "grouped launch")
    ap.add_argument("--split", type=int, default=0,
                    help="MLA workloads: the kernels' split (0 = the library's choice)")
    ap.add_argument("--ncu-launches", type=int, default=0,
                    help="profiling entry: run one producer and N GEMV launches, no timing")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
