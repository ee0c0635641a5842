"""DRAM-cold benchmark of the quantized decode chain on GB300.

A step is one pass of the whole hot path over one synthetic decode token: the fused
RMSNorm -> q8_1 producer on the token's activation row, then the GEMV against that q8_1
activation, reading the next of several rotated weight copies so that no launch finds its
weights in L2.  The default workload (c3) is the m = 1 GEMV at 17408 x 5120 in all three
weight containers (E4M3, E4M3 + block-128 grid, Q8_0), interleaved in a rotating order, each
arm on rotated weight copies totalling more than the 129 MB L2.  --sweep c4 / c5 writes one
JSONL receipt per cell of the GEMV (container x shape x m) and producer grids.

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
              result y is copied device->host and the host waits for it.  Single-GEMV
              workloads add the one-native-call leg (memq_decode_step_host, through the
              binding and straight through the C ABI).
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
DEFAULT_WORKLOAD = "c3"
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
    "gemv_traffic.json": ("memq_dev.cuh", "memq_gemv_kernels.cuh", "memq_gemv_kouter.cuh",
                          "memq_gemv_e4m3.cu", "memq_gemv_blk128.cu", "memq_gemv_q8_0.cu"),
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


# TF32 / bf16 dense tensor throughput ratio (nominal: 1.1 and 2.25 PFLOP/s per GB300)
TF32_PER_BF16 = 1.1 / 2.25
FALLBACK_BF16_TFLOPS = 1900.0


def measured_peak_bf16():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = json.load(f).get("bf16_tflops")
        if v:
            return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


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

    def host_step(self, i, x_host, y_host):
        """The whole decode step for host-resident rows in one native call: x_host -> x, the
        fused step, y -> y_host, and the call's own wait for the stream."""
        c = i % self.copies
        container = {"q8_0": self.memq.Container.Q8_0, "blk": self.memq.Container.E4M3_BLK128,
                     "e4m3": self.memq.Container.E4M3}[self.kind]
        self.memq.memq_decode_step_host(container, x_host, self.x, self.wn, self.w[c],
                                        None if self.aux is None else self.aux[c], y_host, 1e-6,
                                        qs=self.qs, d=self.d, y_dev=self.y)


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


# Sweep grids: C4 (GEMV shapes x m, every container) and C5 (producer rows x widths).
C4_SHAPES = ((5120, 5120), (1024, 5120), (17408, 5120), (5120, 17408))
C4_M = (1, 2, 4, 8)
C5_SHAPES = tuple((ncols, rows) for ncols in (1536, 4096, 8192) for rows in (1, 8, 64, 4096))


def run_sweep(args, dev):
    """One JSONL receipt per cell of the C4 or C5 grid, written to --receipts (first record:
    the command and the peak), and one summary JSON line on stdout.  C4 cell: the GEMV's
    back-to-back period over rotated weight copies totalling more than twice the L2 (CUDA graph
    of 16 launches per copy, CUDA events), its algorithmic bytes, GB/s and fraction of the
    measured peak.  C5 cell: the producer's period per call (z written), from a CUDA graph over
    rotated input copies."""
    import torch
    peak, peak_kind = measured_peak_hbm()
    stream = torch.cuda.Stream(device=dev)
    path = args.receipts or f"{args.sweep}_receipts.jsonl"
    command = "python bench.py " + " ".join(a for a in sys.argv[1:])
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    cells = 0
    with open(path, "w") as f:
        f.write(json.dumps({"sweep": args.sweep, "command": command, "peak_gbs": peak,
                            "peak_source": peak_kind,
                            "timing": "CUDA events around graph replays, DRAM-cold (rotated "
                                      "copies > 2x L2)"}) + "\n")
        if args.sweep == "c4":
            for kind in ("blk", "q8_0", "e4m3"):
                for out_f, in_f in C4_SHAPES:
                    for m in C4_M:
                        wbytes = gemv_bytes(kind, out_f, in_f, m)
                        copies = max(4, -(-2 * L2_BYTES // wbytes))
                        wl = DecodeStep(kind, out_f, in_f, m, copies, dev, fused=False)
                        with torch.cuda.stream(stream):
                            wl.producer()
                            for i in range(copies):
                                wl.gemv(i)
                        stream.synchronize()
                        per = time_gemv_back_to_back(wl, stream, n=16 * copies)
                        fault = wl.memq.memq_device_fault(stream)
                        gbs = wbytes / per / 1e9
                        f.write(json.dumps({
                            "container": {"blk": "blk128", "q8_0": "q8_0", "e4m3": "e4m3"}[kind],
                            "out_f": out_f, "in_f": in_f, "m": m, "copies": copies,
                            "bytes_per_launch": wbytes, "period_us": round(per * 1e6, 3),
                            "gbs": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
                            "fault": fault}) + "\n")
                        f.flush()
                        cells += 1
                        del wl
                        torch.cuda.empty_cache()
        else:
            for ncols, rows in C5_SHAPES:
                wl = ProducerStep(ncols, rows, dev)
                with torch.cuda.stream(stream):
                    for i in range(wl.copies):
                        wl.step(i)
                    n = wl.copies * max(1, -(-64 // wl.copies))
                    g = capture(wl.step, n, stream)
                    g.replay()
                    stream.synchronize()
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for _ in range(4):
                        g.replay()
                    b.record(stream)
                stream.synchronize()
                per = a.elapsed_time(b) / 1e3 / (4 * n)
                fault = wl.memq.memq_device_fault(stream)
                gbs = wl.step_bytes / per / 1e9
                f.write(json.dumps({"ncols": ncols, "rows": rows, "copies": wl.copies,
                                    "bytes_per_call": wl.step_bytes,
                                    "period_us": round(per * 1e6, 3), "gbs": round(gbs, 1),
                                    "frac_of_measured": round(gbs / peak, 4),
                                    "fault": fault}) + "\n")
                f.flush()
                cells += 1
                del wl, g
                torch.cuda.empty_cache()
    clocks = sampler.stop()
    print(json.dumps({"sweep": args.sweep, "cells": cells, "receipts": path, "peak_gbs": peak,
                      "clocks": clocks}), flush=True)


def run_ours(args, world, rank, local):
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from quantized_decode_memq_gb300 import build
    build.build()
    if args.sweep:
        return run_sweep(args, dev)
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
    hcall = time_e2e_host_call(wl, stream, steps=min(K, args.e2e_steps))
    hcall_t, hcall_units = aggregate(hcall["elapsed"], float(hcall["steps"] * wl.step_bytes))
    ccall = time_e2e_c_abi(wl, stream, steps=min(K, args.e2e_steps))
    ccall_t, ccall_units = aggregate(ccall["elapsed"], float(ccall["steps"] * wl.step_bytes))

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
            "host_call": {"value": round(hcall_units / hcall_t / 1e9, 3),
                          "us_per_step": round(hcall_t / hcall["steps"] * 1e6, 2),
                          "mode": "one memq_decode_step_host call per step: H2D of x from "
                                  "pinned memory, the fused step, D2H of y and the wait, in "
                                  "one native call"},
            "host_call_c_abi": {"value": round(ccall_units / ccall_t / 1e9, 3),
                                "us_per_step": round(ccall_t / ccall["steps"] * 1e6, 2),
                                "mode": "the same C entry point called through ctypes with "
                                        "prepared arguments (no Python argument checks)"},
        },
        "gpu_launches": (1 if fused else 2) * K,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


C3_OUT_F, C3_IN_F = 17408, 5120
ARMS = ("e4m3", "blk", "q8_0")
ARM_NAMES = {"e4m3": "E4M3 (per-tensor scale)", "blk": "E4M3 block-128", "q8_0": "Q8_0"}
NOMINAL_HBM_GBS = 8000.0


def _median_event_us(pairs, div=1):
    return float(np.median([a.elapsed_time(b) * 1e3 / div for a, b in pairs]))


def time_isolated(fn, n, stream):
    """Median device time of n individually event-bracketed launches of fn(i) (rotated copies),
    each queued behind a GPU-side sleep so that no host latency lands between its events."""
    import torch
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
            res.append(a.elapsed_time(b) * 1e3)
    return float(np.median(res[2:] if len(res) > 6 else res))


class L2Scrub:
    """Evicts L2 with this library's own RMSNorm -> q8_1 kernel over a 256 MB activation: it reads
    256 MB and writes 256 MB of z plus 64 MB of q8_1 codes, more than twice the 129 MB L2 each
    way (as mla_decode_arm_gate.rs scrubs with an rms_norm pass before every timed launch)."""

    ROWS, NCOLS = 8192, 8192

    def __init__(self, device):
        import torch
        import quantized_decode_memq_gb300 as memq
        self.memq = memq
        self.x = torch.ones((self.ROWS, self.NCOLS), dtype=torch.float32, device=device)
        self.w = torch.ones(self.NCOLS, dtype=torch.float32, device=device)
        self.z = torch.empty_like(self.x)
        self.qs = torch.empty((self.ROWS, self.NCOLS), dtype=torch.int8, device=device)
        self.d = torch.empty((self.ROWS, self.NCOLS // 32), dtype=torch.float32, device=device)

    def __call__(self):
        self.memq.memq_rmsnorm_q8_1(self.x, self.w, 1e-6, qs=self.qs, d=self.d, z=self.z)


def time_isolated_scrubbed(fn, scrub, n, stream):
    """Median device time of n event-bracketed launches of fn(0) -- always the same weights --
    each right after an L2 scrub: the cross-check that the rotated copies leave every launch as
    cold as a scrubbed one."""
    import torch
    res = []
    with torch.cuda.stream(stream):
        for i in range(n):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            scrub()
            torch.cuda._sleep(200000)
            a.record(stream)
            fn(0)
            b.record(stream)
            stream.synchronize()
            res.append(a.elapsed_time(b) * 1e3)
    return float(np.median(res[2:] if len(res) > 6 else res))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def affinity_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_arms(arms, seconds):
    """The f64 oracle (producer + each arm's GEMV on a bounded row sample of the same shape) on
    the host cores: single-threaded, and with the rows split over every core of the process's
    affinity mask (one thread per core calling the unchanged oracle on its row range; the
    oracle's C loops run without the interpreter lock).  GB/s of the whole three-arm step,
    scaled from the sample's bytes; median of 3 timings each."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    ncores = affinity_cores()
    legs = []
    inputs = {kind: _oracle_inputs(kind, wl.out_f, wl.in_f, 1) for kind, wl in arms.items()}
    for cores in (1, ncores):
        per_arm = {}
        for kind, wl in arms.items():
            out_f, in_f = wl.out_f, wl.in_f
            x, wn, w, aux = inputs[kind]
            _, d, qs, _ = oracle.rmsnorm_q8_1(x, wn, 1e-6)
            # rows per timing: sized from a calibration so the three arms x 3 repeats x 2 legs
            # take about `seconds`
            probe = np.arange(min(out_f, 64))
            t0 = time.perf_counter()
            _oracle_gemv(oracle, kind, w, aux, qs, d, in_f, probe)
            per_row = (time.perf_counter() - t0) / len(probe)
            nrows = int(max(cores, min(out_f, seconds / 18.0 * cores / max(per_row, 1e-9))))
            rows = np.arange(nrows)
            chunks = np.array_split(rows, cores)
            times = []
            for _ in range(3):
                t0 = time.perf_counter()
                oracle.rmsnorm_q8_1(x, wn, 1e-6)
                if cores == 1:
                    _oracle_gemv(oracle, kind, w, aux, qs, d, in_f, rows)
                else:
                    with ThreadPoolExecutor(cores) as ex:
                        list(ex.map(lambda r: _oracle_gemv(oracle, kind, w, aux, qs, d, in_f, r),
                                    chunks))
                times.append(time.perf_counter() - t0)
            t = float(np.median(times))
            # whole-arm time: the sampled rows scaled to out_f (the producer is counted once)
            per_arm[kind] = {"rows_sampled": nrows, "s_per_launch": t * out_f / nrows}
        step_s = sum(v["s_per_launch"] for v in per_arm.values())
        in_f = next(iter(arms.values())).in_f
        step_bytes = sum(wl.gemv_bytes for wl in arms.values()) + producer_bytes(1, in_f)
        legs.append({"cores": cores, "value": round(step_bytes / step_s / 1e9, 5), "unit": "GB/s",
                     "ms_per_step": round(step_s * 1e3, 1),
                     "arms": {k: round(v["s_per_launch"] * 1e3, 2) for k, v in per_arm.items()},
                     "rows_sampled": {k: v["rows_sampled"] for k, v in per_arm.items()}})
    best = legs[-1]
    return {"value": best["value"], "unit": "GB/s", "cores": best["cores"], "kind": "oracle",
            "sample": "f64 C oracle: RMSNorm->q8_1 of the activation row, then each arm's GEMV on "
                      "a bounded sample of its output rows (the first rows), scaled to the whole "
                      "step; median of 3 timings", "legs": legs, "cpu_model": cpu_model(),
            "host_cpus": os.cpu_count()}


def _oracle_gemv(oracle, kind, w, aux, qs, d, in_f, rows):
    if kind == "q8_0":
        return oracle.gemv_q8_0(w, in_f, qs, d, rows=rows)
    if kind == "blk":
        return oracle.gemv_e4m3_blk128(w, aux, qs, d, rows=rows)
    return oracle.gemv_e4m3(w, aux, qs, d, rows=rows)


def run_c3(args, world, rank, local, dev, out_f=C3_OUT_F, in_f=C3_IN_F):
    """The default workload: the E4M3, block-128 and Q8_0 GEMVs on the 17408 x 5120 projection at
    m = 1, interleaved (gemv_e4m3_bench.rs, "THE BLOCK-128 ARM" and "PROTOCOL": all arms inside
    one iteration, each on its own rotated weight copies, medians of per-iteration times).

    A step: the RMSNorm -> q8_1 producer on the 5120-wide row, then for each arm -- in an order
    that rotates every step -- a CUDA graph of back-to-back launches over that arm's rotated
    copies (each launch reads weights no launch since has touched: the copies of one arm exceed
    twice the L2), with CUDA events between the arms.  The K timed steps are queued behind a GPU
    sleep so host launch latency never lands inside the region."""
    import torch
    stream = torch.cuda.Stream(device=dev)
    arms = {}
    for kind in ARMS:
        copies = max(4, -(-2 * L2_BYTES // gemv_bytes(kind, out_f, in_f, 1)))
        arms[kind] = DecodeStep(kind, out_f, in_f, 1, copies, dev, fused=False)
    lead = arms["e4m3"]
    for wl in arms.values():  # one activation shared by the three arms
        wl.x, wl.wn, wl.qs, wl.d = lead.x, lead.wn, lead.qs, lead.d
    # 16 launches per copy: each arm's graph boundary (its first launch starts without an
    # overlapping predecessor, and the events around it) is spread over 64 launches
    n = {k: 16 * wl.copies for k, wl in arms.items()}
    with torch.cuda.stream(stream):
        lead.producer()
        for wl in arms.values():
            for i in range(wl.copies):
                wl.gemv(i)
    stream.synchronize()
    with torch.cuda.stream(stream):
        graphs = {k: capture(wl.gemv, n[k], stream) for k, wl in arms.items()}
        g_prod = capture(lambda i: lead.producer(), 1, stream)
    stream.synchronize()

    def run_steps(K, record):
        evs = []
        with torch.cuda.stream(stream):
            torch.cuda._sleep(2_000_000)  # the host queues ahead while the GPU sleeps
            for s in range(K):
                order = ARMS[s % 3:] + ARMS[:s % 3]
                e = [torch.cuda.Event(enable_timing=True) for _ in range(5)] if record else None
                if record:
                    e[0].record(stream)
                g_prod.replay()
                if record:
                    e[1].record(stream)
                for j, kind in enumerate(order):
                    graphs[kind].replay()
                    if record:
                        e[2 + j].record(stream)
                if record:
                    evs.append((order, e))
        return evs

    K, W = args.steps, args.warmup
    run_steps(W, False)
    stream.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    evs = run_steps(K, True)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    elapsed = evs[0][1][0].elapsed_time(evs[-1][1][4]) / 1e3
    per_arm = {k: [] for k in ARMS}
    for order, e in evs:
        for j, kind in enumerate(order):
            per_arm[kind].append(e[1 + j].elapsed_time(e[2 + j]) * 1e3 / n[kind])
    peak, peak_kind = measured_peak_hbm()
    scrub = L2Scrub(dev)
    res = {}
    for kind, wl in arms.items():
        # median period on this rank; across ranks the slowest replica's period with every
        # replica's bytes (replicas only: no data-path collective)
        us_max, bytes_all = aggregate(float(np.median(per_arm[kind])), float(wl.gemv_bytes))
        us = float(np.median(per_arm[kind]))
        iso = time_isolated(wl.gemv, max(8, 2 * wl.copies), stream)
        iso_scrub = time_isolated_scrubbed(wl.gemv, scrub, 12, stream)
        gbs = bytes_all / us_max / 1e3
        res[kind] = {"arm": ARM_NAMES[kind], "us": round(us, 3), "gb_s": round(gbs, 1),
                     "frac_of_measured_peak": round(gbs / peak, 4),
                     "pct_of_nominal_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
                     "spread_us": [round(min(per_arm[kind]), 3), round(max(per_arm[kind]), 3)],
                     "bytes_per_launch": wl.gemv_bytes, "weight_copies": wl.copies,
                     "launches_per_step": n[kind],
                     "isolated_launch_us": round(iso, 3),
                     "isolated_gb_s": round(wl.gemv_bytes / iso / 1e3, 1),
                     "isolated_after_l2_scrub_us": round(iso_scrub, 3),
                     "rotation_vs_scrub": round(iso / iso_scrub, 4),
                     "traffic": profiled_traffic(f"{kind if kind != 'blk' else 'blk128'}_{out_f}x{in_f}_m1")}
    low = min(ARMS, key=lambda k: res[k]["gb_s"])
    dom = max(ARMS, key=lambda k: res[k]["us"])
    value = res[low]["gb_s"]
    step_bytes = sum(wl.gemv_bytes * n[k] for k, wl in arms.items()) + producer_bytes(1, in_f)
    t_max, tot_units = aggregate(elapsed, float(K * step_bytes))

    e2e = time_e2e_arms(arms, lead, stream, steps=min(K, args.e2e_steps), graphs=True)
    eager = time_e2e_arms(arms, lead, stream, steps=min(K, args.e2e_steps), graphs=False)
    c2 = c2_step(args, dev, stream)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": t_max / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8+int8",
        "data": "synthetic",
        "config": {
            "workload": f"c3: E4M3, block-128 and Q8_0 GEMV out_f={out_f} in_f={in_f} m=1 on one "
                        f"q8_1 activation (RMSNorm->q8_1 of a {in_f}-wide row), arms interleaved "
                        f"in a rotating order, each on its own rotated weight copies",
            "value": "the lowest of the three arms' GB/s (each arm: algorithmic bytes per launch / "
                     "median back-to-back launch period over the K steps)",
            "timing": "per step: producer, then per arm a CUDA graph of back-to-back launches "
                      "(programmatic dependent launch) bracketed by CUDA events; K steps queued "
                      "behind a GPU sleep; ms_per_step = the whole region / K",
            "l2": "inputs larger than L2: each arm rotates through copies totalling more than "
                  "twice the 129 MB L2, so every launch reads its weights from DRAM",
            "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
            "step_bytes": step_bytes,
            "target": ">= 80% of the measured HBM peak per arm (back-to-back period); "
                      "t_q8_0 / t_e4m3 within 0.02 of the 34/32 byte ratio",
        },
        "arms": res,
        "step_gbs": round(tot_units / t_max / 1e9, 2),
        "q8_0_to_e4m3_time_ratio": round(res["q8_0"]["us"] / res["e4m3"]["us"], 4),
        "q8_0_to_blk128_time_ratio": round(res["q8_0"]["us"] / res["blk"]["us"], 4),
        "blk128_to_e4m3_time_ratio": round(res["blk"]["us"] / res["e4m3"]["us"], 4),
        "byte_ratio": round(arms["q8_0"].gemv_bytes / arms["e4m3"].gemv_bytes, 4),
        "isolated_q8_0_to_e4m3_time_ratio": round(res["q8_0"]["isolated_launch_us"] /
                                                  res["e4m3"]["isolated_launch_us"], 4),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "pct_of_nominal_8tbs": round(100.0 * value / NOMINAL_HBM_GBS, 2),
        "roofline": {
            "bound": "hbm",
            "achieved": res[dom]["gb_s"],
            "peak": peak,
            "unit": "GB/s",
            "frac": round(res[dom]["gb_s"] / peak, 4),
            "traffic": res[dom]["traffic"],
            "kernel": f"gemv_stream_kernel<{dom}, m=1> (the step's slowest arm)",
            "bytes_per_launch": arms[dom].gemv_bytes,
            "launch_us": res[dom]["us"],
            "launch_timing": "median back-to-back launch period (CUDA events around a graph of "
                             "launches on the launch stream)",
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                           else "fallback 6.8 TB/s",
            "isolated_launch_us": res[dom]["isolated_launch_us"],
        },
        "e2e": e2e | {"eager": eager},
        "c2_decode_step": c2,
        "gpu_launches": K * (1 + sum(n.values())),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_arms(arms, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_e2e_arms(arms, lead, stream, steps, graphs):
    """The public API with host buffers: per step the host->device copy of the activation row
    (pinned), the producer, one launch of each arm, the device->host copy of the three outputs
    and a host wait.  graphs=True replays one CUDA graph per rotated copy holding exactly those
    calls; graphs=False issues them from Python."""
    import torch
    x_pin = torch.from_numpy(lead.x_host.copy()).pin_memory()
    y_pin = {k: torch.empty(wl.y.shape, dtype=torch.float32).pin_memory() for k, wl in arms.items()}
    h2d = x_pin.numel() * 4
    d2h = sum(v.numel() * 4 for v in y_pin.values())
    copies = min(wl.copies for wl in arms.values())

    def one(i):
        lead.x.copy_(x_pin, non_blocking=True)
        lead.producer()
        for k, wl in arms.items():
            wl.gemv(i)
            y_pin[k].copy_(wl.y, non_blocking=True)

    run = one
    if graphs:
        gs = []
        with torch.cuda.stream(stream):
            for c in range(copies):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                    one(c)
                gs.append(g)
        run = lambda i: gs[i % len(gs)].replay()  # noqa: E731
    step_bytes = sum(wl.gemv_bytes for wl in arms.values()) + producer_bytes(1, lead.in_f)
    with torch.cuda.stream(stream):
        for i in range(8):
            run(i)
            stream.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            run(i)
            stream.synchronize()
        wall = time.perf_counter() - t0
    t_max, units = aggregate(wall, float(steps * step_bytes))
    return {"value": round(units / t_max / 1e9, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "us_per_step": round(t_max / steps * 1e6, 2),
            "mode": ("per step: one replay of a CUDA graph holding the public-API calls "
                     if graphs else "per step: the public-API calls issued from Python ")
                    + "(H2D of x from pinned memory, producer, the three GEMVs, D2H of the "
                      "three y), then a host wait; host wall clock"}


def c2_step(args, dev, stream, copies=16, reps=64):
    """The Q8_0 4096 x 4096 decode step (RMSNorm->q8_1 of a 4096-wide row, then the GEMV), 16
    rotated weight copies: `reps` steps as one CUDA graph replay (queued behind a GPU sleep),
    plus the GEMV's back-to-back period and its isolated launch."""
    import torch
    wl = DecodeStep("q8_0", 4096, 4096, 1, copies, dev, fused=False)
    with torch.cuda.stream(stream):
        for i in range(copies):
            wl.step(i)
        g = capture(wl.step, reps, stream)
        g.replay()
    stream.synchronize()
    times = []
    for _ in range(5):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(1_000_000)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
        stream.synchronize()
        times.append(a.elapsed_time(b) / 1e3 / reps)
    step_s = float(np.median(times))
    b2b = time_gemv_back_to_back(wl, stream, n=16 * copies)
    iso = time_isolated(wl.gemv, 2 * copies, stream)
    peak, _ = measured_peak_hbm()
    return {"workload": "q8_0_4096x4096_m1: RMSNorm->q8_1 (1x4096) then Q8_0 GEMV 4096x4096, "
                        "16 rotated copies",
            "step_us": round(step_s * 1e6, 3),
            "step_gbs": round(wl.step_bytes / step_s / 1e9, 2),
            "gemv_back_to_back_us": round(b2b * 1e6, 3),
            "gemv_gbs": round(wl.gemv_bytes / b2b / 1e9, 2),
            "gemv_frac_of_measured_peak": round(wl.gemv_bytes / b2b / 1e9 / peak, 4),
            "gemv_isolated_launch_us": round(iso, 3)}


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
        if t >= 2:
            # The page geometry (d_rope 0, kv_rank 512) at t >= 2 runs the tensor-core kernel:
            # three TF32 MMA products per f32 product, so its peak is the TF32 rate / 3 in
            # f32-equivalent FLOP.
            bf16, kind = measured_peak_bf16()
            peak = round(bf16 * TF32_PER_BF16 / 3.0, 1)
            roof = {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4),
                    "traffic": profiled_traffic(args.workload, "mla_traffic.json"),
                    "peak_kind": f"{kind} bf16 burst x 1.1/2.25 (TF32) / 3 (3xTF32 products per f32 product)",
                    "f32_alu_peak": F32_FMA_TFLOPS,
                    "f32_alu_frac": round(achieved / F32_FMA_TFLOPS, 4)}
        else:
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


def time_e2e_host_call(wl, stream, steps):
    """Per step one memq_decode_step_host call (pinned x in, fused step, pinned y out, the
    call's own wait), rotating the weight copies; host wall clock."""
    import torch
    x_pin = torch.from_numpy(wl.x_host.copy()).pin_memory()
    y_pin = torch.empty(wl.y.shape, dtype=torch.float32).pin_memory()
    with torch.cuda.stream(stream):
        for i in range(8):
            wl.host_step(i, x_pin, y_pin)
        t0 = time.perf_counter()
        for i in range(steps):
            wl.host_step(i, x_pin, y_pin)
        wall = time.perf_counter() - t0
    return {"elapsed": wall, "steps": steps, "h2d": x_pin.numel() * 4, "d2h": y_pin.numel() * 4}


def time_e2e_c_abi(wl, stream, steps):
    """As time_e2e_host_call, calling the C entry point memq_decode_step_host directly through
    ctypes with its arguments prepared once per weight copy: the cost of the C-ABI call itself,
    as a native caller pays it (no Python argument checks)."""
    import ctypes
    import torch
    x_pin = torch.from_numpy(wl.x_host.copy()).pin_memory()
    y_pin = torch.empty(wl.y.shape, dtype=torch.float32).pin_memory()
    memq = wl.memq
    container = {"q8_0": memq.Container.Q8_0, "blk": memq.Container.E4M3_BLK128,
                 "e4m3": memq.Container.E4M3}[wl.kind]
    fn = memq.lib().memq_decode_step_host
    args = [(int(container), x_pin.data_ptr(), wl.x.data_ptr(), wl.wn.data_ptr(),
             ctypes.c_float(1e-6), wl.w[c].data_ptr(),
             None if wl.aux is None else wl.aux[c].data_ptr(), wl.qs.data_ptr(), wl.d.data_ptr(),
             None, wl.y.data_ptr(), y_pin.data_ptr(), wl.out_f, wl.in_f, wl.m, stream.cuda_stream)
            for c in range(wl.copies)]
    bad = 0
    for i in range(8):
        bad |= fn(*args[i % wl.copies])
    t0 = time.perf_counter()
    for i in range(steps):
        bad |= fn(*args[i % wl.copies])
    wall = time.perf_counter() - t0
    if bad:
        raise RuntimeError("memq_decode_step_host failed in the timed loop")
    return {"elapsed": wall, "steps": steps, "h2d": x_pin.numel() * 4, "d2h": y_pin.numel() * 4}


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


def run_reference_c3(args, world):
    """The oracle as the timed arm of the default workload: every step is the producer on the
    5120-wide row plus each arm's GEMV on a bounded sample of its 17408 rows, sized from a
    calibration so that warm-up + K steps take about a minute; GB/s scaled from the sample."""
    import oracle
    oracle.build()
    out_f, in_f = C3_OUT_F, C3_IN_F
    data = {k: _oracle_inputs(k, out_f, in_f, 1) for k in ARMS}
    x, wn = data["e4m3"][0], data["e4m3"][1]
    _, d, qs, _ = oracle.rmsnorm_q8_1(x, wn, 1e-6)
    t0 = time.perf_counter()
    for k in ARMS:
        _oracle_gemv(oracle, k, data[k][2], data[k][3], qs, d, in_f, np.arange(64))
    per_row = (time.perf_counter() - t0) / 64  # one row of each arm
    budget = 60.0 / max(1, args.steps + args.warmup)
    nrows = int(max(1, min(out_f, budget / max(per_row, 1e-9))))
    rng = np.random.default_rng(7)
    samples = [np.sort(rng.choice(out_f, size=nrows, replace=False)) for _ in range(8)]

    def step(i):
        _, dd, qq, _ = oracle.rmsnorm_q8_1(x, wn, 1e-6)
        for k in ARMS:
            _oracle_gemv(oracle, k, data[k][2], data[k][3], qq, dd, in_f, samples[i % 8])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    sample_bytes = producer_bytes(1, in_f) + sum(
        gemv_bytes(k, nrows, in_f, 1) - (4 if k == "e4m3" else 0) for k in ARMS)
    v = args.steps * sample_bytes / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"c3: f64 C oracle of the same step (producer + E4M3, block-128 and "
                               f"Q8_0 GEMV out_f={out_f} in_f={in_f} m=1)",
                   "sample_rows_per_step": nrows},
        "cpu_baseline": {"value": round(v, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: producer 1x{in_f} + {nrows} of {out_f} rows of "
                                   f"each arm's GEMV, f64 C oracle, single thread"},
        "e2e": {"value": round(v, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    """The oracle as the timed arm: every step is the producer plus a bounded row sample of the
    GEMV, sized from a calibration step so that warm-up + K steps take about a minute."""
    if rank != 0:
        return
    if args.workload == "c3":
        return run_reference_c3(args, world)
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
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 50 for c3, whose step is ~50 launches; 100000 "
                         "for the single-launch workloads)")
    ap.add_argument("--warmup", type=int, default=None)
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
    ap.add_argument("--sweep", choices=["c4", "c5"], default=None,
                    help="time every cell of the C4 GEMV grid (3 containers x 4 shapes x m = 1, "
                         "2, 4, 8) or the C5 producer grid and write one JSONL receipt per cell")
    ap.add_argument("--receipts", default=None,
                    help="--sweep output file (default <sweep>_receipts.jsonl)")
    args = ap.parse_args(argv)
    if args.steps is None:
        args.steps = 50 if args.workload == "c3" else 100000
    if args.warmup is None:
        args.warmup = 5 if args.workload == "c3" else 1000
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
