"""Benchmark of the FP8 / MXFP8 transfer codec on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * a 25 MiB DDP gradient bucket held by k = 8 ranks (8 x 13,107,200 bf16,
    ~N(0, 1e-4^2)): blockwise quantize of all 8 shards to e4m3 and to e5m2
    (128-element blocks, fp32 scale = amax / Fmax), then the fused 8-way
    dequant-reduce of each format to bf16 and fp32;
  * the ring of 8 simulated on one GPU: 7 hops, each dequantizing the
    incoming e4m3 chunk, adding the next rank's bf16 partial and
    requantizing (the last hop also writes bf16);
  * BF16 -> MXFP8 prequantization of one Qwen3-30B-A3B-shaped decoder layer
    (128 experts x gate/up [768, 2048] and down [2048, 768], q [4096, 2048],
    k/v [512, 2048], o [2048, 4096]; 622,854,144 weights).
The metric is algorithmic HBM bytes moved per second (bytes each kernel must
read and write, see KERNEL_BYTES), for the device-resident step (`value`),
and end to end with the inputs copied in from pinned host memory and the
outputs copied back every step (`e2e`).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torchrun, one rank per GPU, each rank on its own data
(weak scaling; the ranks exchange nothing but the timing).  `--impl
reference` times the CPU oracle, single-threaded, on a bounded sample of the
same workload, and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import math
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 quant / fused dequant-reduce HBM GB/s and % of GB300 peak, 1 GPU"
WORKLOAD = ("ddp_bucket_25MiB_k8 (e4m3+e5m2 quantize, fused k=8 dequant-reduce -> bf16+fp32, 7-hop e4m3 ring) "
            "+ qwen3_30b_a3b_layer_mxfp8 (622,854,144 weights)")
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


# --------------------------------------------------------------- bytes ----
def nscales(n):
    return (n + 127) // 128


def bytes_quantize(n):
    return 2 * n + n + 4 * nscales(n)


def bytes_reduce(n, k, out_bf16=True, out_f32=True):
    return k * (n + 4 * nscales(n)) + n * (2 * out_bf16 + 4 * out_f32)


def bytes_hop(n, out_bf16):
    return (n + 4 * nscales(n)) + 2 * n + (n + 4 * nscales(n)) + 2 * n * out_bf16


def bytes_mxfp8(b, m, k, scale_bytes):
    return 3 * b * m * k + scale_bytes


# -------------------------------------------------------------- clocks ----
class ClockSampler:
    """SM clock and clock-event reasons of one GPU, sampled from NVML in a
    background thread (read-only queries; nothing is changed)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None, period_s: float = 0.002):
        self.samples = []
        self.ok = False
        self.period = period_s
        self.max_mhz = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if uuid and self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) == 0:
                pass
            elif self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.reason_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except OSError:
            self.ok = False

    def _run(self):
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            a = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
            b = self.reason_fn(self.h, ctypes.byref(rs))
            if a == 0 and b == 0:
                self.samples.append((t, int(mhz.value), int(rs.value)))
            time.sleep(self.period)

    def start(self):
        if not self.ok:
            return
        self._stop = threading.Event()
        self._th = threading.Thread(target=self._run, daemon=True)
        self._th.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._th.join()

    def summary(self, t0, t1):
        if not self.ok or not self.samples:
            return None
        inside = [s for s in self.samples if t0 <= s[0] <= t1] or \
            sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
        reasons = set()
        for _, _, r in inside:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(inside), "source": "nvml"}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for key in ("hbm_gbs", "hbm_GBps", "hbm_gb_s"):
                if key in d:
                    return float(d[key]), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(name):
    src = {"mxfp8_quantize_kernel": "mxfp8.cu", "quantize_blockwise_kernel": "quantize.cu",
           "quantize_group_kernel": "quantize.cu", "dequant_reduce_kernel": "reduce.cu",
           "ring_hop_kernel": "ring_hop.cu", "ring_hop_group_kernel": "ring_hop.cu",
           "mxfp8_dequantize_kernel": "mxfp8_receive.cu", "gather_decode_kernel": "reduce.cu"}[name]
    h = hashlib.sha256()
    for f in (src, "fp8q_device.cuh"):
        with open(os.path.join(ROOT, "weight_transfer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(name):
    """DRAM bytes per launch from a committed ncu summary (a line
    `traffic <kernel>@<source hash> = <bytes> ...` in profiles/*.md), only
    if it was taken on the current source of that kernel (else None)."""
    import glob
    want = f"traffic {name}@{kernel_source_hash(name)}"
    for p in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(p) as f:
            for line in f:
                if line.startswith(want):
                    try:
                        return float(line.split("=")[1].split()[0])
                    except (IndexError, ValueError):
                        return None
    return None


# ------------------------------------------------------- host topology ----
def _cpus(text):
    """'0-3,8,10-11' -> set of CPU numbers."""
    out = set()
    for part in (text or "").split(","):
        part = part.strip()
        if not part:
            continue
        a, _, b = part.partition("-")
        out.update(range(int(a), int(b or a) + 1))
    return out


def _cpu_text(cpus):
    cpus = sorted(cpus)
    runs, i = [], 0
    while i < len(cpus):
        j = i
        while j + 1 < len(cpus) and cpus[j + 1] == cpus[j] + 1:
            j += 1
        runs.append(str(cpus[i]) if i == j else f"{cpus[i]}-{cpus[j]}")
        i = j + 1
    return ",".join(runs)


def bind_to_gpu_numa(torch, dev):
    """Restricts this process to the CPUs local to the GPU (sysfs
    local_cpulist of its PCI function) when they are among the CPUs it may
    use, before any pinned host buffer is allocated, so that the buffers are
    placed on the GPU's side of the host.  Returns what it found and did."""
    p = torch.cuda.get_device_properties(dev)
    bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    info = {"gpu_pci": bdf}

    def read(name):
        try:
            with open(os.path.join("/sys/bus/pci/devices", bdf, name)) as f:
                return f.read().strip()
        except OSError:
            return None

    info["gpu_numa_node"] = read("numa_node")
    local = _cpus(read("local_cpulist"))
    allowed = os.sched_getaffinity(0)
    info["allowed_cpus"] = _cpu_text(allowed)
    info["gpu_local_cpus"] = _cpu_text(local) if local else None
    both = allowed & local
    if both and both != allowed:
        os.sched_setaffinity(0, both)
        info["bound_to"] = _cpu_text(both)
    else:
        info["bound_to"] = None
    return info


# ------------------------------------------------------------- L2 flush ----
class L2Flush:
    """Evicts L2 between timed steps: writes a buffer larger than L2, then
    reads a second one, so that the written lines are back in HBM (and the L2
    holds clean, unrelated lines) before the next step's events start."""

    def __init__(self, torch, dev, nbytes=L2_FLUSH_BYTES):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 4, dtype=torch.float32, device=dev)
        self.i = 0

    def __call__(self):
        self.i += 1
        self.w.fill_(self.i & 0xFF)
        self.r.sum()


# ------------------------------------------------------------ workload ----
def carve(torch, specs, device=None, pin=False):
    """One uint8 allocation holding a tensor of each (shape, dtype) in
    `specs`, at 256-byte aligned offsets (on `device`, or in pinned host
    memory with pin=True).  Returns (buffer, [tensors])."""
    offs, total = [], 0
    for shape, dt in specs:
        nbytes = math.prod(shape) * torch.empty(0, dtype=dt).element_size()
        offs.append((total, nbytes))
        total += (nbytes + 255) // 256 * 256
    if device is None:
        buf = torch.empty(total, dtype=torch.uint8, pin_memory=pin)
    else:
        buf = torch.empty(total, dtype=torch.uint8, device=device)
    views = [buf[o:o + nb].view(dt).view(shape) for (o, nb), (shape, dt) in zip(offs, specs)]
    return buf, views


class DeviceSet:
    """One set of device buffers for a step (inputs and outputs) and the
    step's launch list bound to them, arguments marshalled once so that a
    launch costs one ctypes call."""

    def __init__(self, wl, stream):
        torch, dev, L, n, k = wl.torch, wl.dev, wl.L, wl.n, wl.k
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        nb = nscales(n)
        self.stream = stream
        # the step's inputs in one allocation and the results a caller reads
        # back in another, each a run of tensors (wl.in_specs, wl.out_specs),
        # so that each direction of the end-to-end run is one copy
        self.in_buf, ins = carve(torch, wl.in_specs, dev)
        self.bucket, self.layer = ins[0], ins[1:]
        self.out_buf, outs = carve(torch, wl.out_specs, dev)
        self.q = {0: (outs[0], outs[1]), 1: (outs[2], outs[3])}
        self.red = {0: (outs[4], outs[5]), 1: (outs[6], outs[7])}
        # hops 1..6 are internal; the last hop's codes and scales are results
        self.hops = [(torch.empty(n, dtype=u8, device=dev), torch.empty(nb, dtype=f32, device=dev))
                     for _ in range(k - 2)] + [(outs[8], outs[9])]
        self.ring_bf16 = outs[10]
        self.mx = [(outs[11 + 2 * i], outs[12 + 2 * i], wl.w.mxfp8_swizzled_scale_bytes(b, m, kk))
                   for i, (name, b, m, kk) in enumerate(wl.tensors)]
        self.outputs = outs

        vp = ctypes.c_void_p
        sp_ = vp(stream.cuda_stream)
        launches = []

        def add(kind, nbytes, elems, fn, *args):
            launches.append((kind, nbytes, elems, fn, args))

        # FP8Q_INPUTS_READY holds for every launch of the step but the hops:
        # the bucket and the layer are written only by copies, and each reduce
        # reads codes that the quantize two launches earlier wrote (a kernel
        # of the library lets its successor start only after its own wait)
        ready = ctypes.c_uint(wl.w.FP8Q_INPUTS_READY)
        for f in (0, 1):
            c, sc = self.q[f]
            add("quantize_blockwise_kernel", bytes_quantize(k * n), k * n, L.fp8q_quantize_blockwise_ex,
                vp(self.bucket.data_ptr()), ctypes.c_size_t(k * n), ctypes.c_int(f), vp(c.data_ptr()),
                vp(sc.data_ptr()), ready, sp_)
        self._keep = []
        for f in (0, 1):
            c, sc = self.q[f]
            cp = (vp * k)(*[c[r].data_ptr() for r in range(k)])
            sp = (vp * k)(*[sc[r].data_ptr() for r in range(k)])
            self._keep += [cp, sp]
            ob, of = self.red[f]
            add("dequant_reduce_kernel", bytes_reduce(n, k), n, L.fp8q_dequant_reduce_ex, cp, sp, ctypes.c_int(k),
                ctypes.c_size_t(n), ctypes.c_int(f), vp(ob.data_ptr()), vp(of.data_ptr()), ready, sp_)
        # hop 0 = e4m3 quantize of rank 0's shard; hop h adds shard h, which
        # only the step's input copy writes, so each hop may start reading it
        # while the previous hop drains
        prev = (self.q[0][0][0], self.q[0][1][0])
        for h in range(1, k):
            oc, osc = self.hops[h - 1]
            last = h == k - 1
            hp = (wl.w.fp8q_hop_t * 1)(wl.w.fp8q_hop_t(prev[0].data_ptr(), prev[1].data_ptr(),
                                                        self.bucket[h].data_ptr(), n, oc.data_ptr(),
                                                        osc.data_ptr(), self.ring_bf16.data_ptr() if last else None))
            self._keep.append(hp)
            add("ring_hop_kernel", bytes_hop(n, last), n, L.fp8q_ring_hop_group_ex, hp, ctypes.c_int(1),
                ctypes.c_int(0), ctypes.c_uint(wl.w.FP8Q_HOP_LOCAL_READY), sp_)
            prev = (oc, osc)
        # the whole layer (expert batches and attention matrices) in one launch
        self._group = (wl.w.mxfp8_tensor_t * len(wl.tensors))()
        mx_bytes = mx_elems = 0
        for i, ((name, b, m, kk), x, (c, sc, sb)) in enumerate(zip(wl.tensors, self.layer, self.mx)):
            self._group[i] = wl.w.mxfp8_tensor_t(x.data_ptr(), b, m, kk, c.data_ptr(), sc.data_ptr())
            mx_bytes += bytes_mxfp8(b, m, kk, sb)
            mx_elems += b * m * kk
        add("mxfp8_quantize_kernel", mx_bytes, mx_elems, L.mxfp8_quantize_swizzled_group_ex, self._group,
            ctypes.c_int(len(wl.tensors)), ready, sp_)
        self.launches = launches

    def segments(self):
        """Runs of consecutive launches of one kernel: (kind, first, last)."""
        runs = []
        for i, (kind, _, _, _, _) in enumerate(self.launches):
            if runs and runs[-1][0] == kind:
                runs[-1][2] = i
            else:
                runs.append([kind, i, i])
        return [tuple(r) for r in runs]

    def run(self, events=None, only=None, segments=False):
        """Launch one step on this set's stream; with `events`, bracket each
        launch (or, with `only`, each launch of that kernel; with `segments`,
        each run of launches of one kernel) with a pair of timing events.  An
        event between two launches also ends the overlap of the second with
        the first, so the timed steps bracket only the kernel whose roofline
        is reported."""
        starts = ends = None
        if segments:
            runs = self.segments()
            starts, ends = {r[1] for r in runs}, {r[2] for r in runs}
        for i, (kind, _, _, fn, args) in enumerate(self.launches):
            if events is None:
                before = after = False
            elif segments:
                before, after = i in starts, i in ends
            else:
                before = after = only is None or kind == only
            if before:
                events[2 * i].record(self.stream)
            st = fn(*args)
            if st != 0:
                raise RuntimeError(f"launch {i} failed with status {st}")
            if after:
                events[2 * i + 1].record(self.stream)


class Workload:
    """The step's inputs in pinned host memory and the device sets that run
    it (one for the device-resident timing, two for the copy pipeline)."""

    def __init__(self, dev, rank, torch):
        import gen
        import weight_transfer_gb300 as w
        self.torch, self.w, self.dev = torch, w, dev
        self.L = w.lib()
        n, k = gen.DDP_N, gen.DDP_K
        self.n, self.k = n, k
        self.tensors = gen.QWEN3_TENSORS
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        nb = nscales(n)
        # inputs: the bucket of all 8 ranks (shard r = row r), then the layer's tensors
        self.in_specs = [((k, n), bf)] + [((b, m, kk), bf) for (name, b, m, kk) in self.tensors]
        self.out_specs = [((k, n), u8), ((k, nb), f32), ((k, n), u8), ((k, nb), f32), ((n,), bf), ((n,), f32),
                          ((n,), bf), ((n,), f32), ((n,), u8), ((nb,), f32), ((n,), bf)]
        for (name, b, m, kk) in self.tensors:
            self.out_specs += [((b, m, kk), u8), ((w.mxfp8_swizzled_scale_bytes(b, m, kk),), u8)]
        # the inputs in pinned host memory, laid out as a device set's inputs
        self.h_in, hv = carve(torch, self.in_specs, pin=True)
        for r, seed in enumerate(rank_data_seeds(rank, k)):
            hv[0][r].copy_(gen.ddp_shard(seed))
        for t in range(len(self.tensors)):
            hv[1 + t].copy_(gen.qwen3_tensor(rank, t))
        self.stream = torch.cuda.current_stream(dev)
        self.sets = [DeviceSet(self, self.stream)]
        self.h2d(self.sets[0], self.stream)
        torch.cuda.synchronize(dev)
        self.launches = self.sets[0].launches
        self.step_bytes = sum(l[1] for l in self.launches)
        self.step_elems = sum(l[2] for l in self.launches)
        self.h_out = None

    # the main timed loop and the profile cases use set 0
    @property
    def q(self):
        return self.sets[0].q

    @property
    def red(self):
        return self.sets[0].red

    def run(self, events=None, only=None, segments=False):
        self.sets[0].run(events, only, segments)

    def _copy_all(self, stream, pairs):
        """Copies (dst, src) tensor pairs on `stream`, one cudaMemcpyAsync per
        pair.  Each direction of a step is one pair (the inputs and the
        results each lie in one buffer).  Fanning a direction out over 4 side
        streams in 32 MiB pieces gave 370 GB/s end to end, one copy per tensor
        386 GB/s, one copy per direction 388 GB/s; the host link carries
        about 210 GB/s host to device and 190 GB/s back, by copy engine or SM
        alike."""
        torch = self.torch
        nbytes = 0
        with torch.cuda.stream(stream):
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
                nbytes += dst.numel() * dst.element_size()
        return nbytes

    def h2d(self, ds, stream):
        """Copies the step's inputs from pinned host memory into set `ds`."""
        return self._copy_all(stream, [(ds.in_buf, self.h_in)])

    def d2h(self, ds, stream):
        """Reads every result of set `ds` back into pinned host memory."""
        if self.h_out is None:
            self.h_out_buf, self.h_out = carve(self.torch, self.out_specs, pin=True)
        return self._copy_all(stream, [(self.h_out_buf, ds.out_buf)])

    def e2e(self, steps, warmup=2):
        """Steady-state end-to-end throughput of the public API with host
        buffers: every step copies its inputs in (H2D stream), runs the step
        (compute stream) and reads its results back (D2H stream); two device
        sets let step i's readback overlap step i+1's input copy and kernels.
        Returns (ms per step, H2D bytes per step, D2H bytes per step)."""
        torch = self.torch
        s_in = torch.cuda.Stream(self.dev)
        s_run = torch.cuda.Stream(self.dev)
        s_out = torch.cuda.Stream(self.dev)
        self.sets = [DeviceSet(self, s_run), DeviceSet(self, s_run)]
        Ev = torch.cuda.Event
        # the copy engines alone, for reference: one step's inputs in, outputs
        # out (best of three, after a warm-up copy)
        self.copy_gbps = {}
        for name, fn, st in (("h2d", self.h2d, s_in), ("d2h", self.d2h, s_out)):
            fn(self.sets[0], st)
            torch.cuda.synchronize(self.dev)
            best = 0.0
            for _ in range(3):
                a, b = Ev(enable_timing=True), Ev(enable_timing=True)
                a.record(st)
                nb = fn(self.sets[0], st)
                b.record(st)
                torch.cuda.synchronize(self.dev)
                best = max(best, nb / (a.elapsed_time(b) * 1e-3) / 1e9)
            self.copy_gbps[name] = round(best, 1)
        # both directions at once (step i+1's inputs in while step i's results
        # go out): the pipeline's ceiling when the host side is shared
        best = 0.0
        for _ in range(3):
            a, b, c = Ev(enable_timing=True), Ev(enable_timing=True), Ev(enable_timing=True)
            torch.cuda.synchronize(self.dev)
            a.record(s_in)
            s_out.wait_event(a)
            nb_in = self.h2d(self.sets[0], s_in)
            nb_out = self.d2h(self.sets[1], s_out)
            b.record(s_in)
            c.record(s_out)
            torch.cuda.synchronize(self.dev)
            best = max(best, (nb_in + nb_out) / (max(a.elapsed_time(b), a.elapsed_time(c)) * 1e-3) / 1e9)
        self.copy_gbps["both"] = round(best, 1)
        bi = bo = 0
        total = warmup + steps
        done_run = [None, None]      # compute of the set's previous step finished (inputs free)
        done_out = [None, None]      # readback of the set's previous step finished (outputs free)
        start = Ev(enable_timing=True)
        end = Ev(enable_timing=True)
        for i in range(total):
            if i == warmup:
                torch.cuda.synchronize(self.dev)
                start.record(s_in)
            ds = self.sets[i % 2]
            if done_run[i % 2] is not None:
                s_in.wait_event(done_run[i % 2])
            bi = self.h2d(ds, s_in)
            copied = Ev()
            copied.record(s_in)
            s_run.wait_event(copied)
            if done_out[i % 2] is not None:
                s_run.wait_event(done_out[i % 2])
            ds.run()
            ran = Ev()
            ran.record(s_run)
            done_run[i % 2] = ran
            s_out.wait_event(ran)
            bo = self.d2h(ds, s_out)
            out = Ev()
            out.record(s_out)
            done_out[i % 2] = out
        end.record(s_out)
        torch.cuda.synchronize(self.dev)
        # the sets were built for the pipeline streams; set 0 goes back to the main stream
        self.sets = [DeviceSet(self, self.stream)]
        self.h2d(self.sets[0], self.stream)
        self.sets[0].run()
        self.launches = self.sets[0].launches
        torch.cuda.synchronize(self.dev)
        # the pipelined run's last results, read back to the host, against a
        # device-resident run on the same inputs: byte for byte
        self.e2e_outputs_equal = all(
            torch.equal(h.contiguous().view(-1).view(torch.uint8), d.contiguous().view(-1).cpu().view(torch.uint8))
            for h, d in zip(self.h_out, self.sets[0].outputs))
        return start.elapsed_time(end) / steps, bi, bo


# --------------------------------------------------------- oracle runs ----
_ORACLE_INPUTS = {}


def _oracle_inputs():
    """Host copies of rank 0's step inputs for the oracle (generated once)."""
    if not _ORACLE_INPUTS:
        import numpy as np
        import torch
        import gen
        _ORACLE_INPUTS["shards"] = [gen.ddp_shard(r).view(torch.int16).numpy().view(np.uint16) for r in range(gen.DDP_K)]
        _ORACLE_INPUTS["mats"] = [(gen.qwen3_tensor(0, t).view(torch.int16).numpy().view(np.uint16), b, m, kk)
                                  for t, (_, b, m, kk) in enumerate(gen.QWEN3_TENSORS)]
    return _ORACLE_INPUTS


def _oracle_step(orc, shards, mats, keep=None):
    """One step of the oracle on the given slices of the bucket shards and
    the layer tensors: returns (algorithmic bytes, elements).  With `keep` (a
    dict), its results are stored there for the parity check of the GPU step."""
    k = len(shards)
    n = shards[0].size
    nbytes = elems = 0
    if n:
        q = {}
        red = {}
        hops = []
        for f in (0, 1):
            q[f] = [orc.quantize_blockwise(sh, f) for sh in shards]
            nbytes += bytes_quantize(k * n)
            elems += k * n
        for f in (0, 1):
            red[f] = orc.dequant_reduce([c for c, _ in q[f]], [s for _, s in q[f]], f)
            nbytes += bytes_reduce(n, k)
            elems += n
        c, s = q[0][0]
        for h in range(1, k):
            c, s, hb = orc.ring_hop(c, s, shards[h], 0)
            hops.append((c, s, hb))
            nbytes += bytes_hop(n, h == k - 1)
            elems += n
        if keep is not None:
            keep.update(n=n, q=q, red=red, hops=hops)
    for t, (x, b, m, kk) in enumerate(mats):
        if b * m == 0:
            continue
        mc, ms = orc.mxfp8_quantize_swizzled(x, b, m, kk)
        if keep is not None:
            keep.setdefault("mx", []).append((t, b, m, kk, mc, ms))
        nbytes += bytes_mxfp8(b, m, kk, orc.swizzled_scale_bytes(b, m, kk))
        elems += b * m * kk
    return nbytes, elems


def parity_against_oracle(ds, keep):
    """The GPU step's own outputs (device set `ds`, rank 0's data) against the
    oracle's results on the cpu_baseline sample, the same leading elements of
    every output: codes and scales of both quantizes, both reduce outputs, all
    7 hops (codes, scales, the last hop's bf16) and the MXFP8 codes and
    swizzled scales of the sampled experts / rows.  Bit for bit."""
    import numpy as np
    import torch

    def host(t, count):
        v = t.contiguous().view(-1)[:count]
        if v.dtype in (torch.bfloat16, torch.float16):
            v = v.view(torch.int16)
        return v.cpu().numpy().view(np.uint8)

    def raw(a):
        return np.ascontiguousarray(a).view(np.uint8).ravel()

    checked = mismatched = 0

    def cmp(gpu_bytes, want):
        nonlocal checked, mismatched
        want = raw(want)
        assert gpu_bytes.size == want.size, (gpu_bytes.size, want.size)
        checked += want.size
        mismatched += int(np.count_nonzero(gpu_bytes != want))
    elements = 0
    if "n" in keep:
        n = keep["n"]
        nb = nscales(n)
        for f in (0, 1):
            c, sc = ds.q[f]
            for r, (ec, es) in enumerate(keep["q"][f]):
                cmp(host(c[r], n), ec)
                cmp(host(sc[r], nb), es)
            eb, ef = keep["red"][f]
            cmp(host(ds.red[f][0], n), eb)
            cmp(host(ds.red[f][1], n), ef)
            elements += (len(keep["q"][f]) + 1) * n
        for h, (ec, es, eb) in enumerate(keep["hops"]):
            oc, osc = ds.hops[h]
            cmp(host(oc, n), ec)
            cmp(host(osc, nb), es)
            elements += n
        cmp(host(ds.ring_bf16, n), keep["hops"][-1][2])
    for t, b, m, kk, mc, ms in keep.get("mx", []):
        c, sc, _ = ds.mx[t]
        cmp(host(c, b * m * kk), mc)
        cmp(host(sc, ms.size), ms)
        elements += b * m * kk
    return {"elements": elements, "bytes_compared": checked, "mismatches": mismatched,
            "what": "the GPU step's outputs against the oracle's on the cpu_baseline sample, byte for byte"}


def oracle_sample(fraction, threads=1, keep=None):
    """The oracle on a contiguous fraction of the same workload (rank 0's
    data): returns (algorithmic bytes, elements, seconds, description).  With
    threads > 1 the sample is cut into that many disjoint, 128-aligned parts
    (bucket elements, experts, attention rows) run at once; the oracle's
    calls release the interpreter lock, so the threads run in parallel."""
    import concurrent.futures as cf
    import oracle as orc
    inp = _oracle_inputs()
    n_full = inp["shards"][0].size
    n = max(128, int(n_full * fraction) // 128 * 128)
    mats_all = []
    for x, b, m, kk in inp["mats"]:
        if b > 1:
            mats_all.append((x, max(1, int(round(b * fraction))), m, kk, True))
        else:
            mats_all.append((x, 1, max(128, int(m * fraction) // 128 * 128), kk, False))

    def part(i, t):
        lo, hi = (n // 128) * i // t * 128, (n // 128) * (i + 1) // t * 128
        shards = [sh[lo:hi].copy() for sh in inp["shards"]]
        mats = []
        for x, b, m, kk, batched in mats_all:
            if batched:
                b0, b1 = b * i // t, b * (i + 1) // t
                mats.append((x[b0:b1].copy(), b1 - b0, m, kk))
            else:
                r0, r1 = (m // 128) * i // t * 128, (m // 128) * (i + 1) // t * 128
                mats.append((x[0, r0:r1].copy(), 1, r1 - r0, kk))
        return shards, mats

    parts = [part(i, threads) for i in range(threads)]
    t0 = time.perf_counter()
    if threads == 1:
        res = [_oracle_step(orc, *parts[0], keep=keep)]
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            res = list(ex.map(lambda p_: _oracle_step(orc, *p_), parts))
    dt = time.perf_counter() - t0
    nbytes = sum(r[0] for r in res)
    elems = sum(r[1] for r in res)
    desc = (f"{fraction:.4g} of one step: the first {n} elements of each of the 8 bucket shards (both formats, "
            f"reduce, 7 hops) and the first {fraction:.4g} of the experts / rows of each layer tensor; "
            + ("single-threaded oracle" if threads == 1 else f"cut into {threads} disjoint parts on {threads} threads"))
    return nbytes, elems, dt, desc


def oracle_fraction_for(seconds):
    """The step fraction whose oracle run takes about `seconds`."""
    _, _, t_cal, _ = oracle_sample(1.0 / 256)
    t_full = max(1e-9, t_cal * 256)
    return max(1.0 / 4096, min(1.0, seconds / t_full))


def run_reference(args):
    """--impl reference: the oracle, as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    steps, warmup = args.steps, max(args.warmup, 3)
    # size each step so that the whole run stays within about two minutes
    frac = min(0.25, oracle_fraction_for(100.0 / (steps + warmup)))
    for _ in range(warmup):
        oracle_sample(frac)
    tot_b = tot_t = tot_e = 0.0
    desc = ""
    for _ in range(steps):
        b, e, t, desc = oracle_sample(frac)
        tot_b += b
        tot_t += t
        tot_e += e
    gbs = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warmup, "ms_per_step": round(1e3 * tot_t / steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_fraction_per_step": frac},
            "elements_per_s": round(tot_e / tot_t, 1),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- ranks ----
def combine_over_ranks(dist, device, ms_local, bytes_local, elems_local):
    """Whole-job figures: the slowest rank's step time, and the bytes and
    elements of all ranks (each rank processes its own data).  `dist` is
    torch.distributed with an initialised group, or None for one process."""
    if dist is None:
        return ms_local, bytes_local, elems_local
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([bytes_local, elems_local], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t[0].item()), float(u[0].item()), float(u[1].item())


def rank_data_seeds(rank, k=8):
    """Seeds of the bucket shards a rank works on: rank r takes 8r .. 8r+7,
    so no two ranks quantize the same bytes."""
    return [r + k * rank for r in range(k)]


# -------------------------------------------------------- profile cases ----
# kernel kind and index of its first launch in Workload.launches
PROFILE_CASES = {"quantize": ("quantize_blockwise_kernel", 0), "reduce": ("dequant_reduce_kernel", 2),
                 "ring_hop": ("ring_hop_kernel", 4), "mxfp8": ("mxfp8_quantize_kernel", 11)}


def run_profile_case(case, launches):
    """One kernel of the bench step, launched `launches` times on the bench's
    own inputs (the inputs of each step kernel, prepared once), then exit."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if case == "ring_hop_256MiB":
        # one e4m3 hop of the ring sweep's largest payload (2^27 elements,
        # 256 MiB of bf16; outside the step), without the bf16 output
        import gen
        import weight_transfer_gb300 as w
        n = (256 << 20) // 2
        x0, x1 = gen.ring_partial(0, n).to(dev), gen.ring_partial(1, n).to(dev)
        c0, s0 = w.fp8q_quantize_blockwise(x0, "e4m3")
        c1, s1 = torch.empty_like(c0), torch.empty_like(s0)
        for _ in range(max(1, launches)):
            w.fp8q_ring_hop(c0, s0, x1, "e4m3", out_codes=c1, out_scales=s1)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": case, "kernel": "ring_hop_kernel", "launches": launches,
                          "bytes_per_launch": bytes_hop(n, False)}))
        return
    wl = Workload(dev, 0, torch)
    wl.run()                                   # every kernel's inputs exist
    torch.cuda.synchronize()
    if case == "mxfp8_dequantize":
        # the receiver side on the step's expert gate batch (outside the step)
        name, b, mm, kk = wl.tensors[0]
        c, sc, sb = wl.sets[0].mx[0]
        out = torch.empty((b, mm, kk), dtype=torch.bfloat16, device=dev)
        for _ in range(max(1, launches)):
            wl.w.mxfp8_dequantize_swizzled(c, sc, out=out, stream=wl.stream)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": case, "kernel": "mxfp8_dequantize_kernel", "launches": launches,
                          "bytes_per_launch": 3 * b * mm * kk + sb}))
        return
    if case == "ring_allreduce_sim":
        # the simulated 8-rank ring AllReduce of the bucket (outside the
        # step); its last launch is the all-gather decode (gather_decode_kernel)
        P, n = wl.k, wl.n
        parts = [wl.sets[0].bucket[r] for r in range(P)]
        res = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        ws = torch.empty(int(wl.w.lib().fp8q_ring_allreduce_workspace_bytes(P, n)), dtype=torch.uint8, device=dev)
        for _ in range(max(1, launches)):
            wl.w.fp8q_ring_allreduce_sim(parts, "e4m3", results=res, workspace=ws, stream=wl.stream)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": case, "kernel": "gather_decode_kernel", "launches": launches,
                          "bytes_per_launch": n + 4 * nscales(n) + P * 2 * n}))
        return
    kind, first = PROFILE_CASES[case]
    _, nbytes, _, fn, fargs = wl.launches[first]
    assert wl.launches[first][0] == kind
    for _ in range(max(1, launches)):
        st = fn(*fargs)
        if st != 0:
            raise RuntimeError(f"{case}: status {st}")
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": case, "kernel": kind, "launches": launches, "bytes_per_launch": nbytes}))


def fused_vs_naive(wl, torch, reps=20):
    """Time the fused 8-way reduce against the naive order (dequantize each
    shard to fp32 in HBM, then sum) on the bench's e4m3 codes."""
    L, n, k = wl.L, wl.n, wl.k
    vp = ctypes.c_void_p
    c, sc = wl.q[0]
    cp = (vp * k)(*[c[r].data_ptr() for r in range(k)])
    sp = (vp * k)(*[sc[r].data_ptr() for r in range(k)])
    stride = int(L.fp8q_unfused_stride(n))
    ws = torch.empty(k * stride, dtype=torch.float32, device=wl.dev)
    ob, of = wl.red[0]
    s = vp(wl.stream.cuda_stream)
    flush = L2Flush(torch, wl.dev)

    def fused():
        return L.fp8q_dequant_reduce(cp, sp, k, n, 0, vp(ob.data_ptr()), vp(of.data_ptr()), s)

    def naive():
        return L.fp8q_dequant_reduce_unfused(cp, sp, k, n, 0, vp(ws.data_ptr()), vp(ob.data_ptr()),
                                             vp(of.data_ptr()), s)
    out = {}
    for name, fn in (("fused", fused), ("naive", naive)):
        for _ in range(3):
            fn()
        tot = 0.0
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(wl.stream)
            if fn() != 0:
                raise RuntimeError(f"{name} reduce failed")
            b.record(wl.stream)
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        out[name + "_us"] = round(1e3 * tot / reps, 2)
    out["fused_over_naive"] = round(out["naive_us"] / out["fused_us"], 2)
    out["naive_bytes"] = k * (n + 4 * nscales(n)) + 2 * k * 4 * n + n * 6
    out["fused_bytes"] = bytes_reduce(n, k)
    del ws
    return out


def ring_sweep(wl, torch, payloads=(64 << 20, 128 << 20, 256 << 20), reps=10):
    """The ring at large per-hop payloads, outside the step: the size range
    the >= 70%-of-peak bar is stated for.  Per payload: one hop (e4m3, with
    the bf16 output of a last hop) timed alone, and the 7-hop chain of a ring
    of 8 launched back to back as the step launches it (each hop's local
    partial copied early).  Partials 0 and 1 come from the counter-based
    generator; 2..7 from a seeded device-side draw of the same
    distribution, N(0, 1e-3^2)."""
    import gen
    L = wl.L
    w = wl.w
    vp = ctypes.c_void_p
    s = vp(wl.stream.cuda_stream)
    flush = L2Flush(torch, wl.dev)
    out = {}
    P = gen.RING_PARTIALS

    def ev():
        return torch.cuda.Event(enable_timing=True)
    for payload in payloads:
        n = payload // 2
        nb = nscales(n)
        x0 = gen.ring_partial(0, n).to(wl.dev)
        x1 = gen.ring_partial(1, n).to(wl.dev)
        c0 = torch.empty(n, dtype=torch.uint8, device=wl.dev)
        s0 = torch.empty(nb, dtype=torch.float32, device=wl.dev)
        c1 = torch.empty_like(c0)
        s1 = torch.empty_like(s0)
        ob = torch.empty(n, dtype=torch.bfloat16, device=wl.dev)
        if L.fp8q_quantize_blockwise(vp(x0.data_ptr()), n, 0, vp(c0.data_ptr()), vp(s0.data_ptr()), s) != 0:
            raise RuntimeError("ring sweep quantize failed")
        args = (vp(c0.data_ptr()), vp(s0.data_ptr()), vp(x1.data_ptr()), ctypes.c_size_t(n), ctypes.c_int(0),
                vp(c1.data_ptr()), vp(s1.data_ptr()), vp(ob.data_ptr()), s)
        for _ in range(3):
            L.fp8q_ring_hop(*args)
        tot = 0.0
        for _ in range(reps):
            flush()
            a, b = ev(), ev()
            a.record(wl.stream)
            if L.fp8q_ring_hop(*args) != 0:
                raise RuntimeError("ring sweep hop failed")
            b.record(wl.stream)
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        us = 1e3 * tot / reps
        nbytes = bytes_hop(n, True)
        row = {"us": round(us, 2), "bytes": nbytes, "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1)}
        # the 7-hop chain
        g = torch.Generator(device=wl.dev)
        g.manual_seed(200 + payload)
        parts = [x0, x1] + [torch.randn(n, device=wl.dev, generator=g).mul_(1e-3).to(torch.bfloat16)
                            for _ in range(P - 2)]
        outs = [(torch.empty(n, dtype=torch.uint8, device=wl.dev), torch.empty(nb, dtype=torch.float32, device=wl.dev))
                for _ in range(P - 1)]
        hops = []
        prev = (c0, s0)
        for h in range(1, P):
            oc, os_ = outs[h - 1]
            hops.append((w.fp8q_hop_t * 1)(w.fp8q_hop_t(prev[0].data_ptr(), prev[1].data_ptr(), parts[h].data_ptr(), n,
                                                         oc.data_ptr(), os_.data_ptr(),
                                                         ob.data_ptr() if h == P - 1 else None)))
            prev = (oc, os_)
        ready = ctypes.c_uint(w.FP8Q_HOP_LOCAL_READY)
        times = []
        for i in range(reps + 2):
            flush()
            a, b = ev(), ev()
            a.record(wl.stream)
            for hp in hops:
                if L.fp8q_ring_hop_group_ex(hp, 1, 0, ready, s) != 0:
                    raise RuntimeError("ring sweep chain failed")
            b.record(wl.stream)
            torch.cuda.synchronize()
            if i >= 2:
                times.append(a.elapsed_time(b))
        cms = sorted(times)[len(times) // 2]
        cbytes = (P - 2) * bytes_hop(n, False) + bytes_hop(n, True)
        row["chain_7_hops"] = {"us": round(1e3 * cms, 2), "bytes": cbytes, "GB/s": round(cbytes / (cms * 1e-3) / 1e9, 1)}
        out[f"{payload >> 20}MiB"] = row
        del x0, x1, c0, s0, c1, s1, ob, parts, outs, hops
    return out


def timed(torch, stream, fn, flush, reps=5):
    """Mean event time (ms) of fn() on `stream`, L2 flushed before each rep."""
    fn()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / reps


def extra_rows(wl, torch, peak):
    """The rows beyond the step, each timed on its own on the step's data:
    the simulated 8-rank FP8 ring AllReduce of the bucket, the MXFP8 receiver
    (dequantize the layer's expert gate batch), per-tensor scaling."""
    w, dev, st = wl.w, wl.dev, wl.stream
    flush = L2Flush(torch, dev)
    ds = wl.sets[0]
    P, n = wl.k, wl.n
    m = n // P
    parts = [ds.bucket[r] for r in range(P)]
    res = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    ws = torch.empty(int(w.lib().fp8q_ring_allreduce_workspace_bytes(P, n)), dtype=torch.uint8, device=dev)
    out = {}
    wire = [0]

    def ring(mean=False):
        wire[0] = w.fp8q_ring_allreduce_sim(parts, "e4m3", results=res, workspace=ws, stream=st, mean=mean)[1]
    ms = timed(torch, st, ring, flush)
    ms_mean = timed(torch, st, lambda: ring(True), flush)
    # the all-gather decode reads the one shared copy of the gathered codes
    # once and writes every rank's result
    kbytes = P * bytes_quantize(m) + (P - 1) * P * bytes_hop(m, False) + (n + 4 * nscales(n) + P * 2 * n)
    out["ring_allreduce_sim"] = {
        "ranks": P, "elements": n, "ms": round(ms, 4), "ms_mean": round(ms_mean, 4), "kernel_bytes": kbytes,
        "GB/s": round(kbytes / (ms * 1e-3) / 1e9, 1), "wire_bytes_per_rank": wire[0],
        "bf16_ring_bytes_per_rank": 2 * (P - 1) * m * 2,
        "wire_saving_vs_bf16": round(1 - wire[0] / (2 * (P - 1) * m * 2), 6)}
    del res, ws
    # the same collective at 256 MiB of bf16 per rank (device-drawn partials,
    # N(0, 1e-4^2)): per-rank chunks of 16.8M elements instead of 1.6M
    nl_ = 8 * (1 << 24)
    g = torch.Generator(device=dev)
    g.manual_seed(300)
    big = [torch.randn(nl_, device=dev, generator=g).mul_(1e-4).to(torch.bfloat16) for _ in range(P)]
    bres = [torch.empty(nl_, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    bws = torch.empty(int(w.lib().fp8q_ring_allreduce_workspace_bytes(P, nl_)), dtype=torch.uint8, device=dev)
    ms = timed(torch, st, lambda: w.fp8q_ring_allreduce_sim(big, "e4m3", results=bres, workspace=bws, stream=st),
               flush)
    ml = nl_ // P
    kb2 = P * bytes_quantize(ml) + (P - 1) * P * bytes_hop(ml, False) + (nl_ + 4 * nscales(nl_) + P * 2 * nl_)
    out["ring_allreduce_sim_256MiB_per_rank"] = {
        "ranks": P, "elements": nl_, "ms": round(ms, 4), "kernel_bytes": kb2,
        "GB/s": round(kb2 / (ms * 1e-3) / 1e9, 1), "frac_of_peak": round(kb2 / (ms * 1e-3) / 1e9 / peak, 4)}
    del bws
    out["ring_allreduce_sim_256MiB_per_rank"]["breakdown"] = allreduce_breakdown(w, torch, dev, st, big, bres, peak)
    out["ring_allreduce_sim"]["frac_of_peak"] = round(out["ring_allreduce_sim"]["GB/s"] / peak, 4)
    del big, bres
    name, b, mm, kk = wl.tensors[0]
    c, sc, sb = ds.mx[0]
    outw = torch.empty((b, mm, kk), dtype=torch.bfloat16, device=dev)
    ms = timed(torch, st, lambda: w.mxfp8_dequantize_swizzled(c, sc, out=outw, stream=st), flush)
    nbytes = 3 * b * mm * kk + sb
    out["mxfp8_dequantize"] = {"tensor": name, "elements": b * mm * kk, "us": round(1e3 * ms, 2),
                               "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                               "frac_of_peak": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4)}
    del outw
    # NEXT-4: the layer's MXFP8 weights packed with their scales into transfer
    # buffers of at most 256 MiB (each weight and its scale in one buffer), all
    # buffers filled by one gather launch, then scattered back by one launch
    pairs = [(c.numel(), sb_) for c, _, sb_ in ds.mx]
    slots, sizes = w.fp8q_pack_plan(pairs, 256 << 20)
    bufs = [torch.empty(sz, dtype=torch.uint8, device=dev) for sz in sizes]
    outs_c = [torch.empty_like(c) for c, _, _ in ds.mx]
    outs_s = [torch.empty(sb_, dtype=torch.uint8, device=dev) for _, _, sb_ in ds.mx]
    gather, scatter = [], []
    for (bt, co, so), (c, sc_, sb_), oc, os_ in zip(slots, ds.mx, outs_c, outs_s):
        cv = c.view(-1)
        gather += [(cv, bufs[bt][co:co + cv.numel()]), (sc_[:sb_], bufs[bt][so:so + sb_])]
        scatter += [(bufs[bt][co:co + cv.numel()], oc.view(-1)), (bufs[bt][so:so + sb_], os_)]
    moved = sum(a + b for a, b in pairs)
    ms_g = timed(torch, st, lambda: w.fp8q_copy_segments(gather, stream=st), flush)
    ms_s = timed(torch, st, lambda: w.fp8q_copy_segments(scatter, stream=st), flush)
    torch.cuda.synchronize()
    same = all(torch.equal(oc, c) for oc, (c, _, _) in zip(outs_c, ds.mx)) and \
        all(torch.equal(os_, sc_[:sb_]) for os_, (_, sc_, sb_) in zip(outs_s, ds.mx))
    out["pack_layer"] = {"weights": len(pairs), "buffers": len(sizes), "cap_bytes": 256 << 20, "bytes": moved,
                         "gather_us": round(1e3 * ms_g, 2), "scatter_us": round(1e3 * ms_s, 2),
                         "GB/s": round(2 * moved / (ms_g * 1e-3) / 1e9, 1),
                         "frac_of_peak": round(2 * moved / (ms_g * 1e-3) / 1e9 / peak, 4),
                         "round_trip_equal": same,
                         "bytes_counted": "read + written by the gather launch"}
    del bufs, outs_c, outs_s, gather, scatter
    codes = torch.empty(P * n, dtype=torch.uint8, device=dev)
    sa = torch.empty(4, dtype=torch.float32, device=dev)
    x = ds.bucket.reshape(-1)
    ms = timed(torch, st, lambda: w.fp8q_quantize_tensorwise(x, "e4m3", codes=codes, scale_amax=sa, stream=st), flush)
    nbytes = 2 * 2 * P * n + P * n                        # two passes over the input, one over the codes
    out["quantize_tensorwise"] = {"elements": P * n, "us": round(1e3 * ms, 2),
                                  "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                  "frac_of_peak": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4)}
    return out


def allreduce_breakdown(w, torch, dev, st, parts, res_one_call, peak, reps=10):
    """The simulated ring AllReduce's launches one by one: the same schedule
    as fp8q_ring_allreduce_sim, replayed through the public entry points
    (one grouped quantize, P - 1 hop groups, the all-gather decode), with
    events around each launch (median of `reps`, L2 flushed before each
    pass) and around the whole sequence.  Its results must equal the
    one-call collective's, byte for byte."""
    L = w.lib()
    vp = ctypes.c_void_p
    P, n = len(parts), parts[0].numel()
    m = n // P
    u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
    msg = [[(torch.empty(m, dtype=u8, device=dev), torch.empty(nscales(m), dtype=f32, device=dev)) for _ in range(P)]
           for _ in range(2)]
    fin_c = torch.empty(n, dtype=u8, device=dev)
    fin_s = torch.empty(nscales(n), dtype=f32, device=dev)
    res = [torch.empty(n, dtype=bf, device=dev) for _ in range(P)]
    sp = vp(st.cuda_stream)
    steps = []
    items = (w.fp8q_quant_t * P)(*[w.fp8q_quant_t(parts[i].data_ptr() + 2 * i * m, m, msg[0][i][0].data_ptr(),
                                                  msg[0][i][1].data_ptr()) for i in range(P)])
    steps.append(("quantize_group", P * bytes_quantize(m),
                  lambda: L.fp8q_quantize_blockwise_group(items, P, 0, ctypes.c_uint(0), sp)))
    keep = [items]
    for s_ in range(1, P):
        hops = (w.fp8q_hop_t * P)()
        for i in range(P):
            frm, c = (i - 1) % P, (i - s_) % P
            ic, isc = msg[(s_ - 1) & 1][frm]
            if s_ < P - 1:
                oc, osc = msg[s_ & 1][i][0].data_ptr(), msg[s_ & 1][i][1].data_ptr()
            else:
                oc, osc = fin_c.data_ptr() + c * m, fin_s.data_ptr() + 4 * c * (m // 128)
            hops[i] = w.fp8q_hop_t(ic.data_ptr(), isc.data_ptr(), parts[i].data_ptr() + 2 * c * m, m, oc, osc, None)
        keep.append(hops)
        steps.append((f"hop_group_{s_}", P * bytes_hop(m, False),
                      (lambda h=hops: L.fp8q_ring_hop_group_ex(h, P, 0, ctypes.c_uint(w.FP8Q_HOP_LOCAL_READY), sp))))
    outs = (vp * P)(*[r.data_ptr() for r in res])
    steps.append(("gather_decode", n + 4 * nscales(n) + P * 2 * n,
                  lambda: L.fp8q_gather_decode(vp(fin_c.data_ptr()), vp(fin_s.data_ptr()), n, 0, outs, P,
                                               ctypes.c_uint(0), sp)))
    flush = L2Flush(torch, dev)
    Ev = torch.cuda.Event
    per = [[] for _ in steps]
    whole = []
    for rep in range(reps + 1):
        flush()
        evs = [(Ev(enable_timing=True), Ev(enable_timing=True)) for _ in steps]
        for (name, _, fn), (a, b) in zip(steps, evs):
            a.record(st)
            if fn() != 0:
                raise RuntimeError(f"AllReduce breakdown: {name} failed")
            b.record(st)
        flush()
        a0, b0 = Ev(enable_timing=True), Ev(enable_timing=True)
        a0.record(st)
        for _, _, fn in steps:
            fn()
        b0.record(st)
        torch.cuda.synchronize(dev)
        if rep:
            for i, (a, b) in enumerate(evs):
                per[i].append(a.elapsed_time(b))
            whole.append(a0.elapsed_time(b0))
    equal = all(torch.equal(a, b) for a, b in zip(res, res_one_call))
    rows = []
    for (name, nbytes, _), t in zip(steps, per):
        us = 1e3 * sorted(t)[len(t) // 2]
        rows.append({"launch": name, "us": round(us, 2), "bytes": nbytes,
                     "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "frac_of_peak": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)})
    wm = sorted(whole)[len(whole) // 2]
    return {"launches": rows, "sequence_ms": round(wm, 4),
            "sum_of_launches_ms": round(sum(r["us"] for r in rows) / 1e3, 4),
            "results_equal_one_call": equal,
            "timing": "events around each launch (no overlap between launches), and around the whole sequence "
                      "(dependent launch as in the one-call collective)"}


def vec3p5b_row(wl, torch, peak, reps=3):
    """The 3.5e9-element gradient vector: 4 shards quantized to e4m3 (one
    launch per shard), then the 4-shard fused reduce to bf16 streamed in
    2^27-element chunks (launched back to back).  The inputs are drawn on the
    device from a seeded Philox normal with the vector's distribution
    (N(0, 1e-4^2), 1e-4 outliers x1000, the same 64 zero blocks per shard);
    the full-size parity test uses the counter-based generator instead, which
    is too slow on the host for a timing row.  Medians of `reps`."""
    import gen
    w, dev, st = wl.w, wl.dev, wl.stream
    L = w.lib()
    n, k, chunk = gen.VEC_N, gen.VEC_K, gen.VEC_CHUNK
    nb = nscales(n)
    free, _ = torch.cuda.mem_get_info(dev)
    need = k * (n + 4 * nb) + 2 * 2 * n
    if free < need * 1.1:
        return {"skipped": f"needs {need / 2**30:.1f} GiB, {free / 2**30:.1f} GiB free"}
    x = torch.empty(n, dtype=torch.bfloat16, device=dev)
    codes = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(k)]
    scales = [torch.empty(nb, dtype=torch.float32, device=dev) for _ in range(k)]
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    vp = ctypes.c_void_p
    sp_ = vp(st.cuda_stream)

    def ev():
        return torch.cuda.Event(enable_timing=True)
    q_ms = []
    for r in range(k):
        g = torch.Generator(device=dev)
        g.manual_seed(100 + r)
        for c0 in range(0, n, chunk):
            cnt = min(chunk, n - c0)
            v = torch.randn(cnt, device=dev, generator=g).mul_(1e-4)
            hit = torch.rand(cnt, device=dev, generator=g) < 1e-4
            v[hit] *= 1000.0
            x[c0:c0 + cnt].copy_(v)
            del v, hit
        zb = torch.from_numpy(gen.vec_zero_blocks(r).astype("int64")).to(dev)
        idx = (zb[:, None] * 128 + torch.arange(128, device=dev)[None, :]).reshape(-1)
        x[idx[idx < n]] = 0
        args = (vp(x.data_ptr()), ctypes.c_size_t(n), ctypes.c_int(0), vp(codes[r].data_ptr()),
                vp(scales[r].data_ptr()), sp_)
        torch.cuda.synchronize()
        for _ in range(reps):
            a, b = ev(), ev()
            a.record(st)
            if L.fp8q_quantize_blockwise(*args) != 0:
                raise RuntimeError("3.5B quantize failed")
            b.record(st)
            torch.cuda.synchronize()
            q_ms.append(a.elapsed_time(b))
    del x
    calls = []
    for c0 in range(0, n, chunk):
        cnt = min(chunk, n - c0)
        b0 = c0 // 128
        cp = (vp * k)(*[codes[r].data_ptr() + c0 for r in range(k)])
        spp = (vp * k)(*[scales[r].data_ptr() + 4 * b0 for r in range(k)])
        calls.append((cp, spp, ctypes.c_int(k), ctypes.c_size_t(cnt), ctypes.c_int(0), vp(out.data_ptr() + 2 * c0),
                      vp(None), sp_))
    r_ms = []
    for _ in range(reps):
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record(st)
        for c in calls:
            if L.fp8q_dequant_reduce(*c) != 0:
                raise RuntimeError("3.5B reduce failed")
        b.record(st)
        torch.cuda.synchronize()
        r_ms.append(a.elapsed_time(b))
    del codes, scales, out
    torch.cuda.empty_cache()
    q_med = sorted(q_ms)[len(q_ms) // 2]
    r_med = sorted(r_ms)[len(r_ms) // 2]
    qb = bytes_quantize(n)
    rb = k * (n + 4 * nb) + 2 * n
    return {"elements": n, "shards": k,
            "quantize": {"launches": k * reps, "ms_median": round(q_med, 3), "bytes": qb,
                         "GB/s": round(qb / (q_med * 1e-3) / 1e9, 1),
                         "frac_of_peak": round(qb / (q_med * 1e-3) / 1e9 / peak, 4)},
            "reduce_streamed": {"chunks": len(calls), "ms_median": round(r_med, 3), "bytes": rb,
                                "GB/s": round(rb / (r_med * 1e-3) / 1e9, 1),
                                "frac_of_peak": round(rb / (r_med * 1e-3) / 1e9 / peak, 4)},
            "inputs": "device Philox normal, seeds 100 + shard, with the vector's outliers and zero blocks"}


def mxfp8_stack_row(wl, torch, peak, layers=48, reps=3):
    """MXFP8 prequantization of a whole Qwen3-30B-A3B-shaped stack: 48 layers
    (29.9e9 weights, 59.8 GB of bf16) resident on the device, one grouped
    launch per layer, launched back to back (times: medians of `reps` passes
    over the stack).  A second pass puts events between the layers and gives
    the spread of the per-layer rate.  The weights are drawn on the device
    from seeded Philox normals with the stack's distribution (N(0, 0.02^2),
    1% of rows x50): the counter-based host generator would need minutes for
    29.9e9 values."""
    import gen
    w, dev, st = wl.w, wl.dev, wl.stream
    L = w.lib()
    tensors = gen.QWEN3_TENSORS
    per_layer = sum(3 * b * m * k + w.mxfp8_swizzled_scale_bytes(b, m, k) for _, b, m, k in tensors)
    free, _ = torch.cuda.mem_get_info(dev)
    if free < layers * per_layer * 1.05 + (2 << 30):
        return {"skipped": f"needs {layers * per_layer / 2**30:.1f} GiB, {free / 2**30:.1f} GiB free"}
    g = torch.Generator(device=dev)
    keep, groups = [], []
    for l in range(layers):
        arr = (w.mxfp8_tensor_t * len(tensors))()
        for t, (name, b, m, k) in enumerate(tensors):
            g.manual_seed(10_000 + 100 * l + t)
            x32 = torch.randn((b, m, k), device=dev, generator=g).mul_(0.02)
            rows = torch.rand((b, m, 1), device=dev, generator=g) < 0.01
            x = torch.where(rows, x32 * 50.0, x32).to(torch.bfloat16)
            del x32, rows
            c = torch.empty((b, m, k), dtype=torch.uint8, device=dev)
            sc = torch.empty(w.mxfp8_swizzled_scale_bytes(b, m, k), dtype=torch.uint8, device=dev)
            arr[t] = w.mxfp8_tensor_t(x.data_ptr(), b, m, k, c.data_ptr(), sc.data_ptr())
            keep += [x, c, sc]
        groups.append(arr)
    torch.cuda.synchronize(dev)
    sp = ctypes.c_void_p(st.cuda_stream)
    ready = ctypes.c_uint(w.FP8Q_INPUTS_READY)
    Ev = torch.cuda.Event
    whole, per = [], []
    for rep in range(reps + 1):
        a, b_ = Ev(enable_timing=True), Ev(enable_timing=True)
        a.record(st)
        for arr in groups:
            if L.mxfp8_quantize_swizzled_group_ex(arr, len(tensors), ready, sp) != 0:
                raise RuntimeError("MXFP8 stack launch failed")
        b_.record(st)
        torch.cuda.synchronize(dev)
        if rep:
            whole.append(a.elapsed_time(b_))
    evs = [(Ev(enable_timing=True), Ev(enable_timing=True)) for _ in groups]
    for arr, (a, b_) in zip(groups, evs):
        a.record(st)
        L.mxfp8_quantize_swizzled_group_ex(arr, len(tensors), ready, sp)
        b_.record(st)
    torch.cuda.synchronize(dev)
    per = sorted(per_layer / (a.elapsed_time(b_) * 1e-3) / 1e9 for a, b_ in evs)
    ms = sorted(whole)[len(whole) // 2]
    total = layers * per_layer
    del keep, groups
    torch.cuda.empty_cache()
    return {"layers": layers, "weights": layers * sum(b * m * k for _, b, m, k in tensors), "bytes": total,
            "ms": round(ms, 3), "GB/s": round(total / (ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round(total / (ms * 1e-3) / 1e9 / peak, 4),
            "per_layer_GBps": {"min": round(per[0], 1), "median": round(per[len(per) // 2], 1),
                               "max": round(per[-1], 1)},
            "launches": f"{layers} grouped launches (7 tensors each) back to back; medians of {reps} passes",
            "inputs": "device Philox normal N(0, 0.02^2), 1% of rows x50, seed 10000 + 100 * layer + tensor"}


def graph_timed(wl, torch, flush, steps, dom, barrier, clocks):
    """K replays of the step captured once as a CUDA graph, on its own buffer
    set and stream, with the dominant kernel bracketed by event nodes
    captured in the graph (external events).  L2 is flushed before every
    replay, outside the step events.  Returns (timing dict, None), or
    (None, reason) where this torch cannot record events inside a graph."""
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None, "torch.cuda.Event has no external (graph-node) events"
    dev = wl.dev
    s = torch.cuda.Stream(dev)
    ds = DeviceSet(wl, s)
    wl.h2d(ds, s)
    with torch.cuda.stream(s):
        ds.run()                                   # first-call setup outside the capture
    torch.cuda.synchronize(dev)
    nl = len(ds.launches)
    dom_ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * nl)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ds.run(dom_ev, only=dom)
    main = torch.cuda.current_stream(dev)
    dom_idx = [j for j, l in enumerate(ds.launches) if l[0] == dom]
    step_ms, dom_ms = [], []
    g.replay()                                     # one untimed replay
    torch.cuda.synchronize(dev)
    barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        g.replay()
        b.record(main)
        torch.cuda.synchronize(dev)                # the graph's events are re-recorded by every replay
        step_ms.append(a.elapsed_time(b))
        dom_ms += [dom_ev[2 * j].elapsed_time(dom_ev[2 * j + 1]) for j in dom_idx]
    barrier()
    t1 = time.perf_counter()
    same = all(torch.equal(o.contiguous().view(-1).view(torch.uint8), r.contiguous().view(-1).view(torch.uint8))
               for o, r in zip(ds.outputs, wl.sets[0].outputs))
    del g, ds
    torch.cuda.empty_cache()
    return {"ms_mean": sum(step_ms) / steps, "ms_median": sorted(step_ms)[steps // 2], "dom_ms": dom_ms,
            "outputs_equal_stream_run": same, "clocks": clocks.summary(t0, t1)}, None


def hbm_copy_check(torch, dev, nbytes=2 << 30, reps=5):
    """A device-to-device copy of `nbytes` on this GPU in the same run (read
    plus written bytes over the median time): the box's own copy rate, shown
    next to the peak that the fractions use."""
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    src.fill_(1)
    dst.copy_(src)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = sorted(times)[len(times) // 2]
    del src, dst
    torch.cuda.empty_cache()
    return {"GB/s": round(2 * nbytes / (ms * 1e-3) / 1e9, 1), "bytes_moved": 2 * nbytes, "ms_median": round(ms, 4),
            "what": "device-to-device copy of 2 GiB, median of 5"}


def host_cpu():
    """The host cores the oracle runs on."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "processor name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:                 # Arm: implementer and part numbers
        ids = {}
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    key = line.split(":")[0].strip()
                    if key in ("CPU implementer", "CPU part") and key not in ids:
                        ids[key] = line.split(":", 1)[1].strip()
        except OSError:
            pass
        if ids:
            model = " ".join(f"{k_} {v_}" for k_, v_ in ids.items())
    return {"nproc": os.cpu_count(), "usable": len(os.sched_getaffinity(0)), "model": model,
            "arch": os.uname().machine}


# ---------------------------------------------------------------- main ----
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fp8q", choices=["fp8q", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-vec3p5b", action="store_true", help="skip the 3.5e9-element vector row")
    ap.add_argument("--no-stack", action="store_true", help="skip the 48-layer MXFP8 stack row")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES) + ["mxfp8_dequantize", "ring_allreduce_sim", "ring_hop_256MiB"],
                    help="launch one kernel of the step a few times on its bench inputs and exit (for ncu)")
    ap.add_argument("--profile-launches", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.profile_launches)
        return
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    topo = bind_to_gpu_numa(torch, dev)
    wl = Workload(dev, rank, torch)
    flush = L2Flush(torch, dev)
    warmup = max(args.warmup, 3)
    steps = max(args.steps, 1)
    nl = len(wl.launches)
    for _ in range(warmup):
        flush()
        wl.run()
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(("GPU-" + str(uuid)) if uuid is not None else None)
    clocks.start()
    time.sleep(0.05)

    # ---------------- per-kernel breakdown (before the timed region) ------
    # every launch bracketed by events: the share of each kernel and the
    # kernel whose roofline is reported
    nbreak = min(steps, 50)
    break_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nl)] for _ in range(nbreak)]
    for i in range(nbreak):
        flush()
        wl.run(break_ev[i])
    torch.cuda.synchronize()
    per_kind = {}
    for i in range(nbreak):
        for j, (kind, nbytes, elems, _, _) in enumerate(wl.launches):
            dt = break_ev[i][2 * j].elapsed_time(break_ev[i][2 * j + 1])
            d = per_kind.setdefault(kind, {"launches": 0, "ms": 0.0, "bytes": 0, "elems": 0, "all": []})
            d["launches"] += 1
            d["ms"] += dt
            d["bytes"] += nbytes
            d["elems"] += elems
            d["all"].append(dt)
    dom = max(per_kind, key=lambda k: per_kind[k]["ms"])

    # each run of launches of one kernel timed as a whole: inside a run the
    # launches overlap as they do in the timed steps (no event between them)
    seg_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nl)] for _ in range(nbreak)]
    for i in range(nbreak):
        flush()
        wl.run(seg_ev[i], segments=True)
    torch.cuda.synchronize()
    segments = []
    for kind, a, b in wl.sets[0].segments():
        ms = sum(seg_ev[i][2 * a].elapsed_time(seg_ev[i][2 * b + 1]) for i in range(nbreak)) / nbreak
        nbytes = sum(wl.launches[j][1] for j in range(a, b + 1))
        segments.append({"kernel": kind, "launches": b - a + 1, "us": round(1e3 * ms, 2),
                         "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)})

    # ---------------- timed region: K device-resident steps ----------------
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    launch_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nl)] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush()                                     # evict L2 between steps
        step_ev[i][0].record(wl.stream)
        wl.run(launch_ev[i], only=dom)
        step_ev[i][1].record(wl.stream)
    torch.cuda.synchronize()
    barrier()
    t1 = time.perf_counter()
    clock_info = clocks.summary(t0, t1)

    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms_local = sum(step_ms) / steps
    dom_ms, dom_launches = 0.0, 0
    for i in range(steps):
        for j, (kind, _, _, _, _) in enumerate(wl.launches):
            if kind == dom:
                dom_ms += launch_ev[i][2 * j].elapsed_time(launch_ev[i][2 * j + 1])
                dom_launches += 1
    dom_bytes = per_kind[dom]["bytes"] // per_kind[dom]["launches"]
    stream_timing = {"ms_per_step": round(ms_local, 4), "GB/s": round(wl.step_bytes / (ms_local * 1e-3) / 1e9, 1),
                     "dominant_kernel_avg_us": round(1e3 * dom_ms / dom_launches, 2), "clocks": clock_info}

    # ---------------- timed region, graph form: K replays of the step -------
    graph, graph_why = graph_timed(wl, torch, flush, steps, dom, barrier, clocks)
    if graph is not None and graph["outputs_equal_stream_run"]:
        headline = "cuda_graph"
        ms_local = graph["ms_mean"]
        dom_ms, dom_launches = sum(graph["dom_ms"]), len(graph["dom_ms"])
        clock_info = graph["clocks"]
    else:
        headline = "stream"
    graph_timing = ({"unavailable": graph_why} if graph is None else
                    {"ms_per_step": round(graph["ms_mean"], 4), "ms_median": round(graph["ms_median"], 4),
                     "GB/s": round(wl.step_bytes / (graph["ms_mean"] * 1e-3) / 1e9, 1),
                     "dominant_kernel_avg_us": round(1e3 * sum(graph["dom_ms"]) / max(1, len(graph["dom_ms"])), 2),
                     "outputs_equal_stream_run": graph["outputs_equal_stream_run"], "clocks": graph["clocks"]})

    # the same steps with programmatic dependent launch switched off
    wl.w.fp8q_set_launch_overlap(False)
    noov_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nbreak)]
    for i in range(nbreak):
        flush()
        noov_ev[i][0].record(wl.stream)
        wl.run()
        noov_ev[i][1].record(wl.stream)
    torch.cuda.synchronize()
    wl.w.fp8q_set_launch_overlap(True)
    ms_no_overlap = sum(a.elapsed_time(b) for a, b in noov_ev) / nbreak

    ms_step, bytes_all, elems_all = combine_over_ranks(dist if world > 1 else None, dev, ms_local,
                                                       float(wl.step_bytes), float(wl.step_elems))
    value_gbs = bytes_all / (ms_step * 1e-3) / 1e9

    # ---------------- end to end: host buffers through the C ABI -----------
    # three windows, the median reported: the host link is shared with the
    # machine's other GPUs, and one window can land on a neighbour's transfer
    barrier()
    e2e_windows = []
    for _ in range(3):
        ms_w, bi, bo = wl.e2e(max(1, min(args.e2e_steps, steps)))
        e2e_windows.append(ms_w)
    e2e_local = sorted(e2e_windows)[1]
    barrier()
    clocks.stop()
    e2e_ms, _, _ = combine_over_ranks(dist if world > 1 else None, dev, e2e_local, 0.0, 0.0)
    e2e_gbs = bytes_all / (e2e_ms * 1e-3) / 1e9
    e2e_steps = max(1, min(args.e2e_steps, steps))

    fvn = fused_vs_naive(wl, torch)
    sweep = ring_sweep(wl, torch)
    # a bounded copy wait that ran out leaves invalid outputs and an error
    # bit: every rank reads its bits before reporting anything
    dev_errors = wl.w.fp8q_device_errors(clear=False)
    if dev_errors:
        raise RuntimeError(f"rank {rank}: a kernel raised device error bits {dev_errors:#x}")
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    copy_check = hbm_copy_check(torch, dev)
    extras = extra_rows(wl, torch, peak)
    if not args.no_vec3p5b:
        extras["vec3p5b"] = vec3p5b_row(wl, torch, peak)
    if not args.no_stack:
        extras["mxfp8_48_layers"] = mxfp8_stack_row(wl, torch, peak)
    total_ms = sum(d["ms"] for d in per_kind.values())
    kernels = {}
    for kind, d in per_kind.items():
        avg_ms = d["ms"] / d["launches"]
        gbs = d["bytes"] / (d["ms"] * 1e-3) / 1e9
        med_ms = sorted(d["all"])[len(d["all"]) // 2]
        kernels[kind] = {"launches_per_step": d["launches"] // nbreak, "avg_us": round(1e3 * avg_ms, 2),
                         "median_us": round(1e3 * med_ms, 2),
                         "bytes_per_launch": d["bytes"] // d["launches"], "GB/s": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4), "share": round(d["ms"] / total_ms, 4)}
    achieved = dom_bytes * dom_launches / (dom_ms * 1e-3) / 1e9
    traffic = ncu_traffic(dom)
    line = {
        "metric": METRIC, "value": round(value_gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "bucket_elements_per_shard": wl.n, "shards": wl.k,
                   "layer_weights": sum(b * m * k for _, b, m, k in wl.tensors), "launches_per_step": nl,
                   "l2": "flushed between steps (256 MiB write, then 256 MiB read, outside the step events)",
                   "io": "bf16 in; e4m3/e5m2 codes + fp32 scales, E8M0 swizzled scales, bf16/fp32 sums out"},
        "elements_per_s": round(elems_all / (ms_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": f"{peak_kind} HBM copy GB/s", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "avg_us": round(1e3 * dom_ms / dom_launches, 2),
                     "copy_check": copy_check,
                     "timing": f"events around each launch of this kernel in the K timed steps ({headline} form)"},
        "kernels": kernels,
        "kernels_timing": f"separate pass of {nbreak} steps with events around every launch",
        "segments": [dict(g, frac_of_peak=round(g["GB/s"] / peak, 4)) for g in segments],
        "segments_timing": f"separate pass of {nbreak} steps with events only where the kernel changes",
        "timing": {"headline": headline,
                   "what": "value, ms_per_step and the roofline come from the headline form; both forms run K "
                           "steps with L2 flushed before each, outside the step events",
                   "stream": stream_timing, "cuda_graph": graph_timing},
        "launch_overlap": {"step_ms_on": stream_timing["ms_per_step"], "step_ms_off": round(ms_no_overlap, 4),
                           "steps_off": nbreak,
                           "what": "programmatic dependent launch of every kernel (on in the timed steps)"},
        "e2e": {"value": round(e2e_gbs, 1), "unit": "GB/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "ms_per_step": round(e2e_ms, 3), "steps": e2e_steps,
                "windows_ms_per_step": [round(x, 3) for x in e2e_windows],
                "what": f"median of 3 windows of {e2e_steps} pipelined steps",
                "copy_GBps_alone": getattr(wl, "copy_gbps", None),
                "outputs_equal_device_run": getattr(wl, "e2e_outputs_equal", None),
                "host": topo,
                "pipeline": "H2D, kernels and D2H on three streams (one cudaMemcpyAsync per direction: the "
                            "inputs and the results each lie in one buffer), two device buffer sets"},
        "gpu_launches": nl * steps,
        "fused_vs_naive_reduce": fvn,
        "next_rows": extras,
        "ring_hop_sweep": {k: dict(v, frac_of_peak=round(v["GB/s"] / peak, 4),
                                   chain_7_hops=dict(v["chain_7_hops"],
                                                     frac_of_peak=round(v["chain_7_hops"]["GB/s"] / peak, 4)))
                           for k, v in sweep.items()},
        "clocks": clock_info,
        "cpu_baseline": None,
        "parity_checked": None,
    }
    if world == 1 and not args.no_cpu_baseline:
        keep = {}
        nbytes, elems, dt, desc = oracle_sample(oracle_fraction_for(10.0), keep=keep)
        line["parity_checked"] = parity_against_oracle(wl.sets[0], keep)
        line["cpu_baseline"] = {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": round(dt, 2), "host": host_cpu()}
        ncores = len(os.sched_getaffinity(0))
        if ncores > 1:
            # the same oracle over independent parts on every usable core, a
            # second baseline row; its sample is sized for about 5 s
            frac = min(1.0, oracle_fraction_for(5.0) * ncores)
            nb_all, _, dt_all, desc_all = oracle_sample(frac, threads=ncores)
            line["cpu_baseline_all_cores"] = {"value": round(nb_all / dt_all / 1e9, 4), "unit": "GB/s",
                                              "cores": ncores, "kind": "oracle", "sample": desc_all,
                                              "seconds": round(dt_all, 2)}
    line["device_errors"] = wl.w.fp8q_device_errors(clear=False)
    print(json.dumps(line), flush=True)
    if line["device_errors"]:
        raise RuntimeError(f"a kernel raised device error bits {line['device_errors']:#x}")
    if line["parity_checked"] and line["parity_checked"]["mismatches"]:
        raise RuntimeError(f"the GPU step differs from the oracle: {line['parity_checked']}")
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
