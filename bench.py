"""Benchmark: W8A16 FP8 block-scaled decode GEMM on GB300 (one JSON line).

Headline workload: FFN gate/up, M=16, N=17408, K=5120 (89 MB of E4M3
weights, [128 x 128] FP32 block scales, BF16 X and Y).  One step is one call of
the whole path (weight stream, dequant, tensor-core MMA, two-level fold,
split-K reduction, BF16 store).  Inputs are resident in HBM; the weight
matrix rotates over enough copies (>= 2x the L2 size) that no step finds its
weights in L2.  Calls are launched with weight-prefetch overlap (a call may
start streaming its weights while the previous call finishes; it waits for
that call before it reads X or writes Y), as consecutive decode GEMMs would
run; `--overlap 0` times them strictly one after another.  `value` is
algorithmic bytes per call (W + scales + X + Y, each counted once) / device
time per call.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--quick] [--overlap 0|1]

Under torchrun each rank runs an independent replica (the GEMM has no
exchange step); rank 0 prints the line with the max time over ranks.
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

METRIC = "achieved HBM GB/s (and µs/call) of FP8 block-scaled W8A16 GEMM at M=1..32"
PAGE_BASELINE_GBPS = 342.0   # H100 w8a16_gemv_batch16, gate/up, M=16 (atlas page, WHY table)
HEAD = dict(M=16, N=17408, K=5120, config_id=1)
L2_BYTES = 129 * 1000 * 1000


def fp8_bytes(M, N, K):
    nb, kb = -(-N // 128), -(-K // 128)
    return N * K + nb * kb * 4 + M * K * 2 + M * N * 2


def lut3_bytes(M, N, K):
    return (-(-N // 128)) * (-(-K // 256)) * 16384 + N * (K // 128) * 2 + 16 + M * K * 2 + M * N * 2


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The sources the headline (FP8) kernel is built from: a change to any of
# them makes a stored ncu traffic figure stale.
HEADLINE_KERNEL_SOURCES = ("qg_fp8.cu", "qg_gemm.cuh", "qg_device.cuh", "qg_internal.h")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_quantized_qgemm_gb300", "csrc")
    for name in HEADLINE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(name, calls_bytes):
    """DRAM bytes per launch from a committed ncu summary of the same kernel
    source, else None."""
    path = os.path.join(ROOT, "profiles", f"{name}.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    t = d.get("dram_bytes_per_launch")
    if t is None:
        return None
    scale = d.get("scale_to_full", 1.0)
    return float(t) * float(scale)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None):
        self.rows = []
        self.proc = None
        self.uuid = device_uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._first = threading.Event()
        self._t.start()
        self._first.wait(timeout=5.0)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))
            self._first.set()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        for _, line in self.rows:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def head_config(overlap, world):
    """The headline workload's `config` (shared by both arms of the bench)."""
    M, N, K = HEAD["M"], HEAD["N"], HEAD["K"]
    copies = -(-2 * L2_BYTES // (N * K)) + 1   # as Fp8Case
    return {"workload": "fp8_block gate/up M=16 N=17408 K=5120",
            "M": M, "N": N, "K": K, "weights": "E4M3 [N,K] + FP32 [128x128] block scales",
            "arith": "E4M3 weights as stored into tcgen05 kind::f8f6f4 (no weight dequant); BF16 X split "
                     "per (row, 128-K block) into two power-of-two-scaled E4M3 planes; FP32 two-level fold; "
                     "BF16 out",
            "l2": f"inputs larger than L2: {copies} rotating weight copies ({copies * N * K / 1e6:.0f} MB)",
            "overlap": "weight prefetch overlaps the previous call" if overlap else "off",
            "parallelism": "replicas" if world > 1 else "1 GPU"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, world, device="cuda"):
    """The maximum of x over all ranks of the default process group (x itself
    for one rank): the job's time is its slowest rank's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ----------------------------------------------------------------- our arm
def time_calls(torch, stream, fn, steps, warmup):
    """Device time per call (ms) of `steps` calls issued back to back on
    `stream`, after `warmup` untimed ones; CUDA events on that stream."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            fn(i)
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


class Fp8Case:
    """One FP8 problem resident on the device: enough rotating weight copies
    (>= 2x L2) that no call finds its weights in L2; M <= M_max runs on the
    first M rows of X and Y."""

    def __init__(self, torch, qg, M_max, N, K, config_id):
        import workloads as wl
        self.torch, self.qg = torch, qg
        self.p = wl.make_fp8_problem(M_max, N, K, config_id=config_id)
        self.N, self.K = N, K
        self.copies = -(-2 * L2_BYTES // (N * K)) + 1
        self.W = [torch.from_numpy(self.p.W).cuda() for _ in range(self.copies)]
        self.S = torch.from_numpy(self.p.S).cuda()
        self.X = torch.from_numpy(self.p.X.view(np.int16)).view(torch.bfloat16).cuda()
        self.Y = torch.empty((M_max, N), dtype=torch.bfloat16, device="cuda")
        self.ws = qg.Workspace()

    def stepper(self, M, stream):
        qg, N, K = self.qg, self.N, self.K
        buf = self.ws.get(qg.workspace_bytes(qg.KIND_FP8_BLOCK, M, N, K))
        ws_ptr = buf.data_ptr() if buf is not None else None
        ws_n = buf.numel() if buf is not None else 0
        lib, sptr, copies = qg.lib, stream.cuda_stream, self.copies
        xp, yp, sp = self.X.data_ptr(), self.Y.data_ptr(), self.S.data_ptr()
        wps = [w.data_ptr() for w in self.W]

        def step(i):
            r = lib.qgemm_fp8_block(xp, K, wps[i % copies], sp, yp, N, M, N, K, ws_ptr, ws_n, sptr)
            if r:
                raise RuntimeError(qg.status_string(r))
        return step

    def tune(self, M, stream):
        """The exactness-gated dispatch tuner on this shape (its grid stays in
        the process's dispatch table); returns the grid chosen."""
        g, _ = self.qg.tune_fp8(self.X[:M], self.W, self.S, calls=100, workspace=self.ws, stream=stream)
        return g

    def time(self, M, stream, steps, warmup):
        ms = time_calls(self.torch, stream, self.stepper(M, stream), steps, warmup)
        st = self.qg.last_device_status(stream)
        if st:
            raise RuntimeError(f"device status {self.qg.status_string(st)}")
        return ms

    def free(self):
        self.W = self.S = self.X = self.Y = self.ws = None


class Lut3Case:
    """The 3-bit learned-LUT problem, packed once, rotated over >= 2x L2."""

    def __init__(self, torch, qg, M_max, N, K):
        import workloads as wl
        self.torch, self.qg = torch, qg
        p = wl.make_lut3_problem(M_max, N, K, config_id=4)
        packed = qg.pack_lut3(p.codes)
        self.N, self.K = N, K
        self.copies = -(-2 * L2_BYTES // packed.size) + 1
        self.Wq = [torch.from_numpy(packed).cuda() for _ in range(self.copies)]
        self.qm = torch.from_numpy(p.qmap.view(np.int16)).view(torch.float16).cuda()
        self.sc = torch.from_numpy(p.scales.view(np.int16)).view(torch.float16).cuda()
        self.X = torch.from_numpy(p.X.view(np.int16)).view(torch.float16).cuda()
        self.Y = torch.empty((M_max, N), dtype=torch.float16, device="cuda")
        self.ws = qg.Workspace()

    def tune(self, M, stream):
        g, _ = self.qg.tune_lut3(self.X[:M], self.Wq, self.qm, self.sc, self.N, calls=50, workspace=self.ws,
                                 stream=stream)
        return g

    def time(self, M, stream, steps, warmup):
        qg, N, K = self.qg, self.N, self.K
        buf = self.ws.get(qg.workspace_bytes(qg.KIND_LUT3, M, N, K))
        ws_ptr = buf.data_ptr() if buf is not None else None
        ws_n = buf.numel() if buf is not None else 0
        lib, sptr, copies = qg.lib, stream.cuda_stream, self.copies
        xp, yp, qp, scp = self.X.data_ptr(), self.Y.data_ptr(), self.qm.data_ptr(), self.sc.data_ptr()
        wps = [w.data_ptr() for w in self.Wq]

        def step(i):
            r = lib.qgemm_lut3(xp, K, wps[i % copies], qp, scp, yp, N, M, N, K, ws_ptr, ws_n, sptr)
            if r:
                raise RuntimeError(qg.status_string(r))
        ms = time_calls(self.torch, stream, step, steps, warmup)
        st = qg.last_device_status(stream)
        if st:
            raise RuntimeError(f"device status {qg.status_string(st)}")
        return ms

    def free(self):
        self.Wq = self.qm = self.sc = self.X = self.Y = self.ws = None


def e2e_fp8(torch, qg, stream, case, M, steps, warmup):
    """Through the public Python API with host buffers: X in pinned host
    memory, Y into pinned host memory, every step.  qgemm_fp8_block_host
    moves both inside the timed region: its staging kernel reads X over the
    host link, and the GEMM's epilogue stores Y to the host.  Each step reads
    a different X: the steps rotate over host X buffers of distinct contents
    that together exceed twice the L2 size, so no step's X can come from a
    cache."""
    K, N = case.K, case.N
    slots = -(-2 * L2_BYTES // (M * K * 2)) + 1
    Xh = torch.empty((slots, M, K), dtype=torch.bfloat16).pin_memory()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0x51A7E000 + 7)
    for s0 in range(0, slots, 256):
        s1 = min(slots, s0 + 256)
        Xh[s0:s1].copy_(torch.randn((s1 - s0, M, K), generator=gen, device="cuda").to(torch.bfloat16).cpu())
    Yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    stage = torch.empty(M * K, dtype=torch.bfloat16, device="cuda")
    W, S, ws, copies = case.W, case.S, case.ws, case.copies

    def step(i):
        qg.qgemm_fp8_block_host(Xh[i % slots], W[i % copies], S, Y=Yh, X_stage=stage, workspace=ws, stream=stream)

    ms = time_calls(torch, stream, step, steps, warmup)
    st = qg.last_device_status(stream)
    if st:
        raise RuntimeError(f"device status {qg.status_string(st)}")
    # the last step's Y, read on the host, must be the device path's result
    last = steps - 1
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qg.qgemm_fp8_block(Xh[last % slots].cuda(), W[last % copies], S, Y=ref, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    if not torch.equal(ref.cpu().view(torch.int16), Yh.view(torch.int16)):
        raise RuntimeError("host-buffer path differs from the device path")
    return ms, M * K * 2, Yh.numel() * Yh.element_size(), slots


def time_halves(torch, qg, stream, case, steps, warmup):
    """M = 32 as two calls on contiguous 16-row halves of X and Y (plain row
    offsets), one step = both calls."""
    qg_, N, K = qg, case.N, case.K
    buf = case.ws.get(qg_.workspace_bytes(qg_.KIND_FP8_BLOCK, 16, N, K))
    ws_ptr = buf.data_ptr() if buf is not None else None
    ws_n = buf.numel() if buf is not None else 0
    lib, sptr, copies = qg_.lib, stream.cuda_stream, case.copies
    xp, yp, sp = case.X.data_ptr(), case.Y.data_ptr(), case.S.data_ptr()
    wps = [w.data_ptr() for w in case.W]

    def step(i):
        w = wps[i % copies]
        for h in (0, 1):
            r = lib.qgemm_fp8_block(xp + h * 16 * K * 2, K, w, sp, yp + h * 16 * N * 2, N, 16, N, K, ws_ptr, ws_n,
                                    sptr)
            if r:
                raise RuntimeError(qg_.status_string(r))
    ms = time_calls(torch, stream, step, steps, warmup)
    st = qg_.last_device_status(stream)
    if st:
        raise RuntimeError(f"device status {qg_.status_string(st)}")
    return ms


def bf16_bytes(M, N, K):
    return N * K * 2 + M * K * 2 + M * N * 2


class Bf16Case:
    """Unquantised BF16 output-projection (lm_head) shape, weights rotated
    over copies (>= 2x L2)."""

    def __init__(self, torch, qg, M_max, N, K):
        import workloads as wl
        self.torch, self.qg, self.N, self.K = torch, qg, N, K
        p = wl.make_bf16_problem(M_max, N, K, config_id=5)
        self.copies = -(-2 * L2_BYTES // (N * K * 2)) + 1
        self.W = [torch.from_numpy(p.W.view(np.int16)).view(torch.bfloat16).cuda() for _ in range(self.copies)]
        self.X = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
        self.Y = torch.empty((M_max, N), dtype=torch.bfloat16, device="cuda")
        self.ws = qg.Workspace()

    def tune(self, M, stream):
        g, _ = self.qg.tune_bf16(self.X[:M], self.W, calls=50, workspace=self.ws, stream=stream)
        return g

    def time(self, M, stream, steps, warmup):
        qg, N, K = self.qg, self.N, self.K
        buf = self.ws.get(qg.workspace_bytes(qg.KIND_BF16, M, N, K))
        ws_ptr = buf.data_ptr() if buf is not None else None
        ws_n = buf.numel() if buf is not None else 0
        lib, sptr, copies = qg.lib, stream.cuda_stream, self.copies
        xp, yp = self.X.data_ptr(), self.Y.data_ptr()
        wps = [w.data_ptr() for w in self.W]

        def step(i):
            r = lib.qgemm_bf16(xp, K, wps[i % copies], yp, N, M, N, K, ws_ptr, ws_n, sptr)
            if r:
                raise RuntimeError(qg.status_string(r))
        ms = time_calls(self.torch, stream, step, steps, warmup)
        st = qg.last_device_status(stream)
        if st:
            raise RuntimeError(f"device status {qg.status_string(st)}")
        return ms

    def free(self):
        self.W = self.X = self.Y = self.ws = None


class QkvCase:
    """The attention projections Q (N=6144), K and V (N=1024 each) at
    K=5120 sharing X, weights rotated over copies (>= 2x L2)."""

    NS = (6144, 1024, 1024)

    def __init__(self, torch, qg, M_max, K=5120):
        import workloads as wl
        self.torch, self.qg, self.K = torch, qg, K
        ps = [wl.make_fp8_problem(M_max, N, K, config_id=80 + j) for j, N in enumerate(self.NS)]
        per_set = sum(N for N in self.NS) * K
        self.copies = -(-2 * L2_BYTES // per_set) + 1
        self.sets = [[(torch.from_numpy(p.W).cuda(), torch.from_numpy(p.S).cuda()) for p in ps]
                     for _ in range(self.copies)]
        self.X = torch.from_numpy(ps[0].X.view(np.int16)).view(torch.bfloat16).cuda()
        self.Y = [torch.empty((M_max, N), dtype=torch.bfloat16, device="cuda") for N in self.NS]
        self.ws = qg.Workspace()

    def nbytes(self, M):
        """Algorithmic bytes of the three GEMMs with X counted once."""
        return sum(fp8_bytes(M, N, self.K) for N in self.NS) - 2 * M * self.K * 2

    def time(self, M, stream, steps, warmup, fused):
        qg, K = self.qg, self.K
        X = self.X[:M]
        Ys = [Y[:M] for Y in self.Y]
        ws = self.ws

        def step(i):
            ws_set = self.sets[i % self.copies]
            if fused:
                qg.qgemm_fp8_block_multi(X, ws_set, Ys=Ys, workspace=ws, stream=stream)
            else:
                for (W, S), Y in zip(ws_set, Ys):
                    qg.qgemm_fp8_block(X, W, S, Y=Y, workspace=ws, stream=stream)
        ms = time_calls(self.torch, stream, step, steps, warmup)
        st = qg.last_device_status(stream)
        if st:
            raise RuntimeError(f"device status {qg.status_string(st)}")
        return ms

    def free(self):
        self.sets = self.X = self.Y = self.ws = None


class W8a8Case:
    """W8A8 at prefill batch sizes on the gate/up shape: E4M3 activations and
    their scales resident (the quantiser timed on its own), weights rotated
    over copies (>= 2x L2)."""

    def __init__(self, torch, qg, M_max, N, K):
        import workloads as wl
        self.torch, self.qg, self.N, self.K = torch, qg, N, K
        p = wl.make_w8a8_problem(M_max, N, K, config_id=6)
        self.copies = -(-2 * L2_BYTES // (N * K)) + 1
        self.W = [torch.from_numpy(p.W).cuda() for _ in range(self.copies)]
        self.S = torch.from_numpy(p.S).cuda()
        self.X = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).cuda()
        self.ldsx = -(-M_max // 32) * 32
        self.Xq = torch.empty((M_max, K), dtype=torch.uint8, device="cuda")
        self.Sx = torch.empty((-(-K // 128), self.ldsx), dtype=torch.float32, device="cuda")
        self.Y = torch.empty((M_max, N), dtype=torch.bfloat16, device="cuda")
        self.ws = qg.Workspace()

    def tune(self, M, stream):
        """The dispatch tuner on the GEMM of the first M rows (quantised first)."""
        qg, K = self.qg, self.K
        r = qg.lib.qg_quantize_act_e4m3(self.X.data_ptr(), K, self.Xq.data_ptr(), K, self.Sx.data_ptr(), self.ldsx,
                                        M, K, stream.cuda_stream)
        if r:
            raise RuntimeError(qg.status_string(r))
        g, _ = qg.tune_w8a8(self.Xq[:M], self.Sx, self.W, self.S, calls=20, workspace=self.ws, stream=stream)
        return g

    def time(self, M, stream, steps, warmup, what="gemm"):
        """what: "gemm" (qgemm_w8a8_block on resident codes), "quant"
        (qg_quantize_act_e4m3) or "both" (the two launches of a call from
        BF16 activations)."""
        qg, N, K = self.qg, self.N, self.K
        buf = self.ws.get(qg.workspace_bytes(qg.KIND_W8A8, M, N, K))
        ws_ptr = buf.data_ptr() if buf is not None else None
        ws_n = buf.numel() if buf is not None else 0
        lib, sptr, copies, ldsx = qg.lib, stream.cuda_stream, self.copies, self.ldsx
        xp, xqp, sxp, sp, yp = (self.X.data_ptr(), self.Xq.data_ptr(), self.Sx.data_ptr(), self.S.data_ptr(),
                                self.Y.data_ptr())
        wps = [w.data_ptr() for w in self.W]

        def quant():
            r = lib.qg_quantize_act_e4m3(xp, K, xqp, K, sxp, ldsx, M, K, sptr)
            if r:
                raise RuntimeError(qg.status_string(r))

        def gemm(i):
            r = lib.qgemm_w8a8_block(xqp, K, sxp, ldsx, wps[i % copies], sp, yp, N, M, N, K, ws_ptr, ws_n, sptr)
            if r:
                raise RuntimeError(qg.status_string(r))
        quant()
        if what == "gemm":
            step = gemm
        elif what == "quant":
            def step(i):
                quant()
        else:
            def step(i):
                quant()
                gemm(i)
        ms = time_calls(self.torch, stream, step, steps, warmup)
        st = qg.last_device_status(stream)
        if st:
            raise RuntimeError(f"device status {qg.status_string(st)}")
        return ms

    def free(self):
        self.W = self.X = self.Xq = self.Sx = self.Y = self.ws = None


def fp8_tensor_peak():
    """FP8 dense tensor peak: the measured BF16 GEMM peak times the nominal
    FP8 / BF16 ratio (4.5 / 2.25 PFLOP/s)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]) * 2.0, "2 x measured bf16_tflops"
    return 1900.0 * 2.0, "2 x fallback bf16"


def secondary_lines(torch, qg, stream, peak, steps=2000, warmup=50, tune=True):
    """The other configurations (not the headline): us/call, GB/s, fraction
    of the HBM peak.  With `tune`, each shape first runs the library's
    exactness-gated dispatch tuner (outside the timed calls) and its line
    records the grid chosen."""
    out = {}

    def rec(name, ms, nbytes, grid=None):
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 3), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4)}
        if grid is not None:
            out[name]["grid"] = grid

    def tuned(c, m):
        return c.tune(m, stream) if tune else None

    c = Fp8Case(torch, qg, 16, 17408, 5120, 1)
    for m in (1, 8):
        g = tuned(c, m)
        rec(f"fp8_gateup_M{m}", c.time(m, stream, steps, warmup), fp8_bytes(m, 17408, 5120), g)
    c.free()
    c = Fp8Case(torch, qg, 32, 5120, 17408, 2)
    for m in (1, 16, 32):
        g = tuned(c, m)
        rec(f"fp8_down_M{m}", c.time(m, stream, steps, warmup), fp8_bytes(m, 5120, 17408), g)
    # the same 32 rows as two 16-row calls (the weights stream twice; the
    # fraction is taken against the one-call algorithmic bytes)
    rec("fp8_down_M32_halves", time_halves(torch, qg, stream, c, steps, warmup), fp8_bytes(32, 5120, 17408))
    c.free()
    for n in (1024, 5120, 6144):
        c = Fp8Case(torch, qg, 32, n, 5120, 3)
        for m in (1, 2, 4, 5, 8, 16, 17, 24, 32):
            g = tuned(c, m)
            rec(f"fp8_attn_N{n}_M{m}", c.time(m, stream, steps, warmup), fp8_bytes(m, n, 5120), g)
        c.free()
    c = Fp8Case(torch, qg, 1, 256, 512, 0)
    rec("fp8_small_M1", c.time(1, stream, steps, warmup), fp8_bytes(1, 256, 512))
    c.free()
    # unquantised BF16 output projection (lm_head shape)
    c = Bf16Case(torch, qg, 32, 32768, 5120)
    for m in (1, 16, 32):
        g = tuned(c, m)
        rec(f"bf16_lm_head_M{m}", c.time(m, stream, steps // 4, warmup), bf16_bytes(m, 32768, 5120), g)
    c.free()
    # Q, K and V in one launch against the three calls one after another
    c = QkvCase(torch, qg, 32)
    for m in (1, 16, 32):
        rec(f"fp8_qkv_fused_M{m}", c.time(m, stream, steps, warmup, True), c.nbytes(m))
        rec(f"fp8_qkv_separate_M{m}", c.time(m, stream, steps, warmup, False), c.nbytes(m))
    c.free()
    c = Lut3Case(torch, qg, 16, 28672, 8192)
    for m in (1, 4, 8, 16):
        g = tuned(c, m)
        rec(f"lut3_M{m}", c.time(m, stream, steps, warmup), lut3_bytes(m, 28672, 8192), g)
    c.free()
    # W8A8 beyond the decode tier: tensor-bound, so its lines carry TFLOP/s
    # against the FP8 tensor peak
    tpeak, _ = fp8_tensor_peak()
    c = W8a8Case(torch, qg, 1024, 17408, 5120)
    for m in (64, 256, 1024):
        flops = 2.0 * m * 17408 * 5120
        g = tuned(c, m)
        for what in ("gemm", "both"):
            ms = c.time(m, stream, max(50, steps // 20), warmup, what)
            tf = flops / (ms * 1e-3) / 1e12
            out[f"w8a8_gateup_M{m}_{what}"] = {"us": round(ms * 1e3, 3), "TFLOPs": round(tf, 1),
                                               "frac_fp8_tensor": round(tf / tpeak, 4)}
            if g is not None:
                out[f"w8a8_gateup_M{m}_{what}"]["grid"] = g
        out[f"w8a8_gateup_M{m}_quant"] = {"us": round(c.time(m, stream, max(50, steps // 20), warmup, "quant") * 1e3, 3)}
    c.free()
    qg.dispatch_clear()
    torch.cuda.empty_cache()
    return out


def _oracle_rate(oracle, p, M, K, nthreads, budget_s):
    """GB/s of the oracle on a column sample of the problem sized to about
    `budget_s` seconds, and a description of the sample."""
    N = p.W.shape[0]
    cols = 128 if nthreads == 1 else 512
    t0 = time.perf_counter()
    oracle.qgemm_fp8_block(p.X, p.W[:cols], p.S[: -(-cols // 128)], nthreads=nthreads)
    dt = time.perf_counter() - t0
    n_s = int(min(N, max(128, (budget_s / max(dt, 1e-6)) * cols)) // 128 * 128)
    # whole passes over the sample until the budget is spent
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.qgemm_fp8_block(p.X, p.W[:n_s], p.S[: -(-n_s // 128)], nthreads=nthreads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or passes >= 1000:
            break
    gbs = fp8_bytes(M, n_s, K) * passes / dt / 1e9
    return gbs, f"columns 0..{n_s - 1} of {N} (all {M} rows, full K={K}), {passes} passes; {dt:.2f} s"


def cpu_baseline(M, N, K, config_id, budget_s=10.0):
    """The oracle as it stands, on the host cores (all of them, and one),
    over a column sample of the same workload sized to roughly `budget_s`
    seconds each."""
    import oracle
    import workloads as wl
    p = wl.make_fp8_problem(M, N, K, config_id=config_id)
    nt = oracle.max_threads()
    gbs, sample = _oracle_rate(oracle, p, M, K, nt, budget_s)
    gbs1, sample1 = _oracle_rate(oracle, p, M, K, 1, budget_s)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": nt, "kind": "oracle", "sample": sample,
            "single_thread": {"value": round(gbs1, 5), "unit": "GB/s", "cores": 1, "sample": sample1}}, p


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    import workloads as wl
    M, N, K, cid = HEAD["M"], HEAD["N"], HEAD["K"], HEAD["config_id"]
    p = wl.make_fp8_problem(M, N, K, config_id=cid)
    nt = oracle.max_threads()
    # each step: a column sample of the workload, sized so that the warm-up and
    # timed steps together take about 150 s on these cores (at most 1 s a step)
    step_budget = min(1.0, 150.0 / max(1, args.steps + args.warmup))
    cols = 512
    t0 = time.perf_counter()
    oracle.qgemm_fp8_block(p.X, p.W[:cols], p.S[:cols // 128], nthreads=nt)
    dt = time.perf_counter() - t0
    n_s = int(min(N, max(128, (step_budget / max(dt, 1e-6)) * cols)) // 128 * 128)
    for _ in range(args.warmup):
        oracle.qgemm_fp8_block(p.X, p.W[:n_s], p.S[:n_s // 128], nthreads=nt)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.qgemm_fp8_block(p.X, p.W[:n_s], p.S[:n_s // 128], nthreads=nt)
    dt = time.perf_counter() - t0
    per = dt / args.steps
    gbs = fp8_bytes(M, n_s, K) / per / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": head_config(bool(args.overlap), args.gpus),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": nt, "kind": "oracle",
                         "sample": f"columns 0..{n_s - 1} of {N} per step (all {M} rows, full K)"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only, no secondary configs or CPU baseline")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the headline calls and print their line, nothing else (for profiling the kernel)")
    ap.add_argument("--overlap", type=int, choices=[0, 1], default=1,
                    help="launch with weight-prefetch overlap of consecutive calls (default 1)")
    ap.add_argument("--only", choices=["lut3", "fp8_down_m32", "bf16", "fp8_attn_n5120_m16", "w8a8_m256"],
                    default=None,
                    help="time one secondary workload alone and print its line, for profiling its kernel: "
                         "lut3 = 3-bit LUT, M=16, N=28672, K=8192; fp8_down_m32 = FP8 M=32, N=5120, K=17408; "
                         "bf16 = dense BF16, M=16, N=32768, K=5120; fp8_attn_n5120_m16 = FP8 M=16, N=5120, K=5120; "
                         "w8a8_m256 = W8A8 GEMM, M=256, N=17408, K=5120")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from __graft_entry__ import build
    if rank == 0:
        build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    import weight_only_quantized_qgemm_gb300 as qg

    if args.only is not None:
        stream = torch.cuda.Stream()
        qg.set_weight_prefetch_overlap(bool(args.overlap))
        if args.only == "lut3":
            c = Lut3Case(torch, qg, 16, 28672, 8192)
            ms = c.time(16, stream, args.steps, args.warmup)
            nbytes, name = lut3_bytes(16, 28672, 8192), "lut3 M=16 N=28672 K=8192"
        elif args.only == "bf16":
            c = Bf16Case(torch, qg, 16, 32768, 5120)
            ms = c.time(16, stream, args.steps, args.warmup)
            nbytes, name = bf16_bytes(16, 32768, 5120), "bf16 M=16 N=32768 K=5120"
        elif args.only == "w8a8_m256":
            c = W8a8Case(torch, qg, 256, 17408, 5120)
            ms = c.time(256, stream, args.steps, args.warmup)
            tpeak, tkind = fp8_tensor_peak()
            tf = 2.0 * 256 * 17408 * 5120 / (ms * 1e-3) / 1e12
            print(json.dumps({"workload": "w8a8 gate/up M=256 N=17408 K=5120 (GEMM on resident E4M3 codes)",
                              "us_per_call": round(ms * 1e3, 3), "TFLOPs": round(tf, 1),
                              "frac": round(tf / tpeak, 4), "peak": tpeak, "peak_kind": tkind,
                              "steps": args.steps, "warmup": args.warmup}))
            return 0
        elif args.only == "fp8_attn_n5120_m16":
            c = Fp8Case(torch, qg, 16, 5120, 5120, 3)
            ms = c.time(16, stream, args.steps, args.warmup)
            nbytes, name = fp8_bytes(16, 5120, 5120), "fp8_block M=16 N=5120 K=5120"
        else:
            c = Fp8Case(torch, qg, 32, 5120, 17408, 2)
            ms = c.time(32, stream, args.steps, args.warmup)
            nbytes, name = fp8_bytes(32, 5120, 17408), "fp8_block down M=32 N=5120 K=17408"
        peak, peak_kind = measured_peaks()
        gbs = nbytes / (ms * 1e-3) / 1e9
        print(json.dumps({"workload": name, "us_per_call": round(ms * 1e3, 3),
                          "GBps": round(gbs, 1), "frac": round(gbs / peak, 4), "peak": peak,
                          "peak_kind": peak_kind, "steps": args.steps, "warmup": args.warmup}))
        return 0

    M, N, K, cid = HEAD["M"], HEAD["N"], HEAD["K"], HEAD["config_id"]
    stream = torch.cuda.Stream()
    sampler = ClockSampler(gpu_uuid(torch, local))
    # consecutive calls may overlap: a call streams its weights while the one
    # before it finishes (weights are never written by the preceding call)
    qg.set_weight_prefetch_overlap(bool(args.overlap))

    # headline: warm up, then exactly `steps` calls with clocks sampled alongside
    case = Fp8Case(torch, qg, M, N, K, cid)
    step = case.stepper(M, stream)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms_total = e0.elapsed_time(e1)
    st = qg.last_device_status(stream)
    if st:
        raise RuntimeError(f"device status {qg.status_string(st)}")
    ms_total = max_over_ranks(ms_total, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ms = ms_total / args.steps
    per_call_bytes = fp8_bytes(M, N, K)
    value = per_call_bytes * world / (ms * 1e-3) / 1e9
    achieved = per_call_bytes / (ms * 1e-3) / 1e9
    copies = case.copies
    if args.headline_only:
        if rank == 0:
            peak, _ = measured_peaks()
            print(json.dumps({"workload": "fp8_block gate/up M=16 N=17408 K=5120", "us_per_call": round(ms * 1e3, 3),
                              "GBps": round(achieved, 1), "frac": round(achieved / peak, 4), "steps": args.steps,
                              "warmup": args.warmup, "clocks": clocks}))
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    e2e_ms, h2d, d2h, e2e_slots = e2e_fp8(torch, qg, stream, case, M, steps=max(200, min(args.steps, 5000)),
                                          warmup=args.warmup)
    e2e_ms = max_over_ranks(e2e_ms, world)
    # the same calls strictly one after another (no launch overlap): what one
    # call costs on its own
    iso_ms = None
    if args.overlap:
        qg.set_weight_prefetch_overlap(False)
        iso_ms = case.time(M, stream, max(200, min(args.steps, 5000)), args.warmup)
        qg.set_weight_prefetch_overlap(True)
        iso_ms = max_over_ranks(iso_ms, world)
    case.free()
    torch.cuda.empty_cache()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peak, peak_kind = measured_peaks()
    secondary = {}
    cpu = None
    if not args.quick:
        try:
            secondary = secondary_lines(torch, qg, stream, peak)
        except Exception as e:  # secondary numbers must not hide the headline
            secondary["error"] = repr(e)[:300]
        if world == 1:   # the CPU baseline is taken at one GPU only
            cpu, _ = cpu_baseline(M, N, K, cid)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 6),
        "us_per_call": round(ms * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / world / PAGE_BASELINE_GBPS, 3),
        "vs_baseline_ref": "H100 w8a16_gemv_batch16 gate/up M=16, 342 GB/s (atlas m16_tc page, WHY table): context, other hardware",
        "dtype": "bf16",
        "data": "synthetic",
        "config": head_config(bool(args.overlap), world),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "bytes_per_launch": per_call_bytes,
                     "traffic": profiled_traffic("fp8_gateup_m16", per_call_bytes)},
        "isolated": None if iso_ms is None else {
            "us_per_call": round(iso_ms * 1e3, 3), "GBps": round(per_call_bytes / (iso_ms * 1e-3) / 1e9, 2),
            "frac": round(per_call_bytes / (iso_ms * 1e-3) / 1e9 / peak, 4),
            "how": "same workload, calls launched without weight-prefetch overlap (each waits for the one before)"},
        "e2e": {"value": round(per_call_bytes * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(e2e_ms * 1e3, 3),
                "path": "qgemm_fp8_block_host: pinned host X read by a staging kernel, "
                        "Y stored to pinned host memory by the GEMM epilogue (2 kernels per step)",
                "x_buffers": f"{e2e_slots} pinned host X buffers of distinct contents rotated "
                             f"({e2e_slots * h2d / 1e6:.0f} MB > 2x L2)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "secondary": secondary,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
