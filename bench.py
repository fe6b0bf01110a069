"""Benchmark of the Mamba-3 hot path on GB300.

One step = the SISO scan of the packed input projection of a SISO 1B-layer
batch (B=8, L=2048, H=32, P=64, N=128, A=32, G=1; rows 16384 x width 4480):
m3_siso_forward_packed, the preprocess fused into the chunked scan, whose
output has the bits of m3_preprocess followed by m3_siso_forward (that
two-call step is timed beside it), through the C ABI with device-resident
inputs. The metric is tokens/s (B*L per step, summed over ranks). The JSON line also carries the roofline of the dominant kernel, the
CPU oracle baseline, an end-to-end figure with host buffers, sampled clocks,
and supplementary timings of the MIMO and decode-step entry points.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl m3|reference]
                [--mode fp32|tf32] [--no-parts] [--part NAME]
--part NAME runs only one supplementary part (siso_scan_fp32, mimo_scan_fp32,
mimo_scan_tf32, mimo_packed_tf32, siso_long_scan_fp32, siso_long_scan_tf32, siso_step,
mimo_step, siso_prefill_tf32, siso_backward_fp32, siso_long_backward_fp32,
mimo_backward_fp32, preprocess_backward, train_step_fp32) and prints its JSON, for
profiling it alone.
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas, weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_mamba3_gb300 import inputs as gen  # noqa: E402

METRIC = "Mamba-3 scan tokens/s at 1 GB300 (fwd) and % of roofline; step tokens/s"
UNIT = "tokens/s"
W_MAIN = gen.SISO_1B


def bytes_per_token_scan(w):
    """Algorithmic HBM bytes of one token of a scan: x, z, out [H,P]; B, C rows
    [R*G, N]; adt, dt, trap [H]; angle [A] (float32, each read or written once)."""
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    return 4 * (3 * w.num_heads * w.head_dim + 2 * w.mimo_rank * G * w.state_size +
                3 * w.num_heads + w.num_rope_angles)


def bytes_per_token_packed(w):
    """Algorithmic HBM bytes of one token of the packed-projection scan: its
    packed row read once (W floats) and its output row written once (H*P)."""
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    width = gen.packed_width(w.num_heads * w.head_dim, w.state_size, w.num_heads,
                             w.num_rope_angles, G, w.mimo_rank)
    return 4 * (width + w.num_heads * w.head_dim)


def bytes_per_row_preprocess(w):
    """Algorithmic bytes of one preprocess row: the packed row read once and
    the same number of floats written (x, z, bh, ch, dt, adt, trap, angle)."""
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    width = gen.packed_width(w.num_heads * w.head_dim, w.state_size, w.num_heads,
                             w.num_rope_angles, G, w.mimo_rank)
    return 4 * 2 * width


def bytes_per_row_preprocess_backward(w):
    """Algorithmic bytes of one row of the preprocess adjoint: the eight output
    gradients read (W floats in all), the B / C rows and the dt / a columns of
    the packed row read (2 G R N + 2 H floats; the other columns' gradients do
    not depend on the projection), and the projection gradient row written
    (W floats). The dt_bias sums (H floats per row, re-read) are not counted."""
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    width = gen.packed_width(w.num_heads * w.head_dim, w.state_size, w.num_heads,
                             w.num_rope_angles, G, w.mimo_rank)
    return 4 * (2 * width + 2 * G * w.mimo_rank * w.state_size + 2 * w.num_heads)


def bytes_per_step_call(w):
    """Algorithmic bytes of one decode-step call: ssm state read + written,
    k/v/angle states read + written, per-token operands read, out written."""
    B, H, P, N, A = w.batch_size, w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
    G = H if w.num_groups == 0 else w.num_groups
    R = w.mimo_rank
    state = 2 * B * H * (P * N + R * N + R * P + A)
    tok = B * (3 * H * P + 2 * R * G * N + 3 * H + A)
    return 4 * (state + tok)


def bytes_per_token_backward(w):
    """Algorithmic HBM bytes of one token of the SISO backward: the forward
    operands and the output gradient read once (dout, x, z [H,P]; B, C rows
    [G,N]; adt, dt, trap [H]; angle [A]) and their gradients written once
    (dx, dz; dB, dC; d adt, d dt, d trap; d angle)."""
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    H, P, N, A = w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
    return 4 * ((3 * H * P + 2 * G * N + 3 * H + A) + (2 * H * P + 2 * G * N + 3 * H + A))


def flops_per_token_backward(w):
    """FP32 CUDA-core flops of the two sweeps per token: per state element the
    forward sweep's state update (3 FMA), readout (1 FMA) and dq (1 FMA), and
    the reverse sweep's decay (1 MUL), M k, M^T v and adjoint update (3 FMA);
    an FMA is 2 flops: 17 H P N."""
    return 17 * w.num_heads * w.head_dim * w.state_size


def bytes_per_token_backward_mimo(w):
    """Algorithmic HBM bytes of one token of the MIMO backward: dout, x, z
    [H,P]; B, C rows [R*G,N]; adt, dt, trap [H]; angle [A] read once, and the
    gradients of x, z, B, C, adt, dt, trap and angle written once."""
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    H, P, N, A, R = w.num_heads, w.head_dim, w.state_size, w.num_rope_angles, w.mimo_rank
    return 4 * ((3 * H * P + 2 * R * G * N + 3 * H + A) + (2 * H * P + 2 * R * G * N + 3 * H + A))


def flops_per_token_backward_mimo(w):
    """FP32 flops of the MIMO adjoints per token: per state element the state
    update (a decay multiply and 2R FMA), the y and dq readouts (R FMA each)
    and the reverse sweep (a multiply and 3R FMA): (2 + 14 R) H P N. The second
    forward sweep that the output norm's row-wide adjoint requires is not
    counted."""
    return (2 + 14 * w.mimo_rank) * w.num_heads * w.head_dim * w.state_size


def fp32_alu_peak():
    """FP32 CUDA-core peak in TFLOP/s: 152 SMs x 128 FP32 lanes x 2 flops per
    FMA x the maximum SM clock (MEASURED_PEAKS.json's sm_max_mhz, else the
    nominal 2070 MHz)."""
    mhz, how = 2070.0, "nominal 2070 MHz"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        if "sm_max_mhz" in p:
            mhz, how = float(p["sm_max_mhz"]), "measured sm_max_mhz"
    return 152 * 128 * 2 * mhz * 1e6 / 1e12, f"152 SMs x 128 FP32 lanes x 2 x {how}"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tf32_peak():
    """Dense TF32 tensor peak in TFLOP/s: the measured BF16 GEMM peak times the
    nominal TF32 / BF16 ratio (1.1 / 2.25 PFLOP/s), else the fallback's."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        if "bf16_tflops" in p:
            return float(p["bf16_tflops"]) * 1.1 / 2.25, "measured bf16 x nominal 1.1/2.25"
    return 1900.0 * 1.1 / 2.25, "fallback bf16 x nominal 1.1/2.25"


def mma_flops_per_token_chunked(w, q=64):
    """FLOPs the chunked scan's MMAs execute per token (single pass, Q tokens per
    chunk): S = Q K^T and Yo = G Q^T (2 Q N each per token and head), Yi = X P^T
    (2 Q P) and the state update (2 P N), i.e. 2 (Q (N + P) + 2 P N) per head."""
    P, N, H = w.head_dim, w.state_size, w.num_heads
    return 2 * (q * (N + P) + 2 * P * N) * H


# Sources that make up each kernel the bench reports a roofline for (the
# traffic figure of a capture is valid only while all of them are unchanged).
KERNEL_SOURCES = {
    "k_scan_chunk": ["scan_chunk.cuh", "k_scan_chunk_packed.cu", "tc_ptx.cuh", "m3_internal.cuh"],
    "k_preprocess": ["k_preprocess.cu", "m3_internal.cuh"],
    "k_step_bulk": ["k_step.cu", "tc_ptx.cuh", "m3_internal.cuh"],
}


def kernel_source_sha(kernel):
    """sha1[:12] of the concatenated sources of `kernel` (None if unknown)."""
    import hashlib
    files = KERNEL_SOURCES.get(kernel)
    if not files:
        return None
    h = hashlib.sha1()
    for f in files:
        path = os.path.join(ROOT, "selective_state_space_mamba3_gb300", "csrc", f)
        if not os.path.exists(path):
            return None
        h.update(open(path, "rb").read())
    return h.hexdigest()[:12]


def read_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary
    (profiles/traffic.txt: `<kernel> <source sha1> <bytes per launch> <workload>`),
    or None when absent or when the kernel's sources have changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kernel and not line.startswith("#"):
            return float(parts[2]) if sha is not None and sha == parts[1] else None
    return None


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the
    timed region runs. Through NVML (libnvidia-ml, read-only queries, every
    2 ms) when it loads, else through `nvidia-smi -lms 50`; every sample
    carries a host timestamp, and only those taken between mark_begin() and
    mark_end() are reported (the nearest one if the region was shorter than
    the sampling period)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []          # (time, sm MHz, set of reasons)
        self.smax = None
        self.source = None
        self.t0 = self.t1 = None
        self._stop = threading.Event()

    def _nvml(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.gpu).uuid)
        except Exception:
            uuid = None
        ok = False
        if uuid:
            ok = nv.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) == 0
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
            self.smax = float(mx.value)
        getr = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        return nv, h, getr

    def start(self):
        import ctypes
        try:
            nv, h, getr = self._nvml()
            self.source = "nvml"

            def run():
                clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop.is_set():
                    t = time.perf_counter()
                    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                        why = set()
                        if getr(h, ctypes.byref(rs)) == 0:
                            why = {n for b, n in self.BITS.items() if rs.value & b}
                        self.samples.append((t, float(clk.value), why))
                    time.sleep(0.002)
            self.t = threading.Thread(target=run, daemon=True)
            self.t.start()
            return
        except (OSError, AttributeError):
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_first(self, timeout=5.0):
        """Blocks until the first sample arrived (the sampler is running)."""
        end = time.perf_counter() + timeout
        while not self.samples and time.perf_counter() < end:
            time.sleep(0.005)

    def mark_begin(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            f = [x.strip() for x in line.strip().split(",")]
            if len(f) < 9:
                continue
            try:
                sm, self.smax = float(f[1]), float(f[2])
            except ValueError:
                continue
            why = {n for n, v in zip(names, f[5:9]) if v.lower() == "active"}
            self.samples.append((time.perf_counter(), sm, why))

    def stop(self):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"],
                    "samples": 0}
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.t.join(timeout=2)
        return self.summary()

    def summary(self):
        """Median SM clock, max clock and reasons of the samples in the window."""
        got = list(self.samples)
        inside = [x for x in got if self.t0 is not None and self.t0 <= x[0] <= self.t1]
        if not inside and got and self.t0 is not None:
            mid = 0.5 * (self.t0 + self.t1)
            inside = [min(got, key=lambda x: abs(x[0] - mid))]
        sm = [x[1] for x in inside]
        reasons = set().union(*[x[2] for x in inside]) if inside else set()
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": self.smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": self.source,
                "window_ms": round(1e3 * (self.t1 - self.t0), 3) if self.t0 is not None else None}


def dist_setup(args=None):
    """(world size, rank, local rank) from the torchrun environment."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(world, values, device):
    """Maximum over the ranks of each value (timings in ms) by one
    all_reduce(MAX) on `device` ("cuda" under NCCL, "cpu" under gloo); the
    values themselves when there is one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(world, tokens_per_rank, steps, ms):
    """Tokens/s of the whole job: every rank processes `tokens_per_rank` per
    step (replicas), timed as the slowest rank's `ms` for `steps` steps."""
    return world * tokens_per_rank * steps / (ms * 1e-3)


# --------------------------------------------------------------------- m3 arm

class Step:
    """Device buffers and the two calls of one step (preprocess + SISO scan)."""

    def __init__(self, w, mode):
        import torch
        import selective_state_space_mamba3_gb300 as m3
        self.m3, self.torch, self.w = m3, torch, w
        B, L, H, P, N, A = w.batch_size, w.sequence_length, w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
        G = H if w.num_groups == 0 else w.num_groups
        self.rows = B * L
        proj = gen.layer_projection(w)
        par = gen.scan_params(w)
        self.h_proj = torch.from_numpy(proj["projected"]).pin_memory()
        self.proj = self.h_proj.cuda()
        self.dt_bias = torch.from_numpy(proj["dt_bias"]).cuda()
        self.pcfg = m3.preprocess_config(inner_size=H * P, state_size=N, num_heads=H,
                                         num_rope_angles=A, num_groups=G, mimo_rank=1,
                                         **gen.PRE_DEFAULT)
        e = lambda *s: torch.empty(*s, device="cuda")
        self.x, self.z = e(B, L, H, P), e(B, L, H, P)
        self.bh, self.ch = e(B, L, G, N), e(B, L, G, N)
        self.dt, self.adt, self.trap = e(B, L, H), e(B, L, H), e(B, L, H)
        self.angle = e(B, L, A)
        self.out = e(B, L, H, P)
        self.h_out = torch.empty(B, L, H, P).pin_memory()
        self.cb, self.bb, self.d = (torch.from_numpy(par[k]).cuda() for k in ("c_bias", "b_bias", "d"))
        self.scfg = m3.ssm_config(w.cfg(), mode)
        wsb = m3.m3_siso_forward_workspace(self.scfg)
        self.ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
        wpb = m3.m3_siso_forward_packed_workspace(self.scfg, self.pcfg)
        self.ws_packed = torch.empty(max(wpb, 16), dtype=torch.uint8, device="cuda")

    def packed(self):
        """One step through the fused entry point (packed projection -> out)."""
        self.m3.m3_siso_forward_packed(self.scfg, self.pcfg, self.proj, self.dt_bias, self.cb,
                                       self.bb, self.d, self.out, self.ws_packed)

    def preprocess(self):
        self.m3.m3_preprocess(self.pcfg, self.rows, self.proj, self.dt_bias, self.x, self.z,
                              self.bh, self.ch, self.dt, self.adt, self.trap, self.angle)

    def scan(self, out=None):
        self.m3.m3_siso_forward(self.scfg, self.ch, self.bh, self.x, self.z, self.adt, self.dt,
                                self.trap, self.angle, self.cb, self.bb, self.d,
                                self.out if out is None else out, self.ws)

    def preprocess_rows(self, proj, r0, r1):
        """m3_preprocess of packed rows [r0, r1) of `proj` into the same rows of
        the scan operands (every operand is row-major over the B*L rows)."""
        flat = lambda t: t.view(self.rows, -1)[r0:r1]
        self.m3.m3_preprocess(self.pcfg, r1 - r0, proj[r0:r1], self.dt_bias, flat(self.x),
                              flat(self.z), flat(self.bh), flat(self.ch), flat(self.dt),
                              flat(self.adt), flat(self.trap), flat(self.angle))

    def e2e(self, steps, slices):
        """`steps` end-to-end steps through the public API with host buffers:
        each step copies its packed projection from pinned host memory in
        `slices` row slices on an input copy stream, preprocesses each slice on
        the compute stream as it lands, scans the whole batch, and copies the
        output back to pinned host memory on an output copy stream. Two device
        projection and output buffers let one step's copies overlap the
        neighbouring steps' compute. Returns the average ms per step (CUDA
        events, all three streams joined)."""
        torch = self.torch
        if not hasattr(self, "proj2"):
            self.proj2 = [self.proj, torch.empty_like(self.proj)]
            self.out2 = [self.out, torch.empty_like(self.out)]
            self.streams = [torch.cuda.Stream() for _ in range(3)]
        s_in, s_comp, s_out = self.streams
        bounds = [self.rows * k // slices for k in range(slices + 1)]
        ev = lambda: torch.cuda.Event()
        cur = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur.synchronize()
        e0.record(cur)
        for st in self.streams:
            st.wait_event(e0)
        pre_done, d2h_done = {}, {}
        for i in range(steps):
            buf = i % 2
            proj, out = self.proj2[buf], self.out2[buf]
            landed = []
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(pre_done[i - 2])
                for k in range(slices):
                    r0, r1 = bounds[k], bounds[k + 1]
                    proj[r0:r1].copy_(self.h_proj[r0:r1], non_blocking=True)
                    landed.append(ev())
                    landed[-1].record(s_in)
            with torch.cuda.stream(s_comp):
                for k in range(slices):
                    s_comp.wait_event(landed[k])
                    self.preprocess_rows(proj, bounds[k], bounds[k + 1])
                pre_done[i] = ev()
                pre_done[i].record(s_comp)
                if i >= 2:
                    s_comp.wait_event(d2h_done[i - 2])
                self.scan(out)
                done = ev()
                done.record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                self.h_out.copy_(out, non_blocking=True)
                d2h_done[i] = ev()
                d2h_done[i].record(s_out)
        for st in self.streams:
            cur.wait_stream(st)
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps


def time_events(torch, fn, reps):
    """Average device time (ms) of fn() over reps launches, CUDA events on the
    current stream."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record()
    for _ in range(reps):
        fn()
    ev[1].record()
    torch.cuda.synchronize()
    return ev[0].elapsed_time(ev[1]) / reps


def parts_scan(torch, m3, w, mode, peak):
    """Supplementary: one forward of workload w (device inputs): the MIMO R4
    forward at B4 L4096 H32 P64 N64, the long-context SISO forward at B2
    L16384 H32 G4 P64 N128 A64. Both workloads are stated FP32-exact; TF32 is
    reported beside it."""
    mimo = w.mimo_rank > 1
    ins = gen.scan_inputs(w)
    d = {k: torch.from_numpy(v).cuda() for k, v in ins.items()}
    del ins
    cfg = m3.ssm_config(w.cfg(), mode)
    nws = m3.m3_mimo_forward_workspace(cfg) if mimo else m3.m3_siso_forward_workspace(cfg)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["x"])
    keys = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
    if mimo:
        keys += ("mimo_x", "mimo_z", "mimo_o", "norm_weight")
        fn = lambda: m3.m3_mimo_forward(cfg, *[d[k] for k in keys], out, ws)
    else:
        fn = lambda: m3.m3_siso_forward(cfg, *[d[k] for k in keys], out, ws)
    for _ in range(3):
        fn()
    ms = time_events(torch, fn, 10)
    gbs = w.tokens * bytes_per_token_scan(w) / (ms * 1e-3) / 1e9
    return {"workload": w.name, "mode": "tf32" if mode == m3.M3_MATH_TF32 else "fp32",
            "ms": round(ms, 4), "tokens_per_s": round(w.tokens / (ms * 1e-3)),
            "hbm_gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 4)}


def parts_step(torch, m3, peak, mimo=False):
    """Supplementary: decode step at B256 H32 P64 N128 A32 (SISO), or the MIMO
    step at B256 H32 P64 N64 A32 R4 with the output norm, 512 single-token
    calls cycling over 32 distinct token inputs, states resident on the device."""
    w = gen.DECODE_STEP
    if mimo:
        w = w.with_(name="MIMO decode step B256 H32 G1 P64 N64 A32 R4 norm x512", state_size=64,
                    mimo_rank=4, has_output_norm=1)
    ins = gen.decode_inputs(w, steps=32)
    seq = {k: torch.from_numpy(ins[k]).cuda() for k in ("c", "b", "x", "z", "adt", "dt", "trap", "angle")}
    toks = [[seq[k][:, t:t + 1].contiguous() for k in ("c", "b", "x", "z", "adt", "dt", "trap", "angle")]
            for t in range(32)]
    pkeys = ("c_bias", "b_bias", "d") + (("mimo_x", "mimo_z", "mimo_o", "norm_weight") if mimo else ())
    par = [torch.from_numpy(ins[k]).cuda() for k in pkeys]
    B, H, P, N, A, R = (w.batch_size, w.num_heads, w.head_dim, w.state_size, w.num_rope_angles,
                        w.mimo_rank)
    st = [torch.zeros(s, device="cuda") for s in ((B, H, P, N), (B, H, A), (B, H, R, N),
                                                  (B, H, R, P))]
    out = torch.empty(B, 1, H, P, device="cuda")
    cfg = m3.ssm_config(w.cfg(sequence_length=1))
    step = m3.m3_mimo_step if mimo else m3.m3_siso_step
    i = [0]

    def fn():
        step(cfg, *toks[i[0] % 32], *par, *st, out)
        i[0] += 1
    for _ in range(5):
        fn()
    ms = time_events(torch, fn, w.steps)
    gbs = bytes_per_step_call(w) / (ms * 1e-3) / 1e9
    return {"workload": w.name, "ms_per_call": round(ms, 4),
            "tokens_per_s": round(B / (ms * 1e-3)), "hbm_gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 4)}


def parts_prefill(torch, m3, w, peak):
    """Supplementary: m3_siso_prefill over the 1B-layer workload in TF32 mode,
    from a zero step state, writing the final ssm / angle / k / v states (the
    prefill -> decode hand-off). Algorithmic bytes: the scan's, plus the four
    states written once (and read once as the entry state)."""
    ins = gen.scan_inputs(w)
    d = {k: torch.from_numpy(v).cuda() for k, v in ins.items()}
    del ins
    B, H, P, N, A = w.batch_size, w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
    cfg = m3.ssm_config(w.cfg(), m3.M3_MATH_TF32)
    ws = torch.empty(max(m3.m3_siso_prefill_workspace(cfg), 16), dtype=torch.uint8, device="cuda")
    st = [torch.zeros(s, device="cuda") for s in ((B, H, P, N), (B, H, A), (B, H, N), (B, H, P))]
    out = torch.empty_like(d["x"])
    keys = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
    fn = lambda: m3.m3_siso_prefill(cfg, *[d[k] for k in keys], *st, out, ws)
    for _ in range(3):
        fn()
    ms = time_events(torch, fn, 10)
    nbytes = w.tokens * bytes_per_token_scan(w) + 2 * 4 * B * H * (P * N + A + N + P)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name + " prefill", "mode": "tf32", "ms": round(ms, 4),
            "tokens_per_s": round(w.tokens / (ms * 1e-3)), "hbm_gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 4), "algorithmic_bytes": nbytes}


def parts_packed_mimo(torch, m3, w, mode, peak):
    """Supplementary: m3_mimo_forward_packed over the MIMO R4 workload (B4 L4096
    H32 P64 N64 A32 R4 with the output norm): packed projection rows in, output
    out (the preprocess kernel into the workspace, then the MIMO scan).
    Algorithmic bytes: each packed row read once, the output written once."""
    H, P, N, A = w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
    G = H if w.num_groups == 0 else w.num_groups
    proj = gen.layer_projection(w)
    par = gen.scan_params(w)
    dp = torch.from_numpy(proj["projected"]).cuda()
    db = torch.from_numpy(proj["dt_bias"]).cuda()
    keys = ("c_bias", "b_bias", "d", "mimo_x", "mimo_z", "mimo_o", "norm_weight")
    pv = [torch.from_numpy(par[k]).cuda() for k in keys]
    del proj
    cfg = m3.ssm_config(w.cfg(), mode)
    pcfg = m3.preprocess_config(inner_size=H * P, state_size=N, num_heads=H, num_rope_angles=A,
                                num_groups=G, mimo_rank=w.mimo_rank, **gen.PRE_DEFAULT)
    nws = m3.m3_mimo_forward_packed_workspace(cfg, pcfg)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty(w.batch_size, w.sequence_length, H, P, device="cuda")
    fn = lambda: m3.m3_mimo_forward_packed(cfg, pcfg, dp, db, *pv, out, ws)
    for _ in range(3):
        fn()
    ms = time_events(torch, fn, 10)
    nbytes = w.tokens * bytes_per_token_packed(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name + " packed", "mode": "tf32" if mode == m3.M3_MATH_TF32 else "fp32",
            "entry": "m3_mimo_forward_packed", "ms": round(ms, 4),
            "tokens_per_s": round(w.tokens / (ms * 1e-3)), "hbm_gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 4), "algorithmic_bytes": nbytes}


def cpu_baseline_oracle(w, batch_rows):
    """The CPU oracle (as it stands) on a bounded sample of the workload: the
    first `batch_rows` batch rows, preprocess + SISO scan, all host threads."""
    import oracle
    oracle.build()
    H, P, N, A = w.num_heads, w.head_dim, w.state_size, w.num_rope_angles
    G = H if w.num_groups == 0 else w.num_groups
    L = w.sequence_length
    proj = gen.layer_projection(w)
    par = gen.scan_params(w)
    rows = batch_rows * L
    kw = dict(inner_size=H * P, state_size=N, num_heads=H, num_rope_angles=A, num_groups=G,
              mimo_rank=1, **gen.PRE_DEFAULT)
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    pre = oracle.preprocess(proj["projected"][:rows], proj["dt_bias"], **kw)
    f = lambda k, *s: pre[k].astype(np.float32).reshape(batch_rows, L, *s)
    oracle.scan(w.cfg(batch_size=batch_rows), f("ch", G, N), f("bh", G, N), f("x", H, P),
                f("z", H, P), f("adt", H), f("dt", H), f("trap", H), f("angle", A),
                par["c_bias"], par["b_bias"], par["d"])
    dt = time.perf_counter() - t0
    return {"value": round(rows / dt, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"batch rows 0..{batch_rows - 1} of {w.batch_size} ({rows} of {w.tokens} "
                      f"tokens), preprocess + SISO scan, FP64, {threads} threads, {dt:.2f} s",
            "seconds": round(dt, 3)}


def parts_backward(torch, m3, w, peak):
    """Supplementary: m3_siso_backward (the eleven SISO adjoints, FP32) of
    workload w with device-resident operands and output gradient. Bound: the
    FP32 CUDA-core rate of the two token-sequential sweeps (alu), with the HBM
    fraction beside it."""
    ins = gen.scan_inputs(w)
    d = {k: torch.from_numpy(v).cuda() for k, v in ins.items()}
    go = torch.from_numpy(gen.output_gradient(w)).cuda()
    del ins
    cfg = m3.ssm_config(w.cfg(), m3.M3_MATH_FP32)
    ws = torch.empty(m3.m3_siso_backward_workspace(cfg), dtype=torch.uint8, device="cuda")
    keys = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d")
    g = {k: torch.empty_like(d[k]) for k in keys}
    fn = lambda: m3.m3_siso_backward(cfg, go, *[d[k] for k in keys], *[g[k] for k in keys], ws)
    for _ in range(3):
        fn()
    ms = time_events(torch, fn, 5)
    gbs = w.tokens * bytes_per_token_backward(w) / (ms * 1e-3) / 1e9
    tflops = w.tokens * flops_per_token_backward(w) / (ms * 1e-3) / 1e12
    alu, how = fp32_alu_peak()
    return {"workload": w.name, "mode": "fp32", "ms": round(ms, 4),
            "tokens_per_s": round(w.tokens / (ms * 1e-3)), "hbm_gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 4), "alu_tflops": round(tflops, 2),
            "alu_peak_tflops": round(alu, 1), "alu_peak": how, "frac_alu": round(tflops / alu, 4),
            "algorithmic_bytes": w.tokens * bytes_per_token_backward(w),
            "flops": w.tokens * flops_per_token_backward(w)}


def parts_backward_mimo(torch, m3, w, peak):
    """Supplementary: m3_mimo_backward (the fifteen MIMO adjoints, FP32) of
    workload w with device-resident operands and output gradient."""
    ins = gen.scan_inputs(w)
    d = {k: torch.from_numpy(v).cuda() for k, v in ins.items()}
    go = torch.from_numpy(gen.output_gradient(w)).cuda()
    del ins
    cfg = m3.ssm_config(w.cfg(), m3.M3_MATH_FP32)
    ws = torch.empty(m3.m3_mimo_backward_workspace(cfg), dtype=torch.uint8, device="cuda")
    keys = ("c", "b", "x", "z", "adt", "dt", "trap", "angle", "c_bias", "b_bias", "d", "mimo_x",
            "mimo_z", "mimo_o", "norm_weight")
    g = {k: torch.empty_like(d[k]) for k in keys}
    fn = lambda: m3.m3_mimo_backward(cfg, go, *[d[k] for k in keys], *[g[k] for k in keys], ws)
    for _ in range(3):
        fn()
    ms = time_events(torch, fn, 5)
    gbs = w.tokens * bytes_per_token_backward_mimo(w) / (ms * 1e-3) / 1e9
    tflops = w.tokens * flops_per_token_backward_mimo(w) / (ms * 1e-3) / 1e12
    alu, how = fp32_alu_peak()
    return {"workload": w.name, "mode": "fp32", "ms": round(ms, 4),
            "tokens_per_s": round(w.tokens / (ms * 1e-3)), "hbm_gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 4), "alu_tflops": round(tflops, 2),
            "alu_peak_tflops": round(alu, 1), "alu_peak": how, "frac_alu": round(tflops / alu, 4),
            "algorithmic_bytes": w.tokens * bytes_per_token_backward_mimo(w),
            "flops": w.tokens * flops_per_token_backward_mimo(w)}


def parts_preprocess_backward(torch, m3, w, peak):
    """Supplementary: m3_preprocess_backward (the adjoint of the projection
    preprocess: the packed projection and dt_bias gradients) at workload w's
    layer shape, device-resident inputs; HBM-bound streaming."""
    p = gen.layer_projection(w)
    G = w.num_heads if w.num_groups == 0 else w.num_groups
    kw = dict(inner_size=w.num_heads * w.head_dim, state_size=w.state_size,
              num_heads=w.num_heads, num_rope_angles=w.num_rope_angles, num_groups=G,
              mimo_rank=w.mimo_rank, **gen.PRE_DEFAULT)
    rows = p["projected"].shape[0]
    I, bc, H, A = kw["inner_size"], G * w.mimo_rank * w.state_size, w.num_heads, w.num_rope_angles
    shapes = dict(x=(rows, I), z=(rows, I), bh=(rows, bc), ch=(rows, bc), dt=(rows, H),
                  adt=(rows, H), trap=(rows, H), angle=(rows, A))
    gr = {k: torch.from_numpy(v).cuda() for k, v in gen.preprocess_output_gradient(w, shapes).items()}
    proj = torch.from_numpy(p["projected"]).cuda()
    dtb = torch.from_numpy(p["dt_bias"]).cuda()
    del p
    cfg = m3.preprocess_config(**kw)
    gp = torch.empty_like(proj)
    gb = torch.empty_like(dtb)
    ws = torch.empty(max(m3.m3_preprocess_backward_workspace(cfg, rows), 16), dtype=torch.uint8,
                     device="cuda")
    fn = lambda: m3.m3_preprocess_backward(cfg, rows, proj, dtb, *[gr[k] for k in gen.PRE_OUTPUTS],
                                           gp, gb, ws)
    for _ in range(3):
        fn()
    ms = time_events(torch, fn, 5)
    nbytes = rows * bytes_per_row_preprocess_backward(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name + " (layer rows)", "rows": rows, "ms": round(ms, 4),
            "hbm_gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 4), "algorithmic_bytes": nbytes}


def parts_train_step(torch, m3, w, peak):
    """Supplementary: one training step of the layer's scan through the
    torch.autograd binding (selective_state_space_mamba3_gb300.autograd): the
    packed projection -> m3_preprocess -> m3_siso_forward (FP32-exact) -> loss
    sum(out * W) -> m3_siso_backward -> m3_preprocess_backward, i.e. the
    projection and dt_bias gradients (and those of c_bias, b_bias, D).
    Device-resident inputs; the torch elementwise ops of the loss run beside."""
    from selective_state_space_mamba3_gb300 import autograd as m3ag
    p = gen.layer_projection(w)
    sp = gen.scan_params(w)
    B, L, H, P, N, A = (w.batch_size, w.sequence_length, w.num_heads, w.head_dim, w.state_size,
                        w.num_rope_angles)
    G = H if w.num_groups == 0 else w.num_groups
    pkw = dict(inner_size=H * P, state_size=N, num_heads=H, num_rope_angles=A, num_groups=G,
               mimo_rank=1, **gen.PRE_DEFAULT)
    proj = torch.from_numpy(p["projected"]).cuda().requires_grad_(True)
    dtb = torch.from_numpy(p["dt_bias"]).cuda().requires_grad_(True)
    par = {k: torch.from_numpy(sp[k]).cuda().requires_grad_(True) for k in ("c_bias", "b_bias", "d")}
    wgt = torch.from_numpy(gen.output_gradient(w)).cuda()
    cfg = w.cfg()

    def step():
        x, z, bh, ch, dt, adt, trap, ang = m3ag.preprocess(pkw, proj, dtb)
        out = m3ag.siso_scan(cfg, ch.view(B, L, G, N), bh.view(B, L, G, N), x.view(B, L, H, P),
                             z.view(B, L, H, P), adt.view(B, L, H), dt.view(B, L, H),
                             trap.view(B, L, H), ang.view(B, L, A), par["c_bias"], par["b_bias"],
                             par["d"])
        (out * wgt).sum().backward()
        proj.grad = None
        dtb.grad = None
        for v in par.values():
            v.grad = None
    for _ in range(3):
        step()
    ms = time_events(torch, step, 5)
    return {"workload": w.name, "mode": "fp32", "ms": round(ms, 4),
            "tokens_per_s": round(w.tokens / (ms * 1e-3)),
            "entry": "autograd: m3_preprocess, m3_siso_forward, m3_siso_backward, "
                     "m3_preprocess_backward"}


def part_by_name(torch, m3, name, peak):
    """One supplementary part, by its key in the JSON line's `parts`."""
    table = {
        "siso_scan_fp32": lambda: parts_scan(torch, m3, gen.SISO_1B, m3.M3_MATH_FP32, peak),
        "mimo_scan_fp32": lambda: parts_scan(torch, m3, gen.MIMO_R4, m3.M3_MATH_FP32, peak),
        "mimo_scan_tf32": lambda: parts_scan(torch, m3, gen.MIMO_R4, m3.M3_MATH_TF32, peak),
        "mimo_packed_tf32": lambda: parts_packed_mimo(torch, m3, gen.MIMO_R4, m3.M3_MATH_TF32, peak),
        "siso_long_scan_fp32": lambda: parts_scan(torch, m3, gen.SISO_LONG, m3.M3_MATH_FP32, peak),
        "siso_long_scan_tf32": lambda: parts_scan(torch, m3, gen.SISO_LONG, m3.M3_MATH_TF32, peak),
        "siso_step": lambda: parts_step(torch, m3, peak),
        "mimo_step": lambda: parts_step(torch, m3, peak, mimo=True),
        "siso_prefill_tf32": lambda: parts_prefill(torch, m3, gen.SISO_1B, peak),
        "siso_backward_fp32": lambda: parts_backward(torch, m3, gen.SISO_1B, peak),
        "siso_long_backward_fp32": lambda: parts_backward(torch, m3, gen.SISO_LONG, peak),
        "mimo_backward_fp32": lambda: parts_backward_mimo(torch, m3, gen.MIMO_R4, peak),
        "preprocess_backward": lambda: parts_preprocess_backward(torch, m3, gen.SISO_1B, peak),
        "train_step_fp32": lambda: parts_train_step(torch, m3, gen.SISO_1B, peak),
    }
    if name not in table:
        raise SystemExit(f"bench.py: unknown part {name!r}; one of {sorted(table)}")
    return table[name]()


def run_part(args):
    """--part NAME: one supplementary part alone (for profiling it)."""
    import torch
    import selective_state_space_mamba3_gb300 as m3
    from selective_state_space_mamba3_gb300 import build as m3build
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    m3build.build()
    m3.load_library()
    peak, _ = load_peaks()
    print(json.dumps({"part": args.part, **part_by_name(torch, m3, args.part, peak)}), flush=True)


def run_m3(args):
    import torch
    import selective_state_space_mamba3_gb300 as m3
    from selective_state_space_mamba3_gb300 import build as m3build
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    m3build.build()
    m3.load_library()
    mode = m3.M3_MATH_TF32 if args.mode == "tf32" else m3.M3_MATH_FP32
    peak, peak_kind = load_peaks()
    w = W_MAIN
    s = Step(w, mode)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        s.packed()
        s.preprocess()
        s.scan()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_first()
    barrier()
    torch.cuda.synchronize()
    n0 = m3.launch_count()
    clocks.mark_begin()
    t_start.record()
    for k in range(K):
        ev[k][0].record()
        s.packed()
        ev[k][1].record()
    t_end.record()
    torch.cuda.synchronize()
    clocks.mark_end()
    launches = m3.launch_count() - n0
    barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(world, [t_start.elapsed_time(t_end)], "cuda")[0]
    fused_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    assert m3.m3_workspace_status(s.ws_packed) == m3.M3_OK
    tokens = w.tokens
    value = whole_job_rate(world, tokens, K, total_ms)

    # the two-call step (preprocess, then scan) and its parts, same workload
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    torch.cuda.synchronize()
    for k in range(K):
        ev2[k][0].record()
        s.preprocess()
        ev2[k][1].record()
        s.scan()
        ev2[k][2].record()
    torch.cuda.synchronize()
    pre_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev2]))
    scan_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev2]))
    assert m3.m3_workspace_status(s.ws) == m3.M3_OK

    # roofline of the dominant kernel (algorithmic bytes / live event time):
    # the fused scan (the packed rows read once, the output written once:
    # 4 (W + H P) bytes per token), timed with the short row-norm pass that
    # precedes it in the same call, so the fraction is a lower bound
    scan_bytes = tokens * bytes_per_token_scan(w)
    pre_bytes = s.rows * bytes_per_row_preprocess(w)
    fused_bytes = tokens * bytes_per_token_packed(w)
    kname, kms, kbytes = "k_scan_chunk", fused_ms, fused_bytes
    achieved = kbytes / (kms * 1e-3) / 1e9
    roof = {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
            "algorithmic_bytes": kbytes, "ms": round(kms, 4),
            "timed_with": "k_row_pre (the packed step's row pass, same call)",
            "traffic": read_traffic(kname)}
    # the other roofline term: the MMA flops the kernel executes against the
    # TF32 tensor peak (the larger of the two terms' times is the bound)
    tpeak, tkind = tf32_peak()
    mma_flops = tokens * mma_flops_per_token_chunked(w)
    roof["hbm_us_at_peak"] = round(kbytes / (peak * 1e9) * 1e6, 1)
    roof["tensor_term"] = {"executed_mma_flops": mma_flops, "peak_tflops": round(tpeak, 1),
                           "peak_kind": tkind,
                           "us_at_peak": round(mma_flops / (tpeak * 1e12) * 1e6, 1),
                           "achieved_tflops": round(mma_flops / (kms * 1e-3) / 1e12, 1),
                           "frac": round(mma_flops / (kms * 1e-3) / (tpeak * 1e12), 4)}

    # end to end through the public API with host buffers (pinned), rank-local:
    # every step copies its inputs in and its output out; copies and compute of
    # neighbouring steps overlap on three streams
    KE = max(3, min(K, 10))
    s.e2e(2, 8)
    barrier()
    e2e_ms = max_over_ranks(world, [s.e2e(KE, 8)], "cuda")[0]
    e2e = {"value": round(whole_job_rate(world, tokens, 1, e2e_ms), 1), "unit": UNIT,
           "h2d_bytes_per_step": s.h_proj.numel() * 4, "d2h_bytes_per_step": s.h_out.numel() * 4,
           "ms_per_step": round(e2e_ms, 4)}

    parts = {"fused_step": {"ms": round(fused_ms, 4), "tokens_per_s": round(tokens / (fused_ms * 1e-3)),
                            "hbm_gbs": round(achieved, 1), "frac_hbm": round(achieved / peak, 4),
                            "algorithmic_bytes": fused_bytes,
                            "entry": "m3_siso_forward_packed"},
             "two_call_step": {"ms": round(pre_ms + scan_ms, 4),
                               "tokens_per_s": round(tokens / ((pre_ms + scan_ms) * 1e-3)),
                               "entry": "m3_preprocess + m3_siso_forward"},
             "preprocess": {"ms": round(pre_ms, 4), "hbm_gbs": round(pre_bytes / (pre_ms * 1e-3) / 1e9, 1),
                            "frac_hbm": round(pre_bytes / (pre_ms * 1e-3) / 1e9 / peak, 4),
                            "algorithmic_bytes": pre_bytes},
             "siso_scan": {"ms": round(scan_ms, 4), "tokens_per_s": round(tokens / (scan_ms * 1e-3)),
                           "hbm_gbs": round(scan_bytes / (scan_ms * 1e-3) / 1e9, 1),
                           "frac_hbm": round(scan_bytes / (scan_ms * 1e-3) / 1e9 / peak, 4),
                           "algorithmic_bytes": scan_bytes}}
    del s
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_parts:
        for name in ("siso_scan_fp32", "mimo_scan_fp32", "mimo_scan_tf32", "mimo_packed_tf32",
                     "siso_long_scan_fp32",
                     "siso_long_scan_tf32", "siso_step", "mimo_step", "siso_prefill_tf32",
                     "siso_backward_fp32", "siso_long_backward_fp32", "mimo_backward_fp32",
                     "preprocess_backward", "train_step_fp32"):
            parts[name] = part_by_name(torch, m3, name, peak)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_oracle(w, args.cpu_rows)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
                "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "tf32" if mode == m3.M3_MATH_TF32 else "f32", "data": "synthetic",
                "config": {"workload": w.name, "batch": w.batch_size, "seq_len": w.sequence_length,
                           "heads": w.num_heads, "head_dim": w.head_dim, "state_size": w.state_size,
                           "groups": w.num_groups, "rope_angles": w.num_rope_angles,
                           "step": "m3_siso_forward_packed: 16384 x 4480 packed rows -> out "
                                   "(preprocess fused into the scan)",
                           "math_mode": args.mode, "parallelism": f"replicas x{world}",
                           "l2": "inputs larger than L2 (293.6 MB packed projection read per step)"},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
                "clocks": clk, "parts": parts}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# -------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as it stands, on the host cores, on the same workload's
    configuration: each step is a bounded sample (one batch row: preprocess of
    its 2048 packed rows + the SISO scan over them)."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    w = W_MAIN
    for _ in range(args.warmup):
        cpu_baseline_oracle(w, 1)
    times = []
    for _ in range(args.steps):
        r = cpu_baseline_oracle(w, 1)
        times.append(r["seconds"])
    tot = float(np.sum(times))
    tokens = w.sequence_length * args.steps
    value = tokens / tot
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch_size, "seq_len": w.sequence_length,
                       "heads": w.num_heads, "head_dim": w.head_dim, "state_size": w.state_size,
                       "groups": w.num_groups, "rope_angles": w.num_rope_angles,
                       "step": "oracle preprocess + SISO scan of one batch row (2048 tokens)"},
            "cpu_baseline": {"kind": "oracle", "cores": r["cores"], "sample": r["sample"],
                             "value": round(value, 1), "unit": UNIT},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def relaunch_under_torchrun(n):
    """`--gpus N` with N > 1 outside torchrun: run this same command as N
    ranks under torch.distributed.run (one process per GPU) and return its
    exit status, so that the job never silently runs on one rank."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="m3", choices=["m3", "reference"])
    ap.add_argument("--mode", default="tf32", choices=["fp32", "tf32"])
    ap.add_argument("--no-parts", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=8)
    ap.add_argument("--part", default=None)
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(relaunch_under_torchrun(args.gpus))
    if world != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {world}")
    if args.warmup < 3 and args.impl == "m3":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.part:
        run_part(args)
    else:
        run_m3(args)


if __name__ == "__main__":
    main()
