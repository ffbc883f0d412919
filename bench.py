"""Benchmark of the selective-scan hot path on B300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill scan, Mamba-130M-shaped layer: (batch 8, dim 1536, L 2048, N 16), bf16
    u/delta/z/B/C, fp32 A/D/bias/state, softplus + silu(z) gate, y bf16;
  * d_state = 1 scalar scan (SM1): (8, 1536, 2048, 1), fp32, h0 ~ N(0,1);
  * one decode token on the resident (256, 5120, 16) fp32 state (the token sets
    rotate through 16 seeded sets; the state carries across steps, so K timed
    steps are K consecutive decode tokens).
Metric: Gtoken*channel/s over the whole step (sum of batch*dim*L over the three
parts / step time), with per-part HBM GB/s and roofline fractions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0). Under torchrun each rank runs the same per-GPU
workload on its own GPU (independent problems, no collective in the data path:
weak scaling); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "selective-scan Gtoken·channel/s and achieved HBM GB/s vs B300 peak (prefill+decode)"
UNIT = "Gtoken*channel/s"
WORKLOAD = "mamba130m_layer_step"
N_SM = 148
SM_MAX_MHZ_NOMINAL = 2032.0
FP32_LANES_PER_CLK_SM = 128       # FMA pipe
SFU_EX2_PER_CLK_SM = 32           # ex2 lanes per clock per SM, measured on B300


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL)), "measured"
    return 6400.0, SM_MAX_MHZ_NOMINAL, "fallback"


def _bf16_peak():
    """Measured dense bf16 tensor TFLOP/s (burst), else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1800.0


# ------------------------------------------------------------------------------------------
# workload accounting (algorithmic bytes and work per launch)
# ------------------------------------------------------------------------------------------
def scan_bytes(bt, dim, L, N, ei, eo, has_z, has_h0):
    """Bytes a scan must move at least once: u, delta (, z) in, y out, B and C once per
    batch row, h_last out (and h0 in), A/D/bias."""
    x = bt * dim * L
    return (x * ((3 if has_z else 2) * ei + eo) + 2 * bt * N * L * ei + bt * dim * N * 4 * (2 if has_h0 else 1)
            + dim * (N + 2) * 4)


def decode_bytes(bt, dim, N, ei, eo):
    """State read + write, x/delta/z in, y out, B and C, A/D/bias."""
    return bt * dim * N * 4 * 2 + bt * dim * (3 * ei + eo) + 2 * bt * N * ei + dim * (N + 2) * 4


def conv_bytes(bt, dim, L, width, ei, eo):
    """Causal conv1d: x in and u out once, the conv state in and out, weights and bias."""
    return bt * dim * L * (ei + eo) + 2 * bt * dim * (width - 1) * 4 + dim * (width + 1) * 4


def conv_update_bytes(bt, dim, width, ei, eo):
    """Conv decode update: x in, u out, the state read and written, weights and bias."""
    return bt * dim * (ei + eo + 2 * (width - 1) * 4) + dim * (width + 1) * 4


def ssd_bytes(bt, L, H, P, G, N, eo, has_z, has_h0):
    """Mamba-2 SSD scan: x (, z) in and y out once, dt, B and C once, h_last out (and
    h0 in), A/D/dt_bias."""
    x = bt * L * H * P
    return (x * ((2 if has_z else 1) * 2 + eo) + bt * L * H * 2 + 2 * bt * L * G * N * 2
            + bt * H * P * N * 4 * (2 if has_h0 else 1) + 3 * H * 4)


def ssd_tensor_flops(bt, L, H, P, N, Q=128):
    """Tensor-core FLOPs the SSD kernel issues per launch: per (b, h, chunk of Q) the
    products C B^T (Q x Q x N), the masked matrix times x (Q x P x Q, high and low
    parts), C times the state (Q x P x N, two parts) and the state update (N x P x Q,
    two parts, M padded to 128 rows when N = 64)."""
    chunks = bt * H * ((L + Q - 1) // Q)
    per = 2 * Q * Q * N + 2 * (2 * Q * P * Q) + 2 * (2 * Q * P * N) + 2 * (2 * 128 * P * Q)
    return chunks * per


SFU_HALF_RATE_SLOTS = 2           # lg2 and rcp issue at half the ex2 rate (16/clk/SM measured)


def alu_roof_seconds(elements, tokch, has_z, mhz):
    """Time the SFU and FP32 pipes need at the given clock (the larger of the two):
    per (t, n) element one ex2 and 4 FP32 FMA-pipe ops; per (b, d, t) softplus = ex2 + lg2
    and silu = ex2 + rcp (lg2/rcp at half rate, 2 slots each) and ~10 FP32 ops of the
    fused prologue/epilogue."""
    f = mhz * 1e6 * N_SM
    per_tok = (1 + SFU_HALF_RATE_SLOTS) * (2 if has_z else 1)
    sfu = elements + tokch * per_tok
    fp = 4 * elements + 10 * tokch
    return max(sfu / (SFU_EX2_PER_CLK_SM * f), fp / (FP32_LANES_PER_CLK_SM * f))


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    """Samples the SM clock and clock-event reasons while the timed region runs (NVML
    when importable, else `nvidia-smi -lms`)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting",
               0x10: "sync_boost", 0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.idx = device_index
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self.mode = None
        self.err = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.err = f"NVML: {e}"
            self.mode = "smi"

    def _sample_nvml(self):
        nv = self.nv
        self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
        try:
            self.reasons |= nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
        except Exception:
            self.reasons |= nv.nvmlDeviceGetCurrentClocksThrottleReasons(self.h)

    def _run(self):
        while not self._stop.is_set():
            self._sample_nvml()
            time.sleep(self.period)

    def start(self):
        if self.mode == "nvml":
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        else:
            try:
                self._p = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.idx), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception as e:
                self._p = None
                self.err = f"{self.err}; nvidia-smi: {e}"

    def stop(self):
        if self.mode == "nvml":
            self._sample_nvml()
            self._stop.set()
            self._t.join()
            return
        if self._p is None:
            return
        time.sleep(0.05)
        self._p.terminate()
        out, _ = self._p.communicate(timeout=10)
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 3:
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                    self.reasons |= int(parts[2], 16)
                except ValueError:
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "note": f"no samples ({self.err})"}
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit]
        return {"sm_mhz": float(np.median(self.samples)), "sm_max_mhz": float(self.max_mhz), "reasons": names,
                "samples": len(self.samples), "source": self.mode}


# ------------------------------------------------------------------------------------------
# the step
# ------------------------------------------------------------------------------------------
class Step:
    """Device-resident inputs/outputs of one bench step and the three launches."""

    def __init__(self, torch, ssm, device, algo="auto"):
        from workloads.torch_io import decode_set_to_torch, scan_to_torch, to_torch
        self.torch, self.ssm, self.algo = torch, ssm, algo
        self.pre_cfg = W.CONFIGS["mamba130m"]
        self.sm1_cfg = W.CONFIGS["sm1"]
        self.dec_cfg = W.DECODE_CONFIGS["decode"]
        self.pre_in = W.make_scan_inputs(self.pre_cfg)
        self.sm1_in = W.make_scan_inputs(self.sm1_cfg)
        self.dec_in = W.make_decode_inputs(self.dec_cfg)
        self.pre = scan_to_torch(self.pre_in, device)
        s1 = scan_to_torch(self.sm1_in, device)
        # the scalar entry point's d_state = 1 layouts
        self.sm1 = {"u": s1["u"], "delta": s1["delta"], "A": s1["A"][:, 0].contiguous(),
                    "B": s1["B"][:, 0].contiguous(), "C": s1["C"][:, 0].contiguous(),
                    "delta_bias": s1["delta_bias"], "h0": s1["h0"][:, :, 0].contiguous()}
        self.dec_state = to_torch(self.dec_in["state"], device)
        self.dec_A = to_torch(self.dec_in["A"], device)
        self.dec_D = to_torch(self.dec_in["D"], device)
        self.dec_bias = to_torch(self.dec_in["delta_bias"], device)
        self.dec_sets = [decode_set_to_torch(s, device) for s in self.dec_in["sets"]]
        c = self.pre_cfg
        self.pre_y = torch.empty((c.batch, c.dim, c.seqlen), dtype=torch.bfloat16, device=device)
        self.pre_h = torch.empty((c.batch, c.dim, c.dstate), dtype=torch.float32, device=device)
        self.pre_ws = ssm.alloc_workspace(c.batch, c.dim, c.seqlen, c.dstate, device)
        c = self.sm1_cfg
        self.sm1_y = torch.empty((c.batch, c.dim, c.seqlen), dtype=torch.float32, device=device)
        self.sm1_h = torch.empty((c.batch, c.dim), dtype=torch.float32, device=device)
        self.sm1_ws = ssm.alloc_workspace(c.batch, c.dim, c.seqlen, 1, device)
        c = self.dec_cfg
        self.dec_y = torch.empty((c.batch, c.dim), dtype=torch.bfloat16, device=device)
        self.k = 0

    def run(self, events=None):
        ssm, p, s, c = self.ssm, self.pre, self.sm1, self.dec_sets[self.k % len(self.dec_sets)]
        if events:
            events[0].record()
        ssm.scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"], True, None,
                     y=self.pre_y, h_last=self.pre_h, algo=self.algo, workspace=self.pre_ws)
        if events:
            events[1].record()
        ssm.scalar_scan_fwd(s["u"], s["delta"], s["A"], s["B"], s["C"], None, None, s["delta_bias"], True,
                            s["h0"], y=self.sm1_y, h_last=self.sm1_h, workspace=self.sm1_ws)
        if events:
            events[2].record()
        ssm.state_update(self.dec_state, c["x"], c["delta"], self.dec_A, c["B"], c["C"], self.dec_D, c["z"],
                         self.dec_bias, True, y=self.dec_y)
        if events:
            events[3].record()
        self.k += 1

    def parts(self):
        c, s, d = self.pre_cfg, self.sm1_cfg, self.dec_cfg
        return [
            ("prefill_mamba130m", c.tokens_channels, c.tokens_channels * c.dstate,
             scan_bytes(c.batch, c.dim, c.seqlen, c.dstate, 2, 2, True, False), True),
            ("sm1_scalar_scan", s.tokens_channels, s.tokens_channels,
             scan_bytes(s.batch, s.dim, s.seqlen, 1, 4, 4, False, True), False),
            ("decode_token", d.batch * d.dim, d.batch * d.dim * d.dstate,
             decode_bytes(d.batch, d.dim, d.dstate, 2, 2), True),
        ]


class HostStep:
    """The same step through the public API from pinned HOST buffers: every step copies
    its inputs host->device and its outputs device->host inside the timed region.

    Copies run on their own streams, as a streaming caller would run them: the next
    step's inputs (host->device engine) and the previous step's outputs (device->host
    engine) move while the current step computes. Device inputs and outputs are
    double-buffered so no copy overwrites data a launch still reads; the decode state
    is one buffer, updated in step order on the compute stream."""

    def __init__(self, st: Step):
        import torch
        self.torch = torch
        self.st = st
        p = st.pre
        self.h_pre = {k: p[k].cpu().pin_memory() for k in ("u", "delta", "z", "B", "C")}
        self.h_sm1 = {k: st.sm1[k].cpu().pin_memory() for k in ("u", "delta", "B", "C")}
        self.h_dec = [{k: v.cpu().pin_memory() for k, v in s.items()} for s in st.dec_sets]
        self.o_pre = torch.empty(st.pre_y.shape, dtype=st.pre_y.dtype).pin_memory()
        self.o_sm1 = torch.empty(st.sm1_y.shape, dtype=st.sm1_y.dtype).pin_memory()
        self.o_dec = torch.empty(st.dec_y.shape, dtype=st.dec_y.dtype).pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in list(self.h_pre.values()) + list(self.h_sm1.values()))
        self.h2d += sum(t.numel() * t.element_size() for t in self.h_dec[0].values())
        self.d2h = sum(t.numel() * t.element_size() for t in (self.o_pre, self.o_sm1, self.o_dec))
        # two device buffer sets: inputs that arrive by copy, and the step's outputs
        self.dev = []
        for _ in range(2):
            self.dev.append({
                "pre": {k: torch.empty_like(p[k]) for k in self.h_pre},
                "sm1": {k: torch.empty_like(st.sm1[k]) for k in self.h_sm1},
                "dec": {k: torch.empty_like(v) for k, v in st.dec_sets[0].items()},
                "pre_y": torch.empty_like(st.pre_y), "sm1_y": torch.empty_like(st.sm1_y),
                "dec_y": torch.empty_like(st.dec_y)})
        self.s_h2d = torch.cuda.Stream()
        self.s_d2h = torch.cuda.Stream()
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.out_read = [torch.cuda.Event() for _ in range(2)]
        self.n = 0

    def begin(self):
        """Order the copy streams after everything already on the compute stream."""
        comp = self.torch.cuda.current_stream()
        self.s_h2d.wait_stream(comp)
        self.s_d2h.wait_stream(comp)

    def end(self):
        """Make the compute stream wait for the last copies (the timed region's end)."""
        comp = self.torch.cuda.current_stream()
        comp.wait_stream(self.s_h2d)
        comp.wait_stream(self.s_d2h)

    def run(self):
        torch, st, ssm = self.torch, self.st, self.st.ssm
        comp = torch.cuda.current_stream()
        i = self.n % 2
        d = self.dev[i]
        hd = self.h_dec[st.k % len(self.h_dec)]
        with torch.cuda.stream(self.s_h2d):
            if self.n >= 2:
                self.s_h2d.wait_event(self.computed[i])   # set i's last launches are done with it
            for k, v in self.h_pre.items():
                d["pre"][k].copy_(v, non_blocking=True)
            for k, v in self.h_sm1.items():
                d["sm1"][k].copy_(v, non_blocking=True)
            for k, v in hd.items():
                d["dec"][k].copy_(v, non_blocking=True)
            self.in_ready[i].record(self.s_h2d)
        comp.wait_event(self.in_ready[i])
        if self.n >= 2:
            comp.wait_event(self.out_read[i])            # set i's outputs have left
        p, s, c = d["pre"], d["sm1"], d["dec"]
        pa, sa = st.pre, st.sm1
        ssm.scan_fwd(p["u"], p["delta"], pa["A"], p["B"], p["C"], pa["D"], p["z"], pa["delta_bias"], True, None,
                     y=d["pre_y"], h_last=st.pre_h, algo=st.algo, workspace=st.pre_ws)
        ssm.scalar_scan_fwd(s["u"], s["delta"], sa["A"], s["B"], s["C"], None, None, sa["delta_bias"], True,
                            sa["h0"], y=d["sm1_y"], h_last=st.sm1_h, workspace=st.sm1_ws)
        ssm.state_update(st.dec_state, c["x"], c["delta"], st.dec_A, c["B"], c["C"], st.dec_D, c["z"],
                         st.dec_bias, True, y=d["dec_y"])
        self.computed[i].record(comp)
        with torch.cuda.stream(self.s_d2h):
            self.s_d2h.wait_event(self.computed[i])
            self.o_pre.copy_(d["pre_y"], non_blocking=True)
            self.o_sm1.copy_(d["sm1_y"], non_blocking=True)
            self.o_dec.copy_(d["dec_y"], non_blocking=True)
            self.out_read[i].record(self.s_d2h)
        st.k += 1
        self.n += 1


# ------------------------------------------------------------------------------------------
# oracle timings (CPU baseline and the reference arm)
# ------------------------------------------------------------------------------------------
def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(pre_in, sm1_in, dec_in, min_seconds: float):
    """Time the fp64 oracle on bounded samples of each part; returns per-part token*channel/s."""
    import oracle
    threads = _cores()
    out = {}

    def timed(fn, units):
        t0 = time.perf_counter()
        reps = 0
        while True:
            fn()
            reps += 1
            if time.perf_counter() - t0 >= min_seconds / 3:
                break
        return reps * units / (time.perf_counter() - t0)

    chans = [(0, d) for d in range(256)]
    out["prefill_mamba130m"] = timed(lambda: oracle.scan_inputs(pre_in, chans, threads=threads),
                                     len(chans) * pre_in["seqlen"])
    chans1 = [(0, d) for d in range(1536)]
    out["sm1_scalar_scan"] = timed(lambda: oracle.scan_inputs(sm1_in, chans1, threads=threads),
                                   len(chans1) * sm1_in["seqlen"])
    rows = slice(0, 32)
    st = dec_in["state"][rows].astype(np.float64)
    s = dec_in["sets"][0]
    args = (s["x"].f32()[rows], s["delta"].f32()[rows], dec_in["A"], s["B"].f32()[rows], s["C"].f32()[rows],
            dec_in["D"], s["z"].f32()[rows], dec_in["delta_bias"], True)
    out["decode_token"] = timed(lambda: oracle.state_update(st, *args, threads=threads), 32 * dec_in["dim"])
    sample = ("fp64 oracle on: prefill batch row 0, channels 0-255, full L; SM1 batch row 0, all 1536 "
              "channels; decode batch rows 0-31, one token; each repeated for >= %.1f s" % (min_seconds / 3))
    return out, threads, sample


def step_tokch():
    c, s, d = W.CONFIGS["mamba130m"], W.CONFIGS["sm1"], W.DECODE_CONFIGS["decode"]
    return {"prefill_mamba130m": c.tokens_channels, "sm1_scalar_scan": s.tokens_channels,
            "decode_token": d.batch * d.dim}


def cpu_value(rates):
    tc = step_tokch()
    secs = sum(tc[k] / rates[k] for k in tc)
    return sum(tc.values()) / secs / 1e9


def base_config(extra=None):
    cfg = {"workload": WORKLOAD,
           "parts": {"prefill": "mamba130m (8,1536,2048,16) bf16 in/out, softplus, silu(z), fp32 state",
                     "sm1": "scalar scan (8,1536,2048,1) fp32, h0~N(0,1)",
                     "decode": "one token on (256,5120,16) fp32 state, bf16 x/delta/z/B/C"},
           "l2": "no flush: per-step traffic ~0.68 GB > 126 MB L2, each part's inputs exceed L2 or are "
                 "evicted by the other parts between uses"}
    if extra:
        cfg.update(extra)
    return cfg


def _traffic_record(kernel: str):
    """ncu DRAM bytes (read + write) per launch recorded in profiles/traffic.json, valid
    only while the kernel's sources hash to what they were when the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        p = os.path.join(ROOT, src)
        if not os.path.exists(p):
            return None
        h.update(open(p, "rb").read())
    if h.hexdigest()[:16] != rec["sources_sha"]:
        return None
    return rec["bytes_per_launch"]


# ------------------------------------------------------------------------------------------
# multi-process (one process per GPU, independent replicas)
# ------------------------------------------------------------------------------------------
def rank_env():
    """(world, rank, local_rank) from the torchrun environment; (1, 0, 0) without it."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time: every rank runs the same per-GPU workload, so the job
    takes as long as its slowest rank."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokch_per_rank: int, ms: float) -> float:
    """Whole-job Gtoken*channel/s: all ranks' units over the slowest rank's step time."""
    return world * tokch_per_rank / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--algo", default="auto", choices=["auto", "thread", "warpscan", "lookback"],
                    help="prefill scan algorithm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-configs", action="store_true", help="skip timing the other prefill configs")
    ap.add_argument("--only", choices=["scan", "decode", "conv", "conv_update", "scan_bwd", "ssd", "scan_dir",
                                       "pipes"],
                    help="time one entry point alone on --config (a kernel case for sweeps and ncu)")
    ap.add_argument("--config", default="mamba130m",
                    help="workload of --only: a prefill-scan config name, or 'decode'")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.only:
        return run_case(args)

    world, rank, local_rank = rank_env()

    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import selective_state_space_121_b300 as ssm

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    st = Step(torch, ssm, device, args.algo)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.start()
    start.record(stream)
    for k in range(args.steps):
        st.run(ev[k])
    end.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    ms = start.elapsed_time(end) / args.steps
    part_ms = np.zeros(3)
    for e in ev:
        for i in range(3):
            part_ms[i] += e[i].elapsed_time(e[i + 1])
    part_ms /= args.steps
    if dist:
        ms = max_over_ranks(ms, dist, device)
        dist.barrier()

    # end to end from pinned host buffers through the same public API
    hs = HostStep(st)
    hs.begin()
    for _ in range(3):
        hs.run()
    hs.end()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    hs.begin()
    for _ in range(args.e2e_steps):
        hs.run()
    hs.end()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    if dist:
        e2e_ms = max_over_ranks(e2e_ms, dist, device)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # every prefill config of the hot path on its own (auto algorithm; inputs > L2)
    configs_measured = {}
    step_parts = st.parts()
    step_inputs = (st.pre_in, st.sm1_in, st.dec_in)
    h2d, d2h = hs.h2d, hs.d2h
    if not args.no_configs:
        del st, hs
        torch.cuda.empty_cache()
        for name, steps in (("tiny", 50), ("mamba2p8b", 10), ("long", 5)):
            rec = time_case("scan", name, "auto", steps, 3, device)
            configs_measured[name] = {k: rec[k] for k in ("case", "ms_median", "Gtokch_s", "GB_s", "hbm_frac")}
            torch.cuda.empty_cache()
        # the conv that feeds the scan (prefill and decode update, HBM-bound) and the
        # scan's backward on the Mamba-130M-shaped layer
        for only, cfgname, steps in (("conv", None, 50), ("conv_update", None, 100), ("scan_bwd", "mamba130m", 5),
                                     ("ssd", "ssd_5120", 10), ("scan_dir", "vmamba56", 10)):
            rec = time_case(only, cfgname, "auto", steps, 3, device)
            configs_measured[only] = {k: rec[k] for k in ("case", "ms_median", "Gtokch_s", "GB_s", "hbm_frac")}
            if "tensor_TFLOP_s" in rec:
                configs_measured[only].update({k: rec[k] for k in ("tensor_TFLOP_s", "tensor_frac")})
                configs_measured[only]["traffic"] = _traffic_record("ssd_5120")
            torch.cuda.empty_cache()

    hbm_peak, _, peak_kind = _peaks()
    parts_out = {}
    tot_tokch = 0
    for (name, tokch, elems, nbytes, has_z), pm in zip(step_parts, part_ms):
        tot_tokch += tokch
        sec = pm * 1e-3
        hbm_t = nbytes / (hbm_peak * 1e9)
        alu_t = alu_roof_seconds(elems, tokch, has_z, SM_MAX_MHZ_NOMINAL)
        parts_out[name] = {"ms": round(pm, 5), "Gtokch_s": tokch / sec / 1e9, "GB_s": nbytes / sec / 1e9,
                           "hbm_frac": nbytes / sec / 1e9 / hbm_peak, "alg_bytes": nbytes, "elements": elems,
                           "roof_us": {"hbm": hbm_t * 1e6, "alu": alu_t * 1e6},
                           "roof_frac": max(hbm_t, alu_t) / sec}
    value = job_value(world, tot_tokch, ms)

    # roofline of the dominant kernel (largest share of the step)
    dom_i = int(np.argmax(part_ms))
    name, tokch, elems, nbytes, has_z = step_parts[dom_i]
    sec = part_ms[dom_i] * 1e-3
    hbm_t = nbytes / (hbm_peak * 1e9)
    alu_t = alu_roof_seconds(elems, tokch, has_z, SM_MAX_MHZ_NOMINAL)
    if alu_t > hbm_t:
        flops = 6.0 * elems   # per (t, n): dt*A, (dt*u)*B, a*h+b (2), C*h+y (2)
        peak = 6.0 * elems / alu_t / 1e12
        roofline = {"bound": "alu", "kernel": name, "achieved": flops / sec / 1e12, "peak": peak,
                    "unit": "TFLOP/s", "frac": (flops / sec / 1e12) / peak,
                    "peak_kind": "derived: 148 SMs x 2032 MHz; per (t,n) element 1 ex2 (32/clk/SM, measured) + "
                                 "4 FP32 FMA-pipe ops (128/clk/SM); per (b,d,t) softplus+silu = 6 SFU slots "
                                 "(lg2, rcp at half rate) + 10 FP32 ops; 6 flops/element",
                    "hbm_GB_s": nbytes / sec / 1e9, "hbm_frac_of_measured": nbytes / sec / 1e9 / hbm_peak,
                    "traffic": _traffic_record(name)}
    else:
        roofline = {"bound": "hbm", "kernel": name, "achieved": nbytes / sec / 1e9, "peak": hbm_peak,
                    "unit": "GB/s", "frac": nbytes / sec / 1e9 / hbm_peak,
                    "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)", "traffic": _traffic_record(name)}

    cpu = None
    if not args.no_cpu_baseline:
        rates, cores, sample = oracle_sample(*step_inputs, 12.0)
        cpu = {"value": cpu_value(rates), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "parts_Gtokch_s": {k: v / 1e9 for k, v in rates.items()}}

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32 in, f32 arithmetic and state",
        "data": "synthetic (seeded PCG64 inputs shaped like Mamba-130M layers)",
        "config": base_config({"parallelism": f"replicas x{world} (independent batches per GPU)",
                               "prefill_algo": args.algo}),
        "parts": parts_out,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": job_value(world, tot_tokch, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "copies": "pinned host buffers; host->device and device->host on their own streams, "
                          "device buffers double-buffered, so copies overlap the neighbouring steps"},
        "configs_measured": configs_measured,
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


def run_case(args):
    """One entry point alone on one workload: W warm-up launches, then K launches each
    timed with CUDA events on the launching stream. Prints one JSON line (not the
    bench contract line): median/mean ms, Gtoken*channel/s, algorithmic GB/s.
    `--only pipes` instead prints the measured per-SM pipe throughputs
    (selective_state_space_121_b300.pipes) the compute roof is derived from."""
    import torch
    torch.cuda.set_device(0)
    if args.only == "pipes":
        from selective_state_space_121_b300 import pipes
        print(json.dumps({"pipes": pipes.pipe_rates(), "device": torch.cuda.get_device_name(0)}))
        return
    print(json.dumps(time_case(args.only, args.config, args.algo, args.steps, args.warmup, torch.device("cuda", 0))))


def time_case(only, config, algo, steps, warmup, dev):
    """Times one entry point alone on one workload (see run_case); returns the record."""
    import torch
    import selective_state_space_121_b300 as ssm
    from workloads.torch_io import decode_set_to_torch, scan_to_torch, to_torch
    stream = torch.cuda.current_stream()
    if only == "scan":
        cfg = W.CONFIGS[config]
        inp = W.make_scan_inputs(cfg)
        t = scan_to_torch(inp, dev)
        ei = 2 if cfg.in_dtype == W.BF16 else 4
        eo = 2 if cfg.out_dtype == W.BF16 else 4
        odt = torch.bfloat16 if cfg.out_dtype == W.BF16 else torch.float32
        y = torch.empty((cfg.batch, cfg.dim, cfg.seqlen), dtype=odt, device=dev)
        h = torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32, device=dev)
        ws = ssm.alloc_workspace(cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate, dev)

        def launch():
            ssm.scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                         cfg.softplus, t["h0"], y=y, h_last=h, algo=algo, workspace=ws)
        tokch = cfg.tokens_channels
        nbytes = scan_bytes(cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate, ei, eo, cfg.has_z, t["h0"] is not None)
        label = f"scan {cfg.name} ({cfg.batch},{cfg.dim},{cfg.seqlen},{cfg.dstate}) algo={algo}"
    elif only == "scan_bwd":
        cfg = W.CONFIGS[config]
        inp = W.make_scan_inputs(cfg)
        t = scan_to_torch(inp, dev)
        odt = torch.bfloat16 if cfg.out_dtype == W.BF16 else torch.float32
        dout = torch.randn((cfg.batch, cfg.dim, cfg.seqlen), generator=torch.Generator(dev).manual_seed(1),
                           device=dev).to(odt)
        wsb = torch.empty(max(ssm.scan_bwd_workspace_size(cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate), 16),
                          dtype=torch.uint8, device=dev)

        def launch():
            ssm.scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], cfg.softplus,
                         t["h0"], dout=dout, workspace=wsb, want_dh0=False)
        ei = 2 if cfg.in_dtype == W.BF16 else 4
        eo = 2 if cfg.out_dtype == W.BF16 else 4
        tokch = cfg.tokens_channels
        x = cfg.batch * cfg.dim * cfg.seqlen
        # inputs u, delta, z, dout, B, C read; du, ddelta, dz written; dB, dC fp32 written
        nbytes = x * (3 * ei + eo + 3 * ei) + 2 * cfg.batch * cfg.dstate * cfg.seqlen * (ei + 4)
        label = f"scan_bwd {cfg.name} ({cfg.batch},{cfg.dim},{cfg.seqlen},{cfg.dstate})"
    elif only == "conv":
        cfg = W.CONV_CONFIGS["conv_mamba130m"]
        inp = W.make_conv_inputs(cfg)
        x, w, bias, st = (to_torch(inp[k], dev) for k in ("x", "weight", "bias", "conv_state"))
        odt = torch.bfloat16 if cfg.out_dtype == W.BF16 else torch.float32
        out = torch.empty(x.shape, dtype=odt, device=dev)
        so = torch.empty_like(st)

        def launch():
            ssm.causal_conv1d_fwd(x, w, bias, st, True, out=out, conv_state_out=so)
        ei = 2 if cfg.in_dtype == W.BF16 else 4
        eo = 2 if cfg.out_dtype == W.BF16 else 4
        tokch = cfg.batch * cfg.dim * cfg.seqlen
        nbytes = conv_bytes(cfg.batch, cfg.dim, cfg.seqlen, cfg.width, ei, eo)
        label = f"causal_conv1d {cfg.name} ({cfg.batch},{cfg.dim},{cfg.seqlen}) width={cfg.width}"
    elif only == "conv_update":
        cfg = W.CONV_CONFIGS["conv_decode"]
        # 12 state/input/output sets (12 x 16 MB > the 126 MB L2) taken in turn
        sets = []
        for k in range(12):
            inp = W.make_conv_inputs(dataclasses.replace(cfg, seed_base=cfg.seed_base + 10 * k))
            sets.append((to_torch(inp["conv_state"], dev), to_torch(inp["x"], dev)[..., 0].contiguous(),
                         torch.empty((cfg.batch, cfg.dim), dtype=torch.bfloat16, device=dev)))
        w, bias = to_torch(inp["weight"], dev), to_torch(inp["bias"], dev)
        k = [0]

        def launch():
            st, xt, o = sets[k[0] % len(sets)]
            k[0] += 1
            ssm.causal_conv1d_update(st, xt, w, bias, True, out=o)
        tokch = cfg.batch * cfg.dim
        nbytes = conv_update_bytes(cfg.batch, cfg.dim, cfg.width, 2, 2)
        label = f"causal_conv1d_update ({cfg.batch},{cfg.dim}) width={cfg.width}"
    elif only == "scan_dir":
        # the four-direction image scan: one timed unit runs all four traversals
        cfg = W.CONFIGS["vmamba56"]
        rows, cols = W.IMAGE_GRIDS["vmamba56"]
        inp = W.make_scan_inputs(cfg)
        t = scan_to_torch(inp, dev)
        ys = [torch.empty((cfg.batch, cfg.dim, cfg.seqlen), dtype=torch.bfloat16, device=dev) for _ in range(4)]
        hs = [torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32, device=dev) for _ in range(4)]

        def launch():
            for k, order in enumerate(("raster", "reverse", "columns", "columns_reverse")):
                ssm.scan_fwd_dir(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                                 None, order=order, rows=rows, cols=cols, y=ys[k], h_last=hs[k])
        tokch = 4 * cfg.tokens_channels
        nbytes = 4 * scan_bytes(cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate, 2, 2, True, False)
        label = f"scan_dir vmamba56 ({cfg.batch},{cfg.dim},{rows}x{cols},{cfg.dstate}) x 4 directions"
    elif only == "ssd":
        from workloads.torch_io import ssd_to_torch
        cfg = W.SSD_CONFIGS[config if config in W.SSD_CONFIGS else "ssd_5120"]
        inp = W.make_ssd_inputs(cfg)
        t = ssd_to_torch(inp, dev)
        odt = torch.bfloat16 if cfg.out_dtype == W.BF16 else torch.float32
        y = torch.empty((cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim), dtype=odt, device=dev)
        hl = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), dtype=torch.float32, device=dev)

        def launch():
            ssm.ssd_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["dt_bias"], True, t["h0"],
                             y=y, h_last=hl)
        tokch = cfg.tokens_channels
        nbytes = ssd_bytes(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.ngroups, cfg.dstate,
                           2 if odt == torch.bfloat16 else 4, cfg.has_z, cfg.h0 != "zero")
        flops = ssd_tensor_flops(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate)
        label = (f"ssd {cfg.name} (batch {cfg.batch}, L {cfg.seqlen}, {cfg.nheads} heads x {cfg.headdim}, "
                 f"groups {cfg.ngroups}, d_state {cfg.dstate})")
    else:
        cfg = W.DECODE_CONFIGS["decode"]
        inp = W.make_decode_inputs(cfg)
        # four resident states (4 x 84 MB > the 126 MB L2) taken in turn, so every
        # launch streams its state from HBM as it would with one state per layer
        states = [to_torch(inp["state"], dev) for _ in range(4)]
        A, D, bias = (to_torch(inp[k], dev) for k in ("A", "D", "delta_bias"))
        sets = [decode_set_to_torch(s, dev) for s in inp["sets"]]
        yd = torch.empty((cfg.batch, cfg.dim), dtype=torch.bfloat16, device=dev)
        k = [0]

        def launch():
            s = sets[k[0] % len(sets)]
            state = states[k[0] % len(states)]
            k[0] += 1
            ssm.state_update(state, s["x"], s["delta"], A, s["B"], s["C"], D, s["z"], bias, True, y=yd)
        tokch = cfg.batch * cfg.dim
        nbytes = decode_bytes(cfg.batch, cfg.dim, cfg.dstate, 2, 2)
        label = f"decode ({cfg.batch},{cfg.dim},{cfg.dstate})"
    for _ in range(warmup):
        launch()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        e0.record(stream)
        launch()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = np.array([e0.elapsed_time(e1) for e0, e1 in ev])
    hbm_peak, _, peak_kind = _peaks()
    med = float(np.median(ms))
    rec = {"case": label, "launches": steps, "ms_median": med, "ms_mean": float(ms.mean()),
           "ms_min": float(ms.min()), "Gtokch_s": tokch / (med * 1e-3) / 1e9,
           "alg_bytes": nbytes, "GB_s": nbytes / (med * 1e-3) / 1e9,
           "hbm_frac": nbytes / (med * 1e-3) / 1e9 / hbm_peak, "peak_GB_s": hbm_peak, "peak_kind": peak_kind}
    if only == "ssd":
        tf = flops / (med * 1e-3) / 1e12
        rec.update({"tensor_flops": flops, "tensor_TFLOP_s": tf, "tensor_frac": tf / _bf16_peak(),
                    "inputs_vs_L2": f"inputs {(nbytes - tokch * 2) / 1e6:.0f} MB > 126 MB L2"})
    return rec


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle as it stands, on the host cores, each step a
    bounded sample of the same workload (rank 0 only)."""
    if rank != 0:
        return
    pre_in = W.make_scan_inputs(W.CONFIGS["mamba130m"])
    sm1_in = W.make_scan_inputs(W.CONFIGS["sm1"])
    dec_in = W.make_decode_inputs(W.DECODE_CONFIGS["decode"], token_sets=1)
    for _ in range(args.warmup):
        oracle_sample(pre_in, sm1_in, dec_in, 0.0)
    t0 = time.perf_counter()
    rates_acc = {}
    cores, sample = _cores(), ""
    for _ in range(args.steps):
        rates, cores, sample = oracle_sample(pre_in, sm1_in, dec_in, 0.0)
        for k, v in rates.items():
            rates_acc.setdefault(k, []).append(v)
    wall = time.perf_counter() - t0
    rates = {k: float(np.mean(v)) for k, v in rates_acc.items()}
    value = cpu_value(rates)
    tc = step_tokch()
    ms = sum(tc[k] / rates[k] for k in tc) * 1e3
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs as our arm)",
        "config": base_config(), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                         "wall_s": wall},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


if __name__ == "__main__":
    main()
