"""Benchmark of the selective-scan hot path on B300.

One step = one pass of the whole hot path (every row of the scan's scope: the
chunked prefill scan, its multi-block look-back carry for long sequences, the
d_state = 1 scan and the decode update) over one batch of synthetic input, at the
largest single-GPU configurations:
  * prefill scan, Mamba-2.8B-shaped layer: (batch 4, dim 5120, L 4096, N 16), bf16
    u/delta/z/B/C, fp32 A/D/bias/state, softplus + silu(z) gate, y bf16;
  * prefill scan, long context: (1, 1536, 131072, 16), the same dtypes (time is cut
    into segments joined by the decoupled look-back carry);
  * d_state = 1 scalar scan (SM1): (8, 1536, 2048, 1), fp32, h0 ~ N(0,1);
  * one decode token on the resident (256, 5120, 16) fp32 state (the token sets
    rotate through 16 seeded sets; the state carries across steps, so K timed
    steps are K consecutive decode tokens).
Metric: Gtoken*channel/s over the whole step (sum of batch*dim*L over the parts /
step time), with per-part HBM GB/s and roofline fractions. The Mamba-130M-shaped
prefill and the other entry points are timed on their own in `configs_measured`.

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
WORKLOAD = "mamba2p8b_long_sm1_decode_step"
N_SM = 148
SM_MAX_MHZ_NOMINAL = 2032.0
# per-SM pipe rates measured on this B300 by `python bench.py --only pipes`
# (selective_state_space_121_b300/probe/pipe_rates.cu; summary in profiles/)
FP32_LANES_PER_CLK_SM = 128       # FMA pipe (packed f32x2: the same FMAs per clock)
SFU_EX2_PER_CLK_SM = 32           # ex2 lanes per clock per SM
SFU_HALF_RATE_SLOTS = 2           # lg2 and rcp issue at half the ex2 rate (16/clk/SM)

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
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "10"],
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
        out = {"sm_mhz": float(np.median(self.samples)), "sm_max_mhz": float(self.max_mhz), "reasons": names,
               "samples": len(self.samples), "source": self.mode}
        if self.mode != "nvml" and self.err:
            out["nvml_unavailable"] = self.err[:160]
        return out


# ------------------------------------------------------------------------------------------
# the step
# ------------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Part:
    name: str        # key in the JSON line
    kind: str        # "scan" (ssm_scan_fwd), "scalar" (ssm_scalar_scan_fwd), "decode" (ssm_state_update)
    config: str      # workloads config name
    kernel: str      # the kernel that runs it at this size


PARTS = (
    Part("prefill_mamba2p8b", "scan", "mamba2p8b", "serial_scan_kernel"),
    Part("prefill_long", "scan", "long", "serial_lookback_kernel"),
    Part("sm1_scalar_scan", "scalar", "sm1", "scalar_scan_ring_kernel"),
    Part("decode_token", "decode", "decode", "state_update_tma_kernel"),
)


def part_cfg(p: Part):
    return W.DECODE_CONFIGS[p.config] if p.kind == "decode" else W.CONFIGS[p.config]


def part_units(p: Part):
    """(token*channels, (t, n) elements, algorithmic bytes, has_z) of one launch."""
    c = part_cfg(p)
    if p.kind == "decode":
        return (c.batch * c.dim, c.batch * c.dim * c.dstate, decode_bytes(c.batch, c.dim, c.dstate, 2, 2), True)
    ei = 2 if c.in_dtype == W.BF16 else 4
    eo = 2 if c.out_dtype == W.BF16 else 4
    return (c.tokens_channels, c.tokens_channels * c.dstate,
            scan_bytes(c.batch, c.dim, c.seqlen, c.dstate, ei, eo, c.has_z, c.h0 != "zero"), c.has_z)


def make_part_inputs(p: Part, token_sets=None):
    c = part_cfg(p)
    if p.kind == "decode":
        return W.make_decode_inputs(c, token_sets=token_sets)
    return W.make_scan_inputs(c)


class Step:
    """Device-resident inputs/outputs of one bench step and its launches (one per part)."""

    def __init__(self, torch, ssm, device, algo="auto", inputs=None):
        from workloads.torch_io import decode_set_to_torch, scan_to_torch, to_torch
        self.torch, self.ssm, self.algo = torch, ssm, algo
        self.inputs = inputs or {p.name: make_part_inputs(p) for p in PARTS}
        self.dev = {}
        for p in PARTS:
            c, inp = part_cfg(p), self.inputs[p.name]
            if p.kind == "decode":
                d = {"state": to_torch(inp["state"], device), "A": to_torch(inp["A"], device),
                     "D": to_torch(inp["D"], device), "delta_bias": to_torch(inp["delta_bias"], device),
                     "sets": [decode_set_to_torch(s, device) for s in inp["sets"]],
                     "y": torch.empty((c.batch, c.dim), dtype=torch.bfloat16, device=device)}
            else:
                t = scan_to_torch(inp, device)
                if p.kind == "scalar":   # the scalar entry point's d_state = 1 layouts
                    t = {"u": t["u"], "delta": t["delta"], "A": t["A"][:, 0].contiguous(),
                         "B": t["B"][:, 0].contiguous(), "C": t["C"][:, 0].contiguous(), "D": t["D"],
                         "z": t["z"], "delta_bias": t["delta_bias"],
                         "h0": None if t["h0"] is None else t["h0"][:, :, 0].contiguous()}
                odt = torch.bfloat16 if c.out_dtype == W.BF16 else torch.float32
                d = dict(t)
                d["y"] = torch.empty((c.batch, c.dim, c.seqlen), dtype=odt, device=device)
                d["h_last"] = torch.empty((c.batch, c.dim) + ((c.dstate,) if p.kind == "scan" else ()),
                                          dtype=torch.float32, device=device)
                d["ws"] = ssm.alloc_workspace(c.batch, c.dim, c.seqlen, c.dstate, device)
            self.dev[p.name] = d
        self.k = 0

    def launch(self, p: Part, d=None, y=None):
        """One part's launch; `d` overrides the device inputs (the end-to-end copies)."""
        ssm, c = self.ssm, part_cfg(p)
        base = self.dev[p.name]
        d = d or base
        if p.kind == "decode":
            s = d["sets"][self.k % len(base["sets"])] if "sets" in d else d
            ssm.state_update(base["state"], s["x"], s["delta"], base["A"], s["B"], s["C"], base["D"], s["z"],
                             base["delta_bias"], True, y=base["y"] if y is None else y)
        elif p.kind == "scan":
            ssm.scan_fwd(d["u"], d["delta"], base["A"], d["B"], d["C"], base["D"], d["z"], base["delta_bias"],
                         c.softplus, base["h0"], y=base["y"] if y is None else y, h_last=base["h_last"],
                         algo=self.algo, workspace=base["ws"])
        else:
            ssm.scalar_scan_fwd(d["u"], d["delta"], base["A"], d["B"], d["C"], base["D"], d["z"],
                                base["delta_bias"], c.softplus, base["h0"], y=base["y"] if y is None else y,
                                h_last=base["h_last"], workspace=base["ws"])

    def run(self, events=None):
        for i, p in enumerate(PARTS):
            if events:
                events[i].record()
            self.launch(p)
        if events:
            events[len(PARTS)].record()
        self.k += 1


class HostStep:
    """The same step through the public API from pinned HOST buffers: every step copies
    its inputs host->device and its outputs device->host inside the timed region.

    Copies run on their own streams, as a streaming caller would run them: the next
    step's inputs (host->device engine) and the previous step's outputs (device->host
    engine) move while the current step computes. Device inputs and outputs are
    double-buffered so no copy overwrites data a launch still reads; the decode state
    is one buffer, updated in step order on the compute stream."""

    IN_KEYS = {"scan": ("u", "delta", "z", "B", "C"), "scalar": ("u", "delta", "z", "B", "C"),
               "decode": ("x", "delta", "z", "B", "C")}

    def __init__(self, st: Step):
        import torch
        self.torch = torch
        self.st = st
        self.host_in, self.host_out = {}, {}
        for p in PARTS:
            d = st.dev[p.name]
            if p.kind == "decode":
                self.host_in[p.name] = [{k: v.cpu().pin_memory() for k, v in s.items()} for s in d["sets"]]
            else:
                self.host_in[p.name] = {k: d[k].cpu().pin_memory() for k in self.IN_KEYS[p.kind] if d.get(k) is not None}
            self.host_out[p.name] = torch.empty(d["y"].shape, dtype=d["y"].dtype).pin_memory()
        self.h2d = 0
        for p in PARTS:
            hi = self.host_in[p.name]
            hi = hi[0] if isinstance(hi, list) else hi
            self.h2d += sum(t.numel() * t.element_size() for t in hi.values())
        self.d2h = sum(t.numel() * t.element_size() for t in self.host_out.values())
        self.dev = []
        for _ in range(2):
            bufs = {}
            for p in PARTS:
                hi = self.host_in[p.name]
                hi = hi[0] if isinstance(hi, list) else hi
                bufs[p.name] = {k: torch.empty(v.shape, dtype=v.dtype, device=st.dev[p.name]["y"].device)
                                for k, v in hi.items()}
                bufs[p.name]["_y"] = torch.empty_like(st.dev[p.name]["y"])
            self.dev.append(bufs)
        self.s_h2d = torch.cuda.Stream()
        self.s_d2h = torch.cuda.Stream()
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.out_read = [torch.cuda.Event() for _ in range(2)]
        self.n = 0

    def begin(self):
        comp = self.torch.cuda.current_stream()
        self.s_h2d.wait_stream(comp)
        self.s_d2h.wait_stream(comp)

    def end(self):
        comp = self.torch.cuda.current_stream()
        comp.wait_stream(self.s_h2d)
        comp.wait_stream(self.s_d2h)

    def run(self):
        torch, st = self.torch, self.st
        comp = torch.cuda.current_stream()
        i = self.n % 2
        bufs = self.dev[i]
        with torch.cuda.stream(self.s_h2d):
            if self.n >= 2:
                self.s_h2d.wait_event(self.computed[i])   # set i's last launches are done with it
            for p in PARTS:
                hi = self.host_in[p.name]
                hi = hi[st.k % len(hi)] if isinstance(hi, list) else hi
                for k, v in hi.items():
                    bufs[p.name][k].copy_(v, non_blocking=True)
            self.in_ready[i].record(self.s_h2d)
        comp.wait_event(self.in_ready[i])
        if self.n >= 2:
            comp.wait_event(self.out_read[i])            # set i's outputs have left
        for p in PARTS:
            d = {k: v for k, v in bufs[p.name].items() if k != "_y"}
            for k in self.IN_KEYS[p.kind]:
                d.setdefault(k, None)
            st.launch(p, d, y=bufs[p.name]["_y"])
        self.computed[i].record(comp)
        with torch.cuda.stream(self.s_d2h):
            self.s_d2h.wait_event(self.computed[i])
            for p in PARTS:
                self.host_out[p.name].copy_(bufs[p.name]["_y"], non_blocking=True)
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


# the bounded sample of each part the fp64 oracle runs: (what, number of units)
SAMPLE = {
    "prefill_mamba2p8b": ("batch row 0, channels 0-255, full L", 256),
    "prefill_long": ("batch row 0, channels 0-15, full L", 16),
    "sm1_scalar_scan": ("batch row 0, channels 0-1535, full L", 1536),
    "decode_token": ("batch rows 0-15, all channels, one token", 16),
}


def sample_text():
    return "fp64 oracle on: " + "; ".join(f"{k}: {v[0]}" for k, v in SAMPLE.items())


def oracle_part(p: Part, inp, threads):
    """Runs the oracle once on the part's sample; returns the token*channels it covered."""
    import oracle
    n = SAMPLE[p.name][1]
    if p.kind == "decode":
        rows = slice(0, n)
        st = inp["state"][rows].astype(np.float64)
        s = inp["sets"][0]
        oracle.state_update(st, s["x"].f32()[rows], s["delta"].f32()[rows], inp["A"], s["B"].f32()[rows],
                            s["C"].f32()[rows], inp["D"], s["z"].f32()[rows], inp["delta_bias"], True,
                            threads=threads)
        return n * inp["dim"]
    chans = [(0, d) for d in range(n)]
    oracle.scan_inputs(inp, chans, threads=threads)
    return n * inp["seqlen"]


def oracle_rates(inputs, min_seconds: float):
    """Per-part oracle throughput (token*channels/s), each part repeated for about
    min_seconds / #parts."""
    threads = _cores()
    rates = {}
    for p in PARTS:
        t0 = time.perf_counter()
        units = 0
        while True:
            units += oracle_part(p, inputs[p.name], threads)
            if time.perf_counter() - t0 >= min_seconds / len(PARTS):
                break
        rates[p.name] = units / (time.perf_counter() - t0)
    return rates, threads


def step_value_from_rates(rates):
    """Whole-step Gtoken*channel/s if every part ran at its sampled rate."""
    tc = {p.name: part_units(p)[0] for p in PARTS}
    secs = sum(tc[k] / rates[k] for k in tc)
    return sum(tc.values()) / secs / 1e9


def base_config(extra=None):
    cfg = {"workload": WORKLOAD,
           "parts": {"prefill_mamba2p8b": "(4,5120,4096,16) bf16 in/out, softplus, silu(z), fp32 state",
                     "prefill_long": "(1,1536,131072,16) bf16 in/out, softplus, silu(z), look-back carry",
                     "sm1_scalar_scan": "(8,1536,2048,1) fp32, h0~N(0,1)",
                     "decode_token": "one token on (256,5120,16) fp32 state, bf16 x/delta/z/B/C"},
           "l2": "no flush: per-step traffic ~2.8 GB > 126 MB L2, each part's inputs exceed L2 or are "
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--algo", default="auto", choices=["auto", "thread", "warpscan", "lookback"],
                    help="prefill scan algorithm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--no-configs", action="store_true", help="skip timing the other entry points and configs")
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

    nparts = len(PARTS)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nparts + 1)] for _ in range(args.steps)]
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
    part_ms = np.zeros(nparts)
    for e in ev:
        for i in range(nparts):
            part_ms[i] += e[i].elapsed_time(e[i + 1])
    part_ms /= args.steps
    if dist:
        ms = max_over_ranks(ms, dist, device)
        dist.barrier()

    # end to end from pinned host buffers through the same public API
    hs = HostStep(st)
    hs.begin()
    for _ in range(2):
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

    inputs = st.inputs
    h2d, d2h = hs.h2d, hs.d2h
    del st, hs
    torch.cuda.empty_cache()

    hbm_peak, _, peak_kind = _peaks()
    parts_out = {}
    tot_tokch = 0
    for p, pm in zip(PARTS, part_ms):
        tokch, elems, nbytes, has_z = part_units(p)
        tot_tokch += tokch
        sec = pm * 1e-3
        hbm_t = nbytes / (hbm_peak * 1e9)
        alu_t = alu_roof_seconds(elems, tokch, has_z, SM_MAX_MHZ_NOMINAL)
        parts_out[p.name] = {"kernel": p.kernel, "ms": round(float(pm), 5), "Gtokch_s": tokch / sec / 1e9,
                             "GB_s": nbytes / sec / 1e9, "hbm_frac": nbytes / sec / 1e9 / hbm_peak,
                             "alg_bytes": nbytes, "elements": elems,
                             "roof_us": {"hbm": hbm_t * 1e6, "alu": alu_t * 1e6},
                             "alu_frac": alu_t / sec}
    value = job_value(world, tot_tokch, ms)

    # roofline of the dominant kernel (largest share of the step), against HBM; its
    # compute (SFU / FMA-pipe) roof beside it
    dom_i = int(np.argmax(part_ms))
    dp = PARTS[dom_i]
    tokch, elems, nbytes, has_z = part_units(dp)
    sec = part_ms[dom_i] * 1e-3
    alu_t = alu_roof_seconds(elems, tokch, has_z, SM_MAX_MHZ_NOMINAL)
    alu_peak = 6.0 * elems / alu_t / 1e12
    roofline = {"bound": "hbm", "kernel": dp.kernel, "part": dp.name,
                "achieved": nbytes / sec / 1e9, "peak": hbm_peak, "unit": "GB/s",
                "frac": nbytes / sec / 1e9 / hbm_peak,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)",
                "alg_bytes_per_launch": nbytes, "launch_ms": float(part_ms[dom_i]),
                "traffic": _traffic_record(dp.name),
                "alu": {"achieved": 6.0 * elems / sec / 1e12, "peak": alu_peak, "unit": "TFLOP/s",
                        "frac": alu_t / sec,
                        "peak_kind": "derived from the measured pipe rates (bench.py --only pipes): 148 SMs x "
                                     "2032 MHz; per (t,n) element 1 ex2 (32/clk/SM) + 4 FP32 FMA-pipe ops "
                                     "(128/clk/SM); per (b,d,t) softplus+silu = 6 SFU slots (lg2, rcp at half "
                                     "rate) + 10 FP32 ops; 6 flops/element"}}

    # the other configs and entry points, each timed on its own (graph replay)
    configs_measured = {}
    if not args.no_configs:
        cases = [("scan", "tiny", 50), ("scan", "mamba130m", 20), ("conv", None, 50), ("conv_update", None, 100),
                 ("scan_bwd", "mamba130m", 5), ("ssd", "ssd_5120", 10), ("scan_dir", "vmamba56", 10)]
        for only, cfgname, steps in cases:
            rec = time_case(only, cfgname, "auto", steps, 3, device)
            key = cfgname if only == "scan" else only
            configs_measured[key] = {k: rec[k] for k in ("case", "ms_median", "Gtokch_s", "GB_s", "hbm_frac")
                                     if k in rec}
            for k in ("tensor_TFLOP_s", "tensor_frac", "alu_frac"):
                if k in rec:
                    configs_measured[key][k] = rec[k]
            if only == "ssd":
                configs_measured[key]["traffic"] = _traffic_record("ssd_5120")
            torch.cuda.empty_cache()

    cpu = None
    if not args.no_cpu_baseline:
        rates, cores = oracle_rates(inputs, 16.0)
        cpu = {"value": step_value_from_rates(rates), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample_text() + "; each part repeated for ~4 s, rates combined over the step's units",
               "parts_Gtokch_s": {k: v / 1e9 for k, v in rates.items()}}

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32 in, f32 arithmetic and state",
        "data": "synthetic (seeded PCG64 inputs shaped like Mamba-2.8B / long-context / SM1 / decode layers)",
        "config": base_config(),
        "parallelism": f"replicas x{world} (independent batches per GPU)", "prefill_algo": args.algo,
        "parts": parts_out,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": job_value(world, tot_tokch, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "copies": "pinned host buffers; host->device and device->host on their own streams, "
                          "device buffers double-buffered, so copies overlap the neighbouring steps"},
        "configs_measured": configs_measured,
        "gpu_launches": nparts * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


def run_case(args):
    """One entry point alone on one workload: W warm-up launches, then K launches
    captured in a CUDA graph and replayed (the host's per-call overhead, as large as a
    decode launch, stays out of the timed region), timed with CUDA events on the
    launching stream. Prints one JSON line (not the bench contract line): median
    ms per launch, Gtoken*channel/s, algorithmic GB/s. `--only pipes` instead prints
    the measured per-SM pipe throughputs (selective_state_space_121_b300.pipes) the
    compute roof is derived from."""
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
        # one workspace, reused by the four walks in turn (same stream)
        dir_ws = torch.empty(ssm._lib.ssm_scan_dir_workspace_size(cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate,
                                                                 ssm.SSM_BF16, ssm.SSM_BF16),
                             dtype=torch.uint8, device=dev)

        def launch():
            for k, order in enumerate(("raster", "reverse", "columns", "columns_reverse")):
                ssm.scan_fwd_dir(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True,
                                 None, order=order, rows=rows, cols=cols, y=ys[k], h_last=hs[k], workspace=dir_ws)
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
        ssd_ws = torch.empty(ssm.ssd_workspace_size(cfg.batch, cfg.nheads, cfg.dstate), dtype=torch.uint8, device=dev)

        def launch():
            ssm.ssd_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["dt_bias"], True, t["h0"],
                             y=y, h_last=hl, workspace=ssd_ws)
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
    timing = "graph"
    try:
        # `steps` launches captured once, replayed 5 times
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                for _ in range(steps):
                    launch()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ms = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1) / steps)
        ms = np.array(ms)
        del g
    except Exception as exc:   # a launch path that cannot be captured: per-launch events
        timing = f"events ({type(exc).__name__})"
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
    rec = {"case": label, "launches": steps, "timing": timing, "ms_median": med, "ms_mean": float(ms.mean()),
           "ms_min": float(ms.min()), "Gtokch_s": tokch / (med * 1e-3) / 1e9,
           "alg_bytes": nbytes, "GB_s": nbytes / (med * 1e-3) / 1e9,
           "hbm_frac": nbytes / (med * 1e-3) / 1e9 / hbm_peak, "peak_GB_s": hbm_peak, "peak_kind": peak_kind}
    if only == "scan" and cfg.dstate > 1:
        rec["alu_frac"] = alu_roof_seconds(tokch * cfg.dstate, tokch, cfg.has_z, SM_MAX_MHZ_NOMINAL) / (med * 1e-3)
    if only == "ssd":
        tf = flops / (med * 1e-3) / 1e12
        rec.update({"tensor_flops": flops, "tensor_TFLOP_s": tf, "tensor_frac": tf / _bf16_peak(),
                    "inputs_vs_L2": f"inputs {(nbytes - tokch * 2) / 1e6:.0f} MB > 126 MB L2"})
    return rec


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle as it stands, on the host cores (rank 0 only).
    Each step runs the oracle once over a bounded sample of every part (SAMPLE); the
    line reports the wall time those steps actually took and the token*channels they
    covered, with the same config dict as our arm."""
    if rank != 0:
        return
    inputs = {p.name: make_part_inputs(p, token_sets=1 if p.kind == "decode" else None) for p in PARTS}
    threads = _cores()

    def one_step():
        return sum(oracle_part(p, inputs[p.name], threads) for p in PARTS)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    units = 0
    for _ in range(args.steps):
        units += one_step()
    wall = time.perf_counter() - t0
    value = units / wall / 1e9
    ms = wall / args.steps * 1e3
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs as our arm)",
        "config": base_config(), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample_text() + f"; one pass of each per step ({units // args.steps} "
                                                   "token*channels per step)", "wall_s": wall},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


if __name__ == "__main__":
    main()
