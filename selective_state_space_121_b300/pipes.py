"""Binding of libssmprobe.so (include/ssm_probe.h): per-SM throughput of the pipes
that bound the selective scan, measured on the current CUDA device. Measurement
only; the scan entry points do not use it."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssmprobe.so")

# probe index -> (name, unit of the returned rate)
PROBES = {
    0: ("ex2", "lanes/clk/SM"),
    1: ("lg2", "lanes/clk/SM"),
    2: ("rcp", "lanes/clk/SM"),
    3: ("fma_f32", "lanes/clk/SM"),
    4: ("fma_f32x2", "FP32 FMAs/clk/SM"),
    5: ("lds128_1addr", "warp instr/clk/SM"),
    6: ("lds128_2addr_halfwarp", "warp instr/clk/SM"),
    7: ("lds128_4addr_quarterwarp", "warp instr/clk/SM"),
    8: ("lds128_32_consecutive", "warp instr/clk/SM"),
    9: ("lds64_1addr", "warp instr/clk/SM"),
    10: ("lds64_2addr_halfwarp", "warp instr/clk/SM"),
    11: ("lds32_1addr", "warp instr/clk/SM"),
    12: ("shfl_bfly", "warp instr/clk/SM"),
    13: ("lds128_8addr_per_quarter", "warp instr/clk/SM"),
    14: ("lds128_16addr_per_half", "warp instr/clk/SM"),
}


def pipe_rates(stream=None) -> dict:
    """Runs every probe on torch's current device and stream; returns
    {name: {"rate": r, "unit": u, "cycles": c}}."""
    import torch
    lib = ctypes.CDLL(LIB_PATH)
    lib.ssm_probe_pipe_rate.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
    lib.ssm_probe_pipe_rate.restype = ctypes.c_int
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    out = {}
    for i, (name, unit) in PROBES.items():
        r, c = ctypes.c_double(), ctypes.c_double()
        rc = lib.ssm_probe_pipe_rate(i, ctypes.byref(r), ctypes.byref(c), ctypes.c_void_p(s))
        if rc != 0:
            raise RuntimeError(f"ssm_probe_pipe_rate({i}) returned {rc}")
        out[name] = {"rate": r.value, "unit": unit, "cycles": c.value}
    return out
