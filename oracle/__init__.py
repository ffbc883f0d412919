"""fp64 CPU oracle for the Mamba-1 selective scan -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
legs may import this package. The CUDA product path never does, and the two
share no code: the oracle's arithmetic lives in ssm_oracle.c (sequential
recurrence, plain C, double precision) and forms.py (the pages' closed forms,
numpy fp64, used as pins).

Pins (tests/test_oracle_pins.py) tie the oracle to what the pages and the
mathematics fix: brute-force unrolled sums in exact rationals, an exact integer
case, the SM1 closed form, the LTI convolution kernel, associativity of the
affine pairs, resume from h_last, decode/prefill duality, linearity and limits.
No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library (gcc, fp64, no fast-math)."""
    subprocess.run(["gcc", *_CFLAGS, "-o", out, src, "-lm"], check=True)
    return out


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into oracle/liboracle.so if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleLib:
    """ctypes view of one compiled oracle library (the default one, or a test variant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_scan.argtypes = [P] * 8 + [ctypes.c_int, P, P, P, I64, I64, I64, I64, ctypes.c_int]
        lib.oracle_scan.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = [P] * 9 + [ctypes.c_int, P, I64, I64, I64, ctypes.c_int]
        lib.oracle_state_update.restype = ctypes.c_int
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_scan_bwd.argtypes = [P] * 8 + [ctypes.c_int] + [P] * 12 + [I64] * 4 + [ctypes.c_int]
        lib.oracle_scan_bwd.restype = ctypes.c_int
        lib.oracle_scan_dir.argtypes = [P] * 8 + [ctypes.c_int, P, P, P] + [I64] * 4 + [ctypes.c_int, I64, I64,
                                                                                  ctypes.c_int, ctypes.c_int]
        lib.oracle_scan_dir.restype = ctypes.c_int
        lib.oracle_ssd_scan.argtypes = [P] * 8 + [ctypes.c_int, P, P, P] + [I64] * 6 + [ctypes.c_int]
        lib.oracle_ssd_scan.restype = ctypes.c_int
        lib.oracle_causal_conv1d.argtypes = [P] * 4 + [ctypes.c_int, P, P, I64, I64, I64, I64, ctypes.c_int]
        lib.oracle_causal_conv1d.restype = ctypes.c_int
        lib.oracle_conv_update.argtypes = [P] * 4 + [ctypes.c_int, P, I64, I64, I64, ctypes.c_int]
        lib.oracle_conv_update.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def softplus(self, x: float) -> float:
        return self.lib.oracle_softplus(float(x))

    def silu(self, x: float) -> float:
        return self.lib.oracle_silu(float(x))

    def max_threads(self) -> int:
        return self.lib.oracle_max_threads()

    def scan(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None,
             threads: int = 0):
        """Sequential fp64 selective scan.

        u, delta, z: (batch, dim, L); B, C: (batch, N, L); A: (dim, N); D, delta_bias:
        (dim,); h0: (batch, dim, N). Float inputs are taken as exact values.
        Returns (y (batch, dim, L) fp64, h_last (batch, dim, N) fp64).
        """
        u = _f32(u); delta = _f32(delta); A = _f32(A); B = _f32(B); C = _f32(C)
        D = _f32(D); z = _f32(z); delta_bias = _f32(delta_bias); h0 = _f64(h0)
        bt, dim, L = u.shape
        N = A.shape[1]
        assert delta.shape == u.shape and B.shape == (bt, N, L) and C.shape == (bt, N, L)
        assert A.shape == (dim, N)
        assert z is None or z.shape == u.shape
        assert h0 is None or h0.shape == (bt, dim, N)
        y = np.empty((bt, dim, L), dtype=np.float64)
        hl = np.empty((bt, dim, N), dtype=np.float64)
        rc = self.lib.oracle_scan(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z),
                                  _p(delta_bias), int(bool(softplus)), _p(h0), _p(y), _p(hl),
                                  bt, dim, L, N, int(threads))
        if rc != 0:
            raise ValueError("oracle_scan rejected the sizes")
        return y, hl

    def scan_dir(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None,
                 order=0, rows=0, cols=0, zoh=False, threads: int = 0):
        """The fp64 scan along traversal `order` (0 raster, 1 reversed, 2 column-major
        of a rows x cols image, 3 reversed columns), outputs in raster order, with the
        zero-order-hold input matrix when zoh. Shapes as scan()."""
        u = _f32(u); delta = _f32(delta); A = _f32(A); B = _f32(B); C = _f32(C)
        D = _f32(D); z = _f32(z); delta_bias = _f32(delta_bias); h0 = _f64(h0)
        bt, dim, L = u.shape
        N = A.shape[1]
        assert delta.shape == u.shape and B.shape == (bt, N, L) and C.shape == (bt, N, L)
        assert z is None or z.shape == u.shape
        assert h0 is None or h0.shape == (bt, dim, N)
        y = np.empty((bt, dim, L), dtype=np.float64)
        hl = np.empty((bt, dim, N), dtype=np.float64)
        rc = self.lib.oracle_scan_dir(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                      int(bool(softplus)), _p(h0), _p(y), _p(hl), bt, dim, L, N, int(order),
                                      int(rows), int(cols), int(bool(zoh)), int(threads))
        if rc != 0:
            raise ValueError("oracle_scan_dir rejected the sizes")
        return y, hl

    def state_update(self, state, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                     softplus=True, threads: int = 0):
        """One decode token in fp64; state (batch, dim, N) fp64 is updated IN PLACE.

        x, delta, z: (batch, dim); B, C: (batch, N). Returns y (batch, dim) fp64.
        """
        assert state.dtype == np.float64 and state.flags.c_contiguous
        x = _f32(x); delta = _f32(delta); A = _f32(A); B = _f32(B); C = _f32(C)
        D = _f32(D); z = _f32(z); delta_bias = _f32(delta_bias)
        bt, dim, N = state.shape
        assert x.shape == (bt, dim) and B.shape == (bt, N) and A.shape == (dim, N)
        y = np.empty((bt, dim), dtype=np.float64)
        rc = self.lib.oracle_state_update(_p(state), _p(x), _p(delta), _p(A), _p(B), _p(C),
                                          _p(D), _p(z), _p(delta_bias), int(bool(softplus)),
                                          _p(y), bt, dim, N, int(threads))
        if rc != 0:
            raise ValueError("oracle_state_update rejected the sizes")
        return y


    def scan_bwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None,
                 dout=None, dh_last=None, threads: int = 0):
        """fp64 gradients of the scan for dout = dl/d(out) (batch, dim, L) and dh_last =
        dl/d(h_last) (batch, dim, N) or None. Returns a dict with du, ddelta, dz (None
        without z), dA, dB, dC, dD, ddelta_bias, dh0 (fp64)."""
        u = _f32(u); delta = _f32(delta); A = _f32(A); B = _f32(B); C = _f32(C)
        D = _f32(D); z = _f32(z); delta_bias = _f32(delta_bias); h0 = _f64(h0)
        dout = _f64(dout); dh_last = _f64(dh_last)
        bt, dim, L = u.shape
        N = A.shape[1]
        assert dout.shape == u.shape and B.shape == (bt, N, L) and C.shape == (bt, N, L)
        assert dh_last is None or dh_last.shape == (bt, dim, N)
        out = {k: np.empty(s_, dtype=np.float64) for k, s_ in (
            ("du", (bt, dim, L)), ("ddelta", (bt, dim, L)), ("dA", (dim, N)), ("dB", (bt, N, L)),
            ("dC", (bt, N, L)), ("dD", (dim,)), ("ddelta_bias", (dim,)), ("dh0", (bt, dim, N)))}
        out["dz"] = np.empty((bt, dim, L), dtype=np.float64) if z is not None else None
        rc = self.lib.oracle_scan_bwd(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
                                      int(bool(softplus)), _p(h0), _p(dout), _p(dh_last), _p(out["du"]),
                                      _p(out["ddelta"]), _p(out["dA"]), _p(out["dB"]), _p(out["dC"]),
                                      _p(out["dD"]), _p(out["dz"]), _p(out["ddelta_bias"]), _p(out["dh0"]),
                                      bt, dim, L, N, int(threads))
        if rc != 0:
            raise ValueError("oracle_scan_bwd failed")
        return out

    def ssd_scan(self, x, dt, A, B, C, D=None, z=None, dt_bias=None, softplus=True, h0=None, threads: int = 0):
        """Mamba-2 multi-head SSM by its recurrence in fp64. x, z: (batch, L, H, P); dt: (batch,
        L, H); B, C: (batch, L, G, N); A, D, dt_bias: (H,); h0: (batch, H, P, N). Returns (y
        (batch, L, H, P), h_last (batch, H, P, N)) fp64."""
        x = _f32(x); dt = _f32(dt); A = _f32(A); B = _f32(B); C = _f32(C)
        D = _f32(D); z = _f32(z); dt_bias = _f32(dt_bias); h0 = _f64(h0)
        bt, L, H, P = x.shape
        G, N = B.shape[2], B.shape[3]
        assert dt.shape == (bt, L, H) and B.shape == (bt, L, G, N) and C.shape == B.shape
        y = np.empty((bt, L, H, P), dtype=np.float64)
        hl = np.empty((bt, H, P, N), dtype=np.float64)
        rc = self.lib.oracle_ssd_scan(_p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(z), _p(dt_bias),
                                      int(bool(softplus)), _p(h0), _p(y), _p(hl), bt, L, H, P, G, N, int(threads))
        if rc != 0:
            raise ValueError("oracle_ssd_scan rejected the sizes")
        return y, hl

    def causal_conv1d(self, x, w, bias=None, conv_state=None, silu=True, threads: int = 0):
        """Causal depthwise conv1d (+ silu) in fp64.

        x: (batch, dim, L); w: (dim, width); bias: (dim,); conv_state: (batch, dim,
        width-1) fp64, the inputs before x (zeros when None). Returns (out (batch, dim,
        L) fp64, conv_state_out (batch, dim, width-1) fp64).
        """
        x = _f32(x); w = _f32(w); bias = _f32(bias)
        bt, dim, L = x.shape
        width = w.shape[1]
        assert w.shape == (dim, width) and width >= 1
        st = None if conv_state is None else _f64(conv_state)
        assert st is None or st.shape == (bt, dim, width - 1)
        out = np.empty((bt, dim, L), dtype=np.float64)
        so = np.empty((bt, dim, width - 1), dtype=np.float64)
        rc = self.lib.oracle_causal_conv1d(_p(x), _p(w), _p(bias), _p(st), int(bool(silu)), _p(out),
                                           _p(so), bt, dim, L, width, int(threads))
        if rc != 0:
            raise ValueError("oracle_causal_conv1d rejected the sizes")
        return out, so

    def conv_update(self, conv_state, x, w, bias=None, silu=True, threads: int = 0):
        """One decode token of the convolution; conv_state (batch, dim, width-1) fp64 is
        updated IN PLACE. x: (batch, dim). Returns out (batch, dim) fp64."""
        assert conv_state.dtype == np.float64 and conv_state.flags.c_contiguous
        x = _f32(x); w = _f32(w); bias = _f32(bias)
        bt, dim = x.shape
        width = w.shape[1]
        assert conv_state.shape == (bt, dim, width - 1) and w.shape == (dim, width)
        out = np.empty((bt, dim), dtype=np.float64)
        rc = self.lib.oracle_conv_update(_p(conv_state), _p(x), _p(w), _p(bias), int(bool(silu)),
                                         _p(out), bt, dim, width, int(threads))
        if rc != 0:
            raise ValueError("oracle_conv_update rejected the sizes")
        return out


_default = None


def default() -> OracleLib:
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def softplus(x: float) -> float:
    return default().softplus(x)


def silu(x: float) -> float:
    return default().silu(x)


def max_threads() -> int:
    return default().max_threads()


def scan(*args, **kw):
    return default().scan(*args, **kw)


def state_update(*args, **kw):
    return default().state_update(*args, **kw)


def scan_dir(*args, **kw):
    return default().scan_dir(*args, **kw)


def scan_bwd(*args, **kw):
    return default().scan_bwd(*args, **kw)


def ssd_scan(*args, **kw):
    return default().ssd_scan(*args, **kw)


def causal_conv1d(*args, **kw):
    return default().causal_conv1d(*args, **kw)


def conv_update(*args, **kw):
    return default().conv_update(*args, **kw)


def scan_inputs(inp: dict, channels=None, threads: int = 0):
    """Run the oracle on a workloads.make_scan_inputs() dict.

    channels: None for all, else an iterable of (b, d) pairs; the oracle then runs a
    reduced problem per batch row holding only those channels (channels are
    independent, so this is the same arithmetic). Returns dict {(b, d): (y_row, h_row)}
    when channels is given, else (y, h_last) for the whole tensor.
    """
    A, D, bias, h0 = inp["A"], inp["D"], inp["delta_bias"], inp["h0"]
    z = inp["z"]
    if channels is None:
        return scan(inp["u"].f32(), inp["delta"].f32(), A, inp["B"].f32(), inp["C"].f32(), D,
                    None if z is None else z.f32(), bias, inp["softplus"], h0, threads)
    by_b = {}
    for (b, d) in channels:
        by_b.setdefault(int(b), []).append(int(d))
    out = {}
    for b, ds in by_b.items():
        ds = sorted(set(ds))
        idx = (b, np.array(ds))
        u = inp["u"].rows_f32(idx)[None]
        dl = inp["delta"].rows_f32(idx)[None]
        zz = None if z is None else z.rows_f32(idx)[None]
        Bb = inp["B"].rows_f32(b)[None]
        Cb = inp["C"].rows_f32(b)[None]
        Ad = A[ds]
        Dd = None if D is None else D[ds]
        bd = None if bias is None else bias[ds]
        hh = None if h0 is None else h0[b, ds][None]
        y, hl = scan(u, dl, Ad, Bb, Cb, Dd, zz, bd, inp["softplus"], hh, threads)
        for i, d in enumerate(ds):
            out[(b, d)] = (y[0, i], hl[0, i])
    return out
