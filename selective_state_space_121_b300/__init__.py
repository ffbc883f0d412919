"""B300-native Mamba-1 selective scan: thin Python binding over libssmscan.so.

Every function here only marshals arguments: it checks tensor placement, shape
and dtype, allocates outputs with torch (device memory is torch's job), and
calls the C ABI declared in include/ssm_scan.h on torch's current CUDA stream.
All arithmetic runs in the library's sm_103a kernels; there is no CPU or
PyTorch fallback. If libssmscan.so is missing, importing this package raises.

Entry points (names follow the C ABI):
    scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, h0) -> (y, h_last)
    scalar_scan_fwd(...)  d_state = 1 (SM1) form of scan_fwd
    state_update(state, x, delta, A, B, C, D, z, delta_bias, softplus) -> y
    scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, h0, dout, dh_last) -> gradients
    causal_conv1d_fwd(x, weight, bias, conv_state, silu) -> (u, conv_state_out)
    causal_conv1d_update(conv_state, x, weight, bias, silu) -> u_t
    workspace_size(batch, dim, seqlen, dstate) -> bytes
    query_status(workspace) -> device status word of a look-back scan
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssmscan.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python selective_state_space_121_b300/build.py` "
        "(there is no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_lib.ssm_abi_version.restype = _I
_lib.ssm_status_string.argtypes = [_I]
_lib.ssm_status_string.restype = ctypes.c_char_p
_lib.ssm_scan_workspace_size.argtypes = [_I64] * 4
_lib.ssm_scan_workspace_size.restype = _SZ
_lib.ssm_scan_fwd.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 4 + [_I, _I, _P, _SZ, _P]
_lib.ssm_scan_fwd.restype = _I
_lib.ssm_scan_fwd_algo.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 4 + [_I, _I, _P, _SZ, _I, _P]
_lib.ssm_scan_fwd_algo.restype = _I
_lib.ssm_scalar_scan_fwd.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 3 + [_I, _I, _P, _SZ, _P]
_lib.ssm_scalar_scan_fwd.restype = _I
_lib.ssm_state_update.argtypes = [_P] * 9 + [_I, _P] + [_I64] * 3 + [_I, _I, _P]
_lib.ssm_state_update.restype = _I
_lib.ssm_test_lookback_timeout.argtypes = [_P] * 6 + [_I64] * 4 + [_I, _P, _SZ, _I64, ctypes.c_uint32, _P]
_lib.ssm_test_lookback_timeout.restype = _I
_lib.ssm_ssd_scan_fwd_ws.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 6 + [_I, _I, _P, _SZ, _P]
_lib.ssm_ssd_scan_fwd_ws.restype = _I
_lib.ssm_ssd_workspace_size.argtypes = [_I64] * 3
_lib.ssm_ssd_workspace_size.restype = _SZ
_lib.ssm_test_ssd_wait_fault.argtypes = [_P] * 6 + [_I64] * 6 + [_I, _P, _SZ, _I64, _P]
_lib.ssm_test_serial_handover_timeout.argtypes = [_P] * 6 + [_I64] * 4 + [_I, _P, _SZ, _I64, ctypes.c_uint32, _P]
_lib.ssm_test_serial_handover_timeout.restype = _I
_lib.ssm_test_ssd_wait_fault.restype = _I
_lib.ssm_query_status.argtypes = [_P, _SZ, _P]
_lib.ssm_query_status.restype = _I
_lib.ssm_scan_fwd_lookback_static.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 4 + [_I, _I, _P]
_lib.ssm_scan_fwd_lookback_static.restype = _I
_lib.ssm_scan_bwd_workspace_size.argtypes = [_I64] * 4
_lib.ssm_scan_bwd_workspace_size.restype = _SZ
_lib.ssm_scan_bwd.argtypes = [_P] * 8 + [_I] + [_P] * 12 + [_I64] * 4 + [_I, _I, _P, _SZ, _P]
_lib.ssm_scan_bwd.restype = _I
_lib.ssm_causal_conv1d_fwd.argtypes = [_P] * 6 + [_I64] * 4 + [_I, _I, _I, _P]
_lib.ssm_causal_conv1d_fwd.restype = _I
_lib.ssm_causal_conv1d_update.argtypes = [_P] * 5 + [_I64] * 3 + [_I, _I, _I, _P]
_lib.ssm_causal_conv1d_update.restype = _I
_lib.ssm_ssd_scan_fwd.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 6 + [_I, _I, _P]
_lib.ssm_ssd_scan_fwd.restype = _I
_lib.ssm_ssd_chunk_len.argtypes = []
_lib.ssm_ssd_chunk_len.restype = _I64
_lib.ssm_scan_fwd_dir.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 4 + [_I, _I64, _I64, _I, _I, _I, _P]
_lib.ssm_scan_fwd_dir.restype = _I
_lib.ssm_scan_fwd_dir_ws.argtypes = [_P] * 8 + [_I, _P, _P, _P] + [_I64] * 4 + [_I, _I64, _I64, _I, _I, _I, _P, _SZ, _P]
_lib.ssm_scan_fwd_dir_ws.restype = _I
_lib.ssm_scan_dir_workspace_size.argtypes = [_I64] * 4 + [_I, _I]
_lib.ssm_scan_dir_workspace_size.restype = _SZ
_lib.ssm_device_status.argtypes = [_I, _P]
_lib.ssm_device_status.restype = _I
_lib.ssm_test_math.argtypes = [_I, _P, _P, _I64, _P]
_lib.ssm_test_math.restype = _I

SSM_F32, SSM_BF16 = 0, 1
ALGOS = {"auto": 0, "thread": 1, "warpscan": 2, "lookback": 3}
SSM_ERR_DIM = -2
SSM_ERR_LOOKBACK_TIMEOUT = -7
SSM_ERR_SCRATCH_LIMIT = -11
SSM_ERR_WIDTH = -12
SSM_ERR_SHAPE = -13
SSM_ERR_WAIT_TIMEOUT = -14
SSM_ERR_ORDER = -15
ORDERS = {"raster": 0, "reverse": 1, "columns": 2, "columns_reverse": 3}
STATIC_SCRATCH_BYTES = 4 << 20   # SSM_STATIC_SCRATCH_BYTES

# the C ABI entry-point names, as declared in include/ssm_scan.h
EXPORTS = ("ssm_abi_version", "ssm_status_string", "ssm_scan_workspace_size", "ssm_scan_fwd",
           "ssm_scan_fwd_algo", "ssm_scalar_scan_fwd", "ssm_state_update",
           "ssm_test_lookback_timeout", "ssm_query_status", "ssm_scan_fwd_lookback_static",
           "ssm_causal_conv1d_fwd", "ssm_causal_conv1d_update", "ssm_scan_bwd_workspace_size",
           "ssm_scan_bwd", "ssm_ssd_scan_fwd", "ssm_ssd_chunk_len", "ssm_device_status", "ssm_scan_fwd_dir",
           "ssm_test_math", "ssm_test_ssd_wait_fault", "ssm_ssd_scan_fwd_ws", "ssm_ssd_workspace_size",
           "ssm_test_serial_handover_timeout", "ssm_scan_fwd_dir_ws", "ssm_scan_dir_workspace_size")
MATH = {"exp": 0, "log1p01": 1, "expm1": 2, "softplus": 3, "silu": 4, "softplus_sfu": 5, "silu_sfu": 6}


class SSMError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(_lib.ssm_status_string(status).decode())


def _check(status: int):
    if status != 0:
        raise SSMError(status)


def abi_version() -> int:
    return _lib.ssm_abi_version()


def status_string(status: int) -> str:
    return _lib.ssm_status_string(status).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SSM_F32
    if t == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported dtype {t}: use torch.float32 or torch.bfloat16")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr() or None


def _f32(t, shape, name):
    if t is None:
        return None
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _out(t, shape, name, dtypes=(torch.float32, torch.bfloat16), device=None):
    """A caller-provided output: the library writes exactly `shape` elements of its
    dtype there, so a smaller tensor (or another dtype's element size) would be
    overrun on the device. Checked before any call."""
    if t is None:
        return None
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {[str(d) for d in dtypes]}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the inputs on {device}")
    return t


def _same(ref, named_shapes):
    for name, t, shp in named_shapes:
        if t is None:
            continue
        if t.dtype != ref.dtype:
            raise TypeError(f"{name} must have dtype {ref.dtype}")
        if tuple(t.shape) != tuple(shp):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shp)}")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def workspace_size(batch: int, dim: int, seqlen: int, dstate: int) -> int:
    return int(_lib.ssm_scan_workspace_size(batch, dim, seqlen, dstate))


def alloc_workspace(batch: int, dim: int, seqlen: int, dstate: int, device=None) -> torch.Tensor:
    n = workspace_size(batch, dim, seqlen, dstate)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, *,
             out_dtype=None, return_last_state=True, algo="auto", workspace=None, y=None,
             h_last=None):
    """Selective scan forward. u, delta, z: (batch, dim, L); B, C: (batch, N, L);
    A: (dim, N) fp32; D, delta_bias: (dim,) fp32; h0: (batch, dim, N) fp32.
    Returns (y (batch, dim, L), h_last (batch, dim, N) fp32 or None)."""
    bt, dim, L = u.shape
    N = A.shape[1]
    in_code = _dtype_code(u.dtype)
    _same(u, (("delta", delta, u.shape), ("B", B, (bt, N, L)), ("C", C, (bt, N, L)), ("z", z, u.shape)))
    _f32(A, (dim, N), "A"); _f32(D, (dim,), "D"); _f32(delta_bias, (dim,), "delta_bias")
    _f32(h0, (bt, dim, N), "h0")
    if y is None:
        y = torch.empty((bt, dim, L), dtype=out_dtype or u.dtype, device=u.device)
    if h_last is None and return_last_state:
        h_last = torch.empty((bt, dim, N), dtype=torch.float32, device=u.device)
    _out(y, (bt, dim, L), "y", device=u.device)
    _out(h_last, (bt, dim, N), "h_last", (torch.float32,), u.device)
    if workspace is None and algo in ("auto", "thread", "lookback"):
        workspace = alloc_workspace(bt, dim, L, N, u.device)
    status = _lib.ssm_scan_fwd_algo(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        int(bool(softplus)), _ptr(h0), _ptr(y), _ptr(h_last), bt, dim, L, N, in_code,
        _dtype_code(y.dtype), _ptr(workspace), _nbytes(workspace), ALGOS[algo], _stream())
    _check(status)
    return y, h_last


def scan_fwd_dir(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, *,
                 order="raster", rows=0, cols=0, zoh=False, out_dtype=None, return_last_state=True, y=None,
                 h_last=None, workspace="auto"):
    """Selective scan along a traversal order ("raster", "reverse", "columns",
    "columns_reverse" of a rows x cols image stored in raster order), outputs in
    raster order; zoh selects the zero-order-hold input matrix. Shapes as scan_fwd.
    workspace: a uint8 device tensor (ssm_scan_dir_workspace_size bytes), "auto" to
    allocate one (every walk may then take the time-serial or look-back algorithm, the
    column orders through transposed copies), or None for the warp-scan form alone."""
    bt, dim, L = u.shape
    N = A.shape[1]
    in_code = _dtype_code(u.dtype)
    _same(u, (("delta", delta, u.shape), ("B", B, (bt, N, L)), ("C", C, (bt, N, L)), ("z", z, u.shape)))
    _f32(A, (dim, N), "A"); _f32(D, (dim,), "D"); _f32(delta_bias, (dim,), "delta_bias")
    _f32(h0, (bt, dim, N), "h0")
    if y is None:
        y = torch.empty((bt, dim, L), dtype=out_dtype or u.dtype, device=u.device)
    if h_last is None and return_last_state:
        h_last = torch.empty((bt, dim, N), dtype=torch.float32, device=u.device)
    _out(y, (bt, dim, L), "y", device=u.device)
    _out(h_last, (bt, dim, N), "h_last", (torch.float32,), u.device)
    order_code = ORDERS[order] if isinstance(order, str) else int(order)
    if workspace is None:
        status = _lib.ssm_scan_fwd_dir(
            _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(softplus)), _ptr(h0), _ptr(y), _ptr(h_last), bt, dim, L, N, order_code, int(rows), int(cols),
            int(bool(zoh)), in_code, _dtype_code(y.dtype), _stream())
    else:
        if isinstance(workspace, str):
            n = _lib.ssm_scan_dir_workspace_size(bt, dim, L, N, in_code, _dtype_code(y.dtype))
            workspace = torch.empty(n, dtype=torch.uint8, device=u.device)
        status = _lib.ssm_scan_fwd_dir_ws(
            _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(softplus)), _ptr(h0), _ptr(y), _ptr(h_last), bt, dim, L, N, order_code, int(rows), int(cols),
            int(bool(zoh)), in_code, _dtype_code(y.dtype), _ptr(workspace), _nbytes(workspace), _stream())
    _check(status)
    return y, h_last


def scalar_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, *,
                    out_dtype=None, return_last_state=True, workspace=None, y=None, h_last=None):
    """d_state = 1 scan. u, delta, z: (batch, dim, L); A: (dim,) fp32; B, C: (batch, L);
    h0: (batch, dim) fp32. Returns (y, h_last (batch, dim))."""
    bt, dim, L = u.shape
    in_code = _dtype_code(u.dtype)
    _same(u, (("delta", delta, u.shape), ("B", B, (bt, L)), ("C", C, (bt, L)), ("z", z, u.shape)))
    _f32(A, (dim,), "A"); _f32(D, (dim,), "D"); _f32(delta_bias, (dim,), "delta_bias")
    _f32(h0, (bt, dim), "h0")
    if y is None:
        y = torch.empty((bt, dim, L), dtype=out_dtype or u.dtype, device=u.device)
    if h_last is None and return_last_state:
        h_last = torch.empty((bt, dim), dtype=torch.float32, device=u.device)
    _out(y, (bt, dim, L), "y", device=u.device)
    _out(h_last, (bt, dim), "h_last", (torch.float32,), u.device)
    if workspace is None:
        workspace = alloc_workspace(bt, dim, L, 1, u.device)
    status = _lib.ssm_scalar_scan_fwd(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        int(bool(softplus)), _ptr(h0), _ptr(y), _ptr(h_last), bt, dim, L, in_code,
        _dtype_code(y.dtype), _ptr(workspace), _nbytes(workspace), _stream())
    _check(status)
    return y, h_last


def state_update(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *,
                 out_dtype=None, y=None):
    """One decode token; `state` (batch, dim, N) fp32 is updated in place.
    x, delta, z: (batch, dim); B, C: (batch, N). Returns y (batch, dim)."""
    bt, dim, N = state.shape
    _f32(state, (bt, dim, N), "state")
    in_code = _dtype_code(x.dtype)
    _same(x, (("delta", delta, (bt, dim)), ("B", B, (bt, N)), ("C", C, (bt, N)), ("z", z, (bt, dim))))
    _f32(A, (dim, N), "A"); _f32(D, (dim,), "D"); _f32(delta_bias, (dim,), "delta_bias")
    if y is None:
        y = torch.empty((bt, dim), dtype=out_dtype or x.dtype, device=x.device)
    _out(y, (bt, dim), "y", device=x.device)
    status = _lib.ssm_state_update(
        _ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(delta_bias), int(bool(softplus)), _ptr(y), bt, dim, N, in_code, _dtype_code(y.dtype),
        _stream())
    _check(status)
    return y


def scan_fwd_lookback_static(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, *,
                             y, h_last=None) -> int:
    """The look-back scan on the library's own fixed scratch area
    (ssm_scan_fwd_lookback_static): for callers that cannot allocate device memory or
    pass a workspace. The caller provides y (and h_last) preallocated; this function
    allocates nothing. Returns the ABI status (0 on success, SSM_ERR_SCRATCH_LIMIT
    when the sizes need more than STATIC_SCRATCH_BYTES of scratch)."""
    bt, dim, L = u.shape
    N = A.shape[1]
    in_code = _dtype_code(u.dtype)
    _same(u, (("delta", delta, u.shape), ("B", B, (bt, N, L)), ("C", C, (bt, N, L)), ("z", z, u.shape)))
    _f32(A, (dim, N), "A"); _f32(D, (dim,), "D"); _f32(delta_bias, (dim,), "delta_bias")
    _f32(h0, (bt, dim, N), "h0")
    _out(y, (bt, dim, L), "y", device=u.device)
    _out(h_last, (bt, dim, N), "h_last", (torch.float32,), u.device)
    return int(_lib.ssm_scan_fwd_lookback_static(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        int(bool(softplus)), _ptr(h0), _ptr(y), _ptr(h_last), bt, dim, L, N, in_code, _dtype_code(y.dtype),
        _stream()))


def scan_bwd_workspace_size(batch: int, dim: int, seqlen: int, dstate: int) -> int:
    return int(_lib.ssm_scan_bwd_workspace_size(batch, dim, seqlen, dstate))


def scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None, *, dout,
             dh_last=None, workspace=None, want_dh0=True):
    """Backward of scan_fwd for dout = dl/dy (batch, dim, L) and dh_last = dl/dh_last.
    Returns a dict: du, ddelta, dz (None without z) in u's dtype; dA, dB, dC, dD (None
    without D), ddelta_bias (None without delta_bias), dh0 (None unless want_dh0) fp32."""
    bt, dim, L = u.shape
    N = A.shape[1]
    in_code = _dtype_code(u.dtype)
    _same(u, (("delta", delta, u.shape), ("B", B, (bt, N, L)), ("C", C, (bt, N, L)), ("z", z, u.shape)))
    _f32(A, (dim, N), "A"); _f32(D, (dim,), "D"); _f32(delta_bias, (dim,), "delta_bias")
    _f32(h0, (bt, dim, N), "h0"); _f32(dh_last, (bt, dim, N), "dh_last")
    if tuple(dout.shape) != (bt, dim, L):
        raise ValueError("dout must have u's shape")
    dev = u.device
    f32 = torch.float32
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dz": torch.empty_like(u) if z is not None else None,
         "dA": torch.empty((dim, N), dtype=f32, device=dev), "dB": torch.empty((bt, N, L), dtype=f32, device=dev),
         "dC": torch.empty((bt, N, L), dtype=f32, device=dev),
         "dD": torch.empty((dim,), dtype=f32, device=dev) if D is not None else None,
         "ddelta_bias": torch.empty((dim,), dtype=f32, device=dev) if delta_bias is not None else None,
         "dh0": torch.empty((bt, dim, N), dtype=f32, device=dev) if want_dh0 else None}
    if workspace is None:
        need = scan_bwd_workspace_size(bt, dim, L, N)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    status = _lib.ssm_scan_bwd(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus)),
        _ptr(h0), _ptr(dout), _ptr(dh_last), _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]),
        _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]), bt, dim, L, N,
        in_code, _dtype_code(dout.dtype), _ptr(workspace), _nbytes(workspace), _stream())
    _check(status)
    return g


def causal_conv1d_fwd(x, weight, bias=None, conv_state=None, silu=True, *, out_dtype=None, out=None,
                      conv_state_out=None, return_state=True):
    """Causal depthwise conv1d (+ silu) over x (batch, dim, L): weight (dim, width) fp32,
    bias (dim,), conv_state (batch, dim, width-1) fp32 = the inputs before x (zeros when
    None). Returns (out (batch, dim, L), conv_state_out (batch, dim, width-1) fp32, or
    None when return_state is False and no conv_state_out is given)."""
    bt, dim, L = x.shape
    width = weight.shape[1]
    _f32(weight, (dim, width), "weight"); _f32(bias, (dim,), "bias")
    _f32(conv_state, (bt, dim, width - 1), "conv_state")
    if out is None:
        out = torch.empty((bt, dim, L), dtype=out_dtype or x.dtype, device=x.device)
    if conv_state_out is None and return_state:
        conv_state_out = torch.empty((bt, dim, width - 1), dtype=torch.float32, device=x.device)
    _out(out, (bt, dim, L), "out", device=x.device)
    _out(conv_state_out, (bt, dim, width - 1), "conv_state_out", (torch.float32,), x.device)
    status = _lib.ssm_causal_conv1d_fwd(
        _ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state), _ptr(conv_state_out), _ptr(out), bt, dim, L,
        width, int(bool(silu)), _dtype_code(x.dtype), _dtype_code(out.dtype), _stream())
    _check(status)
    return out, conv_state_out


def causal_conv1d_update(conv_state, x, weight, bias=None, silu=True, *, out_dtype=None, out=None):
    """One decode token of the conv: conv_state (batch, dim, width-1) fp32 is updated in
    place; x (batch, dim). Returns out (batch, dim)."""
    bt, dim = x.shape
    width = weight.shape[1]
    _f32(weight, (dim, width), "weight"); _f32(bias, (dim,), "bias")
    _f32(conv_state, (bt, dim, width - 1), "conv_state")
    if out is None:
        out = torch.empty((bt, dim), dtype=out_dtype or x.dtype, device=x.device)
    _out(out, (bt, dim), "out", device=x.device)
    status = _lib.ssm_causal_conv1d_update(
        _ptr(conv_state), _ptr(x), _ptr(weight), _ptr(bias), _ptr(out), bt, dim, width, int(bool(silu)),
        _dtype_code(x.dtype), _dtype_code(out.dtype), _stream())
    _check(status)
    return out


def ssd_workspace_size(batch: int, nheads: int, dstate: int) -> int:
    return int(_lib.ssm_ssd_workspace_size(batch, nheads, dstate))


def ssd_scan_fwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, softplus=True, h0=None, *,
                 out_dtype=None, y=None, h_last=None, return_last_state=True, workspace="auto"):
    """Mamba-2 SSD scan on the tensor cores. x, z: (batch, L, nheads, 64) bf16; dt: (batch,
    L, nheads) bf16; A, D, dt_bias: (nheads,) fp32; B, C: (batch, L, ngroups, dstate) bf16
    with dstate 64 or 128; h0: (batch, nheads, 64, dstate) fp32. workspace: a uint8 device
    tensor (ssd_workspace_size bytes enable the work-balanced launch), "auto" to allocate
    one, or None for the one-sequence-per-CTA launch. Returns (y, h_last)."""
    bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _same(x, [("dt", dt, (bt, L, H)), ("B", B, (bt, L, G, N)), ("C", C, (bt, L, G, N)), ("z", z, (bt, L, H, P))])
    _f32(A, (H,), "A"); _f32(D, (H,), "D"); _f32(dt_bias, (H,), "dt_bias"); _f32(h0, (bt, H, P, N), "h0")
    if y is None:
        y = torch.empty((bt, L, H, P), dtype=out_dtype or x.dtype, device=x.device)
    if h_last is None and return_last_state:
        h_last = torch.empty((bt, H, P, N), dtype=torch.float32, device=x.device)
    _out(y, (bt, L, H, P), "y", device=x.device)
    _out(h_last, (bt, H, P, N), "h_last", (torch.float32,), x.device)
    if isinstance(workspace, str):
        workspace = torch.empty(ssd_workspace_size(bt, H, N), dtype=torch.uint8, device=x.device)
    status = _lib.ssm_ssd_scan_fwd_ws(
        _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias), int(bool(softplus)),
        _ptr(h0), _ptr(y), _ptr(h_last), bt, L, H, P, G, N, _dtype_code(x.dtype), _dtype_code(y.dtype),
        _ptr(workspace), _nbytes(workspace), _stream())
    _check(status)
    return y, h_last


def ssd_chunk_len() -> int:
    return int(_lib.ssm_ssd_chunk_len())


def device_status(clear: bool = True) -> int:
    """SSM_ERR_WAIT_TIMEOUT if an SSD launch recorded an exhausted wait (syncs the stream)."""
    return int(_lib.ssm_device_status(int(bool(clear)), _stream()))


def query_status(workspace) -> int:
    """Device status word of the last look-back scan that used `workspace` (syncs the stream)."""
    return int(_lib.ssm_query_status(_ptr(workspace), _nbytes(workspace), _stream()))


def test_math(fn: str, x: torch.Tensor) -> torch.Tensor:
    """Evaluates one device math helper (ssm_test_math) on fp32 CUDA values x."""
    if x.dtype != torch.float32:
        raise TypeError("x must be float32")
    x = x.contiguous()
    y = torch.empty_like(x)
    _check(_lib.ssm_test_math(MATH[fn], _ptr(x), _ptr(y), x.numel(), _stream()))
    return y


def run_ssd_wait_fault_test(x, dt, A, B, C, y, wait_limit: int, withhold_arrive: bool, workspace=None,
                            drop_ticket: int = -1) -> int:
    """Runs the SSD kernel's failure paths (see ssm_test_ssd_wait_fault); returns the launch status."""
    bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _same(x, [("dt", dt, (bt, L, H)), ("B", B, (bt, L, G, N)), ("C", C, (bt, L, G, N))])
    _f32(A, (H,), "A")
    _out(y, (bt, L, H, P), "y", (torch.bfloat16,), x.device)
    return int(_lib.ssm_test_ssd_wait_fault(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(y), bt, L, H, G, N,
                                            int(wait_limit), int(bool(withhold_arrive)), _ptr(workspace),
                                            _nbytes(workspace), int(drop_ticket), _stream()))


def run_serial_handover_timeout_test(u, delta, A, B, C, y, workspace, drop_ticket: int, spin_limit: int) -> int:
    """Runs the balanced time-serial scan with one ticket withholding its state
    (see ssm_test_serial_handover_timeout); returns the launch status."""
    bt, dim, L = u.shape
    return int(_lib.ssm_test_serial_handover_timeout(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(y), bt, dim, L, A.shape[1], _dtype_code(u.dtype),
        _ptr(workspace), _nbytes(workspace), int(drop_ticket), int(spin_limit), _stream()))


def run_lookback_timeout_test(u, delta, A, B, C, y, workspace, drop_segment: int, spin_limit: int) -> int:
    """Runs the look-back error path (see ssm_test_lookback_timeout); returns the launch status."""
    bt, dim, L = u.shape
    return int(_lib.ssm_test_lookback_timeout(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(y), bt, dim, L, A.shape[1],
        _dtype_code(u.dtype), _ptr(workspace), _nbytes(workspace), drop_segment, spin_limit,
        _stream()))
