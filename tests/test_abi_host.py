"""CPU-only checks of the C ABI library: it loads, exports every entry point the
header declares, and its host-side logic (argument validation, workspace sizing)
answers without touching a GPU. No kernel is launched here: every call below is
rejected by validation before any CUDA call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^SSM_API\s+[\w\s\*]+?\b(ssm_\w+)\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def ssm():
    import selective_state_space_121_b300 as m
    return m


def test_header_declares_entry_points():
    names = _declared()
    for need in ("ssm_scan_fwd", "ssm_scalar_scan_fwd", "ssm_state_update", "ssm_scan_workspace_size",
                 "ssm_query_status"):
        assert need in names


def test_library_exports_every_declared_symbol(ssm):
    lib = ctypes.CDLL(ssm.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in ssm_scan.h but not exported"
    assert sorted(ssm.EXPORTS) == _declared()


def test_abi_version_matches_header(ssm):
    v = int(re.search(r"#define SSM_SCAN_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert ssm.abi_version() == v


def test_status_strings(ssm):
    for code in range(0, -16, -1):
        assert ssm.status_string(code).startswith("SSM_")
    assert not ssm.status_string(-99).startswith("SSM_")


def test_workspace_size(ssm):
    # at least the 16-byte status header, and grows with the look-back descriptor count
    assert ssm.workspace_size(8, 1536, 2048, 16) >= 16
    small = ssm.workspace_size(1, 16, 1 << 17, 16)
    big = ssm.workspace_size(1, 64, 1 << 17, 16)
    assert big > small > 16
    assert ssm.workspace_size(-1, 4, 4, 16) == 16          # invalid sizes: header only
    assert ssm.workspace_size(1, 4, 4, 3) == 16
    assert ssm.workspace_size(2, 0, 16, 16) >= 16          # empty problems do not divide by zero
    assert ssm.workspace_size(0, 4, 16, 16) >= 16


# argument validation, all rejected before any CUDA call ------------------------------
FAKE = 0x10000          # non-null, 64 KiB aligned: never dereferenced by the host


def _scan(ssm, **kw):
    args = dict(u=FAKE, delta=FAKE * 2, A=FAKE * 3, B=FAKE * 4, C=FAKE * 5, D=None, z=None, bias=None,
                softplus=1, h0=None, y=FAKE * 6, h_last=None, batch=2, dim=4, L=8, N=16, idt=1, odt=1,
                ws=None, wsb=0, algo=2)
    args.update(kw)
    return ssm._lib.ssm_scan_fwd_algo(args["u"], args["delta"], args["A"], args["B"], args["C"], args["D"],
                                      args["z"], args["bias"], args["softplus"], args["h0"], args["y"],
                                      args["h_last"], args["batch"], args["dim"], args["L"], args["N"],
                                      args["idt"], args["odt"], args["ws"], args["wsb"], args["algo"], None)


def test_validation_errors(ssm):
    assert _scan(ssm, idt=7) == -3
    assert _scan(ssm, odt=-1) == -3
    assert _scan(ssm, batch=-1) == -2
    assert _scan(ssm, L=-5) == -2
    assert _scan(ssm, N=3) == -8
    assert _scan(ssm, N=32) == -8
    assert _scan(ssm, algo=9) == -10
    assert _scan(ssm, u=None) == -1
    assert _scan(ssm, A=None) == -1
    assert _scan(ssm, C=None) == -1
    assert _scan(ssm, y=FAKE + 1) == -4                     # bf16 output needs 2-byte alignment
    assert _scan(ssm, D=FAKE * 7 + 2) == -4                 # fp32 needs 4
    assert _scan(ssm, y=FAKE + 16) == -9                    # y overlaps u
    assert _scan(ssm, h_last=FAKE * 3) == -9                # h_last over A
    assert _scan(ssm, h0=FAKE * 8, h_last=FAKE * 8 + 4) == -9   # h_last partly over h0
    assert _scan(ssm, batch=1 << 40, dim=1 << 30) == -2     # size overflow
    # the look-back needs a workspace: a 16-byte header plus, per (channel, segment),
    # a 16-byte descriptor per state -- here 2 x 4 channels, one segment, d_state 16
    assert _scan(ssm, algo=3, ws=None, wsb=0) == -5
    lb_need = 16 + 2 * 4 * 16 * 16
    assert _scan(ssm, algo=3, ws=FAKE * 9, wsb=lb_need - 1) == -5
    # the advertised size covers every algorithm, the look-back's included
    assert ssm.workspace_size(2, 4, 8, 16) >= lb_need


def test_state_update_validation(ssm):
    f = ssm._lib.ssm_state_update

    def call(**kw):
        a = dict(state=FAKE, x=FAKE * 2, delta=FAKE * 3, A=FAKE * 4, B=FAKE * 5, C=FAKE * 6, D=None, z=None,
                 bias=None, sp=1, y=FAKE * 7, batch=2, dim=4, N=16, idt=1, odt=1)
        a.update(kw)
        return f(a["state"], a["x"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["sp"],
                 a["y"], a["batch"], a["dim"], a["N"], a["idt"], a["odt"], None)
    assert call(idt=5) == -3
    assert call(N=5) == -8
    assert call(batch=-2) == -2
    assert call(state=None) == -1
    assert call(state=FAKE + 4) == -4          # 16-byte vector state access for N >= 4
    assert call(y=FAKE + 8) == -9              # y inside the state
    assert call(x=FAKE + 64) == -9             # state overlaps x


def test_query_status_rejects_small_workspace(ssm):
    assert ssm._lib.ssm_query_status(None, 0, None) == -5
    assert ssm._lib.ssm_query_status(FAKE, 8, None) == -5


def test_conv_validation(ssm):
    f = ssm._lib.ssm_causal_conv1d_fwd

    def call(**kw):
        a = dict(x=FAKE, w=FAKE * 2, bias=None, sin=None, sout=None, out=FAKE * 3, batch=2, dim=4, L=8, width=4,
                 silu=1, idt=1, odt=1)
        a.update(kw)
        return f(a["x"], a["w"], a["bias"], a["sin"], a["sout"], a["out"], a["batch"], a["dim"], a["L"],
                 a["width"], a["silu"], a["idt"], a["odt"], None)
    assert call(idt=3) == -3
    assert call(width=0) == -12
    assert call(width=5) == -12
    assert call(L=-1) == -2
    assert call(x=None) == -1
    assert call(w=None) == -1
    assert call(out=FAKE + 1) == -4                   # bf16 output needs 2-byte alignment
    assert call(sin=FAKE * 4 + 2) == -4               # fp32 state needs 4
    assert call(out=FAKE + 32) == -9                  # out overlaps x
    assert call(sout=FAKE * 2) == -9                  # state out over the weights
    assert call(sin=FAKE * 4, sout=FAKE * 4 + 4) == -9  # partly over the incoming state
    assert call(batch=1 << 40, dim=1 << 30) == -2

    g = ssm._lib.ssm_causal_conv1d_update

    def upd(**kw):
        a = dict(st=FAKE, x=FAKE * 2, w=FAKE * 3, bias=None, out=FAKE * 4, batch=2, dim=4, width=4, silu=1,
                 idt=1, odt=1)
        a.update(kw)
        return g(a["st"], a["x"], a["w"], a["bias"], a["out"], a["batch"], a["dim"], a["width"], a["silu"],
                 a["idt"], a["odt"], None)
    assert upd(width=9) == -12
    assert upd(st=None) == -1
    assert upd(out=FAKE + 8) == -9                    # out inside the state
    assert upd(x=FAKE + 16) == -9                     # state overlaps x
    assert upd(st=FAKE + 2) == -4


def test_ssd_validation(ssm):
    """Argument errors of ssm_ssd_scan_fwd come back before any launch (no GPU needed)."""
    f = ssm._lib.ssm_ssd_scan_fwd

    def call(**kw):
        a = dict(x=FAKE, dt=FAKE * 2, A=FAKE * 3, B=FAKE * 4, C=FAKE * 5, D=None, z=None, bias=None, sp=1,
                 h0=None, y=FAKE * 6, hl=None, batch=2, L=8, H=4, P=64, G=1, N=128, idt=1, odt=1)
        a.update(kw)
        return f(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["sp"], a["h0"], a["y"],
                 a["hl"], a["batch"], a["L"], a["H"], a["P"], a["G"], a["N"], a["idt"], a["odt"], None)
    assert call(idt=0) == -3                           # fp32 inputs are not taken
    assert call(odt=5) == -3
    assert call(P=32) == -13
    assert call(N=16) == -13
    assert call(H=3, G=2) == -13                       # heads not a multiple of groups
    assert call(L=-1) == -2
    assert call(x=None) == -1
    assert call(A=None) == -1
    assert call(x=FAKE + 8) == -4                      # x rows need 16-byte alignment
    assert call(B=FAKE * 4 + 2) == -4
    assert call(hl=FAKE * 7 + 2) == -4
    assert call(y=FAKE + 64) == -9                     # y overlaps x
    assert call(hl=FAKE * 3) == -9                     # final state over A
    assert call(h0=FAKE * 7, hl=FAKE * 7 + 4) == -9    # partly over the initial state
    assert call(batch=1 << 40, H=1 << 30) == -2
    assert ssm._lib.ssm_ssd_chunk_len() == 128


def test_scan_dir_validation(ssm):
    """Argument errors of ssm_scan_fwd_dir come back before any launch (no GPU needed)."""
    f = ssm._lib.ssm_scan_fwd_dir

    def call(**kw):
        a = dict(u=FAKE, d=FAKE * 2, A=FAKE * 3, B=FAKE * 4, C=FAKE * 5, D=None, z=None, bias=None, sp=1, h0=None,
                 y=FAKE * 6, hl=None, batch=2, dim=4, L=12, N=16, order=2, rows=3, cols=4, zoh=0, idt=1, odt=1)
        a.update(kw)
        return f(a["u"], a["d"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["sp"], a["h0"], a["y"],
                 a["hl"], a["batch"], a["dim"], a["L"], a["N"], a["order"], a["rows"], a["cols"], a["zoh"], a["idt"],
                 a["odt"], None)
    assert call(order=4) == -15
    assert call(order=-1) == -15
    assert call(order=2, rows=5, cols=4) == -15        # rows * cols != seqlen
    assert call(order=3, rows=0, cols=12) == -15
    assert call(N=3) == -8
    assert call(idt=7) == -3
    assert call(u=None) == -1
    assert call(y=FAKE + 16) == -9                     # y overlaps u
    assert call(batch=1 << 40, dim=1 << 30) == -2


def test_outputs_are_checked_before_any_call(ssm):
    """Every entry point that takes caller-provided outputs checks their shape and dtype
    before calling the library: the library writes the full output shape, so a smaller
    tensor would be overrun on the device. CPU tensors suffice here: the checks raise
    before any pointer is taken."""
    import torch
    bt, dim, L, N = 2, 8, 16, 4
    f32, bf = torch.float32, torch.bfloat16
    u = torch.zeros(bt, dim, L, dtype=bf)
    Bm = torch.zeros(bt, N, L, dtype=bf)
    A = torch.zeros(dim, N, dtype=f32)
    short_y = torch.zeros(bt, dim, L - 1, dtype=bf)
    with pytest.raises(ValueError, match="y has shape"):
        ssm.scan_fwd_lookback_static(u, u, A, Bm, Bm, y=short_y)
    with pytest.raises(TypeError, match="y must have dtype"):
        ssm.scan_fwd_lookback_static(u, u, A, Bm, Bm, y=torch.zeros(bt, dim, L, dtype=torch.float16))
    with pytest.raises(ValueError, match="h_last has shape"):
        ssm.scan_fwd_lookback_static(u, u, A, Bm, Bm, y=torch.zeros(bt, dim, L, dtype=bf),
                                     h_last=torch.zeros(bt, dim, N - 1, dtype=f32))
    with pytest.raises(ValueError, match="y has shape"):
        ssm.scan_fwd(u, u, A, Bm, Bm, y=short_y)
    with pytest.raises(ValueError, match="h_last has shape"):
        ssm.scan_fwd(u, u, A, Bm, Bm, y=torch.zeros(bt, dim, L, dtype=bf), h_last=torch.zeros(bt, dim, 1))
    with pytest.raises(ValueError, match="y has shape"):
        ssm.scan_fwd_dir(u, u, A, Bm, Bm, y=short_y)
    with pytest.raises(ValueError, match="y has shape"):
        ssm.scalar_scan_fwd(u, u, torch.zeros(dim), torch.zeros(bt, L, dtype=bf), torch.zeros(bt, L, dtype=bf),
                            y=short_y)
    state = torch.zeros(bt, dim, N, dtype=f32)
    x = torch.zeros(bt, dim, dtype=bf)
    with pytest.raises(ValueError, match="y has shape"):
        ssm.state_update(state, x, x, A, torch.zeros(bt, N, dtype=bf), torch.zeros(bt, N, dtype=bf),
                         y=torch.zeros(bt, dim - 1, dtype=bf))
    w = torch.zeros(dim, 4, dtype=f32)
    with pytest.raises(ValueError, match="out has shape"):
        ssm.causal_conv1d_fwd(u, w, out=short_y)
    with pytest.raises(ValueError, match="out has shape"):
        ssm.causal_conv1d_update(torch.zeros(bt, dim, 3), x, w, out=torch.zeros(bt, 1, dtype=bf))
    xs = torch.zeros(1, 16, 2, 64, dtype=bf)
    Bs = torch.zeros(1, 16, 1, 64, dtype=bf)
    with pytest.raises(ValueError, match="y has shape"):
        ssm.ssd_scan_fwd(xs, torch.zeros(1, 16, 2, dtype=bf), torch.zeros(2), Bs, Bs,
                         y=torch.zeros(1, 15, 2, 64, dtype=bf))


def test_probe_library_exports_its_declared_symbol():
    """libssmprobe.so (the pipe-throughput probes behind bench.py --only pipes) exports
    every entry point include/ssm_probe.h declares."""
    probe_h = os.path.join(ROOT, "include", "ssm_probe.h")
    names = sorted(set(re.findall(r"^SSM_PROBE_API\s+[\w\s\*]+?\b(ssm_\w+)\(", open(probe_h).read(), flags=re.M)))
    assert names == ["ssm_probe_pipe_rate"]
    lib = ctypes.CDLL(os.path.join(ROOT, "selective_state_space_121_b300", "libssmprobe.so"))
    for name in names:
        assert hasattr(lib, name), f"{name} declared in ssm_probe.h but not exported"
