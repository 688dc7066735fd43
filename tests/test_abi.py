"""The C-ABI library loads, exports every symbol include/kdn.h declares, and
rejects invalid arguments on the host before any launch (CPU only: none of
these calls reaches a CUDA API)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_symbols():
    names = []
    for h in HEADERS:
        text = open(h).read()
        names += re.findall(r"KDN_API\s+[\w\s\*]+?\b(kdn_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from bayesian_scan_gb300 import build
    build.build()
    from bayesian_scan_gb300 import kdn
    return kdn.lib


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("kdn_diag_scan_fwd", "kdn_mobius_scan", "kdn_status_string",
                     "kdn_get_device_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    from bayesian_scan_gb300 import kdn
    for s in (0, -1, -2, -3, -4, -5):
        assert kdn.status_string(s).startswith("KDN_")
    assert "unknown" in kdn.status_string(7)
    assert kdn.version().startswith("kdn ")


FAKE = 0x10000  # 16-byte aligned fake address: only reached by host checks


def _diag(lib, q=FAKE, k=FAKE, v=FAKE, beta=FAKE, d=FAKE, A=FAKE, I_prior=1.0, I0=None,
          mu0=None, out=FAKE, fs=None, B=1, H=1, T=8, dk=16, dv=16, dtype=1):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kdn_diag_scan_fwd(vp(q), vp(k), vp(v), vp(beta), vp(d), vp(A), I_prior, vp(I0),
                                 vp(mu0), vp(out), vp(fs), B, H, T, dk, dv, dtype, None)


@pytest.mark.parametrize("field", ["q", "k", "v", "beta", "d", "A", "out"])
def test_diag_null_pointer(lib, field):
    assert _diag(lib, **{field: None}) == -1
    # with T = 0 the token tensors are not read, but sizes are still checked
    assert _diag(lib, T=0, dk=24, **{field: None}) == -2


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), -1), (dict(H=0), -1), (dict(T=-1), -1), (dict(B=-3), -1),
    (dict(dk=8), -2), (dict(dv=256), -2), (dict(dk=48), -2), (dict(dtype=2), -2),
    (dict(q=FAKE + 8), -1), (dict(v=FAKE + 4), -1), (dict(out=FAKE + 2), -1),
    (dict(I0=FAKE + 8), -1), (dict(mu0=FAKE + 1), -1), (dict(fs=FAKE + 12), -1),
    (dict(A=FAKE + 2), -1), (dict(d=FAKE + 1), -1),
    (dict(B=1 << 30, H=1 << 30, T=1 << 30), -1),
])
def test_diag_rejects(lib, kw, status):
    assert _diag(lib, **kw) == status


def _fused(lib, ma=FAKE, mb=FAKE, mc=FAKE, md=FAKE, l0=FAKE, lout=FAKE, **kw):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, d=FAKE, A=FAKE, I0=None, mu0=None, out=FAKE,
             fs=None, B=1, H=1, T=8, dk=16, dv=16, dtype=1)
    a.update(kw)
    return lib.kdn_diag_mobius_scan_fwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["d"]),
                                        vp(a["A"]), 1.0, vp(a["I0"]), vp(a["mu0"]), vp(a["out"]),
                                        vp(a["fs"]), vp(ma), vp(mb), vp(mc), vp(md), vp(l0), vp(lout),
                                        a["B"], a["H"], a["T"], a["dk"], a["dv"], a["dtype"], None)


@pytest.mark.parametrize("field", ["ma", "mb", "mc", "md", "l0", "lout"])
def test_fused_null_moebius_pointer(lib, field):
    assert _fused(lib, **{field: None}) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(B=0), -1), (dict(dk=8), -2), (dict(dtype=3), -2),
    (dict(ma=FAKE + 2), -1), (dict(lout=FAKE + 1), -1), (dict(l0=FAKE + 3), -1),
    (dict(q=FAKE + 8), -1),
])
def test_fused_rejects(lib, kw, status):
    assert _fused(lib, **kw) == status


def _mob(lib, a=FAKE, b=FAKE, c=FAKE, d=FAKE, l0=FAKE, out=FAKE, N=4, T=16):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kdn_mobius_scan(vp(a), vp(b), vp(c), vp(d), vp(l0), vp(out), N, T, None)


@pytest.mark.parametrize("field", ["a", "b", "c", "d", "l0", "out"])
def test_mobius_null_pointer(lib, field):
    assert _mob(lib, **{field: None}) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(N=-1), -1), (dict(T=-2), -1), (dict(N=1 << 40, T=1 << 40), -1),
    (dict(a=FAKE + 1), -1), (dict(out=FAKE + 2), -1),
])
def test_mobius_rejects(lib, kw, status):
    assert _mob(lib, **kw) == status


def test_mobius_empty_is_a_no_op(lib):
    # nothing to compute: returns OK without touching the (null) buffers
    assert _mob(lib, a=None, b=None, c=None, d=None, l0=None, out=None, N=0, T=16) == 0
    assert _mob(lib, a=None, b=None, c=None, d=None, l0=None, out=None, N=5, T=0) == 0


def _step(lib, q=FAKE, k=FAKE, v=FAKE, beta=FAKE, d=FAKE, A=FAKE, state=FAKE, out=FAKE, B=1, H=1,
          dk=16, dv=16, dtype=1):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kdn_diag_step(vp(q), vp(k), vp(v), vp(beta), vp(d), vp(A), 1.0, vp(state), vp(out),
                             B, H, dk, dv, dtype, None)


@pytest.mark.parametrize("field", ["q", "k", "v", "beta", "d", "A", "state", "out"])
def test_step_null_pointer(lib, field):
    assert _step(lib, **{field: None}) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), -1), (dict(H=-1), -1), (dict(dk=8), -2), (dict(dv=96), -2), (dict(dtype=5), -2),
    (dict(state=FAKE + 8), -1), (dict(q=FAKE + 1), -1), (dict(out=FAKE + 2), -1),
    (dict(A=FAKE + 2), -1), (dict(q=FAKE + 2, dtype=0), -1),
])
def test_step_rejects(lib, kw, status):
    assert _step(lib, **kw) == status


def _host(lib, q=FAKE, k=FAKE, v=FAKE, beta=FAKE, d=FAKE, A=FAKE, out=FAKE, B=1, H=1, T=8,
          dk=16, dv=16, dtype=1):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kdn_diag_scan_fwd_host(vp(q), vp(k), vp(v), vp(beta), vp(d), vp(A), 1.0, None, None,
                                      vp(out), None, B, H, T, dk, dv, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(out=None), -1), (dict(B=0), -1), (dict(T=-1), -1),
    (dict(dk=12), -2), (dict(dtype=3), -2), (dict(q=FAKE + 1), -1), (dict(A=FAKE + 2), -1),
])
def test_host_diag_rejects(lib, kw, status):
    assert _host(lib, **kw) == status


def test_host_mobius_rejects(lib):
    vp = ctypes.c_void_p
    assert lib.kdn_mobius_scan_host(None, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 4, 16, None) == -1
    assert lib.kdn_mobius_scan_host(vp(FAKE + 1), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 4, 16,
                                    None) == -1
    assert lib.kdn_mobius_scan_host(None, None, None, None, None, None, 0, 16, None) == 0


def _bwd(lib, q=FAKE, k=FAKE, v=FAKE, beta=FAKE, d=FAKE, A=FAKE, I0=None, mu0=None, go=FAKE,
         gfs=None, gq=FAKE, gk=FAKE, gv=FAKE, gb=FAKE, gd=FAKE, gA=FAKE, gis=None, B=1, H=1, T=8,
         dk=16, dv=16, dtype=1, ws=None, ws_bytes=0):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kdn_diag_scan_bwd(vp(q), vp(k), vp(v), vp(beta), vp(d), vp(A), 1.0, vp(I0), vp(mu0),
                                 vp(go), vp(gfs), vp(gq), vp(gk), vp(gv), vp(gb), vp(gd), vp(gA),
                                 vp(gis), B, H, T, dk, dv, dtype, vp(ws), ws_bytes, None)


@pytest.mark.parametrize("field", ["q", "k", "v", "beta", "d", "A", "go", "gq", "gk", "gv", "gb", "gd"])
def test_bwd_null_pointer(lib, field):
    assert _bwd(lib, **{field: None}) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), -1), (dict(H=-2), -1), (dict(T=-1), -1), (dict(dk=8), -2), (dict(dv=80), -2),
    (dict(dtype=4), -2), (dict(q=FAKE + 2), -1), (dict(go=FAKE + 4), -1), (dict(gq=FAKE + 8), -1),
    (dict(gis=FAKE + 4), -1), (dict(gfs=FAKE + 8), -1), (dict(I0=FAKE + 4), -1),
    (dict(gd=FAKE + 2), -1), (dict(gA=FAKE + 1), -1), (dict(d=FAKE + 1), -1),
    (dict(B=1 << 20, H=1 << 20, T=1 << 20), -1),
    (dict(ws=FAKE + 16, ws_bytes=1 << 30), -1), (dict(ws=FAKE, ws_bytes=1024), -1),
])
def test_bwd_rejects(lib, kw, status):
    assert _bwd(lib, **kw) == status


def test_bwd_empty_without_state_outputs_is_a_no_op(lib):
    # T = 0 and nothing to write: OK without touching any buffer
    assert _bwd(lib, q=None, k=None, v=None, beta=None, d=None, A=None, go=None, gq=None, gk=None,
                gv=None, gb=None, gd=None, gA=None, T=0) == 0


def test_bwd_workspace_size(lib):
    n = ctypes.c_longlong(-1)
    assert lib.kdn_diag_scan_bwd_workspace(8, 16, 4096, 128, 128, ctypes.byref(n)) == 0
    # every 8th token's state of all heads dominates: B*H*T/8 * 2*dv*dk*4 bytes
    assert n.value >= 8 * 16 * 512 * 2 * 128 * 128 * 4
    assert lib.kdn_diag_scan_bwd_workspace(1, 1, 0, 16, 16, ctypes.byref(n)) == 0 and n.value == 0
    assert lib.kdn_diag_scan_bwd_workspace(1, 1, 8, 24, 16, ctypes.byref(n)) == -2
    assert lib.kdn_diag_scan_bwd_workspace(0, 1, 8, 16, 16, ctypes.byref(n)) == -1


def _lin(lib, q=FAKE, k=FAKE, v=FAKE, beta=FAKE, d=FAKE, A=FAKE, mu0=None, out=FAKE, fm=None,
         B=1, H=1, T=8, dk=16, dv=16, dtype=1):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kdn_lin_scan_fwd(vp(q), vp(k), vp(v), vp(beta), vp(d), vp(A), 1.0, vp(mu0), vp(out),
                                vp(fm), B, H, T, dk, dv, dtype, None)


@pytest.mark.parametrize("field", ["q", "k", "v", "beta", "d", "A", "out"])
def test_lin_null_pointer(lib, field):
    assert _lin(lib, **{field: None}) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), -1), (dict(T=-1), -1), (dict(dk=8), -2), (dict(dv=48), -2), (dict(dtype=2), -2),
    (dict(q=FAKE + 8), -1), (dict(out=FAKE + 4), -1), (dict(mu0=FAKE + 8), -1),
    (dict(fm=FAKE + 2), -1), (dict(A=FAKE + 2), -1), (dict(d=FAKE + 1), -1),
])
def test_lin_rejects(lib, kw, status):
    assert _lin(lib, **kw) == status
