"""Thin ctypes binding of the C ABI in ``include/kdn.h``.

Argument marshalling only: every step of both scans runs in the CUDA
kernels of ``_build/libkdn.so``.  PyTorch provides device memory and the
current stream.  There is no CPU fallback: if the library is missing the
import of this module raises.

Functions mirror the C names:

* :func:`diag_scan_fwd`  -> ``kdn_diag_scan_fwd``
* :func:`diag_mobius_scan_fwd` -> ``kdn_diag_mobius_scan_fwd`` (per-head lambda in the same launch)
* :func:`mobius_scan`    -> ``kdn_mobius_scan``
* :func:`mobius_scan_noalloc` -> ``kdn_mobius_scan_noalloc``
* :func:`diag_scan_plan`, :func:`mobius_scan_plan` -> the ``*_plan`` queries
* :func:`get_device_error`, :func:`set_wait_limit_ns`,
  :func:`debug_stall_mobius_tile`, :func:`status_string`, :func:`version`

When the tensors passed to :func:`diag_scan_fwd` / :func:`mobius_scan` live in
host memory, the call stages them to the current device on the current stream
(pinned memory makes the copies asynchronous), runs the kernels there and
copies the results back; it returns host tensors.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

KDN_OK, KDN_ERR_INVALID_ARG, KDN_ERR_UNSUPPORTED = 0, -1, -2
KDN_ERR_CUDA, KDN_ERR_TIMEOUT, KDN_ERR_ALLOC = -3, -4, -5
KDN_F32, KDN_BF16 = 0, 1

LIB_PATH = _build.LIB


class KdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkdn is not built ({LIB_PATH}); run bayesian_scan_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, fp, i, ll = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    lib.kdn_diag_scan_fwd.restype = i
    lib.kdn_diag_scan_fwd.argtypes = [vp, vp, vp, vp, vp, fp, ctypes.c_float, fp, fp, fp, fp,
                                      i, i, i, i, i, i, vp]
    lib.kdn_mobius_scan.restype = i
    lib.kdn_mobius_scan.argtypes = [fp, fp, fp, fp, fp, fp, ll, ll, vp]
    lib.kdn_diag_mobius_scan_fwd.restype = i
    lib.kdn_diag_mobius_scan_fwd.argtypes = [vp, vp, vp, vp, vp, fp, ctypes.c_float, fp, fp, fp, fp,
                                             fp, fp, fp, fp, fp, fp, i, i, i, i, i, i, vp]
    lib.kdn_lin_scan_fwd.restype = i
    lib.kdn_lin_scan_fwd.argtypes = [vp, vp, vp, vp, vp, fp, ctypes.c_float, fp, fp, fp,
                                     i, i, i, i, i, i, vp]
    lib.kdn_diag_scan_bwd.restype = i
    lib.kdn_diag_scan_bwd.argtypes = [vp, vp, vp, vp, vp, fp, ctypes.c_float, fp, fp, fp, fp,
                                      fp, fp, fp, fp, fp, fp, fp, i, i, i, i, i, i, vp, ll, vp]
    lib.kdn_diag_scan_bwd_workspace.restype = i
    lib.kdn_diag_scan_bwd_workspace.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_longlong)]
    lib.kdn_diag_step.restype = i
    lib.kdn_diag_step.argtypes = [vp, vp, vp, vp, vp, fp, ctypes.c_float, fp, fp, i, i, i, i, i, vp]
    lib.kdn_diag_scan_fwd_host.restype = i
    lib.kdn_diag_scan_fwd_host.argtypes = [vp, vp, vp, vp, vp, fp, ctypes.c_float, fp, fp, fp, fp,
                                           i, i, i, i, i, i, vp]
    lib.kdn_mobius_scan_host.restype = i
    lib.kdn_mobius_scan_host.argtypes = [fp, fp, fp, fp, fp, fp, ll, ll, vp]
    lib.kdn_mobius_scan_noalloc.restype = i
    lib.kdn_mobius_scan_noalloc.argtypes = [fp, fp, fp, fp, fp, fp, ll, ll, vp]
    lib.kdn_status_string.restype = ctypes.c_char_p
    lib.kdn_status_string.argtypes = [i]
    lib.kdn_get_device_error.restype = i
    lib.kdn_get_device_error.argtypes = [vp]
    lib.kdn_set_wait_limit_ns.restype = None
    lib.kdn_set_wait_limit_ns.argtypes = [ll]
    lib.kdn_debug_stall_mobius_tile.restype = None
    lib.kdn_debug_stall_mobius_tile.argtypes = [ll]
    ip, llp = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_longlong)
    lib.kdn_diag_scan_plan.restype = i
    lib.kdn_diag_scan_plan.argtypes = [i, i, i, i, i, i, ip, ip, llp]
    lib.kdn_mobius_scan_plan.restype = i
    lib.kdn_mobius_scan_plan.argtypes = [ll, ll, ip, llp]
    lib.kdn_version.restype = ctypes.c_char_p
    lib.kdn_version.argtypes = []
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.kdn_status_string(int(status)).decode()


def version() -> str:
    return lib.kdn_version().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, name, dtype=None, shape=None):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _on_one_device(stream, **tensors):
    """Every given tensor must be a CUDA tensor on the current device (the
    device whose stream the call is issued on): the C ABI receives raw
    pointers and cannot tell host memory or another GPU's memory apart."""
    given = [(name, t) for name, t in tensors.items() if t is not None]
    for name, t in given:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the call takes device tensors)")
    cur = torch.device("cuda", torch.cuda.current_device())
    for name, t in given:
        if t.device != cur:
            raise ValueError(f"{name} is on {t.device} but the current device is {cur}")
    if stream is not None and getattr(stream, "device", cur) != cur:
        raise ValueError(f"the stream belongs to {stream.device}, not the current device {cur}")


def diag_scan_fwd(q, k, v, beta, d, A, I_prior=1.0, I0=None, mu0=None, out=None,
                  final_state=True, stream=None):
    """Diagonal metaplastic scan with readout (see ``kdn_diag_scan_fwd``).

    q, k [B,H,T,dk]; v, beta [B,H,T,dv]; d [B,H,T] (bf16 or fp32, all the same);
    A [H] fp32; I0, mu0 [B,H,dv,dk] fp32 or None.  ``final_state`` may be
    True (allocate), False/None (skip) or a [2,B,H,dv,dk] fp32 tensor.
    Returns (out [B,H,T,dv] fp32, final_state or None).  With host tensors
    the call goes to ``kdn_diag_scan_fwd_host`` (pipelined copies; outputs
    are host tensors, page-locked when allocated here).
    """
    if not q.is_cuda:
        return _diag_host(q, k, v, beta, d, A, I_prior, I0, mu0, out, final_state, stream)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("inputs must be bf16 or fp32")
    _check(q, "q", dt)
    _check(k, "k", dt, (B, H, T, dk))
    _check(v, "v", dt, (B, H, T, dv))
    _check(beta, "beta", dt, (B, H, T, dv))
    _check(d, "d", dt, (B, H, T))
    _check(A, "A", torch.float32, (H,))
    for name, t in (("I0", I0), ("mu0", mu0)):
        if t is not None:
            _check(t, name, torch.float32, (B, H, dv, dk))
    if out is None:
        out = torch.empty(B, H, T, dv, device=q.device, dtype=torch.float32)
    _check(out, "out", torch.float32, (B, H, T, dv))
    if final_state is True:
        final_state = torch.empty(2, B, H, dv, dk, device=q.device, dtype=torch.float32)
    elif final_state is False:
        final_state = None
    if final_state is not None:
        _check(final_state, "final_state", torch.float32, (2, B, H, dv, dk))
    _on_one_device(stream, q=q, k=k, v=v, beta=beta, d=d, A=A, I0=I0, mu0=mu0, out=out,
                   final_state=final_state)
    st = lib.kdn_diag_scan_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                               float(I_prior), _ptr(I0), _ptr(mu0), _ptr(out), _ptr(final_state),
                               B, H, T, dk, dv, KDN_BF16 if dt == torch.bfloat16 else KDN_F32,
                               _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_diag_scan_fwd")
    return out, final_state


def diag_mobius_scan_fwd(q, k, v, beta, d, A, ma, mb, mc, md, lambda0, I_prior=1.0, I0=None,
                         mu0=None, out=None, final_state=True, lambda_out=None, stream=None):
    """The diagonal scan and the per-head Moebius scan in one launch (see
    ``kdn_diag_mobius_scan_fwd``).  Diagonal-scan arguments as for
    ``diag_scan_fwd`` (device tensors); ma, mb, mc, md [B*H,T] fp32 (row b*H +
    h), lambda0 [B*H] fp32.  Returns (out, final_state or None, lambda
    [B*H,T])."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("inputs must be bf16 or fp32")
    _check(q, "q", dt)
    _check(k, "k", dt, (B, H, T, dk))
    _check(v, "v", dt, (B, H, T, dv))
    _check(beta, "beta", dt, (B, H, T, dv))
    _check(d, "d", dt, (B, H, T))
    _check(A, "A", torch.float32, (H,))
    for name, t in (("I0", I0), ("mu0", mu0)):
        if t is not None:
            _check(t, name, torch.float32, (B, H, dv, dk))
    for name, t in (("ma", ma), ("mb", mb), ("mc", mc), ("md", md)):
        _check(t, name, torch.float32, (B * H, T))
    _check(lambda0, "lambda0", torch.float32, (B * H,))
    _on_one_device(stream, q=q)
    if out is None:
        out = torch.empty(B, H, T, dv, device=q.device, dtype=torch.float32)
    _check(out, "out", torch.float32, (B, H, T, dv))
    if final_state is True:
        final_state = torch.empty(2, B, H, dv, dk, device=q.device, dtype=torch.float32)
    elif final_state is False:
        final_state = None
    if final_state is not None:
        _check(final_state, "final_state", torch.float32, (2, B, H, dv, dk))
    if lambda_out is None:
        lambda_out = torch.empty(B * H, T, device=q.device, dtype=torch.float32)
    _check(lambda_out, "lambda_out", torch.float32, (B * H, T))
    _on_one_device(stream, q=q, k=k, v=v, beta=beta, d=d, A=A, I0=I0, mu0=mu0, out=out,
                   final_state=final_state, ma=ma, mb=mb, mc=mc, md=md, lambda0=lambda0,
                   lambda_out=lambda_out)
    st = lib.kdn_diag_mobius_scan_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                                      float(I_prior), _ptr(I0), _ptr(mu0), _ptr(out),
                                      _ptr(final_state), _ptr(ma), _ptr(mb), _ptr(mc), _ptr(md),
                                      _ptr(lambda0), _ptr(lambda_out), B, H, T, dk, dv,
                                      KDN_BF16 if dt == torch.bfloat16 else KDN_F32, _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_diag_mobius_scan_fwd")
    return out, final_state, lambda_out


def lin_scan_fwd(q, k, v, beta, d, A, I_prior=1.0, mu0=None, out=None, final_mu=True,
                 stream=None):
    """The non-metaplastic limit (importance held at I_prior; see
    ``kdn_lin_scan_fwd``).  Device tensors as for ``diag_scan_fwd``; mu0
    [B,H,dv,dk] fp32 or None; ``final_mu`` True (allocate), False/None or a
    [B,H,dv,dk] fp32 tensor.  Returns (out, final_mu or None)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("inputs must be bf16 or fp32")
    if not q.is_cuda:
        raise ValueError("lin_scan_fwd takes device tensors")
    _check(q, "q", dt)
    _check(k, "k", dt, (B, H, T, dk))
    _check(v, "v", dt, (B, H, T, dv))
    _check(beta, "beta", dt, (B, H, T, dv))
    _check(d, "d", dt, (B, H, T))
    _check(A, "A", torch.float32, (H,))
    if mu0 is not None:
        _check(mu0, "mu0", torch.float32, (B, H, dv, dk))
    if out is None:
        out = torch.empty(B, H, T, dv, device=q.device, dtype=torch.float32)
    _check(out, "out", torch.float32, (B, H, T, dv))
    if final_mu is True:
        final_mu = torch.empty(B, H, dv, dk, device=q.device, dtype=torch.float32)
    elif final_mu is False:
        final_mu = None
    if final_mu is not None:
        _check(final_mu, "final_mu", torch.float32, (B, H, dv, dk))
    _on_one_device(stream, q=q, k=k, v=v, beta=beta, d=d, A=A, mu0=mu0, out=out, final_mu=final_mu)
    st = lib.kdn_lin_scan_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                              float(I_prior), _ptr(mu0), _ptr(out), _ptr(final_mu),
                              B, H, T, dk, dv, KDN_BF16 if dt == torch.bfloat16 else KDN_F32,
                              _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_lin_scan_fwd")
    return out, final_mu


def diag_scan_bwd_workspace(B, H, T, dk, dv) -> int:
    """Bytes of device workspace ``diag_scan_bwd`` needs."""
    n = ctypes.c_longlong(0)
    st = lib.kdn_diag_scan_bwd_workspace(B, H, T, dk, dv, ctypes.byref(n))
    if st != KDN_OK:
        raise KdnError(st, "kdn_diag_scan_bwd_workspace")
    return int(n.value)


def diag_scan_bwd(q, k, v, beta, d, A, grad_out, I_prior=1.0, I0=None, mu0=None,
                  grad_final_state=None, grad_init_state=True, workspace=None, stream=None):
    """Backward pass of ``diag_scan_fwd`` (see ``kdn_diag_scan_bwd``).

    Inputs as for ``diag_scan_fwd`` (device tensors); ``grad_out`` [B,H,T,dv]
    fp32; ``grad_final_state`` [2,B,H,dv,dk] fp32 or None.  ``grad_init_state``
    True (allocate), False/None (skip) or a [2,B,H,dv,dk] fp32 tensor.
    Returns a dict: q, k [B,H,T,dk]; v, beta [B,H,T,dv]; d [B,H,T]; A [H];
    init_state [2,B,H,dv,dk] or None (all fp32).  ``workspace``: a uint8
    device tensor of at least ``diag_scan_bwd_workspace`` bytes, or None (one
    is taken from torch's caching allocator for the call).
    """
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("inputs must be bf16 or fp32")
    if not q.is_cuda:
        raise ValueError("diag_scan_bwd takes device tensors")
    _check(q, "q", dt)
    _check(k, "k", dt, (B, H, T, dk))
    _check(v, "v", dt, (B, H, T, dv))
    _check(beta, "beta", dt, (B, H, T, dv))
    _check(d, "d", dt, (B, H, T))
    _check(A, "A", torch.float32, (H,))
    _check(grad_out, "grad_out", torch.float32, (B, H, T, dv))
    for name, t in (("I0", I0), ("mu0", mu0)):
        if t is not None:
            _check(t, name, torch.float32, (B, H, dv, dk))
    if grad_final_state is not None:
        _check(grad_final_state, "grad_final_state", torch.float32, (2, B, H, dv, dk))
    f32 = dict(device=q.device, dtype=torch.float32)
    g = dict(q=torch.empty(B, H, T, dk, **f32), k=torch.empty(B, H, T, dk, **f32),
             v=torch.empty(B, H, T, dv, **f32), beta=torch.empty(B, H, T, dv, **f32),
             d=torch.empty(B, H, T, **f32), A=torch.empty(H, **f32))
    if grad_init_state is True:
        grad_init_state = torch.empty(2, B, H, dv, dk, **f32)
    elif grad_init_state is False:
        grad_init_state = None
    if grad_init_state is not None:
        _check(grad_init_state, "grad_init_state", torch.float32, (2, B, H, dv, dk))
    g["init_state"] = grad_init_state
    ws_bytes = diag_scan_bwd_workspace(B, H, T, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), device=q.device, dtype=torch.uint8)
    elif workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError(f"workspace must hold {ws_bytes} bytes")
    _on_one_device(stream, q=q, k=k, v=v, beta=beta, d=d, A=A, I0=I0, mu0=mu0, grad_out=grad_out,
                   grad_final_state=grad_final_state, grad_init_state=grad_init_state,
                   workspace=workspace)
    st = lib.kdn_diag_scan_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                               float(I_prior), _ptr(I0), _ptr(mu0), _ptr(grad_out),
                               _ptr(grad_final_state), _ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]),
                               _ptr(g["beta"]), _ptr(g["d"]), _ptr(g["A"]), _ptr(grad_init_state),
                               B, H, T, dk, dv, KDN_BF16 if dt == torch.bfloat16 else KDN_F32,
                               _ptr(workspace), ws_bytes, _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_diag_scan_bwd")
    return g


def diag_step(q, k, v, beta, d, A, state, I_prior=1.0, out=None, stream=None):
    """One token of the diagonal update on a device-resident state (see
    ``kdn_diag_step``): q, k [B,H,dk]; v, beta [B,H,dv]; d [B,H] (bf16 or
    fp32); A [H] fp32; state [2,B,H,dv,dk] fp32 (mu then I), updated in place.
    Returns out [B,H,dv] fp32."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("inputs must be bf16 or fp32")
    for name, t, shape, dtype in (("q", q, (B, H, dk), dt), ("k", k, (B, H, dk), dt),
                                  ("v", v, (B, H, dv), dt), ("beta", beta, (B, H, dv), dt),
                                  ("d", d, (B, H), dt), ("A", A, (H,), torch.float32),
                                  ("state", state, (2, B, H, dv, dk), torch.float32)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        _check(t, name, dtype, shape)
    if out is None:
        out = torch.empty(B, H, dv, device=q.device, dtype=torch.float32)
    _check(out, "out", torch.float32, (B, H, dv))
    _on_one_device(stream, q=q, k=k, v=v, beta=beta, d=d, A=A, state=state, out=out)
    st = lib.kdn_diag_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A), float(I_prior),
                           _ptr(state), _ptr(out), B, H, dk, dv,
                           KDN_BF16 if dt == torch.bfloat16 else KDN_F32, _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_diag_step")
    return out


def mobius_scan(a, b, c, d, lambda0, out=None, stream=None):
    """Moebius precision recursion (see ``kdn_mobius_scan``): a,b,c,d [N,T]
    fp32, lambda0 [N] fp32 -> lambda_1..lambda_T [N,T] fp32.  Host tensors go
    to ``kdn_mobius_scan_host``."""
    if not a.is_cuda:
        return _mobius_host(a, b, c, d, lambda0, out, stream)
    N, T = a.shape
    for name, t in (("a", a), ("b", b), ("c", c), ("d", d)):
        _check(t, name, torch.float32, (N, T))
    _check(lambda0, "lambda0", torch.float32, (N,))
    if out is None:
        out = torch.empty(N, T, device=a.device, dtype=torch.float32)
    _check(out, "out", torch.float32, (N, T))
    _on_one_device(stream, a=a, b=b, c=c, d=d, lambda0=lambda0, out=out)
    st = lib.kdn_mobius_scan(_ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(lambda0), _ptr(out),
                             N, T, _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_mobius_scan")
    return out


def diag_scan_plan(B, H, T, dk, dv, dtype=torch.bfloat16) -> dict:
    """Launch plan of a diagonal-scan call: token parts, kernels, scratch bytes."""
    p, k, sb = ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
    st = lib.kdn_diag_scan_plan(B, H, T, dk, dv, KDN_BF16 if dtype == torch.bfloat16 else KDN_F32,
                                ctypes.byref(p), ctypes.byref(k), ctypes.byref(sb))
    if st != KDN_OK:
        raise KdnError(st, "kdn_diag_scan_plan")
    return dict(parts=p.value, kernels=k.value, scratch_bytes=sb.value)


def mobius_scan_plan(N, T) -> dict:
    """Launch plan of a Moebius-scan call: kernels and scratch bytes."""
    k, sb = ctypes.c_int(), ctypes.c_longlong()
    st = lib.kdn_mobius_scan_plan(N, T, ctypes.byref(k), ctypes.byref(sb))
    if st != KDN_OK:
        raise KdnError(st, "kdn_mobius_scan_plan")
    return dict(kernels=k.value, scratch_bytes=sb.value)


MOBIUS_NOALLOC_MAX_TILES = 43690   # N * ceil(T / 2048) limit of mobius_scan_noalloc


def mobius_scan_noalloc(a, b, c, d, lambda0, out, stream=None):
    """``kdn_mobius_scan_noalloc``: the Moebius scan for callers that must not
    allocate device memory during the call (e.g. a framework that reserved
    the GPU's memory up front).  The caller passes every buffer, ``out``
    included; the look-back scratch is a fixed 1 MiB array in the library.
    Calls that overlap on the GPU share that array and race."""
    N, T = a.shape
    for name, t in (("a", a), ("b", b), ("c", c), ("d", d), ("out", out)):
        _check(t, name, torch.float32, (N, T))
    _check(lambda0, "lambda0", torch.float32, (N,))
    _on_one_device(stream, a=a, b=b, c=c, d=d, lambda0=lambda0, out=out)
    st = lib.kdn_mobius_scan_noalloc(_ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(lambda0), _ptr(out),
                                     N, T, _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_mobius_scan_noalloc")
    return out


def get_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    return int(lib.kdn_get_device_error(_stream(stream)))


def set_wait_limit_ns(ns: int) -> None:
    lib.kdn_set_wait_limit_ns(int(ns))


def debug_stall_mobius_tile(tile: int) -> None:
    lib.kdn_debug_stall_mobius_tile(int(tile))


# ---------------------------------------------------------------------------
# host-buffer calls: kdn_diag_scan_fwd_host / kdn_mobius_scan_host copy in,
# scan and copy out in pipelined chunks (page-locked tensors let the copies
# overlap the scans); results land in host tensors.

def _host_out(t, name, shape):
    """A caller-given host output (checked) or a new page-locked one."""
    if t is None:
        return torch.empty(shape, dtype=torch.float32, pin_memory=True)
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor when the inputs are")
    _check(t, name, torch.float32, shape)
    return t


def _diag_host(q, k, v, beta, d, A, I_prior, I0, mu0, out, final_state, stream):
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("inputs must be bf16 or fp32")
    for name, t, shape, dtype in (("q", q, (B, H, T, dk), dt), ("k", k, (B, H, T, dk), dt),
                                  ("v", v, (B, H, T, dv), dt), ("beta", beta, (B, H, T, dv), dt),
                                  ("d", d, (B, H, T), dt), ("A", A, (H,), torch.float32),
                                  ("I0", I0, (B, H, dv, dk), torch.float32),
                                  ("mu0", mu0, (B, H, dv, dk), torch.float32)):
        if t is not None:
            if t.is_cuda:
                raise ValueError(f"{name} must be a host tensor like q")
            _check(t, name, dtype, shape)
    out = _host_out(out, "out", (B, H, T, dv))
    if final_state is True:
        final_state = None
        fs = _host_out(None, "final_state", (2, B, H, dv, dk))
    elif final_state is False or final_state is None:
        fs = None
    else:
        fs = _host_out(final_state, "final_state", (2, B, H, dv, dk))
    st = lib.kdn_diag_scan_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(d), _ptr(A),
                                    float(I_prior), _ptr(I0), _ptr(mu0), _ptr(out), _ptr(fs),
                                    B, H, T, dk, dv, KDN_BF16 if dt == torch.bfloat16 else KDN_F32,
                                    _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_diag_scan_fwd_host")
    return out, fs


def _mobius_host(a, b, c, d, lambda0, out, stream):
    N, T = a.shape
    for name, t in (("a", a), ("b", b), ("c", c), ("d", d)):
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor like a")
        _check(t, name, torch.float32, (N, T))
    _check(lambda0, "lambda0", torch.float32, (N,))
    out = _host_out(out, "out", (N, T))
    st = lib.kdn_mobius_scan_host(_ptr(a), _ptr(b), _ptr(c), _ptr(d), _ptr(lambda0), _ptr(out),
                                  N, T, _stream(stream))
    if st != KDN_OK:
        raise KdnError(st, "kdn_mobius_scan_host")
    return out
