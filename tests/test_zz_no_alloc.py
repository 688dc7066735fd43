"""kdn_mobius_scan_noalloc, the allocation-free Moebius scan, against
kdn_mobius_scan.

Some callers cannot allocate device memory during a call (a framework that
reserved the GPU's memory up front, a loop where allocator calls are not
allowed); this entry point serves them with look-back scratch in a fixed
array inside the library.  The test calls it through the C ABI (ctypes) and
compares it with the allocating entry point on two calls in a row (the second
call must clear what the first left in the shared array), checks that those
calls took nothing from the device's default memory pool (where the
allocating entry point takes its scratch), then checks that a call needing
more look-back tiles than the array holds is refused.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one; it also passes alone in a fresh process
(the first call on the device does the array's set-up)."""
import ctypes
import os

import pytest
import torch

from bayesian_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-5   # the Moebius parity tolerance used by the other tests
POOL_USED_HIGH = 8   # cudaMemPoolAttrUsedMemHigh


def _call(lib, a, b, c, d, lam0, out):
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kdn_mobius_scan_noalloc(p(a), p(b), p(c), p(d), p(lam0), p(out),
                                       a.shape[0], a.shape[1], stream)


def _rel(x, ref):
    return float((x.double() - ref.double()).abs().max() / ref.double().abs().max())


class DefaultPool:
    """High-water mark of the current device's default memory pool, read
    through the CUDA runtime the library links."""

    def __init__(self):
        from bayesian_scan_gb300 import build
        self.rt = ctypes.CDLL(os.path.join(build._cuda_lib_dir(build._nvcc()), "libcudart.so"))
        self.pool = ctypes.c_void_p()
        dev = torch.cuda.current_device()
        assert self.rt.cudaDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def reset(self):
        zero = ctypes.c_uint64(0)
        assert self.rt.cudaMemPoolSetAttribute(self.pool, POOL_USED_HIGH, ctypes.byref(zero)) == 0

    def used_high(self):
        v = ctypes.c_uint64()
        assert self.rt.cudaMemPoolGetAttribute(self.pool, POOL_USED_HIGH, ctypes.byref(v)) == 0
        return v.value


def test_noalloc_matches_allocating_entry_point_twice():
    from bayesian_scan_gb300 import kdn
    lib = kdn.lib
    # two look-back calls in a row (unaligned rows; few long sequences), then
    # one that the sequence-per-CTA kernel runs without any scratch
    cases = []
    for N, T, seed in [(48, 9001, 21), (5, 30000, 22), (600, 6144, 23)]:
        a, b, c, d, lam0 = (x.cuda() for x in workloads.draw_mobius(N, T, seed=seed))
        cases.append((a, b, c, d, lam0, torch.full((N, T), float("nan"), device="cuda")))
    pool = DefaultPool()
    torch.cuda.synchronize()
    # the probe sees the allocating entry point's scratch ...
    pool.reset()
    ref0 = kdn.mobius_scan(*cases[0][:5])
    torch.cuda.synchronize()
    assert pool.used_high() > 0
    refs = [ref0] + [kdn.mobius_scan(*cs[:5]) for cs in cases[1:]]
    torch.cuda.synchronize()
    # ... and nothing from the allocation-free one
    pool.reset()
    for call, (a, b, c, d, lam0, out) in enumerate(cases):
        st = _call(lib, a, b, c, d, lam0, out)
        assert st == 0, (call, kdn.status_string(st))
    torch.cuda.synchronize()
    assert pool.used_high() == 0
    assert kdn.get_device_error() == 0
    for call, ((*_, out), ref) in enumerate(zip(cases, refs)):
        assert torch.isfinite(out).all(), f"call {call}"
        assert _rel(out, ref) <= TOL, f"call {call}"


def test_noalloc_refuses_more_tiles_than_the_array_holds():
    from bayesian_scan_gb300 import kdn
    # T % 4 != 0 keeps the call on the look-back kernel: 3 tiles per sequence
    N, T = kdn.MOBIUS_NOALLOC_MAX_TILES // 3 + 1, 4097
    x = torch.zeros(N, T, device="cuda")
    lam0 = torch.ones(N, device="cuda")
    out = torch.full((N, T), -7.0, device="cuda")
    assert _call(kdn.lib, x, x, x, x, lam0, out) == kdn.KDN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((out == -7.0).all())        # nothing was launched
