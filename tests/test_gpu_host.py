"""Host-buffer entry points (kdn_diag_scan_fwd_host, kdn_mobius_scan_host):
chunked, pipelined copies around the same kernels.  Checked against the fp64
oracle and against the device entry points, with page-locked and pageable
host tensors, ragged last chunks, given initial states and zero length."""
import pytest
import torch

from bayesian_scan_gb300 import workloads
import parity

pytestmark = pytest.mark.gpu


def draw(B, H, T, dk, dv, dtype=torch.bfloat16, A_law=("uniform", 0.5, 4.0), seed=3):
    q, k, v, beta, d, A = workloads.draw_diag(B, H, T, dk, dv, dtype, A_law, seed=seed)
    return dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=1.0)


def host_diag(inp, I0=None, mu0=None, pin=True, final_state=True):
    from bayesian_scan_gb300 import kdn
    prep = (lambda t: t.pin_memory()) if pin else (lambda t: t)
    xs = [prep(inp[n]) for n in ("q", "k", "v", "beta", "d", "A")]
    o, fs = kdn.diag_scan_fwd(*xs, I_prior=inp["I_prior"],
                              I0=None if I0 is None else prep(I0),
                              mu0=None if mu0 is None else prep(mu0), final_state=final_state)
    assert not o.is_cuda
    assert kdn.get_device_error() == 0
    return o, fs


@pytest.mark.parametrize("T,dk,dtype", [(3001, 64, torch.bfloat16), (4096, 128, torch.bfloat16),
                                        (1500, 32, torch.float32), (100, 16, torch.float32)])
def test_host_diag_matches_oracle(T, dk, dtype):
    inp = draw(1, 2, T, dk, dk, dtype, seed=T)
    o, fs = host_diag(inp)
    ro, rmu, rI = parity.oracle_diag(inp)
    parity.assert_close(o, ro, parity.TOL_DIAG)
    parity.assert_close(fs[0], rmu, parity.TOL_DIAG)
    parity.assert_close(fs[1], rI, parity.TOL_DIAG)


def test_host_diag_initial_state_and_pageable_buffers():
    inp = draw(2, 1, 2100, 64, 64, seed=5)
    g = torch.Generator().manual_seed(4)
    I0 = 0.5 + torch.rand(2, 1, 64, 64, generator=g)
    mu0 = torch.randn(2, 1, 64, 64, generator=g)
    o, fs = host_diag(inp, I0, mu0, pin=False)
    ro, rmu, rI = parity.oracle_diag(inp, I0, mu0)
    parity.assert_close(o, ro, parity.TOL_DIAG)
    parity.assert_close(fs[0], rmu, parity.TOL_DIAG)
    parity.assert_close(fs[1], rI, parity.TOL_DIAG)


def test_host_diag_agrees_with_device_call():
    # chunks carry the state through (mu, I): equal to the one-call result
    # up to that round trip's rounding
    inp = draw(2, 4, 3000, 64, 64, seed=8)
    o_h, fs_h = host_diag(inp)
    o_d, fs_d = parity.gpu_diag(inp)
    assert parity.rel_err(o_h, o_d) < 1e-4
    assert parity.rel_err(fs_h[0], fs_d[0]) < 1e-4
    assert parity.rel_err(fs_h[1], fs_d[1]) < 1e-4


def test_host_diag_outputs_given_and_state_skipped():
    from bayesian_scan_gb300 import kdn
    inp = draw(1, 2, 700, 32, 32, seed=9)
    out = torch.full((1, 2, 700, 32), float("nan")).pin_memory()
    o, fs = kdn.diag_scan_fwd(*(inp[n].pin_memory() for n in ("q", "k", "v", "beta", "d", "A")),
                              I_prior=1.0, out=out, final_state=False)
    assert o.data_ptr() == out.data_ptr() and fs is None
    ro, _, _ = parity.oracle_diag(inp)
    parity.assert_close(o, ro, parity.TOL_DIAG)


@pytest.mark.parametrize("where", ["pinned", "pinned_offset", "pageable"])
def test_host_diag_output_buffers(where):
    # page-locked 16-byte aligned outputs are written by the scan through
    # their mapping; an offset page-locked view and pageable memory are staged
    from bayesian_scan_gb300 import kdn
    inp = draw(1, 2, 1300, 64, 64, seed=11)
    shape = (1, 2, 1300, 64)
    n = 1 * 2 * 1300 * 64
    if where == "pinned":
        out = torch.full(shape, float("nan")).pin_memory()
    elif where == "pinned_offset":
        out = torch.full((n + 1,), float("nan")).pin_memory()[1:].view(shape)
    else:
        out = torch.full(shape, float("nan"))
    o, _ = kdn.diag_scan_fwd(*(inp[n_].pin_memory() for n_ in ("q", "k", "v", "beta", "d", "A")),
                             I_prior=1.0, out=out, final_state=False)
    assert o.data_ptr() == out.data_ptr()
    ro, _, _ = parity.oracle_diag(inp)
    parity.assert_close(o, ro, parity.TOL_DIAG)


def test_host_diag_batch_groups_match_oracle():
    # four or more batches run as groups of whole batches (here 5 groups of
    # one batch: the three group buffers are reused), with an initial state
    inp = draw(5, 2, 300, 32, 32, seed=21)
    g = torch.Generator().manual_seed(22)
    I0 = 0.5 + torch.rand(5, 2, 32, 32, generator=g)
    mu0 = torch.randn(5, 2, 32, 32, generator=g)
    o, fs = host_diag(inp, I0, mu0)
    ro, rmu, rI = parity.oracle_diag(inp, I0, mu0)
    parity.assert_close(o, ro, parity.TOL_DIAG)
    parity.assert_close(fs[0], rmu, parity.TOL_DIAG)
    parity.assert_close(fs[1], rI, parity.TOL_DIAG)


def test_host_diag_batch_groups_uneven_and_pageable():
    # 9 batches in groups of 2 (the last holds one); pageable buffers, so the
    # outputs are staged and copied out
    inp = draw(9, 2, 129, 16, 16, torch.float32, seed=23)
    o, fs = host_diag(inp, pin=False)
    ro, rmu, rI = parity.oracle_diag(inp)
    parity.assert_close(o, ro, parity.TOL_DIAG)
    parity.assert_close(fs[0], rmu, parity.TOL_DIAG)
    parity.assert_close(fs[1], rI, parity.TOL_DIAG)


def test_host_diag_batch_groups_agree_with_device_call():
    # the 750M-shaped pattern (8 batches of 16 heads, d = 128) at 1000 tokens:
    # each group's call plans its own token split, so agreement is to rounding
    inp = draw(8, 16, 1000, 128, 128, seed=24)
    o_h, fs_h = host_diag(inp)
    o_d, fs_d = parity.gpu_diag(inp)
    assert parity.rel_err(o_h, o_d) < 1e-4
    assert parity.rel_err(fs_h[0], fs_d[0]) < 1e-4
    assert parity.rel_err(fs_h[1], fs_d[1]) < 1e-4


def test_host_diag_zero_length_returns_initial_state():
    inp = draw(1, 2, 0, 16, 16)
    g = torch.Generator().manual_seed(2)
    I0 = 0.5 + torch.rand(1, 2, 16, 16, generator=g)
    mu0 = torch.randn(1, 2, 16, 16, generator=g)
    o, fs = host_diag(inp, I0, mu0)
    assert o.shape == (1, 2, 0, 16)
    assert parity.rel_err(fs[0], mu0) < 1e-6 and parity.rel_err(fs[1], I0) < 1e-6


def test_host_rejects_mixed_devices():
    from bayesian_scan_gb300 import kdn
    inp = draw(1, 1, 32, 16, 16)
    xs = [inp[n] for n in ("q", "k", "v", "beta", "d", "A")]
    xs[2] = xs[2].cuda()
    with pytest.raises(ValueError):
        kdn.diag_scan_fwd(*xs)


@pytest.mark.parametrize("N,T", [(1000, 4100), (3, 5003), (600, 2048), (1, 1)])
def test_host_mobius_matches_oracle_and_device(N, T):
    from bayesian_scan_gb300 import kdn
    a, b, c, d, lam0 = workloads.draw_mobius(N, T, seed=N + 2 * T)
    out = kdn.mobius_scan(*(x.pin_memory() for x in (a, b, c, d, lam0)))
    assert not out.is_cuda
    assert kdn.get_device_error() == 0
    ref = parity.oracle.mobius_scan(a, b, c, d, lam0)
    parity.assert_close(out, ref, parity.TOL_MOBIUS)
    dev = parity.gpu_mobius(a, b, c, d, lam0)
    assert parity.rel_err(out, dev) <= 1e-6
