"""Parity at the full workload sizes, in the launch configuration bench.py
times (same shapes through the same entry points), on sampled outputs.

State rows are independent (only the readout sums over the key axis), so the
oracle computes row i of head (b, h) from v[..., i] and beta[..., i] alone:
the sample is a few rows of a few heads over the whole sequence, compared
element by element with the GPU's o[b, h, :, i] and final mu/I rows.
Moebius sequences are independent too: sampled sequences are compared whole.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from bayesian_scan_gb300 import workloads

pytestmark = pytest.mark.gpu

WORKLOADS = ["heads32_t2048_d64", "layer750m", "layer1p3b", "longctx"]


def _sample(w, rng):
    n_heads = 2 if w.T > 20000 else 3
    heads = sorted(set(int(x) for x in rng.choice(w.B * w.H, size=n_heads, replace=False)) |
                   {w.B * w.H - 1})
    rows = sorted(set(int(x) for x in rng.choice(w.dv, size=3, replace=False)) | {0, w.dv - 1})
    return heads, rows


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_sampled(name):
    from bayesian_scan_gb300 import kdn
    w = workloads.get(name)
    inp = workloads.make(w)
    dev = "cuda"
    x = [inp[n].to(dev) for n in ("q", "k", "v", "beta", "d", "A")]
    mob = [inp[n].to(dev) for n in ("ma", "mb", "mc", "md", "lam0")]
    if w.mobius_fused:   # one lambda sequence per head, in the scan's launch (as bench.py times it)
        o, fs, lam = kdn.diag_mobius_scan_fwd(*x, *mob, I_prior=inp["I_prior"])
    else:
        o, fs = kdn.diag_scan_fwd(*x, I_prior=inp["I_prior"])
        lam = kdn.mobius_scan(*mob)
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    rng = np.random.default_rng(sum(map(ord, name)))
    heads, rows = _sample(w, rng)
    H = w.H
    for bh in heads:
        b, h = divmod(bh, H)
        sl = lambda t: t[b:b + 1, h:h + 1]
        q, k, d = sl(inp["q"]), sl(inp["k"]), sl(inp["d"])
        v, beta = sl(inp["v"])[..., rows], sl(inp["beta"])[..., rows]
        ro, rmu, rI = oracle.diag_scan(q, k, v, beta, d, inp["A"][h:h + 1], inp["I_prior"])
        go = o[b, h][:, rows].cpu()
        gmu = fs[0, b, h][rows].cpu()
        gI = fs[1, b, h][rows].cpu()
        parity.assert_close(go, ro[0, 0], parity.TOL_DIAG, (name, bh))
        parity.assert_close(gmu, rmu[0, 0], parity.TOL_DIAG, (name, bh))
        parity.assert_close(gI, rI[0, 0], parity.TOL_DIAG, (name, bh))
    seqs = sorted(set(int(s) for s in rng.choice(w.mobius_N, size=min(4, w.mobius_N),
                                                 replace=False)))
    ref = oracle.mobius_scan(inp["ma"][seqs], inp["mb"][seqs], inp["mc"][seqs], inp["md"][seqs],
                             inp["lam0"][seqs])
    parity.assert_close(lam[seqs].cpu(), ref, parity.TOL_MOBIUS, name)


def test_full_size_compared_in_full():
    """The 32-head d = 64 workload (B=4, H=8, T=2048, bf16) in its bench
    launch (scan and per-head lambda in one launch): every output element
    against the oracle."""
    from bayesian_scan_gb300 import kdn
    w = workloads.get("heads32_t2048_d64")
    inp = workloads.make(w)
    x = [inp[n].cuda() for n in ("q", "k", "v", "beta", "d", "A")]
    mob = [inp[n].cuda() for n in ("ma", "mb", "mc", "md", "lam0")]
    o, fs, lam = kdn.diag_mobius_scan_fwd(*x, *mob, I_prior=inp["I_prior"])
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    ro, rmu, rI = parity.oracle_diag(inp)
    parity.assert_close(o.cpu(), ro, parity.TOL_DIAG, "o")
    parity.assert_close(fs[0].cpu(), rmu, parity.TOL_DIAG, "mu_T")
    parity.assert_close(fs[1].cpu(), rI, parity.TOL_DIAG, "I_T")
    rl = oracle.mobius_scan(inp["ma"], inp["mb"], inp["mc"], inp["md"], inp["lam0"])
    parity.assert_close(lam.cpu(), rl, parity.TOL_MOBIUS, "lambda")


def test_full_size_properties_everywhere():
    """Properties that hold at any size, checked on every output of the 750M
    layer: all finite, and I_T >= I_prior (I_0 = I_prior, evidence >= 0)."""
    from bayesian_scan_gb300 import kdn
    w = workloads.get("layer750m")
    inp = workloads.make(w, with_mobius=False)
    x = [inp[n].to("cuda") for n in ("q", "k", "v", "beta", "d", "A")]
    o, fs = kdn.diag_scan_fwd(*x, I_prior=inp["I_prior"])
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(fs).all())
    assert float(fs[1].min()) >= inp["I_prior"] * (1 - 1e-6)


def test_full_size_backward_sampled_heads():
    """kdn_diag_scan_bwd over the whole 750M-shaped layer (the bench's
    backward configuration); the oracle recomputes two whole heads (heads
    are independent; the gradients of one head depend on that head alone),
    and dA is checked against the per-token gradients it sums."""
    from bayesian_scan_gb300 import kdn
    w = workloads.get("layer750m_bwd")
    inp = workloads.make(w, with_mobius=False)
    gout, _ = workloads.draw_cotangents(w.B, w.H, w.T, w.dk, w.dv, seed=w.seed + 1)
    x = [inp[n].to("cuda") for n in ("q", "k", "v", "beta", "d", "A")]
    g = kdn.diag_scan_bwd(*x, gout.to("cuda"), I_prior=inp["I_prior"], grad_init_state=False)
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    for n in ("q", "k", "v", "beta", "d", "A"):
        assert bool(torch.isfinite(g[n]).all()), n
    # dA_h = sum_b sum_t (d_t / A_h) dd_t   (dd = -A alpha dL/dalpha, dA = -sum d alpha dL/dalpha)
    dd, d = g["d"].double().cpu(), inp["d"].double()
    ref_dA = (d * dd).sum(dim=(0, 2)) / inp["A"].double()
    assert parity.rel_err(g["A"].cpu(), ref_dA) < 1e-4
    H = w.H
    for bh in (5, w.B * H - 1):
        b, h = divmod(bh, H)
        sl = lambda t: t[b:b + 1, h:h + 1]
        r = oracle.diag_scan_bwd(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["beta"]),
                                 sl(inp["d"]), inp["A"][h:h + 1], inp["I_prior"], dout=sl(gout))
        for n, o in parity.BWD_NAMES.items():
            if n == "A":
                continue
            parity.assert_close(g[n][b:b + 1, h:h + 1].cpu(), r[o], parity.TOL_BWD, (n, bh))


@pytest.mark.parametrize("name", ["layer750m_lin", "longctx_lin"])
def test_full_size_lin_sampled(name):
    """kdn_lin_scan_fwd at the bench sizes (the tensor-core path; the long
    context with its token split): rows of the state are independent, so the
    oracle recomputes sampled rows of sampled heads over the whole sequence."""
    from bayesian_scan_gb300 import kdn
    w = workloads.get(name)
    inp = workloads.make(w, with_mobius=False)
    x = [inp[n].to("cuda") for n in ("q", "k", "v", "beta", "d", "A")]
    o, mu = kdn.lin_scan_fwd(*x, I_prior=inp["I_prior"])
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(mu).all())
    rng = np.random.default_rng(sum(map(ord, name)))
    heads, rows = _sample(w, rng)
    for bh in heads:
        b, h = divmod(bh, w.H)
        sl = lambda t: t[b:b + 1, h:h + 1]
        ro, rmu = oracle.lin_scan(sl(inp["q"]), sl(inp["k"]), sl(inp["v"])[..., rows],
                                  sl(inp["beta"])[..., rows], sl(inp["d"]), inp["A"][h:h + 1],
                                  inp["I_prior"])
        # the tensor-core kernel of the non-metaplastic limit (d = 128, bf16)
        et = parity.TOL_ELEM_LIN_TC
        parity.assert_close(o[b, h][:, rows].cpu(), ro[0, 0], parity.TOL_DIAG, (name, bh), et)
        parity.assert_close(mu[b, h][rows].cpu(), rmu[0, 0], parity.TOL_DIAG, (name, bh), et)
