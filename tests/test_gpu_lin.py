"""kdn_lin_scan_fwd (importance held at I_prior) against the fp64 oracle of
the non-metaplastic limit: every (d_k, d_v) pair in bf16 and fp32, ragged
token counts, a given initial mean, the gate laws, the token-split path (few
long heads), resume, and the limit relation to the metaplastic scan."""
import pytest
import torch

import oracle
import parity
from bayesian_scan_gb300 import workloads

pytestmark = pytest.mark.gpu


def run(inp, mu0=None):
    from bayesian_scan_gb300 import kdn
    dev = "cuda"
    x = [inp[n].to(dev) for n in ("q", "k", "v", "beta", "d", "A")]
    o, mu = kdn.lin_scan_fwd(*x, I_prior=inp["I_prior"], mu0=None if mu0 is None else mu0.to(dev))
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    return o.cpu(), mu.cpu()


def check(inp, mu0=None, tol=parity.TOL_DIAG):
    o, mu = run(inp, mu0)
    ro, rmu = oracle.lin_scan(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d"], inp["A"],
                              inp["I_prior"], mu0)
    errs = dict(o=parity.both_errs(o, ro), mu=parity.both_errs(mu, rmu))
    B, H, T, dk = inp["q"].shape
    tc = dk == 128 and inp["v"].shape[-1] == 128 and inp["q"].dtype == torch.bfloat16
    et = parity.TOL_ELEM_LIN_TC if tc else parity.TOL_ELEM
    for k_, (e, ee) in errs.items():
        assert e <= tol and ee <= et, (k_, errs)
    return errs


def make(B, H, T, dk, dv, dtype=torch.bfloat16, law=("uniform", 0.5, 4.0), seed=0, I_prior=1.0):
    q, k, v, beta, d, A = workloads.draw_diag(B, H, T, dk, dv, dtype, law, seed=seed)
    return dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=I_prior)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (64, 64), (128, 128), (128, 32),
                                   (16, 128), (128, 16)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_lin_matches_oracle(dk, dv, dtype):
    check(make(2, 3, 77, dk, dv, dtype, seed=dk + dv))


@pytest.mark.parametrize("T", [0, 1, 15, 16, 17, 100])
def test_lin_token_counts(T):
    inp = make(1, 2, T, 64, 64, seed=T + 1)
    g = torch.Generator().manual_seed(T)
    check(inp, mu0=torch.randn(1, 2, 64, 64, generator=g))


@pytest.mark.parametrize("law", [("const", 0.0), ("const", 1.0), ("uniform", 0.1, 1.0), ("const", 30.0)])
def test_lin_gate_laws(law):
    check(make(2, 2, 200, 128, 128, law=law, seed=5))


@pytest.mark.parametrize("I_prior", [1e-2, 1.0, 1e3])
def test_lin_prior_scale(I_prior):
    check(make(1, 2, 64, 32, 32, I_prior=I_prior, seed=6))


@pytest.mark.parametrize("dk,dtype", [(128, torch.bfloat16), (64, torch.bfloat16), (128, torch.float32)])
def test_lin_token_split(dk, dtype):
    # two heads over 3001 tokens: the call splits the sequence into parts
    from bayesian_scan_gb300 import kdn
    plan = kdn.diag_scan_plan(1, 2, 3001, dk, dk, dtype)
    assert plan["parts"] > 1
    g = torch.Generator().manual_seed(dk)
    check(make(1, 2, 3001, dk, dk, dtype, law=("uniform", 0.1, 1.0), seed=7),
          mu0=torch.randn(1, 2, dk, dk, generator=g))


def test_lin_resume():
    inp = make(2, 2, 90, 64, 32, seed=8)
    o, mu = run(inp)
    h = 37
    first = {n: (inp[n][:, :, :h].contiguous() if n in ("q", "k", "v", "beta", "d") else inp[n]) for n in inp}
    second = {n: (inp[n][:, :, h:].contiguous() if n in ("q", "k", "v", "beta", "d") else inp[n]) for n in inp}
    o1, mu1 = run(first)
    o2, mu2 = run(second, mu1)
    assert parity.rel_err(torch.cat([o1, o2], dim=2), o) < 1e-5
    assert parity.rel_err(mu2, mu) < 1e-5


def test_lin_is_the_metaplastic_limit_on_the_gpu():
    # the metaplastic scan with I_0 = I_prior = 1e6 tends to this scan
    from bayesian_scan_gb300 import kdn
    inp = make(1, 2, 50, 32, 32, dtype=torch.float32, seed=9, I_prior=1e6)
    o_l, _ = run(inp)
    x = [inp[n].to("cuda") for n in ("q", "k", "v", "beta", "d", "A")]
    o_d, _ = kdn.diag_scan_fwd(*x, I_prior=1e6)
    torch.cuda.synchronize()
    assert parity.rel_err(o_d.cpu(), o_l) < 1e-4


@pytest.mark.parametrize("T", [1, 31, 32, 33, 64, 100, 517])
def test_lin_tensor_core_path(T):
    # d_k = d_v = 128 with bf16 inputs runs the chunked tensor-core kernel
    # (64-token chunks): chunk boundaries, a given initial mean, all heads
    g = torch.Generator().manual_seed(T)
    inp = make(2, 3, T, 128, 128, seed=40 + T)
    check(inp, mu0=torch.randn(2, 3, 128, 128, generator=g))


@pytest.mark.parametrize("I_prior,law", [(1e-2, ("const", 1.0)), (1e3, ("uniform", 0.5, 4.0)),
                                         (1.0, ("const", 0.0)), (1.0, ("const", 30.0))])
def test_lin_tensor_core_scales(I_prior, law):
    check(make(1, 4, 96, 128, 128, law=law, seed=50, I_prior=I_prior))
