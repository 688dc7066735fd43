"""kdn_diag_mobius_scan_fwd: the diagonal scan and the per-head Moebius scan
in one launch ("Kalman Linear Attention (KLA)", Metodologia 2, for lambda;
"Learning to Remember, Learn, and Forget in Attention-Based Models",
Metodologia 1-2, for the scan).  Every output is compared element by element
with the fp64 oracle (o, mu_T, I_T with oracle.diag_scan; lambda with
oracle.mobius_scan) on the same inputs, for every head size, with and without
the token split, with an initial state, and on layouts that take the
separate-launch fallback."""
import pytest
import torch

import oracle
import parity
from bayesian_scan_gb300 import workloads

pytestmark = pytest.mark.gpu


def run_and_check(B, H, T, dk, dv, dtype=torch.bfloat16, A_law=("uniform", 0.5, 4.0), seed=0,
                  state=False, lam_offset=0):
    from bayesian_scan_gb300 import kdn
    q, k, v, beta, d, A = workloads.draw_diag(B, H, T, dk, dv, dtype, A_law, seed=seed)
    ma, mb, mc, md, lam0 = workloads.draw_mobius(B * H, T, seed=seed + 1)
    lam0 = lam0 + torch.rand(B * H, generator=torch.Generator().manual_seed(seed))
    I0 = mu0 = None
    if state:
        g = torch.Generator().manual_seed(seed + 2)
        I0 = 0.5 + torch.rand(B, H, dv, dk, generator=g)
        mu0 = torch.randn(B, H, dv, dk, generator=g)
    dev = "cuda"
    cu = lambda t: None if t is None else t.to(dev)
    lam_out = None
    if lam_offset:
        # a view that starts lam_offset floats into its buffer (not 16-byte aligned)
        lam_out = torch.empty(B * H * T + lam_offset, device=dev)[lam_offset:].view(B * H, T)
    o, fs, lam = kdn.diag_mobius_scan_fwd(cu(q), cu(k), cu(v), cu(beta), cu(d), cu(A), cu(ma), cu(mb),
                                          cu(mc), cu(md), cu(lam0), I_prior=1.0, I0=cu(I0), mu0=cu(mu0),
                                          lambda_out=lam_out)
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    ro, rmu, rI = oracle.diag_scan(q, k, v, beta, d, A, 1.0, I0, mu0)
    rl = oracle.mobius_scan(ma, mb, mc, md, lam0)
    parity.assert_close(o.cpu(), ro, parity.TOL_DIAG, "o")
    parity.assert_close(fs[0].cpu(), rmu, parity.TOL_DIAG, "mu_T")
    parity.assert_close(fs[1].cpu(), rI, parity.TOL_DIAG, "I_T")
    parity.assert_close(lam.cpu(), rl, parity.TOL_MOBIUS, "lambda")
    return kdn.diag_scan_plan(B, H, T, dk, dv, dtype)


@pytest.mark.parametrize("dk,dv,dtype", [(128, 128, torch.bfloat16), (64, 64, torch.bfloat16),
                                         (32, 32, torch.bfloat16), (16, 16, torch.float32),
                                         (64, 32, torch.float32), (128, 64, torch.bfloat16)])
def test_fused_matches_oracle(dk, dv, dtype):
    # 12 heads, 3 lambda tiles of the 128-thread walkers (ragged last tile)
    run_and_check(2, 6, 2600, dk, dv, dtype, seed=dk + dv)


def test_fused_with_token_split_and_initial_state():
    plan = run_and_check(1, 2, 2048, 128, 128, A_law=("uniform", 0.1, 1.0), seed=5, state=True)
    assert plan["parts"] > 1


@pytest.mark.parametrize("T", [1, 4, 8, 100, 2049])
def test_fused_short_and_ragged(T):
    run_and_check(1, 3, T, 64, 64, seed=T)


@pytest.mark.parametrize("T,offset", [(1001, 0), (1000, 1)])
def test_fused_unaligned_layouts_take_the_separate_launch(T, offset):
    # T % 4 != 0, or lambda_out not 16-byte aligned: same results through the
    # separate Moebius launch
    run_and_check(2, 2, T, 128, 128, seed=T + offset, lam_offset=offset)


def test_fused_zero_length_writes_the_initial_state():
    from bayesian_scan_gb300 import kdn
    B, H, dk, dv = 1, 2, 64, 64
    x = [torch.empty(B, H, 0, dk, device="cuda", dtype=torch.bfloat16) for _ in range(2)]
    y = [torch.empty(B, H, 0, dv, device="cuda", dtype=torch.bfloat16) for _ in range(2)]
    d = torch.empty(B, H, 0, device="cuda", dtype=torch.bfloat16)
    A = torch.ones(H, device="cuda")
    m = [torch.empty(B * H, 0, device="cuda") for _ in range(4)]
    lam0 = torch.ones(B * H, device="cuda")
    o, fs, lam = kdn.diag_mobius_scan_fwd(x[0], x[1], y[0], y[1], d, A, *m, lam0, I_prior=2.0)
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    assert lam.numel() == 0 and o.numel() == 0
    assert bool((fs[0] == 0).all()) and bool((fs[1] == 2.0).all())


def test_fused_equals_the_two_separate_calls():
    """The fused launch gives the scan's outputs bit for bit (same kernels)
    and lambda within rounding of kdn_mobius_scan (the walkers' tile length
    follows the scan CTA's thread count)."""
    from bayesian_scan_gb300 import kdn
    w = workloads.get("layer1p3b_t1024")
    inp = workloads.make(w)
    x = [inp[n].cuda() for n in ("q", "k", "v", "beta", "d", "A")]
    mob = [inp[n].cuda() for n in ("ma", "mb", "mc", "md", "lam0")]
    o1, fs1 = kdn.diag_scan_fwd(*x, I_prior=inp["I_prior"])
    l1 = kdn.mobius_scan(*mob)
    o2, fs2, l2 = kdn.diag_mobius_scan_fwd(*x, *mob, I_prior=inp["I_prior"])
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(fs1, fs2)
    assert parity.rel_err(l2.cpu(), l1.cpu()) < 1e-6
