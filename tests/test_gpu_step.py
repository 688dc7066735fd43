"""kdn_diag_step (one token on a device-resident state, batched decoding)
against the fp64 oracle's T = 1 scan from the same state, and a run of steps
against one scan call over the same tokens."""
import pytest
import torch

from bayesian_scan_gb300 import workloads
import parity

pytestmark = pytest.mark.gpu


def random_state(B, H, dv, dk, seed, I_lo=0.5):
    g = torch.Generator().manual_seed(seed)
    I = I_lo + torch.rand(B, H, dv, dk, generator=g) * 3.0
    mu = torch.randn(B, H, dv, dk, generator=g)
    return mu, I


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 64), (128, 128), (128, 32), (64, 128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_step_matches_oracle(dk, dv, dtype):
    from bayesian_scan_gb300 import kdn
    B, H = 3, 5
    q, k, v, beta, d, A = workloads.draw_diag(B, H, 1, dk, dv, dtype, ("uniform", 0.5, 4.0), seed=dk + dv)
    mu, I = random_state(B, H, dv, dk, seed=dk * dv)
    state = torch.stack([mu, I]).cuda()
    out = kdn.diag_step(*(x[:, :, 0].contiguous().cuda() if x.dim() >= 3 else x.cuda()
                          for x in (q, k, v, beta, d)), A.cuda(), state, I_prior=1.0)
    torch.cuda.synchronize()
    ro, rmu, rI = oracle_step(q, k, v, beta, d, A, mu, I)
    parity.assert_close(out.cpu(), ro[:, :, 0], parity.TOL_DIAG)
    parity.assert_close(state[0].cpu(), rmu, parity.TOL_DIAG)
    parity.assert_close(state[1].cpu(), rI, parity.TOL_DIAG)


def oracle_step(q, k, v, beta, d, A, mu, I):
    inp = dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=1.0)
    return parity.oracle_diag(inp, I, mu)


def test_steps_equal_a_scan():
    # 64 steps from the prior state == one scan over the same 64 tokens
    from bayesian_scan_gb300 import kdn
    B, H, T, dk, dv = 2, 3, 64, 64, 64
    q, k, v, beta, d, A = workloads.draw_diag(B, H, T, dk, dv, torch.bfloat16, ("uniform", 0.5, 4.0), seed=5)
    inp = dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=1.0)
    o_scan, fs_scan = parity.gpu_diag(inp)
    state = torch.stack([torch.zeros(B, H, dv, dk), torch.ones(B, H, dv, dk)]).cuda()
    dev = [x.cuda() for x in (q, k, v, beta, d)]
    outs = []
    for t in range(T):
        outs.append(kdn.diag_step(*(x[:, :, t].contiguous() for x in dev), A.cuda(), state).cpu())
    torch.cuda.synchronize()
    o_steps = torch.stack(outs, dim=2)
    assert parity.rel_err(o_steps, o_scan) < 1e-4
    assert parity.rel_err(state[0].cpu(), fs_scan[0]) < 1e-4
    assert parity.rel_err(state[1].cpu(), fs_scan[1]) < 1e-4


def test_step_many_heads():
    # more rows than one grid pass (grid-stride loop) and a ragged row count
    from bayesian_scan_gb300 import kdn
    B, H, dk, dv = 40, 130, 128, 128
    q, k, v, beta, d, A = workloads.draw_diag(B, H, 1, dk, dv, torch.bfloat16, ("uniform", 0.5, 4.0), seed=9)
    mu, I = random_state(B, H, dv, dk, seed=9)
    state = torch.stack([mu, I]).cuda()
    out = kdn.diag_step(*(x[:, :, 0].contiguous().cuda() for x in (q, k, v, beta, d)), A.cuda(), state)
    torch.cuda.synchronize()
    # sampled heads against the oracle
    for bh in (0, 777, 40 * 130 - 1):
        b, h = divmod(bh, 130)
        sl = lambda x: x[b:b + 1, h:h + 1]
        ro, rmu, rI = oracle_step(sl(q), sl(k), sl(v), sl(beta), sl(d), A[h:h + 1], sl(mu), sl(I))
        parity.assert_close(out[b:b + 1, h:h + 1].cpu(), ro[:, :, 0], parity.TOL_DIAG)
        parity.assert_close(state[0, b:b + 1, h:h + 1].cpu(), rmu, parity.TOL_DIAG)
        parity.assert_close(state[1, b:b + 1, h:h + 1].cpu(), rI, parity.TOL_DIAG)
