"""The Python binding's own argument checks (bayesian_scan_gb300/kdn.py): they
run before any CUDA call, so they are tested here without a GPU.  The C-ABI's
validation is covered by test_abi.py."""
import pytest
import torch

from bayesian_scan_gb300 import workloads


@pytest.fixture(scope="module")
def kdn():
    from bayesian_scan_gb300 import kdn as k
    return k


def diag_inputs(B=2, H=3, T=5, dk=16, dv=16, dtype=torch.bfloat16):
    q, k, v, beta, d, A = workloads.draw_diag(B, H, T, dk, dv, dtype, ("const", 1.0), seed=1)
    return dict(q=q, k=k, v=v, beta=beta, d=d, A=A)


def test_host_diag_rejects_bad_shapes_and_dtypes(kdn):
    x = diag_inputs()
    bad = dict(x, k=x["k"][:, :, :4].contiguous())
    with pytest.raises(ValueError, match="k must have shape"):
        kdn.diag_scan_fwd(*(bad[n] for n in ("q", "k", "v", "beta", "d", "A")))
    bad = dict(x, A=x["A"].double())
    with pytest.raises(ValueError, match="A must be torch.float32"):
        kdn.diag_scan_fwd(*(bad[n] for n in ("q", "k", "v", "beta", "d", "A")))
    bad = {n: t.to(torch.float16) if n != "A" else t for n, t in x.items()}
    with pytest.raises(ValueError, match="bf16 or fp32"):
        kdn.diag_scan_fwd(*(bad[n] for n in ("q", "k", "v", "beta", "d", "A")))
    bad = dict(x, v=x["v"].transpose(2, 3))
    with pytest.raises(ValueError, match="v must"):
        kdn.diag_scan_fwd(*(bad[n] for n in ("q", "k", "v", "beta", "d", "A")))
    bad_mu0 = torch.zeros(2, 3, 16, 8)
    with pytest.raises(ValueError, match="mu0 must have shape"):
        kdn.diag_scan_fwd(*(x[n] for n in ("q", "k", "v", "beta", "d", "A")), mu0=bad_mu0)


def test_device_only_entry_points_reject_host_tensors(kdn):
    x = diag_inputs()
    args = [x[n] for n in ("q", "k", "v", "beta", "d", "A")]
    with pytest.raises(ValueError, match="device tensors"):
        kdn.lin_scan_fwd(*args)
    gout = torch.zeros(2, 3, 5, 16)
    with pytest.raises(ValueError, match="device tensors"):
        kdn.diag_scan_bwd(*args, gout)
    state = torch.zeros(2, 2, 3, 16, 16)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        kdn.diag_step(*(t[:, :, 0].contiguous() if t.dim() >= 3 else t for t in args[:5]), args[5], state)


def test_lin_and_bwd_reject_other_dtypes(kdn):
    x = diag_inputs()
    args = [x[n].to(torch.float16) if n != "A" else x[n] for n in ("q", "k", "v", "beta", "d", "A")]
    with pytest.raises(ValueError, match="bf16 or fp32"):
        kdn.lin_scan_fwd(*args)
    with pytest.raises(ValueError, match="bf16 or fp32"):
        kdn.diag_scan_bwd(*args, torch.zeros(2, 3, 5, 16))


def test_host_mobius_rejects_bad_shapes(kdn):
    a = torch.ones(4, 7)
    with pytest.raises(ValueError):
        kdn.mobius_scan(a, a, a, torch.ones(4, 6), torch.ones(4))
    with pytest.raises(ValueError):
        kdn.mobius_scan(a, a, a, a, torch.ones(5))
    with pytest.raises(ValueError):
        kdn.mobius_scan(a, a, a, a.double(), torch.ones(4))


def test_bwd_workspace_query(kdn):
    # the size of the backward's scratch: every 8th token's state plus the
    # column blocks' row partials (no GPU work)
    n = kdn.diag_scan_bwd_workspace(8, 16, 4096, 128, 128)
    BH, T, d = 8 * 16, 4096, 128
    assert n >= BH * T * d * d * 4 // 8 + 4 * BH * T * 2 * d * 4
    assert kdn.diag_scan_bwd_workspace(1, 1, 0, 16, 16) == 0
    with pytest.raises(kdn.KdnError):
        kdn.diag_scan_bwd_workspace(1, 1, 8, 24, 16)
    with pytest.raises(kdn.KdnError):
        kdn.diag_scan_bwd_workspace(0, 1, 8, 16, 16)


def test_device_entry_points_reject_host_operands(kdn):
    """Every operand of a device call is checked, not only the first: a host
    tensor among them is refused before the C ABI sees its pointer.  (On a
    machine without a GPU the first operand stands in for a device tensor
    with a meta tensor, which passes the first check and fails the second.)"""
    a = torch.ones(4, 8)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        kdn.mobius_scan_noalloc(a, a, a, a, torch.ones(4), torch.empty(4, 8))
    x = diag_inputs()
    args = [x[n] for n in ("q", "k", "v", "beta", "d", "A")]
    gout = torch.zeros(2, 3, 5, 16)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        kdn._on_one_device(None, q=args[0], gout=gout)


def test_mixed_host_and_device_operands_are_refused(kdn):
    """A call whose first operand is on the device but another one is not
    (here the device operand is a meta tensor, so no GPU is needed: it fails
    the device check the same way a CUDA tensor on another device would)."""
    dev_like = torch.empty(4, 8, device="meta")
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        kdn._on_one_device(None, a=torch.ones(4, 8), b=dev_like)
    host = torch.ones(4, 8)
    with pytest.raises(ValueError, match="lambda0 must be a CUDA tensor"):
        kdn._on_one_device(None, lambda0=host)
