"""Seeded synthetic inputs: deterministic, right shapes, dtypes and laws."""
import torch

from bayesian_scan_gb300 import workloads


def test_deterministic_and_shaped():
    a = workloads.make("small")
    b = workloads.make("small")
    for k in a:
        if torch.is_tensor(a[k]):
            assert torch.equal(a[k], b[k]), k
    w = workloads.get("small")
    assert a["q"].shape == (w.B, w.H, w.T, w.dk) and a["q"].dtype == torch.float32
    assert a["v"].shape == (w.B, w.H, w.T, w.dv)
    assert a["ma"].shape == (w.mobius_N, w.mobius_T)


def test_laws():
    q, k, v, beta, d, A = workloads.draw_diag(2, 4, 512, 64, 32, torch.bfloat16,
                                              ("uniform", 0.5, 4.0), seed=1)
    assert q.dtype == torch.bfloat16 and A.dtype == torch.float32
    norms = k.float().norm(dim=-1)
    assert torch.allclose(norms, torch.ones_like(norms), atol=1e-2)   # L2-normalised keys
    assert float(beta.min()) > 0 and float(beta.max()) < 1            # sigmoid gate
    assert float(d.min()) >= 0                                         # softplus input
    assert float(A.min()) >= 0.5 and float(A.max()) <= 4.0
    a, b_, c, dd, lam0 = workloads.draw_mobius(3, 1000, seed=2)
    assert 0.5 <= float(a.min()) and float(a.max()) <= 1.5
    assert 0.0 <= float(b_.min()) and float(c.max()) <= 0.5
    assert torch.all(lam0 == 1)


def test_named_workloads_match_their_sizes():
    w = workloads.get("layer750m")
    assert (w.B, w.H, w.T, w.dk, w.dv, w.mobius_N, w.mobius_T) == (8, 16, 4096, 128, 128, 128, 4096)
    w = workloads.get("longctx")
    assert (w.B, w.H, w.T, w.mobius_N, w.mobius_T) == (1, 16, 65536, 4096, 16384)
    assert [workloads.get(i).name for i in range(5)] == workloads.ORDER
