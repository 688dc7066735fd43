"""Diagonal scan: CUDA path vs the fp64 oracle, element by element, on
seeded inputs spanning several chunks, ragged tails, token splits, every
supported head dimension and the degenerate cases."""
import pytest
import torch

from bayesian_scan_gb300 import workloads
import parity

pytestmark = pytest.mark.gpu


def draw(B, H, T, dk, dv, dtype=torch.bfloat16, A_law=("uniform", 0.5, 4.0), seed=7):
    q, k, v, beta, d, A = workloads.draw_diag(B, H, T, dk, dv, dtype, A_law, seed=seed)
    return dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=1.0)


def test_small_workload_fp32():
    inp = workloads.make("small", with_mobius=False)
    parity.check_diag(inp)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 32), (64, 64), (128, 128), (32, 64),
                                   (64, 32), (128, 16), (16, 128), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_head_dims(dk, dv, dtype):
    parity.check_diag(draw(2, 3, 77, dk, dv, dtype))


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 33, 48, 100])
def test_short_and_ragged_lengths(T):
    parity.check_diag(draw(1, 2, T, 64, 64))


def test_zero_length_returns_initial_state():
    inp = draw(1, 2, 0, 32, 32)
    g = torch.Generator().manual_seed(3)
    I0 = 0.5 + torch.rand(1, 2, 32, 32, generator=g)
    mu0 = torch.randn(1, 2, 32, 32, generator=g)
    o, fs = parity.gpu_diag(inp, I0, mu0)
    assert o.numel() == 0
    assert parity.rel_err(fs[0], mu0) < 1e-6 and parity.rel_err(fs[1], I0) < 1e-6


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_given_initial_state(dtype):
    inp = draw(2, 2, 90, 64, 64, dtype)
    g = torch.Generator().manual_seed(5)
    I0 = 0.3 + 3 * torch.rand(2, 2, 64, 64, generator=g)
    mu0 = torch.randn(2, 2, 64, 64, generator=g)
    parity.check_diag(inp, I0, mu0)
    parity.check_diag(inp, I0, None)
    parity.check_diag(inp, None, mu0)


def test_heads_not_a_multiple_of_heads_per_block():
    parity.check_diag(draw(1, 3, 40, 64, 32))     # 4 heads per block, 3 heads
    parity.check_diag(draw(3, 5, 21, 16, 16))     # 8 heads per block, 15 heads


@pytest.mark.parametrize("T", [4096, 3001])
def test_token_split_path(T):
    # one head: the library splits the tokens into parts (aggregate, carry, full)
    parity.check_diag(draw(1, 1, T, 128, 128, A_law=("uniform", 0.1, 1.0)))
    parity.check_diag(draw(1, 2, T, 64, 64, A_law=("const", 1.0)))


@pytest.mark.parametrize("law", [("const", 0.0), ("uniform", 0.1, 1.0), ("const", 30.0)])
@pytest.mark.parametrize("T", [2048, 3001])
def test_token_split_tensor_core_aggregates(law, T):
    # d_k = d_v = 128 with bf16 inputs: the parts' end states come from the
    # tensor-core aggregate pass (no decay, slow decay, decay that underflows;
    # a ragged last chunk for T = 3001)
    from bayesian_scan_gb300 import kdn
    assert kdn.diag_scan_plan(1, 2, T, 128, 128)["parts"] > 1
    parity.check_diag(draw(1, 2, T, 128, 128, A_law=law, seed=T))


def test_long_memory_many_parts():
    """8192 tokens forgetting slowly (A d ~ 0.005: a memory of about 300
    tokens) split into 64 parts, 63 carries.  Per tensor the outputs stay
    near 1e-6 of the oracle.  Element-wise at the 1e-3 rms floor the bar is
    looser than 2e-3: the state is fp32 and a memory of ~300 tokens carries
    a few tens of fp32 ulps of rounding per element, which an output that
    cancels down to 1e-3 rms shows as ~1e-3 to 1e-2 of itself (measured
    4e-3)."""
    from bayesian_scan_gb300 import kdn
    assert kdn.diag_scan_plan(1, 2, 8192, 128, 128)["parts"] >= 32
    parity.check_diag(draw(1, 2, 8192, 128, 128, A_law=("const", 0.005), seed=12), tol_elem=1e-2)


def test_token_split_tensor_core_aggregates_initial_state():
    inp = draw(1, 1, 2600, 128, 128, A_law=("const", 0.02))
    g = torch.Generator().manual_seed(10)
    I0 = 0.5 + torch.rand(1, 1, 128, 128, generator=g)
    mu0 = torch.randn(1, 1, 128, 128, generator=g)
    parity.check_diag(inp, I0, mu0)


def test_token_split_fp32_inputs_d128():
    # fp32 inputs keep the CUDA-core aggregate pass
    parity.check_diag(draw(1, 1, 2500, 128, 128, dtype=torch.float32, A_law=("uniform", 0.1, 1.0)))


def test_token_split_with_initial_state():
    inp = draw(1, 1, 2500, 64, 64, A_law=("const", 0.05))
    g = torch.Generator().manual_seed(9)
    I0 = 0.5 + torch.rand(1, 1, 64, 64, generator=g)
    mu0 = torch.randn(1, 1, 64, 64, generator=g)
    parity.check_diag(inp, I0, mu0)


def test_resume_equals_single_call():
    inp = draw(2, 2, 300, 64, 64)
    o_all, fs_all = parity.gpu_diag(inp)
    first = {k_: (v_[:, :, :123] if k_ in ("q", "k", "v", "beta", "d") else v_) for k_, v_ in inp.items()}
    second = {k_: (v_[:, :, 123:].contiguous() if k_ in ("q", "k", "v", "beta", "d") else v_)
              for k_, v_ in inp.items()}
    first = {k_: (v_.contiguous() if torch.is_tensor(v_) else v_) for k_, v_ in first.items()}
    o1, fs1 = parity.gpu_diag(first)
    o2, fs2 = parity.gpu_diag(second, I0=fs1[1], mu0=fs1[0])
    assert parity.rel_err(torch.cat([o1, o2], dim=2), o_all) < 1e-4
    assert parity.rel_err(fs2[0], fs_all[0]) < 1e-4
    assert parity.rel_err(fs2[1], fs_all[1]) < 1e-4


@pytest.mark.parametrize("law", [("const", 0.0), ("const", 1e-3), ("const", 30.0),
                                 ("const", 300.0), ("uniform", 0.5, 4.0)])
@pytest.mark.parametrize("d", [64, 128])
def test_gate_extremes(law, d):
    # A = 0 (no forgetting), tiny A, and very fast forgetting (alpha underflows;
    # the working scale rescales the state on most tokens); d = 128 takes the
    # full pass whose producers scale the rows' inputs by W
    parity.check_diag(draw(1, 2, 203, d, d, A_law=law))


def test_zero_gate_input():
    inp = draw(1, 2, 64, 32, 32)
    inp["d"] = torch.zeros_like(inp["d"])
    parity.check_diag(inp)


@pytest.mark.parametrize("I_prior", [1e-3, 1.0, 50.0, 1e4])
@pytest.mark.parametrize("d", [64, 128])
def test_prior_scale(I_prior, d):
    inp = draw(1, 2, 120, d, d)
    inp["I_prior"] = I_prior
    parity.check_diag(inp)


def test_output_written_only_where_expected():
    from bayesian_scan_gb300 import kdn
    inp = draw(1, 2, 50, 32, 32)
    dev = "cuda"
    out = torch.full((1, 2, 50 + 7, 32), 12345.0, device=dev)  # larger buffer: guard tail
    view = out[:, :, :50]
    args = [inp[n].to(dev) for n in ("q", "k", "v", "beta", "d", "A")]
    o, _ = kdn.diag_scan_fwd(*args, I_prior=1.0, out=torch.empty(1, 2, 50, 32, device=dev),
                             final_state=False)
    torch.cuda.synchronize()
    ro, _, _ = parity.oracle_diag(inp)
    parity.assert_close(o.cpu(), ro, parity.TOL_DIAG)
    assert torch.all(out[:, :, 50:] == 12345.0)
    assert view.shape == (1, 2, 50, 32)
