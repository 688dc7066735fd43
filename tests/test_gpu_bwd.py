"""kdn_diag_scan_bwd against the fp64 reverse-mode oracle: every gradient
(q, k, v, beta, d, A and the initial state), head sizes 16..128 with
d_k != d_v, bf16 and fp32 inputs, ragged token counts (partial last chunk of
the 8-token recompute), with and without an initial state and final-state
gradients."""
import pytest
import torch

from bayesian_scan_gb300 import workloads
import parity

pytestmark = pytest.mark.gpu


def make(B, H, T, dk, dv, dtype, A_law=("uniform", 0.5, 4.0), seed=0, state=False):
    q, k, v, beta, d, A = workloads.draw_diag(B, H, T, dk, dv, dtype, A_law, seed=seed)
    inp = dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=1.0)
    gout, gfs = workloads.draw_cotangents(B, H, T, dk, dv, seed=seed + 1)
    I0 = mu0 = None
    if state:
        g = torch.Generator().manual_seed(seed + 2)
        I0 = 0.5 + 3.0 * torch.rand(B, H, dv, dk, generator=g)
        mu0 = torch.randn(B, H, dv, dk, generator=g)
    return inp, gout, gfs, I0, mu0


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (64, 64), (128, 128), (128, 32),
                                   (16, 128), (128, 16)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bwd_matches_oracle(dk, dv, dtype):
    inp, gout, gfs, _, _ = make(2, 3, 37, dk, dv, dtype, seed=dk + 3 * dv)
    parity.check_bwd(inp, gout, gfs)


@pytest.mark.parametrize("T", [1, 7, 8, 9, 64, 131])
def test_bwd_token_counts(T):
    # chunk boundaries: fewer tokens than a chunk, exactly one, one more, many
    inp, gout, gfs, I0, mu0 = make(1, 2, T, 32, 32, torch.bfloat16, seed=T, state=True)
    parity.check_bwd(inp, gout, gfs, I0, mu0)


@pytest.mark.parametrize("law", [("const", 0.0), ("const", 1.0), ("uniform", 0.1, 1.0), ("const", 30.0)])
def test_bwd_gate_laws(law):
    # no forgetting (A = 0), slow, fast and near-total forgetting
    inp, gout, gfs, I0, mu0 = make(2, 2, 50, 64, 64, torch.bfloat16, A_law=law, seed=4, state=True)
    parity.check_bwd(inp, gout, gfs, I0, mu0)


def test_bwd_without_final_state_gradient():
    inp, gout, _, I0, mu0 = make(1, 3, 45, 128, 64, torch.bfloat16, seed=8, state=True)
    parity.check_bwd(inp, gout, None, I0, mu0)


def test_bwd_only_initial_mean_given():
    inp, gout, gfs, _, mu0 = make(2, 1, 20, 32, 16, torch.float32, seed=9, state=True)
    parity.check_bwd(inp, gout, gfs, None, mu0)


def test_bwd_zero_tokens():
    # T = 0: the initial state is the final state; grad_A = 0
    from bayesian_scan_gb300 import kdn
    B, H, dk, dv = 2, 3, 32, 64
    inp, gout, gfs, I0, mu0 = make(B, H, 0, dk, dv, torch.bfloat16, seed=1, state=True)
    g = parity.gpu_bwd(inp, gout, gfs, I0, mu0)
    # equal up to the rounding of dmu r mu - dmu r mu (fp32)
    assert parity.rel_err(g["init_state"], gfs) < 1e-6
    assert torch.count_nonzero(g["A"]) == 0


def test_bwd_is_deterministic():
    inp, gout, gfs, I0, mu0 = make(2, 2, 70, 64, 128, torch.bfloat16, seed=12, state=True)
    a = parity.gpu_bwd(inp, gout, gfs, I0, mu0)
    b = parity.gpu_bwd(inp, gout, gfs, I0, mu0)
    for n in a:
        assert torch.equal(a[n], b[n]), n


def test_bwd_chain_across_a_split():
    # backward of [h, T) from the carried state seeds the backward of [0, h):
    # together they equal one backward over [0, T) (GPU on both sides)
    from bayesian_scan_gb300 import kdn
    inp, gout, gfs, I0, mu0 = make(1, 2, 40, 64, 64, torch.bfloat16, seed=21, state=True)
    full = parity.gpu_bwd(inp, gout, gfs, I0, mu0)
    h = 17
    first = {n: (inp[n][:, :, :h].contiguous() if n in ("q", "k", "v", "beta", "d") else inp[n])
             for n in inp}
    second = {n: (inp[n][:, :, h:].contiguous() if n in ("q", "k", "v", "beta", "d") else inp[n])
              for n in inp}
    _, fs1 = parity.gpu_diag(first, I0, mu0)
    g2 = parity.gpu_bwd(second, gout[:, :, h:].contiguous(), gfs, fs1[1], fs1[0])
    g1 = parity.gpu_bwd(first, gout[:, :, :h].contiguous(), g2["init_state"], I0, mu0)
    for n in ("q", "k", "v", "beta", "d"):
        e = parity.rel_err(torch.cat([g1[n], g2[n]], dim=2), full[n])
        assert e < 1e-4, (n, e)
    assert parity.rel_err(g1["A"] + g2["A"], full["A"]) < 1e-4
    assert parity.rel_err(g1["init_state"], full["init_state"]) < 1e-4


def test_bwd_library_workspace_and_caller_workspace_agree():
    # workspace NULL: the call takes stream-ordered scratch itself
    import ctypes
    from bayesian_scan_gb300 import kdn
    B, H, T, dk, dv = 1, 2, 29, 64, 32
    inp, gout, gfs, I0, mu0 = make(B, H, T, dk, dv, torch.bfloat16, seed=33, state=True)
    ref = parity.gpu_bwd(inp, gout, gfs, I0, mu0)
    dev = "cuda"
    x = {n: inp[n].to(dev) for n in ("q", "k", "v", "beta", "d", "A")}
    go, gf, i0, m0 = gout.to(dev), gfs.to(dev), I0.to(dev), mu0.to(dev)
    f32 = dict(device=dev, dtype=torch.float32)
    out = dict(q=torch.empty(B, H, T, dk, **f32), k=torch.empty(B, H, T, dk, **f32),
               v=torch.empty(B, H, T, dv, **f32), beta=torch.empty(B, H, T, dv, **f32),
               d=torch.empty(B, H, T, **f32), A=torch.empty(H, **f32),
               init_state=torch.empty(2, B, H, dv, dk, **f32))
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = kdn.lib.kdn_diag_scan_bwd(p(x["q"]), p(x["k"]), p(x["v"]), p(x["beta"]), p(x["d"]),
                                   p(x["A"]), 1.0, p(i0), p(m0), p(go), p(gf), p(out["q"]),
                                   p(out["k"]), p(out["v"]), p(out["beta"]), p(out["d"]),
                                   p(out["A"]), p(out["init_state"]), B, H, T, dk, dv, 1, None, 0,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    for n in out:
        assert torch.equal(out[n].cpu(), ref[n]), n


def _mixed_head_count(sms, dk=128, dv=128):
    """The smallest head count whose 32-column blocks fill whole waves and
    leave a remainder of at most half a wave: the call then finishes the
    remainder's heads with 16-column blocks (two launches of the main
    kernel, each with its own partials and finalize).  A wave is one 8-warp
    CTA per SM (d_v = 128), or two CTAs of up to 4 warps."""
    ncb = dk // 32
    slots = sms * (1 if (dv // 4) * 8 > 128 else 2)
    for bh in range(1, 8 * slots):
        if bh * ncb * 2 <= sms:
            continue   # few heads: 16-column blocks throughout
        waves, rem = divmod(bh * ncb, slots)
        if waves >= 1 and rem > 0 and 2 * rem <= slots and (waves * slots) % ncb == 0:
            return bh
    raise AssertionError("no mixed plan for this SM count")


@pytest.mark.parametrize("dv", [128, 64])
def test_bwd_mixed_column_blocks(dv):
    # heads split between a launch of 32-column and one of 16-column blocks
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = _mixed_head_count(sms, dv=dv)
    inp, gout, gfs, I0, mu0 = make(1, H, 19, 128, dv, torch.bfloat16, seed=40 + dv, state=True)
    parity.check_bwd(inp, gout, gfs, I0, mu0)
