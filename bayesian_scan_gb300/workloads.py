"""Seeded synthetic workloads for the diagonal scan and the Moebius scan.

This module only draws inputs.  It holds none of the scans' arithmetic and
imports neither the CUDA library nor the oracle, so both sides can be fed the
exact same tensors.

Recipe (all draws on the CPU with ``torch.Generator`` in fp32, in this order:
q, k, v, beta, d, A, then the Moebius a, b, c, d):

* q, v ~ N(0, 1); k ~ N(0, 1), then L2-normalised along d_k (in fp32);
* beta = sigmoid(N(0, 1)) on the value axis (d_v);
* d = softplus(N(0, 1)), one scalar per (b, h, t);
* A: 1 for the small cases, U[0.5, 4] per head for the 750M- and 1.3B-shaped
  layers, U[0.1, 1] per head for the long-context case;
* I_prior = 1, no initial state (I_0 = I_prior, mu_0 = 0);
* Moebius coefficients a, d ~ U[0.5, 1.5], b, c ~ U[0, 0.5], lambda_0 = 1;
* q, k, v, beta, d are then cast to the workload dtype (bf16 except the
  smallest case, which stays fp32); A, I_prior and the Moebius arrays stay
  fp32.

The named workloads mirror the model shapes the pages study (750M and 1.3B
parameter layers, long contexts); see ``WORKLOADS``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    dtype: torch.dtype
    A_law: tuple            # ("const", v) or ("uniform", lo, hi)
    mobius_N: int           # number of Moebius sequences
    mobius_T: int           # their length
    mobius_fused: bool      # one lambda sequence per head over the same T
    seed: int
    I_prior: float = 1.0

    @property
    def tokens(self) -> int:
        """Token-heads of one diagonal-scan pass: B*H*T."""
        return self.B * self.H * self.T

    @property
    def mobius_steps(self) -> int:
        return self.mobius_N * self.mobius_T

    def describe(self) -> str:
        dt = "bf16" if self.dtype == torch.bfloat16 else "fp32"
        return (f"B={self.B},H={self.H},T={self.T},d_k={self.dk},d_v={self.dv},{dt} "
                f"inputs, fp32 state; Moebius {self.mobius_N}x{self.mobius_T} fp32")


WORKLOADS = {
    # the small case the oracle finishes in well under a second
    "small": Workload("small", 1, 1, 256, 16, 16, torch.float32, ("const", 1.0), 1, 256, True, 1000),
    # 32 heads of d=64 over 2048 tokens, per-head lambda
    "heads32_t2048_d64": Workload("heads32_t2048_d64", 4, 8, 2048, 64, 64, torch.bfloat16,
                                  ("const", 1.0), 32, 2048, True, 1001),
    # 750M-shaped layer: 8x16 heads of d=128 over 4096 tokens, fused per-head lambda
    "layer750m": Workload("layer750m", 8, 16, 4096, 128, 128, torch.bfloat16,
                          ("uniform", 0.5, 4.0), 128, 4096, True, 1002),
    # 1.3B-shaped layer: 16x32 heads of d=64 over 4096 tokens, per-head lambda
    "layer1p3b": Workload("layer1p3b", 16, 32, 4096, 64, 64, torch.bfloat16,
                          ("uniform", 0.5, 4.0), 512, 4096, True, 1003),
    # long context: 16 heads of d=128 over 65536 tokens (slow forgetting);
    # standalone Moebius scan over 4096 sequences of 16384 steps
    "longctx": Workload("longctx", 1, 16, 65536, 128, 128, torch.bfloat16,
                        ("uniform", 0.1, 1.0), 4096, 16384, False, 1004),
    # the 1.3B-shaped layer's heads over 1024 tokens: one wave of the d=64
    # kernel (inputs still larger than L2), for profiling captures
    "layer1p3b_t1024": Workload("layer1p3b_t1024", 16, 32, 1024, 64, 64, torch.bfloat16,
                                ("uniform", 0.5, 4.0), 512, 1024, True, 1008),
}
# batched decoding (one token per head per step on a device-resident state):
# 128 x 16 heads of d=128, whose 268 MB state is twice the 129 MB L2; 32
# tokens of inputs for successive steps
DECODE = {
    "decode2k": Workload("decode2k", 128, 16, 32, 128, 128, torch.bfloat16,
                         ("uniform", 0.5, 4.0), 0, 0, False, 1005),
}
WORKLOADS.update(DECODE)
# training: the backward pass of the 750M-shaped layer (same inputs, same
# seed); the gradient flowing into the outputs is drawn by draw_cotangents
# from the next seed
TRAIN = {
    "layer750m_bwd": Workload("layer750m_bwd", 8, 16, 4096, 128, 128, torch.bfloat16,
                              ("uniform", 0.5, 4.0), 0, 0, False, 1002),
    # a one-wave case of the same head shape (32 heads x 1024 tokens) for
    # profiling captures
    "heads32_t1024_bwd": Workload("heads32_t1024_bwd", 2, 16, 1024, 128, 128, torch.bfloat16,
                                  ("uniform", 0.5, 4.0), 0, 0, False, 1006),
    # the backward pass of the 1.3B-shaped layer and of the long context
    # (same inputs and seeds as their forward workloads)
    "layer1p3b_bwd": Workload("layer1p3b_bwd", 16, 32, 4096, 64, 64, torch.bfloat16,
                              ("uniform", 0.5, 4.0), 0, 0, False, 1003),
    "longctx_bwd": Workload("longctx_bwd", 1, 16, 65536, 128, 128, torch.bfloat16,
                            ("uniform", 0.1, 1.0), 0, 0, False, 1004),
    # the long context's 16 heads over 4096 tokens (the same 16-column
    # blocks, about 1 GB of checkpoints) for profiling captures
    "heads16_t4096_bwd": Workload("heads16_t4096_bwd", 1, 16, 4096, 128, 128, torch.bfloat16,
                                  ("uniform", 0.1, 1.0), 0, 0, False, 1009),
}
WORKLOADS.update(TRAIN)
# the non-metaplastic limit (importance held at I_prior) on the layer shapes
# and the long context: same inputs and seeds as the metaplastic workloads
LIN = {
    "layer750m_lin": Workload("layer750m_lin", 8, 16, 4096, 128, 128, torch.bfloat16,
                              ("uniform", 0.5, 4.0), 0, 0, False, 1002),
    "longctx_lin": Workload("longctx_lin", 1, 16, 65536, 128, 128, torch.bfloat16,
                            ("uniform", 0.1, 1.0), 0, 0, False, 1004),
    # one wave of the 750M layer's heads over 512 tokens, for profiling captures
    "heads128_t512_lin": Workload("heads128_t512_lin", 8, 16, 512, 128, 128, torch.bfloat16,
                                  ("uniform", 0.5, 4.0), 0, 0, False, 1007),
}
WORKLOADS.update(LIN)

# the five scan configurations in the order the configuration list gives them
ORDER = ["small", "heads32_t2048_d64", "layer750m", "layer1p3b", "longctx"]


def get(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[ORDER[name_or_index]]
    return WORKLOADS[name_or_index]


def draw_diag(B, H, T, dk, dv, dtype=torch.bfloat16, A_law=("const", 1.0), seed=0,
              gen: torch.Generator | None = None):
    """Draw (q, k, v, beta, d, A) on the CPU.  q,k: [B,H,T,dk]; v,beta:
    [B,H,T,dv]; d: [B,H,T] (all ``dtype``); A: [H] fp32."""
    g = gen if gen is not None else torch.Generator().manual_seed(seed)
    f32 = torch.float32
    q = torch.randn(B, H, T, dk, generator=g, dtype=f32)
    k = torch.randn(B, H, T, dk, generator=g, dtype=f32)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    v = torch.randn(B, H, T, dv, generator=g, dtype=f32)
    beta = torch.sigmoid(torch.randn(B, H, T, dv, generator=g, dtype=f32))
    d = torch.nn.functional.softplus(torch.randn(B, H, T, generator=g, dtype=f32))
    if A_law[0] == "const":
        A = torch.full((H,), float(A_law[1]), dtype=f32)
    else:
        A = torch.rand(H, generator=g, dtype=f32) * (A_law[2] - A_law[1]) + A_law[1]
    cast = lambda x: x.to(dtype).contiguous()
    return cast(q), cast(k), cast(v), cast(beta), cast(d), A.contiguous()


def draw_cotangents(B, H, T, dk, dv, seed=0, gen: torch.Generator | None = None):
    """Draw the gradients that flow into a backward call: grad_out
    [B,H,T,dv] and grad_final_state [2,B,H,dv,dk], fp32 N(0,1)."""
    g = gen if gen is not None else torch.Generator().manual_seed(seed)
    gout = torch.randn(B, H, T, dv, generator=g, dtype=torch.float32)
    gfs = torch.randn(2, B, H, dv, dk, generator=g, dtype=torch.float32)
    return gout, gfs


def draw_mobius(N, T, seed=0, gen: torch.Generator | None = None):
    """Draw Moebius coefficients a, b, c, d [N,T] and lambda0 [N] (fp32)."""
    g = gen if gen is not None else torch.Generator().manual_seed(seed)
    f32 = torch.float32
    a = torch.rand(N, T, generator=g, dtype=f32) + 0.5
    b = torch.rand(N, T, generator=g, dtype=f32) * 0.5
    c = torch.rand(N, T, generator=g, dtype=f32) * 0.5
    d = torch.rand(N, T, generator=g, dtype=f32) + 0.5
    lam0 = torch.ones(N, dtype=f32)
    return a, b, c, d, lam0


def make(w: Workload | str | int, with_mobius: bool = True):
    """All inputs of a workload, drawn in the documented order from one seed."""
    if not isinstance(w, Workload):
        w = get(w)
    g = torch.Generator().manual_seed(w.seed)
    q, k, v, beta, d, A = draw_diag(w.B, w.H, w.T, w.dk, w.dv, w.dtype, w.A_law, gen=g)
    out = dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=w.I_prior)
    if with_mobius:
        a, b, c, dd, lam0 = draw_mobius(w.mobius_N, w.mobius_T, gen=g)
        out.update(ma=a, mb=b, mc=c, md=dd, lam0=lam0)
    return out
