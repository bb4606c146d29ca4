"""Offline truncated-SVD factorisation of a dense weight into a factor pair.

The decomposition the method starts from (Spanish page, "Resumen Tecnico"
section 1: W ~ A B; English page section 1: low-rank decomposition such as SVD):
W [d_in, d_out] = U S V^T is truncated to its r largest singular values and
stored as A_r = U_r (the down factor) and B_r = S_r V_r^T (the up factor, so
the singular values sit in B_r), in the library's out-major bf16 layout
At = A_r^T [r][d_in], Bt = B_r^T [d_out][r].  By Eckart-Young the truncation
error is ||W - A_r B_r||_F^2 = sum_{i >= r} s_i^2, reported before the bf16
rounding of the factors.

This is an offline tool: the SVD is torch.linalg.svd (cuSOLVER on a GPU).
The hot path never calls it.
"""

from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction


def rank_for(d_in: int, d_out: int, rho) -> int:
    """Rank removing a fraction rho of a d_in x d_out weight's parameters, rounded to 64 (ties up)."""
    exact = (1 - Fraction(str(rho))) * d_in * d_out / (d_in + d_out)
    return int(64 * max((exact / 64 + Fraction(1, 2)).__floor__(), 1))


@dataclass
class Factorization:
    At: object           # bf16 [r][d_in]
    Bt: object           # bf16 [d_out][r]
    singular_values: object
    rel_error: float     # ||W - A_r B_r||_F / ||W||_F from the discarded singular values


def factorize(W, r: int | None = None, rho=None) -> Factorization:
    """Split a dense weight W [d_in, d_out] (torch tensor, any float dtype) into rank-r factors."""
    import torch
    if (r is None) == (rho is None):
        raise ValueError("give exactly one of r and rho")
    d_in, d_out = W.shape
    if r is None:
        r = rank_for(d_in, d_out, rho)
    if r <= 0 or r > min(d_in, d_out) or r % 64:
        raise ValueError("r must be a positive multiple of 64 and at most min(d_in, d_out)")
    Wf = W.to(torch.float32)
    U, S, Vh = torch.linalg.svd(Wf, full_matrices=False)
    A = U[:, :r]                                   # [d_in, r]
    B = S[:r, None] * Vh[:r]                       # [r, d_out]
    tail = torch.sum(S[r:].double() ** 2)
    total = torch.sum(S.double() ** 2)
    rel = float(torch.sqrt(tail / total)) if float(total) > 0 else 0.0
    At = A.t().contiguous().to(torch.bfloat16)
    Bt = B.t().contiguous().to(torch.bfloat16)
    return Factorization(At, Bt, S, rel)
