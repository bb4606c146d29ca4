"""The offline SVD factorisation tool: rank-r weights are reproduced, Eckart-Young error."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
from rank_decomposed_gb300.factorize import factorize, rank_for  # noqa: E402


def _widen(t):
    return t.to(torch.float64).cpu().numpy()


def test_rank_r_weight_is_reproduced():
    g = torch.Generator().manual_seed(3)
    d_in, d_out, r = 256, 192, 64
    W = torch.randn(d_in, r, generator=g, dtype=torch.float64) @ torch.randn(r, d_out, generator=g, dtype=torch.float64)
    f = factorize(W, r=r)
    assert f.At.shape == (r, d_in) and f.Bt.shape == (d_out, r)
    assert f.rel_error < 1e-6                      # nothing beyond rank r to discard
    Wr = _widen(f.At).T @ _widen(f.Bt).T            # A_r B_r from the stored bf16 factors
    Wn = W.numpy()
    assert np.linalg.norm(Wr - Wn) / np.linalg.norm(Wn) < 1e-2   # bf16 rounding of the factors


def test_eckart_young_error_and_rank_rule():
    g = torch.Generator().manual_seed(4)
    W = torch.randn(256, 320, generator=g, dtype=torch.float64)
    f = factorize(W, rho=0.4)
    assert f.At.shape[0] == rank_for(256, 320, 0.4) == 64 * round(0.6 * 256 * 320 / 576 / 64)
    s = np.linalg.svd(W.numpy(), compute_uv=False)
    r = f.At.shape[0]
    assert abs(f.rel_error - np.sqrt(np.sum(s[r:] ** 2) / np.sum(s ** 2))) < 1e-6
    # the product of the (fp32) factors before rounding has exactly that error
    U, S, Vh = np.linalg.svd(W.numpy(), full_matrices=False)
    Wr = (U[:, :r] * S[:r]) @ Vh[:r]
    assert abs(np.linalg.norm(W.numpy() - Wr) / np.linalg.norm(W.numpy()) - f.rel_error) < 1e-6
    with pytest.raises(ValueError):
        factorize(W, r=100)
