"""The factors a user brings: the pages' orientation (W ~ A_r B_r) and the offline SVD tool.

lr_factor_pack turns row-major A_r [d_in][r] and B_r [r][d_out] into the
library's At = A_r^T and Bt = B_r^T bit for bit; factorize() splits a dense W
by truncated SVD.  The factors then go through lr_linear_forward and are
checked against the oracle of the same (rounded) factors, and the product
against the dense x W within the Eckart-Young truncation bound.
"""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import assert_parity, dev_bits, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402
from rank_decomposed_gb300.factorize import factorize  # noqa: E402


@pytest.mark.parametrize("d_in,d_out,r", [(512, 768, 64), (4096, 4096, 1216), (1024, 320, 192)])
def test_factor_pack_is_an_exact_transpose(d_in, d_out, r):
    A_bits = synth.bf16_normal(31, synth.make_tag(0, 0, synth.KIND_A), (d_in, r), 0.05)
    B_bits = synth.bf16_normal(31, synth.make_tag(0, 0, synth.KIND_B), (r, d_out), 0.05)
    f = lr.factor_pack(dev_bits(A_bits), dev_bits(B_bits))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(f.At), A_bits.T)
    assert np.array_equal(host_bits(f.Bt), B_bits.T)
    assert (f.d_in, f.d_out, f.r) == (d_in, d_out, r)


def test_factorize_then_linear_against_oracle_and_eckart_young():
    d_in, d_out, r, M = 1024, 768, 128, 16
    g = torch.Generator().manual_seed(7)
    # W with a known spectrum: r singular values near 1, the rest 1e-3, so the
    # truncation error is set by the tail (Eckart-Young)
    U, _ = torch.linalg.qr(torch.randn(d_in, d_in, generator=g, dtype=torch.float64))
    V, _ = torch.linalg.qr(torch.randn(d_out, d_out, generator=g, dtype=torch.float64))
    s = torch.cat([1.0 + torch.rand(r, generator=g, dtype=torch.float64), torch.full((d_out - r,), 1e-3,
                                                                                     dtype=torch.float64)])
    W = (U[:, :d_out] * s) @ V.T
    fz = factorize(W.cuda(), r=r)
    f = lr.FactorPair(fz.At, fz.Bt)
    tail = float(torch.sqrt(torch.sum(s[r:] ** 2) / torch.sum(s ** 2)))
    assert abs(fz.rel_error - tail) < 1e-6

    x_bits = synth.bf16_normal(32, synth.make_tag(0, 0, synth.KIND_X), (M, d_in))
    x = dev_bits(x_bits)
    y = torch.empty((M, d_out), dtype=torch.float32, device="cuda")
    ws = torch.zeros(lr.linear_workspace_bytes(M, f), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.linear_forward(x, f, y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    yv = y.cpu().numpy().astype(np.float64)
    xf = oracle.widen_bf16(x_bits)
    A, B = oracle.factor_from_stored(host_bits(fz.At), host_bits(fz.Bt))
    assert_parity(yv, oracle.lowrank_linear(xf, A, B)[1], "factorized W through the library")
    # against the dense product: the truncation (Eckart-Young, spectral norm
    # sigma_{r+1} = 1e-3) plus the bf16 rounding of the factors and of t
    # (about 2^-8 relative per element, summed in quadrature)
    err = np.linalg.norm(yv - xf @ W.numpy())
    bound = np.linalg.norm(xf) * 1e-3 + 4 * 2.0 ** -8 * np.linalg.norm(xf @ W.numpy())
    assert err <= bound, (err, bound)
    # the pages' orientation packs to the same stored factors
    Ar = fz.At.t().contiguous()
    Br = fz.Bt.t().contiguous()
    g2 = lr.factor_pack(Ar, Br)
    torch.cuda.synchronize()
    assert torch.equal(g2.At, fz.At) and torch.equal(g2.Bt, fz.Bt)
