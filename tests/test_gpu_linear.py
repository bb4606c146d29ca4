"""GPU parity of the factorized linear y = (x A_r) B_r against the fp64 oracle."""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import (assert_parity, bf16_f64, dev_bits, dev_factor, gpu_normal, host_bits,
                         host_factor)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


def _run_linear(x, f, M, ydtype, ws=None, ld_extra=0):
    y = torch.full((M, f.d_out + ld_extra), float("nan"), dtype=ydtype, device="cuda")
    if ws is None:
        ws = torch.zeros(max(lr.linear_workspace_bytes(M, f), 256), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.linear_forward(x, f, y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y[:, : f.d_out]


def _ref(x_bits, A, B):
    return oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)[1]


def test_gpu_generator_matches_numpy():
    for shape, std, cs in [((7, 96), 0.5, None), ((64, 512), 1 / 8, synth.sigma_scale(512)),
                           ((300, 64), 2.0, None)]:
        tag = synth.make_tag(3, 2, synth.KIND_B)
        got = host_bits(gpu_normal(shape, 11, tag, std, cs))
        want = synth.bf16_normal(11, tag, shape, std, cs)
        assert np.array_equal(got, want)


def test_config0_single_linear():
    """x [4, 512], A_r [512, 64], B_r = diag(sigma) G [64, 512], seed 0."""
    M, d_in, d_out, r = 4, 512, 512, 64
    x_bits = synth.activations(0, M, d_in)
    At, Bt = synth.factor_pair(0, 0, 0, d_in, d_out, r)
    f = lr.FactorPair(dev_bits(At), dev_bits(Bt))
    A, B = oracle.factor_from_stored(At, Bt)
    y_ref = _ref(x_bits, A, B)
    x = dev_bits(x_bits)
    y32 = _run_linear(x, f, M, torch.float32)
    assert_parity(y32.cpu().numpy(), y_ref, "config0 f32")
    y16 = _run_linear(x, f, M, torch.bfloat16)
    # a bf16 y is the round-to-nearest-even image of the fp32 y
    assert torch.equal(y16, y32.to(torch.bfloat16))


@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 31, 33, 64, 65, 100, 128, 129, 200, 256])
def test_decode_linear_ragged(M):
    d_in, d_out, r = 512, 1088, 192     # d_out = 8.5 tiles of 128
    f = dev_factor(5, 1, 0, d_in, d_out, r)
    A, B = host_factor(5, 1, 0, d_in, d_out, r)
    x_bits = synth.bf16_normal(5, synth.make_tag(M, 0, synth.KIND_X), (M, d_in))
    y = _run_linear(dev_bits(x_bits), f, M, torch.float32)
    assert_parity(y.cpu().numpy(), _ref(x_bits, A, B), "decode M=%d" % M)


@pytest.mark.parametrize("shape", [(4096, 4096, 1216), (4096, 11008, 1792), (11008, 4096, 1792)])
@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_decode_linear_llama7b(shape, M):
    d_in, d_out, r = shape
    f = dev_factor(0, 0, 4, d_in, d_out, r)
    A, B = host_factor(0, 0, 4, d_in, d_out, r)
    x_bits = synth.activations(0, M, d_in)
    y = _run_linear(dev_bits(x_bits), f, M, torch.float32)
    assert_parity(y.cpu().numpy(), _ref(x_bits, A, B), "7B %s M=%d" % (shape, M))
    y16 = _run_linear(dev_bits(x_bits), f, M, torch.bfloat16)
    assert torch.equal(y16, y.to(torch.bfloat16))


@pytest.mark.parametrize("M", [257, 300, 1029])
def test_prefill_linear_ragged(M):
    d_in, d_out, r = 512, 1088, 192
    f = dev_factor(6, 2, 0, d_in, d_out, r)
    A, B = host_factor(6, 2, 0, d_in, d_out, r)
    x_bits = synth.bf16_normal(6, synth.make_tag(M, 0, synth.KIND_X), (M, d_in))
    y = _run_linear(dev_bits(x_bits), f, M, torch.float32)
    assert_parity(y.cpu().numpy(), _ref(x_bits, A, B), "prefill M=%d" % M)
    y16 = _run_linear(dev_bits(x_bits), f, M, torch.bfloat16)
    assert torch.equal(y16, y.to(torch.bfloat16))


@pytest.mark.parametrize("rho", [0.2, 0.4, 0.6])
def test_prefill_llama7b_sampled_rows(rho):
    """M = 8 x 2048 rows at the swept ranks; rows sampled across tiles, oracle row by row."""
    M, d_in, d_out = 16384, 4096, 11008
    r = oracle.rank_for(d_in, d_out, rho)
    f = dev_factor(0, 0, 4, d_in, d_out, r)
    x = gpu_normal((M, d_in), 0, synth.make_tag(0, 0, synth.KIND_X))
    y = _run_linear(x, f, M, torch.bfloat16)
    A, B = host_factor(0, 0, 4, d_in, d_out, r)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 129, 255, 8191, 16383],
                                     synth.uniform_ints(1, 9, 56, 0, M - 1)]))
    x_rows = host_bits(x[torch.from_numpy(rows).cuda()])
    y_ref = _ref(x_rows, A, B)
    # bf16 output: compare against the oracle with the bar on the fp32 scale
    y_rows = bf16_f64(y[torch.from_numpy(rows).cuda()])
    assert_parity(y_rows, y_ref, "prefill 7B rho=%s" % rho)


def test_strided_rows_and_determinism():
    M, d_in, d_out, r = 40, 1024, 640, 128
    f = dev_factor(7, 0, 1, d_in, d_out, r)
    A, B = host_factor(7, 0, 1, d_in, d_out, r)
    x_bits = synth.bf16_normal(7, 77, (M, d_in + 64))
    xs = dev_bits(x_bits)[:, :d_in]               # row stride d_in + 64
    y1 = _run_linear(xs, f, M, torch.float32, ld_extra=8)
    y2 = _run_linear(xs, f, M, torch.float32, ld_extra=8)
    assert torch.equal(y1, y2)
    assert_parity(y1.cpu().numpy(), _ref(x_bits[:, :d_in], A, B), "strided")
    # rows are independent: permuting x permutes y bit for bit
    p = torch.from_numpy(synth.permutation(7, 78, M)).cuda()
    y3 = _run_linear(xs[p].contiguous(), f, M, torch.float32)
    assert torch.equal(y3, y1[p])


def test_zero_rows_is_noop():
    f = dev_factor(8, 0, 0, 512, 512, 64)
    x = torch.zeros((0, 512), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((0, 512), dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lr.linear_forward(x, f, y, ws, None)
