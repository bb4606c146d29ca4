"""GPU parity of the rank-space sharded linear (simulated processes) against the fp64 oracle."""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import assert_parity, dev_bits, dev_factor, host_factor

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


def _run_sharded(x, f, G, M, ydtype=torch.float32):
    y = torch.full((M, f.d_out), float("nan"), dtype=ydtype, device="cuda")
    ws = torch.zeros(max(lr.rank_sharded_workspace_bytes(M, f, G), 256), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.linear_forward_rank_sharded(x, f, G, y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y


def _run_plain(x, f, M, ydtype=torch.float32):
    y = torch.full((M, f.d_out), float("nan"), dtype=ydtype, device="cuda")
    ws = torch.zeros(max(lr.linear_workspace_bytes(M, f), 256), dtype=torch.uint8, device="cuda")
    lr.linear_forward(x, f, y, ws, None)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("M", [1, 37, 64, 300])
@pytest.mark.parametrize("G", [1, 2, 3, 5])
def test_sharded_matches_oracle(M, G):
    """Uneven shards (r = 5 blocks, d_out = 17 blocks of 64) at decode and prefill sizes."""
    d_in, d_out, r = 512, 1088, 320
    f = dev_factor(9, 0, 2, d_in, d_out, r)
    A, B = host_factor(9, 0, 2, d_in, d_out, r)
    x_bits = synth.bf16_normal(9, synth.make_tag(M, G, synth.KIND_X), (M, d_in))
    y = _run_sharded(dev_bits(x_bits), f, G, M)
    _, _, y_ref = oracle.rank_sharded_linear(oracle.widen_bf16(x_bits), A, B, G)
    assert_parity(y.cpu().numpy(), y_ref, "rank-sharded M=%d G=%d" % (M, G))


@pytest.mark.parametrize("M", [1, 64])
def test_sharded_llama70b_q_eight_processes(M):
    """70B q projection (8192 -> 8192, r = 2432 = 38 blocks) over 8 processes: shards of 4 and 5 blocks."""
    d_in, d_out, r = 8192, 8192, 2432
    f = dev_factor(0, 0, 0, d_in, d_out, r)
    A, B = host_factor(0, 0, 0, d_in, d_out, r)
    x_bits = synth.activations(0, M, d_in)
    y = _run_sharded(dev_bits(x_bits), f, 8, M)
    _, _, y_ref = oracle.rank_sharded_linear(oracle.widen_bf16(x_bits), A, B, 8)
    assert_parity(y.cpu().numpy(), y_ref, "70B q G=8 M=%d" % M)


@pytest.mark.parametrize("M", [4, 300])
def test_one_shard_is_the_plain_linear(M):
    """G = 1 runs the same two GEMMs as lr_linear_forward with a copy between: bit-identical."""
    f = dev_factor(10, 0, 1, 1024, 640, 192)
    x = dev_bits(synth.bf16_normal(10, synth.make_tag(M, 0, synth.KIND_X), (M, 1024)))
    assert torch.equal(_run_sharded(x, f, 1, M), _run_plain(x, f, M))
    assert torch.equal(_run_sharded(x, f, 1, M, torch.bfloat16), _run_plain(x, f, M, torch.bfloat16))


def test_sharded_deterministic_and_bf16_is_rounded_f32():
    M, G = 33, 4
    f = dev_factor(11, 0, 3, 512, 1024, 256)
    x = dev_bits(synth.bf16_normal(11, 5, (M, 512)))
    y1 = _run_sharded(x, f, G, M)
    y2 = _run_sharded(x, f, G, M)
    assert torch.equal(y1, y2)
    assert torch.equal(_run_sharded(x, f, G, M, torch.bfloat16), y1.to(torch.bfloat16))


def test_sharded_rejects_too_many_shards():
    f = dev_factor(12, 0, 0, 512, 512, 128)
    x = torch.zeros((4, 512), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4, 512), dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(lr.LrError):
        lr.linear_forward_rank_sharded(x, f, 3, y, ws, None)
