"""The prefill-size factorized linear as one launch on SM pairs.

Above 256 rows a linear runs its down projection (T = x A_r) and its up
projection (y = T B_r) in one launch.  The 256-row bands are taken in groups;
the up-projection tiles of a group are placed `lag` groups after that group's
down-projection tiles and wait for them.  These tests force small lags and
several group sizes, including a ragged last group (so that the wait is taken
in every arrangement), and start from a workspace of NaN bits, so a T tile
read before it is written shows up in y.  Every result is checked against the
fp64 oracle.
"""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import assert_parity, dev_bits, dev_factor, host_factor

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


@pytest.fixture
def lag_hook():
    def set_schedule(lag, group=0):
        lr.lib.lr_test_prefill_schedule(lag, group)
    yield set_schedule
    lr.lib.lr_test_prefill_schedule(0, 0)


# (M, (d_in, d_out, r)): bands of 256 rows with a ragged last band; rank and
# output widths whose last 256-wide tile is 64, 128 or 192 columns.
CASES = [(257, (512, 1088, 192)), (1029, (1024, 640, 320)), (4133, (1024, 1216, 448))]


# lag < 0: the two projections as two launches (grouped order only)
@pytest.mark.parametrize("lag,group", [(1, 1), (2, 1), (1, 2), (2, 3), (0, 3), (0, 0), (-1, 1), (-1, 3), (-1, 0)])
@pytest.mark.parametrize("M,shape", CASES)
def test_fused_linear_parity_at_every_lag(lag_hook, lag, group, M, shape):
    d_in, d_out, r = shape
    lag_hook(lag, group)
    f = dev_factor(21, 0, 0, d_in, d_out, r)
    A, B = host_factor(21, 0, 0, d_in, d_out, r)
    ws = torch.full((lr.linear_workspace_bytes(M, f),), 0xFF, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = None
    for call in range(2):  # the second call meets the first call's T and band counters
        x_bits = synth.bf16_normal(21, synth.make_tag(M, call, synth.KIND_X), (M, d_in))
        y = torch.full((M, d_out), float("nan"), dtype=torch.float32, device="cuda")
        lr.linear_forward(dev_bits(x_bits), f, y, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        want = oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)[1]
        assert_parity(y.cpu().numpy(), want, "fused M=%d lag=%d group=%d call %d" % (M, lag, group, call))
        if prev is not None:
            assert not torch.equal(y, prev)
        prev = y


def test_fused_linear_result_does_not_depend_on_schedule(lag_hook):
    """Every lag and grouping, fused or not, computes the same tiles in the same order of k: equal bits."""
    M, (d_in, d_out, r) = CASES[2]
    f = dev_factor(22, 0, 0, d_in, d_out, r)
    x = dev_bits(synth.bf16_normal(22, synth.make_tag(M, 0, synth.KIND_X), (M, d_in)))
    ws = torch.full((lr.linear_workspace_bytes(M, f),), 0xFF, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for lag, group in ((1, 1), (3, 2), (17, 1), (1, 16), (2, 5), (0, 0), (-1, 0), (-1, 1)):
        lag_hook(lag, group)
        y = torch.empty((M, d_out), dtype=torch.bfloat16, device="cuda")
        lr.linear_forward(x, f, y, ws, st)
        torch.cuda.synchronize()
        outs.append(y)
    assert int(st.item()) == 0
    for y in outs[1:]:
        assert torch.equal(y, outs[0])


def test_fused_linear_under_graph_replay(lag_hook):
    """Captured once; each replay clears the band counters and recomputes."""
    lag_hook(1)
    M, (d_in, d_out, r) = CASES[1]
    f = dev_factor(23, 0, 0, d_in, d_out, r)
    A, B = host_factor(23, 0, 0, d_in, d_out, r)
    x = torch.empty((M, d_in), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, d_out), dtype=torch.float32, device="cuda")
    ws = torch.full((lr.linear_workspace_bytes(M, f),), 0xFF, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.linear_forward(x, f, y, ws, st)  # configure outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            lr.linear_forward(x, f, y, ws, st)
    for rep in range(3):
        x_bits = synth.bf16_normal(23, synth.make_tag(M, rep, synth.KIND_X), (M, d_in))
        x.copy_(dev_bits(x_bits))
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        want = oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)[1]
        assert_parity(y.cpu().numpy(), want, "fused replay %d" % rep)


def test_workspace_holds_band_counters():
    f = dev_factor(24, 0, 0, 512, 512, 64)
    al = lambda n: (n + 255) // 256 * 256
    assert lr.linear_workspace_bytes(256, f) == al(256 * 64 * 2)
    assert lr.linear_workspace_bytes(257, f) == al(257 * 64 * 2) + al(4 * 2)
    assert lr.linear_workspace_bytes(16384, f) == al(16384 * 64 * 2) + al(4 * 64)


@pytest.mark.parametrize("lag", [0, -1])
@pytest.mark.parametrize("ydtype", [torch.float32, torch.bfloat16])
def test_prefill_padded_leading_dimensions(lag_hook, lag, ydtype):
    """Row strides wider than the rows: x with 64 extra columns, y with 8 (fused and two launches).

    The padding columns of y are never written and every valid element matches the oracle
    (bf16 y: the rounding of the fp32 y, which is what the oracle checks).
    """
    M, d_in, d_out, r = 777, 1024, 1216, 320
    lag_hook(lag)
    f = dev_factor(25, 0, 0, d_in, d_out, r)
    A, B = host_factor(25, 0, 0, d_in, d_out, r)
    x_bits = synth.bf16_normal(25, synth.make_tag(M, 0, synth.KIND_X), (M, d_in))
    xf = torch.zeros((M, d_in + 64), dtype=torch.bfloat16, device="cuda")
    xf[:, :d_in] = dev_bits(x_bits)
    ws = torch.full((lr.linear_workspace_bytes(M, f),), 0xFF, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = {}
    for dt in (torch.float32, ydtype):
        yf = torch.full((M, d_out + 8), float("nan"), dtype=dt, device="cuda")
        lr.linear_forward(xf[:, :d_in], f, yf[:, :d_out], ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.isnan(yf[:, d_out:].float()).all()
        ys[dt] = yf[:, :d_out]
    want = oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)[1]
    assert_parity(ys[torch.float32].cpu().numpy(), want, "padded ld, lag %d" % lag)
    assert torch.equal(ys[ydtype], ys[torch.float32].to(ydtype))
