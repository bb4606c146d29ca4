"""Failure detection without a GPU fault: bounded device waits report a status.

The fault is injected on the host side of the launch: with the test hook
lr_test_stall_producer set, the TMA producers of the decode kernel and of the
paired-SM prefill kernel issue no copy, so the MMA thread's wait on the first
stage runs out (about two seconds), and so do the epilogue waits of the other
CTA of a pair.  The kernel must then report LR_ERR_TIMEOUT through the status
word, release its resources (TMEM of both CTAs of a pair) and return, and the
GPU must stay usable.
"""

import numpy as np
import pytest

import synth
from lr_testutil import assert_parity, dev_bits, dev_factor, host_factor

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import rank_decomposed_gb300 as lr  # noqa: E402


def _linear(x, f, M):
    y = torch.zeros((M, f.d_out), dtype=torch.float32, device="cuda")
    ws = torch.zeros(lr.linear_workspace_bytes(M, f), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.linear_forward(x, f, y, ws, st)
    torch.cuda.synchronize()
    return y, int(st.item())


# M = 4: decode kernel; M = 300 and 1029: the paired-SM prefill kernel, as one
# fused launch (its band waits never start) and, with the lag hook, as two
@pytest.mark.parametrize("M,shape,two_launches", [(4, (512, 512, 64), False), (4, (4096, 4096, 1216), False),
                                                  (300, (512, 1088, 192), False), (1029, (1024, 640, 320), True)])
def test_bounded_wait_reports_timeout_and_gpu_recovers(M, shape, two_launches):
    d_in, d_out, r = shape
    f = dev_factor(21, 0, 0, d_in, d_out, r)
    x_bits = synth.activations(21, M, d_in)
    x = dev_bits(x_bits)
    if two_launches:
        lr.lib.lr_test_prefill_schedule(-1, 0)
    lr.lib.lr_test_stall_producer(1)
    try:
        _, status = _linear(x, f, M)
    finally:
        lr.lib.lr_test_stall_producer(0)
        lr.lib.lr_test_prefill_schedule(0, 0)
    assert status == lr.LR_ERR_TIMEOUT
    # the context is intact: the same call now succeeds and matches the oracle
    y, status = _linear(x, f, M)
    assert status == 0
    A, B = host_factor(21, 0, 0, d_in, d_out, r)
    assert_parity(y.cpu().numpy(), oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)[1],
                  "after timeout")

