"""lr_linear_forward_noalloc: the factorized linear for callers that cannot allocate.

Such callers (allocator-free runtimes, plugins handed only raw pointers and a
stream, serving loops with device memory fixed at start-up) get the same
result as lr_linear_forward, with the intermediate kept in the library's
static device array instead of a caller workspace.  This file is collected
last so that a run stopping at the first failure has run every other test.
"""

import ctypes

import numpy as np
import pytest

import synth
from lr_testutil import assert_parity, dev_factor

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


def _call_noalloc(x, f, y, st):
    fc = f.c()
    return lr.lib.lr_linear_forward_noalloc(x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0),
                                            lr.LR_F32, x.shape[0], ctypes.byref(fc), st.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("M,shape", [(4, (512, 512, 64)), (64, (4096, 4096, 1216)),
                                     (300, (1024, 1088, 192))])
def test_noalloc_matches_workspace_entry_point_twice(M, shape):
    d_in, d_out, r = shape
    f = dev_factor(12, 0, 3, d_in, d_out, r)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = torch.empty((M, d_out), dtype=torch.float32, device="cuda")
    ws = torch.zeros(lr.linear_workspace_bytes(M, f), dtype=torch.uint8, device="cuda")
    for call in range(2):          # two calls in a row share the static array
        x_bits = synth.bf16_normal(12, synth.make_tag(call, 0, synth.KIND_X), (M, d_in))
        x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        lr.linear_forward(x, f, ref, ws, st)
        y = torch.full((M, d_out), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(x, f, y, st) == lr.LR_OK, lr.last_error()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_parity(y.cpu().numpy(), ref.cpu().numpy(), "noalloc call %d" % call)


def test_noalloc_rejects_sizes_beyond_the_static_array():
    f = dev_factor(12, 1, 3, 1024, 1024, 1024)
    M = lr.NOALLOC_SCRATCH_BYTES // (2 * f.r) + 1            # one row too many
    x = torch.zeros((M, 1024), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, 1024), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(x, f, y, st) == lr.LR_ERR_UNSUPPORTED
    assert "static array" in lr.last_error()
