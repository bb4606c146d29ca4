"""lr_linear_forward_noalloc: the factorized linear for callers that cannot allocate.

Such callers (allocator-free runtimes, plugins handed only raw pointers and a
stream, serving loops with device memory fixed at start-up) get the same
result as lr_linear_forward, with the intermediate kept in the library's
static device array instead of a caller workspace.  Both entry points run the
same kernels on the same bits, so their outputs must be identical; each is
also checked against the fp64 oracle.  This file is collected last so that a
run stopping at the first failure has run every other test.
"""

import ctypes

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import assert_parity, dev_factor, host_factor

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


def _call_noalloc(x, f, y, st):
    """The raw C symbol: y's dtype picks LR_BF16 or LR_F32, strides are passed through."""
    fc = f.c()
    ydt = lr.LR_BF16 if y.dtype == torch.bfloat16 else lr.LR_F32
    return lr.lib.lr_linear_forward_noalloc(x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0),
                                            ydt, x.shape[0], ctypes.byref(fc), st.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)


def _x(seed, call, M, d_in, ld_extra=0):
    x_bits = synth.bf16_normal(seed, synth.make_tag(call, 0, synth.KIND_X), (M, d_in))
    full = torch.zeros((M, d_in + ld_extra), dtype=torch.bfloat16, device="cuda")
    full[:, :d_in] = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    return x_bits, full[:, :d_in]


@pytest.mark.parametrize("M,shape,ydtype,ld_extra", [
    (4, (512, 512, 64), torch.float32, 0),
    (64, (4096, 4096, 1216), torch.float32, 0),
    (37, (1024, 1088, 192), torch.bfloat16, 0),
    (20, (512, 768, 128), torch.float32, 24),       # padded ldx and ldy
    (300, (1024, 1088, 192), torch.float32, 0),     # prefill kernels
])
def test_noalloc_equals_workspace_entry_point_twice(M, shape, ydtype, ld_extra):
    d_in, d_out, r = shape
    f = dev_factor(12, 0, 3, d_in, d_out, r)
    A, B = host_factor(12, 0, 3, d_in, d_out, r)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.full((lr.linear_workspace_bytes(M, f),), 0xFF, dtype=torch.uint8, device="cuda")
    for call in range(2):          # two calls in a row share the static array
        x_bits, x = _x(12, call, M, d_in, ld_extra)
        ref_full = torch.full((M, d_out + ld_extra), float("nan"), dtype=ydtype, device="cuda")
        ref = ref_full[:, :d_out]
        lr.linear_forward(x, f, ref, ws, st)
        y_full = torch.full((M, d_out + ld_extra), float("nan"), dtype=ydtype, device="cuda")
        y = y_full[:, :d_out]
        assert _call_noalloc(x, f, y, st) == lr.LR_OK, lr.last_error()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(y, ref), "noalloc call %d differs from lr_linear_forward" % call
        if ld_extra:                                  # the padding columns are not written
            assert torch.isnan(y_full[:, d_out:].float()).all()
        want = oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)[1]
        if ydtype == torch.float32:
            assert_parity(y.cpu().numpy(), want, "noalloc call %d vs oracle" % call)
        else:
            # a bf16 y is the round-to-nearest-even image of the fp32 y, whose
            # parity is what the oracle checks (bf16 rounding alone can exceed
            # the bar at this rms)
            y32 = torch.empty((M, d_out), dtype=torch.float32, device="cuda")
            assert _call_noalloc(x, f, y32, st) == lr.LR_OK, lr.last_error()
            torch.cuda.synchronize()
            assert torch.equal(y, y32.to(torch.bfloat16))
            assert_parity(y32.cpu().numpy(), want, "noalloc call %d (fp32) vs oracle" % call)


def test_noalloc_python_wrapper():
    M, (d_in, d_out, r) = 16, (512, 512, 64)
    f = dev_factor(13, 0, 1, d_in, d_out, r)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x_bits, x = _x(13, 0, M, d_in)
    y = torch.empty((M, d_out), dtype=torch.bfloat16, device="cuda")
    ref = torch.empty((M, d_out), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(lr.linear_workspace_bytes(M, f), dtype=torch.uint8, device="cuda")
    lr.linear_forward_noalloc(x, f, y, st)
    lr.linear_forward(x, f, ref, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y, ref)


def test_noalloc_rejects_sizes_beyond_the_static_array():
    f = dev_factor(12, 1, 3, 1024, 1024, 1024)
    M = lr.NOALLOC_SCRATCH_BYTES // (2 * f.r) + 1            # one row too many
    x = torch.zeros((M, 1024), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, 1024), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(x, f, y, st) == lr.LR_ERR_UNSUPPORTED
    assert "static array" in lr.last_error()
