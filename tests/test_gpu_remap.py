"""GPU remap_compact / remap_scatter: bit-exact against the oracle's index loops."""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import dev_bits, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


def _dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("cap,n_active,d", [(64, 64, 4096), (64, 37, 4096), (64, 1, 4096),
                                            (5, 0, 512), (3, 3, 8), (130, 129, 1024)])
def test_compact_matches_oracle(cap, n_active, d):
    pool_bits = synth.bf16_normal(1, 5, (500, d))
    remap = np.full(cap, -1, np.int32)
    remap[:n_active] = synth.permutation(1, 6, 500)[:n_active]
    pool = dev_bits(pool_bits)
    buf = torch.full((cap, d), 7.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.remap_compact(pool, _dev_i32(remap), _dev_i32([n_active]), buf, st)
    torch.cuda.synchronize()
    want, bad = oracle.remap_gather(pool_bits, remap, n_active, cap)
    assert not bad and int(st.item()) == 0
    assert np.array_equal(host_bits(buf), want)


def test_scatter_inverts_compact():
    d, cap, n = 2048, 48, 41
    pool_bits = synth.bf16_normal(2, 5, (300, d))
    remap = np.full(cap, -1, np.int32)
    remap[:n] = synth.permutation(2, 6, 300)[:n]
    pool = dev_bits(pool_bits)
    r, na = _dev_i32(remap), _dev_i32([n])
    buf = torch.empty((cap, d), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.remap_compact(pool, r, na, buf, st)
    out = torch.zeros_like(pool)
    lr.remap_scatter(buf, r, na, out, st)
    torch.cuda.synchronize()
    want, _ = oracle.remap_scatter(host_bits(buf), remap, n, np.zeros_like(pool_bits))
    got = host_bits(out)
    assert np.array_equal(got, want)
    assert np.array_equal(got[remap[:n]], pool_bits[remap[:n]])
    assert int(st.item()) == 0


def test_fp32_rows_and_full_permutation():
    d, n = 96, 200
    pool = torch.randn(n, d, device="cuda")
    p = synth.permutation(3, 1, n)
    inv = np.argsort(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    once = torch.empty_like(pool)
    twice = torch.empty_like(pool)
    lr.remap_compact(pool, _dev_i32(p), _dev_i32([n]), once, st)
    lr.remap_compact(once, _dev_i32(inv), _dev_i32([n]), twice, st)
    torch.cuda.synchronize()
    assert torch.equal(once, pool[torch.from_numpy(p).cuda()])
    assert torch.equal(twice, pool)


def test_out_of_range_entries_report_and_zero():
    d, cap = 512, 6
    pool_bits = synth.bf16_normal(4, 5, (10, d))
    remap = np.array([3, 10, -2, 0, 9, -1], np.int32)
    pool = dev_bits(pool_bits)
    buf = torch.full((cap, d), 1.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.remap_compact(pool, _dev_i32(remap), _dev_i32([5]), buf, st)
    torch.cuda.synchronize()
    assert int(st.item()) == lr.LR_ERR_REMAP_RANGE
    want, bad = oracle.remap_gather(pool_bits, remap, 5, cap)
    assert bad and np.array_equal(host_bits(buf), want)
    # scatter skips the bad entries and reports them too
    st.zero_()
    out = torch.zeros_like(pool)
    lr.remap_scatter(buf, _dev_i32(remap), _dev_i32([5]), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == lr.LR_ERR_REMAP_RANGE
    wout, _ = oracle.remap_scatter(host_bits(buf), remap, 5, np.zeros_like(pool_bits))
    assert np.array_equal(host_bits(out), wout)


def test_n_active_above_cap_is_clamped():
    d, cap = 64, 4
    pool = torch.randn(8, d, device="cuda")
    buf = torch.empty(cap, d, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.remap_compact(pool, _dev_i32([1, 2, 3, 4]), _dev_i32([99]), buf, st)
    torch.cuda.synchronize()
    assert torch.equal(buf, pool[1:5])
