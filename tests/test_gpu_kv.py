"""GPU parity of the low-rank KV reconstruction over a compacted buffer."""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import assert_parity, bf16_f64, dev_bits, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


def _setup(seed, n_seq, r, d_kv, cap_pad):
    L, table, total = synth.paged_batch(seed, n_seq, 20, 300, 16)
    pool_rows = total * 16
    pool_bits = synth.bf16_normal(seed, synth.make_tag(0, 1, synth.KIND_POOL), (pool_rows, r))
    cap = int(L.sum()) + cap_pad
    remap, n, _ = lr.remap_build(L, table, 16, 0, cap)      # every position of every sequence
    At, Bt = synth.factor_pair(seed, 0, synth.PROJ_K, d_kv, d_kv, r)   # Bt: [d_kv][r]
    return pool_bits, remap, n, cap, Bt


@pytest.mark.parametrize("n_seq,r,d_kv,cap_pad", [(12, 576, 1024, 37), (1, 128, 256, 3)])
def test_kv_reconstruct_matches_oracle(n_seq, r, d_kv, cap_pad):
    pool_bits, remap, n, cap, Bt = _setup(31, n_seq, r, d_kv, cap_pad)
    pool = dev_bits(pool_bits)
    buf = torch.full((cap, r), 3.0, dtype=torch.bfloat16, device="cuda")
    out = torch.full((cap, d_kv), 3.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.kv_reconstruct(pool, torch.from_numpy(remap).cuda(),
                      torch.tensor([n], dtype=torch.int32, device="cuda"), buf, dev_bits(Bt), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    B = oracle.widen_bf16(Bt).T
    _, out_ref, bad = oracle.kv_reconstruct(oracle.widen_bf16(pool_bits), remap, n, cap, B)
    assert not bad
    buf_bits, _ = oracle.remap_gather(pool_bits, remap, n, cap)
    assert np.array_equal(host_bits(buf), buf_bits)            # compaction is bit-exact
    assert_parity(bf16_f64(out)[:n], out_ref[:n], "kv rows")
    assert not torch.any(out[n:].float())                      # padding rows reconstruct to zero


def test_kv_reconstruct_graph_replays_new_batches():
    """Captured once, replayed after the remap and n_active change."""
    r, d_kv = 576, 1024
    pool_bits, remap, n, cap, Bt = _setup(32, 8, r, d_kv, 64)
    pool = dev_bits(pool_bits)
    B = oracle.widen_bf16(Bt).T
    d_remap = torch.from_numpy(remap).cuda()
    d_n = torch.tensor([n], dtype=torch.int32, device="cuda")
    buf = torch.zeros((cap, r), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((cap, d_kv), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Btd = dev_bits(Bt)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lr.kv_reconstruct(pool, d_remap, d_n, buf, Btd, out, st, stream=s)   # warm (first use)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            lr.kv_reconstruct(pool, d_remap, d_n, buf, Btd, out, st, stream=s)
    for trial in range(2):
        k = n // (trial + 2)
        rm = np.full(cap, -1, np.int32)
        rm[:k] = synth.permutation(33, trial, pool_bits.shape[0])[:k]
        d_remap.copy_(torch.from_numpy(rm))
        d_n.fill_(k)
        g.replay()
        torch.cuda.synchronize()
        _, out_ref, _ = oracle.kv_reconstruct(oracle.widen_bf16(pool_bits), rm, k, cap, B)
        assert_parity(bf16_f64(out)[:k], out_ref[:k], "kv replay %d" % trial)
        assert not torch.any(out[k:].float())
    # an empty batch: the fixed-size GEMM runs over padding only
    d_remap.fill_(-1)
    d_n.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert not torch.any(out.float()) and not torch.any(buf.float())
    assert int(st.item()) == 0
