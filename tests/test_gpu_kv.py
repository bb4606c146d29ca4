"""GPU parity of the low-rank KV reconstruction over a compacted buffer."""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import assert_parity, assert_parity_bf16, bf16_f64, dev_bits, dev_factor, host_bits

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


# ------------------------------------------------------- block-granular
def _paged_setup(seed, n_seq, r, d_kv, cap_pad):
    L, table, total = synth.paged_batch(seed, n_seq, 20, 300, 16)
    pool_bits = synth.bf16_normal(seed, synth.make_tag(0, 1, synth.KIND_POOL), (total * 16, r))
    cap = sum((int(x) + 15) // 16 for x in L) + cap_pad
    blocks, n, runs = lr.remap_build_blocks(L, table, 16, cap)
    _, Bt = synth.factor_pair(seed, 0, synth.PROJ_V, d_kv, d_kv, r)
    return L, table, pool_bits, blocks, n, cap, Bt


@pytest.mark.parametrize("n_seq,r,d_kv,cap_pad", [(12, 576, 1024, 5), (3, 128, 320, 1), (40, 192, 256, 0)])
def test_kv_reconstruct_paged_matches_oracle(n_seq, r, d_kv, cap_pad):
    """The GEMM reads each listed block straight from the pool (16-row boxes)."""
    L, table, pool_bits, blocks, n, cap, Bt = _paged_setup(41, n_seq, r, d_kv, cap_pad)
    out = torch.full((cap * 16, d_kv), 3.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.kv_reconstruct_paged(dev_bits(pool_bits), torch.from_numpy(blocks).cuda(),
                            torch.tensor([n], dtype=torch.int32, device="cuda"), dev_bits(Bt), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, bad = oracle.kv_reconstruct_paged(oracle.widen_bf16(pool_bits), blocks, n, oracle.widen_bf16(Bt).T)
    assert not bad
    assert_parity(bf16_f64(out)[:n * 16], ref[:n * 16], "paged kv rows")
    assert not torch.any(out[n * 16:].float())                 # padding blocks reconstruct to zero


def test_kv_reconstruct_paged_equals_row_level_path():
    """On every listed position the one-launch paged path equals compaction + GEMM."""
    r, d_kv = 576, 1024
    L, table, pool_bits, blocks, n, cap, Bt = _paged_setup(42, 9, r, d_kv, 0)
    pool, Btd = dev_bits(pool_bits), dev_bits(Bt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_p = torch.empty((cap * 16, d_kv), dtype=torch.bfloat16, device="cuda")
    lr.kv_reconstruct_paged(pool, torch.from_numpy(blocks).cuda(),
                            torch.tensor([n], dtype=torch.int32, device="cuda"), Btd, out_p, st)
    rows, nr, _ = lr.remap_build(L, table, 16, 0, int(L.sum()))
    buf = torch.empty((nr, r), dtype=torch.bfloat16, device="cuda")
    out_r = torch.empty((nr, d_kv), dtype=torch.bfloat16, device="cuda")
    lr.kv_reconstruct(pool, torch.from_numpy(rows).cuda(), torch.tensor([nr], dtype=torch.int32, device="cuda"),
                      buf, Btd, out_r, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    idx, first = [], 0
    for L_s in L:
        idx += [(first + p // 16) * 16 + p % 16 for p in range(int(L_s))]
        first += (int(L_s) + 15) // 16
    # the same bf16 inputs and the same kernel over the same K order: equal bits
    assert torch.equal(out_p[torch.tensor(idx, device="cuda")], out_r)


def test_kv_reconstruct_paged_bad_block_and_graph_replay():
    r, d_kv = 192, 256
    L, table, pool_bits, blocks, n, cap, Bt = _paged_setup(43, 6, r, d_kv, 8)
    pool, Btd = dev_bits(pool_bits), dev_bits(Bt)
    d_blocks = torch.from_numpy(blocks).cuda()
    d_n = torch.tensor([n], dtype=torch.int32, device="cuda")
    out = torch.zeros((cap * 16, d_kv), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lr.kv_reconstruct_paged(pool, d_blocks, d_n, Btd, out, st, stream=s)   # first use outside capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            lr.kv_reconstruct_paged(pool, d_blocks, d_n, Btd, out, st, stream=s)
    pool_blocks = pool_bits.shape[0] // 16
    B = oracle.widen_bf16(Bt).T
    for trial in range(2):
        k = max(1, n - 3 * trial)
        bl = np.full(cap, -1, np.int32)
        bl[:k] = synth.permutation(44, trial, pool_blocks)[:k]
        d_blocks.copy_(torch.from_numpy(bl))
        d_n.fill_(k)
        g.replay()
        torch.cuda.synchronize()
        ref, _ = oracle.kv_reconstruct_paged(oracle.widen_bf16(pool_bits), bl, k, B)
        assert_parity(bf16_f64(out)[:k * 16], ref[:k * 16], "paged replay %d" % trial)
        assert not torch.any(out[k * 16:].float())
    assert int(st.item()) == 0
    # a listed block outside the pool: zero rows and the range status
    bl[1] = pool_blocks + 5
    d_blocks.copy_(torch.from_numpy(bl))
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == lr.LR_ERR_REMAP_RANGE
    assert not torch.any(out[16:32].float())


# -------------------------------------------------- latent KV producer
@pytest.mark.parametrize("M,d_in,r", [(64, 1024, 192), (5, 512, 576), (300, 1024, 128)])
def test_kv_latent_write_rows_and_values(M, d_in, r):
    """The down projection lands in the listed pool rows, bit for bit the t of
    lr_linear_forward, and no other pool row changes."""
    pool_rows = 4 * M + 40
    f = dev_factor(45, 0, synth.PROJ_K, d_in, 256, r)
    x_bits = synth.bf16_normal(45, synth.make_tag(M, 0, synth.KIND_X), (M, d_in))
    x = dev_bits(x_bits)
    rows = synth.permutation(45, M, pool_rows)[:M].astype(np.int32)
    pool0 = synth.bf16_normal(45, synth.make_tag(0, 2, synth.KIND_POOL), (pool_rows, r))
    pool = dev_bits(pool0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.kv_latent_write(x, f.At, torch.from_numpy(rows).cuda(), pool, st)
    # t of the plain linear: the first M * r bf16 of its workspace
    ws = torch.zeros(lr.linear_workspace_bytes(M, f), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, 256), dtype=torch.float32, device="cuda")
    lr.linear_forward(x, f, y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    t = ws[: M * r * 2].view(torch.bfloat16).view(M, r)
    got = pool[torch.from_numpy(rows).long().cuda()]
    assert torch.equal(got, t)
    keep = np.setdiff1d(np.arange(pool_rows), rows)
    assert np.array_equal(host_bits(pool)[keep], pool0[keep])
    A, _ = oracle.factor_from_stored(host_bits(f.At), host_bits(f.Bt))
    ref, bad = oracle.kv_latent_write(oracle.widen_bf16(x_bits), A, rows, oracle.widen_bf16(pool0))
    assert not bad
    assert_parity_bf16(bf16_f64(got), ref[rows], "latent rows")


def test_kv_latent_write_bad_row_and_round_trip():
    """A row outside the pool is skipped and reported; latents written by
    kv_latent_write and rebuilt by kv_reconstruct_paged match the oracle of x A B."""
    d_in, r, d_kv = 512, 128, 256
    f = dev_factor(46, 0, synth.PROJ_V, d_in, d_kv, r)
    n_blocks, pool_blocks = 3, 8
    M = 16 * n_blocks
    blocks = np.array([5, 0, 6], np.int32)
    rows = np.concatenate([16 * b + np.arange(16) for b in blocks]).astype(np.int32)
    x_bits = synth.bf16_normal(46, synth.make_tag(0, 0, synth.KIND_X), (M, d_in))
    pool = torch.zeros((pool_blocks * 16, r), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.kv_latent_write(dev_bits(x_bits), f.At, torch.from_numpy(rows).cuda(), pool, st)
    out = torch.empty((n_blocks * 16, d_kv), dtype=torch.bfloat16, device="cuda")
    lr.kv_reconstruct_paged(pool, torch.from_numpy(blocks).cuda(),
                            torch.tensor([n_blocks], dtype=torch.int32, device="cuda"), f.Bt, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    A, B = oracle.factor_from_stored(host_bits(f.At), host_bits(f.Bt))
    _, dense = oracle.lowrank_linear(oracle.widen_bf16(x_bits), A, B)
    assert_parity_bf16(bf16_f64(out), dense, "latent write + paged reconstruct")
    bad_rows = rows.copy()
    bad_rows[3] = pool_blocks * 16 + 1
    before = pool.clone()
    lr.kv_latent_write(dev_bits(x_bits), f.At, torch.from_numpy(bad_rows).cuda(), pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == lr.LR_ERR_REMAP_RANGE
    assert torch.equal(pool, before)       # the same values again, and nothing at the bad row
