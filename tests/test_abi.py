"""The C-ABI library without a GPU: exports, host-side remap scan, argument checks."""

import ctypes
import json
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import synth
import rank_decomposed_gb300 as lr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def header_functions():
    text = open(os.path.join(ROOT, "include", "lr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s+\**([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert "lr_linear_forward" in names and "remap_compact" in names and "lr_graph_replay" in names
    assert len(names) >= 14
    out = subprocess.run(["nm", "-D", "--defined-only", lr.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(l.split()[-1] for l in out.splitlines() if l.strip())
    missing = [n for n in names if n not in exported]
    assert not missing, missing


def test_status_strings():
    assert lr.status_string(lr.LR_OK) == "ok"
    assert "remap" in lr.status_string(lr.LR_ERR_REMAP_RANGE)
    assert lr.status_string(99) == "unknown status"


def test_remap_build_golden_and_oracle():
    with open(os.path.join(GOLDEN, "remap_build_small.json")) as f:
        g = json.load(f)
    table = np.array(g["block_table"], dtype=np.int32)
    for c in g["cases"]:
        remap, na, nr = lr.remap_build(g["lengths"], table, g["block_rows"], c["tail_rows"], c["cap"])
        assert remap.tolist() == c["remap"]
        assert (na, nr) == (c["n_active"], c["n_runs"])


@pytest.mark.parametrize("tail", [1, 3, 0])
def test_remap_build_matches_oracle_on_paged_batch(tail):
    L, table, total = synth.paged_batch(3, 24, 1, 200, 16)
    cap = int(L.sum()) if tail == 0 else 24 * tail
    got = lr.remap_build(L, table, 16, tail, cap)
    want = oracle.remap_build(L, table, 16, tail, cap)
    assert np.array_equal(got[0], want[0])
    assert got[1:] == want[1:]


def test_remap_build_errors():
    L = np.array([5, 3], np.int32)
    T = np.array([[0, 1], [2, -1]], np.int32)
    with pytest.raises(lr.LrError) as e:
        lr.remap_build(L, T, 4, 0, 7)          # 8 rows > cap 7
    assert e.value.status == lr.LR_ERR_INVALID_ARG
    with pytest.raises(lr.LrError):
        lr.remap_build(np.array([9], np.int32), np.array([[0, 1]], np.int32), 4, 0, 16)  # too long
    with pytest.raises(lr.LrError):
        lr.remap_build(np.array([2, 2], np.int32), np.array([[0], [0]], np.int32), 4, 0, 8)  # same rows
    with pytest.raises(lr.LrError):
        lr.remap_build(np.array([6], np.int32), np.array([[0, -1]], np.int32), 4, 0, 8)  # missing block


def _fake_factor(d_in, d_out, r, addr=0x10000):
    return lr.Factor(addr, addr + 0x100000, d_in, d_out, r)


def _linear(x, ldx, y, ldy, M, f, ws=0x300000, ws_bytes=1 << 30, ydt=lr.LR_F32):
    return lr.lib.lr_linear_forward(x, ldx, y, ldy, ydt, M, ctypes.byref(f), ws, ws_bytes, None, None)


def test_linear_argument_checks_launch_nothing():
    good = _fake_factor(512, 512, 64)
    assert _linear(0x1000, 512, 0x2000, 512, 0, good) == lr.LR_OK           # M = 0: no-op
    assert _linear(0x1000, 512, 0x2000, 512, 4, _fake_factor(500, 512, 64)) == lr.LR_ERR_UNSUPPORTED
    assert _linear(0x1000, 512, 0x2000, 512, 4, _fake_factor(512, 512, 100)) == lr.LR_ERR_UNSUPPORTED
    assert _linear(None, 512, 0x2000, 512, 4, good) == lr.LR_ERR_INVALID_ARG
    assert _linear(0x1008, 512, 0x2000, 512, 4, good) == lr.LR_ERR_INVALID_ARG  # x not 16-byte aligned
    assert _linear(0x1000, 500, 0x2000, 512, 4, good) == lr.LR_ERR_INVALID_ARG  # ldx < d_in
    assert _linear(0x1000, 512, 0x2000, 256, 4, good) == lr.LR_ERR_INVALID_ARG  # ldy < d_out
    assert _linear(0x1000, 512, 0x2000, 512, 4, good, ws_bytes=16) == lr.LR_ERR_INVALID_ARG
    assert _linear(0x1000, 512, 0x2000, 512, 4, good, ws=0x300010) == lr.LR_ERR_INVALID_ARG
    assert _linear(0x1000, 512, 0x2000, 512, 4, good, ydt=7) == lr.LR_ERR_INVALID_ARG
    assert _linear(0x1000, 512, 0x2000, 512, 4, lr.Factor(0x10008, 0x20000, 512, 512, 64)) == lr.LR_ERR_INVALID_ARG
    assert "aligned" in lr.last_error()


def test_workspace_sizes():
    f = _fake_factor(4096, 4096, 1216)
    assert lr.lib.lr_linear_workspace_bytes(64, ctypes.byref(f)) == 64 * 1216 * 2
    assert lr.lib.lr_linear_workspace_bytes(3, ctypes.byref(f)) == 7424  # 3*1216*2 -> 256-aligned


def _fake_block(d=512, dff=1024, nh=8, nkv=2, hd=64, ranks=(64, 64, 64, 64, 128, 128, 128)):
    b = lr.BlockDesc()
    b.d_model, b.d_ff, b.n_heads, b.n_kv_heads, b.head_dim, b.eps = d, dff, nh, nkv, hd, 1e-6
    io = [(d, nh * hd), (d, nkv * hd), (d, nkv * hd), (nh * hd, d), (d, dff), (d, dff), (dff, d)]
    for i, ((a, o), r) in enumerate(zip(io, ranks)):
        b.f[i] = _fake_factor(a, o, r, 0x10000 * (i + 1))
    return b


def test_block_scratch_layout_matches_struct():
    b = _fake_block()
    M = 5
    al = lambda x: (x + 255) // 256 * 256
    want = al(M * 512 * 2) + sum(al(M * r * 2) for r in (64, 64, 64, 64, 128, 128, 128))
    want += al(M * 512 * 2) + 2 * al(M * 128 * 2) + al(M * 512 * 2) + 3 * al(M * 1024 * 2)
    assert lr.lib.lr_block_scratch_bytes(M, ctypes.byref(b)) == want


def test_block_argument_checks():
    b = _fake_block()
    h, s = 0x100000, 0x200000
    call = lambda bb, M=4, sb=1 << 30: lr.lib.lr_block_forward(h, M, ctypes.byref(bb), s, sb, None, None)
    assert call(b, M=0) == lr.LR_OK
    bad = _fake_block(nkv=3)
    assert call(bad) == lr.LR_ERR_INVALID_ARG           # 8 heads not divisible by 3 kv heads
    bad = _fake_block()
    bad.f[1] = _fake_factor(512, 192, 64)               # k factor with the wrong output size
    assert call(bad) == lr.LR_ERR_INVALID_ARG
    assert call(_fake_block(hd=32, nh=16, nkv=4)) == lr.LR_ERR_UNSUPPORTED
    assert call(b, sb=100) == lr.LR_ERR_INVALID_ARG


def test_remap_copy_argument_checks():
    f = lr.lib.remap_compact
    assert f(0x1000, 10, 8192, 0x2000, 0x3000, 0x4000, 0, None, None) == lr.LR_OK   # cap 0
    assert f(0x1000, 10, 100, 0x2000, 0x3000, 0x4000, 4, None, None) == lr.LR_ERR_INVALID_ARG
    assert f(0x1008, 10, 8192, 0x2000, 0x3000, 0x4000, 4, None, None) == lr.LR_ERR_INVALID_ARG
    assert f(0x1000, 10, 8192, None, 0x3000, 0x4000, 4, None, None) == lr.LR_ERR_INVALID_ARG
    g = lr.lib.remap_scatter
    assert g(0x4000, 0x2000, 0x3000, 0x1000, 10, 48, 0, None, None) == lr.LR_OK
    assert g(0x4000, 0x2000, 0x3000, 0x1000, 10, 40, 4, None, None) == lr.LR_ERR_INVALID_ARG


def test_graph_handles_checked():
    assert lr.lib.lr_graph_replay(None, None) == lr.LR_ERR_STATE
    assert lr.lib.lr_graph_destroy(None) == lr.LR_ERR_STATE
    g = ctypes.c_void_p()
    assert lr.lib.lr_graph_capture(None, ctypes.byref(g)) == lr.LR_ERR_INVALID_ARG


# ------------------------------------------------- rank-space sharding (host)
@pytest.mark.parametrize("d_out,r", [(8192, 2432), (1024, 576), (28672, 3840), (8192, 3840),
                                     (4096, 1216), (11008, 1792), (512, 64)])
def test_rank_shard_comm_bytes_matches_ring_simulation(d_out, r):
    """The closed forms equal the busiest process of a step-by-step ring simulation."""
    M, e = 64, 2
    for G in range(1, 10):
        if 64 * G > min(r, d_out):
            with pytest.raises(lr.LrError):
                lr.rank_shard_comm_bytes(M, d_out, r, G, e)
            continue
        rs, fs = lr.rank_shard_comm_bytes(M, d_out, r, G, e)
        rchunks = [b - a for a, b in oracle.shard_columns(r, G)]
        ochunks = [b - a for a, b in oracle.shard_columns(d_out, G)]
        assert rs == max(oracle.ring_allgather_received(rchunks, M, e))
        assert fs == max(oracle.ring_allreduce_received(ochunks, M, e))


def test_rank_shard_comm_bytes_errors():
    out = (ctypes.c_int64(), ctypes.c_int64())
    call = lambda *a: lr.lib.lr_rank_shard_comm_bytes(*a, ctypes.byref(out[0]), ctypes.byref(out[1]))
    assert call(4, 512, 128, 2, 2) == lr.LR_OK
    assert call(-1, 512, 128, 2, 2) == lr.LR_ERR_INVALID_ARG
    assert call(4, 500, 128, 2, 2) == lr.LR_ERR_INVALID_ARG
    assert call(4, 512, 128, 3, 2) == lr.LR_ERR_INVALID_ARG   # 3 shards of 2 rank blocks
    assert call(4, 512, 128, 0, 2) == lr.LR_ERR_INVALID_ARG
    assert lr.lib.lr_rank_shard_comm_bytes(4, 512, 128, 2, 2, None, None) == lr.LR_ERR_INVALID_ARG


def test_rank_sharded_argument_checks_launch_nothing():
    f = _fake_factor(512, 1024, 256)
    ws = lr.lib.lr_rank_sharded_workspace_bytes(5, ctypes.byref(f), 3)
    # gathered t [5][256] plus shards of 64, 64 and 128 rank columns, each 256-byte aligned
    assert ws == 2560 + 768 + 768 + 1280
    assert lr.lib.lr_rank_sharded_workspace_bytes(5, ctypes.byref(f), 5) == 0  # 5 > 256/64
    call = lambda M, G, ws_bytes=1 << 30, y=0x2000: lr.lib.lr_linear_forward_rank_sharded(
        0x1000, 512, y, 1024, lr.LR_F32, M, ctypes.byref(f), G, 0x300000, ws_bytes, None, None)
    assert call(0, 2) == lr.LR_OK                        # M = 0: no-op
    assert call(4, 0) == lr.LR_ERR_INVALID_ARG
    assert call(4, 5) == lr.LR_ERR_INVALID_ARG           # more shards than rank blocks
    assert call(4, 2, ws_bytes=100) == lr.LR_ERR_INVALID_ARG
    assert call(4, 2, y=0) == lr.LR_ERR_INVALID_ARG


def test_factor_pack_argument_checks_launch_nothing():
    """lr_factor_pack: every rejected call returns before any launch (no GPU here)."""
    pack = lambda A, B, d_in, d_out, r, At, Bt: lr.lib.lr_factor_pack(A, B, d_in, d_out, r, At, Bt, None)
    base = 0x100000
    A, B = base, base + 0x100000
    At, Bt = base + 0x200000, base + 0x300000
    assert pack(A, B, 0, 64, 64, At, Bt) == lr.LR_ERR_INVALID_ARG
    assert pack(A, B, 100, 64, 64, At, Bt) == lr.LR_ERR_UNSUPPORTED      # not a multiple of 64
    assert pack(0, B, 64, 64, 64, At, Bt) == lr.LR_ERR_INVALID_ARG
    assert pack(A + 2, B, 64, 64, 64, At, Bt) == lr.LR_ERR_INVALID_ARG    # misaligned
    # A [64][64] bf16 = 8 KB: an At starting 4 KB into A overlaps it
    assert pack(A, B, 64, 64, 64, A + 4096, Bt) == lr.LR_ERR_INVALID_ARG
    assert pack(A, B, 64, 64, 64, At, At + 4096) == lr.LR_ERR_INVALID_ARG  # At and Bt overlap
    assert "overlap" in lr.last_error()


@pytest.mark.parametrize("cap", [40, 200])
def test_remap_build_blocks_matches_oracle(cap):
    L, table, _ = synth.paged_batch(3, 12, 20, 300, 16)
    if cap < sum((int(x) + 15) // 16 for x in L):
        with pytest.raises(lr.LrError):
            lr.remap_build_blocks(L, table, 16, cap)
        return
    got = lr.remap_build_blocks(L, table, 16, cap)
    want = oracle.remap_build_blocks(L, table, 16, cap)
    assert got[0].tolist() == want[0].tolist() and got[1:] == want[1:]


def test_kv_reconstruct_paged_argument_checks_launch_nothing():
    call = lambda r=64, d_kv=128, cap=4, pool=2, ptr=0x1000: lr.lib.lr_kv_reconstruct_paged(
        ptr, pool, r, 0x2000, 0x3000, cap, 0x4000, d_kv, 0x5000, None, None)
    assert call(cap=0) == lr.LR_OK
    assert call(r=100) == lr.LR_ERR_UNSUPPORTED
    assert call(r=0) == lr.LR_ERR_INVALID_ARG
    assert call(ptr=0) == lr.LR_ERR_INVALID_ARG
    assert call(ptr=0x1008) == lr.LR_ERR_INVALID_ARG
    assert call(pool=1 << 28) == lr.LR_ERR_INVALID_ARG       # 2^32 rows overflow int32


def test_kv_latent_write_argument_checks_launch_nothing():
    call = lambda M=4, d_in=512, r=64, x=0x1000, ldx=512: lr.lib.lr_kv_latent_write(
        x, ldx, M, 0x2000, d_in, r, 0x3000, 0x4000, 100, None, None)
    assert call(M=0) == lr.LR_OK
    assert call(r=100) == lr.LR_ERR_UNSUPPORTED
    assert call(x=0) == lr.LR_ERR_INVALID_ARG
    assert call(ldx=500) == lr.LR_ERR_INVALID_ARG
    assert call(x=0x1004) == lr.LR_ERR_INVALID_ARG
