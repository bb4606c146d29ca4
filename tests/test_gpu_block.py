"""GPU parity of the decomposed block and the graph-replayed layer stack."""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import (assert_parity, block_shapes, dev_bits, dev_factor, host_bits, host_factor)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402

SMALL = dict(d=512, d_ff=1024, n_heads=8, n_kv=2, hd=64, ranks=(128, 64, 64, 128, 192, 192, 192))
LLAMA7B = dict(d=4096, d_ff=11008, n_heads=32, n_kv=32, hd=128,
               ranks=(1216, 1216, 1216, 1216, 1792, 1792, 1792))


def make_layer(seed, layer, cfg):
    shapes = block_shapes(cfg["d"], cfg["d_ff"], cfg["n_heads"], cfg["n_kv"], cfg["hd"], cfg["ranks"])
    relu = cfg.get("mlp") == "relu"
    skip = lambda p: relu and p == synth.PROJ_GATE
    dev = [None if skip(p) else dev_factor(seed, layer, p, a, b, r)
           for p, (a, b, r) in enumerate(shapes)]
    host = {synth.PROJ_NAMES[p]: (None if skip(p) else host_factor(seed, layer, p, a, b, r))
            for p, (a, b, r) in enumerate(shapes)}
    blk = lr.Block(cfg["d"], cfg["d_ff"], cfg["n_heads"], cfg["n_kv"], cfg["hd"], dev,
                   mlp=lr.MLP_RELU if relu else lr.MLP_SWIGLU)
    return blk, host


def _h_input(seed, M, d):
    bits = synth.bf16_normal(seed, synth.make_tag(0, 0, synth.KIND_X), (M, d))
    return bits, oracle.widen_bf16(bits)


@pytest.mark.parametrize("M", [1, 4, 37, 300])
def test_block_small_gqa(M):
    cfg = SMALL
    blk, host = make_layer(3, 0, cfg)
    bits, h0 = _h_input(3, M, cfg["d"])
    h = torch.from_numpy(h0.astype(np.float32)).cuda()
    scratch = torch.zeros(lr.block_scratch_bytes(M, blk), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.block_forward(h, blk, scratch, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.block_forward(h0, host, cfg["n_heads"], cfg["n_kv"], cfg["hd"])
    out = h.cpu().numpy().astype(np.float64)
    assert_parity(out - h0, ref - h0, "block delta M=%d" % M)
    assert_parity(out, ref, "block M=%d" % M)


def test_block_llama7b_decode64():
    cfg = LLAMA7B
    M = 64
    blk, host = make_layer(0, 0, cfg)
    bits, h0 = _h_input(0, M, cfg["d"])
    h = torch.from_numpy(h0.astype(np.float32)).cuda()
    scratch = torch.zeros(lr.block_scratch_bytes(M, blk), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.block_forward(h, blk, scratch, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.block_forward(h0, host, cfg["n_heads"], cfg["n_kv"], cfg["hd"])
    out = h.cpu().numpy().astype(np.float64)
    assert_parity(out - h0, ref - h0, "7B block delta")


LLAMA70B = dict(d=8192, d_ff=28672, n_heads=64, n_kv=8, hd=128,
                ranks=(2432, 576, 576, 2432, 3840, 3840, 3840))


@pytest.mark.parametrize("M", [16, 64])
def test_block_llama70b_gqa_decode(M):
    """One 70B-shaped block (GQA, 8 kv heads) in decode against the oracle."""
    cfg = LLAMA70B
    blk, host = make_layer(0, 3, cfg)
    bits, h0 = _h_input(1, M, cfg["d"])
    h = torch.from_numpy(h0.astype(np.float32)).cuda()
    scratch = torch.zeros(lr.block_scratch_bytes(M, blk), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.block_forward(h, blk, scratch, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.block_forward(h0, host, cfg["n_heads"], cfg["n_kv"], cfg["hd"])
    out = h.cpu().numpy().astype(np.float64)
    assert_parity(out - h0, ref - h0, "70B block delta M=%d" % M)


@pytest.mark.parametrize("cfg_name,M,seed", [("7b", 1029, 5), ("70b", 8192, 6)])
def test_block_prefill_full_shapes_sampled_rows(cfg_name, M, seed):
    """Full-size blocks at prefill sizes, checked on sampled rows (rows are independent).

    7B shapes at 1029 rows: every linear runs as one fused launch.  70B-GQA
    shapes at 8192 rows: the q/k/v/o linears are fused, the MLP linears (over
    1.5e12 flops each) run as two launches; both feed the fp32 residual
    through the add epilogue, and o reads the GQA-broadcast v.
    """
    cfg = LLAMA7B if cfg_name == "7b" else LLAMA70B
    blk, host = make_layer(seed, 0, cfg)
    bits, h0 = _h_input(seed, M, cfg["d"])
    h = torch.from_numpy(h0.astype(np.float32)).cuda()
    scratch = torch.zeros(lr.block_scratch_bytes(M, blk), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.block_forward(h, blk, scratch, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, 511, M - 1],
                                     synth.uniform_ints(seed, 9, 12, 0, M - 1)]))
    ref = oracle.block_forward(h0[rows], host, cfg["n_heads"], cfg["n_kv"], cfg["hd"])
    out = h[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    assert_parity(out - h0[rows], ref - h0[rows], "%s block at %d rows, sampled" % (cfg_name, M))


def _make_stack(cfg, n_layers, cap, n_seq, seed=4, mode=0):
    layers, hosts = zip(*[make_layer(seed, l, cfg) for l in range(n_layers)])
    L, table, total = synth.paged_batch(seed, n_seq, 20, 300, 16)
    pool_rows = total * 16
    pool_bits = synth.bf16_normal(seed, synth.make_tag(0, 0, synth.KIND_POOL), (pool_rows, cfg["d"]))
    remap, n_active, _ = lr.remap_build(L, table, 16, 1, cap)
    d = cfg["d"]
    pool = dev_bits(pool_bits)
    dev = dict(
        pool_in=pool, pool_out=pool.clone(),
        remap=torch.from_numpy(remap).cuda(),
        n_active=torch.tensor([n_active], dtype=torch.int32, device="cuda"),
        xbuf=torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda"),
        h=torch.zeros(cap, d, dtype=torch.float32, device="cuda"),
        ybuf=torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda"),
        status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    dev["scratch"] = torch.zeros(lr.Stack.scratch_bytes(cap, layers, mode), dtype=torch.uint8,
                                 device="cuda")
    stack = lr.Stack(list(layers), mode=mode, **dev)
    return stack, list(hosts), pool_bits, remap, n_active


def _oracle_stack(cfg, hosts, pool_bits, remap, n):
    x = oracle.widen_bf16(pool_bits[remap[:n]])
    return oracle.stack_forward(x, hosts, cfg["n_heads"], cfg["n_kv"], cfg["hd"])


def test_stack_eager_graph_and_remap():
    cfg, cap = SMALL, 16
    stack, hosts, pool_bits, remap, n = _make_stack(cfg, 3, cap, 12)
    assert n == 12
    stack.forward()
    torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    h_eager = stack.h.clone()
    out_eager = stack.pool_out.clone()
    ref = _oracle_stack(cfg, hosts, pool_bits, remap, n)
    assert_parity(h_eager[:n].cpu().numpy(), ref, "stack eager")
    assert not torch.any(h_eager[n:])                               # padding rows stay zero
    assert torch.equal(stack.ybuf, h_eager.to(torch.bfloat16))      # narrow is RNE
    got = host_bits(out_eager)
    want = pool_bits.copy()
    want[remap[:n]] = host_bits(stack.ybuf)[:n]
    assert np.array_equal(got, want)                                 # only remapped rows change

    # the captured graph replays the same step bit for bit
    stack.capture()
    stack.pool_out.copy_(stack.pool_in)
    stack.h.fill_(123.0)
    stack.replay()
    torch.cuda.synchronize()
    assert torch.equal(stack.h, h_eager)
    assert torch.equal(stack.pool_out, out_eager)

    # a new batch: only the remap contents and n_active change, the graph stays valid
    for n2 in (5, 1, cap):
        perm = synth.permutation(9, n2, pool_bits.shape[0])[:cap].astype(np.int32)
        stack.remap.copy_(torch.from_numpy(perm))
        stack.n_active.fill_(n2)
        stack.pool_out.copy_(stack.pool_in)
        stack.replay()
        torch.cuda.synchronize()
        assert int(stack.status.item()) == 0
        ref = _oracle_stack(cfg, hosts, pool_bits, perm, n2)
        assert_parity(stack.h[:n2].cpu().numpy(), ref, "stack replay n=%d" % n2)
        assert not torch.any(stack.h[n2:])

    # an empty batch: every row of the fixed buffer is padding and nothing is scattered
    stack.n_active.fill_(0)
    stack.pool_out.copy_(stack.pool_in)
    stack.h.fill_(5.0)
    stack.replay()
    torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    assert not torch.any(stack.h)
    assert torch.equal(stack.pool_out, stack.pool_in)
    stack.destroy()


def test_stack_launch_count():
    # gather + widen, 2 RMSNorm + 8 GEMM + SiLU-GLU launches per block, narrow + scatter
    stack, *_ = _make_stack(SMALL, 2, 8, 6, mode=lr.STACK_LAYERED)
    assert stack.launch_count() == 2 + 2 * 11


@pytest.mark.parametrize("cap,n_seq", [(1, 1), (16, 16), (100, 90), (256, 256)])
def test_stack_caps(cap, n_seq):
    """Every token tile width of the decode kernel (16, 32->64, 128, 256) in a graph step."""
    cfg = SMALL
    stack, hosts, pool_bits, remap, n = _make_stack(cfg, 2, cap, n_seq, seed=5)
    stack.capture()
    stack.replay()
    torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    ref = _oracle_stack(cfg, hosts, pool_bits, remap, n)
    assert_parity(stack.h[:n].cpu().numpy(), ref, "stack cap=%d" % cap)
    stack.destroy()


def test_stack_llama7b_two_layers():
    """Two 7B-shaped layers, 64 rows, replayed twice: the layers' contribution against the oracle."""
    cfg, cap = LLAMA7B, 64
    stack, hosts, pool_bits, remap, n = _make_stack(cfg, 2, cap, 64, seed=6)
    stack.capture()
    for _ in range(2):
        stack.replay()
    torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    ref = _oracle_stack(cfg, hosts, pool_bits, remap, n)
    x0 = oracle.widen_bf16(pool_bits[remap[:n]])
    out = stack.h[:n].cpu().numpy().astype(np.float64)
    assert_parity(out - x0, ref - x0, "7B stack delta")
    stack.destroy()


OPT_SMALL = dict(d=512, d_ff=2048, n_heads=8, n_kv=8, hd=64, ranks=(128, 128, 128, 128, 64, 192, 192),
                 mlp="relu")
MQA_SMALL = dict(d=512, d_ff=1024, n_heads=8, n_kv=1, hd=64, ranks=(128, 64, 64, 128, 192, 192, 192))


@pytest.mark.parametrize("cfg_name,M", [("opt", 4), ("opt", 300), ("mqa", 5), ("mqa", 260)])
def test_block_variants(cfg_name, M):
    """Non-GLU (ReLU) MLP with MHA, and MQA (one kv head), in decode and prefill sizes."""
    cfg = OPT_SMALL if cfg_name == "opt" else MQA_SMALL
    blk, host = make_layer(13, 0, cfg)
    bits, h0 = _h_input(13, M, cfg["d"])
    h = torch.from_numpy(h0.astype(np.float32)).cuda()
    scratch = torch.zeros(lr.block_scratch_bytes(M, blk), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lr.block_forward(h, blk, scratch, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.block_forward(h0, host, cfg["n_heads"], cfg["n_kv"], cfg["hd"],
                               mlp=cfg.get("mlp", "swiglu"))
    out = h.cpu().numpy().astype(np.float64)
    assert_parity(out - h0, ref - h0, "%s block delta M=%d" % (cfg_name, M))


def test_stack_with_per_layer_ranks():
    """Layers of one stack compressed at different ratios (variadic ranks) under graph replay."""
    cfg0 = dict(SMALL)
    cfg1 = dict(SMALL, ranks=(64, 64, 64, 64, 64, 64, 64))
    cfg2 = dict(SMALL, ranks=(256, 128, 128, 256, 320, 320, 320))
    layers, hosts = zip(*[make_layer(14, l, c) for l, c in enumerate((cfg0, cfg1, cfg2))])
    cap, d = 16, SMALL["d"]
    L, table, total = synth.paged_batch(14, 10, 20, 300, 16)
    pool_bits = synth.bf16_normal(14, synth.make_tag(0, 0, synth.KIND_POOL), (total * 16, d))
    remap, n, _ = lr.remap_build(L, table, 16, 1, cap)
    pool = dev_bits(pool_bits)
    stack = lr.Stack(list(layers), pool, pool.clone(), torch.from_numpy(remap).cuda(),
                     torch.tensor([n], dtype=torch.int32, device="cuda"),
                     torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(cap, d, dtype=torch.float32, device="cuda"),
                     torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(lr.Stack.scratch_bytes(cap, layers), dtype=torch.uint8, device="cuda"),
                     torch.zeros(1, dtype=torch.int32, device="cuda"))
    stack.capture()
    stack.replay()
    torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    ref = _oracle_stack(SMALL, list(hosts), pool_bits, remap, n)
    assert_parity(stack.h[:n].cpu().numpy(), ref, "variadic-rank stack")
    stack.destroy()


@pytest.mark.parametrize("cfg_name,cap", [("opt", 16), ("opt", 64), ("mqa", 37), ("mqa", 128)])
def test_stack_variants(cfg_name, cap):
    """Graph steps of a non-GLU (ReLU) MLP stack and an MQA stack."""
    cfg = OPT_SMALL if cfg_name == "opt" else MQA_SMALL
    stack, hosts, pool_bits, remap, n = _make_stack(cfg, 3, cap, cap, seed=16)
    stack.capture()
    stack.replay()
    torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    x = oracle.widen_bf16(pool_bits[remap[:n]])
    ref = oracle.stack_forward(x, hosts, cfg["n_heads"], cfg["n_kv"], cfg["hd"], mlp=cfg.get("mlp", "swiglu"))
    out = stack.h[:n].cpu().numpy().astype(np.float64)
    assert_parity(out - x, ref - x, "stack %s cap=%d" % (cfg_name, cap))
    stack.destroy()


def test_per_layer_ranks_and_replay_determinism():
    """Layers at different ranks in one graph step (48 rows); two replays agree bit for bit."""
    cfgs = (SMALL, dict(SMALL, ranks=(64, 64, 64, 64, 64, 64, 64)),
            dict(SMALL, ranks=(256, 128, 128, 256, 320, 320, 320)))
    layers, hosts = zip(*[make_layer(17, l, c) for l, c in enumerate(cfgs)])
    cap, d = 48, SMALL["d"]
    L, table, total = synth.paged_batch(17, 40, 20, 300, 16)
    pool_bits = synth.bf16_normal(17, synth.make_tag(0, 0, synth.KIND_POOL), (total * 16, d))
    remap, n, _ = lr.remap_build(L, table, 16, 1, cap)
    pool = dev_bits(pool_bits)
    stack = lr.Stack(list(layers), pool, pool.clone(), torch.from_numpy(remap).cuda(),
                     torch.tensor([n], dtype=torch.int32, device="cuda"),
                     torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(cap, d, dtype=torch.float32, device="cuda"),
                     torch.zeros(cap, d, dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(lr.Stack.scratch_bytes(cap, layers), dtype=torch.uint8, device="cuda"),
                     torch.zeros(1, dtype=torch.int32, device="cuda"))
    stack.capture()
    stack.replay()
    torch.cuda.synchronize()
    h1 = stack.h.clone()
    stack.h.fill_(7.0)
    stack.replay()
    torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    assert torch.equal(stack.h, h1)
    ref = _oracle_stack(SMALL, list(hosts), pool_bits, remap, n)
    assert_parity(stack.h[:n].cpu().numpy(), ref, "variadic-rank stack, 48 rows")
    stack.destroy()


@pytest.mark.parametrize("cfg_name,cap", [("glu", 16), ("relu", 16), ("glu", 300), ("relu", 300)])
def test_launch_count_matches_the_kernels_launched(cfg_name, cap):
    """lr_stack_launch_count (the bench's gpu_launches) against the kernels the profiler sees."""
    profiler = torch.profiler
    cfg = SMALL if cfg_name == "glu" else OPT_SMALL
    stack, *_ = _make_stack(cfg, 2, cap, min(cap, 12), seed=15, mode=lr.STACK_LAYERED)
    stack.forward()                    # first use: configuration outside the profiled step
    torch.cuda.synchronize()
    for _ in range(2):                 # the first session of a process may record nothing
        with profiler.profile(activities=[profiler.ProfilerActivity.CUDA]) as prof:
            stack.forward()
            torch.cuda.synchronize()
    assert int(stack.status.item()) == 0
    kernels = [e for e in prof.events()
               if e.device_type == torch.autograd.DeviceType.CUDA
               and "memcpy" not in e.name.lower() and "memset" not in e.name.lower()]
    if not kernels:
        pytest.skip("the profiler recorded no device activity here")
    assert len(kernels) == stack.launch_count(), sorted({e.name[:40] for e in kernels})
