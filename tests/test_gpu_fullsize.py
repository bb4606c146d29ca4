"""Parity at the benchmark's own sizes and launch configuration.

The LLaMA-7B-shaped 32-layer decomposed stack at rho = 0.4, 64 rows compacted
by remap from the paged pool, replayed as one CUDA graph -- the decode step
bench.py times -- against the fp64 oracle on sampled rows.  Rows do not
interact (one-token attention), so the oracle follows each sampled row alone
through all 32 layers, regenerating every layer's factors on the host from the
same seeded recipe.  The LLaMA-70B-GQA shapes at the largest decode batch
(256 rows) and the OPT-30B shapes (ReLU MLP) are checked the same way over a
few layers.
"""

import numpy as np
import pytest

import oracle
import synth
from lr_testutil import assert_parity, host_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import rank_decomposed_gb300 as lr  # noqa: E402


def test_llama7b_32_layer_graph_step_sampled_rows():
    import bench
    m, M = bench.LLAMA7B, 64
    w = bench.Workload(torch, lr, M, m.layers)
    try:
        w.stack.capture()
        w.stack.replay()
        torch.cuda.synchronize()
        assert int(w.stack.status.item()) == 0
        h = w.stack.h.cpu().numpy().astype(np.float64)
        y_bits = host_bits(w.stack.ybuf)
        remap = w.stack.remap.cpu().numpy()
        n = w.n_active
        assert n == M
        # the step's output rows land in the pool at their remap rows, as bf16 of h
        out_rows = host_bits(w.stack.pool_out[w.stack.remap[:n].long()])
        assert np.array_equal(out_rows, y_bits[:n])
        pool_rows = w.stack.pool_in.shape[0]
    finally:
        w.free()
        torch.cuda.empty_cache()

    rows = [0, 17, 63]
    pool = synth.bf16_normal(0, synth.make_tag(0, 0, synth.KIND_POOL), (pool_rows, m.d), 1.0)
    x = oracle.widen_bf16(pool[remap[rows]])
    del pool
    hr = x
    for layer in range(m.layers):
        factors = {}
        for p, (a, b, r) in enumerate(bench.shapes(bench.RHO, m)):
            At, Bt = synth.factor_pair(0, layer, p, a, b, r)
            factors[synth.PROJ_NAMES[p]] = oracle.factor_from_stored(At, Bt)
        hr = oracle.block_forward(hr, factors, m.nh, m.nkv, m.hd)
    assert_parity(h[rows], hr, "7B 32-layer graph step, rows %s" % rows)
    # the layers' own contribution, without the unit-variance input residual
    # that dominates rms(h)
    assert_parity(h[rows] - x, hr - x, "7B 32-layer graph step, h - x0")


def _graph_step_rows(model, M, n_layers, rows):
    """Replay one graph step of the bench workload.

    Returns h at `rows`, the oracle's rows and the step's input rows x0.
    """
    import bench
    w = bench.Workload(torch, lr, M, n_layers, model=model)
    try:
        w.stack.capture()
        w.stack.replay()
        torch.cuda.synchronize()
        assert int(w.stack.status.item()) == 0
        assert w.n_active == M
        h = w.stack.h.cpu().numpy().astype(np.float64)[rows]
        remap = w.stack.remap.cpu().numpy()
        pool_rows = w.stack.pool_in.shape[0]
    finally:
        w.free()
        torch.cuda.empty_cache()
    pool = synth.bf16_normal(0, synth.make_tag(0, 0, synth.KIND_POOL), (pool_rows, model.d), 1.0)
    x0 = oracle.widen_bf16(pool[remap[rows]])
    hr = x0
    del pool
    mlp = "relu" if model.mlp == "relu" else "swiglu"
    for layer in range(n_layers):
        factors = {}
        for p, sh in enumerate(bench.shapes(bench.RHO, model)):
            if sh is None:
                continue
            a, b, r = sh
            At, Bt = synth.factor_pair(0, layer, p, a, b, r)
            factors[synth.PROJ_NAMES[p]] = oracle.factor_from_stored(At, Bt)
        hr = oracle.block_forward(hr, factors, model.nh, model.nkv, model.hd, mlp=mlp)
    return h, hr, x0


def test_llama70b_gqa_256_rows_graph_step():
    """70B-GQA shapes (d 8192, ffn 28672, 8 kv heads) at the largest decode batch, 4 layers."""
    import bench
    h, ref, x0 = _graph_step_rows(bench.LLAMA70B, 256, 4, [0, 129, 255])
    assert_parity(h, ref, "70B GQA graph step M=256")
    assert_parity(h - x0, ref - x0, "70B GQA graph step M=256, h - x0")


def test_opt30b_relu_64_rows_graph_step():
    """OPT-30B shapes (d 7168, ReLU MLP), 4 layers."""
    import bench
    h, ref, x0 = _graph_step_rows(bench.MODELS["opt30b"], 64, 4, [0, 40, 63])
    assert_parity(h, ref, "OPT-30B graph step M=64")
    assert_parity(h - x0, ref - x0, "OPT-30B graph step M=64, h - x0")
