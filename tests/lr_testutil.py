"""Shared test helpers: device inputs from the seeded generator and the parity bar."""

import numpy as np

import synth

# Parity bar for floating-point outputs: per element
#   |y - y_ref| <= REL * rms(y_ref) + ABS
REL_TOL = 1e-2
ABS_TOL = 1e-3


def tol_of(y_ref):
    y_ref = np.asarray(y_ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    return REL_TOL * rms + ABS_TOL


def assert_parity(y, y_ref, what=""):
    """Check the bar element by element; returns max|err| / tol."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    tol = tol_of(y_ref)
    err = np.abs(y - y_ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, "%s: max err %.3g > tol %.3g (at %s)" % (
        what, worst, tol, np.unravel_index(int(err.argmax()), err.shape))
    return worst / tol


def assert_parity_bf16(y, y_ref, what=""):
    """The parity bar for an output stored as bf16: the bar of the fp32 result
    plus the rounding of the stored value (half an ulp is at most 2^-8 |y_ref|
    relative).  Returns max|err| / bound."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    bound = tol_of(y_ref) + 2.0 ** -8 * np.abs(y_ref)
    ratio = np.abs(y - y_ref) / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    assert worst <= 1.0, "%s: max err / bound %.3g (at %s)" % (
        what, worst, np.unravel_index(int(ratio.argmax()), ratio.shape))
    return worst


def dev_bits(bits):
    """numpy uint16 bf16 bits -> torch bfloat16 CUDA tensor (same bits)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    """torch bfloat16 tensor -> numpy uint16 bits."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(t):
    return (host_bits(t).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gpu_normal(shape, seed, tag, std=1.0, col_scale=None):
    """Device bf16 tensor filled by the GPU generator (bit-identical to synth.bf16_normal)."""
    import torch
    rows, cols = shape
    t = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    cs = None
    if col_scale is not None:
        cs = torch.from_numpy(np.asarray(col_scale, dtype=np.float64)).cuda()
    synth.fill_bf16_normal_device(t.data_ptr(), rows, cols, seed, tag, std,
                                  None if cs is None else cs.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return t


def dev_factor(seed, layer, proj, d_in, d_out, r):
    """FactorPair on the device drawn by the GPU generator with the config recipe."""
    import rank_decomposed_gb300 as lr
    sa, sg = synth.factor_stds(d_in, r)
    At = gpu_normal((r, d_in), seed, synth.make_tag(layer, proj, synth.KIND_A), sa)
    Bt = gpu_normal((d_out, r), seed, synth.make_tag(layer, proj, synth.KIND_B), sg,
                    col_scale=synth.sigma_scale(r))
    return lr.FactorPair(At, Bt)


def host_factor(seed, layer, proj, d_in, d_out, r):
    """Oracle-side fp64 (A_r, B_r) regenerated on the CPU from the same recipe."""
    import oracle
    At, Bt = synth.factor_pair(seed, layer, proj, d_in, d_out, r)
    return oracle.factor_from_stored(At, Bt)


def block_shapes(d, d_ff, n_heads, n_kv, hd, ranks):
    dq, dkv = n_heads * hd, n_kv * hd
    io = [(d, dq), (d, dkv), (d, dkv), (dq, d), (d, d_ff), (d, d_ff), (d_ff, d)]
    return [(a, b, r) for (a, b), r in zip(io, ranks)]
