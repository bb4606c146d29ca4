"""Seeded synthetic inputs shared by the oracle and the GPU path.

This module holds only input generation: counter-based random bits, an
approximately normal variate, integer draws for lengths and permutations, and
the fp64 -> bf16 encoding of the drawn values.  It computes none of the
factorized-linear arithmetic.  Both sides of every parity test take their
inputs from here: the oracle through the numpy functions below, the GPU path
either by copying these arrays to the device or through ``synth_gen.cu``, a
CUDA kernel that implements the same definition bit for bit (a GPU test checks
that equality).

Definition (all integer arithmetic is modulo 2**64):

* ``fmix(z)``: the SplitMix64 output function (Steele, Lea & Flood, OOPSLA
  2014): ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
  z *= 0x94D049BB133111EB; z ^= z >> 31``.
* stream key of ``(seed, tag)``: ``fmix(fmix(seed ^ 0x5EED) + tag * G)`` with
  ``G = 0x9E3779B97F4A7C15``.  ``tag = layer * 2**16 + proj * 2**8 + kind``.
* word ``q`` (0..5) of element ``i``: ``w = fmix(key + (6 i + q + 1) G)``; its
  two 32-bit halves are uniform integers.
* normal variate of element ``i``: the Irwin-Hall sum of its 12 uniform
  halves, ``z = (S - 6 * 2**32) / 2**32`` (exact in fp64).  Mean 0, variance 1,
  support [-6, 6]: a stated approximation of N(0, 1).
* value: ``v = z * std`` in fp64, then ``v * col_scale[j]`` for column ``j``
  when a column scale is given (two correctly rounded fp64 products), then
  round-to-nearest-even to bf16 on the fp64 bit pattern.
* integer draw ``i`` of a stream: ``fmix(key + (i + 1) G)``.
"""

from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# kinds of stream
KIND_X = 0          # activations / hidden rows
KIND_A = 1          # down factor
KIND_B = 2          # up factor (the G of B_r = diag(sigma) G)
KIND_LEN = 3        # sequence lengths
KIND_PERM = 4       # permutations (slot order, physical blocks)
KIND_POOL = 5       # paged pool rows

# projection ids inside a block, in the block's order
PROJ_Q, PROJ_K, PROJ_V, PROJ_O, PROJ_GATE, PROJ_UP, PROJ_DOWN = range(7)
PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


# ---------------------------------------------------------------- scalar form
def fmix_int(z: int) -> int:
    """SplitMix64 output function on a Python int (reference form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def make_tag(layer: int = 0, proj: int = 0, kind: int = 0) -> int:
    if not (0 <= proj < 256 and 0 <= kind < 256 and 0 <= layer < (1 << 40)):
        raise ValueError("tag field out of range")
    return (layer << 16) | (proj << 8) | kind


def stream_key(seed: int, tag: int) -> int:
    return fmix_int((fmix_int((seed ^ 0x5EED) & MASK64) + tag * GOLDEN) & MASK64)


def normal_int(key: int, i: int) -> float:
    """Irwin-Hall-12 variate of element ``i`` computed with Python ints."""
    s = 0
    for q in range(6):
        w = fmix_int((key + (6 * i + q + 1) * GOLDEN) & MASK64)
        s += (w & 0xFFFFFFFF) + (w >> 32)
    return float(s - 6 * (1 << 32)) / 4294967296.0


# ------------------------------------------------------------- vector form
def _fmix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(_M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def normal_f64(key: int, n: int, start: int = 0) -> np.ndarray:
    """Variates of elements ``start .. start+n-1`` of stream ``key`` (fp64)."""
    idx = np.arange(start, start + n, dtype=np.uint64)
    base = np.uint64(key) + idx * np.uint64(6 * GOLDEN & MASK64)
    s = np.zeros(n, dtype=np.int64)
    for q in range(6):
        w = _fmix(base + np.uint64((q + 1) * GOLDEN & MASK64))
        s += (w & np.uint64(0xFFFFFFFF)).astype(np.int64)
        s += (w >> np.uint64(32)).astype(np.int64)
    return (s - np.int64(6 << 32)).astype(np.float64) * (1.0 / 4294967296.0)


def uniform_u64(key: int, n: int, start: int = 0) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    return _fmix(np.uint64(key) + idx * np.uint64(GOLDEN))


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even); returns uint16.

    Only zero and normal bf16 results are produced; a value whose bf16 image
    would be subnormal, infinite or NaN raises ValueError (the generator never
    makes one).
    """
    v = np.ascontiguousarray(v, dtype=np.float64)
    b = v.view(np.uint64)
    sign = (b >> np.uint64(63)).astype(np.uint64)
    mag = b & np.uint64(0x7FFFFFFFFFFFFFFF)
    lsb = (mag >> np.uint64(45)) & np.uint64(1)
    r = (mag + np.uint64((1 << 44) - 1) + lsb) >> np.uint64(45)
    exp11 = (r >> np.uint64(7)).astype(np.int64)
    mant = (r & np.uint64(0x7F)).astype(np.uint64)
    exp8 = exp11 - 1023 + 127
    zero = mag == 0
    bad = (~zero) & ((exp8 <= 0) | (exp8 >= 255))
    if np.any(bad):
        raise ValueError("value outside the normal bf16 range")
    exp8 = np.where(zero, 0, exp8).astype(np.uint64)
    mant = np.where(zero, np.uint64(0), mant)
    out = (sign << np.uint64(15)) | (exp8 << np.uint64(7)) | mant
    return out.astype(np.uint16)


_host_lib = None


def _host():
    """The C implementation (synth_host.c), or None when it has not been built."""
    global _host_lib
    if _host_lib is None:
        import ctypes
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth_host.so")
        if not os.path.exists(path):
            return None
        lib = ctypes.CDLL(path)
        lib.synth_bf16_normal_host.restype = ctypes.c_int
        lib.synth_bf16_normal_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p]
        _host_lib = lib
    return _host_lib


def bf16_normal_numpy(seed: int, tag: int, shape, std: float = 1.0,
                      col_scale: np.ndarray | None = None) -> np.ndarray:
    """The definition in numpy (slow; the reference for the C and CUDA versions)."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    v = normal_f64(stream_key(seed, tag), n) * np.float64(std)
    if col_scale is not None:
        cs = np.asarray(col_scale, dtype=np.float64)
        if cs.shape != (shape[-1],):
            raise ValueError("col_scale must have one entry per column")
        v = (v.reshape(-1, shape[-1]) * cs[None, :]).reshape(-1)
    return f64_to_bf16_bits(v).reshape(shape)


def bf16_normal(seed: int, tag: int, shape, std: float = 1.0,
                col_scale: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16, row-major ``shape``) of ``z * std [* col_scale]``."""
    lib = _host()
    shape = tuple(int(s) for s in shape)
    if lib is None or len(shape) == 0:
        return bf16_normal_numpy(seed, tag, shape, std, col_scale)
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    cols = shape[-1]
    out = np.empty(shape, dtype=np.uint16)
    cs = None
    if col_scale is not None:
        cs = np.ascontiguousarray(col_scale, dtype=np.float64)
        if cs.shape != (cols,):
            raise ValueError("col_scale must have one entry per column")
    bad = lib.synth_bf16_normal_host(out.ctypes.data, rows, cols, stream_key(seed, tag),
                                     float(std), None if cs is None else cs.ctypes.data)
    if bad:
        raise ValueError("value outside the normal bf16 range")
    return out


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    """Fisher-Yates permutation of range(n) driven by integer draws."""
    u = uniform_u64(stream_key(seed, tag), max(n, 1))
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(u[i]) % (i + 1)
        p[i], p[j] = p[j], p[i]
    return p


def uniform_ints(seed: int, tag: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers in [lo, hi] (inclusive): ``lo + draw % (hi - lo + 1)``."""
    u = uniform_u64(stream_key(seed, tag), n)
    return (np.int64(lo) + (u % np.uint64(hi - lo + 1)).astype(np.int64))


# ------------------------------------------------ recipes for the workloads
def factor_stds(d_in: int, r: int):
    """Standard deviations of the factor draws.

    A_r ~ N(0, 1/d_in) and G ~ N(0, 1/r), reading the second argument of
    N(0, s) as the variance, so that t = x A_r has unit variance for unit x.
    """
    return float(np.sqrt(1.0 / d_in)), float(np.sqrt(1.0 / r))


def sigma_scale(r: int) -> np.ndarray:
    """sigma_i = (i + 1) ** -0.5 for i = 0 .. r-1 (fp64)."""
    return 1.0 / np.sqrt(np.arange(1, r + 1, dtype=np.float64))


def factor_pair(seed: int, layer: int, proj: int, d_in: int, d_out: int, r: int):
    """bf16 bits of one factor pair in the stored (out-major) layout.

    Returns ``(At, Bt)``: ``At[r][d_in]`` is A_r transposed and ``Bt[d_out][r]``
    is B_r transposed, both row-major.  ``B_r = diag(sigma) G``, so column
    ``j`` of ``Bt`` carries ``sigma_j``.
    """
    sa, sg = factor_stds(d_in, r)
    At = bf16_normal(seed, make_tag(layer, proj, KIND_A), (r, d_in), sa)
    Bt = bf16_normal(seed, make_tag(layer, proj, KIND_B), (d_out, r), sg,
                     col_scale=sigma_scale(r))
    return At, Bt


def activations(seed: int, M: int, d: int, layer: int = 0) -> np.ndarray:
    """x ~ N(0, 1) bf16 bits ``[M][d]``."""
    return bf16_normal(seed, make_tag(layer, 0, KIND_X), (M, d), 1.0)


def paged_batch(seed: int, n_seq: int, len_lo: int, len_hi: int, block_rows: int = 16):
    """Lengths, a paged block table and the pool size of a decode batch.

    Sequence lengths are uniform in [len_lo, len_hi].  Every sequence owns
    ceil(L / block_rows) blocks; physical block ids are a seeded permutation
    of all blocks, so some blocks happen to be adjacent and most are not.
    Returns ``(lengths[n_seq], block_table[n_seq][max_blocks], n_blocks)``;
    unused table entries are -1.
    """
    lengths = uniform_ints(seed, make_tag(0, 0, KIND_LEN), n_seq, len_lo, len_hi)
    nb = (lengths + block_rows - 1) // block_rows
    total = int(nb.sum())
    phys = permutation(seed, make_tag(0, 1, KIND_PERM), total)
    maxb = int(nb.max()) if n_seq else 0
    table = np.full((n_seq, maxb), -1, dtype=np.int32)
    c = 0
    for s in range(n_seq):
        table[s, : nb[s]] = phys[c : c + nb[s]]
        c += int(nb[s])
    return lengths.astype(np.int32), table, total


def gpu_gen_lib_path() -> str:
    import os
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")


_gpu_lib = None


def _gpu():
    global _gpu_lib
    if _gpu_lib is None:
        import ctypes
        lib = ctypes.CDLL(gpu_gen_lib_path())
        lib.synth_bf16_normal.restype = ctypes.c_int
        lib.synth_bf16_normal.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p,
                                          ctypes.c_void_p]
        _gpu_lib = lib
    return _gpu_lib


def fill_bf16_normal_device(ptr: int, rows: int, cols: int, seed: int, tag: int,
                            std: float = 1.0, col_scale_ptr: int | None = None,
                            stream: int | None = None) -> None:
    """Device version of ``bf16_normal``: writes ``rows x cols`` bf16 values at ``ptr``.

    ``col_scale_ptr`` is a device array of ``cols`` fp64 scales (or None).
    """
    rc = _gpu().synth_bf16_normal(ptr, rows, cols, stream_key(seed, tag), float(std),
                                  col_scale_ptr, stream)
    if rc != 0:
        raise RuntimeError("synth_bf16_normal failed with CUDA error %d" % rc)
