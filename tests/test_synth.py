"""The seeded input generator: definition, determinism, bf16 rounding, moments."""

from fractions import Fraction

import numpy as np
import pytest

import synth


def test_fmix_known_values():
    # SplitMix64 with state 0: first outputs of the published generator
    # (state advanced by the golden gamma before mixing).
    s = 0
    outs = []
    for _ in range(3):
        s = (s + synth.GOLDEN) & synth.MASK64
        outs.append(synth.fmix_int(s))
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_vector_matches_scalar():
    key = synth.stream_key(7, synth.make_tag(3, 2, synth.KIND_A))
    v = synth.normal_f64(key, 50, start=1000)
    for i in range(50):
        assert v[i] == synth.normal_int(key, 1000 + i)
    u = synth.uniform_u64(key, 5, start=3)
    for i in range(5):
        assert int(u[i]) == synth.fmix_int((key + (3 + i + 1) * synth.GOLDEN) & synth.MASK64)


def test_irwin_hall_moments():
    key = synth.stream_key(0, synth.make_tag(0, 0, synth.KIND_X))
    z = synth.normal_f64(key, 400_000)
    assert abs(z.mean()) < 0.01
    assert abs(z.var() - 1.0) < 0.01
    assert z.min() >= -6.0 and z.max() <= 6.0
    # fourth moment of the Irwin-Hall-12 sum, standardised: 3 - 1.2/12 = 2.9
    k4 = np.mean(z ** 4)
    assert abs(k4 - 2.9) < 0.05


def _bf16_value(bits: int) -> Fraction:
    s = -1 if bits >> 15 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0:
        return Fraction(0)
    return s * Fraction(128 + m, 128) * Fraction(2) ** (e - 127)


def _rne_bruteforce(x: float) -> int:
    """Nearest bf16 by exact comparison of the two bracketing candidates."""
    if x == 0.0:
        return 0x8000 if np.signbit(x) else 0
    fx = Fraction(x)
    sign = 0x8000 if x < 0 else 0
    a = abs(fx)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    lo_m = int(a * 128)  # floor of the 8-bit significand
    cands = []
    for m in (lo_m, lo_m + 1):
        ee, mm = e, m
        if mm == 256:
            ee, mm = e + 1, 128
        bits = sign | ((ee + 127) << 7) | (mm - 128)
        cands.append(bits)
    d0 = abs(_bf16_value(cands[0]) - fx)
    d1 = abs(_bf16_value(cands[1]) - fx)
    if d0 < d1:
        return cands[0]
    if d1 < d0:
        return cands[1]
    return cands[0] if (cands[0] & 1) == 0 else cands[1]


def test_bf16_rne_bruteforce():
    rng = np.random.default_rng(1)
    xs = list(rng.normal(size=300) * 10.0 ** rng.integers(-6, 6, size=300))
    # exact midpoints and their neighbours: 1 + k/128 + 1/256
    for k in range(0, 8):
        mid = 1.0 + k / 128 + 1 / 256
        xs += [mid, -mid, np.nextafter(mid, 2), np.nextafter(mid, 0)]
    xs += [1.0, -1.0, 0.0, 1.9999999, 255.99]
    xs = np.array(xs, dtype=np.float64)
    got = synth.f64_to_bf16_bits(xs)
    for x, g in zip(xs, got):
        assert int(g) == _rne_bruteforce(float(x)), x


def test_bf16_range_error():
    with pytest.raises(ValueError):
        synth.f64_to_bf16_bits(np.array([1e-45]))
    with pytest.raises(ValueError):
        synth.f64_to_bf16_bits(np.array([1e40]))


def test_permutation_and_ints():
    p = synth.permutation(0, synth.make_tag(0, 0, synth.KIND_PERM), 1000)
    assert sorted(p.tolist()) == list(range(1000))
    assert not np.array_equal(p, np.arange(1000))
    q = synth.permutation(0, synth.make_tag(0, 0, synth.KIND_PERM), 1000)
    assert np.array_equal(p, q)
    L = synth.uniform_ints(0, synth.make_tag(0, 0, synth.KIND_LEN), 5000, 128, 4096)
    assert L.min() >= 128 and L.max() <= 4096
    assert abs(L.mean() - (128 + 4096) / 2) < 40


def test_factor_pair_recipe():
    At, Bt = synth.factor_pair(0, 0, 0, 512, 512, 64)
    assert At.shape == (64, 512) and Bt.shape == (512, 64)
    A = (At.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    B = (Bt.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # A ~ N(0, 1/512): variance
    assert abs(A.var() * 512 - 1.0) < 0.05
    # column j of Bt has std sqrt(1/64) * (j+1)^-0.5
    col_std = B.std(axis=0)
    want = np.sqrt(1 / 64) / np.sqrt(np.arange(1, 65))
    assert np.all(np.abs(col_std / want - 1) < 0.12)


def test_paged_batch():
    L, table, total = synth.paged_batch(0, 64, 128, 4096, 16)
    nb = (L + 15) // 16
    assert total == nb.sum()
    used = np.concatenate([table[s, : nb[s]] for s in range(64)])
    assert sorted(used.tolist()) == list(range(total))
    for s in range(64):
        assert np.all(table[s, nb[s]:] == -1)


def test_c_backend_matches_numpy_definition():
    assert synth._host() is not None, "libsynth_host.so not built"
    for shape, std, cs in [((33, 70), 0.37, None), ((16, 512), 1 / 8, synth.sigma_scale(512)),
                           ((1, 5), 3.0, None)]:
        tag = synth.make_tag(2, 6, synth.KIND_A)
        assert np.array_equal(synth.bf16_normal(9, tag, shape, std, cs),
                              synth.bf16_normal_numpy(9, tag, shape, std, cs))
