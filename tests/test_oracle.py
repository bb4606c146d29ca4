"""Pins for the fp64 oracle: each check rests on something other than the oracle itself."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_matrix(seed, tag, shape, std=1.0):
    return oracle.widen_bf16(synth.bf16_normal(seed, tag, shape, std))


# ----------------------------------------------------------- formats
def _bf16_by_definition(bits: int) -> Fraction:
    """Value of a bf16 pattern from its fields: sign, 8-bit biased exponent, 7-bit fraction.

    Written from the format's definition (the top half of an IEEE binary32), with
    subnormals (exponent field 0) kept exact rather than flushed.
    """
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0:
        return sign * Fraction(m, 128) * Fraction(1, 2 ** 126)
    return sign * Fraction(128 + m, 128) * Fraction(2) ** (e - 127)


def test_widen_bf16_every_pattern():
    """widen_bf16 against the exact decoding of all 65,536 bf16 patterns.

    A wrong shift, a lost sign or a flushed subnormal fails here.  Patterns with
    the exponent field all ones are Inf (fraction 0) or NaN and must map to them.
    """
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):       # signalling-NaN patterns warn in the fp32 -> fp64 cast
        got = oracle.widen_bf16(bits)
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    special = e == 0xFF
    assert np.all(np.isinf(got[special & (m == 0)]))
    assert np.all(np.isnan(got[special & (m != 0)]))
    finite = np.nonzero(~special)[0]
    want = np.array([float(_bf16_by_definition(int(b))) for b in finite])
    assert np.array_equal(got[finite], want)
    # the sign of zero survives
    assert np.signbit(got[0x8000]) and not np.signbit(got[0x0000])
    assert got.dtype == np.float64


def test_factor_from_stored_hand_example():
    """Stored At [r][d_in] and Bt [d_out][r] come back as A_r [d_in][r] and B_r [r][d_out].

    r = 2, d_in = 3, d_out = 4 (no square shape, so a missing transpose fails),
    with bf16 patterns written out by hand: 1 0x3F80, 2 0x4000, 3 0x4040,
    4 0x4080, 5 0x40A0, 6 0x40C0, -1 0xBF80, 0.5 0x3F00, -2 0xC000, 0.25 0x3E80.
    """
    At = np.array([[0x3F80, 0x4000, 0x4040],            # A_r column 0 = (1, 2, 3)
                   [0x4080, 0x40A0, 0x40C0]], np.uint16)  # A_r column 1 = (4, 5, 6)
    Bt = np.array([[0x3F80, 0xBF80],                     # B_r column 0 = (1, -1)
                   [0x3F00, 0x4000],                     # B_r column 1 = (0.5, 2)
                   [0x4040, 0x0000],                     # B_r column 2 = (3, 0)
                   [0xC000, 0x3E80]], np.uint16)         # B_r column 3 = (-2, 0.25)
    A, B = oracle.factor_from_stored(At, Bt)
    assert A.shape == (3, 2) and B.shape == (2, 4)
    assert np.array_equal(A, [[1.0, 4.0], [2.0, 5.0], [3.0, 6.0]])
    assert np.array_equal(B, [[1.0, 0.5, 3.0, -2.0], [-1.0, 2.0, 0.0, 0.25]])
    # x = e_0 picks row 0 of A_r B_r: (1, 4) B_r = (1 - 4, 0.5 + 8, 3, -2 + 1)
    _, y = oracle.lowrank_linear(np.array([[1.0, 0.0, 0.0]]), A, B)
    assert np.array_equal(y[0], [-3.0, 8.5, 3.0, -1.0])


# ----------------------------------------------------------- the linear
def test_linear_exact_rational_bruteforce():
    """y = (x A) B against exact rational arithmetic on tiny bf16 inputs."""
    x = _bf16_matrix(1, 10, (3, 8))
    A = _bf16_matrix(1, 11, (8, 4), 0.3)
    B = _bf16_matrix(1, 12, (4, 6), 0.5)
    _, y = oracle.lowrank_linear(x, A, B)
    for m in range(3):
        for o in range(6):
            exact = Fraction(0)
            for j in range(4):
                tj = sum(Fraction(float(x[m, k])) * Fraction(float(A[k, j])) for k in range(8))
                exact += tj * Fraction(float(B[j, o]))
            assert abs(Fraction(float(y[m, o])) - exact) <= abs(exact) * Fraction(1, 10**13) + Fraction(1, 10**300)


def test_linear_associativity():
    """(x A) B == x (A B): the factor pair acts as the rank-r weight W = A B."""
    x = _bf16_matrix(2, 1, (5, 96))
    A = _bf16_matrix(2, 2, (96, 16), 0.1)
    B = _bf16_matrix(2, 3, (16, 40), 0.25)
    _, y = oracle.lowrank_linear(x, A, B)
    W = np.einsum("kj,jo->ko", A, B)
    y2 = np.einsum("mk,ko->mo", x, W)
    assert np.max(np.abs(y - y2)) <= 1e-12 * np.max(np.abs(y2))


def test_linear_special_cases():
    x = _bf16_matrix(3, 1, (4, 32))
    A = _bf16_matrix(3, 2, (32, 8), 0.2)
    B = _bf16_matrix(3, 3, (8, 24), 0.2)
    # A = I (r = d_in) reduces to one product x B'
    Bsq = _bf16_matrix(3, 4, (32, 24))
    _, y = oracle.lowrank_linear(x, np.eye(32), Bsq)
    assert np.array_equal(y, x @ Bsq)
    # B = I (r = d_out) reduces to x A
    _, y = oracle.lowrank_linear(x, A, np.eye(8))
    assert np.allclose(y, x @ A, rtol=0, atol=1e-13)
    # one-hot rows pick rows of W = A B
    W = A @ B
    for k in (0, 7, 31):
        e = np.zeros((1, 32))
        e[0, k] = 1.0
        _, y = oracle.lowrank_linear(e, A, B)
        assert np.allclose(y[0], W[k], rtol=0, atol=1e-15)
    # zero input gives exact zeros
    t, y = oracle.lowrank_linear(np.zeros((2, 32)), A, B)
    assert not np.any(t) and not np.any(y)
    # rows are independent: permuting rows permutes outputs
    p = np.array([2, 0, 3, 1])
    _, y = oracle.lowrank_linear(x, A, B)
    _, yp = oracle.lowrank_linear(x[p], A, B)
    assert np.array_equal(yp, y[p])


def test_svd_factors_reproduce_rank_r_weight():
    """A dense W of rank r, split by SVD into (U S, V^T), gives the same layer output."""
    rng = np.random.default_rng(5)
    d_in, d_out, r = 48, 40, 6
    W = rng.normal(size=(d_in, r)) @ rng.normal(size=(r, d_out))
    U, s, Vt = np.linalg.svd(W)
    assert np.all(s[r:] <= 1e-10 * s[0])
    A = U[:, :r] * s[:r]
    B = Vt[:r]
    x = rng.normal(size=(7, d_in))
    _, y = oracle.lowrank_linear(x, A, B)
    ref = x @ W
    assert np.max(np.abs(y - ref)) <= 1e-10 * np.max(np.abs(ref))
    # Eckart-Young: truncating to k < r leaves exactly the tail energy
    k = 3
    Wk = (U[:, :k] * s[:k]) @ Vt[:k]
    assert abs(np.linalg.norm(W - Wk) ** 2 - np.sum(s[k:] ** 2)) <= 1e-8 * np.sum(s ** 2)


# ------------------------------------------------------------- the rank rule
def test_rank_table():
    with open(os.path.join(GOLDEN, "rank_table.json")) as f:
        rows = json.load(f)["rows"]
    for d_in, d_out, rho, r in rows:
        assert oracle.rank_for(d_in, d_out, rho) == r, (d_in, d_out, rho)


# --------------------------------------------------------------- the glue
def test_rmsnorm_closed_forms():
    # [3, 4] with eps = 0: mean square 12.5, so [3, 4] / sqrt(12.5)
    y = oracle.rmsnorm(np.array([[3.0, 4.0]]), eps=0.0)
    assert np.allclose(y, [[0.848528137423857, 1.131370849898476]], rtol=1e-15)
    # a constant row c: c / sqrt(c^2 + eps)
    c = 0.01
    y = oracle.rmsnorm(np.full((1, 64), c), eps=1e-6)
    assert np.allclose(y, 0.01 / np.sqrt(1e-4 + 1e-6), rtol=1e-15)
    # positive scale invariance when eps = 0; mean square of the output is 1
    h = _bf16_matrix(4, 1, (3, 256))
    assert np.allclose(oracle.rmsnorm(7.5 * h, eps=0.0), oracle.rmsnorm(h, eps=0.0), rtol=1e-14)
    assert np.allclose(np.mean(oracle.rmsnorm(h, eps=0.0) ** 2, axis=1), 1.0, rtol=1e-14)


def test_silu_identities():
    z = np.linspace(-20, 20, 401)
    s = oracle.silu(z)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    # z*sig(z) - (-z)*sig(-z) = z since sig(z) + sig(-z) = 1
    assert np.allclose(s - oracle.silu(-z), z, rtol=0, atol=1e-13)
    # silu(ln 3) = ln3 * 3/4 (sigmoid(ln 3) = 3/4)
    assert np.isclose(oracle.silu(np.array([np.log(3.0)]))[0], 0.75 * np.log(3.0), rtol=1e-15)
    assert np.all(np.abs(s[z > 15] - z[z > 15]) < 1e-5)
    assert np.all(np.abs(s[z < -15]) < 1e-5)


def _softmax_attention_one_key(q, k, v, n_heads, n_kv, hd):
    """Textbook scaled-dot-product attention over a context of one token."""
    M = q.shape[0]
    g = n_heads // n_kv
    out = np.zeros((M, n_heads * hd))
    for m in range(M):
        for h in range(n_heads):
            kvh = h // g
            qh = q[m, h * hd:(h + 1) * hd]
            kh = k[m, kvh * hd:(kvh + 1) * hd]
            scores = np.array([qh @ kh / np.sqrt(hd)])
            w = np.exp(scores - scores.max())
            w /= w.sum()
            out[m, h * hd:(h + 1) * hd] = w[0] * v[m, kvh * hd:(kvh + 1) * hd]
    return out


@pytest.mark.parametrize("n_heads,n_kv", [(4, 4), (8, 2), (4, 1)])
def test_one_token_attention_is_softmax_attention(n_heads, n_kv):
    hd = 8
    q = _bf16_matrix(6, 1, (3, n_heads * hd))
    k = _bf16_matrix(6, 2, (3, n_kv * hd))
    v = _bf16_matrix(6, 3, (3, n_kv * hd))
    got = oracle.one_token_attention(v, n_heads, n_kv, hd)
    ref = _softmax_attention_one_key(q, k, v, n_heads, n_kv, hd)
    assert np.array_equal(got, ref)


def _zero_factors(d, d_kv, dff, r=8):
    z = lambda a, b: (np.zeros((a, r)), np.zeros((r, b)))
    return {"q": z(d, d), "k": z(d, d_kv), "v": z(d, d_kv), "o": z(d, d),
            "gate": z(d, dff), "up": z(d, dff), "down": z(dff, d)}


def test_block_zero_factors_is_identity():
    h = _bf16_matrix(7, 1, (3, 32))
    f = _zero_factors(32, 16, 48)
    assert np.array_equal(oracle.block_forward(h, f, 4, 2, 8), h)
    assert np.array_equal(oracle.stack_forward(h, [f, f, f], 4, 2, 8), h)


def test_block_attention_path_bruteforce():
    """v = n1[:, :d_kv] and o = I: h1 = h + GQA-broadcast of n1 columns, by index loops."""
    d, n_heads, n_kv, hd = 32, 4, 2, 8
    d_kv = n_kv * hd
    h = _bf16_matrix(8, 1, (2, d))
    f = _zero_factors(d, d_kv, 48)
    f["v"] = (np.eye(d)[:, :d_kv], np.eye(d_kv))
    f["o"] = (np.eye(d), np.eye(d))
    out = oracle.block_forward(h, f, n_heads, n_kv, hd, eps=1e-6, return_all=True)
    n1 = h / np.sqrt(np.mean(h ** 2, axis=1, keepdims=True) + 1e-6)
    want = h.copy()
    for m in range(2):
        for c in range(d):
            head, e = divmod(c, hd)
            kvh = head // (n_heads // n_kv)
            want[m, c] += n1[m, kvh * hd + e]
    assert np.allclose(out["h1"], want, rtol=0, atol=1e-14)
    # MLP factors are zero, so the block output is h1
    assert np.array_equal(out["h2"], out["h1"])


def test_block_mlp_path():
    """gate = up = n2 and down = I: h2 = h1 + silu(n2) * n2."""
    d = 16
    h = _bf16_matrix(9, 1, (2, d))
    f = _zero_factors(d, d, d)
    f["gate"] = (np.eye(d), np.eye(d))
    f["up"] = (np.eye(d), np.eye(d))
    f["down"] = (np.eye(d), np.eye(d))
    out = oracle.block_forward(h, f, 2, 2, 8, return_all=True)
    n2 = out["n2"]
    want = h + (n2 / (1 + np.exp(-n2))) * n2
    assert np.allclose(out["h2"], want, rtol=0, atol=1e-14)


def test_stack_is_composition():
    d, dff = 32, 48
    h = _bf16_matrix(10, 1, (3, d))
    layers = []
    for l in range(2):
        f = {}
        for p, (a, b) in zip(synth.PROJ_NAMES,
                             [(d, d), (d, 16), (d, 16), (d, d), (d, dff), (d, dff), (dff, d)]):
            f[p] = (_bf16_matrix(11, 100 * l + 2 * len(f), (a, 8), a ** -0.5),
                    _bf16_matrix(11, 100 * l + 2 * len(f) + 1, (8, b), 8 ** -0.5))
        layers.append(f)
    s = oracle.stack_forward(h, layers, 4, 2, 8)
    b = oracle.block_forward(oracle.block_forward(h, layers[0], 4, 2, 8), layers[1], 4, 2, 8)
    assert np.array_equal(s, b)


# -------------------------------------------------------------- the remap
def test_remap_build_golden():
    with open(os.path.join(GOLDEN, "remap_build_small.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        remap, n_active, n_runs = oracle.remap_build(g["lengths"], g["block_table"],
                                                     g["block_rows"], c["tail_rows"], c["cap"])
        assert remap.tolist() == c["remap"]
        assert n_active == c["n_active"]
        assert n_runs == c["n_runs"]
    with pytest.raises(ValueError):
        oracle.remap_build(g["lengths"], g["block_table"], g["block_rows"], 0, 17)


def test_remap_permutation_inverse():
    pool = synth.bf16_normal(0, 77, (40, 24))
    p = synth.permutation(0, 78, 40)[:16]           # 16 distinct pool rows
    buf, bad = oracle.remap_gather(pool, p, 16, 20)
    assert not bad
    assert np.array_equal(buf[:16], pool[p])
    assert not np.any(buf[16:])
    # scatter of the gathered rows restores the pool exactly
    back, bad = oracle.remap_scatter(buf, p, 16, np.zeros_like(pool))
    assert not bad
    assert np.array_equal(back[p], pool[p])
    mask = np.ones(40, bool)
    mask[p] = False
    assert not np.any(back[mask])
    # gather with the inverse permutation undoes a full permutation
    q = synth.permutation(0, 79, 40)
    inv = np.argsort(q)
    once, _ = oracle.remap_gather(pool, q, 40, 40)
    twice, _ = oracle.remap_gather(once, inv, 40, 40)
    assert np.array_equal(twice, pool)


def test_remap_out_of_range_and_padding():
    pool = synth.bf16_normal(0, 80, (8, 4))
    buf, bad = oracle.remap_gather(pool, [3, 99, -1, 0], 3, 5)
    assert bad
    assert np.array_equal(buf[0], pool[3])
    assert not np.any(buf[1]) and not np.any(buf[2])   # bad entries give zero rows
    assert not np.any(buf[3:])                         # rows >= n_active are zero


def test_remap_scatter_out_of_range_and_padding():
    """Out-of-range entries are skipped and flagged; rows at or past n_active are not written."""
    buf = synth.bf16_normal(0, 81, (5, 4))
    pool = np.zeros((8, 4), dtype=np.uint16)
    out, bad = oracle.remap_scatter(buf, [2, 99, -1, 5, 6], 4, pool)
    assert bad
    assert np.array_equal(out[2], buf[0]) and np.array_equal(out[5], buf[3])
    others = [i for i in range(8) if i not in (2, 5)]
    assert not np.any(out[others])          # 99 and -1 wrote nothing; row 6 is past n_active
    assert not np.any(pool)                 # the input pool is left alone
    out, bad = oracle.remap_scatter(buf, [2, 99, -1, 5, 6], 1, pool)
    assert not bad                          # the bad entries lie past n_active
    assert np.array_equal(out[2], buf[0]) and np.count_nonzero(np.any(out, axis=1)) <= 1


# ----------------------------------------------------- KV reconstruction
def test_kv_reconstruct_identity_and_commutation():
    """B = I returns the compacted latents; compacting commutes with the row-wise product."""
    pool_bits = synth.bf16_normal(5, 90, (50, 64))
    pool = oracle.widen_bf16(pool_bits)
    remap = np.full(12, -1, np.int32)
    remap[:9] = synth.permutation(5, 91, 50)[:9]
    buf, out, bad = oracle.kv_reconstruct(pool, remap, 9, 12, np.eye(64))
    assert not bad and np.array_equal(out, buf)
    assert np.array_equal(buf[:9], pool[remap[:9]]) and not np.any(buf[9:])
    B = _bf16_matrix(5, 92, (64, 128), 0.125)
    _, out, _ = oracle.kv_reconstruct(pool, remap, 9, 12, B)
    full = np.einsum("pj,jn->pn", pool, B)          # reconstruct every pool row, then gather
    assert np.allclose(out[:9], full[remap[:9]], rtol=0, atol=1e-12)
    assert not np.any(out[9:])


def test_remap_build_blocks_hand_example_and_rows():
    """Block list of a hand-worked paged batch, and its agreement with the row-level scan.

    Lengths 20, 3, 0, 33 with 16-row blocks need 2, 1, 0 and 3 blocks; their
    table rows list the physical blocks in order.  Every listed row of
    remap_build (all positions) is row p % 16 of the block that holds p.
    """
    lengths = [20, 3, 0, 33]
    table = [[7, 2, -1], [5, -1, -1], [-1, -1, -1], [0, 1, 9]]
    blocks, n, runs = oracle.remap_build_blocks(lengths, table, 16, 8)
    assert blocks.tolist() == [7, 2, 5, 0, 1, 9, -1, -1]
    assert n == 6
    assert runs == 5           # 7 | 2 | 5 | 0,1 | 9
    rows, nr, _ = oracle.remap_build(lengths, table, 16, 0, 64)
    assert nr == sum(lengths)
    i = 0
    for s2, L in enumerate(lengths):
        for p2 in range(L):
            blk = int(table[s2][p2 // 16])
            assert rows[i] == blk * 16 + p2 % 16
            i += 1
    with pytest.raises(ValueError):
        oracle.remap_build_blocks(lengths, table, 16, 5)


def test_kv_reconstruct_paged_matches_row_level():
    """Per listed block the paged reconstruction equals the row-level one on the
    sequence's positions; padding entries give zero rows; a bad id is flagged."""
    pool_bits = synth.bf16_normal(6, 93, (10 * 16, 64))
    pool = oracle.widen_bf16(pool_bits)
    B = _bf16_matrix(6, 94, (64, 128), 0.125)
    lengths, table = [20, 35], [[3, 8, -1], [1, 0, 6]]
    blocks, n, _ = oracle.remap_build_blocks(lengths, table, 16, 7)
    out, bad = oracle.kv_reconstruct_paged(pool, blocks, n, B)
    assert not bad and out.shape == (7 * 16, 128)
    rows, nr, _ = oracle.remap_build(lengths, table, 16, 0, 64)
    _, ref, _ = oracle.kv_reconstruct(pool, rows, nr, 64, B)
    i = 0
    for s2, L in enumerate(lengths):
        first = sum((lengths[t] + 15) // 16 for t in range(s2))
        for p2 in range(L):
            assert np.array_equal(out[(first + p2 // 16) * 16 + p2 % 16], ref[i])
            i += 1
    assert not np.any(out[n * 16:])
    blocks[1] = 99
    out2, bad = oracle.kv_reconstruct_paged(pool, blocks, n, B)
    assert bad and not np.any(out2[16:32])


def test_kv_latent_write_then_reconstruct():
    """Writing the latents of new tokens into their pool rows and reconstructing
    those rows gives the dense product x A B of the tokens, and the other rows
    of the pool are untouched; an entry outside the pool is skipped and flagged."""
    x = _bf16_matrix(7, 95, (3, 32))
    A = _bf16_matrix(7, 96, (32, 16), 0.2)
    B = _bf16_matrix(7, 97, (16, 24), 0.2)
    pool = _bf16_matrix(7, 98, (20, 16))
    rows = [17, 2, 9]
    out, bad = oracle.kv_latent_write(x, A, rows, pool)
    assert not bad
    for m, j in enumerate(rows):
        assert np.allclose(out[j], x[m] @ A, rtol=0, atol=1e-13)
    keep = [i for i in range(20) if i not in rows]
    assert np.array_equal(out[keep], pool[keep])
    _, rec, _ = oracle.kv_reconstruct(out, rows, 3, 3, B)
    _, dense = oracle.lowrank_linear(x, A, B)
    assert np.allclose(rec, dense, rtol=0, atol=1e-12)
    out2, bad = oracle.kv_latent_write(x, A, [17, 20, -1], pool)
    assert bad and np.array_equal(np.delete(out2, 17, axis=0), np.delete(pool, 17, axis=0))


def test_block_relu_mlp_path():
    """Non-GLU MLP with up = I and down = I: h2 = h1 + max(n2, 0); the gate factor is never read."""
    d = 16
    h = _bf16_matrix(12, 1, (3, d))
    f = _zero_factors(d, d, d)
    f["up"] = (np.eye(d), np.eye(d))
    f["down"] = (np.eye(d), np.eye(d))
    f["gate"] = None
    out = oracle.block_forward(h, f, 2, 2, 8, return_all=True, mlp="relu")
    n2 = out["n2"]
    want = out["h1"] + np.where(n2 > 0, n2, 0.0)
    assert np.allclose(out["h2"], want, rtol=0, atol=1e-15)
    assert np.array_equal(oracle.relu(np.array([-2.0, -0.0, 0.0, 3.5])), [0.0, 0.0, 0.0, 3.5])


# ------------------------------------------------- rank-space sharding
@pytest.mark.parametrize("n,G", [(64, 1), (256, 2), (2432, 8), (576, 9), (3840, 7), (1216, 19)])
def test_shard_columns_partition(n, G):
    """Contiguous, in process order, whole 64-column blocks, sizes within one block of each other."""
    parts = oracle.shard_columns(n, G)
    assert len(parts) == G
    assert parts[0][0] == 0 and parts[-1][1] == n
    for (a, b), (c, _) in zip(parts, parts[1:]):
        assert b == c
    sizes = [b - a for a, b in parts]
    assert all(s % 64 == 0 and s >= 64 for s in sizes)
    assert max(sizes) - min(sizes) <= 64


def test_rank_sharded_exact_integers():
    """Small-integer inputs make every fp64 product and sum exact: the sharded
    scheme must reproduce the exact integer product x A B, its t_g must be the
    exact columns of x A, and every G gives the same answer."""
    rng = np.random.default_rng(5)
    x = rng.integers(-3, 4, size=(3, 128)).astype(np.float64)
    A = rng.integers(-2, 3, size=(128, 320)).astype(np.float64)
    B = rng.integers(-2, 3, size=(320, 192)).astype(np.float64)
    xi = [[int(v) for v in row] for row in x]
    Ai = [[int(v) for v in row] for row in A]
    Bi = [[int(v) for v in row] for row in B]
    t_exact = [[sum(xi[m][k] * Ai[k][j] for k in range(128)) for j in range(320)] for m in range(3)]
    y_exact = [[sum(t_exact[m][j] * Bi[j][o] for j in range(320)) for o in range(192)] for m in range(3)]
    for G in (1, 2, 3, 5):
        t_parts, t, y = oracle.rank_sharded_linear(x, A, B, G)
        assert np.array_equal(t, np.array(t_exact, dtype=np.float64))
        assert np.array_equal(y, np.array(y_exact, dtype=np.float64))
        for (a, b), tg in zip(oracle.shard_columns(320, G), t_parts):
            assert np.array_equal(tg, np.array(t_exact, dtype=np.float64)[:, a:b])


def test_rank_sharded_equals_unsharded_bf16():
    """On bf16-valued inputs the sharded result equals the plain (x A) B to fp64 rounding."""
    x = _bf16_matrix(3, 40, (5, 256))
    A = _bf16_matrix(3, 41, (256, 384), 1 / 16)
    B = _bf16_matrix(3, 42, (384, 512), 1 / 20)
    _, y_ref = oracle.lowrank_linear(x, A, B)
    for G in (1, 2, 4, 6):
        _, _, y = oracle.rank_sharded_linear(x, A, B, G)
        assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_ring_collectives_equal_chunks(G):
    """Equal chunks: an all-gather delivers the (G-1) chunks a process lacks,
    (G-1)/G of the matrix; a ring all-reduce moves twice that; one process moves nothing."""
    n, M, e = 64 * 8 * 3, 7, 2
    chunks = [n // G] * G
    ag = oracle.ring_allgather_received(chunks, M, e)
    ar = oracle.ring_allreduce_received(chunks, M, e)
    assert ag == [(G - 1) * n // G * M * e] * G
    assert ar == [2 * (G - 1) * n // G * M * e] * G


def test_ring_allgather_delivers_every_other_chunk_once():
    """Uneven chunks: process g receives exactly the chunks it does not own, once each."""
    chunks = [64, 128, 192, 64, 320]
    M, e = 3, 2
    ag = oracle.ring_allgather_received(chunks, M, e)
    for g in range(len(chunks)):
        assert ag[g] == (sum(chunks) - chunks[g]) * M * e
