"""Oracle: a plain, slow, fp64 CPU statement of the factorized-linear path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the ``rank_decomposed_gb300``
package, its CUDA library or its C-ABI) imports or calls this module; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` do.  It shares no code with the GPU path.  Its inputs are the
bf16 bit patterns made by ``synth``; it widens them exactly to fp64 and never
rounds after that.

Sources (DeInfer: Efficient Parallel Inferencing for Decomposed Large Language
Models, Huang, Huang, Liao, Wen; summaries at gist.science/paper/2604.17709 and
gist.science/es/paper/2604.17709):

* low-rank decomposition W ~ A B of every weight -- es page, "Resumen Tecnico"
  section 1; English page, section 1 (Problem Statement).
* down projection then up projection -- English page, section 2.A; es page
  section 2 ("proyecciones hacia abajo / hacia arriba").
* paged memory scanned for contiguous blocks, remapping index list, copy into a
  contiguous buffer, fixed-size GEMM in a static graph -- English page,
  section 2.C; es page section 2 ("Etapa de Preparacion", "Reproduccion del
  Grafico").
* decomposition of attention and MLP projections, MHA/GQA/MQA attention,
  GLU MLP -- es page section 1 and section 2 ("Generalizacion"); English
  page section 2.D.

Readings where the pages are silent (each is listed with its reason in the
repository's design notes): A_r is the down factor [d_in, r] and B_r the up
factor [r, d_out]; the block is a LLaMA block whose attention core is exact
attention over a one-token context (the output of every head is its value
vector, GQA-broadcast); RMSNorm has unit gain and eps = 1e-6; the MLP is
SiLU-GLU; the residual stream is carried in full precision; the paged block
size is 16 rows.

Pins (``tests/test_oracle.py``): every function here is checked against
something other than itself -- exact rational brute force, associativity, the
identity and one-hot special cases, an SVD rank check with the Eckart-Young
error, closed forms of RMSNorm and SiLU, hand-derived remap fixtures under
``tests/golden/`` and permutation inverses.  The pages print no worked
example, no kernel output and no single-GPU value, so no function is pinned to
a number printed on the pages; that part of parity is unpinned.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

LLAMA_RMS_EPS = 1e-6


# --------------------------------------------------------------- formats
def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ rank rule
def rank_for(d_in: int, d_out: int, rho) -> int:
    """Rank that removes a fraction ``rho`` of a d_in x d_out weight's parameters.

    r = (1 - rho) * d_in * d_out / (d_in + d_out), rounded to the nearest
    multiple of 64 (ties up).  Computed in exact rational arithmetic.
    """
    rho = Fraction(str(rho))
    exact = (1 - rho) * d_in * d_out / (d_in + d_out)
    q = exact / 64
    k = (q + Fraction(1, 2)).__floor__()
    return int(64 * max(k, 1))


# ---------------------------------------------------- factorized linear
def lowrank_linear(x: np.ndarray, A: np.ndarray, B: np.ndarray):
    """y = (x A) B for x [M, d_in], A [d_in, r], B [r, d_out]; returns (t, y).

    The down projection t = x A is formed first and then the up projection
    y = t B, the order in which the decomposed layer is evaluated (English
    page, section 2.A).  fp64 throughout, no intermediate rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    t = x @ np.asarray(A, dtype=np.float64)
    y = t @ np.asarray(B, dtype=np.float64)
    return t, y


def factor_from_stored(At_bits, Bt_bits):
    """Stored out-major bf16 factors (A_r^T [r][d_in], B_r^T [d_out][r]) -> fp64 A_r, B_r."""
    return widen_bf16(At_bits).T.copy(), widen_bf16(Bt_bits).T.copy()


# ------------------------------------------------------------ block glue
def rmsnorm(h: np.ndarray, eps: float = LLAMA_RMS_EPS) -> np.ndarray:
    """Row-wise h / sqrt(mean(h^2) + eps) with unit gain."""
    h = np.asarray(h, dtype=np.float64)
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return h / np.sqrt(ms + eps)


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def one_token_attention(v: np.ndarray, n_heads: int, n_kv_heads: int, head_dim: int):
    """Attention over a context of one token: head h returns the value of kv head h // g.

    With a single key the softmax weight is exactly 1, so the output of query
    head h is the value vector of the kv head it shares (g = n_heads /
    n_kv_heads query heads per kv head: GQA; g = 1: MHA; n_kv_heads = 1: MQA).
    """
    M = v.shape[0]
    g = n_heads // n_kv_heads
    out = np.empty((M, n_heads * head_dim), dtype=np.float64)
    for h in range(n_heads):
        j = h // g
        out[:, h * head_dim:(h + 1) * head_dim] = v[:, j * head_dim:(j + 1) * head_dim]
    return out


def relu(z: np.ndarray) -> np.ndarray:
    """max(z, 0)."""
    return np.maximum(np.asarray(z, dtype=np.float64), 0.0)


def block_forward(h: np.ndarray, factors, n_heads: int, n_kv_heads: int, head_dim: int,
                  eps: float = LLAMA_RMS_EPS, return_all: bool = False, mlp: str = "swiglu"):
    """One decomposed LLaMA block, attention core replaced by one-token attention.

    ``factors`` maps "q","k","v","o","gate","up","down" to (A, B) fp64 pairs.
    n1 = rmsnorm(h); q, k, v = LR(n1); h1 = h + LR_o(attn(v));
    n2 = rmsnorm(h1); h2 = h1 + LR_down(silu(LR_gate(n2)) * LR_up(n2)).
    With mlp="relu" (a non-GLU MLP, English page section 2.D) the MLP is
    h2 = h1 + LR_down(relu(LR_up(n2))) and "gate" is not used.
    """
    h = np.asarray(h, dtype=np.float64)
    n1 = rmsnorm(h, eps)
    _, q = lowrank_linear(n1, *factors["q"])
    _, k = lowrank_linear(n1, *factors["k"])
    _, v = lowrank_linear(n1, *factors["v"])
    attn = one_token_attention(v, n_heads, n_kv_heads, head_dim)
    _, o = lowrank_linear(attn, *factors["o"])
    h1 = h + o
    n2 = rmsnorm(h1, eps)
    _, u = lowrank_linear(n2, *factors["up"])
    if mlp == "relu":
        g = None
        a = relu(u)
    else:
        _, g = lowrank_linear(n2, *factors["gate"])
        a = silu(g) * u
    _, dn = lowrank_linear(a, *factors["down"])
    h2 = h1 + dn
    if return_all:
        return dict(n1=n1, q=q, k=k, v=v, attn=attn, o=o, h1=h1, n2=n2, gate=g,
                    up=u, act=a, down=dn, h2=h2)
    return h2


def stack_forward(h: np.ndarray, layers, n_heads: int, n_kv_heads: int, head_dim: int,
                  eps: float = LLAMA_RMS_EPS, mlp: str = "swiglu") -> np.ndarray:
    """Apply ``block_forward`` for each factor set in ``layers`` in order."""
    for f in layers:
        h = block_forward(h, f, n_heads, n_kv_heads, head_dim, eps, mlp=mlp)
    return h


# ------------------------------------------------------------------ remap
def remap_build(lengths, block_table, block_rows: int, tail_rows: int, cap: int):
    """Preparation stage: paged rows -> remap index list over physical rows.

    Sequences are taken in order; for each, its last ``tail_rows`` positions
    (all positions if ``tail_rows <= 0``) are mapped through the block table to
    physical pool rows ``block_table[s][p // block_rows] * block_rows +
    p % block_rows``.  Returns ``(remap[cap], n_active, n_runs)``: unused
    entries are -1 and ``n_runs`` counts maximal runs of consecutive physical
    rows (the contiguous pieces a copy can move as one).  Raises ValueError
    when the rows do not fit in ``cap`` or a needed table entry is negative.
    """
    rows = []
    for s, L in enumerate(lengths):
        L = int(L)
        start = 0 if tail_rows <= 0 else max(0, L - tail_rows)
        for p in range(start, L):
            blk = int(block_table[s][p // block_rows])
            if blk < 0:
                raise ValueError("block table entry missing")
            rows.append(blk * block_rows + p % block_rows)
    if len(rows) > cap:
        raise ValueError("rows exceed capacity")
    remap = np.full(cap, -1, dtype=np.int32)
    remap[: len(rows)] = rows
    n_runs = 0
    for i in range(len(rows)):
        if i == 0 or rows[i] != rows[i - 1] + 1:
            n_runs += 1
    return remap, len(rows), n_runs


def remap_gather(pool: np.ndarray, remap, n_active: int, cap: int):
    """Copy into a fixed [cap, ...] buffer: row i <- pool[remap[i]] for i < n_active.

    Rows at or beyond ``n_active`` are zero.  A remap entry outside the pool
    gives a zero row and sets the returned error flag.
    """
    buf = np.zeros((cap,) + pool.shape[1:], dtype=pool.dtype)
    bad = False
    for i in range(min(n_active, cap)):
        j = int(remap[i])
        if 0 <= j < pool.shape[0]:
            buf[i] = pool[j]
        else:
            bad = True
    return buf, bad


def remap_scatter(buf: np.ndarray, remap, n_active: int, pool: np.ndarray):
    """Inverse copy: pool[remap[i]] <- buf[i] for i < n_active; returns (pool', bad)."""
    out = pool.copy()
    bad = False
    for i in range(min(n_active, buf.shape[0])):
        j = int(remap[i])
        if 0 <= j < pool.shape[0]:
            out[j] = buf[i]
        else:
            bad = True
    return out, bad


def kv_reconstruct(latent_pool: np.ndarray, remap, n_active: int, cap: int, B: np.ndarray):
    """Low-rank KV reconstruction over a compacted buffer (English page, section 2.C).

    The listed latent rows are copied into a [cap, r] buffer (zero past
    n_active) and multiplied by the up factor B [r, d_kv]: rows of K (or V).
    fp64; returns (buffer, reconstructed rows, out-of-range flag).
    """
    buf, bad = remap_gather(latent_pool, remap, n_active, cap)
    return buf, np.asarray(buf, dtype=np.float64) @ np.asarray(B, dtype=np.float64), bad


def kv_latent_write(x, A, rows, pool):
    """The latent KV producer (English page, sections 1 and 2.C).

    Row m of the down projection x A (x [M, d_in], A [d_in, r]) is written to
    row rows[m] of the paged latent pool [pool_rows, r]; other rows keep their
    contents.  Entries outside the pool are skipped and set the returned flag.
    fp64, no rounding; returns (pool', flag).
    """
    t = np.asarray(x, dtype=np.float64) @ np.asarray(A, dtype=np.float64)
    out = np.array(pool, dtype=np.float64, copy=True)
    bad = False
    for m, j in enumerate(rows):
        j = int(j)
        if 0 <= j < out.shape[0]:
            out[j] = t[m]
        else:
            bad = True
    return out, bad


def remap_build_blocks(lengths, block_table, block_rows: int, cap_blocks: int):
    """Preparation stage at block granularity (English page, section 2.C: the
    remapping index list as a new block table).

    For each sequence in order, the physical blocks holding its positions
    0 .. L-1: the first ceil(L / block_rows) entries of its block-table row.
    Returns ``(blocks[cap_blocks], n_blocks, n_runs)`` with unused entries -1
    and ``n_runs`` the maximal runs of consecutive block ids.  Raises
    ValueError when the blocks exceed ``cap_blocks`` or an entry is missing.
    """
    out = []
    for s, L in enumerate(lengths):
        nb = (int(L) + block_rows - 1) // block_rows
        for b in range(nb):
            blk = int(block_table[s][b])
            if blk < 0:
                raise ValueError("block table entry missing")
            out.append(blk)
    if len(out) > cap_blocks:
        raise ValueError("blocks exceed capacity")
    blocks = np.full(cap_blocks, -1, dtype=np.int32)
    blocks[: len(out)] = out
    n_runs = sum(1 for i in range(len(out)) if i == 0 or out[i] != out[i - 1] + 1)
    return blocks, len(out), n_runs


def kv_reconstruct_paged(latent_pool: np.ndarray, blocks, n_blocks: int, B: np.ndarray, block_rows: int = 16):
    """Reconstruction of whole listed blocks (English page, section 2.C).

    Row ``block_rows * i + j`` of the result is row ``j`` of block
    ``blocks[i]`` of the paged latent pool times the up factor B [r, d_kv], for
    i < n_blocks; the rows of the other list entries are zero.  A block id
    outside the pool gives zero rows and sets the returned flag.  fp64.
    """
    cap = len(blocks)
    r = latent_pool.shape[1]
    buf = np.zeros((cap * block_rows, r), dtype=np.float64)
    bad = False
    pool_blocks = latent_pool.shape[0] // block_rows
    for i in range(min(n_blocks, cap)):
        b = int(blocks[i])
        if 0 <= b < pool_blocks:
            buf[i * block_rows:(i + 1) * block_rows] = latent_pool[b * block_rows:(b + 1) * block_rows]
        else:
            bad = True
    return buf @ np.asarray(B, dtype=np.float64), bad


# ------------------------------------------------------ rank-space sharding
def shard_columns(n: int, G: int):
    """Split n columns (a multiple of 64) over G processes in whole 64-column blocks.

    Process g gets [64 * floor(g * nb / G), 64 * floor((g + 1) * nb / G)) with
    nb = n / 64: contiguous, as even as whole blocks allow, in process order.
    """
    nb = n // 64
    return [(64 * (nb * g // G), 64 * (nb * (g + 1) // G)) for g in range(G)]


def rank_sharded_linear(x, A, B, G: int):
    """The low-rank communication scheme for one factorized linear (English page, section 2.A).

    The down projection is split by columns over G processes, its outputs are
    all-gathered in the rank dimension so every process holds the same t, and
    the up projection runs in shard mode: process g computes only its own
    block of output columns, so no reduce-sum is needed.  Returns
    (per-process t_g, gathered t, y).  fp64, no rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    t_parts = [x @ A[:, a:b] for a, b in shard_columns(A.shape[1], G)]
    t = np.concatenate(t_parts, axis=1)
    y = np.concatenate([t @ B[:, a:b] for a, b in shard_columns(B.shape[1], G)], axis=1)
    return t_parts, t, y


def ring_allgather_received(chunk_cols, M: int, elem_bytes: int):
    """Bytes each process receives in a ring all-gather of an [M][sum(chunk_cols)] matrix.

    Process g starts with chunk g.  In step s = 0 .. G-2 every process passes
    the chunk it received in the previous step (its own in step 0) to its
    right neighbour, so process g receives chunk (g - s - 1) mod G.
    """
    G = len(chunk_cols)
    recv = [0] * G
    for s in range(G - 1):
        for g in range(G):
            recv[g] += chunk_cols[(g - s - 1) % G] * M * elem_bytes
    return recv


def ring_allreduce_received(chunk_cols, M: int, elem_bytes: int):
    """Bytes each process receives in a ring all-reduce (reduce-scatter, then all-gather).

    Reduce-scatter: in step s process g receives the running partial sum of
    chunk (g - s - 1) mod G from its left neighbour and adds its own part, so
    after G-1 steps each chunk is fully reduced on one process.  The
    all-gather phase then circulates the reduced chunks as in
    ring_allgather_received.  Both phases move whole chunks.
    """
    G = len(chunk_cols)
    recv = [0] * G
    for s in range(G - 1):  # reduce-scatter
        for g in range(G):
            recv[g] += chunk_cols[(g - s - 1) % G] * M * elem_bytes
    gather = ring_allgather_received(chunk_cols, M, elem_bytes)
    return [a + b for a, b in zip(recv, gather)]
