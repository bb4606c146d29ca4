"""Python binding of liblr, the GB300 factorized-linear inference path.

Argument marshalling only: every computation runs in the CUDA kernels of
``liblr.so`` (see ``include/lr.h`` for the C ABI).  PyTorch provides device
memory and streams; tensors are passed by ``data_ptr()``.  Importing this
package fails if the library has not been built (``build.build()``): there
is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblr.so")

LR_OK = 0
LR_ERR_INVALID_ARG = 1
LR_ERR_UNSUPPORTED = 2
LR_ERR_CUDA = 3
LR_ERR_TIMEOUT = 4
LR_ERR_REMAP_RANGE = 5
LR_ERR_STATE = 6
LR_BF16 = 0
LR_F32 = 1
PROJ = ("q", "k", "v", "o", "gate", "up", "down")


class LrError(RuntimeError):
    def __init__(self, where: str, status: int, detail: str):
        super().__init__("%s: %s (%s)" % (where, status_string(status), detail))
        self.status = status


class Factor(ctypes.Structure):
    _fields_ = [("At", ctypes.c_void_p), ("Bt", ctypes.c_void_p), ("d_in", ctypes.c_int32),
                ("d_out", ctypes.c_int32), ("r", ctypes.c_int32)]


class BlockDesc(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("eps", ctypes.c_float), ("f", Factor * 7),
                ("mlp", ctypes.c_int32)]


MLP_SWIGLU = 0
MLP_RELU = 1


class StackDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("layers", ctypes.POINTER(BlockDesc)),
                ("pool_in", ctypes.c_void_p), ("pool_out", ctypes.c_void_p),
                ("pool_rows", ctypes.c_int64), ("remap", ctypes.c_void_p),
                ("n_active", ctypes.c_void_p), ("cap", ctypes.c_int64),
                ("xbuf", ctypes.c_void_p), ("h", ctypes.c_void_p), ("ybuf", ctypes.c_void_p),
                ("scratch", ctypes.c_void_p), ("scratch_bytes", ctypes.c_size_t),
                ("dev_status", ctypes.c_void_p), ("mode", ctypes.c_int32)]


STACK_AUTO = 0
STACK_LAYERED = 1


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("liblr.so is not built: run rank_decomposed_gb300.build.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "lr_linear_workspace_bytes": (sz, [i64, P(Factor)]),
        "lr_linear_forward": (i32, [vp, i64, vp, i64, i32, i64, P(Factor), vp, sz, vp, vp]),
        "lr_linear_forward_noalloc": (i32, [vp, i64, vp, i64, i32, i64, P(Factor), vp, vp]),
        "lr_factor_pack": (i32, [vp, vp, i32, i32, i32, vp, vp, vp]),
        "lr_block_scratch_bytes": (sz, [i64, P(BlockDesc)]),
        "lr_block_forward": (i32, [vp, i64, P(BlockDesc), vp, sz, vp, vp]),
        "remap_compact": (i32, [vp, i64, i64, vp, vp, vp, i64, vp, vp]),
        "remap_scatter": (i32, [vp, vp, vp, vp, i64, i64, i64, vp, vp]),
        "remap_build": (i32, [vp, i64, vp, i32, i32, i32, i64, vp, vp, vp]),
        "lr_kv_reconstruct": (i32, [vp, i64, i32, vp, vp, i64, vp, vp, i32, vp, vp, vp]),
        "remap_build_blocks": (i32, [vp, i64, vp, i32, i32, i64, vp, vp, vp]),
        "lr_kv_latent_write": (i32, [vp, i64, i64, vp, i32, i32, vp, vp, i64, vp, vp]),
        "lr_kv_reconstruct_paged": (i32, [vp, i64, i32, vp, vp, i64, vp, i32, vp, vp, vp]),
        "lr_rank_sharded_workspace_bytes": (sz, [i64, P(Factor), i32]),
        "lr_linear_forward_rank_sharded": (i32, [vp, i64, vp, i64, i32, i64, P(Factor), i32, vp, sz,
                                                 vp, vp]),
        "lr_rank_shard_comm_bytes": (i32, [i64, i32, i32, i32, i32, P(i64), P(i64)]),
        "lr_stack_forward": (i32, [P(StackDesc), vp]),
        "lr_graph_capture": (i32, [P(StackDesc), P(vp)]),
        "lr_graph_replay": (i32, [vp, vp]),
        "lr_graph_destroy": (i32, [vp]),
        "lr_stack_launch_count": (i64, [P(StackDesc)]),
        "lr_stack_scratch_bytes": (sz, [P(StackDesc)]),
        "lr_status_string": (ctypes.c_char_p, [i32]),
        "lr_last_error": (ctypes.c_char_p, []),
        "lr_test_stall_producer": (None, [i32]),
        "lr_test_prefill_schedule": (None, [i32, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(st: int) -> str:
    return lib.lr_status_string(st).decode()


def last_error() -> str:
    return lib.lr_last_error().decode()


def _check(where: str, st: int):
    if st != LR_OK:
        raise LrError(where, st, last_error())


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _bf16(t, name):
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError("%s must be bfloat16" % name)
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be a row-major 2-D tensor" % name)


@dataclass
class FactorPair:
    """A decomposed projection: At = A_r^T [r][d_in], Bt = B_r^T [d_out][r], bf16 on the device."""
    At: object
    Bt: object

    @property
    def d_in(self):
        return int(self.At.shape[1])

    @property
    def d_out(self):
        return int(self.Bt.shape[0])

    @property
    def r(self):
        return int(self.At.shape[0])

    def c(self) -> Factor:
        _bf16(self.At, "At")
        _bf16(self.Bt, "Bt")
        if self.Bt.shape[1] != self.At.shape[0]:
            raise ValueError("At and Bt disagree on the rank")
        return Factor(self.At.data_ptr(), self.Bt.data_ptr(), self.d_in, self.d_out, self.r)


@dataclass
class Block:
    """Shape and factors of one decomposed block (projections in q,k,v,o,gate,up,down order)."""
    d_model: int
    d_ff: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    factors: list
    eps: float = 1e-6
    mlp: int = MLP_SWIGLU   # MLP_RELU: non-GLU, factors[4] (gate) may be None

    def c(self) -> BlockDesc:
        b = BlockDesc()
        b.d_model, b.d_ff = self.d_model, self.d_ff
        b.n_heads, b.n_kv_heads, b.head_dim = self.n_heads, self.n_kv_heads, self.head_dim
        b.eps = self.eps
        b.mlp = self.mlp
        for i, f in enumerate(self.factors):
            if f is not None:
                b.f[i] = f.c()
        return b


def factor_pack(A, B, stream=None) -> FactorPair:
    """A FactorPair from the pages' orientation: A_r bf16 [d_in][r], B_r bf16 [r][d_out] (device).

    The library stores the transposes (At = A_r^T, Bt = B_r^T); lr_factor_pack
    writes them on the device.  Allocation of the two outputs is done here
    with torch.
    """
    import torch
    _bf16(A, "A")
    _bf16(B, "B")
    if A.shape[1] != B.shape[0]:
        raise ValueError("A [d_in][r] and B [r][d_out] disagree on r")
    d_in, r = A.shape
    d_out = B.shape[1]
    At = torch.empty((r, d_in), dtype=torch.bfloat16, device=A.device)
    Bt = torch.empty((d_out, r), dtype=torch.bfloat16, device=B.device)
    _check("lr_factor_pack", lib.lr_factor_pack(A.data_ptr(), B.data_ptr(), d_in, d_out, r, At.data_ptr(),
                                                Bt.data_ptr(), _stream(stream)))
    return FactorPair(At, Bt)


# --------------------------------------------------------------- linear
def linear_workspace_bytes(M: int, f: FactorPair) -> int:
    return int(lib.lr_linear_workspace_bytes(M, ctypes.byref(f.c())))


def linear_forward(x, f: FactorPair, y, workspace, status, stream=None):
    """y = (x A_r) B_r; y is bf16 or fp32 [M][>= d_out]."""
    import torch
    _bf16(x, "x")
    if y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a row-major 2-D tensor")
    ydt = {torch.bfloat16: LR_BF16, torch.float32: LR_F32}.get(y.dtype)
    if ydt is None:
        raise TypeError("y must be bfloat16 or float32")
    fc = f.c()
    st = lib.lr_linear_forward(x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0), ydt,
                               x.shape[0], ctypes.byref(fc), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _ptr(status),
                               _stream(stream))
    _check("lr_linear_forward", st)


def rank_sharded_workspace_bytes(M: int, f: FactorPair, n_shards: int) -> int:
    fc = f.c()
    return int(lib.lr_rank_sharded_workspace_bytes(M, ctypes.byref(fc), n_shards))


def linear_forward_rank_sharded(x, f: FactorPair, n_shards: int, y, workspace, status, stream=None):
    """y = (x A_r) B_r computed as n_shards simulated processes of the rank-space scheme.

    Each process runs the down projection on its block of rank columns, the
    blocks are all-gathered (device copies) into one t, and each process runs
    the up projection on its block of output columns.
    """
    import torch
    _bf16(x, "x")
    if y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a row-major 2-D tensor")
    ydt = {torch.bfloat16: LR_BF16, torch.float32: LR_F32}.get(y.dtype)
    if ydt is None:
        raise TypeError("y must be bfloat16 or float32")
    fc = f.c()
    st = lib.lr_linear_forward_rank_sharded(x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0), ydt,
                                            x.shape[0], ctypes.byref(fc), n_shards, workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(), _ptr(status),
                                            _stream(stream))
    _check("lr_linear_forward_rank_sharded", st)


def rank_shard_comm_bytes(M: int, d_out: int, r: int, n_shards: int, elem_bytes: int = 2):
    """(rank-space all-gather bytes, full-space all-reduce bytes) received by the busiest process."""
    a, b = ctypes.c_int64(0), ctypes.c_int64(0)
    _check("lr_rank_shard_comm_bytes",
           lib.lr_rank_shard_comm_bytes(M, d_out, r, n_shards, elem_bytes, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


NOALLOC_SCRATCH_BYTES = 4 << 20


def linear_forward_noalloc(x, f: FactorPair, y, status, stream=None):
    """y = (x A_r) B_r with the intermediate kept in the library's static device array.

    For callers that cannot allocate device memory: no workspace argument and
    no allocation.  Requires M * r * 2 <= NOALLOC_SCRATCH_BYTES; calls that
    overlap on the GPU share the array and must be ordered on one stream.
    """
    import torch
    _bf16(x, "x")
    if y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a row-major 2-D tensor")
    ydt = {torch.bfloat16: LR_BF16, torch.float32: LR_F32}.get(y.dtype)
    if ydt is None:
        raise TypeError("y must be bfloat16 or float32")
    fc = f.c()
    st = lib.lr_linear_forward_noalloc(x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0), ydt,
                                       x.shape[0], ctypes.byref(fc), _ptr(status), _stream(stream))
    _check("lr_linear_forward_noalloc", st)


# ---------------------------------------------------------------- block
def block_scratch_bytes(M: int, b: Block) -> int:
    return int(lib.lr_block_scratch_bytes(M, ctypes.byref(b.c())))


def block_forward(h, b: Block, scratch, status, stream=None):
    """One decomposed block applied in place to the fp32 residual h [M][d_model]."""
    import torch
    if h.dtype != torch.float32 or not h.is_contiguous():
        raise TypeError("h must be a contiguous float32 tensor")
    bc = b.c()
    st = lib.lr_block_forward(h.data_ptr(), h.shape[0], ctypes.byref(bc), scratch.data_ptr(),
                              scratch.numel() * scratch.element_size(), _ptr(status),
                              _stream(stream))
    _check("lr_block_forward", st)


# ---------------------------------------------------------------- remap
def remap_compact(pool, remap, n_active, buf, status, stream=None):
    row_bytes = pool.stride(0) * pool.element_size()
    st = lib.remap_compact(pool.data_ptr(), pool.shape[0], row_bytes, remap.data_ptr(),
                           n_active.data_ptr(), buf.data_ptr(), buf.shape[0], _ptr(status),
                           _stream(stream))
    _check("remap_compact", st)


def remap_scatter(buf, remap, n_active, pool, status, stream=None):
    row_bytes = pool.stride(0) * pool.element_size()
    st = lib.remap_scatter(buf.data_ptr(), remap.data_ptr(), n_active.data_ptr(), pool.data_ptr(),
                           pool.shape[0], row_bytes, buf.shape[0], _ptr(status), _stream(stream))
    _check("remap_scatter", st)


def remap_build(lengths, block_table, block_rows: int, tail_rows: int, cap: int):
    """Host scan: returns (remap int32[cap], n_active, n_runs)."""
    L = np.ascontiguousarray(lengths, dtype=np.int32)
    T = np.ascontiguousarray(block_table, dtype=np.int32)
    if T.ndim != 2 or T.shape[0] != L.shape[0]:
        raise ValueError("block_table must be [n_seq][blocks_per_seq]")
    out = np.empty(cap, dtype=np.int32)
    na = ctypes.c_int32(0)
    nr = ctypes.c_int32(0)
    st = lib.remap_build(L.ctypes.data, L.shape[0], T.ctypes.data, T.shape[1], block_rows,
                         tail_rows, cap, out.ctypes.data, ctypes.byref(na), ctypes.byref(nr))
    _check("remap_build", st)
    return out, na.value, nr.value


def kv_reconstruct(latent_pool, remap, n_active, latent_buf, Bt, out, status, stream=None):
    """Compact the listed latent rows into latent_buf, then out = latent_buf Bt^T (bf16)."""
    _bf16(latent_pool, "latent_pool")
    _bf16(latent_buf, "latent_buf")
    _bf16(Bt, "Bt")
    _bf16(out, "out")
    r = latent_pool.shape[1]
    if latent_buf.shape[1] != r or Bt.shape[1] != r or out.shape[1] != Bt.shape[0] \
            or out.shape[0] != latent_buf.shape[0]:
        raise ValueError("kv_reconstruct: inconsistent shapes")
    st = lib.lr_kv_reconstruct(latent_pool.data_ptr(), latent_pool.shape[0], r, remap.data_ptr(),
                               n_active.data_ptr(), latent_buf.shape[0], latent_buf.data_ptr(),
                               Bt.data_ptr(), Bt.shape[0], out.data_ptr(), _ptr(status),
                               _stream(stream))
    _check("lr_kv_reconstruct", st)


def remap_build_blocks(lengths, block_table, block_rows: int, cap_blocks: int):
    """Host scan at block granularity: returns (blocks int32[cap_blocks], n_blocks, n_runs)."""
    L = np.ascontiguousarray(lengths, dtype=np.int32)
    T = np.ascontiguousarray(block_table, dtype=np.int32)
    if T.ndim != 2 or T.shape[0] != L.shape[0]:
        raise ValueError("block_table must be [n_seq][blocks_per_seq]")
    out = np.empty(cap_blocks, dtype=np.int32)
    nb = ctypes.c_int32(0)
    nr = ctypes.c_int32(0)
    st = lib.remap_build_blocks(L.ctypes.data, L.shape[0], T.ctypes.data, T.shape[1], block_rows, cap_blocks,
                                out.ctypes.data, ctypes.byref(nb), ctypes.byref(nr))
    _check("remap_build_blocks", st)
    return out, nb.value, nr.value


def kv_latent_write(x, At, rows, latent_pool, status, stream=None):
    """latent_pool[rows[m]] = bf16(x[m] A_r) for the M rows of x (At = A_r^T [r][d_in])."""
    _bf16(x, "x")
    _bf16(At, "At")
    _bf16(latent_pool, "latent_pool")
    r, d_in = At.shape
    if x.shape[1] != d_in or latent_pool.shape[1] != r or rows.shape[0] != x.shape[0]:
        raise ValueError("kv_latent_write: inconsistent shapes")
    st = lib.lr_kv_latent_write(x.data_ptr(), x.stride(0), x.shape[0], At.data_ptr(), d_in, r, rows.data_ptr(),
                                latent_pool.data_ptr(), latent_pool.shape[0], _ptr(status), _stream(stream))
    _check("lr_kv_latent_write", st)


def kv_reconstruct_paged(latent_pool, blocks, n_blocks, Bt, out, status, stream=None):
    """out[16 i + j] = latent_pool[16 blocks[i] + j] B_r for i < n_blocks (zero rows after)."""
    _bf16(latent_pool, "latent_pool")
    _bf16(Bt, "Bt")
    _bf16(out, "out")
    r = latent_pool.shape[1]
    if latent_pool.shape[0] % 16 or Bt.shape[1] != r or out.shape[1] != Bt.shape[0] \
            or out.shape[0] != 16 * blocks.shape[0]:
        raise ValueError("kv_reconstruct_paged: inconsistent shapes")
    st = lib.lr_kv_reconstruct_paged(latent_pool.data_ptr(), latent_pool.shape[0] // 16, r, blocks.data_ptr(),
                                     n_blocks.data_ptr(), blocks.shape[0], Bt.data_ptr(), Bt.shape[0],
                                     out.data_ptr(), _ptr(status), _stream(stream))
    _check("lr_kv_reconstruct_paged", st)


# ---------------------------------------------------------------- stack
@dataclass
class Stack:
    """A layer stack over fixed buffers: compact -> blocks -> scatter, eager or as a CUDA graph."""
    layers: list
    pool_in: object
    pool_out: object
    remap: object
    n_active: object
    xbuf: object
    h: object
    ybuf: object
    scratch: object
    status: object
    mode: int = STACK_AUTO
    _graph: object = field(default=None, repr=False)
    _desc: object = field(default=None, repr=False)
    _blocks: object = field(default=None, repr=False)

    def desc(self) -> StackDesc:
        if self._desc is None:
            arr = (BlockDesc * len(self.layers))(*[b.c() for b in self.layers])
            d = StackDesc()
            d.n_layers = len(self.layers)
            d.layers = ctypes.cast(arr, ctypes.POINTER(BlockDesc))
            d.pool_in, d.pool_out = self.pool_in.data_ptr(), self.pool_out.data_ptr()
            d.pool_rows = self.pool_in.shape[0]
            d.remap, d.n_active = self.remap.data_ptr(), self.n_active.data_ptr()
            d.cap = self.xbuf.shape[0]
            d.xbuf, d.h, d.ybuf = self.xbuf.data_ptr(), self.h.data_ptr(), self.ybuf.data_ptr()
            d.scratch = self.scratch.data_ptr()
            d.scratch_bytes = self.scratch.numel() * self.scratch.element_size()
            d.dev_status = _ptr(self.status)
            d.mode = self.mode
            self._blocks, self._desc = arr, d
        return self._desc

    @staticmethod
    def scratch_bytes(cap: int, layers, mode: int = STACK_AUTO) -> int:
        """Scratch bytes of a step over `cap` rows (the block buffers)."""
        arr = (BlockDesc * len(layers))(*[b.c() for b in layers])
        d = StackDesc()
        d.n_layers = len(layers)
        d.layers = ctypes.cast(arr, ctypes.POINTER(BlockDesc))
        d.cap = cap
        d.mode = mode
        return int(lib.lr_stack_scratch_bytes(ctypes.byref(d)))

    def launch_count(self) -> int:
        return int(lib.lr_stack_launch_count(ctypes.byref(self.desc())))

    def forward(self, stream=None):
        _check("lr_stack_forward", lib.lr_stack_forward(ctypes.byref(self.desc()), _stream(stream)))

    def capture(self):
        if self._graph is not None:
            self.destroy()
        g = ctypes.c_void_p()
        _check("lr_graph_capture", lib.lr_graph_capture(ctypes.byref(self.desc()), ctypes.byref(g)))
        self._graph = g

    def replay(self, stream=None):
        if self._graph is None:
            raise RuntimeError("capture() first")
        _check("lr_graph_replay", lib.lr_graph_replay(self._graph, _stream(stream)))

    def destroy(self):
        if self._graph is not None:
            _check("lr_graph_destroy", lib.lr_graph_destroy(self._graph))
            self._graph = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass
