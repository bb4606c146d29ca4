/*
 * lr.h -- C ABI of liblr, the GB300 (sm_103a) factorized-linear inference path.
 *
 * What it computes comes from DeInfer: Efficient Parallel Inferencing for
 * Decomposed Large Language Models (Huang, Huang, Liao, Wen), as summarised on
 * gist.science/paper/2604.17709 (English page) and gist.science/es/paper/
 * 2604.17709 (Spanish page).  Every weight W[d_in][d_out] of a transformer
 * block is approximated by two low-rank factors, W ~ A_r B_r (Spanish page,
 * "Resumen Tecnico" section 1; English page section 1), and a layer is
 * evaluated as a down projection followed by an up projection (English page
 * section 2.A).  For decoding under a static CUDA graph, rows scattered over
 * paged memory are first listed in a remap table and copied into a fixed
 * buffer; the graph then runs fixed-size GEMMs on that buffer (English page
 * section 2.C).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers marked "device" are CUDA device pointers owned by the caller; the
 *   library never allocates, frees or keeps them past the call (the graph
 *   object keeps them, see lr_graph_capture).  Pointers marked "host" are
 *   ordinary host memory.
 * - bf16 means IEEE bfloat16 bit patterns (uint16_t).  All matrices are
 *   row-major with the leading dimension given in elements.
 * - Factors are stored out-major, the layout of a linear layer's weight:
 *   the down factor A_r[d_in][r] is stored transposed as At[r][d_in] and the
 *   up factor B_r[r][d_out] as Bt[d_out][r].  Every tensor-core operand is
 *   then contiguous along the reduction dimension.
 * - Work is enqueued on the given stream (0 = the legacy default stream) and
 *   runs asynchronously.  Argument errors are detected on the host before
 *   anything is enqueued and returned as LR_ERR_INVALID_ARG or
 *   LR_ERR_UNSUPPORTED; nothing is launched in that case.
 * - Device-side problems never trap: a kernel that meets one stores the first
 *   error code into the caller's int32 device word `dev_status` (compare-and-
 *   swap from 0) and finishes safely.  The caller reads it after synchronising
 *   and resets it to 0.
 * - Every wait inside a kernel is bounded (about two seconds); a wait that
 *   runs out reports LR_ERR_TIMEOUT through dev_status and the kernel returns.
 * - No exception crosses this interface.  lr_last_error() gives a one-line
 *   description of the last host-side error of the calling thread.
 */
#ifndef LR_H_
#define LR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lr_stream; /* a cudaStream_t */

typedef enum {
  LR_OK = 0,
  LR_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, small buffer */
  LR_ERR_UNSUPPORTED = 2,  /* a dimension outside what the kernels handle */
  LR_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  LR_ERR_TIMEOUT = 4,      /* device: a bounded wait ran out */
  LR_ERR_REMAP_RANGE = 5,  /* device: a remap entry outside the pool */
  LR_ERR_STATE = 6         /* wrong object state (e.g. replaying a destroyed graph) */
} lr_status;

typedef enum { LR_BF16 = 0, LR_F32 = 1 } lr_dtype;

/* One factor pair (A_r, B_r) of a decomposed projection, W ~ A_r B_r.
 * At: device bf16 [r][d_in]  (A_r transposed), row stride d_in.
 * Bt: device bf16 [d_out][r] (B_r transposed), row stride r.
 * d_in, d_out and r must be positive multiples of 64 (LR_ERR_UNSUPPORTED
 * otherwise); both pointers must be 16-byte aligned. */
typedef struct {
  const void* At;
  const void* Bt;
  int32_t d_in;
  int32_t d_out;
  int32_t r;
} lr_factor;

/* lr_factor_pack: the factors in the pages' orientation, W ~ A_r B_r
 * (Spanish page, "Resumen Tecnico" section 1), to the layout above.
 *   A: device bf16 [d_in][r] row-major (A_r);  B: device bf16 [r][d_out]
 *   row-major (B_r).  At: device bf16 [r][d_in], Bt: device bf16 [d_out][r],
 *   written as the exact transposes (bit-for-bit copies of every element).
 *   d_in, d_out, r positive multiples of 64 (LR_ERR_UNSUPPORTED otherwise);
 *   every pointer 16-byte aligned; the four buffers must not overlap
 *   (LR_ERR_INVALID_ARG).  Enqueued on s; a one-time step when a model's
 *   factors are loaded, not part of a decode step. */
lr_status lr_factor_pack(const void* A, const void* B, int32_t d_in, int32_t d_out, int32_t r, void* At,
                         void* Bt, lr_stream s);

/* Projections of a block, in this order (English page section 2.D: attention
 * and MLP projections are all decomposed). */
enum { LR_Q = 0, LR_K = 1, LR_V = 2, LR_O = 3, LR_GATE = 4, LR_UP = 5, LR_DOWN = 6 };

/* A decomposed LLaMA-style block whose attention core is attention over a
 * one-token context (each query head returns the value vector of its kv head).
 * q: d_model -> n_heads*head_dim, k/v: d_model -> n_kv_heads*head_dim,
 * o: n_heads*head_dim -> d_model, gate/up: d_model -> d_ff, down: d_ff -> d_model.
 * n_heads must be a multiple of n_kv_heads (MHA, GQA, MQA); head_dim a multiple
 * of 64; d_model at most 8192; RMSNorm has unit gain and the given eps.
 * The MLP is SiLU-GLU or, with mlp = LR_MLP_RELU, a non-GLU ReLU MLP. */
/* MLP variants (English page section 2.D: GLU and non-GLU MLPs). */
enum { LR_MLP_SWIGLU = 0, /* h += down(silu(gate(n2)) * up(n2)) (LLaMA) */
       LR_MLP_RELU = 1    /* h += down(relu(up(n2))), gate unused (OPT) */ };

typedef struct {
  int32_t d_model;
  int32_t d_ff;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  float eps;
  lr_factor f[7];
  int32_t mlp;  /* LR_MLP_SWIGLU or LR_MLP_RELU; with LR_MLP_RELU f[LR_GATE] is not read */
} lr_block_desc;

/* ---------------------------------------------------------------------------
 * lr_linear_forward: y = (x A_r) B_r for M rows.
 * English page section 2.A (down projection, then up projection); Spanish
 * page "Resumen Tecnico" section 1 (W ~ A B).
 *   x  device bf16 [M][ldx], ldx >= d_in, ldx multiple of 8, x 16-byte aligned.
 *   y  device [M][ldy] of y_dtype (LR_BF16 or LR_F32), ldy >= d_out.
 *   The intermediate t = x A_r is rounded to bf16 (round to nearest even) and
 *   kept in `workspace`; the sums accumulate in fp32.  A bf16 y is the
 *   round-to-nearest-even image of the fp32 y.
 *   workspace: device, at least lr_linear_workspace_bytes(M, f) bytes, 256-byte
 *   aligned; it holds t (M x r bf16) and, for M > 256, one int32 completion
 *   counter per 256-row band of the one-launch prefill form.  Its contents on
 *   entry do not matter (every element that is read was written, or
 *   cleared, by the same call).  Calls that share a workspace must be
 *   ordered on one stream.
 *   M = 0 is a no-op.  M <= 256 runs the decode kernels, larger M the prefill
 *   kernels (on SM pairs; a linear under 1.5e12 flops runs its down and up
 *   projections in one launch).  The result is deterministic (no
 *   floating-point atomics) and the same whichever form runs. */
size_t lr_linear_workspace_bytes(int64_t M, const lr_factor* f);
lr_status lr_linear_forward(const void* x, int64_t ldx, void* y, int64_t ldy, lr_dtype y_dtype,
                            int64_t M, const lr_factor* f, void* workspace, size_t ws_bytes,
                            int32_t* dev_status, lr_stream s);

/* ---------------------------------------------------------------------------
 * lr_linear_forward_noalloc: the same computation as lr_linear_forward for
 * callers that cannot allocate device memory.  The paper has no counterpart;
 * this is an interface convenience.
 *   Some callers cannot hand the library a workspace: code that runs where
 *   cudaMalloc is forbidden or unwanted (an allocator-free embedded runtime, a
 *   plugin that receives only raw pointers and a stream, a serving loop whose
 *   device memory is fixed at start-up), or code that must not risk the
 *   implicit device synchronisation an allocation can cause.  This entry point
 *   keeps the intermediate t = x A_r in a static device array of
 *   LR_NOALLOC_SCRATCH_BYTES (4 MiB) inside the library instead.  Every GPU
 *   that loads the library holds that array until the process exits.  The
 *   call itself allocates nothing (no cudaMalloc/cudaFree, no allocating
 *   library routine).
 *   Arguments, layouts, checks and results are those of lr_linear_forward
 *   without the workspace.  lr_linear_workspace_bytes(M, f) (about M * r * 2)
 *   must not exceed LR_NOALLOC_SCRATCH_BYTES; larger problems are rejected
 *   with LR_ERR_UNSUPPORTED and a message in lr_last_error().
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   All calls share the one array and it keeps the last call's contents.
 *   Nothing in it needs to start at zero (each call writes every element it
 *   reads).  Calls that overlap on the GPU (on different streams, say) race on
 *   it: order them on one stream. */
#define LR_NOALLOC_SCRATCH_BYTES (4u << 20)
lr_status lr_linear_forward_noalloc(const void* x, int64_t ldx, void* y, int64_t ldy,
                                    lr_dtype y_dtype, int64_t M, const lr_factor* f,
                                    int32_t* dev_status, lr_stream s);

/* ---------------------------------------------------------------------------
 * lr_block_forward: one decomposed block applied in place to the fp32 residual
 * stream h (device fp32 [M][d_model], 16-byte aligned):
 *   n1 = RMSNorm(h); q,k,v = LR(n1); h += LR_o(attn(v));
 *   n2 = RMSNorm(h); h += LR_down(silu(LR_gate(n2)) * LR_up(n2))
 *   (non-GLU: h += LR_down(relu(LR_up(n2)))).
 * Spanish page section 1 (attention and MLP projections decomposed) and
 * section 2 "Generalizacion"; English page section 2.D (MHA/GQA/MQA, GLU MLP).
 * Linear inputs are rounded to bf16.  scratch: device, at least
 * lr_block_scratch_bytes(M, b) bytes, 256-byte aligned; its contents on entry
 * do not matter.  M = 0 is a no-op.  Each linear runs as lr_linear_forward
 * would at the same M (decode kernels up to 256 rows, the SM-pair prefill
 * GEMM above, one launch per linear below 1.5e12 flops); the result does not
 * depend on which form runs. */
size_t lr_block_scratch_bytes(int64_t M, const lr_block_desc* b);
lr_status lr_block_forward(float* h, int64_t M, const lr_block_desc* b, void* scratch,
                           size_t scratch_bytes, int32_t* dev_status, lr_stream s);

/* ---------------------------------------------------------------------------
 * remap_compact: the copy of the preparation stage (English page section 2.C):
 *   buf[i][:] = pool[remap[i]][:] for 0 <= i < min(*n_active, cap), zero rows
 *   for i >= *n_active.  Bit-exact byte copy of row_bytes per row.
 *   pool: device [pool_rows][row_bytes]; buf: device [cap][row_bytes];
 *   remap: device int32 [cap]; n_active: device int32 (read on the device, so
 *   the launch parameters never change with the batch).  row_bytes must be a
 *   positive multiple of 16 and every pointer 16-byte aligned.  An entry
 *   outside [0, pool_rows) gives a zero row and LR_ERR_REMAP_RANGE in
 *   dev_status. */
lr_status remap_compact(const void* pool, int64_t pool_rows, int64_t row_bytes,
                        const int32_t* remap, const int32_t* n_active, void* buf, int64_t cap,
                        int32_t* dev_status, lr_stream s);

/* remap_scatter: the inverse copy, pool[remap[i]][:] = buf[i][:] for
 * 0 <= i < min(*n_active, cap).  Same arguments and checks as remap_compact;
 * an out-of-range entry is skipped and reported.  Targets must be distinct
 * (remap_build makes them so); with duplicates the surviving row is
 * unspecified. */
lr_status remap_scatter(const void* buf, const int32_t* remap, const int32_t* n_active,
                        void* pool, int64_t pool_rows, int64_t row_bytes, int64_t cap,
                        int32_t* dev_status, lr_stream s);

/* remap_build (host only): the scan of the preparation stage (English page
 * section 2.C, "remapping index list (a new block table)").
 *   lengths: host int32 [n_seq]; block_table: host int32 [n_seq][blocks_per_seq],
 *   entry (s, b) = physical block of logical block b of sequence s.
 *   For each sequence in order, its last tail_rows positions (all positions if
 *   tail_rows <= 0) are mapped to physical rows
 *   block_table[s][p / block_rows] * block_rows + p % block_rows.
 *   Outputs (host): remap_out[cap] (unused entries -1), *n_active_out, and
 *   *n_runs_out = number of maximal runs of consecutive physical rows.
 *   LR_ERR_INVALID_ARG if the rows exceed cap, a needed table entry is
 *   negative, a length is negative or exceeds the table, or two rows coincide. */
lr_status remap_build(const int32_t* lengths, int64_t n_seq, const int32_t* block_table,
                      int32_t blocks_per_seq, int32_t block_rows, int32_t tail_rows, int64_t cap,
                      int32_t* remap_out, int32_t* n_active_out, int32_t* n_runs_out);

/* ---------------------------------------------------------------------------
 * lr_kv_reconstruct: the reconstruction of a low-rank KV cache under a static
 * graph (English page section 2.C: scattered latent rows are listed by a
 * remap table, copied into a contiguous buffer, and "the contiguous buffer is
 * multiplied by the upward projection matrices to reconstruct the KV cache"
 * in one large fixed-size GEMM; the latent KV grows with the context, English
 * page section 1).
 *   latent_buf[i][:] = latent_pool[remap[i]][:] for i < *n_active, zero rows
 *   otherwise (as remap_compact), then out = latent_buf Bt^T, i.e.
 *   out[i][n] = sum_j latent_buf[i][j] * B_r[j][n].
 *   latent_pool: device bf16 [pool_rows][r]; latent_buf: device bf16 [cap][r];
 *   Bt: device bf16 [d_kv][r] (the up factor transposed); out: device bf16
 *   [cap][d_kv].  r and d_kv positive multiples of 64, pointers 16-byte
 *   aligned.  Rows past *n_active come out zero.  cap and every pointer are
 *   fixed, so the two launches can be captured once and replayed per step.
 *   Out-of-range remap entries give zero rows and LR_ERR_REMAP_RANGE. */
lr_status lr_kv_reconstruct(const void* latent_pool, int64_t pool_rows, int32_t r,
                            const int32_t* remap, const int32_t* n_active, int64_t cap,
                            void* latent_buf, const void* Bt, int32_t d_kv, void* out,
                            int32_t* dev_status, lr_stream s);

/* ---------------------------------------------------------------------------
 * The block-granular form of the same reconstruction: the remap lists whole
 * paged blocks (the pages' "new block table", English page section 2.C), and
 * the up-projection GEMM reads each listed block straight from the latent
 * pool -- no compacted copy is written or read back.
 *
 * remap_build_blocks (host only): for each sequence in order, the physical
 * blocks that hold its positions 0 .. L-1 (the first ceil(L / block_rows)
 * entries of its block-table row).
 *   lengths: host int32 [n_seq]; block_table: host int32 [n_seq][blocks_per_seq].
 *   Outputs (host): blocks_out[cap_blocks] (unused entries -1), *n_blocks_out,
 *   *n_runs_out = maximal runs of consecutive block ids.
 *   LR_ERR_INVALID_ARG if the blocks exceed cap_blocks, a needed entry is
 *   negative, a length does not fit its table row, or a block is listed twice.
 *   Position p of sequence s sits at row block_rows * i + p % block_rows of
 *   the reconstruction, i being the list index of its block. */
lr_status remap_build_blocks(const int32_t* lengths, int64_t n_seq, const int32_t* block_table,
                             int32_t blocks_per_seq, int32_t block_rows, int64_t cap_blocks,
                             int32_t* blocks_out, int32_t* n_blocks_out, int32_t* n_runs_out);

/* lr_kv_latent_write: the producer side of the low-rank KV cache (English
 * page section 1: the latent KV grows with the context; section 2.C: it is
 * kept in paged memory).  The down projection of k or v for M new tokens is
 * written straight into their rows of the paged latent pool:
 *   latent_pool[rows[m]][:] = bf16(x[m] A_r)   for m < M,
 * summed in fp32 and rounded to nearest even, with A_r given transposed as
 * At [r][d_in].  x: device bf16 [M][ldx]; rows: device int32 [M] (for one new
 * token per sequence, remap_build with tail_rows = 1 on the grown lengths);
 * latent_pool: device bf16 [pool_rows][r].  d_in, r positive multiples of 64;
 * pointers 16-byte aligned, ldx >= d_in and a multiple of 8.  Entries of rows
 * outside [0, pool_rows) are skipped and reported as LR_ERR_REMAP_RANGE;
 * rows must be distinct.  Other pool rows are not touched.  The values are
 * those the down launch of lr_linear_forward writes for t.  M = 0 is a
 * no-op. */
lr_status lr_kv_latent_write(const void* x, int64_t ldx, int64_t M, const void* At, int32_t d_in, int32_t r,
                             const int32_t* rows, void* latent_pool, int64_t pool_rows, int32_t* dev_status,
                             lr_stream s);

/* lr_kv_reconstruct_paged: with 16-row blocks,
 *   out[16 i + j][n] = sum_c latent_pool[16 blocks[i] + j][c] * B_r[c][n]
 * for i < *n_blocks and j < 16; rows of blocks i >= *n_blocks are zero.
 *   latent_pool: device bf16 [pool_blocks * 16][r]; blocks: device int32
 *   [cap_blocks]; n_blocks: device int32 (read on the device, so a captured
 *   graph serves every batch); Bt: device bf16 [d_kv][r]; out: device bf16
 *   [cap_blocks * 16][d_kv].  r and d_kv positive multiples of 64; pointers
 *   16-byte aligned.  A listed block outside [0, pool_blocks) reads as zeros
 *   and reports LR_ERR_REMAP_RANGE.  The rows past a sequence's length in its
 *   last block are reconstructed from whatever the pool holds there; the
 *   caller ignores them.  One launch. */
lr_status lr_kv_reconstruct_paged(const void* latent_pool, int64_t pool_blocks, int32_t r, const int32_t* blocks,
                                  const int32_t* n_blocks, int64_t cap_blocks, const void* Bt, int32_t d_kv,
                                  void* out, int32_t* dev_status, lr_stream s);

/* ---------------------------------------------------------------------------
 * Rank-space sharding of one factorized linear, simulated on this GPU (English
 * page section 2.A, "Highly Efficient Low-Rank Communication": the down
 * projection is split by columns and its output all-gathered in the low-rank
 * space; the up projection runs in shard mode, with no reduce-sum).
 *
 * The rank columns are split over G simulated processes in blocks of 64: process g
 * owns rank columns R_g = [64*floor(g*nr/G), 64*floor((g+1)*nr/G)) with
 * nr = r/64, and output columns O_g likewise over d_out/64 blocks.  Then
 *   1. down, per process:  t_g = x A_r[:, R_g]   into process g's own buffer
 *      (bf16 [M][|R_g|], the rows R_g of At);
 *   2. all-gather in rank space, emulated by device-to-device copies of every
 *      t_g into the columns R_g of one gathered t (bf16 [M][r]);
 *   3. up, shard mode, per process:  y[:, O_g] = t B_r[:, O_g]  (the rows O_g
 *      of Bt), written straight into the caller's y.
 * Every launch is issued on `s`, one process after another.  y equals
 * lr_linear_forward's result up to the fp32 summation order of the split GEMMs.
 * Arguments and checks as lr_linear_forward, plus 1 <= n_shards <= r/64 and
 * n_shards <= d_out/64 (else LR_ERR_INVALID_ARG); the workspace (device,
 * 256-byte aligned, caller-owned) holds the G process buffers and the
 * gathered t: lr_rank_sharded_workspace_bytes bytes.  M == 0 is a no-op. */
size_t lr_rank_sharded_workspace_bytes(int64_t M, const lr_factor* f, int32_t n_shards);
lr_status lr_linear_forward_rank_sharded(const void* x, int64_t ldx, void* y, int64_t ldy,
                                         lr_dtype y_dtype, int64_t M, const lr_factor* f,
                                         int32_t n_shards, void* workspace, size_t ws_bytes,
                                         int32_t* dev_status, lr_stream s);

/* lr_rank_shard_comm_bytes (host only): collective bytes that the busiest of
 * the G processes receives for one factorized linear, with the column split
 * above and elements of elem_bytes bytes:
 *   *rank_space = (r - min_g |R_g|) * M * elem_bytes    (ring all-gather of t,
 *                 the low-rank scheme);
 *   *full_space = 2 (d_out - min_g |O_g|) * M * elem_bytes  (ring all-reduce of
 *                 y, i.e. reduce-scatter then all-gather: the reduce-sum in the
 *                 full dimension that a naive split of the two factors needs).
 * LR_ERR_INVALID_ARG on a negative M, non-positive sizes, r or d_out not a
 * multiple of 64, or n_shards outside [1, min(r, d_out)/64]. */
lr_status lr_rank_shard_comm_bytes(int64_t M, int32_t d_out, int32_t r, int32_t n_shards,
                                   int32_t elem_bytes, int64_t* rank_space, int64_t* full_space);

/* ---------------------------------------------------------------------------
 * A decode step of a layer stack over fixed buffers (English page section 2.C:
 * addresses and launch parameters stay fixed while the logical batch changes):
 *   xbuf = remap_compact(pool_in); h = widen(xbuf); for each layer:
 *   lr_block_forward(h, cap rows); ybuf = bf16(h); remap_scatter(ybuf -> pool_out).
 * pool_in/pool_out: device bf16 [pool_rows][d_model] (may be the same buffer);
 * xbuf/ybuf: device bf16 [cap][d_model]; h: device fp32 [cap][d_model];
 * scratch: max over layers of lr_block_scratch_bytes(cap, layer).
 * All layers must share d_model.  Rows i >= *n_active run through the layers
 * as zero rows and are not scattered. */
enum { LR_STACK_AUTO = 0, LR_STACK_LAYERED = 1 };
typedef struct {
  int32_t n_layers;
  const lr_block_desc* layers; /* host array [n_layers]; copied by the calls */
  const void* pool_in;
  void* pool_out;
  int64_t pool_rows;
  const int32_t* remap;
  const int32_t* n_active;
  int64_t cap;
  void* xbuf;
  float* h;
  void* ybuf;
  void* scratch;
  size_t scratch_bytes;
  int32_t* dev_status;
  /* LR_STACK_AUTO (= LR_STACK_LAYERED): one launch per kernel, chained by
   * programmatic dependent launch.  Other values are rejected
   * (LR_ERR_INVALID_ARG). */
  int32_t mode;
} lr_stack_desc;

/* Scratch the step needs: the block buffers of the largest layer (layers run
 * one after another and reuse them).  Uses only n_layers, layers and cap of
 * the descriptor.  A captured graph keeps using its scratch until
 * lr_graph_destroy. */
size_t lr_stack_scratch_bytes(const lr_stack_desc* st);

/* Enqueue one step eagerly on stream s. */
lr_status lr_stack_forward(const lr_stack_desc* st, lr_stream s);

/* Capture one step into a CUDA graph owned by the library (captured on a
 * private stream; the caller's streams are not touched).  The graph keeps the
 * descriptor's device pointers: they must stay valid until lr_graph_destroy.
 * Per step only the contents of remap, *n_active and the pool change. */
typedef struct lr_graph lr_graph;
lr_status lr_graph_capture(const lr_stack_desc* st, lr_graph** out);
lr_status lr_graph_replay(lr_graph* g, lr_stream s);
lr_status lr_graph_destroy(lr_graph* g);

/* Number of kernel launches one step enqueues (eager or in the graph). */
int64_t lr_stack_launch_count(const lr_stack_desc* st);

const char* lr_status_string(lr_status st);
const char* lr_last_error(void);

/* ---------------------------------------------------------------------------
 * Testing hook (no counterpart on the pages).  lr_test_stall_producer(1) makes
 * the TMA producers of every decode-size GEMM and every SM-pair prefill GEMM
 * launched afterwards issue no copy, so the bounded wait of the thread that
 * consumes the copies runs out:
 * the launch reports LR_ERR_TIMEOUT through dev_status (after about two
 * seconds), releases its resources and returns, and the context stays usable.
 * lr_test_stall_producer(0) restores normal launches.  It exists for the
 * failure-detection tests only; nothing else sets it, and no environment
 * variable does. */
void lr_test_stall_producer(int32_t on);

/* Testing hook (no counterpart on the pages).  Prefill-size GEMMs (M > 256)
 * take their 256-row bands in groups, all of a group's bands for one weight
 * tile before the next; a prefill-size linear runs its down and up
 * projections in one launch, the up-projection tiles of each group placed a
 * number of groups (the lag) after that group's down-projection tiles and
 * waiting for them.  lr_test_prefill_schedule(lag, group) fixes the lag (at
 * most the number of groups) and the bands per group of later launches;
 * 0 restores the automatic choice of either, and a negative lag runs the two
 * projections as two launches.  It exists so tests can make
 * the up projection wait and vary the order of the tiles; results do not
 * depend on it.  Nothing else sets it, and no environment variable does. */
void lr_test_prefill_schedule(int32_t lag, int32_t group);


#ifdef __cplusplus
}
#endif
#endif /* LR_H_ */
