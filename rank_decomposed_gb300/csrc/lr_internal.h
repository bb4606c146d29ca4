// Internal declarations shared by the translation units of liblr.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>


#include "../../include/lr.h"

namespace lr {

// Every bounded wait inside a kernel gives up after this long.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Largest number of problems one grouped decode launch carries.
constexpr int kMaxGroup = 3;

// Decode (swap-AB) kernels take at most this many rows.
constexpr int kDecodeMaxRows = 256;

// Largest cluster used for the split-K reduction of the decode kernel.
constexpr int kMaxCluster = 16;

// What a GEMM does with each finished fp32 output element v at (m, n).
enum Epilogue : int32_t {
  EPI_STORE_BF16 = 0,  // out_bf16[m*ldo + n] = rne(v)
  EPI_STORE_F32 = 1,   // out_f32[m*ldo + n] = v
  EPI_ADD_F32 = 2,     // out_f32[m*ldo + n] += v   (residual stream)
  EPI_RELU_BF16 = 3,   // out_bf16[m*ldo + n] = rne(max(v, 0))   (non-GLU MLP)
};

__host__ __device__ inline bool epi_is_bf16(int32_t epi) {
  return epi == EPI_STORE_BF16 || epi == EPI_RELU_BF16;
}

// One problem of a GEMM launch:  out[m][n] = sum_k act[m][k] * W[n][k]
// for m < M, n < N, k < K (K a multiple of 64).  W and act are bf16.
struct GemmOp {
  const void* W;        // [N][ldw]
  int32_t N;
  int32_t K;
  int64_t ldw;
  const void* act;      // [M][ld_act]
  int64_t ld_act;
  int64_t act_cols;     // columns of the act buffer (differs from K under GQA)
  int32_t gqa_head_dim; // 0: act column = k.  Otherwise the act buffer holds
  int32_t gqa_group;    //   kv heads and column k reads kv head (k/hd)/group.
  int32_t epi;
  void* out;
  int64_t ldo;
  // Output row of activation row m: m, or out_rows[m] when given (entries
  // outside [0, out_rows_limit) are skipped and reported as LR_ERR_REMAP_RANGE).
  const int32_t* out_rows;
  int64_t out_rows_limit;
};

// --------------------------------------------------- device-side parameters
struct DecodeProblem {
  int32_t N;
  int32_t nkb;          // K / 64
  int32_t n_tiles;      // ceil(N / 128)
  int32_t item_begin;   // first CTA index of this problem
  int32_t gqa_head_dim;
  int32_t gqa_group;
  int32_t epi;
  int32_t vec_ok;       // out 16-byte aligned and ldo % 8 == 0: vector stores
  void* out;
  int64_t ldo;
  const int32_t* out_rows;  // see GemmOp
  int64_t out_rows_limit;
  int32_t* status;
};

struct DecodeParams {
  int32_t M;            // valid rows (tokens), 1..256
  int32_t n_problems;
  int32_t splits;       // K splits per tile == cluster size
  int32_t stall_producer;  // fault-injection hook: the TMA producer issues nothing
  int32_t prefetch;     // weight stages requested before waiting for the previous kernel
  int32_t* status;
  DecodeProblem prob[kMaxGroup];
};

struct DecodeMaps {
  CUtensorMap w[kMaxGroup];
  CUtensorMap a[kMaxGroup];
};

struct PrefillParams {
  int32_t M, N, K;
  int32_t m_tiles, n_tiles;
  int32_t epi;
  int32_t gqa_head_dim, gqa_group;
  void* out;
  int64_t ldo;
  int32_t* status;
  // Paged activations (blocks != nullptr): activation row 16 i + j is row j of
  // block blocks[i] of a paged pool of pool_blocks 16-row blocks, for
  // i < *n_blocks; later rows, and entries outside the pool, read as zeros
  // (the latter also report LR_ERR_REMAP_RANGE).
  const int32_t* blocks;
  const int32_t* n_blocks;
  int64_t pool_blocks;
  // Output row of activation row m (see GemmOp).
  const int32_t* out_rows;
  int64_t out_rows_limit;
};

// Rows of a block of the paged latent pool.
constexpr int kPageRows = 16;

// ------------------------------------------------------------- host helpers
void set_error(const char* fmt, ...);
lr_status cuda_fail(cudaError_t e, const char* what);

// Argument checks of a factor pair: LR_ERR_INVALID_ARG for null or misaligned
// pointers and non-positive sizes, LR_ERR_UNSUPPORTED for sizes that are not
// multiples of 64.  `name` prefixes the message.
lr_status check_factor(const lr_factor* f, const char* name);
// Checks of a linear's x / y arguments (pointers, dtype, leading dimensions,
// alignment) for M > 0 rows.
lr_status check_linear_io(const char* who, const void* x, int64_t ldx, const void* y, int64_t ldy,
                          lr_dtype y_dtype, int64_t M, const lr_factor* f);
GemmOp make_op(const void* W, int N, int K, const void* act, int64_t ld_act, int64_t act_cols,
               int epi, void* out, int64_t ldo);
// Ops sharing M: one grouped launch at decode sizes, one launch per op above.
lr_status run_ops(int64_t M, const GemmOp* ops, int n, int32_t* status, cudaStream_t s);
// y = (x A_r) B_r with t (bf16 [M][r]) at `t`: the down then the up launch.
// Arguments already checked.
lr_status enqueue_linear(const void* x, int64_t ldx, void* y, int64_t ldy, lr_dtype y_dtype,
                         int64_t M, const lr_factor* f, void* t, int32_t* status, cudaStream_t s);

// Tensor map over a bf16 row-major [rows][cols] matrix with row stride ld
// (elements), box = box_rows x 64 columns, 128-byte swizzle, zero fill
// outside the matrix.
lr_status encode_map_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint64_t ld, uint32_t box_rows);

int num_sms();

// Launchers (lr_decode.cu, lr_prefill.cu, lr_glue.cu).  They assume their
// arguments were validated by the caller.
lr_status launch_decode(int M, const GemmOp* ops, int n_ops, int32_t* status, cudaStream_t s);

lr_status launch_prefill(int64_t M, const GemmOp& op, int32_t* status, cudaStream_t s);
// The same GEMM on SM pairs (tcgen05 cta_group::2, 256 x 256 tiles).
lr_status launch_prefill_pair(int64_t M, const GemmOp& op, int32_t* status, cudaStream_t s);
// A prefill-size factorized linear in one launch on SM pairs: down (writes
// T) and up (reads T) with band-ordered tiles.  band_done: device int32
// [ceil(M / 256)], cleared by the call.
lr_status launch_prefill_pair_fused(int64_t M, const GemmOp& down, const GemmOp& up, int32_t* band_done,
                                    int32_t* status, cudaStream_t s);
size_t prefill_band_counter_bytes(int64_t M);
// Whether a linear of M rows with these down/up GEMMs runs as one fused
// launch (prefill sizes only).
bool prefill_fuse_linear(int64_t M, const GemmOp& down, const GemmOp& up);
// Whether prefill-size GEMMs run on SM pairs (LR_PREFILL_PAIR=0 turns it
// off) and whether a prefill-size linear is one fused launch
// (LR_PREFILL_FUSED=0 turns it off); both read once.
bool prefill_pair_enabled();
bool prefill_fused_enabled();
// Lag and band group fixed by lr_test_prefill_schedule (0: automatic).
int test_prefill_lag();
int test_prefill_group();
// The same GEMM with its activation rows read from a paged pool through a
// block list (see PrefillParams); op.act is the pool, op.ld_act its row
// stride, M = cap_blocks * 16.
lr_status launch_prefill_paged(int64_t M, const GemmOp& op, const int32_t* blocks, const int32_t* n_blocks,
                               int64_t pool_blocks, int32_t* status, cudaStream_t s);
lr_status launch_rmsnorm(const float* h, void* out_bf16, int64_t M, int d, float eps,
                         cudaStream_t s);
lr_status launch_silu_mul(const void* g, const void* u, void* out, int64_t M, int d,
                          cudaStream_t s);
lr_status launch_widen(const void* in_bf16, float* out, int64_t n, cudaStream_t s);
// out = in^T for bf16 [rows][cols], rows and cols multiples of 64.
lr_status launch_transpose_bf16(const void* in, int rows, int cols, void* out, cudaStream_t s);
lr_status launch_narrow(const float* in, void* out_bf16, int64_t n, cudaStream_t s);
// Stack glue, one CTA per row: gather + widen, and narrow + scatter.
lr_status launch_gather_rows(const void* pool, int64_t pool_rows, int d, const int32_t* remap,
                             const int32_t* n_active, void* xbuf, float* h, int64_t cap,
                             int32_t* status, cudaStream_t s);
lr_status launch_scatter_rows(const float* h, void* ybuf, const int32_t* remap,
                              const int32_t* n_active, void* pool, int64_t pool_rows, int d,
                              int64_t cap, int32_t* status, cudaStream_t s);
lr_status launch_gather(const void* pool, int64_t pool_rows, int64_t row_bytes,
                        const int32_t* remap, const int32_t* n_active, void* buf, int64_t cap,
                        int32_t* status, cudaStream_t s);
lr_status launch_scatter(const void* buf, const int32_t* remap, const int32_t* n_active,
                         void* pool, int64_t pool_rows, int64_t row_bytes, int64_t cap,
                         int32_t* status, cudaStream_t s);

// Kernel attributes (dynamic shared memory, cluster size) of the current
// device; done once per device before the first launch or capture.
lr_status configure_decode();
lr_status configure_prefill();
// A bf16 [rows][cols] matrix viewed as [cols / 64][rows][64]: one box of
// {64, box_rows, box_chunks} loads box_chunks consecutive k-blocks.
lr_status encode_map_bf16_chunks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                 uint64_t ld, uint32_t box_rows, uint32_t box_chunks);
lr_status configure_prefill_pair();
lr_status ensure_configured();

// Buffers of one block inside its scratch (offsets in bytes, 256-aligned).
struct BlockLayout {
  size_t n1, t[7], q, k, v, n2, g, u, a, cnt, total;  // cnt: prefill band counters
};
BlockLayout block_layout(int64_t M, const lr_block_desc* b);

// Launch attribute helper: programmatic dependent launch on/off for kernels
// enqueued by this library (on by default).
bool pdl_enabled();

// Fault-injection hook of the bounded-wait tests (lr_test_stall_producer):
// while set, the decode kernels' weight producers issue no copy.
bool test_stall_producer();

}  // namespace lr
