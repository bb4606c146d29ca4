// Host side of liblr: argument validation, tensor-map encoding, the order of
// kernels inside a decomposed linear, a block and a layer stack, the remap
// scan, and CUDA-graph capture/replay.  See include/lr.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "lr_internal.h"

namespace lr {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

lr_status cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  return LR_ERR_CUDA;
}

static lr_status invalid_device() {
  set_error("device ordinal outside the supported range");
  return LR_ERR_UNSUPPORTED;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

static std::atomic<int> g_stall_producer{0};

bool test_stall_producer() { return g_stall_producer.load(std::memory_order_relaxed) != 0; }

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("LR_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

static std::atomic<int> g_prefill_lag{0};
static std::atomic<int> g_prefill_group{0};

int test_prefill_lag() { return g_prefill_lag.load(std::memory_order_relaxed); }
int test_prefill_group() { return g_prefill_group.load(std::memory_order_relaxed); }

bool prefill_pair_enabled() {
  static const bool on = [] {
    const char* v = getenv("LR_PREFILL_PAIR");
    return !(v && v[0] == '0');
  }();
  return on;
}

bool prefill_fused_enabled() {
  static const bool on = [] {
    const char* v = getenv("LR_PREFILL_FUSED");
    return prefill_pair_enabled() && !(v && v[0] == '0');
  }();
  return on && g_prefill_lag.load(std::memory_order_relaxed) >= 0;
}

// cuTensorMapEncodeTiled, looked up once through the runtime so the library
// needs no link-time dependency on the driver library.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

lr_status encode_map_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint64_t ld, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    set_error("cuTensorMapEncodeTiled unavailable");
    return LR_ERR_CUDA;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d): rows=%llu cols=%llu ld=%llu box_rows=%u",
              static_cast<int>(r), (unsigned long long)rows, (unsigned long long)cols,
              (unsigned long long)ld, box_rows);
    return LR_ERR_CUDA;
  }
  return LR_OK;
}

// A 3-D view of a bf16 [rows][cols] matrix whose columns are cut into chunks
// of 64 (cols a multiple of 64): element (c, r, z) is [r][64 z + c].  A box of
// {64, box_rows, box_chunks} then lands in shared memory as box_chunks
// consecutive 128-byte-swizzled [box_rows][64] tiles: several k-blocks of a
// K-major operand in one TMA operation.
lr_status encode_map_bf16_chunks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                 uint64_t ld, uint32_t box_rows, uint32_t box_chunks) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    set_error("cuTensorMapEncodeTiled unavailable");
    return LR_ERR_CUDA;
  }
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {ld * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (3-D) failed (%d): rows=%llu cols=%llu ld=%llu box_rows=%u",
              static_cast<int>(r), (unsigned long long)rows, (unsigned long long)cols,
              (unsigned long long)ld, box_rows);
    return LR_ERR_CUDA;
  }
  return LR_OK;
}

lr_status ensure_configured() {
  static bool done[64] = {false};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return invalid_device();
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return LR_OK;
  lr_status st = configure_decode();
  if (st != LR_OK) return st;
  st = configure_prefill();
  if (st != LR_OK) return st;
  st = configure_prefill_pair();
  if (st != LR_OK) return st;
  done[dev] = true;
  return LR_OK;
}

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lr_status invalid(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return LR_ERR_INVALID_ARG;
}

}  // namespace

lr_status check_factor(const lr_factor* f, const char* name) {
  if (f == nullptr) return invalid("%s: null factor", name);
  if (f->d_in <= 0 || f->d_out <= 0 || f->r <= 0) return invalid("%s: non-positive dims", name);
  if (f->d_in % 64 || f->d_out % 64 || f->r % 64) {
    set_error("%s: d_in=%d d_out=%d r=%d must be multiples of 64", name, f->d_in, f->d_out, f->r);
    return LR_ERR_UNSUPPORTED;
  }
  if (f->At == nullptr || f->Bt == nullptr) return invalid("%s: null factor pointer", name);
  if (!aligned16(f->At) || !aligned16(f->Bt)) return invalid("%s: factors not 16-byte aligned", name);
  return LR_OK;
}

GemmOp make_op(const void* W, int N, int K, const void* act, int64_t ld_act, int64_t act_cols,
               int epi, void* out, int64_t ldo) {
  GemmOp o;
  memset(&o, 0, sizeof(o));
  o.W = W;
  o.N = N;
  o.K = K;
  o.ldw = K;
  o.act = act;
  o.ld_act = ld_act;
  o.act_cols = act_cols;
  o.epi = epi;
  o.out = out;
  o.ldo = ldo;
  return o;
}

// Run a group of ops that share M: one grouped launch for decode sizes, one
// launch per op for prefill sizes.
lr_status run_ops(int64_t M, const GemmOp* ops, int n, int32_t* status, cudaStream_t s) {
  lr_status cst = ensure_configured();
  if (cst != LR_OK) return cst;
  if (M <= kDecodeMaxRows) return launch_decode(static_cast<int>(M), ops, n, status, s);
  for (int i = 0; i < n; ++i) {
    lr_status st = prefill_pair_enabled() ? launch_prefill_pair(M, ops[i], status, s)
                                          : launch_prefill(M, ops[i], status, s);
    if (st != LR_OK) return st;
  }
  return LR_OK;
}

lr_status check_linear_io(const char* who, const void* x, int64_t ldx, const void* y, int64_t ldy,
                          lr_dtype y_dtype, int64_t M, const lr_factor* f) {
  if (x == nullptr || y == nullptr) return invalid("%s: null pointer", who);
  if (y_dtype != LR_BF16 && y_dtype != LR_F32) return invalid("%s: bad y dtype", who);
  if (ldx < f->d_in || ldx % 8 || !aligned16(x))
    return invalid("%s: x must be 16-byte aligned with ldx >= d_in, ldx %% 8 == 0", who);
  if (ldy < f->d_out) return invalid("%s: ldy < d_out", who);
  if (M > kDecodeMaxRows && (!aligned16(y) || ldy % 8))
    return invalid("%s: y must be 16-byte aligned with ldy %% 8 == 0", who);
  return LR_OK;
}

lr_status enqueue_linear(const void* x, int64_t ldx, void* y, int64_t ldy, lr_dtype y_dtype,
                         int64_t M, const lr_factor* f, void* t, int32_t* status, cudaStream_t s) {
  GemmOp down = make_op(f->At, f->r, f->d_in, x, ldx, f->d_in, EPI_STORE_BF16, t, f->r);
  GemmOp up = make_op(f->Bt, f->d_out, f->r, t, f->r, f->r,
                      y_dtype == LR_BF16 ? EPI_STORE_BF16 : EPI_STORE_F32, y, ldy);
  if (prefill_fuse_linear(M, down, up)) {
    lr_status cst = ensure_configured();
    if (cst != LR_OK) return cst;
    int32_t* cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(t) +
                                              align_up(static_cast<size_t>(M) * static_cast<size_t>(f->r) * 2));
    return launch_prefill_pair_fused(M, down, up, cnt, status, s);
  }
  lr_status st = run_ops(M, &down, 1, status, s);
  if (st != LR_OK) return st;
  return run_ops(M, &up, 1, status, s);
}

// ---------------------------------------------------------------- block
BlockLayout block_layout(int64_t M, const lr_block_desc* b) {
  BlockLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align_up(bytes);
    return o;
  };
  const size_t m = static_cast<size_t>(M);
  L.n1 = take(m * b->d_model * 2);
  for (int i = 0; i < 7; ++i) {
    const bool unused = (i == LR_GATE && b->mlp == LR_MLP_RELU);
    L.t[i] = take(unused ? 0 : m * b->f[i].r * 2);
  }
  L.q = take(m * b->f[LR_Q].d_out * 2);
  L.k = take(m * b->f[LR_K].d_out * 2);
  L.v = take(m * b->f[LR_V].d_out * 2);
  L.n2 = take(m * b->d_model * 2);
  L.g = take(m * b->d_ff * 2);
  L.u = take(m * b->d_ff * 2);
  L.a = take(m * b->d_ff * 2);
  L.cnt = take(M > kDecodeMaxRows ? prefill_band_counter_bytes(M) : 0);
  L.total = off;
  return L;
}

namespace {

lr_status check_block(const lr_block_desc* b) {
  if (b == nullptr) return invalid("block: null descriptor");
  static const char* names[7] = {"q", "k", "v", "o", "gate", "up", "down"};
  if (b->mlp != LR_MLP_SWIGLU && b->mlp != LR_MLP_RELU) return invalid("block: bad mlp variant");
  for (int i = 0; i < 7; ++i) {
    if (i == LR_GATE && b->mlp == LR_MLP_RELU) continue;  // not read
    lr_status st = check_factor(&b->f[i], names[i]);
    if (st != LR_OK) return st;
  }
  const int d = b->d_model, dff = b->d_ff, hd = b->head_dim;
  if (d <= 0 || dff <= 0 || hd <= 0 || b->n_heads <= 0 || b->n_kv_heads <= 0)
    return invalid("block: non-positive shape");
  if (b->n_heads % b->n_kv_heads) return invalid("block: n_heads %% n_kv_heads != 0");
  if (hd % 64 || d % 64 || dff % 64) {
    set_error("block: d_model, d_ff and head_dim must be multiples of 64");
    return LR_ERR_UNSUPPORTED;
  }
  if (d > 8192) {
    set_error("block: d_model above 8192 is not supported (RMSNorm keeps a row in registers)");
    return LR_ERR_UNSUPPORTED;
  }
  if (!(b->eps >= 0.f)) return invalid("block: eps must be >= 0");
  const int dq = b->n_heads * hd, dkv = b->n_kv_heads * hd;
  const int want[7][2] = {{d, dq}, {d, dkv}, {d, dkv}, {dq, d}, {d, dff}, {d, dff}, {dff, d}};
  for (int i = 0; i < 7; ++i)
    if (!(i == LR_GATE && b->mlp == LR_MLP_RELU) &&
        (b->f[i].d_in != want[i][0] || b->f[i].d_out != want[i][1]))
      return invalid("block: factor %s is %dx%d, expected %dx%d", names[i], b->f[i].d_in,
                     b->f[i].d_out, want[i][0], want[i][1]);
  return LR_OK;
}

// One launch of a block, in stream order: a GEMM group (ops sharing M and
// their input), an RMSNorm or a SiLU-GLU.
struct Step {
  enum Kind { GEMM, RMSNORM, SILU } kind;
  GemmOp ops[kMaxGroup];
  int n = 0;
  const void* src0 = nullptr;
  const void* src1 = nullptr;
  void* dst = nullptr;
  int d = 0;
  float eps = 0.f;
  int32_t* cnt = nullptr;  // GEMM: band counters for a fused prefill-size linear
};

Step gemm_step(std::initializer_list<GemmOp> ops) {
  Step st;
  st.kind = Step::GEMM;
  for (const GemmOp& o : ops) st.ops[st.n++] = o;
  return st;
}

// The launches of one block: n1 = RMSNorm(h); q, k, v = LR(n1) (down group,
// then up group); h += LR_o(attn(v)); n2 = RMSNorm(h);
// h += LR_down(silu(LR_gate(n2)) * LR_up(n2)) (ReLU variant: the ReLU is
// applied in the up projection's epilogue).
void block_steps_of(float* h, int64_t M, const lr_block_desc* b, uint8_t* ws, std::vector<Step>& out) {
  const BlockLayout L = block_layout(M, b);
  const int d = b->d_model, dff = b->d_ff;
  const lr_factor* f = b->f;
  void* t[7];
  for (int i = 0; i < 7; ++i) t[i] = ws + L.t[i];
  Step norm;
  norm.kind = Step::RMSNORM;
  norm.src0 = h;
  norm.dst = ws + L.n1;
  norm.d = d;
  norm.eps = b->eps;
  out.push_back(norm);
  {
    void* outs[3] = {ws + L.q, ws + L.k, ws + L.v};
    Step dn, up;
    dn.kind = up.kind = Step::GEMM;
    for (int i = 0; i < 3; ++i) {
      dn.ops[i] = make_op(f[i].At, f[i].r, d, ws + L.n1, d, d, EPI_STORE_BF16, t[i], f[i].r);
      up.ops[i] = make_op(f[i].Bt, f[i].d_out, f[i].r, t[i], f[i].r, f[i].r, EPI_STORE_BF16, outs[i],
                          f[i].d_out);
    }
    dn.n = up.n = 3;
    out.push_back(dn);
    out.push_back(up);
  }
  {
    const int dq = b->n_heads * b->head_dim, dkv = b->n_kv_heads * b->head_dim;
    GemmOp od = make_op(f[LR_O].At, f[LR_O].r, dq, ws + L.v, dkv, dkv, EPI_STORE_BF16, t[LR_O],
                        f[LR_O].r);
    if (b->n_heads != b->n_kv_heads) {
      od.gqa_head_dim = b->head_dim;
      od.gqa_group = b->n_heads / b->n_kv_heads;
    }
    out.push_back(gemm_step({od}));
    out.push_back(gemm_step(
        {make_op(f[LR_O].Bt, d, f[LR_O].r, t[LR_O], f[LR_O].r, f[LR_O].r, EPI_ADD_F32, h, d)}));
  }
  norm.dst = ws + L.n2;
  out.push_back(norm);
  if (b->mlp == LR_MLP_SWIGLU) {
    void* outs[2] = {ws + L.g, ws + L.u};
    Step dn, up;
    dn.kind = up.kind = Step::GEMM;
    for (int i = 0; i < 2; ++i) {
      const lr_factor& fi = f[LR_GATE + i];
      dn.ops[i] = make_op(fi.At, fi.r, d, ws + L.n2, d, d, EPI_STORE_BF16, t[LR_GATE + i], fi.r);
      up.ops[i] = make_op(fi.Bt, dff, fi.r, t[LR_GATE + i], fi.r, fi.r, EPI_STORE_BF16, outs[i], dff);
    }
    dn.n = up.n = 2;
    out.push_back(dn);
    out.push_back(up);
    Step act;
    act.kind = Step::SILU;
    act.src0 = ws + L.g;
    act.src1 = ws + L.u;
    act.dst = ws + L.a;
    act.d = dff;
    out.push_back(act);
  } else {
    const lr_factor& fu = f[LR_UP];
    out.push_back(gemm_step({make_op(fu.At, fu.r, d, ws + L.n2, d, d, EPI_STORE_BF16, t[LR_UP], fu.r)}));
    out.push_back(gemm_step({make_op(fu.Bt, dff, fu.r, t[LR_UP], fu.r, fu.r, EPI_RELU_BF16, ws + L.a, dff)}));
  }
  const lr_factor& fd = f[LR_DOWN];
  out.push_back(gemm_step({make_op(fd.At, fd.r, dff, ws + L.a, dff, dff, EPI_STORE_BF16, t[LR_DOWN], fd.r)}));
  out.push_back(gemm_step({make_op(fd.Bt, d, fd.r, t[LR_DOWN], fd.r, fd.r, EPI_ADD_F32, h, d)}));
}

void block_steps(float* h, int64_t M, const lr_block_desc* b, uint8_t* ws, std::vector<Step>& out) {
  const size_t first = out.size();
  block_steps_of(h, M, b, ws, out);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + block_layout(M, b).cnt);
  for (size_t i = first; i < out.size(); ++i) out[i].cnt = cnt;
}

// A GEMM step followed by the GEMM step that reads each of its outputs as
// activations: the down and up projections of the same linears.
bool down_up_pair(const Step& a, const Step& b) {
  if (a.kind != Step::GEMM || b.kind != Step::GEMM || a.n != b.n || a.cnt == nullptr) return false;
  for (int j = 0; j < a.n; ++j)
    if (b.ops[j].act != a.ops[j].out || b.ops[j].K != a.ops[j].N || a.ops[j].out_rows != nullptr)
      return false;
  return true;
}

// Enqueue steps in order.  At prefill sizes each down/up pair runs as one
// fused launch per linear.
lr_status enqueue_steps(const std::vector<Step>& steps, int64_t M, int32_t* status, cudaStream_t s) {
  const bool prefill = M > kDecodeMaxRows && prefill_fused_enabled();
  for (size_t i = 0; i < steps.size(); ++i) {
    const Step& st = steps[i];
    lr_status r;
    if (prefill && i + 1 < steps.size() && down_up_pair(st, steps[i + 1])) {
      r = ensure_configured();
      for (int j = 0; j < st.n && r == LR_OK; ++j) {
        const GemmOp& dn = st.ops[j];
        const GemmOp& up = steps[i + 1].ops[j];
        if (prefill_fuse_linear(M, dn, up)) {
          r = launch_prefill_pair_fused(M, dn, up, st.cnt, status, s);
        } else {
          r = run_ops(M, &dn, 1, status, s);
          if (r == LR_OK) r = run_ops(M, &up, 1, status, s);
        }
      }
      ++i;
    } else if (st.kind == Step::GEMM) {
      r = run_ops(M, st.ops, st.n, status, s);
    } else if (st.kind == Step::RMSNORM) {
      r = launch_rmsnorm(static_cast<const float*>(st.src0), st.dst, M, st.d, st.eps, s);
    } else {
      r = launch_silu_mul(st.src0, st.src1, st.dst, M, st.d, s);
    }
    if (r != LR_OK) return r;
  }
  return LR_OK;
}

lr_status enqueue_block(float* h, int64_t M, const lr_block_desc* b, uint8_t* ws,
                        int32_t* status, cudaStream_t s) {
  std::vector<Step> steps;
  block_steps(h, M, b, ws, steps);
  return enqueue_steps(steps, M, status, s);
}

int64_t block_launches(int64_t M, const lr_block_desc* b) {
  // rmsnorm x2, the GEMM launches (grouped at decode sizes) and, for SiLU-GLU,
  // a silu_mul launch; ReLU is applied in the up projection's epilogue.
  const int64_t glu = b->mlp == LR_MLP_RELU ? 0 : 1;
  if (M <= kDecodeMaxRows) return 2 + glu + 8;
  // two launches per linear: down and up, or a counter-clearing launch and
  // the fused launch
  return 2 + glu + 2 * (b->mlp == LR_MLP_RELU ? 6 : 7);
}

// ---------------------------------------------------------------- stack
size_t block_region_bytes(const lr_stack_desc* st) {
  size_t need = 0;
  for (int l = 0; l < st->n_layers; ++l)
    need = std::max(need, block_layout(st->cap, &st->layers[l]).total);
  return align_up(need);
}

lr_status check_stack(const lr_stack_desc* st) {
  if (st == nullptr) return invalid("stack: null descriptor");
  if (st->n_layers < 0 || (st->n_layers > 0 && st->layers == nullptr))
    return invalid("stack: bad layer array");
  if (st->n_layers == 0) return invalid("stack: no layers");
  if (st->cap <= 0 || st->cap > kDecodeMaxRows * 64) return invalid("stack: bad cap");
  if (st->mode != LR_STACK_AUTO && st->mode != LR_STACK_LAYERED) return invalid("stack: bad mode");
  if (!st->pool_in || !st->pool_out || !st->remap || !st->n_active || !st->xbuf || !st->h ||
      !st->ybuf || !st->scratch)
    return invalid("stack: null pointer");
  if (!aligned16(st->pool_in) || !aligned16(st->pool_out) || !aligned16(st->xbuf) ||
      !aligned16(st->h) || !aligned16(st->ybuf) || (reinterpret_cast<uintptr_t>(st->scratch) % kAlign))
    return invalid("stack: misaligned buffer");
  if (st->pool_rows <= 0) return invalid("stack: empty pool");
  const int d = st->layers[0].d_model;
  for (int l = 0; l < st->n_layers; ++l) {
    lr_status s2 = check_block(&st->layers[l]);
    if (s2 != LR_OK) return s2;
    if (st->layers[l].d_model != d) return invalid("stack: layers disagree on d_model");
  }
  const size_t need = lr_stack_scratch_bytes(st);
  if (st->scratch_bytes < need) return invalid("stack: scratch %zu < %zu bytes", st->scratch_bytes, need);
  return LR_OK;
}

// One step with one launch per kernel.
lr_status enqueue_layered(const lr_stack_desc* st, cudaStream_t s) {
  const int d = st->layers[0].d_model;
  const int64_t row_bytes = static_cast<int64_t>(d) * 2;
  uint8_t* ws = static_cast<uint8_t*>(st->scratch);
  lr_status r;
  const bool decode = st->cap <= kDecodeMaxRows;
  if (decode) {
    r = launch_gather_rows(st->pool_in, st->pool_rows, d, st->remap, st->n_active, st->xbuf, st->h,
                           st->cap, st->dev_status, s);
  } else {
    r = launch_gather(st->pool_in, st->pool_rows, row_bytes, st->remap, st->n_active, st->xbuf,
                      st->cap, st->dev_status, s);
    if (r == LR_OK) r = launch_widen(st->xbuf, st->h, st->cap * d, s);
  }
  if (r != LR_OK) return r;
  std::vector<Step> steps;
  for (int l = 0; l < st->n_layers; ++l) block_steps(st->h, st->cap, &st->layers[l], ws, steps);
  r = enqueue_steps(steps, st->cap, st->dev_status, s);
  if (r != LR_OK) return r;
  if (decode)
    return launch_scatter_rows(st->h, st->ybuf, st->remap, st->n_active, st->pool_out,
                               st->pool_rows, d, st->cap, st->dev_status, s);
  r = launch_narrow(st->h, st->ybuf, st->cap * d, s);
  if (r != LR_OK) return r;
  return launch_scatter(st->ybuf, st->remap, st->n_active, st->pool_out, st->pool_rows,
                        row_bytes, st->cap, st->dev_status, s);
}

}  // namespace
}  // namespace lr

struct lr_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  uint32_t magic = 0x4C524750u;
};

using namespace lr;

extern "C" {

const char* lr_status_string(lr_status st) {
  switch (st) {
    case LR_OK: return "ok";
    case LR_ERR_INVALID_ARG: return "invalid argument";
    case LR_ERR_UNSUPPORTED: return "unsupported shape";
    case LR_ERR_CUDA: return "CUDA error";
    case LR_ERR_TIMEOUT: return "device wait timed out";
    case LR_ERR_REMAP_RANGE: return "remap entry outside the pool";
    case LR_ERR_STATE: return "bad object state";
  }
  return "unknown status";
}

const char* lr_last_error(void) { return g_err; }

void lr_test_stall_producer(int32_t on) { g_stall_producer.store(on != 0 ? 1 : 0); }

void lr_test_prefill_schedule(int32_t lag, int32_t group) {
  g_prefill_lag.store(lag > 0 ? lag : (lag < 0 ? -1 : 0));
  g_prefill_group.store(group > 0 ? group : 0);
}

size_t lr_linear_workspace_bytes(int64_t M, const lr_factor* f) {
  if (f == nullptr || M < 0) return 0;
  size_t n = align_up(static_cast<size_t>(M) * static_cast<size_t>(f->r) * 2);
  if (M > kDecodeMaxRows) n += align_up(prefill_band_counter_bytes(M));
  return n;
}

lr_status lr_linear_forward(const void* x, int64_t ldx, void* y, int64_t ldy, lr_dtype y_dtype,
                            int64_t M, const lr_factor* f, void* workspace, size_t ws_bytes,
                            int32_t* dev_status, lr_stream s) {
  lr_status st = check_factor(f, "linear");
  if (st != LR_OK) return st;
  if (M < 0 || M > (int64_t(1) << 31) - 1) return invalid("linear: bad M");
  if (M == 0) return LR_OK;
  st = check_linear_io("linear", x, ldx, y, ldy, y_dtype, M, f);
  if (st != LR_OK) return st;
  if (workspace == nullptr) return invalid("linear: null workspace");
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return invalid("linear: workspace not 256-byte aligned");
  if (ws_bytes < lr_linear_workspace_bytes(M, f)) return invalid("linear: workspace too small");
  return enqueue_linear(x, ldx, y, ldy, y_dtype, M, f, workspace, dev_status,
                        reinterpret_cast<cudaStream_t>(s));
}

lr_status lr_factor_pack(const void* A, const void* B, int32_t d_in, int32_t d_out, int32_t r, void* At,
                         void* Bt, lr_stream s) {
  if (d_in <= 0 || d_out <= 0 || r <= 0) return invalid("factor_pack: non-positive dims");
  if (d_in % 64 || d_out % 64 || r % 64) {
    set_error("factor_pack: d_in=%d d_out=%d r=%d must be multiples of 64", d_in, d_out, r);
    return LR_ERR_UNSUPPORTED;
  }
  if (!A || !B || !At || !Bt) return invalid("factor_pack: null pointer");
  if (!aligned16(A) || !aligned16(B) || !aligned16(At) || !aligned16(Bt))
    return invalid("factor_pack: pointers must be 16-byte aligned");
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(A), b0 = reinterpret_cast<uintptr_t>(B);
  const uintptr_t at0 = reinterpret_cast<uintptr_t>(At), bt0 = reinterpret_cast<uintptr_t>(Bt);
  const uintptr_t na = static_cast<uintptr_t>(d_in) * r * 2, nb = static_cast<uintptr_t>(r) * d_out * 2;
  auto overlap = [](uintptr_t x, uintptr_t nx, uintptr_t y, uintptr_t ny) { return x < y + ny && y < x + nx; };
  if (overlap(a0, na, at0, na) || overlap(a0, na, bt0, nb) || overlap(b0, nb, at0, na) ||
      overlap(b0, nb, bt0, nb) || overlap(at0, na, bt0, nb))
    return invalid("factor_pack: inputs and outputs must not overlap");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  lr_status st = launch_transpose_bf16(A, d_in, r, At, cs);
  if (st != LR_OK) return st;
  return launch_transpose_bf16(B, r, d_out, Bt, cs);
}

size_t lr_block_scratch_bytes(int64_t M, const lr_block_desc* b) {
  if (b == nullptr || M < 0) return 0;
  return block_layout(M, b).total;
}

lr_status lr_block_forward(float* h, int64_t M, const lr_block_desc* b, void* scratch,
                           size_t scratch_bytes, int32_t* dev_status, lr_stream s) {
  lr_status st = check_block(b);
  if (st != LR_OK) return st;
  if (M < 0 || M > (int64_t(1) << 31) - 1) return invalid("block: bad M");
  if (M == 0) return LR_OK;
  if (h == nullptr || scratch == nullptr) return invalid("block: null pointer");
  if (!aligned16(h) || reinterpret_cast<uintptr_t>(scratch) % kAlign)
    return invalid("block: h must be 16-byte and scratch 256-byte aligned");
  if (scratch_bytes < lr_block_scratch_bytes(M, b)) return invalid("block: scratch too small");
  return enqueue_block(h, M, b, static_cast<uint8_t*>(scratch), dev_status,
                       reinterpret_cast<cudaStream_t>(s));
}

lr_status remap_compact(const void* pool, int64_t pool_rows, int64_t row_bytes,
                        const int32_t* remap, const int32_t* n_active, void* buf, int64_t cap,
                        int32_t* dev_status, lr_stream s) {
  if (cap < 0 || pool_rows < 0) return invalid("remap_compact: negative size");
  if (row_bytes <= 0 || row_bytes % 16) return invalid("remap_compact: row_bytes must be a positive multiple of 16");
  if (cap == 0) return LR_OK;
  if (!pool || !remap || !n_active || !buf) return invalid("remap_compact: null pointer");
  if (!aligned16(pool) || !aligned16(buf)) return invalid("remap_compact: misaligned buffer");
  if (cap > 0x7FFFFFFF) return invalid("remap_compact: cap too large");
  return launch_gather(pool, pool_rows, row_bytes, remap, n_active, buf, cap, dev_status,
                       reinterpret_cast<cudaStream_t>(s));
}

lr_status remap_scatter(const void* buf, const int32_t* remap, const int32_t* n_active,
                        void* pool, int64_t pool_rows, int64_t row_bytes, int64_t cap,
                        int32_t* dev_status, lr_stream s) {
  if (cap < 0 || pool_rows < 0) return invalid("remap_scatter: negative size");
  if (row_bytes <= 0 || row_bytes % 16) return invalid("remap_scatter: row_bytes must be a positive multiple of 16");
  if (cap == 0) return LR_OK;
  if (!pool || !remap || !n_active || !buf) return invalid("remap_scatter: null pointer");
  if (!aligned16(pool) || !aligned16(buf)) return invalid("remap_scatter: misaligned buffer");
  if (cap > 0x7FFFFFFF) return invalid("remap_scatter: cap too large");
  return launch_scatter(buf, remap, n_active, pool, pool_rows, row_bytes, cap, dev_status,
                        reinterpret_cast<cudaStream_t>(s));
}

lr_status lr_kv_reconstruct(const void* latent_pool, int64_t pool_rows, int32_t r,
                            const int32_t* remap, const int32_t* n_active, int64_t cap,
                            void* latent_buf, const void* Bt, int32_t d_kv, void* out,
                            int32_t* dev_status, lr_stream s) {
  if (r <= 0 || d_kv <= 0 || cap < 0 || pool_rows < 0) return invalid("kv_reconstruct: bad sizes");
  if (r % 64 || d_kv % 64) {
    set_error("kv_reconstruct: r=%d and d_kv=%d must be multiples of 64", r, d_kv);
    return LR_ERR_UNSUPPORTED;
  }
  if (cap == 0) return LR_OK;
  if (cap > 0x7FFFFFFF) return invalid("kv_reconstruct: cap too large");
  if (!latent_pool || !remap || !n_active || !latent_buf || !Bt || !out)
    return invalid("kv_reconstruct: null pointer");
  if (!aligned16(latent_pool) || !aligned16(latent_buf) || !aligned16(Bt) || !aligned16(out))
    return invalid("kv_reconstruct: buffers must be 16-byte aligned");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  lr_status st = launch_gather(latent_pool, pool_rows, static_cast<int64_t>(r) * 2, remap,
                               n_active, latent_buf, cap, dev_status, cs);
  if (st != LR_OK) return st;
  GemmOp up = make_op(Bt, d_kv, r, latent_buf, r, r, EPI_STORE_BF16, out, d_kv);
  return run_ops(cap, &up, 1, dev_status, cs);
}

}  // extern "C"

namespace {

// Columns [shard_begin(g), shard_begin(g + 1)) of an n-column dimension (n a
// multiple of 64) belong to process g of G: whole 64-column blocks, as even as
// possible.
int64_t shard_begin(int64_t n, int g, int G) { return 64 * ((n / 64) * g / G); }

}  // namespace

extern "C" {

size_t lr_rank_sharded_workspace_bytes(int64_t M, const lr_factor* f, int32_t n_shards) {
  if (f == nullptr || M < 0 || n_shards < 1 || f->r < 64 * n_shards) return 0;
  const size_t m = static_cast<size_t>(M);
  size_t total = align_up(m * static_cast<size_t>(f->r) * 2);
  for (int g = 0; g < n_shards; ++g) {
    const int64_t w = shard_begin(f->r, g + 1, n_shards) - shard_begin(f->r, g, n_shards);
    total += align_up(m * static_cast<size_t>(w) * 2);
  }
  return total;
}

lr_status lr_linear_forward_rank_sharded(const void* x, int64_t ldx, void* y, int64_t ldy,
                                         lr_dtype y_dtype, int64_t M, const lr_factor* f,
                                         int32_t n_shards, void* workspace, size_t ws_bytes,
                                         int32_t* dev_status, lr_stream s) {
  lr_status st = check_factor(f, "rank_sharded");
  if (st != LR_OK) return st;
  const int G = n_shards;
  if (G < 1 || 64 * G > f->r || 64 * G > f->d_out)
    return invalid("rank_sharded: n_shards=%d outside [1, min(r, d_out)/64]", G);
  if (M < 0 || M > (int64_t(1) << 31) - 1) return invalid("rank_sharded: bad M");
  if (M == 0) return LR_OK;
  if (x == nullptr || y == nullptr || workspace == nullptr) return invalid("rank_sharded: null pointer");
  if (y_dtype != LR_BF16 && y_dtype != LR_F32) return invalid("rank_sharded: bad y dtype");
  if (ldx < f->d_in || ldx % 8 || !aligned16(x))
    return invalid("rank_sharded: x must be 16-byte aligned with ldx >= d_in, ldx %% 8 == 0");
  if (ldy < f->d_out) return invalid("rank_sharded: ldy < d_out");
  if (M > kDecodeMaxRows && (!aligned16(y) || ldy % 8))
    return invalid("rank_sharded: y must be 16-byte aligned with ldy %% 8 == 0");
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return invalid("rank_sharded: workspace not 256-byte aligned");
  if (ws_bytes < lr_rank_sharded_workspace_bytes(M, f, G)) return invalid("rank_sharded: workspace too small");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  const size_t m = static_cast<size_t>(M);
  uint8_t* t = static_cast<uint8_t*>(workspace);  // gathered [M][r]
  uint8_t* local = t + align_up(m * static_cast<size_t>(f->r) * 2);
  const int esz = y_dtype == LR_BF16 ? 2 : 4;
  const uint16_t* At = static_cast<const uint16_t*>(f->At);
  const uint16_t* Bt = static_cast<const uint16_t*>(f->Bt);
  // 1. down projection of every process into its own buffer
  uint8_t* tg = local;
  for (int g = 0; g < G; ++g) {
    const int64_t r0 = shard_begin(f->r, g, G), w = shard_begin(f->r, g + 1, G) - r0;
    GemmOp down = make_op(At + r0 * f->d_in, static_cast<int>(w), f->d_in, x, ldx, f->d_in,
                          EPI_STORE_BF16, tg, w);
    st = run_ops(M, &down, 1, dev_status, cs);
    if (st != LR_OK) return st;
    tg += align_up(m * static_cast<size_t>(w) * 2);
  }
  // 2. all-gather in rank space: every t_g lands in its columns of t
  tg = local;
  for (int g = 0; g < G; ++g) {
    const int64_t r0 = shard_begin(f->r, g, G), w = shard_begin(f->r, g + 1, G) - r0;
    cudaError_t e = cudaMemcpy2DAsync(t + r0 * 2, static_cast<size_t>(f->r) * 2, tg,
                                      static_cast<size_t>(w) * 2, static_cast<size_t>(w) * 2, m,
                                      cudaMemcpyDeviceToDevice, cs);
    if (e != cudaSuccess) return cuda_fail(e, "rank_sharded: all-gather copy");
    tg += align_up(m * static_cast<size_t>(w) * 2);
  }
  // 3. up projection of every process on its output columns (shard mode)
  for (int g = 0; g < G; ++g) {
    const int64_t o0 = shard_begin(f->d_out, g, G), w = shard_begin(f->d_out, g + 1, G) - o0;
    GemmOp up = make_op(Bt + o0 * f->r, static_cast<int>(w), f->r, t, f->r, f->r,
                        y_dtype == LR_BF16 ? EPI_STORE_BF16 : EPI_STORE_F32,
                        static_cast<uint8_t*>(y) + o0 * esz, ldy);
    st = run_ops(M, &up, 1, dev_status, cs);
    if (st != LR_OK) return st;
  }
  return LR_OK;
}

lr_status lr_rank_shard_comm_bytes(int64_t M, int32_t d_out, int32_t r, int32_t n_shards,
                                   int32_t elem_bytes, int64_t* rank_space, int64_t* full_space) {
  if (rank_space == nullptr || full_space == nullptr) return invalid("comm_bytes: null output");
  if (M < 0 || d_out <= 0 || r <= 0 || elem_bytes <= 0) return invalid("comm_bytes: bad sizes");
  if (r % 64 || d_out % 64) return invalid("comm_bytes: r and d_out must be multiples of 64");
  const int G = n_shards;
  if (G < 1 || 64 * G > r || 64 * G > d_out) return invalid("comm_bytes: bad n_shards");
  int64_t min_r = r, min_o = d_out;
  for (int g = 0; g < G; ++g) {
    min_r = std::min(min_r, shard_begin(r, g + 1, G) - shard_begin(r, g, G));
    min_o = std::min(min_o, shard_begin(d_out, g + 1, G) - shard_begin(d_out, g, G));
  }
  *rank_space = (r - min_r) * M * elem_bytes;
  *full_space = 2 * (d_out - min_o) * M * elem_bytes;
  return LR_OK;
}

lr_status remap_build_blocks(const int32_t* lengths, int64_t n_seq, const int32_t* block_table,
                             int32_t blocks_per_seq, int32_t block_rows, int64_t cap_blocks,
                             int32_t* blocks_out, int32_t* n_blocks_out, int32_t* n_runs_out) {
  if (n_seq < 0 || cap_blocks < 0 || block_rows <= 0 || blocks_per_seq < 0)
    return invalid("remap_build_blocks: bad sizes");
  if ((n_seq > 0 && (!lengths || !block_table)) || (cap_blocks > 0 && !blocks_out) || !n_blocks_out ||
      !n_runs_out)
    return invalid("remap_build_blocks: null pointer");
  int64_t n = 0;
  for (int64_t s = 0; s < n_seq; ++s) {
    const int64_t L = lengths[s];
    if (L < 0 || L > static_cast<int64_t>(blocks_per_seq) * block_rows)
      return invalid("remap_build_blocks: length %lld of sequence %lld does not fit its table row",
                     (long long)L, (long long)s);
    const int64_t nb = (L + block_rows - 1) / block_rows;
    for (int64_t b = 0; b < nb; ++b) {
      const int32_t blk = block_table[s * blocks_per_seq + b];
      if (blk < 0) return invalid("remap_build_blocks: missing block for sequence %lld", (long long)s);
      if (n >= cap_blocks) return invalid("remap_build_blocks: blocks exceed cap %lld", (long long)cap_blocks);
      blocks_out[n++] = blk;
    }
  }
  std::vector<int32_t> sorted(blocks_out, blocks_out + n);
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
    return invalid("remap_build_blocks: a physical block is listed twice");
  int32_t runs = 0;
  for (int64_t i = 0; i < n; ++i)
    if (i == 0 || blocks_out[i] != blocks_out[i - 1] + 1) ++runs;
  for (int64_t i = n; i < cap_blocks; ++i) blocks_out[i] = -1;
  *n_blocks_out = static_cast<int32_t>(n);
  *n_runs_out = runs;
  return LR_OK;
}

lr_status lr_kv_latent_write(const void* x, int64_t ldx, int64_t M, const void* At, int32_t d_in, int32_t r,
                             const int32_t* rows, void* latent_pool, int64_t pool_rows, int32_t* dev_status,
                             lr_stream s) {
  if (d_in <= 0 || r <= 0 || M < 0 || pool_rows < 0) return invalid("kv_latent_write: bad sizes");
  if (d_in % 64 || r % 64) {
    set_error("kv_latent_write: d_in=%d and r=%d must be multiples of 64", d_in, r);
    return LR_ERR_UNSUPPORTED;
  }
  if (M == 0) return LR_OK;
  if (M > 0x7FFFFFFF) return invalid("kv_latent_write: bad M");
  if (!x || !At || !rows || !latent_pool) return invalid("kv_latent_write: null pointer");
  if (ldx < d_in || ldx % 8 || !aligned16(x) || !aligned16(At) || !aligned16(latent_pool))
    return invalid("kv_latent_write: x, At and the pool must be 16-byte aligned with ldx >= d_in, ldx %% 8 == 0");
  GemmOp down = make_op(At, r, d_in, x, ldx, d_in, EPI_STORE_BF16, latent_pool, r);
  down.out_rows = rows;
  down.out_rows_limit = pool_rows;
  return run_ops(M, &down, 1, dev_status, reinterpret_cast<cudaStream_t>(s));
}

lr_status lr_kv_reconstruct_paged(const void* latent_pool, int64_t pool_blocks, int32_t r, const int32_t* blocks,
                                  const int32_t* n_blocks, int64_t cap_blocks, const void* Bt, int32_t d_kv,
                                  void* out, int32_t* dev_status, lr_stream s) {
  if (r <= 0 || d_kv <= 0 || cap_blocks < 0 || pool_blocks < 0)
    return invalid("kv_reconstruct_paged: bad sizes");
  if (r % 64 || d_kv % 64) {
    set_error("kv_reconstruct_paged: r=%d and d_kv=%d must be multiples of 64", r, d_kv);
    return LR_ERR_UNSUPPORTED;
  }
  if (cap_blocks == 0) return LR_OK;
  if (pool_blocks * kPageRows > 0x7FFFFFFF || cap_blocks * kPageRows > 0x7FFFFFFF)
    return invalid("kv_reconstruct_paged: pool or capacity rows overflow int32");
  if (!latent_pool || !blocks || !n_blocks || !Bt || !out) return invalid("kv_reconstruct_paged: null pointer");
  if (!aligned16(latent_pool) || !aligned16(Bt) || !aligned16(out))
    return invalid("kv_reconstruct_paged: buffers must be 16-byte aligned");
  lr_status st = ensure_configured();
  if (st != LR_OK) return st;
  GemmOp up = make_op(Bt, d_kv, r, latent_pool, r, r, EPI_STORE_BF16, out, d_kv);
  return launch_prefill_paged(cap_blocks * kPageRows, up, blocks, n_blocks, pool_blocks, dev_status,
                              reinterpret_cast<cudaStream_t>(s));
}

lr_status remap_build(const int32_t* lengths, int64_t n_seq, const int32_t* block_table,
                      int32_t blocks_per_seq, int32_t block_rows, int32_t tail_rows, int64_t cap,
                      int32_t* remap_out, int32_t* n_active_out, int32_t* n_runs_out) {
  if (n_seq < 0 || cap < 0 || block_rows <= 0 || blocks_per_seq < 0)
    return invalid("remap_build: bad sizes");
  if ((n_seq > 0 && (!lengths || !block_table)) || (cap > 0 && !remap_out) || !n_active_out ||
      !n_runs_out)
    return invalid("remap_build: null pointer");
  int64_t n = 0;
  for (int64_t s = 0; s < n_seq; ++s) {
    const int64_t L = lengths[s];
    if (L < 0 || L > static_cast<int64_t>(blocks_per_seq) * block_rows)
      return invalid("remap_build: length %lld of sequence %lld does not fit its table row",
                     (long long)L, (long long)s);
    const int64_t start = tail_rows <= 0 ? 0 : std::max<int64_t>(0, L - tail_rows);
    for (int64_t p = start; p < L; ++p) {
      const int32_t blk = block_table[s * blocks_per_seq + p / block_rows];
      if (blk < 0) return invalid("remap_build: missing block for sequence %lld", (long long)s);
      if (n >= cap) return invalid("remap_build: rows exceed cap %lld", (long long)cap);
      const int64_t row = static_cast<int64_t>(blk) * block_rows + p % block_rows;
      if (row > 0x7FFFFFFF) return invalid("remap_build: row index overflows int32");
      remap_out[n++] = static_cast<int32_t>(row);
    }
  }
  // Distinct targets: the scatter writes each pool row at most once.
  std::vector<int32_t> sorted(remap_out, remap_out + n);
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
    return invalid("remap_build: two rows map to the same physical row");
  int32_t runs = 0;
  for (int64_t i = 0; i < n; ++i)
    if (i == 0 || remap_out[i] != remap_out[i - 1] + 1) ++runs;
  for (int64_t i = n; i < cap; ++i) remap_out[i] = -1;
  *n_active_out = static_cast<int32_t>(n);
  *n_runs_out = runs;
  return LR_OK;
}

size_t lr_stack_scratch_bytes(const lr_stack_desc* st) {
  if (st == nullptr || st->layers == nullptr || st->n_layers <= 0 || st->cap <= 0) return 0;
  return block_region_bytes(st);
}

lr_status lr_stack_forward(const lr_stack_desc* st, lr_stream s) {
  lr_status r = check_stack(st);
  if (r != LR_OK) return r;
  r = ensure_configured();
  if (r != LR_OK) return r;
  return enqueue_layered(st, reinterpret_cast<cudaStream_t>(s));
}

int64_t lr_stack_launch_count(const lr_stack_desc* st) {
  if (st == nullptr || st->layers == nullptr) return 0;
  const bool decode = st->cap <= kDecodeMaxRows;
  int64_t n = decode ? 2 : 4;  // gather(+widen), (narrow+)scatter
  for (int l = 0; l < st->n_layers; ++l) n += block_launches(st->cap, &st->layers[l]);
  return n;
}

lr_status lr_graph_capture(const lr_stack_desc* st, lr_graph** out) {
  if (out == nullptr) return invalid("graph_capture: null output");
  *out = nullptr;
  lr_status r = check_stack(st);
  if (r != LR_OK) return r;
  r = ensure_configured();
  if (r != LR_OK) return r;
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "graph_capture: stream");
  lr_graph* g = new lr_graph();
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    r = cuda_fail(e, "graph_capture: begin");
  } else {
    lr_status r2 = enqueue_layered(st, cs);
    e = cudaStreamEndCapture(cs, &g->graph);
    if (r2 != LR_OK) r = r2;
    else if (e != cudaSuccess) r = cuda_fail(e, "graph_capture: end");
    else {
      e = cudaGraphInstantiate(&g->exec, g->graph, 0);
      if (e != cudaSuccess) r = cuda_fail(e, "graph_capture: instantiate");
    }
  }
  cudaStreamDestroy(cs);
  if (r != LR_OK) {
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    return r;
  }
  *out = g;
  return LR_OK;
}

lr_status lr_graph_replay(lr_graph* g, lr_stream s) {
  if (g == nullptr || g->magic != 0x4C524750u || g->exec == nullptr) {
    set_error("graph_replay: not a live graph");
    return LR_ERR_STATE;
  }
  cudaError_t e = cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) return cuda_fail(e, "graph_replay");
  return LR_OK;
}

lr_status lr_graph_destroy(lr_graph* g) {
  if (g == nullptr || g->magic != 0x4C524750u) {
    set_error("graph_destroy: not a live graph");
    return LR_ERR_STATE;
  }
  g->magic = 0;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
  return LR_OK;
}

}  // extern "C"
