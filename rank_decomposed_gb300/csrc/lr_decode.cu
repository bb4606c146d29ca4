// Decode-size GEMMs (M <= 256 rows): out[m][n] = sum_k act[m][k] * W[n][k].
//
// These are the down and up projections of a decomposed layer (DeInfer, English
// summary page section 2.A) at decode batch sizes, where the time is the
// stream of factor bytes from HBM.  Design for sm_103a:
//  * swap-AB on the 5th-generation tensor cores: a 128-row tile of the weight
//    is the MMA's M side and the (padded) tokens are its N side, so M = 1..256
//    tokens all run on tcgen05 with an fp32 accumulator in TMEM;
//  * weight and activation tiles arrive by TMA (128-byte swizzle) through a
//    multi-stage mbarrier ring; one thread issues the MMAs;
//  * the K dimension of each 128-row tile is split over the CTAs of one
//    thread-block cluster; their fp32 partial tiles are summed in a fixed
//    order through distributed shared memory, by all six warps once the main
//    loop is done, so no workspace, no counters and no floating-point atomics
//    are involved and the result is deterministic;
//  * an unsplit tile leaves TMEM through a shared-memory staging tile and one
//    bulk copy per token row (a bulk fp32 add for the residual stream);
//  * up to three problems with the same input (q/k/v, gate/up) share one
//    launch;
//  * programmatic dependent launch: weight tiles (which never depend on the
//    previous kernel) are requested before griddepcontrol.wait, activation
//    tiles after it.
#include <cuda_bf16.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "lr_ptx.cuh"

namespace lr {
namespace {

// warp 0: TMA, warp 1: MMA, warps 2..5: epilogue (TMEM lane quadrants 2, 3,
// 0, 1); all six warps share the split-K reduction.
constexpr int kThreads = 192;
constexpr int kTileN = 128;    // weight rows per tile = MMA M
constexpr int kBK = 64;        // reduction depth of one pipeline stage
constexpr int kWBytes = kTileN * kBK * 2;

template <int NT>
struct DecodeCfg;
template <> struct DecodeCfg<16> { static constexpr int kStages = 6; static constexpr int kSlots = 2; };
template <> struct DecodeCfg<32> { static constexpr int kStages = 5; static constexpr int kSlots = 2; };
template <> struct DecodeCfg<64> { static constexpr int kStages = 4; static constexpr int kSlots = 2; };
template <> struct DecodeCfg<128> { static constexpr int kStages = 3; static constexpr int kSlots = 2; };
template <> struct DecodeCfg<256> { static constexpr int kStages = 4; static constexpr int kSlots = 1; };

template <int NT>
constexpr int decode_smem_bytes() {
  return DecodeCfg<NT>::kStages * (kWBytes + NT * kBK * 2) + 1024;
}

// After the MMAs the ring holds the fp32 partial tile [NT][128] and, behind
// it, the staged output slice of at most ceil(NT / 2) tokens (S >= 2); with
// S == 1 it holds the staged [NT][128] tile alone.
template <int NT>
constexpr bool decode_epilogue_fits() {
  return NT * kTileN * 4 + ((NT + 1) / 2) * kTileN * 4 <= DecodeCfg<NT>::kStages * (kWBytes + NT * kBK * 2);
}
static_assert(decode_epilogue_fits<16>() && decode_epilogue_fits<32>() && decode_epilogue_fits<64>() &&
                  decode_epilogue_fits<128>() && decode_epilogue_fits<256>(),
              "decode epilogue staging does not fit in the ring");

__device__ __forceinline__ int act_col(const DecodeProblem& P, int kb) {
  const int k = kb * kBK;
  if (P.gqa_head_dim > 0) {
    const int head = k / P.gqa_head_dim;
    return (head / P.gqa_group) * P.gqa_head_dim + (k % P.gqa_head_dim);
  }
  return k;
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

// Remote shared-memory load.  No memory clobber: the loads are ordered after
// the cluster barrier that precedes them (which is a compiler barrier), and
// leaving them free lets the compiler keep many in flight.
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float relu_f(float v) { return v > 0.0f ? v : 0.0f; }

// Output row of token `tok`: the token itself, or its entry in the problem's
// row list (-1 for an entry outside the output, which is reported).
__device__ __forceinline__ int64_t out_row(const DecodeProblem& P, int tok) {
  if (P.out_rows == nullptr) return tok;
  const int64_t r = P.out_rows[tok];
  if (r >= 0 && r < P.out_rows_limit) return r;
  report_status(P.status, LR_ERR_REMAP_RANGE);
  return -1;
}

// Four consecutive outputs (m, n .. n+3) of one problem.
__device__ __forceinline__ void store_out4(const DecodeProblem& P, int m, int n, float4 v) {
  const int64_t orow = out_row(P, m);
  if (orow < 0) return;
  const int64_t off = orow * P.ldo + n;
  if (P.epi == EPI_RELU_BF16) {
    v.x = relu_f(v.x); v.y = relu_f(v.y); v.z = relu_f(v.z); v.w = relu_f(v.w);
  }
  if (epi_is_bf16(P.epi)) {
    uint16_t* o = static_cast<uint16_t*>(P.out) + off;
    const uint16_t b0 = f32_to_bf16_rn(v.x), b1 = f32_to_bf16_rn(v.y);
    const uint16_t b2 = f32_to_bf16_rn(v.z), b3 = f32_to_bf16_rn(v.w);
    if (P.vec_ok) {
      *reinterpret_cast<uint2*>(o) = make_uint2(static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16),
                                                static_cast<uint32_t>(b2) | (static_cast<uint32_t>(b3) << 16));
    } else {
      o[0] = b0; o[1] = b1; o[2] = b2; o[3] = b3;
    }
  } else {
    float* o = static_cast<float*>(P.out) + off;
    if (P.epi == EPI_ADD_F32) {
      if (P.vec_ok) {
        const float4 h = *reinterpret_cast<const float4*>(o);
        v.x += h.x; v.y += h.y; v.z += h.z; v.w += h.w;
      } else {
        v.x += o[0]; v.y += o[1]; v.z += o[2]; v.w += o[3];
      }
    }
    if (P.vec_ok) {
      *reinterpret_cast<float4*>(o) = v;
    } else {
      o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
  }
}

// Bytes of one output element.
__device__ __forceinline__ int out_elem_bytes(const DecodeProblem& P) {
  return epi_is_bf16(P.epi) ? 2 : 4;
}

// Token `tok` of the tile, staged in shared memory as 128 consecutive output
// elements, goes to out[tok][n0 ..] with one bulk copy (a bulk fp32 add at L2
// for the residual epilogue); rows past N are not written.  Needs vec_ok.
__device__ __forceinline__ void store_staged_row(const DecodeProblem& P, int tok, int n0,
                                                 const uint8_t* row) {
  const int esz = out_elem_bytes(P);
  const int rows = P.N - n0 < kTileN ? P.N - n0 : kTileN;
  const int64_t orow = out_row(P, tok);
  if (orow < 0) return;
  uint8_t* dst = static_cast<uint8_t*>(P.out) + (orow * P.ldo + n0) * esz;
  if (P.epi == EPI_ADD_F32)
    bulk_add_f32(dst, row, static_cast<uint32_t>(rows * esz));
  else
    bulk_store(dst, row, static_cast<uint32_t>(rows * esz));
}

// Sum tokens [t0, t1) x 128 rows of the tile over the S partial tiles of the
// cluster, in rank order, four rows at a time, by `nthr` threads (et is this
// thread's index among them); CH chunks per iteration keep CH * S remote loads
// in flight.  With `stage` the sums are written there as
// [t1 - t0][128] output elements (the residual add is left to the bulk copy);
// without it they are stored to the output directly.
template <int CH, int MAXS>
__device__ __forceinline__ void reduce_slice(const DecodeProblem& P, const float* ptile, int S,
                                             int t0, int t1, int n0, int et, int nthr, uint8_t* stage) {
  const int nchunks = (t1 - t0) * (kTileN / 4);
  const uint32_t pbase = smem_u32(ptile);
  uint32_t rbase[MAXS];
#pragma unroll
  for (int s2 = 0; s2 < MAXS; ++s2)
    rbase[s2] = s2 < S ? cluster_addr(pbase, static_cast<uint32_t>(s2)) : 0u;
  for (int c = et; c < nchunks; c += nthr * CH) {
    float4 v[CH][MAXS];
#pragma unroll
    for (int h = 0; h < CH; ++h) {
      const int cc = c + h * nthr;
      if (cc < nchunks) {
        const uint32_t off = static_cast<uint32_t>(((t0 + cc / 32) * kTileN + (cc % 32) * 4) * 4);
#pragma unroll
        for (int s2 = 0; s2 < MAXS; ++s2)
          if (s2 < S) v[h][s2] = ld_cluster_f32x4(rbase[s2] + off);
      }
    }
#pragma unroll
    for (int h = 0; h < CH; ++h) {
      const int cc = c + h * nthr;
      if (cc >= nchunks) break;
      const int tok = t0 + cc / 32;
      const int row = (cc % 32) * 4;
      if (n0 + row >= P.N) continue;  // N is a multiple of 64: 4 rows all in or all out
      float4 acc = v[h][0];
#pragma unroll
      for (int s2 = 1; s2 < MAXS; ++s2)
        if (s2 < S) {
          acc.x += v[h][s2].x;
          acc.y += v[h][s2].y;
          acc.z += v[h][s2].z;
          acc.w += v[h][s2].w;
        }
      if (stage == nullptr) {
        store_out4(P, tok, n0 + row, acc);
      } else if (epi_is_bf16(P.epi)) {
        if (P.epi == EPI_RELU_BF16) {
          acc.x = relu_f(acc.x); acc.y = relu_f(acc.y); acc.z = relu_f(acc.z); acc.w = relu_f(acc.w);
        }
        const uint32_t lo = static_cast<uint32_t>(f32_to_bf16_rn(acc.x)) |
                            (static_cast<uint32_t>(f32_to_bf16_rn(acc.y)) << 16);
        const uint32_t hi = static_cast<uint32_t>(f32_to_bf16_rn(acc.z)) |
                            (static_cast<uint32_t>(f32_to_bf16_rn(acc.w)) << 16);
        *reinterpret_cast<uint2*>(stage + ((tok - t0) * kTileN + row) * 2) = make_uint2(lo, hi);
      } else {
        *reinterpret_cast<float4*>(stage + ((tok - t0) * kTileN + row) * 4) = acc;
      }
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, DecodeCfg<NT>::kSlots)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ DecodeMaps maps) {
  constexpr int kStages = DecodeCfg<NT>::kStages;
  constexpr int kABytes = NT * kBK * 2;
  constexpr uint32_t kStageBytes = kWBytes + kABytes;
  constexpr uint32_t kTmemCols = NT < 32 ? 32 : NT;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTileN, NT);
  // Unsplit tiles, and split tiles of the 128- and 256-token shapes, are
  // staged in shared memory and written by bulk copies; split tiles of the
  // smaller shapes are stored by the threads (measured faster there).
  constexpr bool kBulkEpi = NT >= 128;
  // TMEM column chunks (16 tokens each) loaded before one wait in the epilogue.
  constexpr int kChunksPerWait = NT / 16 < 4 ? NT / 16 : 4;

  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accum_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  extern __shared__ uint8_t dyn_smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.splits;
  const int item = blockIdx.x;
  int g = 0;
#pragma unroll
  for (int i = 1; i < kMaxGroup; ++i)
    if (i < p.n_problems && item >= p.prob[i].item_begin) g = i;
  // A register copy of this CTA's problem, selected with static indices.  A
  // reference into the parameter array at a run-time index is a generic
  // pointer, and the compiler would re-read every field after each global
  // store of the epilogue (it cannot prove the two disjoint).
  DecodeProblem P = p.prob[0];
#pragma unroll
  for (int i = 1; i < kMaxGroup; ++i)
    if (i == g) P = p.prob[i];
  const int local = item - P.item_begin;
  const int tile = local / S;
  const int split = local % S;  // == rank inside the cluster
  const int kb0 = split * P.nkb / S;
  const int nk = (split + 1) * P.nkb / S - kb0;
  const int n0 = tile * kTileN;

  const uint32_t raw = smem_u32(dyn_smem);
  uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* w_smem = smem;
  uint8_t* a_smem = smem + kStages * kWBytes;
  float* ptile = reinterpret_cast<float*>(smem);  // [NT][128] once the MMAs are done

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accum_bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  pdl_launch_dependents();

  if (warp == 0) {
    // (With the fault-injection hook set the producer issues nothing: the MMA
    // thread's bounded wait runs out and the launch reports LR_ERR_TIMEOUT.)
    if (lane == 0 && !p.stall_producer) {
      const CUtensorMap* mw = &maps.w[g];
      const CUtensorMap* ma = &maps.a[g];
      prefetch_tensormap(mw);
      prefetch_tensormap(ma);
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_a = l2_policy_evict_last();
      const int npre = nk < kStages ? nk : kStages;
      const int nw = npre < p.prefetch ? npre : p.prefetch;
      // Weight tiles do not depend on earlier kernels: the first `nw` are
      // requested before the wait for the previous kernel.
      for (int i = 0; i < nw; ++i) {
        mbar_arrive_expect_tx(&full_bar[i], kStageBytes);
        tma_load_2d(w_smem + i * kWBytes, mw, &full_bar[i], (kb0 + i) * kBK, n0, pol_w);
      }
      pdl_wait();
      for (int i = 0; i < nw; ++i)
        tma_load_2d(a_smem + i * kABytes, ma, &full_bar[i], act_col(P, kb0 + i), 0, pol_a);
      for (int i = nw; i < npre; ++i) {
        mbar_arrive_expect_tx(&full_bar[i], kStageBytes);
        tma_load_2d(w_smem + i * kWBytes, mw, &full_bar[i], (kb0 + i) * kBK, n0, pol_w);
        tma_load_2d(a_smem + i * kABytes, ma, &full_bar[i], act_col(P, kb0 + i), 0, pol_a);
      }
      int issued = npre;
      for (int i = npre; i < nk; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&empty_bar[s], ((i / kStages) - 1) & 1, &abort_sh)) {
          abort_sh = 1;
          report_status(p.status, LR_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
        tma_load_2d(w_smem + s * kWBytes, mw, &full_bar[s], (kb0 + i) * kBK, n0, pol_w);
        tma_load_2d(a_smem + s * kABytes, ma, &full_bar[s], act_col(P, kb0 + i), 0, pol_a);
        ++issued;
      }
      if (abort_sh) {
        // Let the copies already issued land before the CTA can exit.
        for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
          mbar_wait(&full_bar[i % kStages], (i / kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&full_bar[s], (i / kStages) & 1, &abort_sh)) {
          abort_sh = 1;
          report_status(p.status, LR_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint64_t ad = smem_desc_sw128(smem_u32(w_smem + s * kWBytes));
        const uint64_t bd = smem_desc_sw128(smem_u32(a_smem + s * kABytes));
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          tc_mma_bf16(tmem, ad + 2 * k, bd + 2 * k, kIdesc, (i | k) != 0 ? 1u : 0u);
        tc_commit(&empty_bar[s]);
      }
      tc_commit(&accum_bar);
      // Every MMA issued by this thread completes before TMEM is released.
      mbar_wait(&accum_bar, 0, nullptr);
    }
  } else if (S == 1) {
    // Epilogue, whole K in this CTA: TMEM lanes 32*(warp%4) .. +31 hold weight
    // rows, the columns are tokens.
    const int q = warp & 3;
    const int n = n0 + q * 32 + lane;
    bool ok = mbar_wait(&accum_bar, 0, &abort_sh);
    // One decision for all four epilogue warps: the staged path below meets
    // at a named barrier, which every one of them must reach.
    ok = named_bar_and(1, 128, ok);
    if (ok && P.vec_ok) {
      // Stage the tile as [token][128 rows] of output elements in the (now
      // idle) ring, then one bulk copy per token row.
      tc_fence_after();
      uint8_t* stage = smem;
      const int row = q * 32 + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < NT / 16; c0 += kChunksPerWait) {
        if (c0 * 16 >= p.M) break;
        uint32_t r[kChunksPerWait][16];
#pragma unroll
        for (int b = 0; b < kChunksPerWait; ++b)
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + (c0 + b) * 16, r[b]);
        tmem_ld_wait();
#pragma unroll
        for (int b = 0; b < kChunksPerWait; ++b)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = (c0 + b) * 16 + j;
            if (epi_is_bf16(P.epi)) {
              const float v = __uint_as_float(r[b][j]);
              reinterpret_cast<uint16_t*>(stage)[tok * kTileN + row] =
                  f32_to_bf16_rn(P.epi == EPI_RELU_BF16 ? relu_f(v) : v);
            } else {
              reinterpret_cast<uint32_t*>(stage)[tok * kTileN + row] = r[b][j];
            }
          }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      pdl_wait();  // outputs (e.g. the residual stream) belong to earlier kernels
      const int et = threadIdx.x - 64;
      const int esz = out_elem_bytes(P);
      for (int t = et; t < p.M; t += 128) store_staged_row(P, t, n0, stage + t * kTileN * esz);
      bulk_commit();
      bulk_wait_all();
    } else if (ok) {
      tc_fence_after();
      pdl_wait();  // outputs (e.g. the residual stream) belong to earlier kernels
#pragma unroll 1
      for (int c = 0; c < NT / 16; ++c) {
        if (c * 16 >= p.M) break;
        uint32_t r[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 16, r);
        tmem_ld_wait();
        if (n < P.N && P.out_rows != nullptr) {
          // rows scattered through the problem's row list, one token at a time
          const int nt = p.M - c * 16 < 16 ? p.M - c * 16 : 16;
          for (int j = 0; j < nt; ++j) {
            const int64_t orow = out_row(P, c * 16 + j);
            if (orow < 0) continue;
            const float v = __uint_as_float(r[j]);
            if (epi_is_bf16(P.epi))
              static_cast<uint16_t*>(P.out)[orow * P.ldo + n] =
                  f32_to_bf16_rn(P.epi == EPI_RELU_BF16 ? relu_f(v) : v);
            else if (P.epi == EPI_STORE_F32)
              static_cast<float*>(P.out)[orow * P.ldo + n] = v;
            else
              static_cast<float*>(P.out)[orow * P.ldo + n] += v;
          }
        } else if (n < P.N) {
          const int nt = p.M - c * 16 < 16 ? p.M - c * 16 : 16;
          if (P.epi == EPI_ADD_F32) {
            float* o = static_cast<float*>(P.out) + n;
            float hv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j < nt) hv[j] = o[static_cast<int64_t>(c * 16 + j) * P.ldo];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j < nt) o[static_cast<int64_t>(c * 16 + j) * P.ldo] = hv[j] + __uint_as_float(r[j]);
          } else if (P.epi == EPI_STORE_F32) {
            float* o = static_cast<float*>(P.out) + n;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j < nt) o[static_cast<int64_t>(c * 16 + j) * P.ldo] = __uint_as_float(r[j]);
          } else {
            uint16_t* o = static_cast<uint16_t*>(P.out) + n;
            const bool rl = P.epi == EPI_RELU_BF16;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j < nt) {
                const float v = __uint_as_float(r[j]);
                o[static_cast<int64_t>(c * 16 + j) * P.ldo] = f32_to_bf16_rn(rl ? relu_f(v) : v);
              }
          }
        }
      }
    } else if (lane == 0) {
      abort_sh = 1;
      report_status(p.status, LR_ERR_TIMEOUT);
    }
  } else {
    // Epilogue warps, K split over the cluster: copy the valid tokens of the
    // TMEM accumulator into this CTA's partial tile.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    bool ok = mbar_wait(&accum_bar, 0, &abort_sh);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < NT / 16; c0 += kChunksPerWait) {
        if (c0 * 16 >= p.M) break;
        uint32_t r[kChunksPerWait][16];
#pragma unroll
        for (int b = 0; b < kChunksPerWait; ++b)
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + (c0 + b) * 16, r[b]);
        tmem_ld_wait();
#pragma unroll
        for (int b = 0; b < kChunksPerWait; ++b)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = (c0 + b) * 16 + j;
            if (tok < p.M) ptile[tok * kTileN + row] = __uint_as_float(r[b][j]);
          }
      }
    } else if (lane == 0) {
      abort_sh = 1;
      report_status(p.status, LR_ERR_TIMEOUT);
    }
  }

  if (S > 1) {
  __syncwarp();
  cluster_sync_all();  // every partial tile of the cluster is in shared memory

  {
    // Reduce this CTA's share of the tile -- tokens [t0, t1) x 128 rows -- over
    // the S partial tiles of the cluster, with every warp of the CTA (the
    // producer and MMA warps are done by now).
    pdl_wait();  // outputs (e.g. the residual stream) belong to earlier kernels
    const int et = threadIdx.x;
    const int t0 = split * p.M / S;
    const int t1 = (split + 1) * p.M / S;
    // The reduced slice is staged behind the partial tile (which the other
    // CTAs of the cluster are still reading) and leaves by bulk copies.
    uint8_t* stage = (kBulkEpi && P.vec_ok) ? smem + NT * kTileN * 4 : nullptr;
    if (S <= 4)
      reduce_slice<4, 4>(P, ptile, S, t0, t1, n0, et, kThreads, stage);
    else if (S <= 8)
      reduce_slice<2, 8>(P, ptile, S, t0, t1, n0, et, kThreads, stage);
    else
      reduce_slice<1, kMaxCluster>(P, ptile, S, t0, t1, n0, et, kThreads, stage);
    if (stage != nullptr) {
      fence_proxy_async_smem();
      named_bar_sync(1, kThreads);
      const int esz = out_elem_bytes(P);
      for (int t = et; t < t1 - t0; t += kThreads) store_staged_row(P, t0 + t, n0, stage + t * kTileN * esz);
      bulk_commit();
    }
  }

  __syncwarp();
  cluster_sync_all();  // no CTA leaves while others read its shared memory
  if (kBulkEpi && P.vec_ok) bulk_wait_all();  // staged rows have been written
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  return (v && *v) ? atoi(v) : dflt;
}

// Pick the number of K splits (= cluster size) of a launch: minimise, in units
// of one 128 x 64 weight tile, the per-SM share of weight tiles, plus a fixed
// cost per wave of CTAs (launch, pipeline fill, epilogue) and the cluster
// reduction, which reads S partial tiles of M tokens.  The weights were fitted
// by sweeping them on the 7B- and 70B-shaped decode steps: the reduction
// weighs more for the 256-token shape, which runs one CTA per SM.
// LR_DECODE_SPLITS forces a split count (a measurement switch).
struct CostOverride {
  bool set = false;
  double overhead = 0.0, red = 0.0;
};

// LR_DECODE_COST="overhead,red" replaces the two weights of the split cost
// model (a measurement switch, read once per process).
const CostOverride& cost_override() {
  static const CostOverride c = [] {
    CostOverride o;
    if (const char* v = getenv("LR_DECODE_COST"))
      o.set = sscanf(v, "%lf,%lf", &o.overhead, &o.red) == 2;
    return o;
  }();
  return c;
}

int choose_splits(const GemmOp* ops, int n_ops, int slots, int M) {
  static const int forced = env_int("LR_DECODE_SPLITS", 0);
  double overhead = 16.0;
  double red = slots == 1 ? 1.25 : 0.5;
  if (cost_override().set) {
    overhead = cost_override().overhead;
    red = cost_override().red;
  }
  int tiles = 0, min_nkb = 1 << 30;
  for (int g = 0; g < n_ops; ++g) {
    tiles += (ops[g].N + kTileN - 1) / kTileN;
    min_nkb = std::min(min_nkb, ops[g].K / kBK);
  }
  const int smax = std::min(kMaxCluster, min_nkb);
  if (forced > 0) return std::min(forced, smax);
  const int sms = num_sms();
  int best = 1;
  double best_cost = 1e30;
  for (int S = 1; S <= smax; ++S) {
    const long C = static_cast<long>(tiles) * S;
    int umax = 0;
    for (int g = 0; g < n_ops; ++g) umax = std::max(umax, (ops[g].K / kBK + S - 1) / S);
    const double per_sm = std::ceil(static_cast<double>(C) / sms) * umax;
    const double waves = std::ceil(static_cast<double>(C) / (static_cast<double>(sms) * slots));
    // the cluster reduction reads S partial tiles of M tokens per tile
    const double cost = per_sm + overhead * waves + (S > 1 ? red * S * M / 64.0 : 0.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

template <int NT>
lr_status configure_nt() {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       decode_smem_bytes<NT>());
  if (e != cudaSuccess) return cuda_fail(e, "decode: set smem");
  e = cudaFuncSetAttribute(decode_kernel<NT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return cuda_fail(e, "decode: allow clusters of 16");
  return LR_OK;
}

template <int NT>
lr_status launch_nt(int M, const GemmOp* ops, int n_ops, int32_t* status, cudaStream_t s) {
  constexpr int kSmem = decode_smem_bytes<NT>();
  DecodeParams prm;
  memset(&prm, 0, sizeof(prm));
  DecodeMaps maps;
  memset(&maps, 0, sizeof(maps));
  prm.M = M;
  prm.n_problems = n_ops;
  prm.status = status;
  const int S = choose_splits(ops, n_ops, DecodeCfg<NT>::kSlots, M);
  prm.splits = S;
  // Weight stages requested before griddepcontrol.wait (LR_DECODE_PREFETCH
  // overrides it: a measurement switch, read once per process).
  static const int pf = env_int("LR_DECODE_PREFETCH", -1);
  prm.prefetch = pf >= 0 ? std::min(pf, DecodeCfg<NT>::kStages) : DecodeCfg<NT>::kStages;
  // Fault injection for the timeout path, set only through lr_test_stall_producer.
  prm.stall_producer = test_stall_producer() ? 1 : 0;
  int items = 0;
  for (int g = 0; g < n_ops; ++g) {
    const GemmOp& o = ops[g];
    lr_status st = encode_map_bf16(&maps.w[g], o.W, o.N, o.K, o.ldw, kTileN);
    if (st != LR_OK) return st;
    st = encode_map_bf16(&maps.a[g], o.act, M, o.act_cols, o.ld_act, NT);
    if (st != LR_OK) return st;
    DecodeProblem& P = prm.prob[g];
    P.N = o.N;
    P.nkb = o.K / kBK;
    P.n_tiles = (o.N + kTileN - 1) / kTileN;
    P.item_begin = items;
    P.gqa_head_dim = o.gqa_head_dim;
    P.gqa_group = o.gqa_group;
    P.epi = o.epi;
    P.out = o.out;
    P.ldo = o.ldo;
    P.vec_ok = (reinterpret_cast<uintptr_t>(o.out) % 16 == 0) && (o.ldo % 8 == 0) ? 1 : 0;
    P.out_rows = o.out_rows;
    P.out_rows_limit = o.out_rows_limit;
    P.status = status;
    items += P.n_tiles * S;
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(items, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = S;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<NT>, prm, maps);
  if (e != cudaSuccess) return cuda_fail(e, "decode: launch");
  return LR_OK;
}

}  // namespace

lr_status configure_decode() {
  lr_status st;
  if ((st = configure_nt<16>()) != LR_OK) return st;
  if ((st = configure_nt<32>()) != LR_OK) return st;
  if ((st = configure_nt<64>()) != LR_OK) return st;
  if ((st = configure_nt<128>()) != LR_OK) return st;
  return configure_nt<256>();
}

lr_status launch_decode(int M, const GemmOp* ops, int n_ops, int32_t* status, cudaStream_t s) {
  if (M <= 16) return launch_nt<16>(M, ops, n_ops, status, s);
  if (M <= 32) return launch_nt<32>(M, ops, n_ops, status, s);
  if (M <= 64) return launch_nt<64>(M, ops, n_ops, status, s);
  if (M <= 128) return launch_nt<128>(M, ops, n_ops, status, s);
  return launch_nt<256>(M, ops, n_ops, status, s);
}

}  // namespace lr
