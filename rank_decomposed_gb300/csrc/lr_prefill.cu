// Prefill-size GEMM: out[m][n] = sum_k act[m][k] * W[n][k] for M > 256 rows.
//
// Used twice per decomposed linear (DeInfer, English summary page section
// 2.A): T = X A_r (act = X, W = A_r^T) and Y = T B_r (act = T, W = B_r^T).
// Here the tensor pipe is the bound.  Design for sm_103a:
//  * persistent kernel, one CTA per SM, 128 x 256 output tiles walked with the
//    N tiles of one M band adjacent so the band's activation rows are read
//    from HBM once and reused from L2;
//  * warp-specialised: one TMA producer thread, one tcgen05 MMA thread and
//    four epilogue warps;
//  * 4-stage ring of 48 KB stages (128x64 activation + 256x64 weight, 128-byte
//    swizzle);
//  * two 256-column fp32 accumulators in TMEM, so the epilogue of one tile
//    overlaps the MMAs of the next;
//  * paged activations (KV reconstruction, English summary page section
//    2.C): a 128-row activation tile is eight 16-row blocks of a paged pool,
//    each loaded by its own TMA box at its block's row; a 16-row box lands on
//    a 2 KB boundary, so the 128-byte swizzle of the stage is the same as
//    that of one 128-row box.
#include <cuda_bf16.h>

#include <cstring>

#include "lr_ptx.cuh"

namespace lr {
namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmem = kStages * kStageBytes + 1024;
constexpr uint32_t kTmemCols = 512;      // two accumulators of 256 columns

__device__ __forceinline__ int act_col(const PrefillParams& p, int kb) {
  const int k = kb * kBK;
  if (p.gqa_head_dim > 0) {
    const int head = k / p.gqa_head_dim;
    return (head / p.gqa_group) * p.gqa_head_dim + (k % p.gqa_head_dim);
  }
  return k;
}

__device__ __forceinline__ void tile_coords(const PrefillParams& p, int t, int& m0, int& n0) {
  m0 = (t / p.n_tiles) * kBM;
  n0 = (t % p.n_tiles) * kBN;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_w) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN);
  // The last N tile of a width that is not a multiple of kBN (N is a multiple
  // of 64) runs a narrower MMA instead of multiplying zero-filled rows.
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  extern __shared__ uint8_t dyn_smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = p.K / kBK;
  const int tiles = p.m_tiles * p.n_tiles;

  const uint32_t raw = smem_u32(dyn_smem);
  uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(&drain_bar, 1);
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
    if (lane == 0) {
      prefetch_tensormap(&map_a);
      prefetch_tensormap(&map_w);
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_last();
      pdl_wait();
      const bool paged = p.blocks != nullptr;
      const int nb = paged ? *reinterpret_cast<const volatile int32_t*>(p.n_blocks) : 0;
      // paged: the block ids of a tile's eight blocks, loaded one tile ahead
      constexpr int kTB = kBM / kPageRows;
      int32_t bnext[kTB];
      auto load_ids = [&](int t) {
#pragma unroll
        for (int j = 0; j < kTB; ++j) {
          const int i = (t / p.n_tiles) * kTB + j;
          bnext[j] = (t < tiles && i < nb && i * kPageRows < p.M) ? p.blocks[i] : -1;
        }
      };
      if (paged) load_ids(blockIdx.x);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        int m0, n0;
        tile_coords(p, t, m0, n0);
        // paged: the pool row of each block (pool_blocks * 16, past the pool,
        // for padding and bad entries: it reads as zeros)
        int32_t brow[kTB];
        if (paged) {
#pragma unroll
          for (int j = 0; j < kTB; ++j) {
            int64_t b = bnext[j];
            if (b >= p.pool_blocks || (b < 0 && m0 / kPageRows + j < nb && (m0 / kPageRows + j) * kPageRows < p.M)) {
              report_status(p.status, LR_ERR_REMAP_RANGE);
              b = -1;
            }
            brow[j] = static_cast<int32_t>((b < 0 ? p.pool_blocks : b) * kPageRows);
          }
          load_ids(t + gridDim.x);
        }
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&empty_bar[s], ((it / kStages) & 1) ^ 1, &abort_sh)) {
            abort_sh = 1;
            report_status(p.status, LR_ERR_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
          if (paged) {
#pragma unroll
            for (int j = 0; j < kBM / kPageRows; ++j)
              tma_load_2d(st + j * kPageRows * kBK * 2, &map_a, &full_bar[s], kb * kBK, brow[j], pol_a);
          } else {
            tma_load_2d(st, &map_a, &full_bar[s], act_col(p, kb), m0, pol_a);
          }
          tma_load_2d(st + kABytes, &map_w, &full_bar[s], kb * kBK, n0, pol_w);
        }
      }
      if (!ok) {
        for (int i = it > kStages ? it - kStages : 0; i < it; ++i)
          mbar_wait(&full_bar[i % kStages], (i / kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++lt) {
        const int b = lt & 1;
        if (!mbar_wait(&acce_bar[b], ((lt >> 1) & 1) ^ 1, &abort_sh)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + b * kBN;
        int m0t, n0t;
        tile_coords(p, t, m0t, n0t);
        const uint32_t idesc = p.N - n0t >= kBN ? kIdesc : idesc_bf16_f32(kBM, p.N - n0t);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&full_bar[s], (it / kStages) & 1, &abort_sh)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * kStageBytes);
          const uint64_t ad = smem_desc_sw128(sa);
          const uint64_t bd = smem_desc_sw128(sa + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          tc_commit(&empty_bar[s]);
        }
        tc_commit(&accf_bar[b]);
      }
      if (!ok) {
        abort_sh = 1;
        report_status(p.status, LR_ERR_TIMEOUT);
      }
      // Every MMA issued by this thread completes before TMEM is released.
      tc_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, nullptr);
    }
  } else {
    pdl_wait();  // outputs (e.g. the residual stream) belong to earlier kernels
    const int q = warp & 3;
    int lt = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++lt) {
      const int b = lt & 1;
      bool ok = mbar_wait(&accf_bar[b], (lt >> 1) & 1, &abort_sh);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          abort_sh = 1;
          report_status(p.status, LR_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      int m0, n0;
      tile_coords(p, t, m0, n0);
      const int m = m0 + q * 32 + lane;
      const uint32_t tbase = tmem + b * kBN + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < kBN / 16; ++c) {
        const int n = n0 + c * 16;
        if (n >= p.N) break;  // N is a multiple of 64: whole chunks are in or out
        uint32_t r[16];
        tmem_ld16(tbase + c * 16, r);
        tmem_ld_wait();
        int64_t orow = m < p.M ? m : -1;
        if (orow >= 0 && p.out_rows != nullptr) {
          orow = p.out_rows[m];
          if (orow < 0 || orow >= p.out_rows_limit) {
            if (c == 0) report_status(p.status, LR_ERR_REMAP_RANGE);
            orow = -1;
          }
        }
        if (orow >= 0) {
          const int64_t off = orow * p.ldo + n;
          if (epi_is_bf16(p.epi)) {
            if (p.epi == EPI_RELU_BF16) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (__uint_as_float(r[j]) < 0.0f) r[j] = 0u;
            }
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              w[j] = static_cast<uint32_t>(f32_to_bf16_rn(__uint_as_float(r[2 * j]))) |
                     (static_cast<uint32_t>(f32_to_bf16_rn(__uint_as_float(r[2 * j + 1]))) << 16);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + off);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          } else if (p.epi == EPI_STORE_F32) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.out) + off);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float4 v = dst[j];
              v.x += __uint_as_float(r[4 * j]);
              v.y += __uint_as_float(r[4 * j + 1]);
              v.z += __uint_as_float(r[4 * j + 2]);
              v.w += __uint_as_float(r[4 * j + 3]);
              dst[j] = v;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[b]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

lr_status configure_prefill() {
  cudaError_t e =
      cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return cuda_fail(e, "prefill: set smem");
  return LR_OK;
}

lr_status launch_prefill_impl(int64_t M, const GemmOp& op, const int32_t* blocks, const int32_t* n_blocks,
                              int64_t pool_blocks, int32_t* status, cudaStream_t s) {
  PrefillParams p;
  memset(&p, 0, sizeof(p));
  p.blocks = blocks;
  p.n_blocks = n_blocks;
  p.pool_blocks = pool_blocks;
  p.M = static_cast<int32_t>(M);
  p.N = op.N;
  p.K = op.K;
  p.m_tiles = static_cast<int32_t>((M + kBM - 1) / kBM);
  p.n_tiles = (op.N + kBN - 1) / kBN;
  p.epi = op.epi;
  p.gqa_head_dim = op.gqa_head_dim;
  p.gqa_group = op.gqa_group;
  p.out = op.out;
  p.ldo = op.ldo;
  p.status = status;
  p.out_rows = op.out_rows;
  p.out_rows_limit = op.out_rows_limit;
  CUtensorMap ma, mw;
  // paged: the map spans the pool, one 16-row block per box
  lr_status st = blocks != nullptr
                     ? encode_map_bf16(&ma, op.act, static_cast<uint64_t>(pool_blocks) * kPageRows, op.act_cols,
                                       op.ld_act, kPageRows)
                     : encode_map_bf16(&ma, op.act, static_cast<uint64_t>(M), op.act_cols, op.ld_act, kBM);
  if (st != LR_OK) return st;
  st = encode_map_bf16(&mw, op.W, op.N, op.K, op.ldw, kBN);
  if (st != LR_OK) return st;
  const int tiles = p.m_tiles * p.n_tiles;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_kernel, p, ma, mw);
  if (e != cudaSuccess) return cuda_fail(e, "prefill: launch");
  return LR_OK;
}

lr_status launch_prefill(int64_t M, const GemmOp& op, int32_t* status, cudaStream_t s) {
  return launch_prefill_impl(M, op, nullptr, nullptr, 0, status, s);
}

lr_status launch_prefill_paged(int64_t M, const GemmOp& op, const int32_t* blocks, const int32_t* n_blocks,
                               int64_t pool_blocks, int32_t* status, cudaStream_t s) {
  return launch_prefill_impl(M, op, blocks, n_blocks, pool_blocks, status, s);
}

}  // namespace lr
