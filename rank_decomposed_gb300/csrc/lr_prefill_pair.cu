// Prefill-size GEMM on SM pairs: out[m][n] = sum_k act[m][k] * W[n][k] for
// M > 256 rows, the same operation as the one-SM prefill kernel (the two
// GEMMs of a decomposed linear, DeInfer English summary page section 2.A).
//
// A 2-CTA cluster shares one 256 x 256 output tile through tcgen05's
// cta_group::2 form: the leader CTA issues a 256-row MMA whose A operand is
// the 128 activation rows held in each CTA's shared memory and whose B
// operand is the 128 weight rows (output columns) held in each CTA's shared
// memory; each CTA's TMEM receives its own 128 rows of the 256-column result.
// Per SM this halves the weight bytes staged per k-block compared with a
// 128 x 256 tile on one SM (32 KB instead of 48 KB a stage).
//  * persistent: one pair per two SMs, tiles taken in groups of 256-row
//    bands, all of a group's bands for one weight tile before the next (see
//    PairParams), so activations and weights are both re-read from L2;
//  * a factorized linear can run as one launch: the down projection's tiles,
//    then the up projection's, each waiting on per-band completion counters;
//  * each CTA's producer loads its own halves, signalling the leader's
//    full barrier (the leader alone arms it with both CTAs' bytes);
//  * the leader's commits arrive on the empty/accumulator-full barriers of
//    both CTAs (multicast); the epilogue warps of both CTAs arrive on the
//    leader's accumulator-empty barrier;
//  * 3-stage ring of 64 KB stages, two k-blocks each, loaded by one 3-D TMA
//    operation per operand (per-operation cost, not bytes in flight, was
//    the limit of a 7-stage ring of single k-blocks); two 256-column fp32
//    accumulators.
#include <cuda_bf16.h>

#include <cstring>

#include "lr_ptx.cuh"

namespace lr {
namespace {

constexpr int kThreads = 192;
constexpr int kPM = 256;   // rows of a pair tile, 128 per CTA
constexpr int kPN = 256;   // columns of a pair tile, split 128 / 128 between the CTAs
constexpr int kHalf = 128;
constexpr int kBK = 64;
constexpr int kKB = 2;       // k-blocks per stage, loaded by one TMA operation per operand
constexpr int kStages = 3;
constexpr int kSubBytes = kHalf * kBK * 2;   // 16 KB: one k-block of 128 rows
constexpr int kABytes = kKB * kSubBytes;     // this CTA's activation rows
constexpr int kBBytes = kKB * kSubBytes;     // this CTA's weight rows
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmem = kStages * kStageBytes + 1024;  // 193 KB with the alignment pad
constexpr uint32_t kTmemCols = 512;  // two accumulators of 256 columns
constexpr uint16_t kPairMask = 0x3;  // both CTAs of the cluster

__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of `local` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(rank));
  return a;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (own or peer).
__device__ __forceinline__ void mbar_arrive_at(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Tile load into this CTA's shared memory whose completion bytes go to an
// mbarrier of either CTA of the pair (given by its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The same with a 3-D tensor map (chunked K; see encode_map_bf16_chunks).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y, int32_t z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar_cluster), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_mma_pair_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at the same shared-memory offset in every CTA of
// `mask` once the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// One GEMM of a pair launch (see GemmOp); n_tiles = ceil(N / 256).
struct PairGemm {
  int32_t N, K, n_tiles, epi;
  int32_t gqa_head_dim, gqa_group;
  int32_t act_pairs;  // a stage's two activation k-blocks are adjacent chunks: one box
  void* out;
  int64_t ldo;
  const int32_t* out_rows;
  int64_t out_rows_limit;
};

// A launch runs g[0] alone (fused == 0) or a factorized linear (fused == 1):
// g[0] writes T = act A_r (bf16) and g[1] reads T as its activations.
//
// Tile order.  The 256-row bands are taken in groups of `group` bands (the
// last group may be smaller); inside a group the tiles go output tile by
// output tile, all of the group's bands for one weight tile before the next,
// so that a weight tile is read from memory once per group while the group's
// activation rows stay in L2.  Step s of the schedule holds the first-GEMM
// tiles of group s and, when fused, the second-GEMM tiles of group s - lag,
// so that a group's T rows are read back while they are still in L2.
// band_done[b] counts the epilogue warps that have stored a first-GEMM tile
// of band b (4 per CTA, 8 per pair tile); a second-GEMM tile of band b
// starts loading once it reaches 8 * g[0].n_tiles.
struct PairParams {
  int32_t M, m_tiles;  // m_tiles = ceil(M / 256) bands
  int32_t group, n_groups;
  int32_t fused, lag;  // lag in groups, 1 <= lag <= n_groups
  PairGemm g[2];
  int32_t* band_done;
  int32_t* status;
  int32_t stall_producer;  // fault-injection hook: the TMA producers issue nothing
};

struct Unit {
  int g, band, m0, n0, nt;
};

// Position in the schedule: step and offset inside the step.
struct Sched {
  int step, off;
};

__device__ __forceinline__ int group_bands(const PairParams& p, int grp) {
  const int b = p.m_tiles - grp * p.group;
  return b < p.group ? b : p.group;
}

__device__ __forceinline__ int step_first(const PairParams& p, int s) {
  return s < p.n_groups ? group_bands(p, s) * p.g[0].n_tiles : 0;
}

__device__ __forceinline__ int step_second(const PairParams& p, int s) {
  return (p.fused && s >= p.lag && s - p.lag < p.n_groups) ? group_bands(p, s - p.lag) * p.g[1].n_tiles : 0;
}

// Move k tiles forward; false once past the last tile.
__device__ __forceinline__ bool sched_advance(const PairParams& p, Sched& it, int k) {
  const int steps = p.n_groups + (p.fused ? p.lag : 0);
  it.off += k;
  while (it.step < steps) {
    const int sz = step_first(p, it.step) + step_second(p, it.step);
    if (it.off < sz) return true;
    it.off -= sz;
    ++it.step;
  }
  return false;
}

__device__ __forceinline__ Unit sched_unit(const PairParams& p, const Sched& it) {
  const int c1 = step_first(p, it.step);
  int grp, o;
  Unit x;
  if (it.off < c1) {
    x.g = 0;
    grp = it.step;
    o = it.off;
  } else {
    x.g = 1;
    grp = it.step - p.lag;
    o = it.off - c1;
  }
  const int gb = group_bands(p, grp);
  x.band = grp * p.group + o % gb;
  x.m0 = x.band * kPM;
  x.n0 = (o / gb) * kPN;
  const int rest = p.g[x.g].N - x.n0;
  x.nt = rest < kPN ? rest : kPN;  // a multiple of 64
  return x;
}

__device__ __forceinline__ int act_col(const PairGemm& g, int kb) {
  const int k = kb * kBK;
  if (g.gqa_head_dim > 0) {
    const int head = k / g.gqa_head_dim;
    return (head / g.gqa_group) * g.gqa_head_dim + (k % g.gqa_head_dim);
  }
  return k;
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Generic-proxy global writes and async-proxy (TMA) global reads are ordered
// across this fence.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *cnt >= want (another CTA's release).  False on timeout
// or when *abort is set.
__device__ __forceinline__ bool wait_count(const int32_t* cnt, int32_t want, volatile int* abort) {
  if (ld_acquire_gpu(cnt) >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(cnt) >= want) return true;
    if ((it & 15u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PairParams p, const __grid_constant__ CUtensorMap map_a0,
                        const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_a1,
                        const __grid_constant__ CUtensorMap map_w1) {
  __shared__ __align__(8) uint64_t full_bar[kStages];  // armed and waited on in the leader only
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];  // leader only: 4 epilogue warps x 2 CTAs
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  extern __shared__ uint8_t dyn_smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank_in_cluster();  // 0: leader, issues the MMAs
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  // Both CTAs run the same code with the same static shared memory, so the
  // aligned ring sits at the same offset in each, as the pair MMA requires.
  const uint32_t raw = smem_u32(dyn_smem);
  uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 8);
    }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_barrier();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0 && !p.stall_producer) {
      prefetch_tensormap(&map_a0);
      prefetch_tensormap(&map_w0);
      if (p.fused) {
        prefetch_tensormap(&map_a1);
        prefetch_tensormap(&map_w1);
      }
      const uint64_t pol = l2_policy_evict_last();
      pdl_wait();
      const int32_t band_full = 8 * p.g[0].n_tiles;
      int it = 0;
      bool ok = true;
      Sched sc = {0, 0};
      for (bool more = sched_advance(p, sc, pair); more && ok; more = sched_advance(p, sc, npairs)) {
        const Unit x = sched_unit(p, sc);
        const PairGemm& G = p.g[x.g];
        const CUtensorMap* ma = x.g ? &map_a1 : &map_a0;
        const CUtensorMap* mw = x.g ? &map_w1 : &map_w0;
        if (x.g == 1) {
          if (!wait_count(p.band_done + x.band, band_full, &abort_sh)) {
            abort_sh = 1;
            report_status(p.status, LR_ERR_TIMEOUT);
            break;
          }
          fence_proxy_async_global();
        }
        const int arow = x.m0 + static_cast<int>(rank) * kHalf;
        const int wrow = x.n0 + static_cast<int>(rank) * (x.nt >> 1);
        const int nst = (G.K / kBK + kKB - 1) / kKB;  // stages; the last may hold one k-block
        for (int ks = 0; ks < nst; ++ks, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&empty_bar[s], ((it / kStages) & 1) ^ 1, &abort_sh)) {
            abort_sh = 1;
            report_status(p.status, LR_ERR_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          const uint32_t fb = peer_addr(smem_u32(&full_bar[s]), 0);
          if (leader) mbar_arrive_expect_tx(&full_bar[s], 2 * kStageBytes);
          // (a k-block past K, in an odd last stage, reads zeros or unused data)
          if (G.act_pairs) {
            tma_load_3d_pair(st, ma, fb, 0, arow, act_col(G, kKB * ks) / kBK, pol);
          } else {
#pragma unroll
            for (int h = 0; h < kKB; ++h)
              tma_load_3d_pair(st + h * kSubBytes, ma, fb, 0, arow, act_col(G, kKB * ks + h) / kBK, pol);
          }
          tma_load_3d_pair(st + kABytes, mw, fb, 0, wrow, kKB * ks, pol);
        }
      }
      if (abort_sh) {
        // Loads still in flight land within microseconds; do not leave
        // before they have (they write this CTA's shared memory).
        if (leader) {
          for (int i = it > kStages ? it - kStages : 0; i < it; ++i)
            mbar_wait(&full_bar[i % kStages], (i / kStages) & 1, nullptr);
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      Sched sc = {0, 0};
      for (bool more = sched_advance(p, sc, pair); more && ok; more = sched_advance(p, sc, npairs), ++lt) {
        const int b = lt & 1;
        if (!mbar_wait(&acce_bar[b], ((lt >> 1) & 1) ^ 1, &abort_sh)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + b * kPN;
        const Unit x = sched_unit(p, sc);
        const uint32_t idesc = idesc_bf16_f32(kPM, x.nt);
        const int nkb = p.g[x.g].K / kBK;
        const int nst = (nkb + kKB - 1) / kKB;
        for (int ks = 0; ks < nst; ++ks, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&full_bar[s], (it / kStages) & 1, &abort_sh)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * kStageBytes);
#pragma unroll
          for (int h = 0; h < kKB; ++h) {
            if (kKB * ks + h >= nkb) break;
            const uint64_t ad = smem_desc_sw128(sa + h * kSubBytes);
            const uint64_t bd = smem_desc_sw128(sa + kABytes + h * kSubBytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              tc_mma_pair_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (ks | h | k) != 0 ? 1u : 0u);
          }
          tc_commit_pair(&empty_bar[s], kPairMask);
        }
        tc_commit_pair(&accf_bar[b], kPairMask);
      }
      if (!ok) {
        abort_sh = 1;
        report_status(p.status, LR_ERR_TIMEOUT);
      }
      // Every MMA issued by this thread completes before either CTA frees TMEM.
      tc_commit_pair(&drain_bar, kPairMask);
      mbar_wait(&drain_bar, 0, nullptr);
    } else if (!leader && lane == 0) {
      mbar_wait(&drain_bar, 0, nullptr);
    }
  } else {
    pdl_wait();  // outputs (e.g. the residual stream) belong to earlier kernels
    const int q = warp & 3;
    const uint32_t acce0 = peer_addr(smem_u32(&acce_bar[0]), 0);
    const uint32_t acce1 = peer_addr(smem_u32(&acce_bar[1]), 0);
    int lt = 0;
    Sched sc = {0, 0};
    for (bool more = sched_advance(p, sc, pair); more; more = sched_advance(p, sc, npairs), ++lt) {
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
      const Unit x = sched_unit(p, sc);
      const PairGemm& G = p.g[x.g];
      const int m = x.m0 + static_cast<int>(rank) * kHalf + q * 32 + lane;
      const uint32_t tbase = tmem + b * kPN + (static_cast<uint32_t>(q * 32) << 16);
      int64_t orow = m < p.M ? m : -1;
      if (orow >= 0 && G.out_rows != nullptr) {
        orow = G.out_rows[m];
        if (orow < 0 || orow >= G.out_rows_limit) {
          report_status(p.status, LR_ERR_REMAP_RANGE);
          orow = -1;
        }
      }
#pragma unroll 1
      for (int c = 0; c < x.nt / 16; ++c) {
        const int n = x.n0 + c * 16;
        uint32_t r[16];
        tmem_ld16(tbase + c * 16, r);
        tmem_ld_wait();
        if (orow >= 0) {
          const int64_t off = orow * G.ldo + n;
          if (epi_is_bf16(G.epi)) {
            if (G.epi == EPI_RELU_BF16) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (__uint_as_float(r[j]) < 0.0f) r[j] = 0u;
            }
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              w[j] = static_cast<uint32_t>(f32_to_bf16_rn(__uint_as_float(r[2 * j]))) |
                     (static_cast<uint32_t>(f32_to_bf16_rn(__uint_as_float(r[2 * j + 1]))) << 16);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(G.out) + off);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          } else if (G.epi == EPI_STORE_F32) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(G.out) + off);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(G.out) + off);
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
      if (p.fused && x.g == 0) {
        // This warp's T rows are stored: publish them to the second GEMM's
        // TMA loads, which run on other SMs.
        __threadfence();
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) atomicAdd(p.band_done + x.band, 1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_at(b ? acce1 : acce0);
    }
  }

  tc_fence_before();
  __syncwarp();
  // Neither CTA leaves while its peer may still arrive on its barriers or
  // read its shared memory; then both free their TMEM together.
  cluster_barrier();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Zero the band counters of a fused launch once the previous kernel (which
// may be the previous fused launch on the same workspace) has finished.
__global__ void __launch_bounds__(256) clear_band_counters(int32_t* band_done, int n) {
  pdl_wait();
  for (int i = threadIdx.x; i < n; i += blockDim.x) band_done[i] = 0;
  pdl_launch_dependents();
}

}  // namespace

lr_status configure_prefill_pair() {
  cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return cuda_fail(e, "prefill pair: set smem");
  return LR_OK;
}

// Pairs that can be resident at once (clusters of two one-CTA-per-SM CTAs).
static int pair_slots() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms() / 2;
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

PairGemm pair_gemm(const GemmOp& op) {
  PairGemm g;
  memset(&g, 0, sizeof(g));
  g.N = op.N;
  g.K = op.K;
  g.n_tiles = (op.N + kPN - 1) / kPN;
  g.epi = op.epi;
  g.gqa_head_dim = op.gqa_head_dim;
  g.gqa_group = op.gqa_group;
  // the head broadcast keeps k-blocks 2j, 2j+1 adjacent when a head spans whole pairs
  g.act_pairs = (op.gqa_head_dim == 0 || op.gqa_head_dim % (kKB * kBK) == 0) ? 1 : 0;
  g.out = op.out;
  g.ldo = op.ldo;
  g.out_rows = op.out_rows;
  g.out_rows_limit = op.out_rows_limit;
  return g;
}

lr_status launch_pair(const PairParams& p, const GemmOp* ops, int32_t* band_done, cudaStream_t s) {
  const int n = p.fused ? 2 : 1;
  CUtensorMap ma[2], mw[2];
  for (int i = 0; i < n; ++i) {
    lr_status st = encode_map_bf16_chunks(&ma[i], ops[i].act, static_cast<uint64_t>(p.M), ops[i].act_cols,
                                          ops[i].ld_act, kHalf, p.g[i].act_pairs ? kKB : 1);
    if (st != LR_OK) return st;
    st = encode_map_bf16_chunks(&mw[i], ops[i].W, ops[i].N, ops[i].K, ops[i].ldw, kHalf, kKB);
    if (st != LR_OK) return st;
  }
  if (n == 1) {
    ma[1] = ma[0];
    mw[1] = mw[0];
  }
  PairParams q = p;
  // Fault injection for the timeout path, set only through lr_test_stall_producer.
  q.stall_producer = test_stall_producer() ? 1 : 0;
  if (p.fused) {
    // A kernel rather than a memset, so that the chain of programmatic
    // dependent launches is not broken.
    cudaLaunchConfig_t cc;
    memset(&cc, 0, sizeof(cc));
    cc.gridDim = dim3(1, 1, 1);
    cc.blockDim = dim3(256, 1, 1);
    cc.stream = s;
    cudaLaunchAttribute ca[1];
    ca[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    ca[0].val.programmaticStreamSerializationAllowed = 1;
    cc.attrs = ca;
    cc.numAttrs = pdl_enabled() ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cc, clear_band_counters, band_done, p.m_tiles);
    if (e != cudaSuccess) return cuda_fail(e, "prefill pair: clear band counters");
  }
  const int units = p.m_tiles * (p.g[0].n_tiles + (p.fused ? p.g[1].n_tiles : 0));
  const int slots = pair_slots();
  const int pairs = units < slots ? units : slots;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = 2;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_pair_kernel, q, ma[0], mw[0], ma[1], mw[1]);
  if (e != cudaSuccess) return cuda_fail(e, "prefill pair: launch");
  return LR_OK;
}

// Bands per group: the group's activation rows (256 x K bf16 per band) stay
// in L2 while its weight tiles stream past, so their total is kept near
// 32 MB; at most 16 bands.
int band_group(int K) {
  if (test_prefill_group() > 0) return test_prefill_group();
  const int64_t per_band = static_cast<int64_t>(kPM) * K * 2;
  int64_t g = (int64_t(32) << 20) / per_band;
  if (g < 1) g = 1;
  if (g > 16) g = 16;
  return static_cast<int>(g);
}

void set_groups(PairParams& p, int group) {
  if (group > p.m_tiles) group = p.m_tiles;
  p.group = group;
  p.n_groups = (p.m_tiles + group - 1) / group;
}

}  // namespace

lr_status launch_prefill_pair(int64_t M, const GemmOp& op, int32_t* status, cudaStream_t s) {
  PairParams p;
  memset(&p, 0, sizeof(p));
  p.M = static_cast<int32_t>(M);
  p.m_tiles = static_cast<int32_t>((M + kPM - 1) / kPM);
  set_groups(p, band_group(op.K));
  p.g[0] = pair_gemm(op);
  p.status = status;
  return launch_pair(p, &op, nullptr, s);
}

size_t prefill_band_counter_bytes(int64_t M) {
  return sizeof(int32_t) * static_cast<size_t>((M + kPM - 1) / kPM);
}

bool prefill_fuse_linear(int64_t M, const GemmOp& down, const GemmOp& up) {
  if (M <= kDecodeMaxRows || !prefill_fused_enabled()) return false;
  if (test_prefill_lag() > 0) return true;
  // Measured on the LLaMA-shaped projections: one launch wins for the 7B
  // ones (0.3-0.9 TFLOP at 16384 rows, +3-5 %: one launch boundary less),
  // two launches win for the 70B q/o/MLP ones (2.6-9.3 TFLOP at 32768 rows,
  // by 2-3 %), whose launches are long enough that a boundary costs little.
  const double flops = 2.0 * static_cast<double>(M) * down.N * (static_cast<double>(down.K) + up.N);
  return flops < 1.5e12;
}

lr_status launch_prefill_pair_fused(int64_t M, const GemmOp& down, const GemmOp& up, int32_t* band_done,
                                    int32_t* status, cudaStream_t s) {
  PairParams p;
  memset(&p, 0, sizeof(p));
  p.M = static_cast<int32_t>(M);
  p.m_tiles = static_cast<int32_t>((M + kPM - 1) / kPM);
  const int g1 = band_group(down.K), g2 = band_group(up.K);
  set_groups(p, g1 < g2 ? g1 : g2);
  p.fused = 1;
  p.g[0] = pair_gemm(down);
  p.g[1] = pair_gemm(up);
  // All of the down projection's tiles, then all of the up projection's:
  // measured faster than placing each group's up-projection tiles a few
  // groups after its down-projection tiles (which keeps T in L2 but runs
  // both GEMMs' tiles side by side).  A fixed lag (testing) uses that order.
  p.lag = test_prefill_lag() > 0 && test_prefill_lag() < p.n_groups ? test_prefill_lag() : p.n_groups;
  p.band_done = band_done;
  p.status = status;
  const GemmOp ops[2] = {down, up};
  return launch_pair(p, ops, band_done, s);
}

}  // namespace lr
