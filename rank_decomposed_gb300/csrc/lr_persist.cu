// One decode step of a decomposed layer stack as a single persistent kernel.
//
// The step is the graph-replay stage of DeInfer (English summary page,
// section 2.C): compact the batch's rows out of the paged pool, run every
// decomposed block on the fixed buffer, scatter the rows back.  At decode
// sizes the time is the stream of factor bytes from HBM, and a chain of
// separate kernels leaves HBM idle at every launch boundary.  Here one CTA per
// SM (a cooperative launch) walks a program built on the host:
//  * phases: gather, and per layer RMSNorm, q/k/v down, q/k/v up, o down,
//    o up (+residual), RMSNorm, gate/up down, gate/up up, SiLU-GLU, down down,
//    down up (+residual); then scatter.  A grid barrier (a global arrival
//    counter) separates phases;
//  * a GEMM phase (out[m][n] = sum_k act[m][k] W[n][k]) is cut stream-K
//    style: the phase's (tile, k-block) units are split evenly over the CTAs,
//    each CTA's range becomes segments of 128-row tiles;
//  * warp roles: a TMA producer thread issues weight tiles as far ahead as the
//    shared-memory ring allows -- across phase boundaries, since weights never
//    depend on activations -- and issues activation tiles once the previous
//    phase's barrier has passed; one thread issues tcgen05 MMAs into two TMEM
//    accumulators (swap-AB: weights on the 128-row side, tokens as N); four
//    epilogue warps drain TMEM and run the glue phases;
//  * a tile split over several CTAs is reduced cooperatively: every
//    contributor writes its fp32 partial, waits (bounded) for the others on
//    the tile's counter, then sums one slice of tokens over all partials in
//    contributor order.  Deterministic, no floating-point atomics.
// Every wait is bounded; on a timeout the kernel raises a global abort flag,
// reports LR_ERR_TIMEOUT, drains its own copies and MMAs, and returns.
#include <cuda_bf16.h>

#include <cstring>

#include "lr_ptx.cuh"

namespace lr {
namespace {

constexpr int kThreads = 224;  // w0 TMA, w1 MMA + TMEM, w2 spare, w3..w6 epilogue
constexpr int kEpiWarp0 = 3;
constexpr int kTileN = 128;
constexpr int kBK = 64;
constexpr int kWBytes = kTileN * kBK * 2;
constexpr int kSmemBudget = 200 * 1024;

template <int NT>
struct PCfg {
  static constexpr int kABytes = NT * kBK * 2;
  static constexpr int kStageBytes = kWBytes + kABytes;
  static constexpr int kStages = kSmemBudget / kStageBytes;
  static constexpr int kSmem = kStages * kStageBytes + 1024;
  static constexpr uint32_t kTmemCols = (2 * NT) < 32 ? 32 : 2 * NT;
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_volatile_i32(const int32_t* p) {
  return *reinterpret_cast<const volatile int32_t*>(p);
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

__device__ __forceinline__ void epi_sync() { named_bar_sync(1, 128); }

__device__ __forceinline__ int act_col(const PProblem& P, int kb) {
  const int k = kb * kBK;
  if (P.gqa_head_dim > 0) {
    const int head = k / P.gqa_head_dim;
    return (head / P.gqa_group) * P.gqa_head_dim + (k % P.gqa_head_dim);
  }
  return k;
}

struct Abort {
  int32_t* flag;
  int32_t* status;
  __device__ bool raised() const { return ld_volatile_i32(flag) != 0; }
  __device__ void raise() const {
    atomicExch(flag, 1);
    report_status(status, LR_ERR_TIMEOUT);
  }
};

// Spin until *ctr >= target (acquire).  Returns false on abort / timeout.
__device__ bool wait_counter(const uint32_t* ctr, uint32_t target, const Abort& ab) {
  if (ld_acquire_u32(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_u32(ctr) >= target) return true;
    __nanosleep(32);
    if ((it & 63u) == 0u) {
      if (ab.raised()) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        ab.raise();
        return false;
      }
    }
  }
}

// -------------------------------------------------------------- glue phases
__device__ void glue_gather(const PersistParams& p, const PPhase& ph, int cta, int tid) {
  const int d8 = ph.d / 8;
  const int n = min(max(ld_volatile_i32(p.n_active), 0), p.M);
  for (int i = cta; i < p.M; i += p.G) {
    const uint4* src = nullptr;
    if (i < n) {
      const int64_t j = p.remap[i];
      if (j >= 0 && j < p.pool_rows)
        src = static_cast<const uint4*>(ph.src0) + j * d8;
      else if (tid == 0)
        report_status(p.status, LR_ERR_REMAP_RANGE);
    }
    uint4* xb = static_cast<uint4*>(ph.dst1) + static_cast<int64_t>(i) * d8;
    float4* h = static_cast<float4*>(ph.dst0) + static_cast<int64_t>(i) * 2 * d8;
    for (int v0 = tid; v0 < d8; v0 += 4 * 128) {
      uint4 wv[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int v = v0 + b * 128;
        wv[b] = (src != nullptr && v < d8) ? __ldcg(src + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int v = v0 + b * 128;
        if (v >= d8) break;
        const uint4 w = wv[b];
        xb[v] = w;
        h[2 * v] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                               __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
        h[2 * v + 1] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u),
                                   __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
      }
    }
  }
}

// Row width handled by the register-resident RMSNorm: 128 threads x 16 float4.
constexpr int kNormVec = 16;

__device__ void glue_rmsnorm(const PersistParams& p, const PPhase& ph, int cta, int tid,
                             float* red) {
  const int d4 = ph.d / 4;
  for (int i = cta; i < p.M; i += p.G) {
    const float4* x = static_cast<const float4*>(ph.src0) + static_cast<int64_t>(i) * d4;
    float4 v[kNormVec];
#pragma unroll
    for (int j = 0; j < kNormVec; ++j) {
      const int idx = tid + j * 128;
      v[j] = idx < d4 ? __ldcg(x + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kNormVec; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    epi_sync();
    const float tot = (red[0] + red[1]) + (red[2] + red[3]);
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(ph.d) + ph.eps);
    uint2* y = static_cast<uint2*>(ph.dst0) + static_cast<int64_t>(i) * d4;
#pragma unroll
    for (int j = 0; j < kNormVec; ++j) {
      const int idx = tid + j * 128;
      if (idx < d4) {
        uint2 w;
        w.x = static_cast<uint32_t>(f32_to_bf16_rn(v[j].x * inv)) |
              (static_cast<uint32_t>(f32_to_bf16_rn(v[j].y * inv)) << 16);
        w.y = static_cast<uint32_t>(f32_to_bf16_rn(v[j].z * inv)) |
              (static_cast<uint32_t>(f32_to_bf16_rn(v[j].w * inv)) << 16);
        y[idx] = w;
      }
    }
    epi_sync();  // `red` is reused by the next row
  }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ uint32_t silu_mul2(uint32_t gw, uint32_t uw) {
  const float g0 = bf16_to_f32(static_cast<uint16_t>(gw & 0xFFFFu));
  const float g1 = bf16_to_f32(static_cast<uint16_t>(gw >> 16));
  const float u0 = bf16_to_f32(static_cast<uint16_t>(uw & 0xFFFFu));
  const float u1 = bf16_to_f32(static_cast<uint16_t>(uw >> 16));
  return static_cast<uint32_t>(f32_to_bf16_rn(silu_f(g0) * u0)) |
         (static_cast<uint32_t>(f32_to_bf16_rn(silu_f(g1) * u1)) << 16);
}

__device__ void glue_silu(const PersistParams& p, const PPhase& ph, int cta, int tid) {
  constexpr int kB = 4;
  const int64_t n8 = static_cast<int64_t>(p.M) * ph.d / 8;
  const int64_t stride = static_cast<int64_t>(p.G) * 128;
  const uint4* g = static_cast<const uint4*>(ph.src0);
  const uint4* u = static_cast<const uint4*>(ph.src1);
  uint4* a = static_cast<uint4*>(ph.dst0);
  for (int64_t i0 = static_cast<int64_t>(cta) * 128 + tid; i0 < n8; i0 += kB * stride) {
    uint4 gv[kB], uv[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int64_t i = i0 + b * stride;
      if (i < n8) {
        gv[b] = __ldcg(g + i);
        uv[b] = __ldcg(u + i);
      }
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int64_t i = i0 + b * stride;
      if (i < n8)
        a[i] = make_uint4(silu_mul2(gv[b].x, uv[b].x), silu_mul2(gv[b].y, uv[b].y),
                          silu_mul2(gv[b].z, uv[b].z), silu_mul2(gv[b].w, uv[b].w));
    }
  }
}

__device__ void glue_scatter(const PersistParams& p, const PPhase& ph, int cta, int tid) {
  const int d8 = ph.d / 8;
  const int n = min(max(ld_volatile_i32(p.n_active), 0), p.M);
  for (int i = cta; i < p.M; i += p.G) {
    const float4* h = static_cast<const float4*>(ph.src0) + static_cast<int64_t>(i) * 2 * d8;
    uint4* yb = static_cast<uint4*>(ph.dst1) + static_cast<int64_t>(i) * d8;
    uint4* dst = nullptr;
    if (i < n) {
      const int64_t j = p.remap[i];
      if (j >= 0 && j < p.pool_rows)
        dst = static_cast<uint4*>(ph.dst0) + j * d8;
      else if (tid == 0)
        report_status(p.status, LR_ERR_REMAP_RANGE);
    }
    for (int v0 = tid; v0 < d8; v0 += 4 * 128) {
      float4 av[4], bv[4];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int v = v0 + bb * 128;
        if (v < d8) {
          av[bb] = __ldcg(h + 2 * v);
          bv[bb] = __ldcg(h + 2 * v + 1);
        }
      }
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
      const int v = v0 + bb * 128;
      if (v >= d8) break;
      const float4 a = av[bb], b = bv[bb];
      uint4 w;
      w.x = static_cast<uint32_t>(f32_to_bf16_rn(a.x)) | (static_cast<uint32_t>(f32_to_bf16_rn(a.y)) << 16);
      w.y = static_cast<uint32_t>(f32_to_bf16_rn(a.z)) | (static_cast<uint32_t>(f32_to_bf16_rn(a.w)) << 16);
      w.z = static_cast<uint32_t>(f32_to_bf16_rn(b.x)) | (static_cast<uint32_t>(f32_to_bf16_rn(b.y)) << 16);
      w.w = static_cast<uint32_t>(f32_to_bf16_rn(b.z)) | (static_cast<uint32_t>(f32_to_bf16_rn(b.w)) << 16);
      yb[v] = w;
      if (dst) dst[v] = w;
      }
    }
  }
}

// ------------------------------------------------------------ GEMM epilogue
__device__ __forceinline__ void store1(const PProblem& P, int m, int n, float v) {
  const int64_t off = static_cast<int64_t>(m) * P.ldo + n;
  if (P.epi == EPI_STORE_BF16) {
    static_cast<uint16_t*>(P.out)[off] = f32_to_bf16_rn(v);
  } else if (P.epi == EPI_STORE_F32) {
    static_cast<float*>(P.out)[off] = v;
  } else {
    float* o = static_cast<float*>(P.out) + off;
    *o = __ldcg(o) + v;
  }
}

__device__ __forceinline__ void store4(const PProblem& P, int m, int n, float4 v) {
  const int64_t off = static_cast<int64_t>(m) * P.ldo + n;
  if (P.epi == EPI_STORE_BF16) {
    uint16_t* o = static_cast<uint16_t*>(P.out) + off;
    const uint16_t b0 = f32_to_bf16_rn(v.x), b1 = f32_to_bf16_rn(v.y);
    const uint16_t b2 = f32_to_bf16_rn(v.z), b3 = f32_to_bf16_rn(v.w);
    if (P.vec_ok) {
      *reinterpret_cast<uint2*>(o) = make_uint2(static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16),
                                                static_cast<uint32_t>(b2) | (static_cast<uint32_t>(b3) << 16));
    } else {
      o[0] = b0; o[1] = b1; o[2] = b2; o[3] = b3;
    }
    return;
  }
  float* o = static_cast<float*>(P.out) + off;
  if (P.epi == EPI_ADD_F32) {
    if (P.vec_ok) {
      const float4 h = __ldcg(reinterpret_cast<const float4*>(o));
      v.x += h.x; v.y += h.y; v.z += h.z; v.w += h.w;
    } else {
      v.x += __ldcg(o); v.y += __ldcg(o + 1); v.z += __ldcg(o + 2); v.w += __ldcg(o + 3);
    }
  }
  if (P.vec_ok) {
    *reinterpret_cast<float4*>(o) = v;
  } else {
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    persist_kernel(const __grid_constant__ PersistParams p) {
  constexpr int kStages = PCfg<NT>::kStages;
  constexpr int kABytes = PCfg<NT>::kABytes;
  constexpr uint32_t kStageBytes = PCfg<NT>::kStageBytes;
  constexpr uint32_t kTmemCols = PCfg<NT>::kTmemCols;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTileN, NT);

  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ float red_sh[4];
  extern __shared__ uint8_t dyn_smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const Abort ab{p.abort_flag, p.status};
  const int seg0 = p.seg_begin[cta];
  const int seg1 = p.seg_begin[cta + 1];

  const uint32_t raw = smem_u32(dyn_smem);
  uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* w_smem = smem;
  uint8_t* a_smem = smem + kStages * kWBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 4);
    }
    mbar_init(&drain_bar, 1);
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

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (1 thread)
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_a = l2_policy_evict_last();
      int wseg = seg0, wkb = (seg0 < seg1) ? p.segs[seg0].kb0 : 0;
      int aseg = seg0, akb = wkb;
      int pseg = seg0, pkb = wkb;   // L2 prefetch cursor, runs ahead of the W cursor
      long wi = 0, ai = 0, pi = 0;
      uint32_t seen = 0;
      uint64_t t_last = globaltimer_ns();
      bool ok = true;
      uint32_t idle = 0;
      while (aseg < seg1) {
        bool did = false;
        // 1. activation tiles of stages whose weight tile is issued, as far as
        //    the last observed barrier count allows (no polling here)
        while (ai < wi) {
          const PSeg sg = p.segs[aseg];
          if (seen < static_cast<uint32_t>(sg.phase) * static_cast<uint32_t>(p.G)) break;
          const PProblem& P = p.probs[sg.prob];
          const int s = static_cast<int>(ai % kStages);
          tma_load_2d(a_smem + s * kABytes, p.maps + P.amap, &full_bar[s], act_col(P, akb), 0, pol_a);
          ++ai;
          if (++akb == sg.kb1) {
            ++aseg;
            if (aseg < seg1) akb = p.segs[aseg].kb0;
          }
          did = true;
        }
        // 2. weight tiles into every free slot: they never wait for a barrier
        while (wseg < seg1) {
          const int s = static_cast<int>(wi % kStages);
          if (!mbar_try_wait(&empty_bar[s], static_cast<uint32_t>(((wi / kStages) & 1) ^ 1))) break;
          const PSeg sg = p.segs[wseg];
          const PProblem& P = p.probs[sg.prob];
          mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
          tma_load_2d(w_smem + s * kWBytes, p.maps + P.wmap, &full_bar[s], wkb * kBK,
                      sg.tile * kTileN, pol_w);
          ++wi;
          if (++wkb == sg.kb1) {
            ++wseg;
            if (wseg < seg1) wkb = p.segs[wseg].kb0;
          }
          did = true;
        }
        // 2b. L2 prefetch of weight tiles further ahead: HBM keeps streaming
        //     while this phase's barrier and reductions complete
        if (pi < wi) {
          pi = wi;
          pseg = wseg;
          pkb = wkb;
        }
        while (pseg < seg1 && pi < wi + p.pf_ahead) {
          const PSeg sg = p.segs[pseg];
          tma_prefetch_l2_2d(p.maps + p.probs[sg.prob].wmap, pkb * kBK, sg.tile * kTileN);
          ++pi;
          if (++pkb == sg.kb1) {
            ++pseg;
            if (pseg < seg1) pkb = p.segs[pseg].kb0;
          }
          did = true;
        }
        if (did) {
          idle = 0;
          t_last = 0;
          continue;
        }
        // 3. nothing to issue: refresh the barrier count (one L2 round trip)
        //    if an activation tile is waiting for it, else back off
        if (ai < wi) {
          const uint32_t v = ld_acquire_u32(p.gbar);
          if (v != seen) {
            seen = v;
            fence_proxy_async();
            continue;
          }
        }
        if (++idle > 4) __nanosleep(32);
        if ((idle & 15u) == 0u) {
          const uint64_t now = globaltimer_ns();
          if (t_last == 0) t_last = now;
          if (ab.raised()) { ok = false; break; }
          if (now - t_last > kWaitLimitNs) { ab.raise(); ok = false; break; }
        }
      }
      if (!ok) {
        // A stage whose weight tile is issued also expects its activation tile:
        // issue the missing ones (the data no longer matters) so every stage
        // can complete, then let the copies in flight land before exiting.
        while (ai < wi) {
          const PSeg sg = p.segs[aseg];
          const PProblem& P = p.probs[sg.prob];
          const int s = static_cast<int>(ai % kStages);
          tma_load_2d(a_smem + s * kABytes, p.maps + P.amap, &full_bar[s], act_col(P, akb), 0, pol_a);
          ++ai;
          if (++akb == sg.kb1) {
            ++aseg;
            if (aseg < seg1) akb = p.segs[aseg].kb0;
          }
        }
        for (long i = wi > kStages ? wi - kStages : 0; i < wi; ++i)
          mbar_wait(&full_bar[i % kStages], static_cast<uint32_t>((i / kStages) & 1), nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer (1 thread)
    if (lane == 0) {
      long it = 0;
      int k = 0;
      bool ok = true;
      for (int sidx = seg0; sidx < seg1 && ok; ++sidx, ++k) {
        const PSeg sg = p.segs[sidx];
        const int b = k & 1;
        if (!mbar_wait(&acce_bar[b], static_cast<uint32_t>(((k >> 1) & 1) ^ 1), ab.flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + b * NT;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
          const int s = static_cast<int>(it % kStages);
          if (!mbar_wait(&full_bar[s], static_cast<uint32_t>((it / kStages) & 1), ab.flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(smem_u32(w_smem + s * kWBytes));
          const uint64_t bd = smem_desc_sw128(smem_u32(a_smem + s * kABytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (kb != sg.kb0 || kk != 0) ? 1u : 0u);
          tc_commit(&empty_bar[s]);
        }
        if (ok) tc_commit(&accf_bar[b]);
      }
      if (!ok && !ab.raised()) ab.raise();
      tc_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, nullptr);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------- epilogue + glue (4 warps, 128 threads)
    const int tid = threadIdx.x - kEpiWarp0 * 32;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    __shared__ int flag_sh;
    __shared__ int vote_sh[2][4];
    int sidx = seg0, k = 0;
    bool ok = true;
    for (int ph = 0; ph < p.n_phases && ok; ++ph) {
      const PPhase phase = p.phases[ph];
      // The barrier is one cumulative arrival counter, so "count >= ph * G"
      // means "phases 0 .. ph-1 are complete" only if no CTA arrives at a
      // barrier before the previous one has completed: every CTA waits here,
      // whether or not it has work in this phase.
      const uint32_t need = static_cast<uint32_t>(ph) * static_cast<uint32_t>(p.G);
      if (tid == 0) flag_sh = wait_counter(p.gbar, need, ab) ? 1 : 0;
      epi_sync();
      if (!flag_sh) { ok = false; break; }
      if (phase.kind != PH_GEMM) {
        if (phase.kind == PH_GATHER) glue_gather(p, phase, cta, tid);
        else if (phase.kind == PH_RMSNORM) glue_rmsnorm(p, phase, cta, tid, red_sh);
        else if (phase.kind == PH_SILU) glue_silu(p, phase, cta, tid);
        else glue_scatter(p, phase, cta, tid);
      } else {
        // Pass 1: drain every segment of the phase as its accumulator
        // completes -- whole tiles straight to the output, split tiles as
        // partials followed by an arrival on the tile's counter.
        const int sbeg = sidx;
        for (; sidx < seg1 && p.segs[sidx].phase == ph; ++sidx, ++k) {
          const PSeg sg = p.segs[sidx];
          const PProblem& P = p.probs[sg.prob];
          const int b = k & 1;
          // The four warps must agree before any of them leaves the loop:
          // a warp that left would strand the others at a named barrier.
          bool got = mbar_wait(&accf_bar[b], static_cast<uint32_t>((k >> 1) & 1), ab.flag);
          got = __all_sync(0xffffffffu, got);
          if (lane == 0) vote_sh[k & 1][q] = got ? 1 : 0;
          epi_sync();
          got = vote_sh[k & 1][0] && vote_sh[k & 1][1] && vote_sh[k & 1][2] && vote_sh[k & 1][3];
          if (!got) { ok = false; break; }
          tc_fence_after();
          const uint32_t tb = tmem + b * NT + (static_cast<uint32_t>(q * 32) << 16);
          const int n = sg.tile * kTileN + row;
          float* part = p.partials + static_cast<int64_t>(sg.slot + sg.j) * NT * kTileN;
#pragma unroll 1
          for (int c = 0; c < NT / 16 && c * 16 < p.M; ++c) {
            uint32_t r[16];
            tmem_ld16(tb + c * 16, r);
            tmem_ld_wait();
            if (sg.nc == 1) {
              if (n < P.N) {
                if (P.epi == EPI_ADD_F32) {
                  // issue the 16 residual loads before any store
                  float hv[16];
                  float* o = static_cast<float*>(P.out) + n;
#pragma unroll
                  for (int jj = 0; jj < 16; ++jj)
                    hv[jj] = (c * 16 + jj < p.M) ? __ldcg(o + static_cast<int64_t>(c * 16 + jj) * P.ldo) : 0.f;
#pragma unroll
                  for (int jj = 0; jj < 16; ++jj)
                    if (c * 16 + jj < p.M) o[static_cast<int64_t>(c * 16 + jj) * P.ldo] = hv[jj] + __uint_as_float(r[jj]);
                } else {
#pragma unroll
                  for (int jj = 0; jj < 16; ++jj)
                    if (c * 16 + jj < p.M) store1(P, c * 16 + jj, n, __uint_as_float(r[jj]));
                }
              }
            } else {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                if (c * 16 + jj < p.M) __stcg(part + (c * 16 + jj) * kTileN + row, __uint_as_float(r[jj]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce_bar[b]);
          if (sg.nc > 1) {
            __threadfence();
            epi_sync();
            if (tid == 0) atomicAdd(p.counters + sg.ctr, 1u);
          }
        }
        if (!ok) break;
        // Pass 2: for every split tile, wait (bounded) until all contributors
        // have written their partials, then sum this contributor's slice of
        // tokens over the partials in contributor order.
        for (int s2 = sbeg; s2 < sidx; ++s2) {
          const PSeg sg = p.segs[s2];
          if (sg.nc == 1) continue;
          const PProblem& P = p.probs[sg.prob];
          if (tid == 0)
            flag_sh = wait_counter(p.counters + sg.ctr, static_cast<uint32_t>(sg.nc), ab) ? 1 : 0;
          epi_sync();
          if (!flag_sh) { ok = false; break; }
          const int t0 = sg.j * p.M / sg.nc, t1 = (sg.j + 1) * p.M / sg.nc;
          const float* base = p.partials + static_cast<int64_t>(sg.slot) * NT * kTileN;
          const int nch = (t1 - t0) * (kTileN / 4);
          for (int cidx = tid; cidx < nch; cidx += 128) {
            const int tok = t0 + cidx / (kTileN / 4);
            const int r4 = (cidx % (kTileN / 4)) * 4;
            if (sg.tile * kTileN + r4 >= P.N) continue;
            const float* src = base + tok * kTileN + r4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j0 = 0; j0 < sg.nc; j0 += 8) {
              float4 v[8];
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
                if (j0 + jj < sg.nc)
                  v[jj] = __ldcg(reinterpret_cast<const float4*>(src + static_cast<int64_t>(j0 + jj) * NT * kTileN));
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
                if (j0 + jj < sg.nc) {
                  if (j0 + jj == 0) {
                    acc = v[0];
                  } else {
                    acc.x += v[jj].x; acc.y += v[jj].y; acc.z += v[jj].z; acc.w += v[jj].w;
                  }
                }
            }
            store4(P, tok, sg.tile * kTileN + r4, acc);
          }
          epi_sync();  // flag_sh is reused by the next tile
        }
        if (!ok) break;
      }
      // arrive at the barrier that ends phase `ph`
      fence_proxy_async();
      __threadfence();
      epi_sync();
      if (tid == 0) atomicAdd(p.gbar, 1u);
    }
    if (!ok && tid == 0 && !ab.raised()) ab.raise();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NT>
lr_status configure_nt() {
  cudaError_t e = cudaFuncSetAttribute(persist_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PCfg<NT>::kSmem);
  if (e != cudaSuccess) return cuda_fail(e, "persist: set smem");
  return LR_OK;
}

template <int NT>
lr_status launch_nt(const PersistParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(p.G, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = PCfg<NT>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, persist_kernel<NT>, p);
  if (e != cudaSuccess) return cuda_fail(e, "persist: launch");
  return LR_OK;
}

}  // namespace

int persist_max_rows() { return 256; }
int persist_grid() { return num_sms(); }

lr_status configure_persist() {
  lr_status st;
  if ((st = configure_nt<16>()) != LR_OK) return st;
  if ((st = configure_nt<32>()) != LR_OK) return st;
  if ((st = configure_nt<64>()) != LR_OK) return st;
  if ((st = configure_nt<128>()) != LR_OK) return st;
  return configure_nt<256>();
}

lr_status launch_persist(const PersistParams& p, int nt, void* zero_base, size_t zero_bytes,
                         cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(zero_base, 0, zero_bytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "persist: memset");
  switch (nt) {
    case 16: return launch_nt<16>(p, s);
    case 32: return launch_nt<32>(p, s);
    case 64: return launch_nt<64>(p, s);
    case 128: return launch_nt<128>(p, s);
    default: return launch_nt<256>(p, s);
  }
}

}  // namespace lr
