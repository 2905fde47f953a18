// out_tc.cu -- the output projection of up to 64 tokens in one launch on
// sm_103a tensor cores: o_i = W^UV_i o~_i per head ([kasblo] "V側は、小さな表現
// の加重和を先に求める") and u = W^O [o_1; ...; o_n_h] ([qiita] "Attention 計算").
//
// u needs every head's o_i, so the launch has two phases with one hand-off
// through global memory between them:
// * the grid is the W^O product's: 128-row tiles of u (grid y) with the
//   d_h n_h-long k range split over the CTAs of a cluster (grid x), one CTA
//   per SM, every CTA resident at once (checked on the host);
// * phase 1: CTA c also owns heads c, c + ctas, ...: o_i = W^UV_i o~_i (M = the
//   head's d_h = 128 rows, K = d_c) into TMEM, rounded once to bf16 into a
//   scratch [n_tok, n_h d_h] -- the same rounding as the separate route;
// * each CTA then adds one to a counter of the handle; the W^O loads of a
//   CTA's o columns wait (bounded) until every CTA has added its one, while
//   the first W^O weight tiles (which need nothing) are already in flight;
// * phase 2: the CTA's share of u's tile (TMEM), the cluster's fp32 partial
//   tiles summed through distributed shared memory in rank order, bf16 u.
// The last CTA to finish sets the counters back to zero for the next call.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kOm = 128;                  // weight rows per tile
constexpr int kOk = 64;                   // k per stage
constexpr int kOn = 64;                   // token columns (at most 64 tokens)
constexpr uint32_t kOA = kOm * kOk * 2;   // 16 KB weight tile
constexpr uint32_t kOB = kOn * kOk * 2;   // 8 KB token tile
constexpr uint32_t kOStage = kOA + kOB;
constexpr int kOStages = 8;
constexpr uint32_t kOOffBars = kOStages * kOStage;
constexpr uint32_t kOOffStg = kOOffBars + 256;         // phase 1: 4 KB per epilogue warp, [token][32 columns]
constexpr uint32_t kOSmem = kOOffStg + 4 * kOn * 64 + 1024;
constexpr int kOThreads = 256;
constexpr int kOMaxHeadsPerCta = 2;
constexpr int kOSplit = 3;                // cluster size along the k range of W^O
static_assert(kOStages * kOStage >= kOn * kOm * 4, "the reduction buffer reuses the stages");

struct OutMaps {
  CUtensorMap wuv;   // W^UV [n_h d_h, d_c]
  CUtensorMap olat;  // o~ [n_tok, n_h d_c]
  CUtensorMap wo;    // W^O [d_model, n_h d_h]
  CUtensorMap obuf;  // o [n_tok, n_h d_h] (the scratch phase 1 writes)
};

struct OutParams {
  int n_tok, n_h, ctas;
  int uv_blocks;      // d_c / 64
  int o_blocks;       // n_h d_h / 64
  int d_model;
  __nv_bfloat16* obuf;
  __nv_bfloat16* u;
  unsigned int* counters;  // [0] CTAs past phase 1, [1] CTAs finished (reset by the last)
  int* status;
  long long wait_limit;
};

struct OutBars {
  uint64_t full[kOStages], empty[kOStages], p1_done[kOMaxHeadsPerCta], p2_done, drain;
  uint32_t tmem;
  int abort;
};

// Bounded wait (sites: producer 1 stage free, 2 every CTA past phase 1; MMA
// warp 3 stage landed; epilogue warps 4 o_i in TMEM, 5 u tile in TMEM).
__device__ __forceinline__ bool ot_wait(uint64_t* bar, uint32_t parity, const OutParams& p, OutBars* bs, int site) {
  if (mbar_test_wait(bar, parity)) return true;
  for (long long i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= p.wait_limit || *reinterpret_cast<volatile int*>(&bs->abort)) {
      if (i >= p.wait_limit) report_site(p.status, site, -1);
      else report(p.status, MLA_ERR_DEVICE_TIMEOUT);
      atomicExch(&bs->abort, 1);
      return false;
    }
  }
}
__device__ __forceinline__ bool ot_wait_warp(uint64_t* bar, uint32_t parity, const OutParams& p, OutBars* bs,
                                             int site) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = ot_wait(bar, parity, p, bs, site);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* a) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

__global__ void __cluster_dims__(kOSplit, 1, 1) __launch_bounds__(kOThreads, 1)
    out_kernel(const __grid_constant__ OutMaps maps, const OutParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  OutBars* bs = reinterpret_cast<OutBars*>(smem + kOOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = static_cast<int>(cluster_ctarank());
  const int tile = blockIdx.y;                                  // u rows [128 tile, +128)
  const int cta = static_cast<int>(blockIdx.y) * kOSplit + split;
  int n_heads = 0;                                              // heads cta, cta + ctas, ...
  for (int hd = cta; hd < p.n_h && n_heads < kOMaxHeadsPerCta; hd += p.ctas) ++n_heads;
  const int kb0 = static_cast<int>(static_cast<long long>(split) * p.o_blocks / kOSplit);
  const int kb1 = static_cast<int>(static_cast<long long>(split + 1) * p.o_blocks / kOSplit);
  const int n1 = n_heads * p.uv_blocks, n2 = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kOStages; ++s) {
      mbar_init(&bs->full[s], 1);
      mbar_init(&bs->empty[s], 1);
    }
    for (int h = 0; h < kOMaxHeadsPerCta; ++h) mbar_init(&bs->p1_done[h], 1);
    mbar_init(&bs->p2_done, 1);
    mbar_init(&bs->drain, 1);
    bs->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bs->tmem, 256);  // o_i of up to two heads (64 columns each) | u partial (64)
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bs->tmem;
  constexpr uint32_t kTmemU = 128;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.wuv);
      tma_prefetch_desc(&maps.olat);
      tma_prefetch_desc(&maps.wo);
      tma_prefetch_desc(&maps.obuf);
      // the step's last weight reads: evict-first, also on the lines an L2
      // prefetch brought in, so that none of them outlives the step
      const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
      auto load_w = [&](int i, uint8_t* st, uint64_t* bar) {
        if (i < n1) {
          const int hd = cta + (i / p.uv_blocks) * p.ctas, kb = i % p.uv_blocks;
          tma_load_2d_hint(st, &maps.wuv, bar, kb * kOk, hd * kOm, pol_w);
        } else {
          tma_load_2d_hint(st, &maps.wo, bar, (kb0 + i - n1) * kOk, tile * kOm, pol_w);
        }
      };
      auto load_x = [&](int i, uint8_t* st, uint64_t* bar) {
        if (i < n1) {
          const int hd = cta + (i / p.uv_blocks) * p.ctas, kb = i % p.uv_blocks;
          tma_load_2d_hint(st + kOA, &maps.olat, bar, hd * p.uv_blocks * kOk + kb * kOk, 0, pol_x);
        } else {
          tma_load_2d_hint(st + kOA, &maps.obuf, bar, (kb0 + i - n1) * kOk, 0, pol_x);
        }
      };
      const int total = n1 + n2;
      // the first stages' weights before the wait for the previous kernel
      const int early = total < kOStages ? total : kOStages;
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx(&bs->full[i], kOStage);
        load_w(i, smem + i * kOStage, &bs->full[i]);
      }
      pdl_wait();
      bool ok = true;
      int it = 0;
      for (; it < early && it < n1; ++it) load_x(it, smem + it * kOStage, &bs->full[it]);
      // The rest of phase 1 (weights and o~), then the first stages of phase 2
      // with their weights only: their o columns wait for every CTA's phase 1.
      int w_issued = early, x_issued = it;
      const int w_ahead = n1 + kOStages < total ? n1 + kOStages : total;
      for (; ok && w_issued < w_ahead; ++w_issued) {
        const int s = w_issued % kOStages;
        if (!(ok = ot_wait(&bs->empty[s], ((w_issued / kOStages) - 1) & 1, p, bs, 1))) break;
        mbar_arrive_expect_tx(&bs->full[s], kOStage);
        load_w(w_issued, smem + s * kOStage, &bs->full[s]);
        if (w_issued < n1) {
          load_x(w_issued, smem + s * kOStage, &bs->full[s]);
          x_issued = w_issued + 1;
        }
      }
      if (ok && n2 > 0) {
        // every CTA's o_i is in the scratch
        for (long long i = 0;; ++i) {
          if (ld_acquire_gpu(p.counters) >= static_cast<unsigned int>(p.ctas)) break;
          if (i >= p.wait_limit || *reinterpret_cast<volatile int*>(&bs->abort)) {
            if (i >= p.wait_limit) report_site(p.status, 2, -1);
            atomicExch(&bs->abort, 1);
            ok = false;
            break;
          }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");  // the TMA reads what other CTAs stored
      }
      // the o columns of the stages whose weights went ahead (after a timeout
      // too, so that every issued copy completes before the CTA exits)
      for (int i = x_issued > n1 ? x_issued : n1; i < w_issued; ++i)
        load_x(i, smem + (i % kOStages) * kOStage, &bs->full[i % kOStages]);
      for (; ok && w_issued < total; ++w_issued) {
        const int s = w_issued % kOStages;
        if (!(ok = ot_wait(&bs->empty[s], ((w_issued / kOStages) - 1) & 1, p, bs, 1))) break;
        mbar_arrive_expect_tx(&bs->full[s], kOStage);
        load_w(w_issued, smem + s * kOStage, &bs->full[s]);
        load_x(w_issued, smem + s * kOStage, &bs->full[s]);
      }
      if (!ok) {
        // every issued copy must land before the CTA may exit
        for (int k = w_issued > kOStages ? w_issued - kOStages : 0; k < w_issued; ++k)
          for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->full[k % kOStages], (k / kOStages) & 1); ++i) {
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kOm, kOn, false, false);
    bool ok = true;
    int it = 0;
    for (int hs = 0; hs < n_heads && ok; ++hs) {
      for (int kb = 0; kb < p.uv_blocks && ok; ++kb, ++it) {
        const int s = it % kOStages;
        if (!(ok = ot_wait_warp(&bs->full[s], (it / kOStages) & 1, p, bs, 3))) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + s * kOStage);
        mma_ss_kblock_elect<2, 2>(tmem + hs * kOn, smem_desc(a, 16, 1024, kSwizzle128B),
                                  smem_desc(a + kOA, 16, 1024, kSwizzle128B), idesc, kb > 0 ? 1u : 0u);
        mma_commit_elect(&bs->empty[s]);
      }
      if (ok) mma_commit_elect(&bs->p1_done[hs]);
    }
    for (int kb = 0; kb < n2 && ok; ++kb, ++it) {
      const int s = it % kOStages;
      if (!(ok = ot_wait_warp(&bs->full[s], (it / kOStages) & 1, p, bs, 3))) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * kOStage);
      mma_ss_kblock_elect<2, 2>(tmem + kTmemU, smem_desc(a, 16, 1024, kSwizzle128B),
                                smem_desc(a + kOA, 16, 1024, kSwizzle128B), idesc, kb > 0 ? 1u : 0u);
      mma_commit_elect(&bs->empty[s]);
    }
    if (ok) mma_commit_elect(&bs->p2_done);
    if (!ok) {
      mma_commit_elect(&bs->drain);
      for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->drain, 0); ++i) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue warps
    const int w = warp - 4, r = 32 * w + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * w) << 16;
    if (lane == 0) pdl_wait();  // the scratch and u may still be read by the previous kernel
    __syncwarp();
    bool ok = true;
    // o_i column 32 w + lane of every token, through this warp's 4 KB of
    // staging ([token][32 columns]), then as 16-byte pieces (the 64-byte run
    // of each token's row this warp owns): 8 stores a lane, not 64 two-byte ones
    uint8_t* stg = smem + kOOffStg + w * (kOn * 64);
    for (int hs = 0; hs < n_heads && ok; ++hs) {
      if (!(ok = ot_wait_warp(&bs->p1_done[hs], 0, p, bs, 4))) break;
      tc_fence_after();
      uint32_t v[kOn];
      tmem_ld32(tmem + lanes + hs * kOn, v);
      tmem_ld32(tmem + lanes + hs * kOn + 32, v + 32);
      tmem_ld_wait();
      const int hd = cta + hs * p.ctas;
#pragma unroll
      for (int n = 0; n < kOn; ++n)
        *reinterpret_cast<__nv_bfloat16*>(stg + n * 64 + lane * 2) = __float2bfloat16_rn(__uint_as_float(v[n]));
      __syncwarp();
      for (int i = lane; i < p.n_tok * 4; i += 32) {
        const int n = i >> 2, piece = i & 3;
        *reinterpret_cast<uint4*>(p.obuf + static_cast<size_t>(n) * p.n_h * kOm + static_cast<size_t>(hd) * kOm +
                                  32 * w + 8 * piece) = *reinterpret_cast<const uint4*>(stg + n * 64 + piece * 16);
      }
      __syncwarp();  // the staging is reused by the next head
    }
    // this CTA's o columns are stored: count it (all 128 epilogue threads
    // fence their stores, meet, and one of them adds)
    __threadfence();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (threadIdx.x == 32 * 4) atomicAdd(p.counters, 1u);
    if (ok && n2 > 0) ok = ot_wait(&bs->p2_done, 0, p, bs, 5);
    if (ok && n2 > 0) {
      tc_fence_after();
      // u partial tile (row r of the tile, 64 tokens) into the reduction
      // buffer [64 columns][128 rows] fp32 over the stages (all consumed)
      float* red = reinterpret_cast<float*>(smem);
#pragma unroll
      for (int c = 0; c < kOn / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lanes + kTmemU + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) red[(32 * c + j) * kOm + r] = __uint_as_float(v[j]);
      }
    }
    if (!ok) atomicExch(&bs->abort, 1);
  }
  __syncthreads();
  const bool good = !*reinterpret_cast<volatile int*>(&bs->abort);
  // the cluster's partial tiles: CTA `split` finishes the 4-row groups
  // [g0, g1) of every column, summing the three partials in rank order
  cluster_arrive();
  cluster_wait();
  if (good && n2 > 0) {
    const uint32_t red_addr = smem_u32(smem);
    const int g0 = split * (kOm / 4) / kOSplit, g1 = (split + 1) * (kOm / 4) / kOSplit, my = g1 - g0;
    for (int f = threadIdx.x; f < my * kOn; f += kOThreads) {
      const int col = f / my, row0 = 4 * (g0 + f % my);
      if (col >= p.n_tok) continue;
      const uint32_t off = static_cast<uint32_t>((col * kOm + row0) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 v[kOSplit];
#pragma unroll
      for (int q = 0; q < kOSplit; ++q) v[q] = ld_cluster_v4(map_to_rank(red_addr + off, q));
#pragma unroll
      for (int q = 0; q < kOSplit; ++q) {
        acc.x += v[q].x; acc.y += v[q].y; acc.z += v[q].z; acc.w += v[q].w;
      }
      const int o = tile * kOm + row0;
      if (o < p.d_model) {
        __nv_bfloat16* dst = p.u + static_cast<size_t>(col) * p.d_model + o;
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
      }
    }
  }
  cluster_arrive();  // the partial tiles stay until every CTA of the cluster has read them
  cluster_wait();
  if (threadIdx.x == 0) {
    // the last CTA of the launch sets the counters back for the next call
    __threadfence();
    if (atomicAdd(p.counters + 1, 1u) == static_cast<unsigned int>(p.ctas) - 1u) {
      atomicExch(p.counters, 0u);
      atomicExch(p.counters + 1, 0u);
    }
    pdl_trigger();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

int out_fused_max_tokens() { return kOn; }

// Returns cudaErrorNotSupported when the fused launch does not apply (the
// caller then runs the two separate launches).
cudaError_t launch_out_tc(const mla_handle* h, const void* o_lat, const void* w_uv, const void* w_o, int n_tok,
                          void* obuf, void* u, cudaStream_t s) {
  const mla_dims& d = h->dims;
  const int tiles = d.d_model / kOm;
  const int ctas = tiles * kOSplit;
  if (n_tok < 1 || n_tok > kOn || d.d_model % kOm != 0 || (d.n_h * d.d_h) % kOk != 0 || d.d_c % kOk != 0 ||
      d.d_h != kOm || (d.n_h + ctas - 1) / ctas > kOMaxHeadsPerCta || !h->out_counters)
    return cudaErrorNotSupported;
  cudaError_t e = kernel_attrs_once(h, reinterpret_cast<const void*>(out_kernel), kOSmem, false);
  if (e != cudaSuccess) return e;
  // every CTA waits for every other one: all must be resident at once
  static int resident[16] = {};
  int dev = h->device;
  int ncl = (dev >= 0 && dev < 16) ? resident[dev] : 0;
  if (ncl == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kOSplit, tiles);
    cfg.blockDim = dim3(kOThreads);
    cfg.dynamicSmemBytes = kOSmem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = kOSplit;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&ncl, out_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      ncl = -1;
    }
    if (ncl == 0) ncl = -1;
    if (dev >= 0 && dev < 16) resident[dev] = ncl;
  }
  if (ncl < tiles) return cudaErrorNotSupported;
  const long long H = static_cast<long long>(d.n_h) * d.d_h;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  OutMaps maps;
  if (!tensor_map_2d(h, &maps.wuv, w_uv, d.d_c, H, kOk, kOm, sw) ||
      !tensor_map_2d(h, &maps.olat, o_lat, static_cast<long long>(d.n_h) * d.d_c, n_tok, kOk, kOn, sw) ||
      !tensor_map_2d(h, &maps.wo, w_o, H, d.d_model, kOk, kOm, sw) ||
      !tensor_map_2d(h, &maps.obuf, obuf, H, n_tok, kOk, kOn, sw))
    return cudaErrorInvalidValue;
  OutParams p;
  p.n_tok = n_tok;
  p.n_h = d.n_h;
  p.ctas = ctas;
  p.uv_blocks = d.d_c / kOk;
  p.o_blocks = static_cast<int>(H / kOk);
  p.d_model = d.d_model;
  p.obuf = static_cast<__nv_bfloat16*>(obuf);
  p.u = static_cast<__nv_bfloat16*>(u);
  p.counters = h->out_counters;
  p.status = h->status;
  p.wait_limit = h->wait_limit;
  return launch_pdl(out_kernel, dim3(kOSplit, tiles), dim3(kOThreads), kOSmem, s, 1, maps, p);
}

}  // namespace mla
