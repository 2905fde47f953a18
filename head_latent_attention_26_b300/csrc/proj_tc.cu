// proj_tc.cu -- the projection steps of the layer on sm_103a tensor cores.
//
// Every projection of the decode step is a skinny product Y[n, o] =
// sum_k X[n, k] W[o, k]: a few new tokens (n) against a weight matrix that is
// read once per step.  The work is bound by streaming the weights out of HBM,
// so the kernel is built around that stream:
// * the weight rows are the M = 128 side of every tcgen05 MMA and the tokens
//   the N side (N = 64, 128 or 256 per tile), accumulators in TMEM;
// * one warp issues TMA loads of 128 x 64 weight tiles (128B swizzle, L2
//   evict-first) and token tiles (evict-last: every output tile re-reads
//   them) into a ring of shared-memory stages, one thread issues the MMAs;
// * when one output tile has too few k-blocks to keep enough SMs streaming,
//   the k range is split over the CTAs of a thread-block cluster and the fp32
//   partial tiles are summed through distributed shared memory in a fixed
//   order, so no global workspace or second kernel is needed.
//
// Three epilogues serve the steps of the path:
// * linear: Y[n, o] in bf16 -- c^Q = W^DQ h, q^C = W^UQ c^Q, W^QR c^Q
//   ([qiita] "Query の圧縮", "RoPE の扱い"), o_i = W^UV_i o~_i per head and
//   u = W^O [o_1; ...] ([kasblo] "V側は、小さな表現の加重和を先に求める",
//   [qiita] "Attention 計算");
// * append: the cache row [c^KV ; RoPE_pos(k^R)] = [W^DKV h ; RoPE(W^KR h)]
//   ([0h-n0] "MLA: 低ランクKV結合圧縮", [qiita] "RoPE の扱い") rounded once to
//   bf16 and written to pool row block_table[b][pos/64]*64 + pos%64;
// * absorb: q~_i = W^UK_i^T q^C_i ([0h-n0] "行列吸収トリック") with the W^UK
//   tile read as an MN-major A operand (no transpose copy), plus the RoPE of
//   q^R_i, written as one latent query row [q~_i ; RoPE_pos(q^R_i)];
// * folded query: the same latent query row straight from c^Q with the
//   folded weight W~^UQ_i = W^UK_i^T W^UQ_i ([0h-n0] "行列吸収トリック": the
//   product can be formed ahead of inference) as the first product and W^QR
//   as the second, rotated in the epilogue.
//
// [0h-n0] = "論文解説: DeepSeek-V2 — … Multi-head Latent Attention",
// [qiita] = MLA notes on qiita.com, [kasblo] = MLA explainer on kasblo.com.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kBM = 128;                       // weight rows per output tile
constexpr int kBK = 64;                        // k per stage (one 128-byte swizzle atom)
constexpr uint32_t kABytes = kBM * kBK * 2;    // 16 KB weight tile
constexpr int kThreads = 128;
constexpr int kMaxSplit = 16;                  // cluster size (above 8 needs the non-portable opt-in)
constexpr int kMaxDevices = 16;                // devices whose resident-cluster counts are cached

enum : int { kModeLinear = 0, kModeAppend = 1, kModeAbsorb = 2, kModeQFolded = 3, kModeLinearAppend = 4 };

struct ProjMaps {
  CUtensorMap w;   // weights
  CUtensorMap x;   // tokens
  CUtensorMap w2;  // linear mode: weights of a second product with the same tokens
};

struct ProjParams {
  int n_tok, out, k_blocks;
  int tiles_per_group;  // output tiles sharing one window of X columns
  int x_group_cols;     // X column offset of group g = g * x_group_cols
  int w_group_rows;     // absorb: W^UK row offset of head g = g * w_group_rows
  __nv_bfloat16* y;
  long long ldy;
  // linear mode: output tiles >= seg1_tiles belong to a second product
  // (maps.w2 -> y2) over the same tokens and k range
  int seg1_tiles, out2;
  __nv_bfloat16* y2;
  long long ldy2;
  int y_f16, y2_f16;  // linear mode: write y / y2 as fp16 instead of bf16
  // append
  const int* seq_idx;
  const int* pos;
  const int* block_table;
  int max_blocks, batch, n_pool_blocks, max_pos, d_c, d_hr, width, block;
  int dense;  // append: row n of the tile goes to row n of `pool` (a dense [n_new, width] buffer)
  __nv_bfloat16* pool;
  const float* rope_cos;
  const float* rope_sin;
  // absorb
  __nv_bfloat16* q_lat;
  const __nv_bfloat16* q_r;
  int n_h;
  int* status;
  long long wait_limit;
};

template <int STAGES, int NT>
struct ProjShared {
  uint64_t full[STAGES], empty[STAGES], done;
  uint32_t tmem;
  int abort;
  int slot[NT];  // append: destination pool row of each token of the tile (-1 = skip)
  int tpos[NT];  // append: its position
};

__device__ __forceinline__ bool proj_wait(uint64_t* bar, uint32_t parity, const ProjParams& p, int* abort) {
  for (long long i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= p.wait_limit || *reinterpret_cast<volatile int*>(abort)) {
      report(p.status, MLA_ERR_DEVICE_TIMEOUT);
      atomicExch(abort, 1);
      return false;
    }
  }
}

__device__ __forceinline__ void store_pair(__nv_bfloat16* dst, float a, float b) {
  *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(a, b);
}
// the same pair as bf16 or, when f16, as fp16 (one rounding either way)
__device__ __forceinline__ void store_pair_as(__nv_bfloat16* dst, float a, float b, int f16) {
  if (f16) {
    const __half2 v = __floats2half2_rn(a, b);
    *reinterpret_cast<__half2*>(dst) = v;
  } else {
    store_pair(dst, a, b);
  }
}

// One CTA computes MT output tiles of 128 weight rows (one TMEM accumulator of
// NT columns each) over its share [kb0, kb1) of the k blocks.
template <int NT, int STAGES, int MODE, int MT>
__global__ void __launch_bounds__(kThreads, 1) proj_kernel(const __grid_constant__ ProjMaps maps, const ProjParams p) {
  constexpr uint32_t kBBytes = NT * kBK * 2;
  constexpr uint32_t kStage = kABytes + kBBytes;
  constexpr uint32_t kRedCols = 64;  // epilogue chunk: 64 token columns of fp32
  static_assert(STAGES * kStage >= kRedCols * kBM * 4, "reduction buffer reuses the stages");
  using Shared = ProjShared<STAGES, NT>;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared* ss = reinterpret_cast<Shared*>(smem + STAGES * kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = static_cast<int>(cluster_ctarank());
  const int nsplit = static_cast<int>(cluster_nctarank());
  const int n0 = blockIdx.z * NT;
  // first output tile of this CTA; in linear mode tiles past seg1_tiles are
  // tiles of the second product
  const bool seg2 = (MODE == kModeLinear || MODE == kModeQFolded || MODE == kModeLinearAppend) &&
                    static_cast<int>(blockIdx.y) * MT >= p.seg1_tiles;
  // tiles that write cache rows: every tile of the append mode, the second
  // product's tiles of the linear + append mode
  const bool appends = MODE == kModeAppend || (MODE == kModeLinearAppend && seg2);
  const int tile0 = static_cast<int>(blockIdx.y) * MT - (seg2 ? p.seg1_tiles : 0);
  const CUtensorMap* wmap = seg2 ? &maps.w2 : &maps.w;
  const int group = tile0 / p.tiles_per_group;  // all MT tiles share it (MT divides tiles_per_group)
  const int kb0 = static_cast<int>(static_cast<long long>(split) * p.k_blocks / nsplit);
  const int kb1 = static_cast<int>(static_cast<long long>(split + 1) * p.k_blocks / nsplit);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ss->full[s], 1);
      mbar_init(&ss->empty[s], 1);
    }
    mbar_init(&ss->done, 1);
    ss->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ss->tmem, NT * MT);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ss->tmem;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(wmap);
      tma_prefetch_desc(&maps.x);
      const uint64_t pol_w = l2_policy_evict_normal(), pol_x = l2_policy_evict_last();
      const int x_off = group * p.x_group_cols;
      // The weights do not depend on earlier kernels: the first STAGES weight
      // tiles go out before the wait for the previous kernel, their token
      // tiles right after it.
      const int n_loads = MT * (kb1 - kb0);
      const int early = n_loads < STAGES ? n_loads : STAGES;
      auto load_w = [&](int i, uint8_t* st, uint64_t* bar) {
        const int o_tile = tile0 + i / (kb1 - kb0), kb = kb0 + i % (kb1 - kb0);
        if (MODE == kModeAbsorb) {
          // W^UK_i^T tile: 64 rows of head i (the k side) x 128 latent columns (the M side)
          const int m = o_tile % p.tiles_per_group;
          const int y = group * p.w_group_rows + kb * kBK;
          tma_load_2d_hint(st, wmap, bar, m * kBM, y, pol_w);
          tma_load_2d_hint(st + kABytes / 2, wmap, bar, m * kBM + 64, y, pol_w);
        } else {
          tma_load_2d_hint(st, wmap, bar, kb * kBK, o_tile * kBM, pol_w);
        }
      };
      auto load_x = [&](int i, uint8_t* st, uint64_t* bar) {
        const int kb = kb0 + i % (kb1 - kb0);
        tma_load_2d_hint(st + kABytes, &maps.x, bar, x_off + kb * kBK, n0, pol_x);
      };
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx(&ss->full[i], kStage);
        load_w(i, smem + i * kStage, &ss->full[i]);
      }
      pdl_wait();
      for (int i = 0; i < early; ++i) load_x(i, smem + i * kStage, &ss->full[i]);
      uint32_t it = early;
      for (int i = early; i < n_loads; ++i, ++it) {
        const int s = it % STAGES;
        if (!proj_wait(&ss->empty[s], ((it / STAGES) - 1) & 1, p, &ss->abort)) break;
        uint8_t* st = smem + s * kStage;
        mbar_arrive_expect_tx(&ss->full[s], kStage);
        load_w(i, st, &ss->full[s]);
        load_x(i, st, &ss->full[s]);
      }
      if (ss->abort) {
        // every issued copy must land before the CTA may exit
        for (uint32_t k = (it > STAGES ? it - STAGES : 0); k < it; ++k)
          for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&ss->full[k % STAGES], (k / STAGES) & 1); ++i) {
          }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (warp-uniform operands); one elected lane
    // issues each k block's four MMAs.
    {
      const uint32_t idesc = idesc_bf16_f32(kBM, NT, MODE == kModeAbsorb, false);
      uint32_t it = 0;
      bool go = true;
      for (int mi = 0; mi < MT && go; ++mi) {
        const uint32_t d = tmem + mi * NT;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % STAGES;
          bool ok = true;
          if (lane == 0) ok = proj_wait(&ss->full[s], (it / STAGES) & 1, p, &ss->abort);
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
            go = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + s * kStage), b = a + kABytes;
          const uint64_t bd = smem_desc(b, 16, 1024, kSwizzle128B);
          if (MODE == kModeAbsorb)
            mma_ss_kblock_elect<128, 2>(d, smem_desc(a, 8192, 1024, kSwizzle128B), bd, idesc, kb > kb0 ? 1u : 0u);
          else
            mma_ss_kblock_elect<2, 2>(d, smem_desc(a, 16, 1024, kSwizzle128B), bd, idesc, kb > kb0 ? 1u : 0u);
          mma_commit_elect(&ss->empty[s]);
        }
      }
      mma_commit_elect(&ss->done);  // arrives once every MMA above has finished
    }
  } else if (appends) {
    // ---------------------------------------------------------------- destination rows
    pdl_wait();
    for (int j = threadIdx.x - 64; j < NT; j += 64) {
      const int n = n0 + j;
      int slot = -1, tp = 0;
      if (n < p.n_tok) {
        const int b = __ldg(p.seq_idx + n);
        tp = __ldg(p.pos + n);
        if (b < 0 || b >= p.batch || tp < 0 || tp >= p.max_pos || tp / p.block >= p.max_blocks) {
          report(p.status, MLA_ERR_DEVICE_BOUNDS);
        } else {
          const int blk = __ldg(p.block_table + static_cast<size_t>(b) * p.max_blocks + tp / p.block);
          if (blk < 0 || blk >= p.n_pool_blocks) report(p.status, MLA_ERR_DEVICE_BOUNDS);
          else slot = p.dense ? n : blk * p.block + tp % p.block;
        }
      }
      ss->slot[j] = slot;
      ss->tpos[j] = tp;
    }
  }
  __syncthreads();

  // -------------------------------------------------------------------- epilogue
  bool ok = proj_wait(&ss->done, 0, p, &ss->abort) && !*reinterpret_cast<volatile int*>(&ss->abort);
  tc_fence_after();
  if (threadIdx.x == 0) pdl_trigger();  // every CTA of this grid is resident: the next may launch
  float* red = reinterpret_cast<float*>(smem);  // [64 columns][128 rows] fp32, stages reused
  const uint32_t red_addr = smem_u32(red);
  const int r = warp * 32 + lane;  // TMEM lane = output row of the tile
  // CTA `split` of the cluster finishes the 4-row groups [g0, g1) of each
  // column: contiguous 16-byte reads, so the SM-to-SM transfers are whole
  const int g0 = split * (kBM / 4) / nsplit, g1 = (split + 1) * (kBM / 4) / nsplit, my_groups = g1 - g0;
  const int half = p.d_hr / 2;
#pragma unroll 1
  for (int cc = 0; cc < MT * NT; cc += kRedCols) {
    const int mi = cc / NT, c0 = cc % NT;
    const int o_tile = tile0 + mi;
    if (ok) {
#pragma unroll
      for (int ch = 0; ch < kRedCols / 16; ++ch) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc + ch * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) red[(ch * 16 + j) * kBM + r] = __uint_as_float(v[j]);
      }
    }
    if (nsplit > 1) {
      cluster_arrive();
      cluster_wait();
    } else {
      __syncthreads();
    }
    if (ok) {
      for (int f = threadIdx.x; f < my_groups * kRedCols; f += kThreads) {
        const int col = f / my_groups;
        const int row0 = 4 * (g0 + f % my_groups);
        const int n = n0 + c0 + col;
        if (n >= p.n_tok) continue;
        const uint32_t off = static_cast<uint32_t>((col * kBM + row0) * 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (nsplit > 1) {
          // all partials in flight at once, then summed in rank order
          float4 v[kMaxSplit];
#pragma unroll
          for (int q = 0; q < kMaxSplit; ++q)
            v[q] = q < nsplit ? ld_cluster_v4(map_to_rank(red_addr + off, q)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < kMaxSplit; ++q) {
            acc.x += v[q].x;
            acc.y += v[q].y;
            acc.z += v[q].z;
            acc.w += v[q].w;
          }
        } else {
          acc = *reinterpret_cast<const float4*>(reinterpret_cast<const uint8_t*>(red) + off);
        }
        const float2 pr[2] = {make_float2(acc.x, acc.y), make_float2(acc.z, acc.w)};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = row0 + 2 * e;
          const float2 a = pr[e];
          if (MODE == kModeLinear || (MODE == kModeLinearAppend && !seg2)) {
            const int o = o_tile * kBM + row;
            if (!seg2 && o < p.out) store_pair_as(p.y + static_cast<size_t>(n) * p.ldy + o, a.x, a.y, p.y_f16);
            if (seg2 && o < p.out2) store_pair_as(p.y2 + static_cast<size_t>(n) * p.ldy2 + o, a.x, a.y, p.y2_f16);
          } else if (appends) {
            const int o = o_tile * kBM + row;
            const int slot = ss->slot[c0 + col];
            if (o >= (MODE == kModeLinearAppend ? p.out2 : p.out) || slot < 0) continue;
            __nv_bfloat16* dst = p.pool + static_cast<size_t>(slot) * p.width + o;
            if (o < p.d_c) {
              store_pair(dst, a.x, a.y);
            } else {
              const int k = (o - p.d_c) >> 1;
              const size_t t = static_cast<size_t>(ss->tpos[c0 + col]) * half + k;
              const float cs = __ldg(p.rope_cos + t), sn = __ldg(p.rope_sin + t);
              store_pair(dst, a.x * cs - a.y * sn, a.x * sn + a.y * cs);
            }
          } else if (MODE == kModeQFolded) {
            const int o = o_tile * kBM + row;
            if (!seg2) {
              // W~^UQ row o = latent column o % d_c of head o / d_c
              if (o < p.out)
                store_pair(p.q_lat + (static_cast<size_t>(n) * p.n_h + o / p.d_c) * p.width + o % p.d_c, a.x, a.y);
            } else if (o < p.out2) {
              // W^QR row o = positional column o % d_hr of head o / d_hr: rotate the pair
              const int tp = __ldg(p.pos + n);
              if (tp < 0 || tp >= p.max_pos) {
                report(p.status, MLA_ERR_DEVICE_BOUNDS);
                continue;
              }
              const int k2 = o % p.d_hr;
              const size_t t = static_cast<size_t>(tp) * half + (k2 >> 1);
              const float cs = __ldg(p.rope_cos + t), sn = __ldg(p.rope_sin + t);
              store_pair(p.q_lat + (static_cast<size_t>(n) * p.n_h + o / p.d_hr) * p.width + p.d_c + k2,
                         a.x * cs - a.y * sn, a.x * sn + a.y * cs);
            }
          } else {
            const int o = (o_tile % p.tiles_per_group) * kBM + row;  // latent column of head `group`
            if (o < p.out)
              store_pair(p.q_lat + (static_cast<size_t>(n) * p.n_h + group) * p.width + o, a.x, a.y);
          }
        }
      }
    }
    if (nsplit > 1) {
      cluster_arrive();  // the partial tiles stay until every CTA has read them
      cluster_wait();
    } else {
      __syncthreads();
    }
  }
  if (MODE == kModeAbsorb && ok) {
    // the positional part of the latent query: RoPE_pos(q^R_i) ([qiita] "RoPE の扱い"),
    // shared out over the CTAs of the head; each thread gathers the operands
    // of a batch of items before using any, so their loads overlap
    const int m = ((tile0 % p.tiles_per_group) / MT) * nsplit + split, nm = (p.tiles_per_group / MT) * nsplit;
    const int items = NT * half;
    constexpr int kBatch = 8;
    const int stride = kThreads * nm;
    for (int base = threadIdx.x + kThreads * m; base < items; base += stride * kBatch) {
      int tp[kBatch];
      __nv_bfloat162 x[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int f = base + b * stride;
        const int n = n0 + f / half, k = f % half;
        const bool live = f < items && n < p.n_tok;
        tp[b] = live ? __ldg(p.pos + n) : -1;
        x[b] = live ? *reinterpret_cast<const __nv_bfloat162*>(p.q_r + (static_cast<size_t>(n) * p.n_h + group) * p.d_hr + 2 * k)
                    : __nv_bfloat162();
      }
      float cs[kBatch], sn[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int f = base + b * stride, k = f % half;
        const bool live = tp[b] >= 0 && tp[b] < p.max_pos;
        const size_t t = live ? static_cast<size_t>(tp[b]) * half + k : 0;
        cs[b] = live ? __ldg(p.rope_cos + t) : 0.f;
        sn[b] = live ? __ldg(p.rope_sin + t) : 0.f;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int f = base + b * stride;
        const int n = n0 + f / half, k = f % half;
        if (f >= items || n >= p.n_tok) continue;
        if (tp[b] < 0 || tp[b] >= p.max_pos) {
          report(p.status, MLA_ERR_DEVICE_BOUNDS);
          continue;
        }
        const float x0 = __bfloat162float(x[b].x), x1 = __bfloat162float(x[b].y);
        const size_t hn = static_cast<size_t>(n) * p.n_h + group;
        store_pair(p.q_lat + hn * p.width + p.d_c + 2 * k, x0 * cs[b] - x1 * sn[b], x0 * sn[b] + x1 * cs[b]);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, NT * MT);
  }
}

template <int NT, int STAGES, int MODE, int MT>
cudaError_t launch_proj_nt(const mla_handle* h, const ProjMaps& maps, const ProjParams& p, int nsplit,
                           int tile_groups, int n_tiles, cudaStream_t s) {
  constexpr size_t kSmem = STAGES * (kABytes + NT * kBK * 2) + sizeof(ProjShared<STAGES, NT>) + 1024;
  auto kern = proj_kernel<NT, STAGES, MODE, MT>;
  // both attributes once per handle (the cluster opt-in is harmless for small splits)
  cudaError_t e = kernel_attrs_once(h, reinterpret_cast<const void*>(kern), static_cast<int>(kSmem), true);
  if (e != cudaSuccess) return e;
  // The largest split (cluster size) not above nsplit whose clusters can all
  // be resident at once: clusters are placed within one GPC, so a split that
  // fits the SM count can still leave a second wave.  Per device and cluster
  // size, the resident-cluster count is asked once and kept.
  static int resident[kMaxDevices][kMaxSplit + 1];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
  const int clusters = tile_groups * n_tiles;
  for (; nsplit > 1; --nsplit) {
    int ncl = dev >= 0 ? resident[dev][nsplit] : 0;
    if (ncl == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(nsplit, tile_groups, n_tiles);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = kSmem;
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = nsplit;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = 1;
      cfg.attrs = a;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();  // not fatal: fall back to the SM-count estimate
        break;
      }
      if (ncl <= 0) ncl = -1;
      if (dev >= 0) resident[dev][nsplit] = ncl;
    }
    if (ncl >= clusters) break;
  }
  return launch_pdl(kern, dim3(nsplit, tile_groups, n_tiles), dim3(kThreads, 1, 1), kSmem, s, nsplit, maps, p);
}

// Token-tile width: the smallest of 64/128/256 that holds every token, else
// 256-token tiles.  Stages: enough for ~100-200 KB of loads in flight per SM.
// With 64-token tiles, a grid whose unsplit tiles fit the SMs runs one CTA
// per SM with eight stages (a lone CTA with four stages keeps too little in
// flight to reach its share of HBM bandwidth); larger grids run two CTAs per
// SM with four.
template <int MODE, int MT>
cudaError_t launch_proj(const mla_handle* h, const ProjMaps& maps, const ProjParams& p, int nsplit, int o_tiles,
                        cudaStream_t s) {
  const int groups = o_tiles / MT;
  if (p.n_tok <= 64) {
    if (groups <= h->num_sms) return launch_proj_nt<64, 8, MODE, MT>(h, maps, p, nsplit, groups, 1, s);
    return launch_proj_nt<64, 4, MODE, MT>(h, maps, p, nsplit, groups, 1, s);
  }
  if (p.n_tok <= 128) return launch_proj_nt<128, 4, MODE, MT>(h, maps, p, nsplit, groups, 1, s);
  return launch_proj_nt<256, 3, MODE, (MT > 2 ? 2 : MT)>(h, maps, p, nsplit, o_tiles / (MT > 2 ? 2 : MT),
                                                        (p.n_tok + 255) / 256, s);
}

int token_tile(int n_tok) { return n_tok <= 64 ? 64 : n_tok <= 128 ? 128 : 256; }

// k-range split: the largest that keeps the grid within one wave (two CTAs
// per SM for 64-token tiles, one otherwise) and gives every CTA a k block.
int pick_split(const mla_handle* h, int ctas_per_split, int n_tok, int k_blocks) {
  const int nt = token_tile(n_tok);
  const long long base = static_cast<long long>(ctas_per_split) * ((n_tok + nt - 1) / nt);
  const long long slots = static_cast<long long>(h->num_sms) * (nt == 64 ? 2 : 1);
  int sp = 1;
  while (sp + 1 <= kMaxSplit && sp + 1 <= k_blocks && base * (sp + 1) <= slots) ++sp;
  return sp;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 [rows, cols] (rows ld elements apart; 0: cols) with 128B-swizzled
// boxes, through the handle's map cache
bool encode_bf16_2d(const mla_handle* h, CUtensorMap* m, const void* base, long long cols, long long rows,
                    int box_cols, int box_rows, long long ld = 0) {
  return tensor_map_2d(h, m, base, cols, rows, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ld);
}

namespace {
ProjParams base_params(const mla_handle* h, int n_tok) {
  ProjParams p = {};
  p.n_tok = n_tok;
  p.tiles_per_group = 1 << 30;
  p.status = h->status;
  p.wait_limit = h->wait_limit;
  p.max_pos = h->max_pos;
  p.d_c = h->dims.d_c;
  p.d_hr = h->dims.d_hr;
  p.width = h->dims.d_c + h->dims.d_hr;
  p.block = h->dims.block;
  p.n_h = h->dims.n_h;
  p.rope_cos = h->rope_cos;
  p.rope_sin = h->rope_sin;
  return p;
}
}  // namespace

cudaError_t launch_linear_tc(const mla_handle* h, const void* X, int x_cols, const void* W, int in, int out,
                             int groups, int x_group_cols, void* Y, long long ldy, int n_tok, cudaStream_t s) {
  ProjMaps maps;
  const int nt = token_tile(n_tok);
  if (!encode_bf16_2d(h, &maps.w, W, in, out, kBK, kBM) || !encode_bf16_2d(h, &maps.x, X, x_cols, n_tok, kBK, nt))
    return cudaErrorInvalidValue;
  maps.w2 = maps.w;
  ProjParams p = base_params(h, n_tok);
  const int o_tiles = (out + kBM - 1) / kBM;
  p.out = out;
  p.k_blocks = (in + kBK - 1) / kBK;
  p.tiles_per_group = groups > 1 ? o_tiles / groups : 1 << 30;
  p.x_group_cols = groups > 1 ? x_group_cols : 0;
  p.y = static_cast<__nv_bfloat16*>(Y);
  p.ldy = ldy;
  p.seg1_tiles = 1 << 30;
  return launch_proj<kModeLinear, 1>(h, maps, p, pick_split(h, o_tiles, n_tok, p.k_blocks), o_tiles, s);
}

cudaError_t launch_linear2_tc(const mla_handle* h, const void* X, int in, const void* W1, int out1, void* Y1,
                              long long ldy1, const void* W2, int out2, void* Y2, long long ldy2, int n_tok,
                              cudaStream_t s, long long x_ld, int f16_mask) {
  ProjMaps maps;
  const int nt = token_tile(n_tok);
  if (!encode_bf16_2d(h, &maps.w, W1, in, out1, kBK, kBM) || !encode_bf16_2d(h, &maps.w2, W2, in, out2, kBK, kBM) ||
      !encode_bf16_2d(h, &maps.x, X, in, n_tok, kBK, nt, x_ld))
    return cudaErrorInvalidValue;
  ProjParams p = base_params(h, n_tok);
  const int t1 = (out1 + kBM - 1) / kBM, t2 = (out2 + kBM - 1) / kBM;
  p.out = out1;
  p.out2 = out2;
  p.k_blocks = (in + kBK - 1) / kBK;
  p.y = static_cast<__nv_bfloat16*>(Y1);
  p.ldy = ldy1;
  p.y2 = static_cast<__nv_bfloat16*>(Y2);
  p.ldy2 = ldy2;
  p.y_f16 = f16_mask & 1;
  p.y2_f16 = (f16_mask >> 1) & 1;
  p.seg1_tiles = t1;
  return launch_proj<kModeLinear, 1>(h, maps, p, pick_split(h, t1 + t2, n_tok, p.k_blocks), t1 + t2, s);
}

cudaError_t launch_q_absorbed_tc(const mla_handle* h, const void* c_q, const void* w_abs, const void* w_qr,
                                 const int* pos, int n_tok, void* q_lat, cudaStream_t s) {
  const mla_dims& d = h->dims;
  const int out1 = d.n_h * d.d_c, out2 = d.n_h * d.d_hr;
  ProjMaps maps;
  if (!encode_bf16_2d(h, &maps.w, w_abs, d.d_cq, out1, kBK, kBM) || !encode_bf16_2d(h, &maps.w2, w_qr, d.d_cq, out2, kBK, kBM) ||
      !encode_bf16_2d(h, &maps.x, c_q, d.d_cq, n_tok, kBK, token_tile(n_tok)))
    return cudaErrorInvalidValue;
  ProjParams p = base_params(h, n_tok);
  const int t1 = (out1 + kBM - 1) / kBM, t2 = (out2 + kBM - 1) / kBM;
  p.out = out1;
  p.out2 = out2;
  p.k_blocks = (d.d_cq + kBK - 1) / kBK;
  p.seg1_tiles = t1;
  p.pos = pos;
  p.q_lat = static_cast<__nv_bfloat16*>(q_lat);
  return launch_proj<kModeQFolded, 1>(h, maps, p, pick_split(h, t1 + t2, n_tok, p.k_blocks), t1 + t2, s);
}

cudaError_t launch_cache_append_tc(const mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx,
                                   const int* pos, int n_new, const int* block_table, int max_blocks, int batch,
                                   void* pool, int n_pool_blocks, cudaStream_t s) {
  const mla_dims& d = h->dims;
  const int width = d.d_c + d.d_hr;
  ProjMaps maps;
  if (!encode_bf16_2d(h, &maps.w, w_dkr, d.d_model, width, kBK, kBM) ||
      !encode_bf16_2d(h, &maps.x, x, d.d_model, n_new, kBK, token_tile(n_new)))
    return cudaErrorInvalidValue;
  ProjParams p = base_params(h, n_new);
  const int o_tiles = (width + kBM - 1) / kBM;
  p.out = width;
  p.k_blocks = (d.d_model + kBK - 1) / kBK;
  p.seq_idx = seq_idx;
  p.pos = pos;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.batch = batch;
  p.n_pool_blocks = n_pool_blocks;
  p.pool = static_cast<__nv_bfloat16*>(pool);
  maps.w2 = maps.w;
  p.seg1_tiles = 1 << 30;
  return launch_proj<kModeAppend, 1>(h, maps, p, pick_split(h, o_tiles, n_new, p.k_blocks), o_tiles, s);
}

// c^Q = W^DQ x (into c_q, [n_tok, d_cq]) and the cache rows of the same tokens
// (mla_cache_append's product and epilogue) in one launch: both products
// read the same token tiles.
cudaError_t launch_q_down_append_tc(const mla_handle* h, const void* x, const void* w_dq, void* c_q,
                                   const void* w_dkr, const int* seq_idx, const int* pos, int n_new,
                                   const int* block_table, int max_blocks, int batch, void* pool, int n_pool_blocks,
                                   cudaStream_t s) {
  const mla_dims& d = h->dims;
  const int width = d.d_c + d.d_hr;
  ProjMaps maps;
  if (!encode_bf16_2d(h, &maps.w, w_dq, d.d_model, d.d_cq, kBK, kBM) ||
      !encode_bf16_2d(h, &maps.w2, w_dkr, d.d_model, width, kBK, kBM) ||
      !encode_bf16_2d(h, &maps.x, x, d.d_model, n_new, kBK, token_tile(n_new)))
    return cudaErrorInvalidValue;
  ProjParams p = base_params(h, n_new);
  const int t1 = (d.d_cq + kBM - 1) / kBM, t2 = (width + kBM - 1) / kBM;
  p.out = d.d_cq;
  p.y = static_cast<__nv_bfloat16*>(c_q);
  p.ldy = d.d_cq;
  p.out2 = width;
  p.seg1_tiles = t1;
  p.k_blocks = (d.d_model + kBK - 1) / kBK;
  p.seq_idx = seq_idx;
  p.pos = pos;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.batch = batch;
  p.n_pool_blocks = n_pool_blocks;
  p.pool = static_cast<__nv_bfloat16*>(pool);
  return launch_proj<kModeLinearAppend, 1>(h, maps, p, pick_split(h, t1 + t2, n_new, p.k_blocks), t1 + t2, s);
}

// The cache rows of the new tokens, [n_new, d_c + d_hr] bf16 in token order
// (the append epilogue with the block-table scatter replaced by row n).  The
// block table is still read to check each token's sequence and position.
cudaError_t launch_cache_rows_dense_tc(const mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx,
                                       const int* pos, int n_new, const int* block_table, int max_blocks, int batch,
                                       int n_pool_blocks, void* rows, cudaStream_t s) {
  const mla_dims& d = h->dims;
  const int width = d.d_c + d.d_hr;
  ProjMaps maps;
  if (!encode_bf16_2d(h, &maps.w, w_dkr, d.d_model, width, kBK, kBM) ||
      !encode_bf16_2d(h, &maps.x, x, d.d_model, n_new, kBK, token_tile(n_new)))
    return cudaErrorInvalidValue;
  ProjParams p = base_params(h, n_new);
  const int o_tiles = (width + kBM - 1) / kBM;
  p.out = width;
  p.k_blocks = (d.d_model + kBK - 1) / kBK;
  p.seq_idx = seq_idx;
  p.pos = pos;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.batch = batch;
  p.n_pool_blocks = n_pool_blocks;
  p.pool = static_cast<__nv_bfloat16*>(rows);
  p.dense = 1;
  maps.w2 = maps.w;
  p.seg1_tiles = 1 << 30;
  return launch_proj<kModeAppend, 1>(h, maps, p, pick_split(h, o_tiles, n_new, p.k_blocks), o_tiles, s);
}

cudaError_t launch_absorb_q_tc(const mla_handle* h, const void* q_c, const void* q_r, const int* pos, int n_tok,
                               const void* w_uk, void* q_lat, cudaStream_t s) {
  const mla_dims& d = h->dims;
  ProjMaps maps;
  // W^UK as [n_h*d_h rows, d_c columns]; boxes of 64 rows x 64 latent columns
  if (!encode_bf16_2d(h, &maps.w, w_uk, d.d_c, static_cast<long long>(d.n_h) * d.d_h, 64, kBK) ||
      !encode_bf16_2d(h, &maps.x, q_c, static_cast<long long>(d.n_h) * d.d_h, n_tok, kBK, token_tile(n_tok)))
    return cudaErrorInvalidValue;
  ProjParams p = base_params(h, n_tok);
  const int per_head = (d.d_c + kBM - 1) / kBM;
  p.out = d.d_c;
  p.k_blocks = (d.d_h + kBK - 1) / kBK;
  p.tiles_per_group = per_head;
  p.x_group_cols = d.d_h;
  p.w_group_rows = d.d_h;
  p.pos = pos;
  p.q_lat = static_cast<__nv_bfloat16*>(q_lat);
  p.q_r = static_cast<const __nv_bfloat16*>(q_r);
  maps.w2 = maps.w;
  p.seg1_tiles = 1 << 30;
  // Up to 64 tokens: one 128-column tile per CTA with two stages (the tile's
  // two k blocks both in flight), four CTAs per SM, so all n_h * d_c / 128
  // tiles stream in one wave and the epilogue and the RoPE items are spread
  // over four CTAs per head.  At 64 tokens this takes 9.8 us against 17.6 us
  // for one eight-stage CTA per head (back-to-back calls, weights not in L2).
  if (n_tok <= 64) return launch_proj_nt<64, 2, kModeAbsorb, 1>(h, maps, p, 1, per_head * d.n_h, 1, s);
  // more tokens: all of a head's output tiles in one CTA (they share the q^C tile)
  constexpr int kMT = 4;
  if (per_head % kMT != 0) return cudaErrorInvalidValue;
  // d_h = 128 is two k blocks: no split, so no cluster reduction
  return launch_proj<kModeAbsorb, kMT>(h, maps, p, 1, per_head * d.n_h, s);
}

}  // namespace mla
