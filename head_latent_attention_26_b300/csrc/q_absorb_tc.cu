// q_absorb_tc.cu -- the latent query of up to 64 tokens straight from c^Q, in
// one launch on sm_103a tensor cores.
//
// The latent query row of head i is [q~_i ; RoPE_pos(q^R_i)] with
// q^C_i = W^UQ_i c^Q and q^R_i = W^QR_i c^Q ([qiita] "Query の圧縮",
// "RoPE の扱い") and q~_i = W^UK_i^T q^C_i ([0h-n0] "行列吸収トリック").  Each
// head's q^C_i is exactly the input of its own absorption, so one CTA per head
// chains the two products without a trip through HBM:
// * phase 1: q^C_i = W^UQ_i c^Q (M = 128 rows of W^UQ_i, N = the tokens,
//   K = d_c' streamed in 64-wide blocks through a ring of shared-memory stages
//   by TMA) into TMEM;
// * hand-off: warps 4..7 read q^C_i out of TMEM, round it once to bf16 (the
//   rounding the separate route applies when it stores q_c) and write it into
//   shared memory as the MN-major B operand of phase 2 -- into the token
//   halves of the first two stages, which phase 2's weight loads leave free;
// * phase 2: q~_i = W^UK_i^T q^C_i, four 128-row blocks of the 512 latent
//   columns (A = the W^UK_i tile read MN-major, no transposed copy; K = d_h),
//   into four TMEM accumulators, then written to q_lat.
// Another n_h d_hR / 128 CTAs compute W^QR c^Q tiles and rotate each (2k,
// 2k+1) pair of rows by its token's position into q_lat's last d_hR columns.
// The weights are read once: W^UQ 50.3 MB, W^QR 25.2 MB and W^UK 16.8 MB at
// the DeepSeek-V2 sizes.  Every wait is bounded (MLA_ERR_DEVICE_TIMEOUT).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kQm = 128;                     // weight rows per tile
constexpr int kQk = 64;                      // k per stage (one 128-byte swizzle atom)
constexpr int kQn = 64;                      // token columns (at most 64 tokens)
constexpr uint32_t kQA = kQm * kQk * 2;      // 16 KB weight tile
constexpr uint32_t kQB = kQn * kQk * 2;      // 8 KB token tile
constexpr uint32_t kQStage = kQA + kQB;
constexpr int kQStages = 4;
constexpr uint32_t kQOffBars = kQStages * kQStage;
constexpr uint32_t kQSmem = kQOffBars + 256 + 1024;  // + alignment slack: two CTAs per SM
constexpr int kQThreads = 256;
constexpr int kQLatBlocks = 4;               // 512 latent columns = four 128-row blocks of W^UK_i^T
constexpr int kQDc = 512, kQDhr = 64, kQWidth = kQDc + kQDhr, kQDh = 128;

struct QAbsMaps {
  CUtensorMap wuq;  // W^UQ [n_h d_h, d_c'], boxes 64 x 128
  CUtensorMap wqr;  // W^QR [n_h d_hR, d_c'], boxes 64 x 128
  CUtensorMap cq;   // c^Q [n_tok, d_c'], boxes 64 x 64
  CUtensorMap wuk;  // W^UK [n_h d_h, d_c], boxes 64 x 64
};

struct QAbsParams {
  int n_tok, n_h, k_blocks;  // k_blocks = d_c' / 64
  const int* pos;
  int max_pos;
  const float* rope_cos;
  const float* rope_sin;
  __nv_bfloat16* q_lat;  // [n_tok, n_h, d_c + d_hR]
  int* status;
  long long wait_limit;
};

struct QAbsBars {
  uint64_t full[kQStages], empty[kQStages], qc_done, qc_ready, done, drain;
  uint32_t tmem;
  int abort;
};

// Bounded wait (sites: producer 1 stage free; MMA warp 2 stage landed, 3 q^C
// written; epilogue warps 4 q^C ready in TMEM, 5 q~ ready in TMEM).
__device__ __forceinline__ bool qa_wait(uint64_t* bar, uint32_t parity, const QAbsParams& p, QAbsBars* bs,
                                        int site) {
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
__device__ __forceinline__ bool qa_wait_warp(uint64_t* bar, uint32_t parity, const QAbsParams& p, QAbsBars* bs,
                                             int site) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = qa_wait(bar, parity, p, bs, site);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__global__ void __launch_bounds__(kQThreads, 2)  // two CTAs per SM: 128 registers a thread
    q_absorb_kernel(const __grid_constant__ QAbsMaps maps, const QAbsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  QAbsBars* bs = reinterpret_cast<QAbsBars*>(smem + kQOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool head_cta = static_cast<int>(blockIdx.x) < p.n_h;
  const int head = blockIdx.x;                                   // head CTAs
  const int rtile = static_cast<int>(blockIdx.x) - p.n_h;        // W^QR CTAs: rows [128 rtile, +128)
  const int nk = p.k_blocks;
  const int n_loads = head_cta ? nk + kQLatBlocks * (kQDh / kQk) : nk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bs->full[s], 1);
      mbar_init(&bs->empty[s], 1);
    }
    mbar_init(&bs->qc_done, 1);
    mbar_init(&bs->qc_ready, 4);
    mbar_init(&bs->done, 1);
    mbar_init(&bs->drain, 1);
    bs->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bs->tmem, kQLatBlocks * kQn);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bs->tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(head_cta ? &maps.wuq : &maps.wqr);
      tma_prefetch_desc(&maps.cq);
      if (head_cta) tma_prefetch_desc(&maps.wuk);
      const uint64_t pol_w = l2_policy_evict_normal(), pol_x = l2_policy_evict_last();
      // load i: phase-1 weight tile (i < nk) or W^UK_i^T tile (m, kb) of phase 2
      auto stage_bytes = [&](int i) { return i < nk ? kQStage : kQA; };
      auto load_w = [&](int i, uint8_t* st, uint64_t* bar) {
        if (i < nk) {
          if (head_cta) tma_load_2d_hint(st, &maps.wuq, bar, i * kQk, head * kQm, pol_w);
          else tma_load_2d_hint(st, &maps.wqr, bar, i * kQk, rtile * kQm, pol_w);
        } else {
          const int j = i - nk, m = j >> 1, kb = j & 1;  // latent block m, d_h block kb
          const int y = head * kQDh + kb * kQk;
          tma_load_2d_hint(st, &maps.wuk, bar, m * kQm, y, pol_w);
          tma_load_2d_hint(st + kQA / 2, &maps.wuk, bar, m * kQm + 64, y, pol_w);
        }
      };
      // The weights do not depend on earlier kernels: the first stages' weight
      // tiles go out before the wait for the previous kernel, their token
      // tiles (c^Q, written by it) right after.
      const int early = n_loads < kQStages ? n_loads : kQStages;
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx(&bs->full[i], stage_bytes(i));
        load_w(i, smem + i * kQStage, &bs->full[i]);
      }
      pdl_wait();
      for (int i = 0; i < early; ++i)
        if (i < nk) tma_load_2d_hint(smem + i * kQStage + kQA, &maps.cq, &bs->full[i], i * kQk, 0, pol_x);
      bool ok = true;
      int it = early;
      for (; it < n_loads && ok; ++it) {
        const int s = it % kQStages;
        if (!(ok = qa_wait(&bs->empty[s], ((it / kQStages) - 1) & 1, p, bs, 1))) break;
        uint8_t* st = smem + s * kQStage;
        mbar_arrive_expect_tx(&bs->full[s], stage_bytes(it));
        load_w(it, st, &bs->full[s]);
        if (it < nk) tma_load_2d_hint(st + kQA, &maps.cq, &bs->full[s], it * kQk, 0, pol_x);
      }
      if (!ok) {
        // every issued copy must land before the CTA may exit
        for (int k = it > kQStages ? it - kQStages : 0; k < it; ++k)
          for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->full[k % kQStages], (k / kQStages) & 1); ++i) {
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) pdl_wait();  // (the producer's token tiles already depend on it)
    __syncwarp();
    const uint32_t idesc1 = idesc_bf16_f32(kQm, kQn, false, false);
    const uint32_t idesc2 = idesc_bf16_f32(kQm, kQn, true, true);  // W^UK_i^T and q^C both MN-major
    bool ok = true;
    int it = 0;
    for (; it < nk && ok; ++it) {
      const int s = it % kQStages;
      if (!(ok = qa_wait_warp(&bs->full[s], (it / kQStages) & 1, p, bs, 2))) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * kQStage);
      mma_ss_kblock_elect<2, 2>(tmem, smem_desc(a, 16, 1024, kSwizzle128B), smem_desc(a + kQA, 16, 1024, kSwizzle128B),
                                idesc1, it > 0 ? 1u : 0u);
      mma_commit_elect(&bs->empty[s]);
    }
    if (ok) mma_commit_elect(&bs->qc_done);
    if (ok && head_cta) {
      if ((ok = qa_wait_warp(&bs->qc_ready, 0, p, bs, 3))) {
        tc_fence_after();
        for (; it < n_loads && ok; ++it) {
          const int s = it % kQStages;
          if (!(ok = qa_wait_warp(&bs->full[s], (it / kQStages) & 1, p, bs, 2))) break;
          tc_fence_after();
          const int j = it - nk, m = j >> 1, kb = j & 1;
          const uint32_t a = smem_u32(smem + s * kQStage);
          const uint32_t b = smem_u32(smem + kb * kQStage + kQA);  // q^C rows [64 kb, 64 kb + 64)
          mma_ss_kblock_elect<128, 128>(tmem + m * kQn, smem_desc(a, kQA / 2, 1024, kSwizzle128B),
                                        smem_desc(b, kQB, 1024, kSwizzle128B), idesc2, kb > 0 ? 1u : 0u);
          mma_commit_elect(&bs->empty[s]);
        }
        if (ok) mma_commit_elect(&bs->done);
      }
    }
    if (!ok) {
      // every issued MMA must finish before TMEM is released
      mma_commit_elect(&bs->drain);
      for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->drain, 0); ++i) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue warps
    const int w = warp - 4, r = 32 * w + lane;  // TMEM lane = weight row of the tile
    const uint32_t lanes = static_cast<uint32_t>(32 * w) << 16;
    if (lane == 0) pdl_wait();  // q_lat may still be read by the previous kernel's readers
    __syncwarp();
    bool ok = qa_wait(&bs->qc_done, 0, p, bs, 4);
    if (ok) {
      tc_fence_after();
      uint32_t v[kQn];
      tmem_ld32(tmem + lanes, v);
      tmem_ld32(tmem + lanes + 32, v + 32);
      tmem_ld_wait();
      if (head_cta) {
        // q^C_i row r (d_h index r) for the 64 tokens, bf16, as row r % 64 of
        // the 128B-swizzled token half of stage r / 64 (16-byte chunk c at
        // c ^ (row % 8))
        uint32_t pk[kQn / 2];
#pragma unroll
        for (int j = 0; j < kQn / 2; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        const int row = r & 63;
        uint8_t* dst = smem + (r >> 6) * kQStage + kQA + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(dst + ((c ^ (row & 7)) * 16)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        fence_proxy_async_smem();  // the MMAs read it through the async proxy
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bs->qc_ready);
        if ((ok = qa_wait_warp(&bs->done, 0, p, bs, 5))) {
          tc_fence_after();
          // q~_i: this warp holds latent columns 128 m + 32 w + lane (m = 0..3)
          // of every token.  They go through the warp's 16 KB of the (now
          // idle) stages, [token][m][32 columns], and leave as 16-byte pieces
          // (the four 64-byte runs of each token's row), 32 stores a lane
          // instead of 256 two-byte ones.
          uint8_t* stg = smem + w * (kQn * kQLatBlocks * 64);
#pragma unroll 1
          for (int m = 0; m < kQLatBlocks; ++m) {
            uint32_t q[kQn];
            tmem_ld32(tmem + lanes + m * kQn, q);
            tmem_ld32(tmem + lanes + m * kQn + 32, q + 32);
            tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < kQn; ++n)
              *reinterpret_cast<__nv_bfloat16*>(stg + n * (kQLatBlocks * 64) + m * 64 + lane * 2) =
                  __float2bfloat16_rn(__uint_as_float(q[n]));
          }
          __syncwarp();
          for (int i = lane; i < p.n_tok * kQLatBlocks * 4; i += 32) {
            const int n = i / (kQLatBlocks * 4), m = (i / 4) % kQLatBlocks, piece = i % 4;
            *reinterpret_cast<uint4*>(p.q_lat + (static_cast<size_t>(n) * p.n_h + head) * kQWidth + m * kQm + 32 * w +
                                      8 * piece) =
                *reinterpret_cast<const uint4*>(stg + n * (kQLatBlocks * 64) + m * 64 + piece * 16);
          }
        }
      } else {
        // W^QR row 128 rtile + r = positional column k2 of head hq; the pair
        // (2k, 2k + 1) sits in adjacent lanes and turns by pos * theta_k
        // Eight tokens at a time: their positions, then their cos / sin,
        // every load of a group in flight before the group's products (one
        // token after another, each load waited on, took a round trip each).
        const int o = rtile * kQm + r, hq = o / kQDhr, k2 = o % kQDhr, k = k2 >> 1;
        constexpr int kG = 8;
#pragma unroll
        for (int n0 = 0; n0 < kQn; n0 += kG) {
          if (n0 >= p.n_tok) break;
          int tp[kG];
#pragma unroll
          for (int i = 0; i < kG; ++i) tp[i] = n0 + i < p.n_tok ? __ldg(p.pos + n0 + i) : 0;
          float cs[kG], sn[kG];
#pragma unroll
          for (int i = 0; i < kG; ++i) {
            const bool in = tp[i] >= 0 && tp[i] < p.max_pos;
            const size_t t = static_cast<size_t>(in ? tp[i] : 0) * (kQDhr / 2) + k;
            cs[i] = __ldg(p.rope_cos + t);
            sn[i] = __ldg(p.rope_sin + t);
          }
#pragma unroll
          for (int i = 0; i < kG; ++i) {
            const int n = n0 + i;
            if (n >= p.n_tok) break;
            const float x = __uint_as_float(v[n]);
            const float y = __shfl_xor_sync(0xffffffffu, x, 1);
            if (tp[i] < 0 || tp[i] >= p.max_pos) {
              if (k2 == 0) report(p.status, MLA_ERR_DEVICE_BOUNDS);
              continue;
            }
            const float out = (k2 & 1) ? y * sn[i] + x * cs[i] : x * cs[i] - y * sn[i];
            p.q_lat[(static_cast<size_t>(n) * p.n_h + hq) * kQWidth + kQDc + k2] = __float2bfloat16_rn(out);
          }
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kQLatBlocks * kQn);
  }
}

}  // namespace

int q_absorb_max_tokens() { return kQn; }

cudaError_t launch_q_absorb_tc(const mla_handle* h, const void* c_q, const void* w_uq, const void* w_qr,
                               const void* w_uk, const int* pos, int n_tok, void* q_lat, cudaStream_t s) {
  const mla_dims& d = h->dims;
  if (n_tok < 1 || n_tok > kQn) return cudaErrorInvalidValue;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  QAbsMaps maps;
  if (!tensor_map_2d(h, &maps.wuq, w_uq, d.d_cq, static_cast<long long>(d.n_h) * d.d_h, kQk, kQm, sw) ||
      !tensor_map_2d(h, &maps.wqr, w_qr, d.d_cq, static_cast<long long>(d.n_h) * d.d_hr, kQk, kQm, sw) ||
      !tensor_map_2d(h, &maps.cq, c_q, d.d_cq, n_tok, kQk, kQn, sw) ||
      !tensor_map_2d(h, &maps.wuk, w_uk, d.d_c, static_cast<long long>(d.n_h) * d.d_h, 64, kQk, sw))
    return cudaErrorInvalidValue;
  QAbsParams p;
  p.n_tok = n_tok;
  p.n_h = d.n_h;
  p.k_blocks = d.d_cq / kQk;
  p.pos = pos;
  p.max_pos = h->max_pos;
  p.rope_cos = h->rope_cos;
  p.rope_sin = h->rope_sin;
  p.q_lat = static_cast<__nv_bfloat16*>(q_lat);
  p.status = h->status;
  p.wait_limit = h->wait_limit;
  cudaError_t e = kernel_attrs_once(h, reinterpret_cast<const void*>(q_absorb_kernel), kQSmem, false);
  if (e != cudaSuccess) return e;
  const int ctas = d.n_h + d.n_h * d.d_hr / kQm;
  return launch_pdl(q_absorb_kernel, dim3(ctas), dim3(kQThreads), kQSmem, s, 1, maps, p);
}

}  // namespace mla
