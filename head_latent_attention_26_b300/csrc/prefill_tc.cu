// prefill_tc.cu -- causal attention of a whole prompt over expanded keys and
// values, on sm_103a tensor cores.
//
// [perforder] "極限最適化の代償：MLA特有の学習負荷と独自Tritonカーネルという障壁"
// notes that when many tokens are processed together (prefill) the latent
// vectors are up-projected to full keys and values by a large matrix product;
// [kasblo] "「キャッシュを減らせた」と「その割合だけ速い」は別の評価" names that
// expanded branch of the reference implementation.  The prompt's keys and
// values are therefore formed explicitly (K^C_i = C W^UK_i^T, V_i = C W^UV_i^T,
// one two-product GEMM launch of the projection kernel), and this kernel runs
// causal attention per head over them ([qiita] "Attention 計算": query t sees
// keys j <= t; the score is q_i.k_i / sqrt(d_h + d_hR) with q_i = [q^C_i ;
// RoPE_t(q^R_i)] and k_i = [K^C_i ; k^R]).
//
// One CTA per (128-query tile, head), 256 threads:
// The MMAs multiply fp16 operands with fp32 accumulation: the expansion
// writes K^C and V in fp16, and the bf16 query parts and k^R are exact in
// fp16, so the only roundings past the inputs are K^C, V, the rotated q^R and
// P (11-bit mantissas) and the bf16 output.
// * warp 0 issues TMA loads: the tile's q^C (two 64-column boxes), then per
//   128-key tile K^C (two boxes) and k^R (one box, read from the cache rows)
//   into one of two K stages and V (two boxes) into one of two V stages;
// * warp 1 issues the MMAs: S = Q K^T (M=128 queries, N=128 keys, K=192, A and
//   B in shared memory) into TMEM, and O += P V (K=128 keys, A = P in TMEM,
//   B = the V stage read MN-major) with the next tile's S issued before the
//   current O so that the softmax of one tile overlaps the other's MMAs;
// * warps 2 and 3 turn each K stage's k^R box from bf16 into fp16 in place;
// * warps 4..7 own one query row per thread (TMEM lane = row): they turn the
//   row's q^C into fp16 and write RoPE_t(q^R) into the third Q box, then per
//   key tile read the row of S, mask the diagonal tile, keep a running max in
//   log2 units (raised only when a tile's max exceeds it by more than 8, which
//   bounds every exp2 argument by 8 and keeps the result exact), write P
//   (fp16) to TMEM and rescale O's row when the max moved; at the end O / l
//   goes out as bf16 with the row's lse.
// Every wait is bounded (MLA_ERR_DEVICE_TIMEOUT, with the wait's site).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kPq = 128;                     // queries per tile
constexpr int kPk = 128;                     // keys per tile
constexpr int kPdh = 128, kPdhr = 64, kPdc = 512, kPwidth = kPdc + kPdhr;
constexpr uint32_t kPBox = 128 * 128;        // one 64-column 16-bit box of 128 rows (16 KB, 128B swizzle)
constexpr int kPStages = 2;
constexpr uint32_t kPOffQ = 0;                                  // q^C | q^C | RoPE(q^R)
constexpr uint32_t kPOffK = kPOffQ + 3 * kPBox;                 // stages of K^C | K^C | k^R
constexpr uint32_t kPOffV = kPOffK + kPStages * 3 * kPBox;      // stages of V | V
constexpr uint32_t kPOffBars = kPOffV + kPStages * 2 * kPBox;
constexpr uint32_t kPSmem = kPOffBars + 1024 + 1024;            // + alignment slack
static_assert(kPSmem <= 232448, "shared memory per CTA");
constexpr uint32_t kPTmemS = 0, kPTmemO = 128, kPTmemP = 256;   // fp32 S | fp32 O | fp16 P (packed pairs)
constexpr int kPThreads = 256;
constexpr int kPFirstRowWarp = 4;
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kPRescale = 8.0f;

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// two bf16 values (one 32-bit word) as fp16x2
__device__ __forceinline__ uint32_t bf16x2_as_f16x2(uint32_t w) {
  return pack_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

struct PrefillMaps {
  CUtensorMap qc;  // q^C as [P, n_h * d_h]
  CUtensorMap k;   // K^C as [P, n_h * d_h]
  CUtensorMap v;   // V as [P, n_h * d_h]
  CUtensorMap kr;  // the cache rows [P, d_c + d_hR] (k^R = columns d_c..)
};

struct PrefillParams {
  int P, n_h;
  const __nv_bfloat16* q_r;  // [P, n_h, d_hR], before RoPE
  const float* rope_cos;     // [max_pos, d_hR / 2]
  const float* rope_sin;
  float scale_log2;          // log2(e) / sqrt(d_h + d_hR)
  __nv_bfloat16* o;          // [P, n_h, d_h]
  float* lse;                // [P, n_h]
  int* status;
  long long wait_limit;
};

struct PrefillBars {
  uint64_t q_full, q_rope;
  uint64_t k_full[kPStages], kr_ready[kPStages], k_empty[kPStages], v_full[kPStages], v_empty[kPStages];
  uint64_t s_full, s_free, p_full, o_done, drain;
  uint32_t tmem;
  int abort;
};

// Bounded wait (site numbers: producer 1 K stage free, 2 V stage free; MMA
// warp 3 query ready, 4 K ready, 5 S read, 6 P written, 7 V landed; row
// warps 8 S ready, 9 previous O MMA done, 10 last O MMA done, 11 query
// landed; k^R converters 12 K landed).
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, const PrefillParams& p, PrefillBars* bs,
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
__device__ __forceinline__ bool pf_wait_warp(uint64_t* bar, uint32_t parity, const PrefillParams& p, PrefillBars* bs,
                                             int site) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = pf_wait(bar, parity, p, bs, site);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__global__ void __launch_bounds__(kPThreads, 1)
    prefill_attn_kernel(const __grid_constant__ PrefillMaps maps, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PrefillBars* bs = reinterpret_cast<PrefillBars*>(smem + kPOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (p.P + kPq - 1) / kPq;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.x);  // the longest rows first
  const int head = blockIdx.y;
  const int n_kv = qt + 1;                                 // key tiles 0..qt (kPk == kPq)

  if (threadIdx.x == 0) {
    mbar_init(&bs->q_full, 1);
    mbar_init(&bs->q_rope, 4);
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&bs->k_full[s], 1);
      mbar_init(&bs->kr_ready[s], 2);  // the two warps that turn the k^R box into fp16
      mbar_init(&bs->k_empty[s], 1);
      mbar_init(&bs->v_full[s], 1);
      mbar_init(&bs->v_empty[s], 1);
    }
    mbar_init(&bs->s_full, 1);
    mbar_init(&bs->s_free, 4);
    mbar_init(&bs->p_full, 4);
    mbar_init(&bs->o_done, 1);
    mbar_init(&bs->drain, 1);
    bs->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bs->tmem, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bs->tmem;
  pdl_wait();  // queries, cache rows and the expanded keys and values come from earlier kernels

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.qc);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.kr);
      const uint64_t pol_q = l2_policy_evict_first();  // the query tile is read once
      const uint64_t pol_kv = l2_policy_evict_last();  // key tile j serves query tiles j..n_qt-1
      const int col = head * kPdh;
      mbar_arrive_expect_tx(&bs->q_full, 2 * kPBox);
      tma_load_2d_hint(smem + kPOffQ, &maps.qc, &bs->q_full, col, qt * kPq, pol_q);
      tma_load_2d_hint(smem + kPOffQ + kPBox, &maps.qc, &bs->q_full, col + 64, qt * kPq, pol_q);
      bool ok = true;
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int s = j & 1;
        if (j >= kPStages && !(ok = pf_wait(&bs->k_empty[s], ((j >> 1) - 1) & 1, p, bs, 1))) break;
        uint8_t* kst = smem + kPOffK + s * 3 * kPBox;
        mbar_arrive_expect_tx(&bs->k_full[s], 3 * kPBox);
        tma_load_2d_hint(kst, &maps.k, &bs->k_full[s], col, j * kPk, pol_kv);
        tma_load_2d_hint(kst + kPBox, &maps.k, &bs->k_full[s], col + 64, j * kPk, pol_kv);
        tma_load_2d_hint(kst + 2 * kPBox, &maps.kr, &bs->k_full[s], kPdc, j * kPk, pol_kv);
        ++k_issued;
        if (j >= kPStages && !(ok = pf_wait(&bs->v_empty[s], ((j >> 1) - 1) & 1, p, bs, 2))) break;
        uint8_t* vst = smem + kPOffV + s * 2 * kPBox;
        mbar_arrive_expect_tx(&bs->v_full[s], 2 * kPBox);
        tma_load_2d_hint(vst, &maps.v, &bs->v_full[s], col, j * kPk, pol_kv);
        tma_load_2d_hint(vst + kPBox, &maps.v, &bs->v_full[s], col + 64, j * kPk, pol_kv);
        ++v_issued;
      }
      if (!ok) {
        // every issued copy must land before the CTA may exit
        for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->q_full, 0); ++i) {
        }
        for (int j = k_issued > kPStages ? k_issued - kPStages : 0; j < k_issued; ++j)
          for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->k_full[j & 1], (j >> 1) & 1); ++i) {
          }
        for (int j = v_issued > kPStages ? v_issued - kPStages : 0; j < v_issued; ++j)
          for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->v_full[j & 1], (j >> 1) & 1); ++i) {
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_f16_f32(kPq, kPk, false, false);
    const uint32_t idesc_o = idesc_f16_f32(kPq, kPdh, false, true);  // V read MN-major
    const uint32_t q_addr = smem_u32(smem + kPOffQ);
    bool ok = pf_wait_warp(&bs->q_full, 0, p, bs, 3) && pf_wait_warp(&bs->q_rope, 0, p, bs, 3);
    // S(j) = Q K_j^T over the three 64-column boxes (q^C, q^C, RoPE(q^R))
    auto issue_s = [&](int j) -> bool {
      const int s = j & 1;
      if (!pf_wait_warp(&bs->kr_ready[s], (j >> 1) & 1, p, bs, 4)) return false;  // landed and converted
      if (j >= 1 && !pf_wait_warp(&bs->s_free, (j - 1) & 1, p, bs, 5)) return false;  // S(j-1) read out
      tc_fence_after();
      const uint32_t k_addr = smem_u32(smem + kPOffK + s * 3 * kPBox);
#pragma unroll
      for (int b = 0; b < 3; ++b)
        mma_ss_kblock_elect<2, 2>(tmem + kPTmemS, smem_desc(q_addr + b * kPBox, 16, 1024, kSwizzle128B),
                                  smem_desc(k_addr + b * kPBox, 16, 1024, kSwizzle128B), idesc_s, b > 0 ? 1u : 0u);
      mma_commit_elect(&bs->s_full);
      mma_commit_elect(&bs->k_empty[s]);
      return true;
    };
    if (ok) {
      tc_fence_after();
      ok = issue_s(0);
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      if (j + 1 < n_kv && !(ok = issue_s(j + 1))) break;
      const int s = j & 1;
      if (!(ok = pf_wait_warp(&bs->p_full, j & 1, p, bs, 6))) break;
      if (!(ok = pf_wait_warp(&bs->v_full[s], (j >> 1) & 1, p, bs, 7))) break;
      tc_fence_after();
      // O += P V_j: eight K-steps of 16 keys (8 packed P columns, 16 rows of
      // 128 B of the V stage = 2048 B = 128 descriptor units per step)
      const uint64_t vd = smem_desc(smem_u32(smem + kPOffV + s * 2 * kPBox), kPBox, 1024, kSwizzle128B);
#pragma unroll
      for (int k = 0; k < kPk / 16; ++k)
        mma_ts_elect(tmem + kPTmemO, tmem + kPTmemP + 8 * k, vd + 128 * k, idesc_o, (j > 0 || k > 0) ? 1u : 0u);
      mma_commit_elect(&bs->o_done);
      mma_commit_elect(&bs->v_empty[s]);
    }
    if (!ok) {
      // every issued MMA must finish before TMEM is released
      mma_commit_elect(&bs->drain);
      for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->drain, 0); ++i) {
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ k^R to fp16
    // The cache rows hold k^R in bf16; each K stage's k^R box becomes fp16 in
    // place (exact: bf16 values within the fp16 range) before its S MMA.
    const int tid = threadIdx.x - 64;  // 0..63
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int s = j & 1;
      if (!(ok = pf_wait(&bs->k_full[s], (j >> 1) & 1, p, bs, 12))) break;
      uint4* box = reinterpret_cast<uint4*>(smem + kPOffK + s * 3 * kPBox + 2 * kPBox);
#pragma unroll 4
      for (int i = tid; i < static_cast<int>(kPBox / 16); i += 64) {
        const uint4 w = box[i];
        box[i] = make_uint4(bf16x2_as_f16x2(w.x), bf16x2_as_f16x2(w.y), bf16x2_as_f16x2(w.z), bf16x2_as_f16x2(w.w));
      }
      fence_proxy_async_smem();  // the MMAs read the box through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&bs->kr_ready[s]);
    }
  } else if (warp >= kPFirstRowWarp) {
    // ------------------------------------------------------------ softmax rows
    const int w = warp - kPFirstRowWarp;  // TMEM lanes 32w..32w+31 (warp % 4 == w)
    const int r = 32 * w + lane;          // query row of the tile
    const int t = qt * kPq + r;           // its position in the prompt
    const bool live = t < p.P;
    const uint32_t lanes = static_cast<uint32_t>(32 * w) << 16;
    // the row's q^C (two boxes, as loaded) to fp16 in place, then RoPE_t(q^R)
    // as fp16 into the third Q box (row r, 128B swizzle: 16-byte chunk c at
    // position c ^ (r % 8)); pairs (2k, 2k+1) turn by t theta_k
    bool ok = pf_wait(&bs->q_full, 0, p, bs, 11);
    if (ok) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint4* qrow = reinterpret_cast<uint4*>(smem + kPOffQ + b * kPBox + r * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = qrow[c];
          qrow[c] = make_uint4(bf16x2_as_f16x2(x.x), bf16x2_as_f16x2(x.y), bf16x2_as_f16x2(x.z), bf16x2_as_f16x2(x.w));
        }
      }
      uint32_t rq[kPdhr / 2];
      if (live) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_r + (static_cast<size_t>(t) * p.n_h + head) * kPdhr);
        uint4 x[kPdhr / 8];
#pragma unroll
        for (int i = 0; i < kPdhr / 8; ++i) x[i] = __ldg(src + i);
        const float* cs = p.rope_cos + static_cast<size_t>(t) * (kPdhr / 2);
        const float* sn = p.rope_sin + static_cast<size_t>(t) * (kPdhr / 2);
#pragma unroll
        for (int k = 0; k < kPdhr / 2; ++k) {
          const uint4 xv = x[k / 4];
          const uint32_t wd = (k % 4 == 0) ? xv.x : (k % 4 == 1) ? xv.y : (k % 4 == 2) ? xv.z : xv.w;
          const float x0 = __uint_as_float(wd << 16), x1 = __uint_as_float(wd & 0xFFFF0000u);
          const float c = __ldg(cs + k), sv = __ldg(sn + k);
          rq[k] = pack_h2(x0 * c - x1 * sv, x0 * sv + x1 * c);
        }
      } else {
#pragma unroll
        for (int k = 0; k < kPdhr / 2; ++k) rq[k] = 0u;
      }
      uint8_t* row = smem + kPOffQ + 2 * kPBox + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) * 16)) = make_uint4(rq[4 * c], rq[4 * c + 1], rq[4 * c + 2], rq[4 * c + 3]);
      fence_proxy_async_smem();  // the MMAs read the box through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&bs->q_rope);
    }
    float m = -INFINITY, l = 0.f;  // running max (log2 units) and this row's sum
    for (int j = 0; j < n_kv && ok; ++j) {
      if (!(ok = pf_wait(&bs->s_full, j & 1, p, bs, 8))) break;
      tc_fence_after();
      uint32_t sv[kPk];
#pragma unroll
      for (int c = 0; c < kPk / 32; ++c) tmem_ld32(tmem + lanes + kPTmemS + 32 * c, sv + 32 * c);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bs->s_free);
      float x[kPk];
#pragma unroll
      for (int c = 0; c < kPk; ++c) x[c] = __uint_as_float(sv[c]);
      if (j == qt) {  // the diagonal tile: key j*128 + c is visible to row r when c <= r
#pragma unroll
        for (int c = 0; c < kPk; ++c)
          if (c > r) x[c] = -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c + 1 < kPk; c += 2) mx = max3(mx, x[c], x[c + 1]);
      mx = fmaxf(mx, x[kPk - 1]) * p.scale_log2;  // log2 units (the scale is positive)
      float mn = m, fa = 1.f;
      if (j == 0) {
        mn = mx;
      } else if (mx > m + kPRescale) {
        mn = mx;
        fa = ex2_approx(m - mx);
      }
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-mn, -mn);
      uint32_t pk[kPk / 2];
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < kPk / 2; ++c) {
        const float2 a = fma_f32x2(make_float2(x[2 * c], x[2 * c + 1]), sc2, nm2);
        const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        acc = add_f32x2(acc, e);
        pk[c] = pack_h2(e.x, e.y);
      }
      // P and O belong to O(j-1) until its MMA is done
      if (j >= 1 && !(ok = pf_wait(&bs->o_done, (j - 1) & 1, p, bs, 9))) break;
      tc_fence_after();
      if (__any_sync(0xffffffffu, fa != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < kPdh / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lanes + kPTmemO + 32 * c, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * fa);
          tmem_st32(tmem + lanes + kPTmemO + 32 * c, ov);
        }
      }
      tmem_st32(tmem + lanes + kPTmemP, pk);
      tmem_st32(tmem + lanes + kPTmemP + 32, pk + 32);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bs->p_full);
      l = l * fa + (acc.x + acc.y);
      m = mn;
    }
    if (ok) ok = pf_wait(&bs->o_done, (n_kv - 1) & 1, p, bs, 10);
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      __nv_bfloat16* dst = p.o + (static_cast<size_t>(t) * p.n_h + head) * kPdh;
#pragma unroll 1
      for (int c = 0; c < kPdh / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lanes + kPTmemO + 32 * c, ov);
        tmem_ld_wait();
        uint32_t ob[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) ob[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
        if (live) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(ob[4 * i], ob[4 * i + 1], ob[4 * i + 2], ob[4 * i + 3]);
        }
      }
      if (live) p.lse[static_cast<size_t>(t) * p.n_h + head] = (m + log2f(l)) * (1.f / kPLog2e);
      tc_fence_before();
    }
  }

  __syncthreads();
  if (threadIdx.x == 0) pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_prefill_attn_tc(const mla_handle* h, const void* rows, const void* q_c, const void* q_r, int P,
                                   const void* k_c, const void* v, void* o, float* lse, cudaStream_t s) {
  const mla_dims& d = h->dims;
  const long long cols = static_cast<long long>(d.n_h) * d.d_h;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  PrefillMaps maps;
  if (!tensor_map_2d(h, &maps.qc, q_c, cols, P, 64, kPq, sw) || !tensor_map_2d(h, &maps.k, k_c, cols, P, 64, kPk, sw) ||
      !tensor_map_2d(h, &maps.v, v, cols, P, 64, kPk, sw) || !tensor_map_2d(h, &maps.kr, rows, kPwidth, P, 64, kPk, sw))
    return cudaErrorInvalidValue;
  PrefillParams p;
  p.P = P;
  p.n_h = d.n_h;
  p.q_r = static_cast<const __nv_bfloat16*>(q_r);
  p.rope_cos = h->rope_cos;
  p.rope_sin = h->rope_sin;
  p.scale_log2 = d.scale * kPLog2e;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = h->status;
  p.wait_limit = h->wait_limit;
  cudaError_t e = kernel_attrs_once(h, reinterpret_cast<const void*>(prefill_attn_kernel), kPSmem, false);
  if (e != cudaSuccess) return e;
  return launch_pdl(prefill_attn_kernel, dim3((P + kPq - 1) / kPq, d.n_h), dim3(kPThreads), kPSmem, s, 1, maps, p);
}

}  // namespace mla
