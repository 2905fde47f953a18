// decode_tc.cu -- latent-cache attention on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ([qiita] "Attention 計算", absorbed form of [0h-n0]
// "行列吸収トリック" and [kasblo] "V側は、小さな表現の加重和を先に求める"):
//   s_ij  = scale * (q~_i . c_j + q^R_i . k^R_j)   for every cached row j <= t
//   o~_i  = sum_j softmax_j(s_ij) c_j,   lse_i = ln sum_j exp(s_ij)
// for all 128 heads i of one query token at once: the heads form the M = 128
// dimension of every MMA, each 64-row cache block is one key tile.
//
// Layout of the work (fixed sizes: n_h = 128, d_c = 512, d_hr = 64, block = 64):
// * A worker is a cluster of two CTAs.  The fp32 accumulator O for 128 heads x
//   512 latent columns fills one SM's TMEM, so it is split by columns: CTA c
//   owns latent columns [256c, 256c+256) and RoPE columns [512+32c, +32) of
//   every cached row and TMA-loads only those 288 columns of each tile (36 KB).
// * Scores: CTA c computes the partial score over its 288 columns,
//   S_c = Q~[:, own] . C[:, own]^T  (M=128, N=64, K=288), with its half of the
//   latent query (latent and RoPE parts) resident in TMEM as the A operand.
// * Each softmax ("row") warp owns 16 heads and writes their 16 x 64 block of
//   partial scores, scaled to log2 units and rounded to fp16, to its outbox;
//   the exchange warp ships it to the same warp's inbox in the peer CTA with
//   one bulk shared-to-shared copy (completion counted on the peer's mbarrier,
//   no fence), one tile ahead of the tile it combines, so the exchange hides
//   behind a tile of work.  The exchange is bound by the SM-to-SM network
//   (about 16 bytes per clock per SM on this part; bulk copies beat 16-byte
//   st.async stores by 1.6x), which is why only fp16 partials travel.  Each
//   CTA adds the peer's fp16 partial to its own fp32 partial and runs the
//   online softmax on the result; no softmax state is exchanged.  (The two
//   CTAs' scores differ by the fp16 rounding of one partial, a few 1e-4 in
//   log2 units; each CTA normalises its half of O with its own sum, so each
//   half is a consistent softmax average.)
// * Values: CTA c accumulates O[:, own 256 latent columns] += P . C[:, own]
//   (M=128, N=256, K=64) in TMEM, with P (bf16) in TMEM and the key tile read
//   again from the same shared-memory stage as an MN-major B operand.  No K or
//   V is ever expanded.
// * Two warps issue the MMAs: one the scores, one the values.  A tcgen05.mma
//   issue stalls while the tensor pipe's queue is full, so a single issuer
//   busy pushing an 18-MMA score batch could not see that P is ready; with two
//   issuers each kind goes in as soon as its inputs are.  S runs ahead of the
//   softmax: while the row warps turn tile t into probabilities they hold
//   S(t+1) in registers and the tensor pipe runs O(t-1) and S(t+2).  S has a
//   single TMEM buffer (O 256 + q~ 128 + q^R 16 + P 32 + S 64 = 496 of the 512
//   columns), so S(t+2) waits for every row warp to have read S(t+1); on the
//   B=64 x T=4096 workload a row warp waits about 490 of the tile's ~2600
//   cycles for its next S.
// * Rescaling of O is lazy: the running max only moves when a tile's max
//   exceeds it by more than 2^8, which keeps every exp2 argument <= 8 and the
//   result exact (numerator and denominator share the stale max).
// * The plan gives each worker either whole tokens (few tokens of similar
//   length) or a balanced contiguous range of the global tile list; split
//   pieces write fp32 partials that a separate log-sum-exp combine kernel
//   merges.
//
// Warp roles per CTA (384 threads): warp 0 = TMA producer, warp 1 = score
// MMA issuer + TMEM owner, warp 2 = value MMA issuer (each issuer runs its
// loop as a whole warp, one elected lane issues each batch of MMAs), warp 3 =
// exchange issuer, warps 4..11 = softmax warps of 16 heads each (16-lane TMEM
// shapes: thread t holds heads base + t/4 and base + t/4 + 8).  The softmax
// warps report progress to the issuers through release/acquire counters in
// shared memory; MMA completions reach them through mbarriers.
// Every wait is bounded; a wait that runs out records MLA_ERR_DEVICE_TIMEOUT,
// raises a CTA-wide abort flag and the roles drain and exit.
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

constexpr int kHeads = 128;
constexpr int kTile = 64;               // keys per tile = rows per cache block
constexpr int kBlockRows = 64;
constexpr int kWidth = 576;             // d_c + d_hr
constexpr int kDc = 512;
constexpr int kRopeSlots = 3;          // RoPE boxes live only until their score MMA
constexpr uint32_t kBoxBytes = kTile * 128;                 // 64 keys x 64 cols bf16 (128B swizzle)
constexpr uint32_t kRopeBoxBytes = kTile * 64;              // 64 keys x 32 cols bf16 (64B swizzle)
constexpr uint32_t kStageBytes = 4 * kBoxBytes;             // 32768: the latent columns of a tile
constexpr int kRowWarps = 8;                                // softmax warps: 16 heads each
constexpr uint32_t kXBlockBytes = 16 * kTile * 2;           // one warp's 16 heads x 64 keys fp16
constexpr uint32_t kXSlotBytes = kRowWarps * kXBlockBytes;  // all row warps
// Quantised cache rows (672 bytes: 512 int8 codes | 16 fp16 scales | 64 bf16
// k^R): a CTA's raw slot holds its 256 codes and 8 scales of every row of a tile.
constexpr int kQ8RowBytes = 672;
constexpr uint32_t kCodeBytes = kTile * 256, kScaleBytes = kTile * 16;
constexpr uint32_t kRawBytes = kCodeBytes + kScaleBytes + kRopeBoxBytes;  // codes | scales | RoPE box

// Shared memory of the two cache formats.  bf16 rows: five stages of the
// tile's latent columns and three RoPE slots.  Quantised rows: three raw
// slots (codes, scales and RoPE box as loaded) and three fp16 stages they are
// turned into, each with its RoPE box after the latent columns (so a stage
// and its RoPE box are freed together).
constexpr int kMaxRawSlots = 3;
template <bool Q8>
struct Layout {
  static constexpr int kStages = Q8 ? 3 : 5;
  static constexpr int kRawSlots = Q8 ? kMaxRawSlots : 0;
  static constexpr uint32_t kStageStride = kStageBytes + (Q8 ? kRopeBoxBytes : 0);
  static constexpr uint32_t kOffStages = 0;
  static constexpr uint32_t kOffRaw = kOffStages + kStages * kStageStride;
  static constexpr uint32_t kOffRope = kOffRaw + kRawSlots * kRawBytes;  // bf16 rows: the RoPE slots
  static constexpr uint32_t kOffInbox = kOffRope + (Q8 ? 0 : kRopeSlots * kRopeBoxBytes);
  static constexpr uint32_t kOffOutbox = kOffInbox + 2 * kXSlotBytes;  // one slot: a copy reads it long before reuse
  static constexpr uint32_t kOffBars = kOffOutbox + kXSlotBytes;
  static constexpr uint32_t kSmemBytes = kOffBars + 1024 + 1024;     // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kOffRaw % 1024 == 0 && kRawBytes % 1024 == 0 && kOffRope % 1024 == 0, "TMA destinations");
};
constexpr int kMaxStages = 5;
// TMEM columns (512 allocated): O half | Q~ latent half | Q~ RoPE half | P | S
// (bf16 operands hold two elements per 32-bit column)
constexpr uint32_t kTmemO = 0, kTmemQ = 256, kTmemQR = 384, kTmemP = 416, kTmemS = 448;
constexpr int kValueWarp = 2;                  // value-MMA issuer
constexpr int kXchgWarp = 3;                   // ships the softmax warps' partial blocks to the peer
constexpr int kFirstRowWarp = 4;               // softmax warps 4 .. 4 + kRowWarps - 1
constexpr int kThreads = 32 * (kFirstRowWarp + kRowWarps);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Maps {
  CUtensorMap latent;  // bf16 pool as [rows, 576], box 64 cols x 64 rows, 128B swizzle
  CUtensorMap rope;    // the RoPE columns: bf16 box 32 cols x 64 rows, or the same 64 bytes of a quantised row; 64B swizzle
  CUtensorMap codes;   // quantised pool as [rows, 672] bytes: box 256 x 64 rows (a CTA's codes)
  CUtensorMap scales;  // the same tensor: box 16 x 64 rows (a CTA's 8 scales)
};

struct Params {
  const __nv_bfloat16* q_lat;
  const int* block_table;
  const int* seq_lens;
  const int* cu_q;
  const int* prefix;  // [n_tok+1] tiles before each token (workspace)
  const int2* tok_info;      // [n_tok] (sequence, position) of each query token (workspace)
  const int* worker_plan;    // [workers][4] tile range [lo, hi) and first token of each worker (workspace)
  const int* plan_flags;     // [1] 1 when worker ranges split tokens (workspace)
  __nv_bfloat16* o_lat;
  float* lse;
  float* part_o;      // [2W][128][512]
  float* part_lse;    // [2W][128]
  int* status;
  long long wait_limit;
  int max_blocks, batch, n_tok, n_pool_blocks, workers;
  float scale_log2;
  // Up to two device ranges a later kernel reads (16-byte aligned, multiples
  // of 16 bytes; 0 bytes = unused), fetched into L2 while the cache streams.
  const uint8_t* pf_ptr[2];
  long long pf_bytes[2];
};

struct Bars {
  uint64_t full[kMaxStages], empty[kMaxStages], rope_empty[kRopeSlots];
  uint64_t raw_full[kMaxRawSlots], raw_empty[kMaxRawSlots];  // quantised cache: raw slot loaded / turned into a stage
  uint64_t s_full, p_free;
  // progress counters of the row warps, polled by the MMA issuers: query
  // tokens loaded into TMEM, S tiles read out of TMEM, P tiles written
  uint32_t n_q[kRowWarps], n_s_read[kRowWarps], n_p_done[kRowWarps];
  // outbox hand-off between row warp q and the exchange warp: blocks written,
  // blocks whose copy to the peer has finished reading the outbox
  uint32_t n_out_ready[kRowWarps], n_out_free[kRowWarps];
  uint64_t xin_full[2][kRowWarps];    // peer warp w's partial scores landed in inbox slot
  uint64_t inbox_free[2][kRowWarps];  // peer warp w has consumed the slot this CTA writes into
  uint64_t drain, drain_o;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");
constexpr uint32_t kBarSlot = kRowWarps * sizeof(uint64_t);  // stride of one slot of xin_full / inbox_free

// A bounded wait ran out (or another role's did): records the timeout, with
// the wait's site and tile the first time, and raises the CTA's abort flag.
// Sites: producer 1 stage free, 2 RoPE slot free; score issuer 3 query
// loaded, 4 stage landed, 5 S read by every row warp; value issuer 6 P
// written by every row warp; exchange warp 7 partial block written, 8 peer
// inbox slot free, 9 peer consumed the last blocks; row warps 10 outbox free,
// 12 S ready, 13 peer partial scores landed, 14 previous O MMA done, 16
// outbox free (epilogue), 17 last O MMA done (epilogue).
__device__ __forceinline__ bool timed_out(long long i, const Params& p, Bars* bs, int site) {
  if (i >= p.wait_limit || *reinterpret_cast<volatile int*>(&bs->abort)) {
    if (i >= p.wait_limit) report_site(p.status, site, -1);
    else report(p.status, MLA_ERR_DEVICE_TIMEOUT);
    atomicExch(&bs->abort, 1);
    return true;
  }
  return false;
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Params& p, Bars* bs, int site,
                                         bool cluster_scope = false) {
  // an already completed phase is seen by the cheaper non-blocking test
  if (cluster_scope ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity)) return true;
  for (long long i = 0;; ++i) {
    if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (timed_out(i, p, bs, site)) return false;
  }
}

// The same for a warp that runs converged: lane 0 polls, every lane gets the
// outcome (and elect.sync later picks lane 0, the lane that observed it).
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, const Params& p, Bars* bs, int site) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, p, bs, site);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// The same for the row warps' progress counters: every lane < kRowWarps polls
// one counter until all have reached `target` (bounded like wait_bar).
__device__ __forceinline__ bool wait_counters(const uint32_t* ctr, uint32_t target, const Params& p, Bars* bs,
                                              int site) {
  const int lane = threadIdx.x & 31;
  for (long long i = 0;; ++i) {
    const bool mine = lane >= kRowWarps || static_cast<int32_t>(ld_acquire_u32(ctr + lane) - target) >= 0;
    if (__all_sync(0xffffffffu, mine)) return true;
    bool out = false;
    if (lane == 0) out = timed_out(i, p, bs, site);
    if (__shfl_sync(0xffffffffu, out ? 1 : 0, 0)) return false;
  }
}

// All lanes of a warp poll one counter until it reaches `target` (bounded).
__device__ __forceinline__ bool wait_counter(const uint32_t* ctr, uint32_t target, const Params& p, Bars* bs,
                                             int site) {
  for (long long i = 0;; ++i) {
    if (static_cast<int32_t>(ld_acquire_u32(ctr) - target) >= 0) return true;
    if (timed_out(i, p, bs, site)) return false;
  }
}

// Contiguous slice [lo, hi) of the global tile list handled by worker g.
__device__ __forceinline__ void worker_range(int g, int workers, int total, int& lo, int& hi) {
  lo = static_cast<int>(static_cast<long long>(g) * total / workers);
  hi = static_cast<int>(static_cast<long long>(g + 1) * total / workers);
}

struct Unit {
  int n;          // query token
  int t0;         // tiles of all tokens before this one
  int ta, tb;     // tile range within the token
  int pos;        // token position (last visible key)
  int b;          // sequence
  int slot;       // partial slot, or -1 when the unit covers the whole token
};

// Iterates the units of a worker; every role walks the same list.  The plan
// kernel stored what a unit needs (tile prefix sums, each token's sequence and
// position, each worker's first token), so a unit costs one round of
// independent loads instead of chains of dependent searches.
struct UnitIter {
  int x, hi, n, first;
  __device__ bool next(const Params& p, int g, Unit& u) {
    while (x < hi) {
      const int t0 = __ldg(p.prefix + n), t1 = __ldg(p.prefix + n + 1);
      if (t1 <= x) { ++n; continue; }
      u.n = n;
      u.t0 = t0;
      u.ta = x - t0;
      u.tb = min(hi, t1) - t0;
      const int2 info = __ldg(p.tok_info + n);
      u.b = info.x;
      u.pos = info.y;
      const bool complete = (u.ta == 0 && u.tb == t1 - t0);
      u.slot = complete ? -1 : 2 * g + (first ? 0 : 1);
      first = 0;
      x = t0 + u.tb;
      ++n;
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ UnitIter make_iter(const Params& p, int g) {
  UnitIter it;
  const int4 wp = __ldg(reinterpret_cast<const int4*>(p.worker_plan) + g);
  it.x = wp.x;
  it.hi = wp.y;
  it.n = it.x < it.hi ? wp.z : 0;
  it.first = 1;
  return it;
}

// L2 prefetch of the ranges in Params, spread over the launch.  The ranges,
// taken end to end, are split between the two CTAs of a pair (CTA c takes
// the c-th half) and each half is cut into one piece per tile of the global
// tile list, so the extra HBM reads follow the cache stream's pace whatever
// the plan.  The score-MMA issuer, idle for most of a tile, asks for each
// tile's piece right after that tile's score MMAs.  A request occupies the
// SM's copy engine, which the stage loads and the score exchange also use:
// issued from the TMA producer, or for four or sixteen tiles at once, the
// requests lengthened the kernel more (by 5.5, 4.3 and 11 µs against 3.5 µs
// at B = 64, T = 4096).
constexpr int kL2PrefetchTiles = 1;
constexpr long long kL2PrefetchMaxRequest = 1ll << 30;  // bytes per request (the size operand is 32-bit)
// Bytes per (tile, CTA), a multiple of 16; 0 when nothing is to be fetched.
__device__ __forceinline__ long long l2_prefetch_piece(const Params& p, long long& tiles) {
  const long long total = p.pf_bytes[0] + p.pf_bytes[1];
  tiles = total > 0 ? static_cast<long long>(__ldg(p.prefix + p.n_tok)) : 0;
  return tiles > 0 ? ((total + 2 * tiles - 1) / (2 * tiles) + 15) & ~15ll : 0;
}
// Fetches CTA c's pieces of global tiles [first, first + n).
__device__ __forceinline__ void l2_prefetch_tiles(const Params& p, long long piece, long long tiles, long long first,
                                                  int n, uint32_t c) {
  long long off = (c * tiles + first) * piece, len = n * piece;
  for (int r = 0; r < 2 && len > 0; ++r) {
    const long long sz = p.pf_bytes[r];
    if (off >= sz) {
      off -= sz;
      continue;
    }
    const long long m = len < sz - off ? len : sz - off;
    for (long long d = 0; d < m; d += kL2PrefetchMaxRequest)
      bulk_prefetch_l2(p.pf_ptr[r] + off + d, static_cast<uint32_t>(m - d < kL2PrefetchMaxRequest ? m - d : kL2PrefetchMaxRequest));
    len -= m;
    off = 0;
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Physical pool row of tile t of sequence b (a bad table entry is reported
// and replaced by block 0).
__device__ __forceinline__ int tile_row(const Params& p, int b, int t) {
  int blk = t < p.max_blocks ? __ldg(p.block_table + static_cast<size_t>(b) * p.max_blocks + t) : -1;
  if (blk < 0 || blk >= p.n_pool_blocks) {
    report(p.status, MLA_ERR_DEVICE_BOUNDS);
    blk = 0;
  }
  return blk * kBlockRows;
}

// Two int8 codes of w (bytes j, j + 1) times the fp16 scale d2, as fp16x2:
// each biased code u = code + 128 goes into the mantissa of the fp16 number
// 1024 + u (one byte permute), 1152 is subtracted (exact: an integer below
// 2048) and the product with the scale is rounded once.
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t w_biased, uint32_t sel, __half2 d2) {
  const uint32_t bits = __byte_perm(w_biased, 0x64646464u, sel);
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&bits), __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  const __half2 r = __hmul2(v, d2);
  return *reinterpret_cast<const uint32_t*>(&r);
}
// Two bf16 values (one 32-bit word) as fp16x2 (exact for fp16-range values).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 r = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Quantised cache, warps 0 and 3: turn every tile's int8 codes into the fp16
// stage the MMAs read (the quantised path multiplies in fp16: an 11-bit
// mantissa keeps code x scale within one rounding of 2^-11).  Warp 0 converts
// rows 0..31 and warp 3 rows 32..63 of the tile (lane = a group of 8
// columns; value = code x its run's fp16 scale, rounded once, written in the
// 128B-swizzled layout a TMA load of 16-bit rows would give) and the same
// rows of the RoPE box, bf16 to fp16 in place; lane 0 of warp 0 also issues
// the TMA loads of the codes, scales and RoPE box, kRawSlots tiles ahead.
__device__ __noinline__ void dequantise_role(const Maps& maps, const Params& p, Bars* bs, uint8_t* smem, int g,
                                             uint32_t c, int warp, int lane) {
  using L = Layout<true>;
  const int half = warp == 0 ? 0 : 1;
  const bool loader = warp == 0 && lane == 0;
  const int4 wp = __ldg(reinterpret_cast<const int4*>(p.worker_plan) + g);
  const uint32_t total = wp.y > wp.x ? static_cast<uint32_t>(wp.y - wp.x) : 0u;
  const uint64_t pol = l2_policy_evict_first();  // every cache row is read once
  UnitIter li = make_iter(p, g);
  Unit lu;
  int lt = 0, lt_end = 0;
  uint32_t lit = 0;  // tiles whose loads were issued
  // issues the loads of the next tile of this worker (lane 0 of warp 0)
  auto load_next = [&]() -> bool {
    while (lt >= lt_end) {
      if (!li.next(p, g, lu)) return true;
      lt = lu.ta;
      lt_end = lu.tb;
    }
    constexpr uint32_t R = L::kRawSlots;
    const uint32_t r = lit % R;
    if (lit >= R && !wait_bar(&bs->raw_empty[r], ((lit / R) - 1) & 1, p, bs, 19)) return false;
    const int y = tile_row(p, lu.b, lt);
    uint8_t* raw = smem + L::kOffRaw + r * kRawBytes;
    mbar_arrive_expect_tx(&bs->raw_full[r], kRawBytes);
    tma_load_2d_hint(raw, &maps.codes, &bs->raw_full[r], 256 * c, y, pol);
    tma_load_2d_hint(raw + kCodeBytes, &maps.scales, &bs->raw_full[r], kDc + 16 * c, y, pol);
    tma_load_2d_hint(raw + kCodeBytes + kScaleBytes, &maps.rope, &bs->raw_full[r], kDc + 32 + 64 * c, y, pol);
    ++lt;
    ++lit;
    return true;
  };
  bool ok = true;
  if (loader) {
    tma_prefetch_desc(&maps.codes);
    tma_prefetch_desc(&maps.scales);
    tma_prefetch_desc(&maps.rope);
    for (int i = 0; i < L::kRawSlots && ok; ++i) ok = load_next();
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  const int box = lane >> 3, chunk = lane & 7;  // this lane's 8 columns: box `box`, 16-byte chunk `chunk`
  for (uint32_t k = 0; k < total && ok; ++k) {
    if (!(ok = wait_bar_warp(&bs->raw_full[k % L::kRawSlots], (k / L::kRawSlots) & 1, p, bs, 20))) break;
    const int s = k % L::kStages;
    if (k >= L::kStages && !(ok = wait_bar_warp(&bs->empty[s], ((k / L::kStages) - 1) & 1, p, bs, 1))) break;
    const uint8_t* raw = smem + L::kOffRaw + (k % L::kRawSlots) * kRawBytes;
    uint8_t* st = smem + L::kOffStages + s * L::kStageStride + box * kBoxBytes;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const int r = 32 * half + i;
      const uint2 cw = *reinterpret_cast<const uint2*>(raw + r * 256 + lane * 8);
      const __half d = *reinterpret_cast<const __half*>(raw + kCodeBytes + r * 16 + (lane >> 2) * 2);
      const __half2 d2 = __halves2half2(d, d);
      const uint32_t x0 = cw.x ^ 0x80808080u, x1 = cw.y ^ 0x80808080u;  // code + 128 in every byte
      const uint4 o = make_uint4(codes_to_f16x2(x0, 0x4140u, d2), codes_to_f16x2(x0, 0x4342u, d2),
                                 codes_to_f16x2(x1, 0x4140u, d2), codes_to_f16x2(x1, 0x4342u, d2));
      *reinterpret_cast<uint4*>(st + r * 128 + ((chunk ^ (r & 7)) * 16)) = o;
    }
    {
      // the RoPE box, rows [32 half, 32 half + 32) (2 KB, 512 contiguous
      // bytes a pass of the warp), into the stage's RoPE box at the same
      // (swizzled) positions
      const uint4* rs = reinterpret_cast<const uint4*>(raw + kCodeBytes + kScaleBytes + half * 2048);
      uint4* rd = reinterpret_cast<uint4*>(smem + L::kOffStages + s * L::kStageStride + kStageBytes + half * 2048);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = rs[32 * j + lane];
        rd[32 * j + lane] =
            make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
      }
    }
    fence_proxy_async_smem();  // the MMAs read the stage through the async proxy
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&bs->full[s]);
      mbar_arrive(&bs->raw_empty[k % L::kRawSlots]);
    }
    if (warp == 0) {
      bool okl = true;
      if (loader && lit < total) okl = load_next();
      ok = __shfl_sync(0xffffffffu, okl ? 1 : 0, 0) != 0;
    }
  }
  // every issued load must land before the CTA may exit
  if (!ok && loader) {
    constexpr uint32_t R = L::kRawSlots;
    for (uint32_t k = lit > R ? lit - R : 0; k < lit; ++k)
      for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->raw_full[k % R], (k / R) & 1); ++i) {
      }
  }
}

template <bool Q8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ Maps maps, const Params p) {
  using L = Layout<Q8>;
  constexpr int kStages = L::kStages;
  constexpr uint32_t kOffStages = L::kOffStages, kOffRope = L::kOffRope, kOffInbox = L::kOffInbox;
  constexpr uint32_t kOffOutbox = L::kOffOutbox, kOffBars = L::kOffBars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bs = reinterpret_cast<Bars*>(smem + kOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t c = cluster_ctarank();  // which half of the columns this CTA owns
  const uint32_t peer = c ^ 1u;
  const int g = blockIdx.x >> 1;         // worker index

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bs->full[s], Q8 ? 2 : 1);  // quantised cache: the two warps that turn codes into the stage
      mbar_init(&bs->empty[s], 1);
    }
    for (int r = 0; r < kMaxRawSlots; ++r) {
      mbar_init(&bs->raw_full[r], 1);
      mbar_init(&bs->raw_empty[r], 2);
    }
    for (int s = 0; s < kRopeSlots; ++s) mbar_init(&bs->rope_empty[s], 1);
    mbar_init(&bs->s_full, 1);
    for (int w = 0; w < kRowWarps; ++w)
      bs->n_q[w] = bs->n_s_read[w] = bs->n_p_done[w] = bs->n_out_ready[w] = bs->n_out_free[w] = 0;
    mbar_init(&bs->p_free, 1);
    for (int s = 0; s < 2; ++s)
      for (int w = 0; w < kRowWarps; ++w) {
        mbar_init(&bs->xin_full[s][w], 1);
        mbar_init(&bs->inbox_free[s][w], 1);
      }
    mbar_init(&bs->drain, 1);
    mbar_init(&bs->drain_o, 1);
    bs->abort = 0;
    fence_mbar_init();
    // first phase of every inbox barrier: one arrival (this one) + the bytes
    for (int s = 0; s < 2; ++s)
      for (int w = 0; w < kRowWarps; ++w) mbar_arrive_expect_tx(&bs->xin_full[s][w], kXBlockBytes);
  }
  if (warp == 1) {
    tmem_alloc(&bs->tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  cluster_arrive();  // peer barriers are initialised before any remote access
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = bs->tmem_base;
  pdl_wait();  // the plan, the latent queries and the cache rows are written by earlier kernels

  if (Q8 && (warp == 0 || warp == kXchgWarp)) {
    // ------------------------------------------------------------ quantised cache: loads and dequantisation
    if constexpr (Q8) dequantise_role(maps, p, bs, smem, g, c, warp, lane);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.latent);
      tma_prefetch_desc(&maps.rope);
      const uint64_t pol = l2_policy_evict_first();  // every cache row is read once
      UnitIter iter = make_iter(p, g);
      Unit u;
      uint32_t it = 0;
      bool ok = true;
      while (ok && iter.next(p, g, u)) {
        for (int t = u.ta; t < u.tb && ok; ++t, ++it) {
          const int s = it % kStages;
          if (it >= kStages) ok = wait_bar(&bs->empty[s], ((it / kStages) - 1) & 1, p, bs, 1);
          const int rs = it % kRopeSlots;
          if (ok && it >= kRopeSlots) ok = wait_bar(&bs->rope_empty[rs], ((it / kRopeSlots) - 1) & 1, p, bs, 2);
          if (!ok) break;
          const int y = tile_row(p, u.b, t);
          uint8_t* st = smem + kOffStages + s * kStageBytes;
          mbar_arrive_expect_tx(&bs->full[s], kStageBytes + kRopeBoxBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tma_load_2d_hint(st + j * kBoxBytes, &maps.latent, &bs->full[s], 256 * c + 64 * j, y, pol);
          tma_load_2d_hint(smem + kOffRope + rs * kRopeBoxBytes, &maps.rope, &bs->full[s], 512 + 32 * c, y, pol);
        }
      }
      // drain: every issued stage must land before the CTA may exit
      if (!ok) {
        for (uint32_t k = (it > kStages ? it - kStages : 0); k < it; ++k)
          for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->full[k % kStages], (k / kStages) & 1); ++i) {
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ score MMA issuer
    // The whole warp runs this loop (operands stay warp-uniform); one elected
    // lane issues each batch of MMAs.
    {
      const uint32_t idesc_s = Q8 ? idesc_f16_f32(128, kTile, false, false) : idesc_bf16_f32(128, kTile, false, false);
      long long pf_tiles;
      const long long pf_piece = l2_prefetch_piece(p, pf_tiles);
      UnitIter iter = make_iter(p, g);
      Unit u;
      uint32_t k = 0;  // S tiles issued (global); tile k sits in stage k % kStages
      uint32_t n_units = 0;
      bool ok = true;
      while (ok && iter.next(p, g, u)) {
        ok = wait_counters(bs->n_q, n_units + 1, p, bs, 3);
        ++n_units;
        if (!ok) break;
        tc_fence_after();
        for (int t = u.ta; t < u.tb && ok; ++t, ++k) {
          // S(k) into the single S buffer once the row warps have read S(k-1) out of it
          if (!(ok = wait_bar_warp(&bs->full[k % kStages], (k / kStages) & 1, p, bs, 4))) break;
          if (k >= 1 && !(ok = wait_counters(bs->n_s_read, k, p, bs, 5))) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + kOffStages + (k % kStages) * L::kStageStride);
          const uint32_t rope = Q8 ? st + kStageBytes : smem_u32(smem + kOffRope + (k % kRopeSlots) * kRopeBoxBytes);
          mma_score_tile_elect<kBoxBytes>(tmem + kTmemS, tmem + kTmemQ, tmem + kTmemQR,
                                          smem_desc(st, 16, 1024, kSwizzle128B),
                                          smem_desc(rope, 16, 512, kSwizzle64B), idesc_s);
          mma_commit_elect(&bs->s_full);
          if (!Q8) mma_commit_elect(&bs->rope_empty[k % kRopeSlots]);
          // a worker's tiles are consecutive in the global list
          if (pf_piece && k % kL2PrefetchTiles == 0 && lane == 0)
            l2_prefetch_tiles(p, pf_piece, pf_tiles, u.t0 + t, kL2PrefetchTiles, c);
        }
      }
      if (!ok) {
        // every issued MMA must finish before TMEM is released
        mma_commit_elect(&bs->drain);
        for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->drain, 0); ++i) {
        }
      }
    }
  } else if (warp == kValueWarp) {
    // ------------------------------------------------------------ value MMA issuer
    {
      const uint32_t idesc_o = Q8 ? idesc_f16_f32(128, 256, false, true) : idesc_bf16_f32(128, 256, false, true);
      UnitIter iter = make_iter(p, g);
      Unit u;
      uint32_t k = 0;  // O MMAs issued (global)
      bool ok = true;
      while (ok && iter.next(p, g, u)) {
        for (int t = u.ta; t < u.tb && ok; ++t, ++k) {
          // P(k) is in TMEM (and S(k) done, so the stage has landed)
          if (!(ok = wait_counters(bs->n_p_done, k + 1, p, bs, 6))) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + kOffStages + (k % kStages) * L::kStageStride);
          mma_value_tile_elect<kTile / 16>(tmem + kTmemO, tmem + kTmemP, smem_desc(st, kBoxBytes, 1024, kSwizzle128B),
                                           idesc_o, t > u.ta ? 1u : 0u);
          mma_commit_elect(&bs->p_free);
          mma_commit_elect(&bs->empty[k % kStages]);
        }
      }
      if (!ok) {
        mma_commit_elect(&bs->drain_o);
        for (long long i = 0; i < p.wait_limit && !mbar_try_wait(&bs->drain_o, 0); ++i) {
        }
      }
    }
  } else if (warp >= kFirstRowWarp) {
    // ------------------------------------------------------------ row warps
    // Softmax warp rw owns 16 heads: TMEM lanes 32q + 16hh .. +16 of its
    // quadrant q, read and written with the 16-lane shapes.  Thread t holds
    // heads ha = 32q + 16hh + t/4 and ha + 8 and, of every 64-key tile, the
    // key pairs 4j + t%4 (keys 8j + 2(t%4), +1; j = 0..7): register pair k =
    // 2j + e is key pair 4j + t%4 of head ha (e = 0) or ha + 8 (e = 1).  The
    // four threads of a head share its running max through two shuffles.
    const int rw = warp - kFirstRowWarp;
    const int q = warp & 3;
    const int hh = rw >> 2;
    const int t4 = lane & 3;
    const int ha = q * 32 + hh * 16 + (lane >> 2);
    const int tr = threadIdx.x - 32 * kFirstRowWarp;  // 0..255 among the row warps
    const uint32_t lane16 = static_cast<uint32_t>(q * 32 + hh * 16) << 16;
    const uint32_t lane32 = static_cast<uint32_t>(q * 32) << 16;
    // this warp's 2 KB block of inbox slot s sits at inbox0 + s * kXSlotBytes,
    // at the same offset in the peer; row = thread (64 B), 16-byte chunks XOR-swizzled
    const uint8_t* const inbox0 = smem + kOffInbox + rw * kXBlockBytes;
    uint8_t* const outbox = smem + kOffOutbox + rw * kXBlockBytes;
    const uint32_t peer_free0 = map_to_rank(smem_u32(&bs->inbox_free[0][rw]), peer);
    // quantised cache: this warp ships its own blocks (warp 3 dequantises)
    const uint32_t peer_inbox_rw = map_to_rank(smem_u32(inbox0), peer);
    const uint32_t peer_xin_rw = map_to_rank(smem_u32(&bs->xin_full[0][rw]), peer);
    const int sw = (lane >> 1) & 3;
    const float2 scale2 = make_float2(p.scale_log2, p.scale_log2);
    UnitIter iter = make_iter(p, g);
    Unit u;
    uint32_t n_s = 0;      // S tiles read out of TMEM (global)
    uint32_t n_send = 0;   // partial blocks sent to the peer
    uint32_t n_recv = 0;   // partial blocks received from it
    uint32_t n_p = 0;      // P tiles written (global) = tile index for the stage ring
    uint32_t n_units_q = 0;  // query tokens loaded
    bool ok = true;

    // Reads this thread's 32 scores of S out of TMEM, scaled to log2 units
    // (kept in `own`, fp32), and hands their fp16 rounding to the exchange warp.
    auto send = [&](float2* own) -> bool {
      if (!wait_bar(&bs->s_full, n_s & 1, p, bs, 12)) return false;
      ++n_s;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld_16x256b_x8(tmem + lane16 + kTmemS, v);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) st_release_u32(&bs->n_s_read[rw], n_s);
      uint32_t h[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        own[k] = mul_f32x2(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), scale2);
        h[k] = pack_half2(own[k].x, own[k].y);
      }
      // the copy of the previous block has read the outbox
      if constexpr (Q8) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      } else {
        if (n_send >= 1 && !wait_counter(&bs->n_out_free[rw], n_send, p, bs, 10)) return false;
      }
      uint8_t* row = outbox + lane * 64;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4*>(row + ((ch ^ sw) * 16)) = make_uint4(h[4 * ch], h[4 * ch + 1], h[4 * ch + 2], h[4 * ch + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if constexpr (Q8) {
        // into inbox slot n_send % 2 of the peer's same warp, once the peer has
        // consumed what went there two blocks ago
        const uint32_t slot = n_send & 1;
        if (n_send >= 2 && !wait_bar(&bs->inbox_free[slot][rw], ((n_send >> 1) - 1) & 1, p, bs, 8, true))
          return false;
        if (lane == 0) {
          bulk_copy_to_peer(peer_inbox_rw + slot * kXSlotBytes, outbox, kXBlockBytes, peer_xin_rw + slot * kBarSlot);
          bulk_commit();
        }
      } else {
        if (lane == 0) st_release_u32(&bs->n_out_ready[rw], n_send + 1);  // the exchange warp ships it
      }
      ++n_send;
      return true;
    };

    while (ok && iter.next(p, g, u)) {
      // ---- latent query: the first softmax warp of each quadrant writes its
      // 32 heads' own 256 latent + 32 RoPE columns (thread = head = TMEM lane)
      if (hh == 0) {
        const int r = q * 32 + lane;
        const uint4* src = reinterpret_cast<const uint4*>(p.q_lat + (static_cast<size_t>(u.n) * kHeads + r) * kWidth + 256 * c);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t v[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w = __ldg(src + ch * 4 + j);
            v[4 * j] = w.x; v[4 * j + 1] = w.y; v[4 * j + 2] = w.z; v[4 * j + 3] = w.w;
          }
          if constexpr (Q8) {  // the quantised path's MMAs take fp16 operands
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = bf16x2_to_f16x2(v[j]);
          }
          tmem_st16(tmem + lane32 + kTmemQ + ch * 16, v);
        }
        const uint4* rsrc = reinterpret_cast<const uint4*>(p.q_lat + (static_cast<size_t>(u.n) * kHeads + r) * kWidth + 512 + 32 * c);
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = __ldg(rsrc + j);
          v[4 * j] = w.x; v[4 * j + 1] = w.y; v[4 * j + 2] = w.z; v[4 * j + 3] = w.w;
        }
        if constexpr (Q8) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = bf16x2_to_f16x2(v[j]);
        }
        tmem_st16(tmem + lane32 + kTmemQR, v);
        tmem_st_wait();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) st_release_u32(&bs->n_q[rw], n_units_q + 1);
      ++n_units_q;
      const int n = u.tb - u.ta;
      float2 cur[16], nxt[16];  // this thread's key pairs of the tile being combined / the next tile
      if (!(ok = send(cur))) break;
      // running max of heads ha / ha + 8 (the same in the head's four threads)
      // and this thread's partial row sums
      float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
      for (int tt = 0; tt < n && ok; ++tt) {
        const int t = u.ta + tt;
        if (tt + 1 < n && !(ok = send(nxt))) break;
        // ---- 1. s = own + peer partial scores of this tile (log2 units)
        const uint32_t rslot = n_recv & 1;
        {
          if (!(ok = wait_bar(&bs->xin_full[rslot][rw], (n_recv >> 1) & 1, p, bs, 13, true))) break;
          ++n_recv;
          if (lane == 0) mbar_arrive_expect_tx(&bs->xin_full[rslot][rw], kXBlockBytes);  // arm the next phase
          const uint8_t* row = inbox0 + rslot * kXSlotBytes + lane * 64;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint4 w = *reinterpret_cast<const uint4*>(row + ((ch ^ sw) * 16));
            cur[4 * ch] = add_f32_f16x2(cur[4 * ch], w.x);
            cur[4 * ch + 1] = add_f32_f16x2(cur[4 * ch + 1], w.y);
            cur[4 * ch + 2] = add_f32_f16x2(cur[4 * ch + 2], w.z);
            cur[4 * ch + 3] = add_f32_f16x2(cur[4 * ch + 3], w.w);
          }
        }
        // ---- 2. online softmax in the log2 domain, causal mask on the last tile
        const int valid = min(kTile, u.pos - t * kTile + 1);  // keys of this tile the token sees
        if (valid < kTile) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int key = 8 * (k >> 1) + 2 * t4;
            if (key >= valid) cur[k].x = -INFINITY;
            if (key + 1 >= valid) cur[k].y = -INFINITY;
          }
        }
        // tile max of each head: this thread's 16 scores, then its three partners
        float xa = max3(max3(cur[0].x, cur[0].y, cur[2].x), max3(cur[2].y, cur[4].x, cur[4].y),
                        max3(cur[6].x, cur[6].y, cur[8].x));
        xa = max3(xa, max3(cur[8].y, cur[10].x, cur[10].y), max3(cur[12].x, cur[12].y, fmaxf(cur[14].x, cur[14].y)));
        float xb = max3(max3(cur[1].x, cur[1].y, cur[3].x), max3(cur[3].y, cur[5].x, cur[5].y),
                        max3(cur[7].x, cur[7].y, cur[9].x));
        xb = max3(xb, max3(cur[9].y, cur[11].x, cur[11].y), max3(cur[13].x, cur[13].y, fmaxf(cur[15].x, cur[15].y)));
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
        float mua = ma, mub = mb, fa = 1.f, fb = 1.f;
        if (tt == 0) {
          mua = xa;
          mub = xb;
        } else {
          if (xa > ma + kRescaleThreshold) { mua = xa; fa = ex2_approx(ma - xa); }
          if (xb > mb + kRescaleThreshold) { mub = xb; fb = ex2_approx(mb - xb); }
        }
        const float2 nma = make_float2(-mua, -mua), nmb = make_float2(-mub, -mub);
        uint32_t pk[16];
        float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 x = add_f32x2(cur[k], (k & 1) ? nmb : nma);
          const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (k & 1) sb = add_f32x2(sb, e); else sa = add_f32x2(sa, e);
          pk[k] = Q8 ? pack_half2(e.x, e.y) : pack_bf16x2(e.x, e.y);
        }
        la = (tt == 0) ? sa.x + sa.y : la * fa + (sa.x + sa.y);
        lb = (tt == 0) ? sb.x + sb.y : lb * fb + (sb.x + sb.y);
        ma = mua;
        mb = mub;
        // ---- 3. the previous O MMA is done (P is free); rescale O if a max moved; write P
        if (n_p >= 1 && !(ok = wait_bar(&bs->p_free, (n_p - 1) & 1, p, bs, 14))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, fa != 1.f || fb != 1.f)) {
#pragma unroll 1
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t v[16];
            tmem_ld_16x256b_x4(tmem + lane16 + kTmemO + ch * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * ((j & 2) ? fb : fa));
            tmem_st_16x256b_x4(tmem + lane16 + kTmemO + ch * 32, v);
          }
        }
        tmem_st_16x128b_x8(tmem + lane16 + kTmemP, pk);
        tmem_st_wait();
        // rows past the token's position may hold anything: zero them for the O MMA
        if (valid < kTile) {
          uint8_t* st = smem + kOffStages + (n_p % kStages) * L::kStageStride;
          for (int idx = tr; idx < (kTile - valid) * 32; idx += 32 * kRowWarps) {
            const int row = valid + (idx >> 5), box = (idx >> 3) & 3, ch = idx & 7;
            *reinterpret_cast<uint4*>(st + box * kBoxBytes + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();  // each warp's P counter release covers its own share
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          st_release_u32(&bs->n_p_done[rw], n_p + 1);
          mbar_arrive_relaxed_cluster(peer_free0 + rslot * kBarSlot);  // its values are consumed
        }
        ++n_p;
#pragma unroll
        for (int k = 0; k < 16; ++k) cur[k] = nxt[k];
      }
      if (!ok) break;
      // ---- epilogue: O / l for heads ha, ha + 8 and this CTA's 256 latent columns
      la += __shfl_xor_sync(0xffffffffu, la, 1);
      lb += __shfl_xor_sync(0xffffffffu, lb, 1);
      la += __shfl_xor_sync(0xffffffffu, la, 2);
      lb += __shfl_xor_sync(0xffffffffu, lb, 2);
      if (!(ok = wait_bar(&bs->p_free, (n_p - 1) & 1, p, bs, 17))) break;
      tc_fence_after();
      const float inv_la = 1.f / la, inv_lb = 1.f / lb;
      // O leaves TMEM in 32-column chunks staged through this warp's (idle)
      // outbox block (16 rows x 128 B fp32, 8-byte slots XOR-swizzled by row)
      // so that every global store covers whole row segments.
      if constexpr (Q8) {  // no copy still reads the outbox
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      } else {
        if (!(ok = wait_counter(&bs->n_out_free[rw], n_send, p, bs, 16))) break;
      }
      uint8_t* const stg = outbox;
      const int ra = lane >> 2;  // staging rows ra (head ha) and ra + 8 (head ha + 8)
      const size_t row0 = static_cast<size_t>(u.slot < 0 ? u.n : u.slot) * kHeads + q * 32 + hh * 16;
#pragma unroll 1
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t v[16];
        tmem_ld_16x256b_x4(tmem + lane16 + kTmemO + ch * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 4 * j + t4;  // float2 slot of columns 8j + 2 t4, +1
          *reinterpret_cast<float2*>(stg + ra * 128 + 8 * (e ^ (4 * (ra & 3)))) =
              make_float2(__uint_as_float(v[4 * j]) * inv_la, __uint_as_float(v[4 * j + 1]) * inv_la);
          *reinterpret_cast<float2*>(stg + (ra + 8) * 128 + 8 * (e ^ (4 * ((ra + 8) & 3)))) =
              make_float2(__uint_as_float(v[4 * j + 2]) * inv_lb, __uint_as_float(v[4 * j + 3]) * inv_lb);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 4 * i + (lane >> 3), cu = lane & 7;  // row, 16-byte unit of 4 columns
          const float4 w = *reinterpret_cast<const float4*>(stg + rr * 128 + 16 * (cu ^ (2 * (rr & 3))));
          const size_t off = (row0 + rr) * kDc + 256 * c + ch * 32 + 4 * cu;
          if (u.slot < 0)
            *reinterpret_cast<uint2*>(p.o_lat + off) = make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w));
          else
            *reinterpret_cast<float4*>(p.part_o + off) = w;
        }
        __syncwarp();
      }
      if (c == 0 && t4 == 0) {
        const float lse_a = (ma + log2f(la)) * 0.69314718055994531f, lse_b = (mb + log2f(lb)) * 0.69314718055994531f;
        float* dst = u.slot < 0 ? p.lse + static_cast<size_t>(u.n) * kHeads : p.part_lse + static_cast<size_t>(u.slot) * kHeads;
        dst[ha] = lse_a;
        dst[ha + 8] = lse_b;
      }
      tc_fence_before();
    }
    if constexpr (Q8) {
      // copies into the peer must have landed before the final cluster barrier
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  } else if (!Q8 && warp == kXchgWarp) {
    // ------------------------------------------------------------ exchange issuer
    // Lane rw ships softmax warp rw's fp16 partial block of every tile to the
    // same warp's inbox in the peer: once the block is written, and once the peer
    // has consumed what it received into that inbox slot two tiles ago.  This
    // keeps the copy issue and its waits off the softmax warps' chain.
    const int rw = lane & (kRowWarps - 1);
    const uint8_t* const outbox_rw = smem + kOffOutbox + rw * kXBlockBytes;
    const uint32_t peer_inbox_rw = map_to_rank(smem_u32(smem + kOffInbox + rw * kXBlockBytes), peer);
    const uint32_t peer_xin_rw = map_to_rank(smem_u32(&bs->xin_full[0][rw]), peer);
    UnitIter iter = make_iter(p, g);
    Unit u;
    uint32_t i = 0;  // blocks shipped per row warp
    bool ok = true;
    while (ok && iter.next(p, g, u)) {
      for (int t = u.ta; t < u.tb && ok; ++t, ++i) {
        if (!(ok = wait_counters(bs->n_out_ready, i + 1, p, bs, 7))) break;
        const uint32_t slot = i & 1;
        bool good = true;
        if (lane < kRowWarps) {
          if (i >= 2) good = wait_bar(&bs->inbox_free[slot][rw], ((i >> 1) - 1) & 1, p, bs, 8, true);
          if (good) {
            bulk_copy_to_peer(peer_inbox_rw + slot * kXSlotBytes, outbox_rw, kXBlockBytes, peer_xin_rw + slot * kBarSlot);
            bulk_commit();
            bulk_wait_read<0>();
            st_release_u32(&bs->n_out_free[rw], i + 1);
          }
        }
        ok = __all_sync(0xffffffffu, good);
      }
    }
    // a copy into the peer must not outlive the peer: wait until the peer has
    // consumed everything shipped (its inbox_free arrivals)
    if (lane < kRowWarps) {
      bulk_wait_all();
      for (uint32_t k = (i > 2 ? i - 2 : 0); ok && k < i; ++k)
        ok = wait_bar(&bs->inbox_free[k & 1][rw], (k >> 1) & 1, p, bs, 9, true);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0) pdl_trigger();
  cluster_arrive();  // no CTA leaves while its peer may still touch its shared memory
  cluster_wait();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__device__ __forceinline__ int worker_of(long long x, int workers, int total) {
  int g = static_cast<int>(x * workers / total);
  while (g + 1 < workers && static_cast<long long>(g + 1) * total / workers <= x) ++g;
  while (g > 0 && static_cast<long long>(g) * total / workers > x) --g;
  return g;
}

constexpr int kPlanSmemSeqs = 4096;  // cu_q entries the plan kernel keeps in shared memory
// Whole tokens per worker when the longest token has at most this many tiles
// more than an even share: splitting costs each split worker a partial write
// and the call a combine pass, about that many tiles of work.
constexpr int kWholeTokenSlack = 12;

// The plan of a decode call, from the sequence metadata:
//   prefix[n]         = tiles of all tokens before n (tiles of token n = pos_n/64 + 1)
//   tok_info[n]       = (sequence, position) of token n
//   worker_plan[g]    = (lo, hi, first token, 0): worker g's range [lo, hi) of
//                       the global tile list and the token holding tile lo
//   plan_flags[0]     = 1 when ranges split tokens (the combine kernel merges)
// Two layouts: with no more tokens than workers and tokens of similar length,
// worker g takes token g whole (nothing to merge); otherwise the tile list is
// cut into W balanced contiguous ranges.  One CTA; cu_q sits in shared memory
// so that finding a token's sequence is a search in shared memory rather than
// a chain of dependent global loads.
__global__ void __launch_bounds__(1024) plan_kernel(const int* __restrict__ seq_lens, const int* __restrict__ cu_q,
                                                    int batch, int n_tok, int max_blocks, int workers,
                                                    int* __restrict__ prefix, int2* __restrict__ tok_info,
                                                    int* __restrict__ worker_plan, int* __restrict__ plan_flags,
                                                    int* status) {
  __shared__ int warp_sums[32];
  __shared__ int carry, max_tiles;
  __shared__ int s_cu[kPlanSmemSeqs + 1];
  // The plan reads only the caller's sequence metadata, which no kernel of the
  // library writes, and its outputs are read only by this call's decode and
  // combine kernels: it runs while the previous kernel finishes and waits for
  // it only before exiting, so that a kernel waiting on the plan has the
  // previous kernel's results too.
  if (threadIdx.x == 0) pdl_trigger();  // the decode CTAs may set up meanwhile
  const bool cu_smem = batch <= kPlanSmemSeqs;
  if (cu_smem)
    for (int i = threadIdx.x; i <= batch; i += blockDim.x) s_cu[i] = __ldg(cu_q + i);
  if (threadIdx.x == 0) { carry = 0; max_tiles = 0; prefix[0] = 0; }
  if (threadIdx.x == 0 && __ldg(cu_q + batch) != n_tok) report(status, MLA_ERR_DEVICE_BOUNDS);
  __syncthreads();
  const int* cu = cu_smem ? s_cu : cu_q;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < n_tok; base += 1024) {
    const int n = base + threadIdx.x;
    int tiles = 0;
    if (n < n_tok) {
      const int b = seq_of_token(cu, batch, n);
      const int c0 = cu[b], c1 = cu[b + 1];
      const int pos = __ldg(seq_lens + b) - (c1 - n);
      if (pos < 0 || n < c0 || n >= c1 || pos / kBlockRows >= max_blocks) {
        report(status, MLA_ERR_DEVICE_BOUNDS);
        tiles = pos >= 0 ? min(pos / kTile + 1, max_blocks * (kBlockRows / kTile)) : 0;
      } else {
        tiles = pos / kTile + 1;
      }
      tok_info[n] = make_int2(b, pos);
      atomicMax(&max_tiles, tiles);
    }
    int v = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = v + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    if (n < n_tok) prefix[n + 1] = incl;
    __syncthreads();
    if (threadIdx.x == 1023) carry = incl;
    __syncthreads();
  }
  const int total = carry;
  const bool whole = n_tok <= workers && max_tiles <= (total + workers - 1) / workers + kWholeTokenSlack;
  if (threadIdx.x == 0) plan_flags[0] = whole ? 0 : 1;
  for (int g = threadIdx.x; g < workers; g += blockDim.x) {
    int lo, hi;
    if (whole) {
      lo = g < n_tok ? prefix[g] : total;  // prefix written above by this CTA
      hi = g < n_tok ? prefix[g + 1] : total;
    } else {
      worker_range(g, workers, total, lo, hi);
    }
    worker_plan[4 * g] = lo;
    worker_plan[4 * g + 1] = hi;
    worker_plan[4 * g + 2] = whole && g < n_tok ? g : 0;
    worker_plan[4 * g + 3] = 0;
  }
  if (whole || total <= 0) {
    pdl_wait();
    return;
  }
  __syncthreads();
  // balanced ranges: every worker's first tile g * total / W lies in exactly one token
  for (int n = threadIdx.x; n < n_tok; n += blockDim.x) {
    const int t0 = prefix[n], t1 = prefix[n + 1];
    if (t1 <= t0) continue;
    for (int g = worker_of(t0, workers, total); g < workers; ++g) {
      const long long lo = static_cast<long long>(g) * total / workers;
      if (lo >= t1) break;
      if (lo >= t0) worker_plan[4 * g + 2] = n;
    }
  }
  pdl_wait();
}

// Merge the pieces of every token whose keys were split across workers:
// lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s (the standard
// identity for a softmax split over disjoint key ranges; not on the pages).
// Each CTA takes (token, head) pairs blockIdx.x, blockIdx.x + gridDim.x, ...
// (at most eight CTAs per SM, so a call that split nothing costs one short
// wave of early exits); the pieces of a token are the workers g0..g1
// whose ranges meet its tiles.  Worker g wrote slot 2g when its range starts
// inside the token, else 2g+1 (its range started in an earlier token).  The
// pieces are spread over the CTA's eight warps (each lane holds 16 of the 512
// columns), so their loads are in flight together; the warps' sums meet in
// shared memory.
__device__ __forceinline__ int piece_slot(int k, int g0, int t0, int workers, int total) {
  const int g = g0 + k;
  int lo, hi;
  worker_range(g, workers, total, lo, hi);
  if (lo >= hi) return -1;  // an empty range wrote nothing
  return (k == 0 && lo < t0) ? 2 * g + 1 : 2 * g;
}

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(
    const int* __restrict__ prefix, const int* __restrict__ plan_flags, int n_tok, int workers,
    const float* __restrict__ part_o, const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ o_lat,
    float* __restrict__ lse) {
  __shared__ float s_red[kCombineWarps];
  __shared__ float4 s_acc[kCombineWarps][kDc / 4];
  pdl_wait();
  // The next decode call's plan may overwrite the plan data, so the next
  // kernel may launch only once every CTA has read all of it: CTAs that stop
  // here exit (an exit counts as the trigger); the others trigger once they
  // have read the plan values of their last pair (the merge itself reads only
  // the partials, which the next call rewrites only after this grid ends).
  if (__ldg(plan_flags) == 0) return;  // whole tokens per worker: nothing was split
  const int total = __ldg(prefix + n_tok);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int pair = blockIdx.x; pair < n_tok * kHeads; pair += gridDim.x) {
    const int n = pair / kHeads, h = pair % kHeads;
    const int t0 = __ldg(prefix + n), t1 = __ldg(prefix + n + 1);
    if (pair + static_cast<int>(gridDim.x) >= n_tok * kHeads) {  // this CTA's last pair
      __syncthreads();
      if (threadIdx.x == 0) pdl_trigger();
    }
    if (t1 <= t0) continue;
    const int g0 = worker_of(t0, workers, total), g1 = worker_of(t1 - 1, workers, total);
    if (g0 == g1) continue;  // whole token inside one worker: already final
    const int npieces = g1 - g0 + 1;
    // L = ln sum_s exp(lse_s), block-wide: max, then the sum of exponentials
    float mx = -INFINITY;
    for (int k = threadIdx.x; k < npieces; k += blockDim.x) {
      const int slot = piece_slot(k, g0, t0, workers, total);
      if (slot >= 0) mx = fmaxf(mx, __ldg(part_lse + static_cast<size_t>(slot) * kHeads + h));
    }
    mx = warp_max(mx);
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    mx = s_red[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, s_red[w]);
    __syncthreads();
    float sum = 0.f;
    for (int k = threadIdx.x; k < npieces; k += blockDim.x) {
      const int slot = piece_slot(k, g0, t0, workers, total);
      if (slot >= 0) sum += expf(__ldg(part_lse + static_cast<size_t>(slot) * kHeads + h) - mx);
    }
    sum = warp_sum(sum);
    if (lane == 0) s_red[warp] = sum;
    __syncthreads();
    sum = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) sum += s_red[w];
    const float L = mx + logf(sum);
    // o = sum_s exp(lse_s - L) o_s: warp w takes pieces w, w + 8, ...
    float4 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int k = warp; k < npieces; k += kCombineWarps) {
      const int slot = piece_slot(k, g0, t0, workers, total);
      if (slot < 0) continue;
      const float wk = expf(__ldg(part_lse + static_cast<size_t>(slot) * kHeads + h) - L);
      const float4* src = reinterpret_cast<const float4*>(part_o + (static_cast<size_t>(slot) * kHeads + h) * kDc);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v = __ldg(src + lane + 32 * j);
        acc[j].x += wk * v.x; acc[j].y += wk * v.y; acc[j].z += wk * v.z; acc[j].w += wk * v.w;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) s_acc[warp][lane + 32 * j] = acc[j];
    __syncthreads();
    // thread i finishes the 4 columns of float4 slot i (i < 128) of the 512
    if (threadIdx.x < kDc / 4) {
      float4 o = s_acc[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < kCombineWarps; ++w) {
        const float4 v = s_acc[w][threadIdx.x];
        o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
      }
      __nv_bfloat16* dst = o_lat + (static_cast<size_t>(n) * kHeads + h) * kDc + 4 * threadIdx.x;
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
    }
    if (threadIdx.x == 0) lse[static_cast<size_t>(n) * kHeads + h] = L;
    __syncthreads();  // s_red and s_acc are reused by the next pair
  }
}

bool encode_pool_maps(const mla_handle* h, Maps* maps, const void* pool, long long rows) {
  maps->codes = maps->scales = CUtensorMap{};
  return tensor_map_2d(h, &maps->latent, pool, kWidth, rows, 64, kTile, CU_TENSOR_MAP_SWIZZLE_128B) &&
         tensor_map_2d(h, &maps->rope, pool, kWidth, rows, 32, kTile, CU_TENSOR_MAP_SWIZZLE_64B);
}

// The quantised pool as [rows, 672] bytes: a CTA's 256 codes, its 8 scales
// and its 64 bytes of k^R per row.
bool encode_q8_pool_maps(const mla_handle* h, Maps* maps, const void* pool, long long rows) {
  maps->latent = CUtensorMap{};
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return tensor_map_2d(h, &maps->codes, pool, kQ8RowBytes, rows, 256, kTile, CU_TENSOR_MAP_SWIZZLE_NONE, u8) &&
         tensor_map_2d(h, &maps->scales, pool, kQ8RowBytes, rows, 16, kTile, CU_TENSOR_MAP_SWIZZLE_NONE, u8) &&
         tensor_map_2d(h, &maps->rope, pool, kQ8RowBytes, rows, 64, kTile, CU_TENSOR_MAP_SWIZZLE_64B, u8);
}

// plan -> decode -> combine, each allowed to launch while its predecessor finishes.
template <bool Q8>
cudaError_t launch_decode_kernels(const mla_handle* h, const Maps& maps, const Params& prm, int W, int n_tok,
                                  const int* seq_lens, const int* cu_q, int batch, int max_blocks, float* lse,
                                  int* status, cudaStream_t s) {
  cudaError_t e = launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, s, 1, seq_lens, cu_q, batch, n_tok, max_blocks, W,
                             const_cast<int*>(prm.prefix), const_cast<int2*>(prm.tok_info),
                             const_cast<int*>(prm.worker_plan), const_cast<int*>(prm.plan_flags), status);
  if (e != cudaSuccess) return e;
  constexpr int kSmemBytes = static_cast<int>(Layout<Q8>::kSmemBytes);
  e = kernel_attrs_once(h, reinterpret_cast<const void*>(decode_tc_kernel<Q8>), kSmemBytes, false);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_tc_kernel<Q8>, dim3(2 * W), dim3(kThreads), kSmemBytes, s, 1, maps, prm);
  if (e != cudaSuccess) return e;
  const int pairs = n_tok * kHeads, grid = pairs < 8 * h->num_sms ? pairs : 8 * h->num_sms;
  return launch_pdl(combine_kernel, dim3(grid), dim3(32 * kCombineWarps), 0, s, 1, static_cast<const int*>(prm.prefix),
                    prm.plan_flags, n_tok, W, static_cast<const float*>(prm.part_o), static_cast<const float*>(prm.part_lse), prm.o_lat,
                    lse);
}

int resolve_workers(const mla_handle* h, int num_workers) {
  return num_workers > 0 ? num_workers : max(1, h->num_sms / 2);
}

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of the decode workspace: plan (prefix sums, token info, worker
// ranges, layout flag), then the split-KV partial outputs and their
// log-sum-exps.
struct WsLayout {
  size_t prefix, tok_info, worker_plan, plan_flags, part_o, part_lse, total;
};
constexpr WsLayout ws_layout(size_t n_tok, size_t W) {
  WsLayout l{};
  l.prefix = 0;
  l.tok_info = l.prefix + align256(sizeof(int) * (n_tok + 1));
  l.worker_plan = l.tok_info + align256(sizeof(int2) * n_tok);
  l.plan_flags = l.worker_plan + align256(sizeof(int4) * W);
  l.part_o = l.plan_flags + 256;
  l.part_lse = l.part_o + align256(sizeof(float) * 2 * W * kHeads * kDc);
  l.total = l.part_lse + align256(sizeof(float) * 2 * W * kHeads);
  return l;
}

void set_workspace(Params& prm, uint8_t* w, const WsLayout& l) {
  prm.prefix = reinterpret_cast<const int*>(w + l.prefix);
  prm.tok_info = reinterpret_cast<const int2*>(w + l.tok_info);
  prm.worker_plan = reinterpret_cast<const int*>(w + l.worker_plan);
  prm.plan_flags = reinterpret_cast<const int*>(w + l.plan_flags);
  prm.part_o = reinterpret_cast<float*>(w + l.part_o);
  prm.part_lse = reinterpret_cast<float*>(w + l.part_lse);
}

}  // namespace

size_t decode_tc_workspace_bytes(const mla_handle* h, int n_tok, int num_workers) {
  return ws_layout(static_cast<size_t>(n_tok), static_cast<size_t>(resolve_workers(h, num_workers))).total;
}

cudaError_t launch_decode_tc(const mla_handle* h, const void* q_lat, const void* pool, int n_pool_blocks,
                             const int* block_table, int max_blocks, const int* seq_lens, const int* cu_q,
                             int batch, int n_tok, int num_workers, void* ws, size_t ws_bytes, void* o_lat,
                             float* lse, cudaStream_t s, bool q8) {
  const int W = resolve_workers(h, num_workers);
  Maps maps;
  const long long rows = static_cast<long long>(n_pool_blocks) * kBlockRows;
  if (!(q8 ? encode_q8_pool_maps(h, &maps, pool, rows) : encode_pool_maps(h, &maps, pool, rows)))
    return cudaErrorInvalidValue;
  Params prm{};
  set_workspace(prm, static_cast<uint8_t*>(ws), ws_layout(static_cast<size_t>(n_tok), static_cast<size_t>(W)));
  {
    std::lock_guard<std::mutex> lock(h->mu);
    for (int r = 0; r < 2; ++r) {
      prm.pf_ptr[r] = static_cast<const uint8_t*>(h->l2_prefetch_ptr[r]);
      prm.pf_bytes[r] = h->l2_prefetch_bytes[r];
    }
  }
  prm.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.cu_q = cu_q;
  prm.o_lat = static_cast<__nv_bfloat16*>(o_lat);
  prm.lse = lse;
  prm.status = h->status;
  prm.wait_limit = h->wait_limit;
  prm.max_blocks = max_blocks;
  prm.batch = batch;
  prm.n_tok = n_tok;
  prm.n_pool_blocks = n_pool_blocks;
  prm.workers = W;
  prm.scale_log2 = h->dims.scale * kLog2e;

  if (q8) return launch_decode_kernels<true>(h, maps, prm, W, n_tok, seq_lens, cu_q, batch, max_blocks, lse, h->status, s);
  return launch_decode_kernels<false>(h, maps, prm, W, n_tok, seq_lens, cu_q, batch, max_blocks, lse, h->status, s);
}


}  // namespace mla

namespace mla {
namespace {
// Waits on a barrier that nothing ever arrives at, with the bounded wait of
// the decode kernel; must return having recorded MLA_ERR_DEVICE_TIMEOUT.
__global__ void wait_timeout_selftest_kernel(int* status, long long wait_limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool done = false;
    for (long long i = 0; i < wait_limit && !done; ++i) done = mbar_try_wait(&bar, 0);
    if (!done) report_site(status, 1, -1);
    mbar_arrive(&bar);  // complete the phase so the barrier is idle at exit
  }
}
}  // namespace

cudaError_t launch_wait_timeout_selftest(const mla_handle* h, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(h->status, h->wait_limit);
  return cudaGetLastError();
}
}  // namespace mla

// ---------------------------------------------------------------------------
// Decode without caller-provided workspace.
//
// Some callers cannot allocate device memory at call time: a plugin hosted by
// a serving engine that has reserved the whole device-memory budget up front
// and hands the plugin no allocator, or a latency-critical loop that must not
// call cudaMalloc because it can synchronise the device and take unbounded
// time.  For them the split-KV scratch (token prefix sums and per-worker
// partial outputs) lives in the fixed array below, which every device that
// loads this library keeps until the process exits.
// ---------------------------------------------------------------------------
namespace mla {
namespace {
constexpr int kNoAllocMaxTokens = 8192;
constexpr int kNoAllocMaxWorkers = 32;
constexpr WsLayout kNoAllocLayout = ws_layout(kNoAllocMaxTokens, kNoAllocMaxWorkers);
constexpr size_t kNoAllocScratchBytes = kNoAllocLayout.total;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace

cudaError_t decode_noalloc_scratch_address(void** ptr) {
  // the array's host-side name stands in for it; its device address on the
  // current device comes from the runtime
  *ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(ptr, g_noalloc_scratch);
  return e == cudaSuccess && *ptr == nullptr ? cudaErrorInvalidSymbol : e;
}

size_t decode_noalloc_scratch_bytes() { return kNoAllocScratchBytes; }
int decode_noalloc_max_tokens() { return kNoAllocMaxTokens; }
int decode_noalloc_max_workers() { return kNoAllocMaxWorkers; }

// 0 = ok, 1 = sizes beyond the fixed scratch, 2 = CUDA error.
int launch_decode_tc_noalloc(const mla_handle* h, const void* q_lat, const void* pool, int n_pool_blocks,
                             const int* block_table, int max_blocks, const int* seq_lens, const int* cu_q,
                             int batch, int n_tok, int num_workers, void* o_lat, float* lse, cudaStream_t s) {
  const int W = num_workers > 0 ? num_workers : min(max(1, h->num_sms / 2), kNoAllocMaxWorkers);
  if (n_tok > kNoAllocMaxTokens || W > kNoAllocMaxWorkers) return 1;
  // the handle looked up the array's device address when it was created
  if (!h->noalloc_scratch) return 2;
  Maps maps;
  const long long rows = static_cast<long long>(n_pool_blocks) * kBlockRows;
  if (!encode_pool_maps(h, &maps, pool, rows)) return 2;
  Params prm{};
  set_workspace(prm, static_cast<uint8_t*>(h->noalloc_scratch), kNoAllocLayout);
  prm.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.cu_q = cu_q;
  prm.o_lat = static_cast<__nv_bfloat16*>(o_lat);
  prm.lse = lse;
  prm.status = h->status;
  prm.wait_limit = h->wait_limit;
  prm.max_blocks = max_blocks;
  prm.batch = batch;
  prm.n_tok = n_tok;
  prm.n_pool_blocks = n_pool_blocks;
  prm.workers = W;
  prm.scale_log2 = h->dims.scale * kLog2e;
  return launch_decode_kernels<false>(h, maps, prm, W, n_tok, seq_lens, cu_q, batch, max_blocks, lse, h->status, s) ==
                 cudaSuccess
             ? 0
             : 2;
}
}  // namespace mla
