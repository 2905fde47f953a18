// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA, tcgen05/TMEM,
// cluster shared memory.  Every wait here is bounded by the caller.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mla {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, "
      "p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking completion test of a phase: when the phase has already
// completed (the common case on the softmax warps' waits) this returns sooner
// than try_wait, which the waits then fall back to.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, "
      "p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Same as mbar_try_wait, with acquire at cluster scope (data written by the peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared-memory counters with release / acquire semantics: a cheaper hand-off
// than an mbarrier round trip between warps of one CTA (the consumer polls).
__device__ __forceinline__ void st_release_u32(uint32_t* addr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(addr)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* addr) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(addr)) : "memory");
  return v;
}

// ------------------------------------------------------------------ programmatic dependent launch
// Kernels of the library are launched so that the next kernel in the stream
// may start while this one finishes.  Every kernel waits (pdl_wait) before it
// reads anything an earlier kernel wrote or writes anything an earlier kernel
// reads, and lets its successor launch (pdl_trigger) once its own CTAs no
// longer need to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Map a local shared::cta address to the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Bulk copy of `bytes` from this CTA's shared memory to a peer CTA's shared
// memory; completes `bytes` of transaction count on the peer's barrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster_addr, const void* src, uint32_t bytes,
                                                  uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster_addr),
      "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster_addr)
      : "memory");
}
// Remote arrive without release semantics (pure flow control).
__device__ __forceinline__ void mbar_arrive_relaxed_cluster(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N bulk groups of this thread still read their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
// 2-D tiled TMA load of the box at (x, y) into shared memory, completing its
// bytes on `bar`, with an L2 eviction-priority policy (see l2_policy_*).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                                 int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// L2 eviction priorities.  Evict-first: the latent cache, read once and
// never worth a line that anything else holds.  Normal: streamed weights, so
// that one step's weight reads replace each other's lines in least-recently-
// used order (a weight range prefetched during the attention, also at normal
// priority, outlives the evict-first cache stream until its kernel reads it,
// and is gone again once the next step's weights have streamed).  Evict-last:
// activations that several CTAs read.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Asks the L2 cache to fetch `bytes` (a multiple of 16) of global memory at
// `src` (16-byte aligned); nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
// Shared-memory matrix descriptor: start, leading/stride byte offsets,
// version 1, swizzle layout (0 none, 2 = 128B, 4 = 64B, 6 = 32B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}
constexpr uint32_t kSwizzle128B = 2, kSwizzle64B = 4, kSwizzleNone = 0;

// Instruction descriptor for kind::f16 with bf16 A/B and f32 accumulation.
// a_mn / b_mn select the MN-major (transposed) operand layout.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// The same with fp16 A and B.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Warp-converged forms: every lane of the warp executes them (so operands stay
// warp-uniform and need no per-instruction register moves) and one elected
// lane issues the instruction.
__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
// One score tile, issued by one elected lane of a converged warp:
// S (+)= Q~[:, own 256 latent] . C^T (16 K-steps, A in TMEM, B a 128B-swizzled
// K-major stage of four 64-column boxes BOX bytes apart) + Q~[:, own 32 RoPE]
// . C_rope^T (2 K-steps, 64B swizzle).  Descriptors advance by constants
// inside the block, so the warp-uniform bases reach the uniform datapath once
// per tile.
template <int BOX>
__device__ __forceinline__ void mma_score_tile_elect(uint32_t d_tmem, uint32_t a_lat, uint32_t a_rope,
                                                     uint64_t b_lat, uint64_t b_rope, uint32_t idesc) {
  constexpr int kB = BOX / 16;  // box stride in descriptor units
  asm volatile(
      "{\n\t.reg .pred e, f, t;\n\t.reg .b64 bd;\n\t.reg .b32 ad;\n\t"
      "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 f, 0, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %5, f;\n\t"
      "add.u32 ad, %1, 8;\n\tadd.s64 bd, %3, 2;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 16;\n\tadd.s64 bd, %3, 4;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 24;\n\tadd.s64 bd, %3, 6;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 32;\n\tadd.s64 bd, %3, %6;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 40;\n\tadd.s64 bd, %3, %7;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 48;\n\tadd.s64 bd, %3, %8;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 56;\n\tadd.s64 bd, %3, %9;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 64;\n\tadd.s64 bd, %3, %10;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 72;\n\tadd.s64 bd, %3, %11;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 80;\n\tadd.s64 bd, %3, %12;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 88;\n\tadd.s64 bd, %3, %13;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 96;\n\tadd.s64 bd, %3, %14;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 104;\n\tadd.s64 bd, %3, %15;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 112;\n\tadd.s64 bd, %3, %16;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "add.u32 ad, %1, 120;\n\tadd.s64 bd, %3, %17;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %4, %5, t;\n\t"
      "add.u32 ad, %2, 8;\n\tadd.s64 bd, %4, 2;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %5, t;\n\t"
      "}" ::"r"(d_tmem),
      "r"(a_lat), "r"(a_rope), "l"(b_lat), "l"(b_rope), "r"(idesc), "n"(kB), "n"(kB + 2), "n"(kB + 4), "n"(kB + 6),
      "n"(2 * kB), "n"(2 * kB + 2), "n"(2 * kB + 4), "n"(2 * kB + 6), "n"(3 * kB), "n"(3 * kB + 2), "n"(3 * kB + 4),
      "n"(3 * kB + 6)
      : "memory");
}
// O (+)= P . C[:, own 256 latent] over KSTEPS x 16 keys, A = P in TMEM, B =
// the same stage read MN-major.  `accumulate` = 0 starts O afresh.
template <int KSTEPS>
__device__ __forceinline__ void mma_value_tile_elect(uint32_t d_tmem, uint32_t a_p, uint64_t b_desc, uint32_t idesc,
                                                     uint32_t accumulate) {
  static_assert(KSTEPS == 2 || KSTEPS == 4, "value tile of 32 or 64 keys");
  if (KSTEPS == 2) {
    asm volatile(
        "{\n\t.reg .pred e, f, t;\n\t.reg .b64 bd;\n\t.reg .b32 ad;\n\t"
        "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 f, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, f;\n\t"
        "add.u32 ad, %1, 8;\n\tadd.s64 bd, %2, 128;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %3, t;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_p), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, f, t;\n\t.reg .b64 bd;\n\t.reg .b32 ad;\n\t"
        "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 f, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, f;\n\t"
        "add.u32 ad, %1, 8;\n\tadd.s64 bd, %2, 128;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %3, t;\n\t"
        "add.u32 ad, %1, 16;\n\tadd.s64 bd, %2, 256;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %3, t;\n\t"
        "add.u32 ad, %1, 24;\n\tadd.s64 bd, %2, 384;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ad], bd, %3, t;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_p), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
// Four K-steps of 16 (one 64-wide k block) with A and B in shared memory,
// issued by one elected lane of a converged warp; descriptors advance by
// A_STEP / B_STEP (16-byte units) per step.  `accumulate` = 0 starts D afresh.
template <int A_STEP, int B_STEP>
__device__ __forceinline__ void mma_ss_kblock_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, f, t;\n\t.reg .b64 ad, bd;\n\t"
      "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 f, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
      "add.s64 ad, %1, %5;\n\tadd.s64 bd, %2, %6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.s64 ad, %1, %7;\n\tadd.s64 bd, %2, %8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.s64 ad, %1, %9;\n\tadd.s64 bd, %2, %10;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(A_STEP), "n"(B_STEP), "n"(2 * A_STEP),
      "n"(2 * B_STEP), "n"(3 * A_STEP), "n"(3 * B_STEP)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
// One MMA with A in TMEM and B a shared-memory descriptor, issued by one
// elected lane of a converged warp; `accumulate` = 0 starts D afresh.
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, f;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 f, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, f;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x on the SFU, flushing subnormal results to zero (x <= 8 here).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-lane TMEM shapes (lane base = the address's lane field, 16-aligned).
// 16x256b: thread t holds TMEM lanes base + t/4 and base + t/4 + 8; for each
// 8-column group j, registers 4j, 4j+1 = columns 8j + 2(t%4), +1 of the first
// lane and 4j+2, 4j+3 the same columns of the second.
// 16x128b: register 2j = column 4j + t%4 of the first lane, 2j+1 of the second.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Packed fp32 pairs (one instruction for two lanes of arithmetic).
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)), "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&r);
}
// (a.x + lo(h), a.y + hi(h)) with h two fp16 values, added in fp32.
__device__ __forceinline__ float2 add_f32_f16x2(float2 a, uint32_t h) {
  float x, y;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %4;\n\t}"
      : "=f"(x), "=f"(y)
      : "r"(h), "f"(a.x), "f"(a.y));
  return make_float2(x, y);
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace mla
