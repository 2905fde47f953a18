// internal.cuh -- handle layout, device status word, scalar helpers shared by
// the kernels of the library (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <unordered_map>
#include <unordered_set>
#include <utility>

#include "mla.h"

namespace mla {
// What a 2-D tiled tensor map encodes: the same key always gives the same map,
// so a handle encodes each one once and reuses it on later calls.
struct MapKey {
  const void* base;
  long long cols, rows, ld;
  int box_cols, box_rows, swizzle, dtype;
  bool operator==(const MapKey& o) const {
    return base == o.base && cols == o.cols && rows == o.rows && ld == o.ld && box_cols == o.box_cols &&
           box_rows == o.box_rows && swizzle == o.swizzle && dtype == o.dtype;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = std::hash<const void*>()(k.base);
    for (long long v : {k.cols, k.rows, k.ld, static_cast<long long>(k.box_cols), static_cast<long long>(k.box_rows),
                        static_cast<long long>(k.swizzle), static_cast<long long>(k.dtype)})
      h = h * 1000003u ^ std::hash<long long>()(v);
    return h;
  }
};
}  // namespace mla

struct mla_handle {
  mla_dims dims;
  int max_pos;
  int device;
  int num_sms;
  float* rope_cos;  // [max_pos, d_hr/2], cos(pos * base^(-2k/d_hr)) rounded from double
  float* rope_sin;
  int* status;      // [4]: first device-side error code (0 = none), then where the first
                    // bounded wait gave up: site word, CTA, tile (see report_site)
  int last_site[3];  // the site words read back by the last mla_check_device_status
  // two device counters of the one-launch output projection (CTAs past its
  // first phase, CTAs finished), zero between calls: the words after the
  // status word in the same allocation
  unsigned int* out_counters;
  long long wait_limit;
  bool tensor_path;  // tcgen05 decode serves these dims
  bool proj_tc;      // tcgen05 projection kernels serve these dims
  // Device address of the decode's fixed scratch array on this handle's
  // device (looked up in mla_create with the device current), or null.
  void* noalloc_scratch;
  // Device ranges that mla_decode calls fetch into L2 while they stream the
  // cache (mla_set_decode_l2_prefetch); guarded by `mu`.
  const void* l2_prefetch_ptr[2];
  long long l2_prefetch_bytes[2];
  // Host-side launch state kept across calls so that a call does no repeated
  // driver work: encoded tensor maps and the kernels whose attributes are set.
  mutable std::mutex mu;
  mutable std::unordered_map<mla::MapKey, CUtensorMap, mla::MapKeyHash> maps;
  mutable std::unordered_set<const void*> attrs_set;
};

namespace mla {

constexpr long long kDefaultWaitLimit = 1ll << 24;  // mbarrier polls (about 0.1 us each) before giving up

// Records `code` in the status word unless an earlier error is already there.
__device__ __forceinline__ void report(int* status, int code) { atomicCAS(status, 0, code); }
// A bounded wait ran out: records MLA_ERR_DEVICE_TIMEOUT and, for the first
// such wait of the call, which one it was (a site number of the kernel, the
// warp), the CTA and the tile it waited for.
__device__ __forceinline__ void report_site(int* status, int site, int k) {
  report(status, MLA_ERR_DEVICE_TIMEOUT);
  const int word = 0x40000000 | (site << 8) | static_cast<int>(threadIdx.x >> 5);
  if (atomicCAS(status + 1, 0, word) == 0) {
    status[2] = static_cast<int>(blockIdx.x);
    status[3] = k;
  }
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sequence owning query row n: the largest b with cu_q[b] <= n.
__device__ __forceinline__ int seq_of_token(const int* cu_q, int batch, int n) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu_q[mid] <= n) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace mla

// Launches `kern` on `s` with programmatic stream serialisation (the kernel
// must call pdl_wait before touching data of earlier kernels) and, when
// cluster_x > 1, thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_x,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- launchers implemented in the kernel translation units ----------------
namespace mla {
cudaError_t launch_linear(const mla_handle* h, const void* X, int ldx, const void* W, int in, int out,
                          void* Y, int ldy, int n_tok, cudaStream_t s);
cudaError_t launch_cache_append_simt(const mla_handle* h, const void* x, const void* w_dkr,
                                     const int* seq_idx, const int* pos, int n_new,
                                     const int* block_table, int max_blocks, int batch, void* pool,
                                     int n_pool_blocks, cudaStream_t s);
cudaError_t launch_absorb_q_simt(const mla_handle* h, const void* q_c, const void* q_r, const int* pos,
                                 int n_tok, const void* w_uk, void* q_lat, cudaStream_t s);
// W~^UQ_i = W^UK_i^T W^UQ_i for every head (any dims, fp32 sums)
cudaError_t launch_absorb_weights(const mla_handle* h, const void* w_uq, const void* w_uk, void* w_abs,
                                  cudaStream_t s);
cudaError_t launch_q_absorbed_simt(const mla_handle* h, const void* c_q, const void* w_abs, const void* w_qr,
                                   const int* pos, int n_tok, void* q_lat, cudaStream_t s);
cudaError_t launch_decode_simt(const mla_handle* h, const void* q_lat, const void* pool,
                               int n_pool_blocks, const int* block_table, int max_blocks,
                               const int* seq_lens, const int* cu_q, int batch, int n_tok, void* o_lat,
                               float* lse, cudaStream_t s);
cudaError_t launch_up_project_simt(const mla_handle* h, const void* o_lat, const void* w_uv, int n_tok,
                                   void* o, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(const mla_handle* h, cudaStream_t s);

// tcgen05 decode (dims n_h=128, d_c=512, d_hr=64, block=64, bf16)
size_t decode_tc_workspace_bytes(const mla_handle* h, int n_tok, int num_workers);
cudaError_t launch_decode_tc(const mla_handle* h, const void* q_lat, const void* pool,
                             int n_pool_blocks, const int* block_table, int max_blocks,
                             const int* seq_lens, const int* cu_q, int batch, int n_tok,
                             int num_workers, void* ws, size_t ws_bytes, void* o_lat, float* lse,
                             cudaStream_t s, bool q8 = false);
// cuTensorMapEncodeTiled from the driver (looked up once); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tma_encoder();
// A 2-D tiled tensor map of a row-major [rows, cols] tensor with boxes of
// box_cols x box_rows, 16-bit (bf16) or 8-bit (u8) elements, rows `ld`
// elements apart (0: cols), encoded once per handle and key and copied out of
// the handle's cache afterwards.
bool tensor_map_2d(const mla_handle* h, CUtensorMap* out, const void* base, long long cols, long long rows,
                   int box_cols, int box_rows, CUtensorMapSwizzle sw,
                   CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, long long ld = 0);
// Sets a kernel's dynamic shared-memory size (and, when asked, the
// non-portable cluster-size opt-in) the first time this handle launches it.
cudaError_t kernel_attrs_once(const mla_handle* h, const void* fn, int smem_bytes, bool nonportable_cluster);
// Device address of the decode's fixed scratch array for the current device.
cudaError_t decode_noalloc_scratch_address(void** ptr);
// tcgen05 projections (bf16, d_h = 128, widths multiples of 64)
cudaError_t launch_linear_tc(const mla_handle* h, const void* X, int x_cols, const void* W, int in, int out,
                             int groups, int x_group_cols, void* Y, long long ldy, int n_tok, cudaStream_t s);
// Two products of the same tokens in one launch: Y1 = X W1^T, Y2 = X W2^T
// (token rows of X are x_ld elements apart, 0: in; bit 0 / bit 1 of f16_mask
// write Y1 / Y2 as fp16 instead of bf16).
cudaError_t launch_linear2_tc(const mla_handle* h, const void* X, int in, const void* W1, int out1, void* Y1,
                              long long ldy1, const void* W2, int out2, void* Y2, long long ldy2, int n_tok,
                              cudaStream_t s, long long x_ld = 0, int f16_mask = 0);
// The latent query of up to q_absorb_max_tokens() tokens straight from c^Q:
// W^UQ_i then W^UK_i^T per head in one CTA, W^QR with RoPE in the others.
int q_absorb_max_tokens();
cudaError_t launch_q_absorb_tc(const mla_handle* h, const void* c_q, const void* w_uq, const void* w_qr,
                               const void* w_uk, const int* pos, int n_tok, void* q_lat, cudaStream_t s);
// W^UV per head and W^O in one launch (up to out_fused_max_tokens() tokens);
// cudaErrorNotSupported when it does not apply (then two launches).
int out_fused_max_tokens();
cudaError_t launch_out_tc(const mla_handle* h, const void* o_lat, const void* w_uv, const void* w_o, int n_tok,
                          void* obuf, void* u, cudaStream_t s);
// Prefill attention over expanded keys and values (tcgen05): see mla_prefill.
cudaError_t launch_prefill_attn_tc(const mla_handle* h, const void* rows, const void* q_c, const void* q_r, int P,
                                   const void* k_c, const void* v, void* o, float* lse, cudaStream_t s);
// W^DQ and the cache-row product of the same tokens in one launch.
cudaError_t launch_q_down_append_tc(const mla_handle* h, const void* x, const void* w_dq, void* c_q,
                                   const void* w_dkr, const int* seq_idx, const int* pos, int n_new,
                                   const int* block_table, int max_blocks, int batch, void* pool, int n_pool_blocks,
                                   cudaStream_t s);
cudaError_t launch_cache_append_tc(const mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx,
                                   const int* pos, int n_new, const int* block_table, int max_blocks, int batch,
                                   void* pool, int n_pool_blocks, cudaStream_t s);
// Latent query from c^Q with the folded weight: [W~^UQ c^Q ; RoPE_pos(W^QR c^Q)]
// straight into q_lat, both products in one launch.
cudaError_t launch_q_absorbed_tc(const mla_handle* h, const void* c_q, const void* w_abs, const void* w_qr,
                                 const int* pos, int n_tok, void* q_lat, cudaStream_t s);
cudaError_t launch_absorb_q_tc(const mla_handle* h, const void* q_c, const void* q_r, const int* pos, int n_tok,
                               const void* w_uk, void* q_lat, cudaStream_t s);
cudaError_t launch_cache_rows_dense_tc(const mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx,
                                       const int* pos, int n_new, const int* block_table, int max_blocks, int batch,
                                       int n_pool_blocks, void* rows, cudaStream_t s);
// Quantised latent cache (rows of 672 bytes: int8 codes of c^KV, fp16 block
// scales, bf16 k^R): quantise dense bf16 rows into the pool slots.
cudaError_t launch_quantize_scatter_q8(const mla_handle* h, const void* rows, const int* seq_idx, const int* pos,
                                       int n_new, const int* block_table, int max_blocks, int batch, void* pool,
                                       int n_pool_blocks, cudaStream_t s);
// Same kernels with their scratch in a fixed device array (no allocation).
int launch_decode_tc_noalloc(const mla_handle* h, const void* q_lat, const void* pool, int n_pool_blocks,
                             const int* block_table, int max_blocks, const int* seq_lens, const int* cu_q,
                             int batch, int n_tok, int num_workers, void* o_lat, float* lse, cudaStream_t s);
size_t decode_noalloc_scratch_bytes();
int decode_noalloc_max_tokens();
int decode_noalloc_max_workers();
}  // namespace mla
