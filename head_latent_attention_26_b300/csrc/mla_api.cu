// mla_api.cu -- the C ABI declared in include/mla.h: handle life cycle,
// host-side argument checks, dispatch to the kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "internal.cuh"
#include "mla.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
size_t elem_bytes(const mla_handle* h) { return h->dims.dtype == MLA_BF16 ? 2 : 4; }

#define MLA_TRY_CUDA(expr)                            \
  do {                                                \
    cudaError_t e_ = (expr);                          \
    if (e_ != cudaSuccess) return MLA_ERR_CUDA;       \
  } while (0)

bool dims_ok(const mla_dims* d) {
  return d && d->n_h > 0 && d->d_h > 0 && d->d_hr >= 2 && d->d_hr % 2 == 0 && d->d_c > 0 &&
         d->d_cq > 0 && d->d_model > 0 && d->block > 0 && d->rope_base > 0.f &&
         std::isfinite(d->scale) && d->scale > 0.f && (d->dtype == MLA_BF16 || d->dtype == MLA_F32);
}

// Shapes the generic path handles: the latent sum keeps d_c/32 values per lane.
bool simt_ok(const mla_dims* d) { return d->d_c <= 512; }

bool tensor_path_dims(const mla_dims* d) {
  return d->n_h == 128 && d->d_c == 512 && d->d_hr == 64 && d->block == 64 && d->dtype == MLA_BF16;
}

// The projection kernels tile weights in 128-row slabs that must not straddle
// heads, and stream k in 64-column (128-byte) steps.
bool proj_tc_dims(const mla_dims* d) {
  return d->dtype == MLA_BF16 && d->d_h == 128 && d->d_c % 128 == 0 && d->d_hr % 2 == 0 &&
         d->d_model % 64 == 0 && d->d_cq % 64 == 0 && (d->d_c + d->d_hr) % 8 == 0;
}

}  // namespace

namespace mla {

bool tensor_map_2d(const mla_handle* h, CUtensorMap* out, const void* base, long long cols, long long rows,
                   int box_cols, int box_rows, CUtensorMapSwizzle sw, CUtensorMapDataType dt, long long ld) {
  const int eb = dt == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1 : 2;
  if (ld <= 0) ld = cols;
  const MapKey key{base, cols, rows, ld, box_cols, box_rows, static_cast<int>(sw), static_cast<int>(dt)};
  std::lock_guard<std::mutex> lock(h->mu);
  auto it = h->maps.find(key);
  if (it != h->maps.end()) {
    *out = it->second;
    return true;
  }
  auto enc = tma_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * eb};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUtensorMap m;
  if (enc(&m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  // a serving loop reuses a handful of buffers; a caller that keeps handing
  // new ones only ever pays for one encode per call
  if (h->maps.size() >= 1024) h->maps.clear();
  h->maps.emplace(key, m);
  *out = m;
  return true;
}

cudaError_t kernel_attrs_once(const mla_handle* h, const void* fn, int smem_bytes, bool nonportable_cluster) {
  std::lock_guard<std::mutex> lock(h->mu);
  if (h->attrs_set.count(fn)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess && nonportable_cluster)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) h->attrs_set.insert(fn);
  return e;
}

}  // namespace mla

extern "C" {

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MLA_ERR_DEVICE_BOUNDS: return "device-side index check failed";
  }
  return "unknown status";
}

mla_status mla_create(const mla_dims* dims, int max_pos, mla_handle** out) {
  if (!out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims_ok(dims) || max_pos < 1) return MLA_ERR_INVALID_ARG;
  if (!simt_ok(dims)) return MLA_ERR_UNSUPPORTED;
  mla_handle* h = new mla_handle();
  h->dims = *dims;
  h->max_pos = max_pos;
  h->wait_limit = mla::kDefaultWaitLimit;
  h->tensor_path = tensor_path_dims(dims);
  h->proj_tc = proj_tc_dims(dims);
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return MLA_ERR_CUDA;
  }
  // RoPE angles pos * base^(-2k/d_hr) in double, cos/sin rounded to float.
  const int half = dims->d_hr / 2;
  const size_t n = static_cast<size_t>(max_pos) * half;
  std::vector<float> c(n), s(n);
  for (int p = 0; p < max_pos; ++p)
    for (int k = 0; k < half; ++k) {
      const double theta = std::pow(static_cast<double>(dims->rope_base), -2.0 * k / dims->d_hr);
      const double ang = static_cast<double>(p) * theta;
      c[static_cast<size_t>(p) * half + k] = static_cast<float>(std::cos(ang));
      s[static_cast<size_t>(p) * half + k] = static_cast<float>(std::sin(ang));
    }
  bool ok = cudaMalloc(&h->rope_cos, n * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&h->rope_sin, n * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&h->status, 8 * sizeof(int)) == cudaSuccess &&
            cudaMemcpy(h->rope_cos, c.data(), n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(h->rope_sin, s.data(), n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemset(h->status, 0, 8 * sizeof(int)) == cudaSuccess;
  // The fixed scratch of mla_decode_noalloc: its device address on this
  // device, looked up now with the device current.  The lookup also loads the
  // library's device code here, so the array is reserved at creation rather
  // than at the first decode call.
  if (ok && h->tensor_path) ok = mla::decode_noalloc_scratch_address(&h->noalloc_scratch) == cudaSuccess;
  if (ok) h->out_counters = reinterpret_cast<unsigned int*>(h->status + 4);  // words 4 and 5, zero
  if (!ok) {
    mla_destroy(h);
    return MLA_ERR_CUDA;
  }
  *out = h;
  return MLA_OK;
}

void mla_destroy(mla_handle* h) {
  if (!h) return;
  if (h->rope_cos) cudaFree(h->rope_cos);
  if (h->rope_sin) cudaFree(h->rope_sin);
  if (h->status) cudaFree(h->status);
  delete h;
}

int mla_num_sms(const mla_handle* h) { return h ? h->num_sms : 0; }
int mla_uses_tensor_path(const mla_handle* h) { return h && h->tensor_path ? 1 : 0; }

mla_status mla_set_wait_limit(mla_handle* h, long long polls) {
  if (!h || polls < 0) return MLA_ERR_INVALID_ARG;
  h->wait_limit = polls == 0 ? mla::kDefaultWaitLimit : polls;
  return MLA_OK;
}

mla_status mla_set_decode_l2_prefetch(mla_handle* h, const void* const* ptrs, const size_t* bytes, int n) {
  if (!h || n < 0 || n > 2 || (n > 0 && (!ptrs || !bytes))) return MLA_ERR_INVALID_ARG;
  for (int r = 0; r < n; ++r)
    if (bytes[r] && (!ptrs[r] || reinterpret_cast<uintptr_t>(ptrs[r]) % 16 || bytes[r] % 16 ||
                     bytes[r] > (static_cast<size_t>(1) << 40)))
      return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(h->mu);
  for (int r = 0; r < 2; ++r) {
    const bool used = r < n && bytes[r];
    h->l2_prefetch_ptr[r] = used ? ptrs[r] : nullptr;
    h->l2_prefetch_bytes[r] = used ? static_cast<long long>(bytes[r]) : 0;
  }
  return MLA_OK;
}

// ---------------------------------------------------------------- a0
size_t mla_q_proj_workspace_bytes(const mla_handle* h, int n_tok) {
  if (!h || n_tok < 0) return 0;
  return (static_cast<size_t>(n_tok) * h->dims.d_cq * elem_bytes(h) + 255) & ~static_cast<size_t>(255);
}

mla_status mla_q_proj(mla_handle* h, const void* x, const void* w_dq, const void* w_uq, const void* w_qr,
                      int n_tok, void* q_c, void* q_r, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!h || n_tok < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  for (const void* p : {x, w_dq, w_uq, w_qr, static_cast<const void*>(q_c), static_cast<const void*>(q_r)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < mla_q_proj_workspace_bytes(h, n_tok)) return MLA_ERR_WORKSPACE;
  const mla_dims& d = h->dims;
  if (h->proj_tc) {
    MLA_TRY_CUDA(mla::launch_linear_tc(h, x, d.d_model, w_dq, d.d_model, d.d_cq, 1, 0, ws, d.d_cq, n_tok, stream));
    MLA_TRY_CUDA(mla::launch_linear2_tc(h, ws, d.d_cq, w_uq, d.n_h * d.d_h, q_c, d.n_h * d.d_h, w_qr,
                                        d.n_h * d.d_hr, q_r, d.n_h * d.d_hr, n_tok, stream));
    return MLA_OK;
  }
  MLA_TRY_CUDA(mla::launch_linear(h, x, d.d_model, w_dq, d.d_model, d.d_cq, ws, d.d_cq, n_tok, stream));
  MLA_TRY_CUDA(mla::launch_linear(h, ws, d.d_cq, w_uq, d.d_cq, d.n_h * d.d_h, q_c, d.n_h * d.d_h, n_tok,
                                  stream));
  MLA_TRY_CUDA(mla::launch_linear(h, ws, d.d_cq, w_qr, d.d_cq, d.n_h * d.d_hr, q_r, d.n_h * d.d_hr,
                                  n_tok, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- a1
mla_status mla_cache_append(mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx,
                            const int* pos, int n_new, const int* block_table, int max_blocks, int batch,
                            void* pool, int n_pool_blocks, cudaStream_t stream) {
  if (!h || n_new < 0) return MLA_ERR_INVALID_ARG;
  if (n_new == 0) return MLA_OK;
  if (!x || !w_dkr || !pool || !aligned16(x) || !aligned16(w_dkr) || !aligned16(pool))
    return MLA_ERR_INVALID_ARG;
  if (!seq_idx || !pos || !block_table || !aligned4(seq_idx) || !aligned4(pos) || !aligned4(block_table))
    return MLA_ERR_INVALID_ARG;
  if (max_blocks < 1 || batch < 1 || n_pool_blocks < 1) return MLA_ERR_INVALID_ARG;
  if (h->proj_tc) {
    MLA_TRY_CUDA(mla::launch_cache_append_tc(h, x, w_dkr, seq_idx, pos, n_new, block_table, max_blocks, batch,
                                             pool, n_pool_blocks, stream));
    return MLA_OK;
  }
  MLA_TRY_CUDA(mla::launch_cache_append_simt(h, x, w_dkr, seq_idx, pos, n_new, block_table, max_blocks,
                                             batch, pool, n_pool_blocks, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- a0 + a1 in one call
mla_status mla_q_proj_append(mla_handle* h, const void* x, const void* w_dq, const void* w_uq, const void* w_qr,
                             const void* w_dkr, const int* seq_idx, const int* pos, int n_tok,
                             const int* block_table, int max_blocks, int batch, void* pool, int n_pool_blocks,
                             void* q_c, void* q_r, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!h || n_tok < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  for (const void* p : {x, w_dq, w_uq, w_qr, w_dkr, static_cast<const void*>(pool), static_cast<const void*>(q_c),
                        static_cast<const void*>(q_r)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  if (!seq_idx || !pos || !block_table || !aligned4(seq_idx) || !aligned4(pos) || !aligned4(block_table))
    return MLA_ERR_INVALID_ARG;
  if (max_blocks < 1 || batch < 1 || n_pool_blocks < 1) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < mla_q_proj_workspace_bytes(h, n_tok)) return MLA_ERR_WORKSPACE;
  if (!h->proj_tc) {
    // the generic kernels: the two calls one after the other
    const mla_status st = mla_q_proj(h, x, w_dq, w_uq, w_qr, n_tok, q_c, q_r, ws, ws_bytes, stream);
    if (st != MLA_OK) return st;
    return mla_cache_append(h, x, w_dkr, seq_idx, pos, n_tok, block_table, max_blocks, batch, pool, n_pool_blocks,
                            stream);
  }
  const mla_dims& d = h->dims;
  MLA_TRY_CUDA(mla::launch_q_down_append_tc(h, x, w_dq, ws, w_dkr, seq_idx, pos, n_tok, block_table, max_blocks,
                                            batch, pool, n_pool_blocks, stream));
  MLA_TRY_CUDA(mla::launch_linear2_tc(h, ws, d.d_cq, w_uq, d.n_h * d.d_h, q_c, d.n_h * d.d_h, w_qr,
                                      d.n_h * d.d_hr, q_r, d.n_h * d.d_hr, n_tok, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- a0 + a1 + a2 in one call
size_t mla_q_latent_append_workspace_bytes(const mla_handle* h, int n_tok) {
  if (!h || n_tok < 0) return 0;
  const mla_dims& d = h->dims;
  auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  const size_t n = static_cast<size_t>(n_tok), e = elem_bytes(h);
  return al(n * d.d_cq * e) + al(n * d.n_h * d.d_h * e) + al(n * d.n_h * d.d_hr * e);
}

mla_status mla_q_latent_append(mla_handle* h, const void* x, const void* w_dq, const void* w_uq, const void* w_qr,
                               const void* w_uk, const void* w_dkr, const int* seq_idx, const int* pos, int n_tok,
                               const int* block_table, int max_blocks, int batch, void* pool, int n_pool_blocks,
                               void* q_lat, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!h || n_tok < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  for (const void* p : {x, w_dq, w_uq, w_qr, w_uk, w_dkr, static_cast<const void*>(pool), static_cast<const void*>(q_lat)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  if (!seq_idx || !pos || !block_table || !aligned4(seq_idx) || !aligned4(pos) || !aligned4(block_table))
    return MLA_ERR_INVALID_ARG;
  if (max_blocks < 1 || batch < 1 || n_pool_blocks < 1) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < mla_q_latent_append_workspace_bytes(h, n_tok)) return MLA_ERR_WORKSPACE;
  const mla_dims& d = h->dims;
  auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  const size_t n = static_cast<size_t>(n_tok), e = elem_bytes(h);
  uint8_t* c_q = static_cast<uint8_t*>(ws);
  uint8_t* q_c = c_q + al(n * d.d_cq * e);
  uint8_t* q_r = q_c + al(n * d.n_h * d.d_h * e);
  if (h->proj_tc && h->tensor_path && n_tok <= mla::q_absorb_max_tokens()) {
    // W^DQ with the cache rows, then W^UQ -> W^UK^T per head with W^QR + RoPE
    MLA_TRY_CUDA(mla::launch_q_down_append_tc(h, x, w_dq, c_q, w_dkr, seq_idx, pos, n_tok, block_table, max_blocks,
                                              batch, pool, n_pool_blocks, stream));
    MLA_TRY_CUDA(mla::launch_q_absorb_tc(h, c_q, w_uq, w_qr, w_uk, pos, n_tok, q_lat, stream));
    return MLA_OK;
  }
  // otherwise the three calls' kernels one after the other, q^C and q^R in ws
  mla_status st = mla_q_proj_append(h, x, w_dq, w_uq, w_qr, w_dkr, seq_idx, pos, n_tok, block_table, max_blocks,
                                    batch, pool, n_pool_blocks, q_c, q_r, c_q, al(n * d.d_cq * e), stream);
  if (st != MLA_OK) return st;
  return mla_absorb_q(h, q_c, q_r, pos, n_tok, w_uk, q_lat, stream);
}

// ---------------------------------------------------------------- a1, quantised cache
size_t mla_cache_append_q8_workspace_bytes(const mla_handle* h, int n_new) {
  if (!h || n_new < 0) return 0;
  const size_t n = static_cast<size_t>(n_new) * (h->dims.d_c + h->dims.d_hr) * 2;
  return (n + 255) & ~static_cast<size_t>(255);
}

mla_status mla_cache_append_q8(mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx, const int* pos,
                               int n_new, const int* block_table, int max_blocks, int batch, void* pool_q8,
                               int n_pool_blocks, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!h || n_new < 0) return MLA_ERR_INVALID_ARG;
  if (!h->tensor_path || !h->proj_tc) return MLA_ERR_UNSUPPORTED;
  if (n_new == 0) return MLA_OK;
  if (!x || !w_dkr || !pool_q8 || !aligned16(x) || !aligned16(w_dkr) || !aligned16(pool_q8))
    return MLA_ERR_INVALID_ARG;
  if (!seq_idx || !pos || !block_table || !aligned4(seq_idx) || !aligned4(pos) || !aligned4(block_table))
    return MLA_ERR_INVALID_ARG;
  if (max_blocks < 1 || batch < 1 || n_pool_blocks < 1) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < mla_cache_append_q8_workspace_bytes(h, n_new)) return MLA_ERR_WORKSPACE;
  MLA_TRY_CUDA(mla::launch_cache_rows_dense_tc(h, x, w_dkr, seq_idx, pos, n_new, block_table, max_blocks, batch,
                                               n_pool_blocks, ws, stream));
  MLA_TRY_CUDA(mla::launch_quantize_scatter_q8(h, ws, seq_idx, pos, n_new, block_table, max_blocks, batch, pool_q8,
                                               n_pool_blocks, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- prefill
size_t mla_prefill_workspace_bytes(const mla_handle* h, int P) {
  if (!h || P < 0) return 0;
  const size_t one = static_cast<size_t>(P) * h->dims.n_h * h->dims.d_h * 2;  // K^C or V, bf16
  return 2 * ((one + 255) & ~static_cast<size_t>(255));
}

mla_status mla_prefill(mla_handle* h, const void* rows, const void* q_c, const void* q_r, int P, const void* w_uk,
                       const void* w_uv, void* ws, size_t ws_bytes, void* o, float* lse, cudaStream_t stream) {
  if (!h || P < 0) return MLA_ERR_INVALID_ARG;
  if (!h->tensor_path || !h->proj_tc) return MLA_ERR_UNSUPPORTED;
  if (P == 0) return MLA_OK;
  if (P > h->max_pos) return MLA_ERR_INVALID_ARG;
  for (const void* p : {rows, q_c, q_r, w_uk, w_uv, static_cast<const void*>(o)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  if (!lse || !aligned4(lse)) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < mla_prefill_workspace_bytes(h, P)) return MLA_ERR_WORKSPACE;
  const mla_dims& d = h->dims;
  const int cols = d.n_h * d.d_h;
  uint8_t* k_c = static_cast<uint8_t*>(ws);
  uint8_t* v = k_c + mla_prefill_workspace_bytes(h, P) / 2;
  // K^C = C W^UK^T and V = C W^UV^T for every head at once, in fp16 (the
  // attention multiplies fp16 operands); C = the first d_c columns of each
  // cache row
  MLA_TRY_CUDA(mla::launch_linear2_tc(h, rows, d.d_c, w_uk, cols, k_c, cols, w_uv, cols, v, cols, P, stream,
                                      d.d_c + d.d_hr, 3));
  MLA_TRY_CUDA(mla::launch_prefill_attn_tc(h, rows, q_c, q_r, P, k_c, v, o, lse, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- a2
mla_status mla_absorb_q(mla_handle* h, const void* q_c, const void* q_r, const int* pos, int n_tok,
                        const void* w_uk, void* q_lat, cudaStream_t stream) {
  if (!h || n_tok < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  for (const void* p : {q_c, q_r, w_uk, static_cast<const void*>(q_lat)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  if (!pos || !aligned4(pos)) return MLA_ERR_INVALID_ARG;
  if (h->proj_tc) {
    MLA_TRY_CUDA(mla::launch_absorb_q_tc(h, q_c, q_r, pos, n_tok, w_uk, q_lat, stream));
    return MLA_OK;
  }
  MLA_TRY_CUDA(mla::launch_absorb_q_simt(h, q_c, q_r, pos, n_tok, w_uk, q_lat, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- folded query weight
mla_status mla_absorb_weights(mla_handle* h, const void* w_uq, const void* w_uk, void* w_uq_abs,
                              cudaStream_t stream) {
  if (!h) return MLA_ERR_INVALID_ARG;
  for (const void* p : {w_uq, w_uk, static_cast<const void*>(w_uq_abs)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  MLA_TRY_CUDA(mla::launch_absorb_weights(h, w_uq, w_uk, w_uq_abs, stream));
  return MLA_OK;
}

mla_status mla_q_proj_absorbed(mla_handle* h, const void* x, const void* w_dq, const void* w_uq_abs,
                               const void* w_qr, const int* pos, int n_tok, void* q_lat, void* ws,
                               size_t ws_bytes, cudaStream_t stream) {
  if (!h || n_tok < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  for (const void* p : {x, w_dq, w_uq_abs, w_qr, static_cast<const void*>(q_lat)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  if (!pos || !aligned4(pos)) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < mla_q_proj_workspace_bytes(h, n_tok)) return MLA_ERR_WORKSPACE;
  const mla_dims& d = h->dims;
  if (h->proj_tc) {
    MLA_TRY_CUDA(mla::launch_linear_tc(h, x, d.d_model, w_dq, d.d_model, d.d_cq, 1, 0, ws, d.d_cq, n_tok, stream));
    MLA_TRY_CUDA(mla::launch_q_absorbed_tc(h, ws, w_uq_abs, w_qr, pos, n_tok, q_lat, stream));
    return MLA_OK;
  }
  MLA_TRY_CUDA(mla::launch_linear(h, x, d.d_model, w_dq, d.d_model, d.d_cq, ws, d.d_cq, n_tok, stream));
  MLA_TRY_CUDA(mla::launch_q_absorbed_simt(h, ws, w_uq_abs, w_qr, pos, n_tok, q_lat, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- a3 + a4
size_t mla_decode_workspace_bytes(const mla_handle* h, int n_tok, int num_workers) {
  if (!h || n_tok < 0 || num_workers < 0) return 0;
  if (h->tensor_path) return mla::decode_tc_workspace_bytes(h, n_tok, num_workers);
  return 0;
}

mla_status mla_decode(mla_handle* h, const void* q_lat, const void* pool, int n_pool_blocks,
                      const int* block_table, int max_blocks, const int* seq_lens, const int* cu_q,
                      int batch, int n_tok, int num_workers, void* ws, size_t ws_bytes, void* o_lat,
                      float* lse, cudaStream_t stream) {
  if (!h || n_tok < 0 || batch < 0 || num_workers < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  if (batch < 1 || max_blocks < 1 || n_pool_blocks < 1) return MLA_ERR_INVALID_ARG;
  for (const void* p : {q_lat, pool, static_cast<const void*>(o_lat), static_cast<const void*>(lse)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  for (const int* p : {block_table, seq_lens, cu_q})
    if (!p || !aligned4(p)) return MLA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_bytes(h, n_tok, num_workers);
  if (need > 0 && (!ws || !aligned16(ws) || ws_bytes < need)) return MLA_ERR_WORKSPACE;
  if (h->tensor_path) {
    MLA_TRY_CUDA(mla::launch_decode_tc(h, q_lat, pool, n_pool_blocks, block_table, max_blocks, seq_lens,
                                       cu_q, batch, n_tok, num_workers, ws, ws_bytes, o_lat, lse, stream));
  } else {
    MLA_TRY_CUDA(mla::launch_decode_simt(h, q_lat, pool, n_pool_blocks, block_table, max_blocks, seq_lens,
                                         cu_q, batch, n_tok, o_lat, lse, stream));
  }
  return MLA_OK;
}

mla_status mla_decode_q8(mla_handle* h, const void* q_lat, const void* pool_q8, int n_pool_blocks,
                         const int* block_table, int max_blocks, const int* seq_lens, const int* cu_q, int batch,
                         int n_tok, int num_workers, void* ws, size_t ws_bytes, void* o_lat, float* lse,
                         cudaStream_t stream) {
  if (!h || n_tok < 0 || batch < 0 || num_workers < 0) return MLA_ERR_INVALID_ARG;
  if (!h->tensor_path) return MLA_ERR_UNSUPPORTED;
  if (n_tok == 0) return MLA_OK;
  if (batch < 1 || max_blocks < 1 || n_pool_blocks < 1) return MLA_ERR_INVALID_ARG;
  for (const void* p : {q_lat, pool_q8, static_cast<const void*>(o_lat), static_cast<const void*>(lse)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  for (const int* p : {block_table, seq_lens, cu_q})
    if (!p || !aligned4(p)) return MLA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_bytes(h, n_tok, num_workers);
  if (!ws || !aligned16(ws) || ws_bytes < need) return MLA_ERR_WORKSPACE;
  MLA_TRY_CUDA(mla::launch_decode_tc(h, q_lat, pool_q8, n_pool_blocks, block_table, max_blocks, seq_lens, cu_q,
                                     batch, n_tok, num_workers, ws, ws_bytes, o_lat, lse, stream, true));
  return MLA_OK;
}

// ---------------------------------------------------------------- a3 + a4, fixed scratch
mla_status mla_decode_noalloc(mla_handle* h, const void* q_lat, const void* pool, int n_pool_blocks,
                              const int* block_table, int max_blocks, const int* seq_lens, const int* cu_q,
                              int batch, int n_tok, int num_workers, void* o_lat, float* lse,
                              cudaStream_t stream) {
  if (!h || n_tok < 0 || batch < 0 || num_workers < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  if (batch < 1 || max_blocks < 1 || n_pool_blocks < 1) return MLA_ERR_INVALID_ARG;
  for (const void* p : {q_lat, pool, static_cast<const void*>(o_lat), static_cast<const void*>(lse)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  for (const int* p : {block_table, seq_lens, cu_q})
    if (!p || !aligned4(p)) return MLA_ERR_INVALID_ARG;
  if (!h->tensor_path) {  // the generic kernels need no scratch at all
    MLA_TRY_CUDA(mla::launch_decode_simt(h, q_lat, pool, n_pool_blocks, block_table, max_blocks, seq_lens,
                                         cu_q, batch, n_tok, o_lat, lse, stream));
    return MLA_OK;
  }
  const int r = mla::launch_decode_tc_noalloc(h, q_lat, pool, n_pool_blocks, block_table, max_blocks, seq_lens,
                                              cu_q, batch, n_tok, num_workers, o_lat, lse, stream);
  if (r == 1) return MLA_ERR_WORKSPACE;
  return r == 0 ? MLA_OK : MLA_ERR_CUDA;
}

// ---------------------------------------------------------------- a5
size_t mla_out_workspace_bytes(const mla_handle* h, int n_tok) {
  if (!h || n_tok < 0) return 0;
  const size_t n = static_cast<size_t>(n_tok) * h->dims.n_h * h->dims.d_h * elem_bytes(h);
  return (n + 255) & ~static_cast<size_t>(255);
}

mla_status mla_out(mla_handle* h, const void* o_lat, const void* w_uv, const void* w_o, int n_tok, void* u,
                   void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!h || n_tok < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0) return MLA_OK;
  for (const void* p : {o_lat, w_uv, w_o, static_cast<const void*>(u)})
    if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < mla_out_workspace_bytes(h, n_tok)) return MLA_ERR_WORKSPACE;
  const mla_dims& d = h->dims;
  const int H = d.n_h * d.d_h;
  if (h->proj_tc && h->tensor_path && n_tok <= mla::out_fused_max_tokens()) {
    const cudaError_t e = mla::launch_out_tc(h, o_lat, w_uv, w_o, n_tok, ws, u, stream);
    if (e != cudaErrorNotSupported) {
      MLA_TRY_CUDA(e);
      return MLA_OK;
    }
  }
  if (h->proj_tc) {
    MLA_TRY_CUDA(mla::launch_linear_tc(h, o_lat, d.n_h * d.d_c, w_uv, d.d_c, H, d.n_h, d.d_c, ws, H, n_tok, stream));
    MLA_TRY_CUDA(mla::launch_linear_tc(h, ws, H, w_o, H, d.d_model, 1, 0, u, d.d_model, n_tok, stream));
    return MLA_OK;
  }
  MLA_TRY_CUDA(mla::launch_up_project_simt(h, o_lat, w_uv, n_tok, ws, stream));
  MLA_TRY_CUDA(mla::launch_linear(h, ws, H, w_o, H, d.d_model, u, d.d_model, n_tok, stream));
  return MLA_OK;
}

// ---------------------------------------------------------------- status
mla_status mla_check_device_status(mla_handle* h, cudaStream_t stream) {
  if (!h) return MLA_ERR_INVALID_ARG;
  MLA_TRY_CUDA(cudaStreamSynchronize(stream));
  int v[4] = {0, 0, 0, 0};
  MLA_TRY_CUDA(cudaMemcpy(v, h->status, sizeof(v), cudaMemcpyDeviceToHost));
  MLA_TRY_CUDA(cudaMemset(h->status, 0, sizeof(v)));
  h->last_site[0] = v[1];
  h->last_site[1] = v[2];
  h->last_site[2] = v[3];
  return static_cast<mla_status>(v[0]);
}

mla_status mla_device_error_site(const mla_handle* h, int* site, int* cta, int* tile) {
  if (!h || !site || !cta || !tile) return MLA_ERR_INVALID_ARG;
  *site = h->last_site[0];
  *cta = h->last_site[1];
  *tile = h->last_site[2];
  return MLA_OK;
}

mla_status mla_selftest_wait_timeout(mla_handle* h, cudaStream_t stream) {
  if (!h) return MLA_ERR_INVALID_ARG;
  MLA_TRY_CUDA(mla::launch_wait_timeout_selftest(h, stream));
  return MLA_OK;
}

}  // extern "C"
