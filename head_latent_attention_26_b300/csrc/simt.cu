// simt.cu -- generic CUDA-core path for every step, any layer sizes, fp32
// arithmetic with bf16 or f32 storage.  It serves the layer sizes the tensor
// path does not (e.g. the tiny 4-head layer) and the projection steps.
//
// Equations: [0h-n0] = "論文解説: DeepSeek-V2 — … Multi-head Latent Attention",
// [qiita] = MLA notes on qiita.com, [kasblo] = MLA explainer on kasblo.com.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace mla {
namespace {

// Y[n, o] = sum_k X[n, k] W[o, k]: one warp per output feature, NT tokens per
// block so each weight row is read once per NT tokens.
template <typename T, int NT>
__global__ void __launch_bounds__(256) linear_kernel(const T* __restrict__ X, int ldx,
                                                     const T* __restrict__ W, int in, int out,
                                                     T* __restrict__ Y, int ldy, int n_tok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o = blockIdx.x * 8 + warp;
  const int n0 = blockIdx.y * NT;
  if (o >= out) return;
  float acc[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j] = 0.f;
  const T* w = W + static_cast<size_t>(o) * in;
  for (int k = lane; k < in; k += 32) {
    const float wk = to_f(w[k]);
#pragma unroll
    for (int j = 0; j < NT; ++j)
      if (n0 + j < n_tok) acc[j] = fmaf(wk, to_f(X[static_cast<size_t>(n0 + j) * ldx + k]), acc[j]);
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float v = warp_sum(acc[j]);
    if (lane == 0 && n0 + j < n_tok) Y[static_cast<size_t>(n0 + j) * ldy + o] = from_f<T>(v);
  }
}

// One block per new token: row = [W^DKV x ; RoPE_pos(W^KR x)] ([0h-n0]
// "MLA: 低ランクKV結合圧縮", [qiita] "RoPE の扱い"), rounded once, written to
// pool row block_table[b][pos/block]*block + pos%block.
template <typename T>
__global__ void __launch_bounds__(256) cache_append_kernel(
    const T* __restrict__ x, const T* __restrict__ w_dkr, const int* __restrict__ seq_idx,
    const int* __restrict__ pos, const int* __restrict__ block_table, int max_blocks, int batch,
    T* __restrict__ pool, int n_pool_blocks, int d_model, int d_c, int d_hr, int block,
    const float* __restrict__ rope_cos, const float* __restrict__ rope_sin, int max_pos,
    int* status) {
  extern __shared__ float row[];
  const int n = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int width = d_c + d_hr;
  const T* xn = x + static_cast<size_t>(n) * d_model;
  for (int o = warp; o < width; o += 8) {
    const T* w = w_dkr + static_cast<size_t>(o) * d_model;
    float acc = 0.f;
    for (int k = lane; k < d_model; k += 32) acc = fmaf(to_f(w[k]), to_f(xn[k]), acc);
    acc = warp_sum(acc);
    if (lane == 0) row[o] = acc;
  }
  __syncthreads();
  const int b = seq_idx[n], p = pos[n];
  if (b < 0 || b >= batch || p < 0 || p >= max_pos || p / block >= max_blocks) {
    if (threadIdx.x == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  const int blk = block_table[static_cast<size_t>(b) * max_blocks + p / block];
  if (blk < 0 || blk >= n_pool_blocks) {
    if (threadIdx.x == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  T* dst = pool + (static_cast<size_t>(blk) * block + p % block) * width;
  for (int k = threadIdx.x; k < d_c; k += blockDim.x) dst[k] = from_f<T>(row[k]);
  const int half = d_hr / 2;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const float c = rope_cos[static_cast<size_t>(p) * half + k];
    const float s = rope_sin[static_cast<size_t>(p) * half + k];
    const float x0 = row[d_c + 2 * k], x1 = row[d_c + 2 * k + 1];
    dst[d_c + 2 * k] = from_f<T>(x0 * c - x1 * s);
    dst[d_c + 2 * k + 1] = from_f<T>(x0 * s + x1 * c);
  }
}

// One block per (head, token): q~_i = W^UK_i^T q^C_i ([0h-n0] "行列吸収トリック")
// and RoPE_pos(q^R_i), written as one latent query row.
template <typename T>
__global__ void __launch_bounds__(256) absorb_q_kernel(const T* __restrict__ q_c,
                                                       const T* __restrict__ q_r,
                                                       const int* __restrict__ pos,
                                                       const T* __restrict__ w_uk, T* __restrict__ q_lat,
                                                       int n_h, int d_h, int d_hr, int d_c,
                                                       const float* __restrict__ rope_cos,
                                                       const float* __restrict__ rope_sin, int max_pos,
                                                       int* status) {
  extern __shared__ float qc[];
  const int i = blockIdx.x, n = blockIdx.y;
  const size_t hn = static_cast<size_t>(n) * n_h + i;
  for (int r = threadIdx.x; r < d_h; r += blockDim.x) qc[r] = to_f(q_c[hn * d_h + r]);
  __syncthreads();
  T* out = q_lat + hn * (d_c + d_hr);
  const T* w = w_uk + static_cast<size_t>(i) * d_h * d_c;
  for (int k = threadIdx.x; k < d_c; k += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < d_h; ++r) acc = fmaf(to_f(w[static_cast<size_t>(r) * d_c + k]), qc[r], acc);
    out[k] = from_f<T>(acc);
  }
  const int p = pos[n];
  if (p < 0 || p >= max_pos) {
    if (threadIdx.x == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  const int half = d_hr / 2;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const float c = rope_cos[static_cast<size_t>(p) * half + k];
    const float s = rope_sin[static_cast<size_t>(p) * half + k];
    const float x0 = to_f(q_r[hn * d_hr + 2 * k]), x1 = to_f(q_r[hn * d_hr + 2 * k + 1]);
    out[d_c + 2 * k] = from_f<T>(x0 * c - x1 * s);
    out[d_c + 2 * k + 1] = from_f<T>(x0 * s + x1 * c);
  }
}

// Folded query weight W~^UQ_i = W^UK_i^T W^UQ_i ([0h-n0] "行列吸収トリック":
// formed once, ahead of inference): Wt[i*d_c + c, k] = sum_e W_uk[i*d_h + e, c]
// W_uq[i*d_h + e, k], fp32 sums rounded once.  One 64 x 64 output tile of one
// head per block (blockIdx.z = head); 16 x 16 threads, 4 x 4 outputs each,
// both operand tiles staged through shared memory 16 rows of e at a time.
template <typename T>
__global__ void __launch_bounds__(256) absorb_weights_kernel(const T* __restrict__ w_uq,
                                                             const T* __restrict__ w_uk, T* __restrict__ w_abs,
                                                             int d_h, int d_c, int d_cq) {
  __shared__ float a[16][64];  // W_uk rows e, latent columns c
  __shared__ float b[16][64];  // W_uq rows e, input columns k
  const int i = blockIdx.z;
  const int c0 = blockIdx.y * 64, k0 = blockIdx.x * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  const T* uk = w_uk + static_cast<size_t>(i) * d_h * d_c;
  const T* uq = w_uq + static_cast<size_t>(i) * d_h * d_cq;
  for (int e0 = 0; e0 < d_h; e0 += 16) {
    for (int f = threadIdx.x; f < 16 * 64; f += 256) {
      const int e = e0 + f / 64, col = f % 64;
      a[f / 64][col] = (e < d_h && c0 + col < d_c) ? to_f(uk[static_cast<size_t>(e) * d_c + c0 + col]) : 0.f;
      b[f / 64][col] = (e < d_h && k0 + col < d_cq) ? to_f(uq[static_cast<size_t>(e) * d_cq + k0 + col]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float av[4], bv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        av[r] = a[e][ty * 4 + r];
        bv[r] = b[e][tx * 4 + r];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(av[r], bv[q], acc[r][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = c0 + ty * 4 + r;
    if (c >= d_c) continue;
    T* dst = w_abs + (static_cast<size_t>(i) * d_c + c) * d_cq;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (k0 + tx * 4 + q < d_cq) dst[k0 + tx * 4 + q] = from_f<T>(acc[r][q]);
  }
}

// One block per (head, token): the latent query straight from c^Q with the
// folded weight, [W~^UQ_i c^Q ; RoPE_pos(W^QR_i c^Q)] ([0h-n0] "行列吸収トリック",
// [qiita] "RoPE の扱い"), one warp per output feature.
template <typename T>
__global__ void __launch_bounds__(256) q_absorbed_kernel(const T* __restrict__ c_q, const T* __restrict__ w_abs,
                                                         const T* __restrict__ w_qr, const int* __restrict__ pos,
                                                         T* __restrict__ q_lat, int n_h, int d_cq, int d_hr,
                                                         int d_c, const float* __restrict__ rope_cos,
                                                         const float* __restrict__ rope_sin, int max_pos,
                                                         int* status) {
  extern __shared__ float sh[];  // c^Q [d_cq], then the raw positional query [d_hr]
  float* cq = sh;
  float* qr = sh + d_cq;
  const int i = blockIdx.x, n = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = threadIdx.x; k < d_cq; k += blockDim.x) cq[k] = to_f(c_q[static_cast<size_t>(n) * d_cq + k]);
  __syncthreads();
  const size_t hn = static_cast<size_t>(n) * n_h + i;
  T* out = q_lat + hn * (d_c + d_hr);
  for (int o = warp; o < d_c + d_hr; o += 8) {
    const T* w = o < d_c ? w_abs + (static_cast<size_t>(i) * d_c + o) * d_cq
                         : w_qr + (static_cast<size_t>(i) * d_hr + (o - d_c)) * d_cq;
    float acc = 0.f;
    for (int k = lane; k < d_cq; k += 32) acc = fmaf(to_f(w[k]), cq[k], acc);
    acc = warp_sum(acc);
    if (lane == 0) {
      if (o < d_c) out[o] = from_f<T>(acc);
      else qr[o - d_c] = acc;
    }
  }
  __syncthreads();
  const int p = pos[n];
  if (p < 0 || p >= max_pos) {
    if (threadIdx.x == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  const int half = d_hr / 2;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const float c = rope_cos[static_cast<size_t>(p) * half + k];
    const float s = rope_sin[static_cast<size_t>(p) * half + k];
    const float x0 = qr[2 * k], x1 = qr[2 * k + 1];
    out[d_c + 2 * k] = from_f<T>(x0 * c - x1 * s);
    out[d_c + 2 * k + 1] = from_f<T>(x0 * s + x1 * c);
  }
}

// One block (4 warps) per (token, head).  Warp w takes keys j = w, w+4, ...
// up to the token's position, keeps a running max / sum / weighted latent sum
// (online softmax), and the four warps are merged at the end.
// [qiita] "Attention 計算" in the absorbed form of [kasblo]
// "V側は、小さな表現の加重和を先に求める".
constexpr int kDecodeMaxPerLane = 16;  // d_c <= 512

template <typename T>
__global__ void __launch_bounds__(128) decode_kernel(
    const T* __restrict__ q_lat, const T* __restrict__ pool, int n_pool_blocks,
    const int* __restrict__ block_table, int max_blocks, const int* __restrict__ seq_lens,
    const int* __restrict__ cu_q, int batch, int n_tok, T* __restrict__ o_lat, float* __restrict__ lse,
    int n_h, int d_c, int d_hr, int block, float scale, int* status) {
  extern __shared__ float sm[];
  const int width = d_c + d_hr;
  float* q = sm;                     // [width]
  float* wm = q + width;             // [4]
  float* wl = wm + 4;                // [4]
  float* wacc = wl + 4;              // [4][d_c]
  const int n = blockIdx.x, i = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t hn = static_cast<size_t>(n) * n_h + i;
  const int b = seq_of_token(cu_q, batch, n);
  const int q_end = cu_q[b + 1];
  const int t = seq_lens[b] - (q_end - n);  // this token's position
  if (t < 0 || n >= q_end || n < cu_q[b] || cu_q[batch] != n_tok) {
    if (threadIdx.x == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  for (int k = threadIdx.x; k < width; k += blockDim.x) q[k] = to_f(q_lat[hn * width + k]);
  __syncthreads();
  float m = -INFINITY, l = 0.f;
  float acc[kDecodeMaxPerLane];
#pragma unroll
  for (int v = 0; v < kDecodeMaxPerLane; ++v) acc[v] = 0.f;
  bool bad = false;
  for (int j = warp; j <= t; j += 4) {
    const int lb = j / block;
    const int blk = lb < max_blocks ? block_table[static_cast<size_t>(b) * max_blocks + lb] : -1;
    if (blk < 0 || blk >= n_pool_blocks) { bad = true; continue; }
    const T* row = pool + (static_cast<size_t>(blk) * block + j % block) * width;
    float s = 0.f;
    for (int k = lane; k < width; k += 32) s = fmaf(q[k], to_f(row[k]), s);
    s = warp_sum(s) * scale;
    const float m_new = fmaxf(m, s);
    const float corr = expf(m - m_new);
    const float p = expf(s - m_new);
    l = l * corr + p;
#pragma unroll
    for (int v = 0; v < kDecodeMaxPerLane; ++v) {
      const int k = lane + 32 * v;
      if (k < d_c) acc[v] = acc[v] * corr + p * to_f(row[k]);
    }
    m = m_new;
  }
  if (bad && lane == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
  if (lane == 0) { wm[warp] = m; wl[warp] = l; }
#pragma unroll
  for (int v = 0; v < kDecodeMaxPerLane; ++v) {
    const int k = lane + 32 * v;
    if (k < d_c) wacc[warp * d_c + k] = acc[v];
  }
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w]);
  float L = 0.f, f[4];
  for (int w = 0; w < 4; ++w) {
    f[w] = wl[w] > 0.f ? expf(wm[w] - M) : 0.f;
    L += wl[w] * f[w];
  }
  for (int k = threadIdx.x; k < d_c; k += blockDim.x) {
    float o = 0.f;
    for (int w = 0; w < 4; ++w) o += wacc[w * d_c + k] * f[w];
    o_lat[hn * d_c + k] = from_f<T>(L > 0.f ? o / L : 0.f);
  }
  if (threadIdx.x == 0) lse[hn] = L > 0.f ? M + logf(L) : -INFINITY;
}

// One block per (head, token): o_i = W^UV_i o~_i, one warp per output row.
template <typename T>
__global__ void __launch_bounds__(256) up_project_kernel(const T* __restrict__ o_lat,
                                                         const T* __restrict__ w_uv, T* __restrict__ o,
                                                         int n_h, int d_h, int d_c) {
  extern __shared__ float ol[];
  const int i = blockIdx.x, n = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t hn = static_cast<size_t>(n) * n_h + i;
  for (int k = threadIdx.x; k < d_c; k += blockDim.x) ol[k] = to_f(o_lat[hn * d_c + k]);
  __syncthreads();
  for (int r = warp; r < d_h; r += 8) {
    const T* w = w_uv + (static_cast<size_t>(i) * d_h + r) * d_c;
    float acc = 0.f;
    for (int k = lane; k < d_c; k += 32) acc = fmaf(to_f(w[k]), ol[k], acc);
    acc = warp_sum(acc);
    if (lane == 0) o[hn * d_h + r] = from_f<T>(acc);
  }
}

}  // namespace

#define MLA_DISPATCH(h, BODY)                        \
  do {                                               \
    if ((h)->dims.dtype == MLA_BF16) {               \
      using T = __nv_bfloat16;                       \
      BODY;                                          \
    } else {                                         \
      using T = float;                               \
      BODY;                                          \
    }                                                \
  } while (0)

cudaError_t launch_linear(const mla_handle* h, const void* X, int ldx, const void* W, int in, int out,
                          void* Y, int ldy, int n_tok, cudaStream_t s) {
  constexpr int NT = 8;
  dim3 grid((out + 7) / 8, (n_tok + NT - 1) / NT);
  MLA_DISPATCH(h, (linear_kernel<T, NT><<<grid, 256, 0, s>>>(
                      static_cast<const T*>(X), ldx, static_cast<const T*>(W), in, out,
                      static_cast<T*>(Y), ldy, n_tok)));
  return cudaGetLastError();
}

cudaError_t launch_cache_append_simt(const mla_handle* h, const void* x, const void* w_dkr,
                                     const int* seq_idx, const int* pos, int n_new,
                                     const int* block_table, int max_blocks, int batch, void* pool,
                                     int n_pool_blocks, cudaStream_t s) {
  const mla_dims& d = h->dims;
  const size_t smem = sizeof(float) * (d.d_c + d.d_hr);
  MLA_DISPATCH(h, (cache_append_kernel<T><<<n_new, 256, smem, s>>>(
                      static_cast<const T*>(x), static_cast<const T*>(w_dkr), seq_idx, pos,
                      block_table, max_blocks, batch, static_cast<T*>(pool), n_pool_blocks,
                      d.d_model, d.d_c, d.d_hr, d.block, h->rope_cos, h->rope_sin, h->max_pos,
                      h->status)));
  return cudaGetLastError();
}

cudaError_t launch_absorb_q_simt(const mla_handle* h, const void* q_c, const void* q_r, const int* pos,
                                 int n_tok, const void* w_uk, void* q_lat, cudaStream_t s) {
  const mla_dims& d = h->dims;
  dim3 grid(d.n_h, n_tok);
  MLA_DISPATCH(h, (absorb_q_kernel<T><<<grid, 256, sizeof(float) * d.d_h, s>>>(
                      static_cast<const T*>(q_c), static_cast<const T*>(q_r), pos,
                      static_cast<const T*>(w_uk), static_cast<T*>(q_lat), d.n_h, d.d_h, d.d_hr,
                      d.d_c, h->rope_cos, h->rope_sin, h->max_pos, h->status)));
  return cudaGetLastError();
}

cudaError_t launch_absorb_weights(const mla_handle* h, const void* w_uq, const void* w_uk, void* w_abs,
                                  cudaStream_t s) {
  const mla_dims& d = h->dims;
  dim3 grid((d.d_cq + 63) / 64, (d.d_c + 63) / 64, d.n_h);
  MLA_DISPATCH(h, (absorb_weights_kernel<T><<<grid, 256, 0, s>>>(
                      static_cast<const T*>(w_uq), static_cast<const T*>(w_uk), static_cast<T*>(w_abs), d.d_h,
                      d.d_c, d.d_cq)));
  return cudaGetLastError();
}

cudaError_t launch_q_absorbed_simt(const mla_handle* h, const void* c_q, const void* w_abs, const void* w_qr,
                                   const int* pos, int n_tok, void* q_lat, cudaStream_t s) {
  const mla_dims& d = h->dims;
  dim3 grid(d.n_h, n_tok);
  const size_t smem = sizeof(float) * (d.d_cq + d.d_hr);
  if (smem > 48 * 1024) {
    MLA_DISPATCH(h, (cudaFuncSetAttribute(q_absorbed_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem))));
  }
  MLA_DISPATCH(h, (q_absorbed_kernel<T><<<grid, 256, smem, s>>>(
                      static_cast<const T*>(c_q), static_cast<const T*>(w_abs), static_cast<const T*>(w_qr), pos,
                      static_cast<T*>(q_lat), d.n_h, d.d_cq, d.d_hr, d.d_c, h->rope_cos, h->rope_sin,
                      h->max_pos, h->status)));
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const mla_handle* h, const void* q_lat, const void* pool,
                               int n_pool_blocks, const int* block_table, int max_blocks,
                               const int* seq_lens, const int* cu_q, int batch, int n_tok, void* o_lat,
                               float* lse, cudaStream_t s) {
  const mla_dims& d = h->dims;
  dim3 grid(n_tok, d.n_h);
  const size_t smem = sizeof(float) * (d.d_c + d.d_hr + 8 + 4 * d.d_c);
  if (smem > 48 * 1024) {
    MLA_DISPATCH(h, (cudaFuncSetAttribute(decode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem))));
  }
  MLA_DISPATCH(h, (decode_kernel<T><<<grid, 128, smem, s>>>(
                      static_cast<const T*>(q_lat), static_cast<const T*>(pool), n_pool_blocks,
                      block_table, max_blocks, seq_lens, cu_q, batch, n_tok, static_cast<T*>(o_lat),
                      lse, d.n_h, d.d_c, d.d_hr, d.block, d.scale, h->status)));
  return cudaGetLastError();
}

cudaError_t launch_up_project_simt(const mla_handle* h, const void* o_lat, const void* w_uv, int n_tok,
                                   void* o, cudaStream_t s) {
  const mla_dims& d = h->dims;
  dim3 grid(d.n_h, n_tok);
  MLA_DISPATCH(h, (up_project_kernel<T><<<grid, 256, sizeof(float) * d.d_c, s>>>(
                      static_cast<const T*>(o_lat), static_cast<const T*>(w_uv), static_cast<T*>(o),
                      d.n_h, d.d_h, d.d_c)));
  return cudaGetLastError();
}

}  // namespace mla
