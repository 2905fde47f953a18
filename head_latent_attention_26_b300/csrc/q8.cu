// q8.cu -- the quantised latent cache.
//
// [0h-n0] "量子化との組み合わせ" notes that the compressed c^KV can be stored
// further with KV-cache quantisation of the Q8_0 kind.  The format taken here
// is that kind's definition: every run of 32 consecutive c^KV values of a row
// shares one scale d = max|x| / 127 kept in fp16, and each value becomes the
// int8 code round(x / d), nearest with ties away from zero (d = 0 and codes 0
// for an all-zero run).  k^R, shared by all heads and carrying the rotation,
// stays bf16.  A cached row is 672 bytes:
//   [ 512 int8 codes | 16 fp16 scales | 64 bf16 k^R ]
// against 1152 for the bf16 row.  The values quantised are the bf16 row the
// plain append would store (the same projection and rounding), and the scale
// and codes are decided in fp32 with correctly rounded divisions, so the
// codes are a function of that bf16 row alone.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kDc = 512, kDhr = 64, kWidth = kDc + kDhr;
constexpr int kQBlock = 32;                        // values per scale
constexpr int kRowBytes = kDc + 2 * (kDc / kQBlock) + 2 * kDhr;  // 672
constexpr int kScalesAt = kDc, kRopeAt = kDc + 2 * (kDc / kQBlock);

// One warp per new token: lanes 0..15 quantise one 32-value run of c^KV each,
// lanes 16..31 copy the 128 bytes of k^R; the row goes to pool slot
// block_table[b][pos / block] * block + pos % block.
__global__ void __launch_bounds__(256) quantize_scatter_q8_kernel(
    const __nv_bfloat16* __restrict__ rows, const int* __restrict__ seq_idx, const int* __restrict__ pos, int n_new,
    const int* __restrict__ block_table, int max_blocks, int batch, uint8_t* __restrict__ pool, int n_pool_blocks,
    int block, int* status) {
  pdl_wait();  // the rows come from the previous kernel
  if (threadIdx.x == 0) pdl_trigger();
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (n >= n_new) return;
  const int b = __ldg(seq_idx + n), tp = __ldg(pos + n);
  if (b < 0 || b >= batch || tp < 0 || tp / block >= max_blocks) {
    if (lane == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  const int blk = __ldg(block_table + static_cast<size_t>(b) * max_blocks + tp / block);
  if (blk < 0 || blk >= n_pool_blocks) {
    if (lane == 0) report(status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  uint8_t* dst = pool + (static_cast<size_t>(blk) * block + tp % block) * kRowBytes;
  const __nv_bfloat16* src = rows + static_cast<size_t>(n) * kWidth;
  if (lane < kDc / kQBlock) {
    float v[kQBlock];
    const uint4* s4 = reinterpret_cast<const uint4*>(src + kQBlock * lane);
#pragma unroll
    for (int i = 0; i < kQBlock / 8; ++i) {
      const uint4 w = s4[i];
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * i + 2 * j] = __uint_as_float(ww[j] << 16);
        v[8 * i + 2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kQBlock; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const __half d16 = __float2half_rn(__fdiv_rn(amax, 127.f));
    const float d = __half2float(d16);
    uint32_t packed[kQBlock / 4];
#pragma unroll
    for (int i = 0; i < kQBlock / 4; ++i) packed[i] = 0;
    if (d > 0.f) {
#pragma unroll
      for (int i = 0; i < kQBlock; ++i) {
        const float q = __fdiv_rn(v[i], d);
        float r = floorf(fabsf(q) + 0.5f);  // nearest, ties away from zero
        r = fminf(r, 127.f);
        const int code = q < 0.f ? -static_cast<int>(r) : static_cast<int>(r);
        packed[i / 4] |= (static_cast<uint32_t>(code) & 0xFFu) << (8 * (i % 4));
      }
    }
    uint4* c4 = reinterpret_cast<uint4*>(dst + kQBlock * lane);
    c4[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    c4[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    *reinterpret_cast<__half*>(dst + kScalesAt + 2 * lane) = d16;
  } else {
    const int i = lane - kDc / kQBlock;  // 16 lanes x 8 bytes of k^R
    *reinterpret_cast<uint2*>(dst + kRopeAt + 8 * i) = *reinterpret_cast<const uint2*>(src + kDc + 4 * i);
  }
}

}  // namespace

cudaError_t launch_quantize_scatter_q8(const mla_handle* h, const void* rows, const int* seq_idx, const int* pos,
                                       int n_new, const int* block_table, int max_blocks, int batch, void* pool,
                                       int n_pool_blocks, cudaStream_t s) {
  return launch_pdl(quantize_scatter_q8_kernel, dim3((n_new + 7) / 8), dim3(256), 0, s, 1,
                    static_cast<const __nv_bfloat16*>(rows), seq_idx, pos, n_new, block_table, max_blocks, batch,
                    static_cast<uint8_t*>(pool), n_pool_blocks, h->dims.block, h->status);
}

}  // namespace mla
