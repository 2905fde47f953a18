/*
 * mla.h -- C ABI of the B300 (sm_103a) Multi-head Latent Attention decode library.
 *
 * Sources, cited by page and section heading:
 *   [0h-n0]  "論文解説: DeepSeek-V2 — MoEモデルのKVキャッシュを93.3%削減する
 *            Multi-head Latent Attention" (0h-n0.github.io)
 *   [kasblo] MLA explainer, kasblo.com
 *   [qiita]  MLA notes, qiita.com/joule
 *
 * The problem statement these calls follow: during generation only the new
 * token's query is computed while past keys/values come from a cache
 * ([qiita] "MHA における KV Cache の問題"); MLA caches, per token and layer,
 * the joint latent c^KV (d_c) and the shared RoPE key k^R (d_h^R) instead of
 * per-head K and V ([0h-n0] "Decoupled RoPE"), and attends to that cache
 * directly by absorbing W^UK into the query and W^UV into the output
 * ([0h-n0] "行列吸収トリック"; [kasblo] "V側は、小さな表現の加重和を先に求める").
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, 16-byte
 *   aligned, row-major and densely packed with the shape given at the call.
 *   The library never allocates or frees memory in these calls; the only
 *   allocation is in mla_create (RoPE table, status word).
 * - Floating-point buffers hold dims.dtype (bf16 or f32) unless stated
 *   otherwise; lse is always f32.  Integer buffers are int32.
 * - Calls are asynchronous on `stream`.  Arguments are validated on the host
 *   before anything is launched; a rejected call launches nothing and
 *   returns MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED or MLA_ERR_WORKSPACE.
 *   A failed launch returns MLA_ERR_CUDA.
 * - Values only the device can see (a block id outside the pool, a position
 *   outside the RoPE table, a sequence shorter than its query count) are
 *   checked in the kernels: the offending access is skipped and a bit is set
 *   in the handle's device status word, read back by
 *   mla_check_device_status.  Every wait inside a kernel is bounded; a wait
 *   that runs out sets MLA_ERR_DEVICE_TIMEOUT there as well.
 * - A call with zero tokens is a valid no-op.
 * - Head i owns rows [i*d_h, (i+1)*d_h) of W^UQ, W^UK, W^UV and rows
 *   [i*d_hr, (i+1)*d_hr) of W^QR; W^O consumes the head-major concatenation.
 * - RoPE rotates interleaved pairs (x[2k], x[2k+1]) by pos * rope_base^(-2k/d_hr),
 *   positions 0-based; the cos/sin table is computed on the host in double.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, inconsistent dims */
  MLA_ERR_UNSUPPORTED = 2,    /* valid request the library does not implement */
  MLA_ERR_WORKSPACE = 3,      /* workspace pointer null or smaller than required */
  MLA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  MLA_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait ran out */
  MLA_ERR_DEVICE_BOUNDS = 6   /* a device-side index check failed; access skipped */
} mla_status;

typedef enum { MLA_BF16 = 0, MLA_F32 = 1 } mla_dtype;

/* Layer sizes in the pages' notation ([0h-n0] "技術的詳細"; [qiita]
 * "Multi-Head Latent Attention"): n_h heads of width d_h, RoPE width d_hr
 * (d_h^R), KV latent d_c, query latent d_cq (d_c'), hidden d_model (d).
 * block = cache rows per block of the paged pool.  scale multiplies every
 * score; 1/sqrt(d_h + d_hr) per [qiita] "Attention 計算". */
typedef struct {
  int n_h, d_h, d_hr, d_c, d_cq, d_model, block;
  float rope_base;
  float scale;
  mla_dtype dtype;
} mla_dims;

typedef struct mla_handle mla_handle;

/* Creates a handle on the current CUDA device: copies dims, builds the RoPE
 * cos/sin table for positions [0, max_pos) and a 4-byte device status word.
 * Rejects odd d_hr, non-positive sizes, max_pos < 1.  *out is owned by the
 * caller and released with mla_destroy. */
mla_status mla_create(const mla_dims* dims, int max_pos, mla_handle** out);
void mla_destroy(mla_handle* h);
const char* mla_status_string(mla_status s);

/* Number of streaming multiprocessors the handle plans for, and whether the
 * tcgen05 path serves these dims (n_h=128, d_c=512, d_hr=64, block=64, bf16). */
int mla_num_sms(const mla_handle* h);
int mla_uses_tensor_path(const mla_handle* h);

/* Upper bound, in device polls, on every bounded wait of later launches
 * (0 = library default, 2^24 polls of roughly 0.1 us each, about 2 s).
 * Used to exercise the timeout path. */
mla_status mla_set_wait_limit(mla_handle* h, long long polls);

/* ---- a0: query projection --------------------------------------------------
 * [qiita] "Query の圧縮": c^Q = W^DQ x, q^C_i = W^UQ_i c^Q;
 * [qiita] "RoPE の扱い": q^R_i = W^QR_i c^Q (returned before the rotation,
 * which mla_absorb_q applies).
 *   x    [n_tok, d_model]     w_dq [d_cq, d_model]
 *   w_uq [n_h*d_h, d_cq]      w_qr [n_h*d_hr, d_cq]
 *   q_c  [n_tok, n_h, d_h]    q_r  [n_tok, n_h, d_hr]   (outputs)
 *   ws: mla_q_proj_workspace_bytes(h, n_tok) bytes (holds c^Q). */
size_t mla_q_proj_workspace_bytes(const mla_handle* h, int n_tok);
mla_status mla_q_proj(mla_handle* h, const void* x, const void* w_dq, const void* w_uq,
                      const void* w_qr, int n_tok, void* q_c, void* q_r, void* ws,
                      size_t ws_bytes, cudaStream_t stream);

/* ---- a1: cache append ------------------------------------------------------
 * [0h-n0] "MLA: 低ランクKV結合圧縮": c^KV_t = W^DKV h_t; [qiita] "RoPE の扱い":
 * k^R_t = RoPE(W^KR h_t); [0h-n0] "Decoupled RoPE": the cached row is
 * [c^KV_t ; k^R_t], d_c + d_hr elements, k^R stored after the rotation.
 *   x          [n_new, d_model]     new tokens' hidden states
 *   w_dkr      [d_c + d_hr, d_model] rows 0..d_c-1 = W^DKV, rows d_c.. = W^KR
 *   seq_idx    [n_new]  sequence of each new token, in [0, batch)
 *   pos        [n_new]  its 0-based position in that sequence
 *   block_table[batch, max_blocks]  physical block of each logical block
 *   pool       [n_pool_blocks, block, d_c + d_hr]  (written)
 * Row of token (b, p) = block_table[b*max_blocks + p/block]*block + p%block.
 * A block id outside [0, n_pool_blocks) or p/block >= max_blocks skips the
 * row and sets MLA_ERR_DEVICE_BOUNDS. */
mla_status mla_cache_append(mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx,
                            const int* pos, int n_new, const int* block_table, int max_blocks,
                            int batch, void* pool, int n_pool_blocks, cudaStream_t stream);

/* ---- a0 + a1 + a2 in one call: the latent query and the cache rows --------
 * mla_q_proj_append followed by mla_absorb_q for the same new tokens, without
 * q^C and q^R leaving the GPU's on-chip memory when there are at most 64
 * tokens: one launch computes c^Q = W^DQ x together with the cache rows, a
 * second gives each head a CTA that chains q^C_i = W^UQ_i c^Q and
 * q~_i = W^UK_i^T q^C_i ([0h-n0] "行列吸収トリック") and rotates W^QR c^Q
 * ([qiita] "RoPE の扱い") into q_lat.  Beyond 64 tokens, or for sizes outside
 * the tensor path, it runs the two calls' kernels.
 *   x, w_dq, w_uq, w_qr, w_dkr, seq_idx, pos, block_table, pool: as in
 *   mla_q_proj / mla_cache_append; w_uk as in mla_absorb_q
 *   q_lat [n_tok, n_h, d_c + d_hr] (output)
 *   ws: mla_q_latent_append_workspace_bytes(h, n_tok) bytes (c^Q, and q^C /
 *       q^R when they are formed)
 * q^C is rounded once to bf16 before the absorption, as on the separate
 * route; the rotation of q^R is applied to its fp32 sum (the separate route
 * rotates the stored bf16 q^R). */
size_t mla_q_latent_append_workspace_bytes(const mla_handle* h, int n_tok);
mla_status mla_q_latent_append(mla_handle* h, const void* x, const void* w_dq, const void* w_uq,
                               const void* w_qr, const void* w_uk, const void* w_dkr,
                               const int* seq_idx, const int* pos, int n_tok,
                               const int* block_table, int max_blocks, int batch, void* pool,
                               int n_pool_blocks, void* q_lat, void* ws, size_t ws_bytes,
                               cudaStream_t stream);

/* ---- a0 + a1 in one call ---------------------------------------------------
 * mla_q_proj and mla_cache_append for the same new tokens (x is their input
 * h, n_tok of them), with the two products that read x -- c^Q = W^DQ x and
 * the cache rows [W^DKV x ; RoPE_pos(W^KR x)] -- issued as one launch.  The
 * arguments are those of the two calls (ws: mla_q_proj_workspace_bytes(h,
 * n_tok) bytes); the results are theirs up to the order of the fp32 sums.
 * Sizes outside the tensor path run the two calls one after the other. */
mla_status mla_q_proj_append(mla_handle* h, const void* x, const void* w_dq, const void* w_uq,
                             const void* w_qr, const void* w_dkr, const int* seq_idx, const int* pos,
                             int n_tok, const int* block_table, int max_blocks, int batch, void* pool,
                             int n_pool_blocks, void* q_c, void* q_r, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* ---- a1 with the quantised latent cache -------------------------------------
 * [0h-n0] "量子化との組み合わせ": c^KV can further be stored with KV-cache
 * quantisation of the Q8_0 kind.  Each cached row becomes 672 bytes:
 *   bytes [0, 512)    int8 codes of c^KV, value j in byte j
 *   bytes [512, 544)  16 fp16 scales, scale b for values [32b, 32b+32)
 *   bytes [544, 672)  k^R, 64 bf16 values (stored after the rotation)
 * Value j stands for code_j * scale_(j/32).  The row quantised is the bf16
 * row mla_cache_append would store; per 32-value run, scale = fp16(max|x| /
 * 127) and code = x / scale rounded to nearest with ties away from zero (both
 * divisions in fp32, correctly rounded), 0 when the run is all zero.
 *   x, w_dkr, seq_idx, pos, block_table, max_blocks, batch: as in
 *   mla_cache_append
 *   pool_q8 [n_pool_blocks, block, 672] bytes (written), 16-byte aligned
 *   ws: mla_cache_append_q8_workspace_bytes(h, n_new) bytes (the bf16 rows)
 * Tensor-path sizes only (n_h = 128, d_c = 512, d_hr = 64, block = 64, bf16);
 * others return MLA_ERR_UNSUPPORTED.  Bounds errors as in mla_cache_append. */
size_t mla_cache_append_q8_workspace_bytes(const mla_handle* h, int n_new);
mla_status mla_cache_append_q8(mla_handle* h, const void* x, const void* w_dkr, const int* seq_idx,
                               const int* pos, int n_new, const int* block_table, int max_blocks,
                               int batch, void* pool_q8, int n_pool_blocks, void* ws, size_t ws_bytes,
                               cudaStream_t stream);

/* ---- a2: query absorption --------------------------------------------------
 * [0h-n0] "行列吸収トリック": q~_i = W^UK_i^T q^C_i (d_c), and q^R_i rotated at
 * the token's position ([qiita] "RoPE の扱い").
 *   q_c [n_tok, n_h, d_h]   q_r [n_tok, n_h, d_hr] (raw)   pos [n_tok]
 *   w_uk [n_h*d_h, d_c]
 *   q_lat [n_tok, n_h, d_c + d_hr] = [q~_i ; RoPE_pos(q^R_i)]   (output) */
mla_status mla_absorb_q(mla_handle* h, const void* q_c, const void* q_r, const int* pos,
                        int n_tok, const void* w_uk, void* q_lat, cudaStream_t stream);

/* ---- a0 + a2 with the folded query weight ----------------------------------
 * [0h-n0] "行列吸収トリック": W~^UQ_i = W^UK_i^T W^UQ_i can be formed once,
 * ahead of inference; the latent content query is then the single product
 * W~^UQ_i c^Q, and no q^C is formed.
 *
 * mla_absorb_weights forms the folded weight (a preparation step, not part
 * of the decode step): fp32 sums over the head's d_h rows, rounded once.
 *   w_uq [n_h*d_h, d_cq]   w_uk [n_h*d_h, d_c]
 *   w_uq_abs [n_h*d_c, d_cq]  (output; rows [i*d_c, (i+1)*d_c) = head i)
 *
 * mla_q_proj_absorbed replaces mla_q_proj + mla_absorb_q:
 * c^Q = W^DQ x, then q_lat = [W~^UQ_i c^Q ; RoPE_pos(W^QR_i c^Q)].
 *   x [n_tok, d_model]   w_dq [d_cq, d_model]   w_uq_abs as above
 *   w_qr [n_h*d_hr, d_cq]   pos [n_tok] int32 (0-based positions)
 *   q_lat [n_tok, n_h, d_c + d_hr]  (output, the layout mla_decode reads)
 *   ws: mla_q_proj_workspace_bytes(h, n_tok) bytes (holds c^Q).
 * A position outside [0, max_pos) leaves that token's positional part
 * unwritten and sets MLA_ERR_DEVICE_BOUNDS.  Which is faster depends on
 * n_tok: the folded weight is d_c/d_h = 4 times the size of W^UQ. */
mla_status mla_absorb_weights(mla_handle* h, const void* w_uq, const void* w_uk, void* w_uq_abs,
                              cudaStream_t stream);
mla_status mla_q_proj_absorbed(mla_handle* h, const void* x, const void* w_dq, const void* w_uq_abs,
                               const void* w_qr, const int* pos, int n_tok, void* q_lat, void* ws,
                               size_t ws_bytes, cudaStream_t stream);

/* ---- a3 + a4: latent attention over the paged cache -----------------------
 * [qiita] "Attention 計算" in absorbed form: s_ij = scale*(q~_i.c_j + q^R_i.k^R_j)
 * for every cached row j <= t (t = the query's position), softmax over j,
 * o~_i = sum_j a_ij c_j ([kasblo] "V側は、小さな表現の加重和を先に求める"),
 * lse_i = ln sum_j exp(s_ij).
 *   q_lat [n_tok, n_h, d_c + d_hr]
 *   pool, n_pool_blocks, block_table, max_blocks: as in mla_cache_append
 *   seq_lens [batch]  cached rows of each sequence INCLUDING this step's tokens
 *   cu_q [batch+1]    query tokens of sequence b are rows cu_q[b]..cu_q[b+1]-1;
 *                     they sit at positions seq_lens[b]-q_len .. seq_lens[b]-1
 *                     and see rows 0..their own position (causal, inclusive)
 *   num_workers       0 = one worker per available SM pair; otherwise the
 *                     number of workers (two SMs each) launched.  On the
 *                     device the plan gives each worker one whole token when
 *                     there are no more tokens than workers and their key
 *                     counts are close, else a balanced range of all keys;
 *                     keys of a token split across workers are merged by a
 *                     log-sum-exp combine (not on the pages).
 *   ws                mla_decode_workspace_bytes(h, n_tok, num_workers) bytes
 *   o_lat [n_tok, n_h, d_c]  (output, dims.dtype)   lse [n_tok, n_h] f32 (output)
 * n_tok must equal cu_q[batch] (checked on the device). */
size_t mla_decode_workspace_bytes(const mla_handle* h, int n_tok, int num_workers);
mla_status mla_decode(mla_handle* h, const void* q_lat, const void* pool, int n_pool_blocks,
                      const int* block_table, int max_blocks, const int* seq_lens,
                      const int* cu_q, int batch, int n_tok, int num_workers, void* ws,
                      size_t ws_bytes, void* o_lat, float* lse, cudaStream_t stream);

/* ---- L2 prefetch during the attention --------------------------------------
 * Not on the pages: a scheduling aid for the step of [qiita] "Attention 計算",
 * whose output projection u = W^O [o_1; ...; o_nh] (with o_i = W^UV_i o~_i,
 * [kasblo] "V側は、小さな表現の加重和を先に求める") reads its weights right
 * after the attention.  The attention leaves HBM bandwidth unused, so later
 * mla_decode and mla_decode_q8 calls on this handle fetch up to two device
 * ranges into L2 while they stream the cache, spread evenly over the call:
 * the ranges end to end are cut into one piece per 64-row tile of the call
 * and per SM of the pair that loads it.  The cache is read at evict-first
 * priority and the prefetch lands at normal priority, so what fits in L2
 * beside the other normal-priority data is still there when the next kernel
 * on the stream reads it.  The query-side projection kernels read their
 * weights at normal priority too: a step's query weights replace the lines
 * the previous step prefetched, so each step fetches its ranges from HBM
 * again.
 * Only addresses and sizes are kept: the ranges must stay valid while such
 * calls run, and nothing reads them for results (a stale range costs
 * bandwidth only).
 *   ptrs[n], bytes[n]  n <= 2; each pointer 16-byte aligned, each size a
 *                      multiple of 16 (0 = unused); n = 0 clears.
 * Returns MLA_ERR_INVALID_ARG otherwise.  mla_decode_noalloc does not
 * prefetch.  Thread-safe against concurrent calls on the handle. */
mla_status mla_set_decode_l2_prefetch(mla_handle* h, const void* const* ptrs, const size_t* bytes, int n);

/* ---- a3 + a4 over the quantised latent cache -------------------------------
 * The attention of mla_decode with the cache rows of mla_cache_append_q8
 * ([0h-n0] "量子化との組み合わせ"): row j stands for [code_j * scale_(j/32) ;
 * k^R], and each value is rounded once to fp16 on chip before the MMAs (which
 * take fp16 operands for this path; the queries and P are rounded to fp16).  The
 * cache stream is 672 bytes per row instead of 1152.
 *   pool_q8 [n_pool_blocks, block, 672] bytes; every other argument, the
 *   workspace (mla_decode_workspace_bytes) and the outputs as in mla_decode.
 * Tensor-path sizes only; others return MLA_ERR_UNSUPPORTED. */
mla_status mla_decode_q8(mla_handle* h, const void* q_lat, const void* pool_q8, int n_pool_blocks,
                         const int* block_table, int max_blocks, const int* seq_lens, const int* cu_q,
                         int batch, int n_tok, int num_workers, void* ws, size_t ws_bytes, void* o_lat,
                         float* lse, cudaStream_t stream);

/* ---- decode without a workspace argument ------------------------------------
 * The pages have no counterpart to this call; it is a convenience of this
 * library.  It computes exactly what mla_decode computes, for callers that
 * cannot allocate device memory when they call: for example a plugin whose
 * host serving engine has reserved the whole device-memory budget and offers
 * it no allocator, or a latency-critical loop that must not call cudaMalloc
 * because that call can synchronise the device and take unbounded time.
 *
 * Its split-KV scratch is one fixed array in device memory (16,909,312 bytes
 * on the tensor path) that every device holding the library keeps until the
 * process exits.  It is reserved on a device when the first handle with the
 * tensor-path sizes is created there: mla_create looks up the array's device
 * address with that device current (which loads the library's device code
 * there) and keeps it in the handle, so a caller that must not allocate later
 * creates its handles before it hands the rest of the memory away.  Limits:
 * n_tok <= 8192 and at most 32 workers (num_workers = 0 picks
 * min(SMs/2, 32)); larger requests return MLA_ERR_WORKSPACE without
 * launching.  Layer sizes outside the tensor path need no scratch and run the
 * generic kernels.
 *
 * Every call shares the one array: calls whose kernels overlap on the GPU
 * (other streams, other threads, other handles of the same device) race on
 * it and must be serialised by the caller.  Nothing in the array needs to
 * start at zero; each call writes every scratch byte it later reads.
 * This call allocates nothing and frees nothing.  Arguments and outputs are
 * those of mla_decode. */
mla_status mla_decode_noalloc(mla_handle* h, const void* q_lat, const void* pool, int n_pool_blocks,
                              const int* block_table, int max_blocks, const int* seq_lens,
                              const int* cu_q, int batch, int n_tok, int num_workers, void* o_lat,
                              float* lse, cudaStream_t stream);

/* ---- prefill over expanded keys and values ---------------------------------
 * Causal attention of a whole prompt in the un-absorbed form the pages give
 * for prefill: with many tokens at once the latent vectors are up-projected
 * to full keys and values by a large matrix product ([perforder]
 * "極限最適化の代償：MLA特有の学習負荷と独自Tritonカーネルという障壁"; the
 * reference's "naive" branch, [kasblo] "「キャッシュを減らせた」と「その割合だけ
 * 速い」は別の評価").  Per head i: K^C_i = C W^UK_i^T and V_i = C W^UV_i^T for
 * the prompt's latent rows C; for query t and key j <= t ([qiita] "Attention
 * 計算") s_tj = (q^C_t,i . K^C_j,i + RoPE_t(q^R_t,i) . k^R_j) / sqrt(d_h + d_hr),
 * a softmax over j and o_t,i = sum_j a_tj V_j,i.  Positions are 0..P-1.
 *   rows [P, d_c + d_hr]  the prompt's cache rows in position order, bf16, as
 *                         mla_cache_append writes them (c^KV ; rotated k^R)
 *   q_c [P, n_h, d_h], q_r [P, n_h, d_hr]  as mla_q_proj writes them (q^R
 *                         before its rotation)
 *   w_uk, w_uv [n_h*d_h, d_c]
 *   ws: mla_prefill_workspace_bytes(h, P) bytes (K^C and V, fp16: the
 *       attention multiplies fp16 operands with fp32 accumulation)
 *   o [P, n_h, d_h] bf16 (output), lse [P, n_h] f32 natural log (output)
 * P <= max_pos.  Tensor-path sizes only; others return MLA_ERR_UNSUPPORTED. */
size_t mla_prefill_workspace_bytes(const mla_handle* h, int P);
mla_status mla_prefill(mla_handle* h, const void* rows, const void* q_c, const void* q_r, int P,
                       const void* w_uk, const void* w_uv, void* ws, size_t ws_bytes, void* o,
                       float* lse, cudaStream_t stream);

/* ---- a5: output ------------------------------------------------------------
 * o_i = W^UV_i o~_i ([kasblo] "V側は、小さな表現の加重和を先に求める") and
 * u = W^O [o_1; ...; o_n_h] ([qiita] "Attention 計算").
 *   o_lat [n_tok, n_h, d_c]   w_uv [n_h*d_h, d_c]   w_o [d_model, n_h*d_h]
 *   u [n_tok, d_model] (output)
 *   ws: mla_out_workspace_bytes(h, n_tok) bytes (holds the per-head o_i).
 * Up to 64 tokens at the tensor-path sizes this is one launch: every CTA
 * first computes the o_i of one or two heads (bf16, into ws), a counter of
 * the handle then releases the W^O phase once every CTA has done so.  Two
 * mla_out calls of one handle must therefore not run on the GPU at the same
 * time (other streams or threads): the handle's counters are shared. */
size_t mla_out_workspace_bytes(const mla_handle* h, int n_tok);
mla_status mla_out(mla_handle* h, const void* o_lat, const void* w_uv, const void* w_o,
                   int n_tok, void* u, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, returns the first error any kernel recorded in the
 * device status word since the last check (MLA_OK if none) and clears it. */
mla_status mla_check_device_status(mla_handle* h, cudaStream_t stream);

/* Where the first bounded wait that ran out (MLA_ERR_DEVICE_TIMEOUT) gave up,
 * as read back by the last mla_check_device_status: *site = 0 when none did,
 * else 0x40000000 | (wait site within its kernel << 8) | warp; *cta = the
 * CTA's linear index; *tile = the tile it waited for, or -1 where the kernel
 * does not record it.
 * Diagnostic only; the sites are numbered in the kernels' sources. */
mla_status mla_device_error_site(const mla_handle* h, int* site, int* cta, int* tile);

/* Runs one kernel that waits on a barrier no one arrives at, with the
 * handle's wait limit; it must come back with MLA_ERR_DEVICE_TIMEOUT recorded
 * in the status word.  Exercises the bounded-wait path without a fault. */
mla_status mla_selftest_wait_timeout(mla_handle* h, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
