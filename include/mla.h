/*
 * mla.h — C ABI of the B300 (sm_103a) MLA latent-cache decode library.
 *
 * One decode step of one Multi-head Latent Attention (MLA) layer over its
 * compressed KV cache. Every cached token holds a 512-wide latent c_KV plus a
 * shared 64-wide decoupled RoPE key k^R: 576 elements per token per layer.
 *   "DeepSeek-V2 机制拆解：KV 缓存压缩 93.3% 是怎么做到的" (discosf.com),
 *     §"长上下文推理的第一瓶颈": decode re-reads every previous token's K/V; only
 *     the d_c = 512 latent is cached and K/V are up-projected from it; W_UK can
 *     be absorbed into the query side and W_UV into the output side.
 *   Same page, §"解耦 RoPE 与 YaRN": RoPE is carried by a decoupled per-head query
 *     and a shared key of width 64 so that absorption survives.
 *   "DeepSeek-V2: A Strong, Economical, and Efficient Mixture-of-Experts Language
 *     Model - 中文验证版" (ai-papers.xuzou.cn), §"瓶颈" and §"方法适配": cache
 *     formula (d_c + d_h^R)·l, d_c = 512, d_h^R = 64, 128 heads.
 *
 * The step is these calls on the caller's stream (the last two, or their fused form):
 *   mla_absorb_q   q_lat[b,h] = [ W_UK[h]^T q^C[b,h]  ‖  RoPE(q^R[b,h], pos[b]) ]
 *   mla_decode_fwd split-KV attention of every head over the 576-wide cache rows
 *   mla_combine    log-sum-exp merge of the per-split partial results
 *   mla_up_v       o[b,h] = W_UV[h] o_lat[b,h]
 *   mla_combine_up_v  the two calls above in one launch
 *
 * Conventions shared by every call
 *   - All pointers except `cache` (a host struct) are DEVICE pointers; the caller
 *     allocates and owns every buffer. The library allocates nothing, keeps no
 *     state beyond a per-device attribute cache, and never synchronises the stream.
 *   - Tensors are dense row-major with the shapes given; base addresses must be
 *     16-byte aligned.
 *   - bf16 means IEEE bfloat16 stored as 16-bit words.
 *   - Arguments are validated on the host before any CUDA call; a bad argument
 *     returns MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED and launches nothing.
 *     A launch failure reported by the runtime returns MLA_ERR_CUDA.
 *   - Problems only the device can see (a page id outside the pool, a bounded
 *     wait that ran out) are written to the optional device status word
 *     (first error wins; the caller zeroes it) and the affected work is skipped.
 *   - Fixed widths: d_h = 128 (q^C), d_h^R = 64, d_c = 512, row = 576.
 *     n_h must be 16, 32, 64 or 128.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#define MLA_ABI_VERSION 1
#define MLA_D_NOPE 128
#define MLA_D_ROPE 64
#define MLA_D_LATENT 512
#define MLA_D_ROW 576
#define MLA_D_Q 192
#define MLA_PAGE_SIZE 64
#define MLA_MAX_SPLITS 256

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size          */
  MLA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. n_h = 96)  */
  MLA_ERR_WORKSPACE = 3,     /* a size/limit of a caller buffer exceeded   */
  MLA_ERR_CUDA = 4,          /* the CUDA runtime reported an error         */
  MLA_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up             */
  MLA_ERR_DEVICE_BOUNDS = 6  /* device: a page id fell outside the pool    */
} mla_status;

typedef enum mla_kv_dtype {
  MLA_KV_BF16 = 0,      /* rows of 576 bf16 (1152 bytes)                      */
  MLA_KV_FP8_E4M3 = 1   /* rows of 576 e4m3 codes (576 bytes) + fp32 scale    */
} mla_kv_dtype;

/*
 * View of one layer's latent cache (host struct; the pointers inside are device
 * memory owned by the caller). Token t of sequence b lives in row
 *   contiguous (block_table == NULL): b * seq_stride_tokens + t
 *   paged      (block_table != NULL): block_table[b * max_pages + t / 64] * 64 + t % 64
 * Row r starts at byte r * 1152 (bf16) or r * 576 (e4m3) of `data`; columns
 * 0..511 are c_KV and 512..575 the RoPE key, stored already rotated at t.
 * For e4m3 the token's value is code * scales[r] (one fp32 scale per row).
 * Rows in [L_b, ...) of a sequence's last page are never used for attention.
 */
typedef struct mla_cache {
  int32_t dtype;                /* mla_kv_dtype                                   */
  int32_t page_size;            /* must be 64 when block_table != NULL            */
  const void* data;             /* device rows                                    */
  const float* scales;          /* device [num_rows] fp32 (e4m3 only), else NULL  */
  const int32_t* block_table;   /* device [B, max_pages] page ids, or NULL        */
  int32_t max_pages;            /* row stride of block_table (entries)            */
  int32_t reserved;             /* must be 0                                      */
  int64_t seq_stride_tokens;    /* contiguous only: rows between sequences        */
  int64_t num_rows;             /* rows addressable through data (bounds checks)  */
} mla_cache;

/*
 * mla_absorb_q — fold W_UK into the query and rotate the decoupled query part.
 *   ("DeepSeek-V2 机制拆解", §"长上下文推理的第一瓶颈" (absorption) and
 *    §"解耦 RoPE 与 YaRN" (decoupled RoPE).)
 *   q     [B, n_h, 192] bf16: q^C = q[..., 0:128], q^R = q[..., 128:192]
 *   w_uk  [n_h, 128, 512] bf16 (K_h = W_UK[h] · c)
 *   pos   [B] int32 query position (>= 0), normally L_b - 1
 *   q_lat [B, n_h, 576] bf16 out:
 *         q_lat[b,h,j]       = sum_d q^C[b,h,d] W_UK[h,d,j]          (j < 512)
 *         q_lat[b,h,512 + i] = rotate-half RoPE of q^R[b,h] at pos[b],
 *                              pair (i, i+32), angle pos * rope_base^(-i/32)
 *   Accumulation fp32, RoPE angles reduced in fp64, result rounded to bf16.
 */
MLA_API mla_status mla_absorb_q(const void* q, const void* w_uk, const int32_t* pos,
                        int B, int n_h, float rope_base, void* q_lat,
                        cudaStream_t stream);

/*
 * RoPE of the decoupled query and key, for the _ex entry points.
 *   ("DeepSeek-V2 机制拆解", §"解耦 RoPE 与 YaRN": the 128K context comes from YaRN on
 *    the decoupled shared key, scale 40, alpha 1, beta 32, target 160K; "中文验证版",
 *    §"计算设置": pre-training length 4K. The pages give no formula; this follows the
 *    published YaRN frequency rule.)
 *   Pair i's frequency is theta_i = base^(-i/32) (plain RoPE, yarn_scale = 1), or with
 *   YaRN, from the turns r_i = original_max_pos * theta_i / (2 pi) the pair makes over
 *   the original context: theta_i when r_i >= yarn_beta, theta_i / yarn_scale when
 *   r_i <= yarn_alpha, and (1 - g) theta_i / yarn_scale + g theta_i with
 *   g = (r_i - yarn_alpha) / (yarn_beta - yarn_alpha) in between. YaRN's attention
 *   temperature is the caller's softmax_scale (mla_decode_fwd). The pages' setting:
 *   {10000, 40, 1, 32, 4096, 0}.
 */
typedef struct mla_rope {
  float base;                   /* > 1                                              */
  float yarn_scale;             /* 1: plain RoPE; > 1: YaRN                          */
  float yarn_alpha;             /* YaRN: 0 <= alpha < beta (turns over the context)  */
  float yarn_beta;
  int32_t original_max_pos;     /* YaRN: the original context length (>= 1)          */
  int32_t reserved;             /* must be 0                                         */
} mla_rope;

/* mla_absorb_q with the RoPE of `rope` (host struct) instead of plain RoPE of base
 * rope_base. mla_absorb_q(..., base, ...) equals this with {base, 1, 0, 0, 0, 0}. */
MLA_API mla_status mla_absorb_q_ex(const void* q, const void* w_uk, const int32_t* pos,
                                   int B, int n_h, const mla_rope* rope, void* q_lat,
                                   cudaStream_t stream);

/*
 * mla_decode_fwd — split-KV attention of all heads over the latent cache.
 *   Scores s[h,t] = softmax_scale * (q_lat[b,h,:] . row_t[0:576]), softmax over
 *   the tokens of each split with a running maximum, and the value is the latent
 *   itself: o_part = sum_t p[h,t] row_t[0:512] / sum_t p[h,t].
 *   ("DeepSeek-V2 机制拆解", §"长上下文推理的第一瓶颈": with W_UK/W_UV absorbed,
 *    all heads attend directly over the cached latent.)
 *   q_lat      [B, n_h, 576] bf16
 *   cache      host pointer to the cache view above
 *   seq_lens   [B] int32 device, 0 <= L_b <= max_seq_len
 *   max_seq_len host upper bound of seq_lens (sizes the launch)
 *   num_splits S, 1..MLA_MAX_SPLITS: uniform splits; or 0: the library's schedule
 *              with S = mla_num_splits(B, max_seq_len, n_h) slots per sequence
 *   o_part     [B, S, n_h, 512] fp32 out, normalised per slot
 *   lse_part   [B, S, n_h] fp32 out, natural-log normaliser of the slot
 *   status     optional device int32 (may be NULL)
 *   Uniform splits (num_splits >= 1): slot s of sequence b covers the tokens
 *   mla_split_range(L_b, S, s) returns; a slot without tokens gets lse = -inf, o = 0.
 *   Library schedule (num_splits = 0): for a paged bf16 cache the batch's 128-token
 *   tiles, sequence after sequence, are shared out evenly among the GPU's SM pairs
 *   (or, when every sequence has the same tile count and that is cheaper, each
 *   sequence is cut into equal pieces); each sequence is cut into at most S pieces
 *   (one per slot, in token order); slots a sequence does not use get lse = -inf and
 *   their o_part is left as it was. For a contiguous cache and for an e4m3 cache the
 *   schedule is uniform splits, sized for max_seq_len, over the first slots. Either
 *   way mla_combine over the S slots gives the whole-sequence result.
 *   A cache of 2^31 - 256 rows or more returns MLA_ERR_UNSUPPORTED (32-bit TMA rows).
 */
MLA_API mla_status mla_decode_fwd(const void* q_lat, const mla_cache* cache,
                          const int32_t* seq_lens, int B, int n_h, int max_seq_len,
                          float softmax_scale, int num_splits,
                          float* o_part, float* lse_part, int32_t* status,
                          cudaStream_t stream);

/*
 * mla_combine — merge split partials by log-sum-exp.
 *   m = max_s lse[s];  w_s = exp(lse[s] - m);  o_lat = sum_s w_s o_part[s] / sum_s w_s;
 *   lse = m + ln sum_s w_s.  Splits with lse = -inf weigh 0; if all are empty the
 *   result is o_lat = 0, lse = -inf.
 *   o_part [B, S, n_h, 512] fp32, lse_part [B, S, n_h] fp32
 *   o_lat  [B, n_h, 512] fp32 out;  lse [B, n_h] fp32 out (may be NULL)
 */
MLA_API mla_status mla_combine(const float* o_part, const float* lse_part, int B,
                       int num_splits, int n_h, float* o_lat, float* lse,
                       cudaStream_t stream);

/*
 * mla_up_v — apply W_UV on the output side.
 *   ("DeepSeek-V2 机制拆解", §"长上下文推理的第一瓶颈": V = W_UV · c, absorbed.)
 *   o[b,h,d] = sum_j W_UV[h,d,j] o_lat[b,h,j]
 *   o_lat [B, n_h, 512] fp32, w_uv [n_h, 128, 512] bf16, o [B, n_h, 128] fp32 out
 *   (W_O, which would follow, is outside this library.)
 */
MLA_API mla_status mla_up_v(const float* o_lat, const void* w_uv, int B, int n_h,
                    float* o, cudaStream_t stream);

/*
 * mla_combine_up_v — mla_combine and mla_up_v as one kernel launch.
 *   ("DeepSeek-V2 机制拆解", §"长上下文推理的第一瓶颈": the weighted sum over the cached
 *   latents, then W_UV; the split partials are merged as mla_combine defines.)
 *   o[b,h,d] = sum_j W_UV[h,d,j] o_lat[b,h,j], with o_lat the merge of o_part's slots.
 *   o_part [B, num_splits, n_h, 512] fp32, lse_part [B, num_splits, n_h] fp32 (as
 *   mla_decode_fwd writes them), w_uv [n_h, 128, 512] bf16, o [B, n_h, 128] fp32 out.
 *   o_lat [B, n_h, 512] fp32 and lse [B, n_h] fp32 are optional outputs (NULL: not
 *   written); when given they hold mla_combine's results up to fp32 rounding order.
 *   The merged o_lat never passes through memory on its way to W_UV.
 *   Errors: NULL o_part, lse_part, w_uv or o, misalignment (16 bytes; lse 4 bytes),
 *   B or num_splits out of range -> MLA_ERR_INVALID_ARG; n_h not 16/32/64/128 ->
 *   MLA_ERR_UNSUPPORTED. o must not alias the inputs.
 */
MLA_API mla_status mla_combine_up_v(const float* o_part, const float* lse_part, int B,
                            int num_splits, int n_h, const void* w_uv, float* o,
                            float* o_lat, float* lse, cudaStream_t stream);

/*
 * mla_cache_append — write the cache rows of T new tokens.
 *   ("DeepSeek-V2 机制拆解", §"长上下文推理的第一瓶颈": each token's hidden state is
 *    down-projected to the cached latent c_KV, d_c = 512; §"解耦 RoPE 与 YaRN": the
 *    shared 64-wide key carries the position, rotated where it is made; hidden size
 *    5120: "中文验证版", §"计算设置".)
 *   c_KV[t] = W_DKV h[t];  k^R[t] = RoPE(W_KR h[t], pos[t]) (the pairing of mla_absorb_q)
 *   row[t]  = bf16([c_KV[t] ‖ k^R[t]]) stored as token pos[t] of sequence seq_ids[t]:
 *     contiguous cache: row seq * seq_stride_tokens + pos
 *     paged cache:      page block_table[seq, pos / 64], slot pos % 64
 *   For an e4m3 cache the bf16 row is written to `staging` and then quantised as by
 *   mla_quantize_fp8 into the cache's codes and scales at that row.
 *   h        [T, d_model] bf16 (d_model a multiple of 512, at most 32768)
 *   w_dkv    [512, d_model] bf16;  w_kr [64, d_model] bf16
 *   seq_ids, pos  [T] int32 device
 *   num_seqs sequences of the cache (rows of the block table, or contiguous sequences)
 *   cache    the layer's cache; its rows (and scales) are WRITTEN
 *   staging  [T, 576] bf16 device scratch, required for an e4m3 cache, else ignored
 *   status   optional device word: MLA_ERR_DEVICE_BOUNDS for a token whose sequence,
 *            position or page lies outside the cache (that token is not written)
 *   T = 0 is a no-op. Two tokens with the same destination race (one of them wins).
 */
MLA_API mla_status mla_cache_append(const void* h, const void* w_dkv, const void* w_kr,
                                    const int32_t* seq_ids, const int32_t* pos, int T,
                                    int d_model, float rope_base, const mla_cache* cache,
                                    int num_seqs, void* staging, int32_t* status,
                                    cudaStream_t stream);

/* mla_cache_append with the RoPE of `rope` (see mla_rope) for the shared key. */
MLA_API mla_status mla_cache_append_ex(const void* h, const void* w_dkv, const void* w_kr,
                                       const int32_t* seq_ids, const int32_t* pos, int T,
                                       int d_model, const mla_rope* rope,
                                       const mla_cache* cache, int num_seqs, void* staging,
                                       int32_t* status, cudaStream_t stream);

/*
 * mla_multi_token_view — several new query tokens per sequence (speculative or chunked
 * decoding), decoded as B*T sequences of one paged view of the same cache.
 *   ("DeepSeek-V2 机制拆解", §"长上下文推理的第一瓶颈": every new token attends to all
 *    earlier tokens; with T new tokens at the end of sequence b, query j sits at
 *    position L_b - T + j and sees tokens 0 .. L_b - T + j.)
 *   Sequence v = b*T + j of the view: view_seq_lens[v] = max(L_b - T + j + 1, 0),
 *   view_pos[v] = max(view_seq_lens[v] - 1, 0) (the query position for mla_absorb_q),
 *   block-table row v = the pages of sequence b (a paged cache's own row, or for a
 *   contiguous cache its rows b*seq_stride .. taken 64 at a time, which needs
 *   seq_stride_tokens and num_rows to be multiples of 64, else MLA_ERR_UNSUPPORTED).
 *   `*view` (host) receives the paged view: the same rows and scales, this block table.
 *   The step is then mla_absorb_q (B*T queries, view_pos), mla_decode_fwd over `view`
 *   with view_seq_lens, mla_combine and mla_up_v, all on B*T sequences.
 *   seq_lens [B] int32 device; view_seq_lens, view_pos [B*T] int32 device out;
 *   view_block_table [B*T, view_max_pages] int32 device out, view_max_pages >=
 *   ceil(max_seq_len / 64). B*T <= 65535.
 */
MLA_API mla_status mla_multi_token_view(const mla_cache* cache, const int32_t* seq_lens, int B,
                                        int T, int max_seq_len, int32_t* view_seq_lens,
                                        int32_t* view_pos, int32_t* view_block_table,
                                        int view_max_pages, mla_cache* view,
                                        cudaStream_t stream);

/*
 * mla_quantize_fp8 — cache-write helper: bf16 rows → e4m3 rows + per-row scale.
 *   The pages report a low-bit KV cache for serving ("DeepSeek-V2 机制拆解",
 *   §"推理参数与 128K 上下文的使用注意"; "中文验证版", §"方法适配") without its format;
 *   this library's stand-in is e4m3 with one fp32 scale per token:
 *   scale = amax/448 (amax = max |x| over the 576 elements; 1 for a zero row),
 *   code  = e4m3(x / scale), fp32 division, round-to-nearest-even, saturating.
 *   rows [num_rows, 576] bf16; codes [num_rows, 576] uint8 out; scales [num_rows] fp32 out
 */
MLA_API mla_status mla_quantize_fp8(const void* rows, int64_t num_rows, uint8_t* codes,
                            float* scales, cudaStream_t stream);

/*
 * mla_quantize_fp6 — bf16 rows → the ~6-bit cache format (a reading of the pages'
 *   "about 6 bits per element": "DeepSeek-V2 机制拆解", §"推理参数与 128K 上下文的使用注意";
 *   "中文验证版", §"瓶颈"; the pages give no format). No decode kernel reads it yet.
 *   The layout is the published microscaling one for 6-bit elements (MXFP6 E2M3):
 *   each row's 576 elements form eighteen blocks of 32 that share a power-of-two
 *   scale X = 2^se, se = floor(log2 amax) - 2 clamped to -127..127 (0 for an all-zero
 *   block), stored as the byte se + 127; each element is coded e2m3(x / X): 6 bits
 *   s ee mmm, exponent bias 1, values up to 7.5, round to nearest with ties to the
 *   even code, saturating. Codes 4t .. 4t+3 of a row are the little-endian 24-bit word
 *   c0 | c1 << 6 | c2 << 12 | c3 << 18 at bytes 3t .. 3t+2.
 *   rows [num_rows, 576] bf16 (finite values; 16-byte aligned);
 *   packed [num_rows, 432] uint8 out; scales [num_rows, 18] uint8 out.
 *   Errors: NULL pointers, misaligned rows, num_rows < 0 -> MLA_ERR_INVALID_ARG;
 *   num_rows = 0 is a no-op.
 */
MLA_API mla_status mla_quantize_fp6(const void* rows, int64_t num_rows, uint8_t* packed,
                            uint8_t* scales, cudaStream_t stream);

/*
 * mla_decode_combine_static — mla_decode_fwd followed by mla_combine with the split
 * partials kept in a fixed device array inside the library instead of caller memory.
 *   (No counterpart on the pages: it exists for callers that cannot allocate device
 *   memory, e.g. an extension under a host framework that owns all of the GPU's memory,
 *   or latency-critical code that cannot afford cudaMalloc's implicit synchronisation.)
 *   Arguments as for mla_decode_fwd and mla_combine; o_lat [B, n_h, 512] fp32 out,
 *   lse [B, n_h] fp32 out (may be NULL).
 *   The partials need B * S * n_h * 2052 bytes (each of the two parts rounded up to
 *   256 bytes); more than MLA_STATIC_SCRATCH_BYTES returns MLA_ERR_WORKSPACE before any
 *   launch. The array (MLA_STATIC_SCRATCH_BYTES on every GPU that loads the library,
 *   held until exit) is shared by all calls and keeps the last call's partials: calls
 *   that overlap on the GPU race, and the caller must serialise them. The first call
 *   on a device (and the first after a device reset replaced its context) looks the
 *   array's device address up (cudaGetSymbolAddress) and should come before any stream
 *   capture. Allocates nothing.
 */
#define MLA_STATIC_SCRATCH_BYTES (64 << 20)
MLA_API mla_status mla_decode_combine_static(const void* q_lat, const mla_cache* cache, const int32_t* seq_lens,
                                             int B, int n_h, int max_seq_len, float softmax_scale, int num_splits,
                                             float* o_lat, float* lse, int32_t* status, cudaStream_t stream);

/* Decode kernels (mla_decode_kernel's answer). */
#define MLA_KERNEL_TC_BF16 1    /* tcgen05 tensor-core kernel, bf16 operands, fp32 accum.*/
#define MLA_KERNEL_TC_E4M3 2     /* tcgen05 kernel for an e4m3 cache: QK^T on the codes
                                    (kind::f8f6f4, the query as two e4m3 parts), PV on f16
                                    operands converted from the codes; fp32 accumulation */

/* Which decode kernel mla_decode_fwd runs for this cache dtype and head count
 * (-1 for an invalid combination). Host only. */
MLA_API int mla_decode_kernel(int kv_dtype, int n_h);

/* Slots per sequence that num_splits = 0 uses (>= 1, <= MLA_MAX_SPLITS): the o_part /
 * lse_part sizes to allocate for it. Host only. */
MLA_API int mla_num_splits(int B, int max_seq_len, int n_h);

/*
 * Token range [*start, *end) of split `split` of a sequence of seq_len tokens
 * under num_splits splits: chunk = 64 * ceil(ceil(seq_len / 64) / num_splits),
 * start = min(split * chunk, seq_len), end = min(start + chunk, seq_len).
 * Host only; returns MLA_ERR_INVALID_ARG for bad arguments.
 */
MLA_API mla_status mla_split_range(int seq_len, int num_splits, int split, int* start, int* end);

MLA_API const char* mla_status_string(int status);
MLA_API int mla_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
