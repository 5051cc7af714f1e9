/*
 * mla.h -- C ABI of libmla.so: DeepSeek Multi-head Latent Attention (MLA)
 * decode in absorb mode over a paged 576-wide latent cache, on one GB300
 * (sm_103a).
 *
 * What is computed (citations name the source page by its title and section):
 *
 *   Each cached token is ONE row shared by all heads: the KV latent c (d_c =
 *   512 values) followed by the decoupled RoPE key k_r (d_rope = 64), rotated
 *   at the token's absolute position before it is stored
 *   ("DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.4, 576 =
 *   512 + 64 elements per token and layer).
 *
 *   A decode step of sequence b with context length L = ctx_len[b] computes,
 *   for every head h, with the query at position L - 1:
 *
 *     q_lat[h] = W_UK[h]^T q_nope[h]                        (key absorption, §2.2)
 *     s_t      = scale * ( q_lat[h] . c_t + RoPE(q_pe[h], L-1) . k_r,t )
 *     o_lat[h] = sum_t softmax(s)_t c_t                     (latent sum, §2.3)
 *     out[h]   = W_UV[h] o_lat[h]                           (value absorption, §2.3)
 *
 *   with scale = 1/sqrt(d_nope + d_rope) unless set.  In exact arithmetic this
 *   equals standard MLA, which expands K = [W_UK c ; k_r] and V = W_UV c per
 *   head ("80 行 PyTorch 从零写 DeepSeek 的 MLA" §4-§5).  RoPE rotates
 *   interleaved pairs (2i, 2i+1) by pos * base^(-2i/d_rope) (same page,
 *   附录 A).  The decode reads B * s_ctx * (d_c + d_rope) * e bytes of cache,
 *   with no head count in it ("G5 MLA KV 访存建模设计规格" 算法与公式,
 *   eq. gmkv-read).
 *
 * Conventions for every call:
 *   - Tensor arguments are DEVICE pointers to caller-owned memory, row-major,
 *     densely packed unless a stride is given.  bf16 means IEEE bfloat16 bits.
 *   - Work is enqueued asynchronously on the given stream (NULL = legacy
 *     default stream); the call returns after launching.  Host-side argument
 *     checks happen before anything is launched: on error nothing is enqueued.
 *   - mla_kv_append and mla_decode allocate nothing.
 *   - Data-dependent problems found ON THE DEVICE (a context length or page id
 *     out of range, an append index out of range) never trap: the affected
 *     sequence's output is zeroed (or the row is not written) and a bit is
 *     set in the handle's device check word, read by mla_get_status().
 *   - The library is built for sm_103a only; there is no CPU or other-GPU
 *     path.  mla_create fails with MLA_ERR_UNSUPPORTED on any other device.
 *   - Error messages are kept per host thread; mla_last_error() returns the
 *     message of the calling thread's last failed call.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* identical to cudaStream_t's target */
typedef struct CUstream_st* mla_stream_t;
typedef struct mla_handle_s* mla_handle_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_MISSING_FIELD = 1,   /* a mandatory mla_config_t field is 0 / unset  */
  MLA_ERR_INVALID_ARG = 2,     /* a pointer, size or stride argument is invalid */
  MLA_ERR_UNSUPPORTED = 3,     /* valid but not built: shape, dtype, device     */
  MLA_ERR_WORKSPACE = 4,       /* workspace NULL, too small or misaligned       */
  MLA_ERR_CUDA = 5,            /* a CUDA runtime / driver call failed           */
  MLA_ERR_DEVICE_CHECK = 6     /* mla_get_status: the device check word was set */
} mla_status_t;

typedef enum {
  MLA_CACHE_BF16 = 1,          /* 576 bf16 per row: 1152 bytes                  */
  MLA_CACHE_FP8_E4M3 = 2,      /* 576 OCP e4m3 bytes per row, one fp32 scale    */
  MLA_CACHE_FP8_E4M3_BLOCK = 3 /* 656 bytes per row: 512 e4m3 latent codes, 4
                                  fp32 scales (one per 128 latent values), 64
                                  bf16 RoPE-key values ("G5 MLA KV 访存建模设计
                                  规格" 附录 A: FlashMLA's FP8 row of 656 bytes
                                  with per-block scales)                        */
} mla_cache_dtype_t;

/* Bits of the device check word (mla_get_status's *device_flags). */
#define MLA_CHECK_CTX_LEN      0x1u  /* ctx_len[b] < 1 or > max_ctx                  */
#define MLA_CHECK_PAGE_ID      0x2u  /* a block-table entry outside [0, num_pages)   */
#define MLA_CHECK_APPEND_INDEX 0x4u  /* append: seq or pos out of range              */
#define MLA_CHECK_TIMEOUT      0x8u  /* a bounded in-kernel wait ran out             */

/*
 * Layer configuration.  Every field is mandatory: a zero (unset) integer or
 * float field fails mla_create with MLA_ERR_MISSING_FIELD, and the message
 * names the field and says it came from mla_config_t ("G5 MLA KV
 * 访存建模设计规格" 约束: kv_lora_rank and qk_rope_head_dim must be given and
 * a missing field raises with its name and source, never a silent default).
 * The two exceptions are stated on their fields.
 */
typedef struct mla_config {
  int32_t d_c;          /* KV latent width (kv_lora_rank).  Built: 512.                  */
  int32_t d_rope;       /* decoupled RoPE key width (qk_rope_head_dim).  Built: 64.      */
  int32_t n_h;          /* query heads.  Built: 1..128.                                   */
  int32_t d_nope;       /* no-RoPE query/key width per head.  Built: 128.                 */
  int32_t d_v;          /* value width per head.  Built: 128.                             */
  int32_t page_size;    /* tokens per cache page.  Built: 64.                             */
  int32_t cache_dtype;  /* mla_cache_dtype_t.                                             */
  int32_t max_position; /* size of the RoPE table: positions 0..max_position-1.  <= 2^20. */
  float rope_base;      /* RoPE base (10000 for the configurations here).                 */
  float softmax_scale;  /* EXCEPTION: 0 means 1/sqrt(d_nope + d_rope).                    */
  float fp8_scale;      /* EXCEPTION: mandatory (> 0) only for MLA_CACHE_FP8_E4M3, where a
                           stored code x represents x * fp8_scale; ignored otherwise (the
                           per-block format carries its scales in every row).             */
} mla_config_t;

/*
 * mla_create -- validate the configuration, copy the weights, build tables.
 *
 *   cfg     host pointer to the configuration (copied).
 *   w_uk    device, [n_h][d_nope][d_c] bf16: W_UK[h] maps a latent c to the
 *           no-RoPE key of head h (k = W_UK[h] c; the first half of each head's
 *           rows of kv_b_proj / wkv_b, "DeepSeek MLA 吸收式缓存" §3.3).
 *   w_uv    device, [n_h][d_v][d_c] bf16: W_UV[h] maps a latent to head h's value.
 *   stream  the copies run on it; mla_create synchronizes it before returning,
 *           so the caller may free w_uk / w_uv afterwards.
 *   out     receives the handle.
 *
 * The handle owns device copies of both weights (as given), an fp32 RoPE
 * cos/sin table (angles computed in float64 on the host) and a device check
 * word.  Errors: MLA_ERR_MISSING_FIELD, MLA_ERR_INVALID_ARG (NULL pointer),
 * MLA_ERR_UNSUPPORTED (shape other than the built ones, or not an sm_103
 * device), MLA_ERR_CUDA.
 */
mla_status_t mla_create(const mla_config_t* cfg, const void* w_uk, const void* w_uv,
                        mla_stream_t stream, mla_handle_t* out);

/* mla_destroy -- synchronize the device and free everything the handle owns. NULL is a no-op. */
mla_status_t mla_destroy(mla_handle_t h);

/*
 * mla_kv_append -- write n token rows into the paged cache.
 *
 * Row i (rows[i], d_c + d_rope bf16 values: latent first, then the UNROTATED
 * RoPE key) is token pos[i] of sequence seq[i].  It is stored at page
 * block_table[seq[i] * bt_stride + pos[i] / page_size], slot pos[i] % page_size:
 * the latent copied unchanged, the RoPE key rotated at position pos[i]
 * ("DeepSeek MLA 吸收式缓存" §2.4: the rope key depends on position and is
 * cached; "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2: keys rotated at their
 * absolute positions).  For an FP8 cache all d_c + d_rope stored values are
 * divided by fp8_scale in fp32 and encoded e4m3, nearest-even, saturating at
 * +-448.  For a per-block FP8 cache each block of 128 latent values gets the
 * scale max|x| / 448 (fp32 division; 0 for an all-zero block, whose codes are
 * 0), its values are divided by it in fp32 and encoded as above, and the RoPE
 * key is stored in bf16 as in a bf16 cache.  The rotation is computed in fp32
 * with fp32 cos/sin, each product and sum rounded separately.
 *
 *   rows         device [n][d_c + d_rope] bf16.
 *   seq, pos     device [n] int32.
 *   n            rows to write (0 is a no-op).
 *   block_table  device [bt_rows][bt_stride] int32 page ids.
 *   cache        device [num_pages][page_size][row], row = 1152 (bf16), 576 (e4m3) or
 *                656 (per-block e4m3) bytes.
 *
 * Rows written by one call must target distinct slots.  Device checks: seq
 * outside [0, bt_rows), pos outside [0, max_position) or past the block-table
 * row, or a page id outside [0, num_pages): the row is skipped and
 * MLA_CHECK_APPEND_INDEX / MLA_CHECK_PAGE_ID is set.
 */
mla_status_t mla_kv_append(mla_handle_t h, const void* rows, const int32_t* seq,
                           const int32_t* pos, int32_t n, const int32_t* block_table,
                           int32_t bt_rows, int32_t bt_stride, void* cache,
                           int32_t num_pages, mla_stream_t stream);

/*
 * mla_kv_project_append -- the down-projection of n hidden states into cache rows, written into
 * the paged cache in the same call.
 *
 * Row i = x[i] . W_DKV^T ("DeepSeek-V2-Lite 真实权重执行审计" §3.1: kv_a_proj_with_mqa maps a
 * hidden state to the [d_c | d_rope] row; the kv norm is the identity here), each value the
 * bf16 rounding of an fp32 sum, is then stored exactly as mla_kv_append stores a row (same
 * slot, rotation, encoding and device checks): the bytes equal those of mla_project into a
 * rows buffer followed by mla_kv_append, for every cache format (with the per-block FP8
 * cache a CTA projects whole rows, since a block's scale needs all 128 of its values).
 *
 *   x            device [n][hidden] bf16, 16-byte aligned.
 *   hidden       a positive multiple of 256.
 *   w_dkv        device [d_c + d_rope][hidden] bf16, 16-byte aligned (caller-owned).
 *   seq, pos, n, block_table, bt_rows, bt_stride, cache, num_pages: as in mla_kv_append.
 */
mla_status_t mla_kv_project_append(mla_handle_t h, const void* x, int32_t hidden, const void* w_dkv,
                                   const int32_t* seq, const int32_t* pos, int32_t n,
                                   const int32_t* block_table, int32_t bt_rows, int32_t bt_stride,
                                   void* cache, int32_t num_pages, mla_stream_t stream);

/*
 * mla_project -- y = x . W^T for a few rows: the query projection (W_Q: [n_h (d_nope +
 * d_rope)][hidden], giving q in the layout mla_decode takes, "80 行 PyTorch 从零写 DeepSeek 的
 * MLA" §2) and the output projection over the heads' concatenated values (W_O).
 *
 *   x            device [m][k] bf16, 16-byte aligned; m >= 0 rows (0 is a no-op).
 *   k            a positive multiple of 256.
 *   w            device [n_out][k] bf16, 16-byte aligned (caller-owned).
 *   n_out        a positive multiple of 16.
 *   y            device [m][n_out] bf16, 4-byte aligned: each value the bf16 rounding of an
 *                fp32 sum accumulated in a fixed order.
 */
mla_status_t mla_project(mla_handle_t h, const void* x, int32_t m, int32_t k, const void* w, int32_t n_out,
                         void* y, mla_stream_t stream);

/*
 * mla_rmsnorm -- RMSNorm of m rows: y = x / sqrt(mean(x^2) + eps) * w (Zhang & Sennrich 2019;
 * "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §3.3 names the latent's norm,
 * kv_a_layernorm / kv_norm).  Sum of squares and scaling in fp32, each value (x * inv) * w
 * rounded to bf16.  Rows are strided, so the latent part of [d_c + d_rope] rows can be
 * normalised in place (y == x, ld_y == ld_x) between mla_project and mla_kv_append, and the
 * low-rank query's qz between its two projections.
 *
 *   x            device [m][ld_x] bf16, 16-byte aligned; values 0 .. n - 1 of each row are used.
 *   m            rows (0 is a no-op).
 *   n            a positive multiple of 8, at most 8192.
 *   ld_x, ld_y   row strides in values: multiples of 8, >= n.
 *   w            device [n] bf16, 16-byte aligned (caller-owned).
 *   eps          >= 0, added to the mean square under the root.
 *   y            device [m][ld_y] bf16, 16-byte aligned; may be x.
 */
mla_status_t mla_rmsnorm(mla_handle_t h, const void* x, int32_t m, int32_t n, int32_t ld_x, const void* w, float eps,
                         void* y, int32_t ld_y, mla_stream_t stream);

/*
 * mla_expand_kv -- the standard-mode (naive) cache of an MLA layer, for comparison with the
 * absorbed path ("80 行 PyTorch 从零写 DeepSeek 的 MLA" §3/§5: the naive mode caches each
 * head's key and value; "DeepSeek-V2-Lite 真实权重执行审计" §3.2: 10,240 bytes per token at
 * 16 heads against 1,152 for the latent row).
 *
 * For every slot of every page: key_h = [W_UK[h] c ; k_r] (d_nope + d_rope) and value_h =
 * W_UV[h] c (d_v), each product an fp32 sum rounded to bf16, k_r copied as cached (already
 * rotated).  Slots that hold no token produce values nobody reads.
 *
 *   cache        device, a bf16 cache as written by mla_kv_append (an FP8 cache is
 *                MLA_ERR_UNSUPPORTED), 16-byte aligned.
 *   num_pages    pages of cache (and of kvx).
 *   kvx          device [num_pages][page_size][n_h][d_nope + d_rope + d_v] bf16, 16-byte aligned.
 */
mla_status_t mla_expand_kv(mla_handle_t h, const void* cache, int32_t num_pages, void* kvx, mla_stream_t stream);

/* mla_decode_naive_workspace_size -- device workspace bytes of mla_decode_naive. */
mla_status_t mla_decode_naive_workspace_size(mla_handle_t h, int32_t batch, int32_t max_ctx, size_t* bytes);

/*
 * mla_decode_naive -- standard-mode decode over the expanded cache: per sequence and head,
 * o_h = sum_t softmax_t(q_h . key_h,t * scale) value_h,t with q_h = [q_nope ; RoPE(q_pe,
 * ctx_len - 1)] -- the same function as mla_decode (the pages' naive = absorbed identity),
 * computed without absorption, reading n_h (d_nope + d_rope + d_v) values per token.
 *
 * Arguments as in mla_decode, with kvx (from mla_expand_kv, same block table and page ids) in
 * place of the latent cache; out is [batch][n_h][d_v] bf16.  Split-KV over 256-token pieces
 * merged by log-sum-exp.  Device checks as in mla_decode (bad lengths and page ids zero that
 * sequence's output and set the check word).
 */
mla_status_t mla_decode_naive(mla_handle_t h, const void* q, const int32_t* ctx_len, int32_t batch, int32_t max_ctx,
                              const int32_t* block_table, int32_t bt_stride, const void* kvx, int32_t num_pages,
                              void* workspace, size_t workspace_bytes, void* out, mla_stream_t stream);

/* mla_prefill_workspace_size -- device workspace bytes of mla_prefill:
 * batch * round_up(max_ctx, 128) * (2 n_h d_nope + d_rope) * 2 (the expanded keys and values)
 * + 256 (the attention kernel's work counter).  Calls sharing a workspace run in stream order. */
mla_status_t mla_prefill_workspace_size(mla_handle_t h, int32_t batch, int32_t max_ctx, size_t* bytes);

/*
 * mla_prefill -- causal prefill of a chunk of query tokens per sequence over the sequence's
 * cached rows, in MHA mode ("G5 MLA KV 访存建模设计规格", 名词定义 and 用例 2: prefill takes
 * every prompt token at once and is compute-bound; "DeepSeek MLA 吸收式缓存：真实权重执行与
 * FlashMLA 架构边界" §6.1: FlashMLA's dense prefill runs in MHA mode).
 *
 * The chunk's rows must already be in the cache (mla_kv_append / mla_kv_project_append).  Query
 * i of sequence b is at position ctx_len[b] - q_len[b] + i and attends the cached rows 0 .. that
 * position:  o_h = sum_t softmax_t(scale q_h . [W_UK[h] c_t ; k_r,t]) W_UV[h] c_t,  q_h =
 * [q_nope ; RoPE(q_pe, position)].  A whole prompt is q_len = ctx_len; a chunk after a cached
 * prefix is q_len < ctx_len.  Keys and values are expanded per head into the workspace (bf16
 * values of fp32 sums), then attention runs on the tensor cores: fp32 scores and sums, bf16 P.
 *
 *   q            device [total_q][n_h][d_nope + d_rope] bf16, 16-byte aligned, unrotated (as in
 *                mla_decode); the rows of sequence b are q_start[b] .. q_start[b] + q_len[b] - 1.
 *   q_start      device [batch] int32: first query row of each sequence.
 *   q_len        device [batch] int32: query tokens of each sequence, 0 <= q_len <= ctx_len and
 *                q_len <= max_q.
 *   total_q      rows of q and out (>= 1).
 *   max_q        host bound on q_len, 1 <= max_q <= max_ctx (sets the grid).
 *   ctx_len, batch, max_ctx, block_table, bt_stride, num_pages: as in mla_decode.
 *   cache        device, the handle's cache format, 128-byte aligned (an FP8 cache's values are
 *                decoded -- codes times the tensor scale, or times their block's scale -- as the
 *                expansion loads them).
 *   workspace    device, >= mla_prefill_workspace_size bytes, 256-byte aligned; overwritten.
 *   out          device [total_q][n_h][d_v] bf16, 32-byte aligned: row q_start[b] + i is the
 *                output of query i of sequence b; other rows are not written.
 *
 * Device checks (mla_get_status): a sequence whose q_start / q_len do not fit [0, total_q)
 * or exceed max_q sets MLA_CHECK_CTX_LEN and writes nothing; one whose ctx_len is outside
 * [1, max_ctx] or below q_len sets MLA_CHECK_CTX_LEN and gets zero rows; a page id outside
 * [0, num_pages) in the pages its queries see sets MLA_CHECK_PAGE_ID and zeroes those rows.
 */
mla_status_t mla_prefill(mla_handle_t h, const void* q, const int32_t* q_start, const int32_t* q_len,
                         int32_t total_q, int32_t max_q, const int32_t* ctx_len, int32_t batch, int32_t max_ctx,
                         const int32_t* block_table, int32_t bt_stride, const void* cache, int32_t num_pages,
                         void* workspace, size_t workspace_bytes, void* out, mla_stream_t stream);

/*
 * mla_decode_workspace_size -- bytes of device workspace mla_decode needs for
 * a batch of `batch` sequences of at most `max_ctx` tokens.  The workspace
 * holds the split plan, the absorbed queries and the split partials.
 */
mla_status_t mla_decode_workspace_size(mla_handle_t h, int32_t batch, int32_t max_ctx,
                                       size_t* bytes);

/*
 * mla_decode -- one decode step for `batch` sequences (one query token each).
 *
 *   q            device [batch][n_h][d_nope + d_rope] bf16: per head the no-RoPE
 *                part, then the unrotated RoPE part.  The query sits at position
 *                ctx_len[b] - 1 (its own row must already be appended).
 *   ctx_len      device [batch] int32, each in [1, max_ctx].
 *   block_table  device [batch][bt_stride] int32: row b lists sequence b's pages.
 *   cache        device, as written by mla_kv_append.
 *   workspace    device, >= mla_decode_workspace_size(h, batch, max_ctx) bytes,
 *                256-byte aligned; contents are scratch (not kept between calls).
 *   out          device [batch][n_h][d_v] bf16: per head the attention output
 *                before the output projection W_O.
 *
 * Long contexts are split across SM pairs and merged by log-sum-exp; the
 * result does not depend on the split beyond fp32 rounding.  Device checks:
 * a bad ctx_len or page id zeroes that sequence's output and sets
 * MLA_CHECK_CTX_LEN / MLA_CHECK_PAGE_ID.
 */
mla_status_t mla_decode(mla_handle_t h, const void* q, const int32_t* ctx_len, int32_t batch,
                        int32_t max_ctx, const int32_t* block_table, int32_t bt_stride,
                        const void* cache, int32_t num_pages, void* workspace,
                        size_t workspace_bytes, void* out, mla_stream_t stream);

/* Size of the scratch array that mla_decode_fixed_scratch uses on each device. */
#define MLA_FIXED_SCRATCH_BYTES (32u << 20)

/*
 * mla_decode_fixed_scratch -- mla_decode without a caller workspace.  The pages
 * describing the method have no counterpart: this is a deployment convenience
 * for callers that cannot allocate device memory at the point of the call.
 *
 * Arguments, output and device checks are those of mla_decode.  The scratch is
 * one array of MLA_FIXED_SCRATCH_BYTES inside the library (one per device);
 * nothing is allocated by the call.
 *
 *   - A batch whose mla_decode_workspace_size exceeds MLA_FIXED_SCRATCH_BYTES
 *     fails with MLA_ERR_WORKSPACE before anything is enqueued (on a 152-SM GB300
 *     up to 25 sequences fit at 128 heads, up to 422 at 16 heads).
 *   - The handle's device must be current (else MLA_ERR_INVALID_ARG).
 *   - Every call writes the scratch before reading it; it never needs clearing.
 *   - All calls on one device share the array, whatever the handle or stream:
 *     calls whose execution overlaps race and corrupt each other's results.
 *     Order them on one stream, or with events.
 *   - The first call in a CUDA context looks the array up (cudaGetSymbolAddress),
 *     which may load the library's module there: make it before any stream
 *     capture begins.  The address is cached with the context it was taken in;
 *     after a device reset, or with another context current, the next call looks
 *     it up again, and that call too must come before any stream capture.
 */
mla_status_t mla_decode_fixed_scratch(mla_handle_t h, const void* q, const int32_t* ctx_len,
                                      int32_t batch, int32_t max_ctx, const int32_t* block_table,
                                      int32_t bt_stride, const void* cache, int32_t num_pages,
                                      void* out, mla_stream_t stream);

/*
 * mla_get_status -- synchronize `stream`, read and clear the device check word.
 * Returns MLA_OK when it was clear, else MLA_ERR_DEVICE_CHECK with the bits in
 * *device_flags (may be NULL) and a message naming them.
 */
mla_status_t mla_get_status(mla_handle_t h, mla_stream_t stream, uint32_t* device_flags);

/* Options for mla_set_option. */
#define MLA_OPT_SPLITS  1   /* value 0: the planner chooses; k > 0: split every sequence into
                               k chunks (capped at its page count).  Used to test that the
                               result does not depend on the split. */
#define MLA_OPT_PROFILE 2   /* value 1: record CUDA events around each kernel mla_decode and
                               mla_prefill launch (which serialises them); mla_profile_read
                               returns the durations. 0: off. */
#define MLA_OPT_TEST_STALL 3 /* test of the bounded in-kernel waits: every later mla_decode
                               withholds one copy, so the thread waiting for it gives up after
                               about a second (of 2e9 clocks), the kernel drains what it has in
                               flight, the step still completes, mla_get_status reports
                               MLA_CHECK_TIMEOUT and that step's output is undefined.
                               value 1: the query-absorb kernel's query copy; 2: one cache tile
                               of the first decode work unit (its first CTA's tile 1); 3: one
                               partial-score copy between the two CTAs of that unit (tile 1, the
                               second CTA's first lane quarter).  For mla_prefill: 4: one weight
                               box of the expansion kernel's first CTA; 5: one key box of the
                               attention kernel (sequence 0, head 0, first query block).  0 (the default): off.  A CUDA
                               graph keeps the value it was captured with. */
#define MLA_OPT_FP8_MMA 4   /* per-tensor FP8 cache (MLA_CACHE_FP8_E4M3): value 1 (the default) runs the decode's
                               contractions on FP8 tensor cores ("G5 MLA KV 访存建模设计规格" use case 1,
                               the FP8 latent cache): QK^T reads the cached e4m3 codes as
                               they are, against the absorbed query quantised to e4m3 with one scale per
                               head (max |q| / 448 over each half of the latent columns; the RoPE part
                               stays bf16), and P . C reads P in e4m3 (P <= 2^8) against a transposed
                               copy of the tile's codes (the default).  Value 0: the codes are
                               converted to bf16 in shared memory and both contractions run in bf16.
                               The two differ by the e4m3 rounding of q and P (within the FP8
                               tolerance of the tests).  No effect on other caches. */
#define MLA_OPT_SMALL_HEADS 5 /* bf16 cache with n_h <= 32: value 1 runs the decode with heads on the
                               MMAs' N dimension, one CTA per work unit ("G5 MLA KV 访存建模设计规格"
                               附录 B's streamed decode; V2-Lite has 16 heads): no partial-score exchange
                               between two CTAs, and the 128-head layout's idle MMA rows are gone.
                               Value 0 (the default): the 128-row layout for every shape.  The
                               results differ by fp32 rounding only.  No effect on other shapes or
                               caches.  A workspace sized by mla_decode_workspace_size serves both. */

mla_status_t mla_set_option(mla_handle_t h, int32_t option, int64_t value);

/*
 * mla_profile_read -- with MLA_OPT_PROFILE on, synchronize and return the
 * device time in milliseconds of each kernel of the last profiled mla_decode
 * (q-absorb + plan, decode, combine + W_UV) or mla_prefill (expansion,
 * attention) call, in launch order.  *count receives the number of kernels; at
 * most `capacity` values are written.  mla_profile_last_name(h, i) names kernel
 * i of that call ("" past the end); mla_profile_kernel_name(i) names the
 * kernels of mla_decode.
 */
mla_status_t mla_profile_read(mla_handle_t h, float* kernel_ms, int32_t capacity, int32_t* count);
const char* mla_profile_kernel_name(int32_t index);
const char* mla_profile_last_name(mla_handle_t h, int32_t index);

/* Thread-local message of this thread's last failed call ("" if none). */
const char* mla_last_error(void);
const char* mla_status_string(mla_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
