// internal.cuh -- types shared by the host API and the kernels of libmla.so.
//
// Shapes built: d_c = 512, d_rope = 64, d_nope = d_v = 128, page = 64 tokens,
// 1 <= n_h <= 128.  A cache row is [c (512) | k_r (64)] = 576 values.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/mla.h"

namespace mla {

constexpr int kDc = 512;          // KV latent width
constexpr int kDr = 64;           // RoPE key width
constexpr int kRow = kDc + kDr;   // 576 values per cached token
constexpr int kDn = 128;          // no-RoPE query width per head
constexpr int kDq = kDn + kDr;    // 192 query values per head
constexpr int kDv = 128;          // value width per head
constexpr int kPage = 64;         // tokens per page
constexpr int kMaxHeads = 128;    // heads padded to one 128-row MMA tile
constexpr int kMaxPosition = 1 << 20;

// One unit of decode work: tokens [page_begin * 64, min(page_end * 64, ctx_len)) of sequence b.
struct Unit {
  int32_t b;
  int32_t page_begin;
  int32_t page_end;
  int32_t part;        // index of this unit's partial slot, or -1 when the unit is the whole sequence
};

// Per-sequence plan entry.
struct SeqPlan {
  int32_t first_unit;  // first unit of the sequence (units of a sequence are consecutive)
  int32_t nsplit;      // 0: invalid sequence (output zeroed), 1: unsplit, >1: split
};
static_assert(sizeof(SeqPlan) == 8, "plan entries are read as int2");

// Device-side views of the workspace (all regions 256-byte aligned).
struct Workspace {
  int32_t* counters;        // [0] = number of units, [1] = number of partial slots
  Unit* units;              // [max_units]
  SeqPlan* seqs;            // [B]
  __nv_bfloat16* q_abs;     // [B][n_h][576]: absorbed query (latent 512 | rotated rope 64)
  __nv_bfloat16* o_lat;     // [B][n_h][512]: normalised latent sum of unsplit sequences
  float* part_o;            // [max_parts][n_h][512]: normalised partial latent sums
  float* part_lse;          // [max_parts][n_h]: natural-log normaliser of each partial
  int32_t* bad;             // [B]: set by the decode kernel when a page id is out of range
  int max_units;
  int max_parts;
};

struct Handle {
  mla_config_t cfg;
  float scale;              // softmax scale actually used
  int device;
  int num_sms;
  int num_pairs;            // SM pairs available to the decode kernel
  __nv_bfloat16* w_uk;      // [n_h][d_nope][d_c] (as given)
  __nv_bfloat16* w_uv;      // [n_h][d_v][d_c]   (as given)
  float2* rope_cs;          // [max_position][d_rope / 2] (cos, sin) fp32 from float64 angles
  unsigned* check_word;     // device check word
  int force_splits;         // MLA_OPT_SPLITS
  int profile;              // MLA_OPT_PROFILE
  int test_stall;           // MLA_OPT_TEST_STALL
  int fp8_mma;              // MLA_OPT_FP8_MMA
  int small_heads;          // MLA_OPT_SMALL_HEADS
  cudaEvent_t ev[8];
  int n_ev_recorded;
  int prof_prefill;         // the last profiled call was mla_prefill (else mla_decode)
  alignas(64) unsigned char tmap[128];   // TMA descriptor (CUtensorMap) of the last cache seen
  alignas(64) unsigned char tmap_rope[128];  // same cache, RoPE-key columns (32-column boxes)
  alignas(64) unsigned char tmap_scale[128]; // per-block FP8 cache: the rows' scale bytes
  alignas(64) unsigned char tmap8[128];      // per-tensor FP8 cache: 128-code boxes, 128-byte swizzle (FP8 MMAs)
  alignas(64) unsigned char tmap_wuk[128];  // TMA descriptors of the handle's weight copies
  alignas(64) unsigned char tmap_wuv[128];
  const void* tmap_cache;
  int tmap_pages;
};

// TMA descriptors of the weights (built once in mla_create).
cudaError_t prepare_weight_maps(Handle& h);
// TMA descriptors of a cache in h.tmap / h.tmap_rope (64- and 32-column boxes of one page).
cudaError_t cache_maps(const Handle& h, const void* cache, int num_pages);

// Workspace sizing and carving (host).  The unit bound sizes the decode grid (two CTAs a unit).
constexpr long long kMaxUnits = 1LL << 28;
long long decode_unit_bound(const Handle& h, int batch, int max_ctx);
size_t workspace_bytes(const Handle& h, int batch, int max_ctx, Workspace* carve, char* base);

// The calling thread's message for mla_last_error (kept in api.cu).
void clear_last_error();
mla_status_t set_last_error(mla_status_t s, const char* msg);

// Kernel launchers (each returns the launch error).
// Standard-mode (expanded) decode: the per-head key/value cache and its decode.
size_t naive_workspace_bytes(int n_h, int batch, int max_ctx);
cudaError_t launch_expand_kv(const Handle& h, const void* cache, int num_pages, void* kvx, cudaStream_t st);
cudaError_t launch_decode_naive(const Handle& h, const void* q, const int32_t* ctx_len, int batch, int max_ctx,
                                const int32_t* block_table, int bt_stride, const void* kvx, int num_pages,
                                void* workspace, void* out, cudaStream_t st);
// Causal prefill in MHA mode: per-head expansion of the cached rows, then attention.
size_t prefill_workspace_bytes(int n_h, int batch, int max_ctx);
cudaError_t launch_prefill(const Handle& h, const void* q, const int32_t* q_start, const int32_t* q_len, int total_q,
                           int max_q, const int32_t* ctx_len, int batch, int max_ctx, const int32_t* block_table,
                           int bt_stride, const void* cache, int num_pages, void* workspace, void* out,
                           cudaStream_t st, cudaEvent_t between = nullptr);
// RMSNorm of m strided rows of n values (n a multiple of 8); y may be x.
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, int m, int n, int ld_x, const __nv_bfloat16* w, float eps,
                           __nv_bfloat16* y, int ld_y, cudaStream_t st);
// y[m][n_out] = bf16(x[m][k] . w[n_out][k]^T); k a multiple of 256, n_out of 16.
cudaError_t launch_project(const __nv_bfloat16* x, int m, int k, const __nv_bfloat16* w, int n_out,
                           __nv_bfloat16* y, cudaStream_t st);
// rows = x[n][k] . w_dkv[576][k]^T written into the paged cache as mla_kv_append writes rows.
cudaError_t launch_kv_project_append(const Handle& h, const __nv_bfloat16* x, int n, int k,
                                     const __nv_bfloat16* w, const int32_t* seq, const int32_t* pos,
                                     const int32_t* block_table, int bt_rows, int bt_stride, void* cache,
                                     int num_pages, cudaStream_t st);
cudaError_t launch_kv_append(const Handle& h, const __nv_bfloat16* rows, const int32_t* seq,
                             const int32_t* pos, int n, const int32_t* block_table, int bt_rows,
                             int bt_stride, void* cache, int num_pages, cudaStream_t st);
// Query absorption; one extra CTA of the same launch runs the split planner.
cudaError_t launch_q_absorb(const Handle& h, const __nv_bfloat16* q, const int32_t* ctx_len,
                            int batch, int max_ctx, const Workspace& ws, cudaStream_t st);
// The decode for few heads (decode_sh.cu): a bf16 cache and n_h <= kShMaxHeads, one CTA per
// work unit (so the planner's one wave is num_sms units, not num_pairs).
constexpr int kShMaxHeads = 32;
bool small_head_decode(const Handle& h);
inline int decode_wave(const Handle& h) { return small_head_decode(h) ? h.num_sms : h.num_pairs; }
cudaError_t launch_decode_small_heads(const Handle& h, const int32_t* ctx_len, int batch, const int32_t* block_table,
                                      int bt_stride, const void* cache, int num_pages, const Workspace& ws,
                                      cudaStream_t st);
cudaError_t launch_decode(const Handle& h, const int32_t* ctx_len, int batch,
                          const int32_t* block_table, int bt_stride, const void* cache,
                          int num_pages, const Workspace& ws, cudaStream_t st);
cudaError_t launch_combine_uv(const Handle& h, int batch, const Workspace& ws,
                              __nv_bfloat16* out, cudaStream_t st);

// Launch a kernel as a programmatic dependent of the previous work in the stream: it may
// be scheduled while that work finishes and must call griddep_wait() before touching
// anything it produced.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device check word bits (same values as the public MLA_CHECK_* macros).
constexpr unsigned kCheckCtxLen = MLA_CHECK_CTX_LEN;
constexpr unsigned kCheckPageId = MLA_CHECK_PAGE_ID;
constexpr unsigned kCheckAppend = MLA_CHECK_APPEND_INDEX;
constexpr unsigned kCheckTimeout = MLA_CHECK_TIMEOUT;

}  // namespace mla
