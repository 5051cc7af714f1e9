// api.cu -- host side of the libmla.so C ABI (include/mla.h): argument and
// configuration checks, the handle (weights, RoPE table, device check word),
// workspace layout and the launch sequence of a decode step.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "internal.cuh"

namespace {

thread_local std::string g_last_error;

mla_status_t fail(mla_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

mla_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define MLA_CUDA_TRY(expr, what)                         \
  do {                                                   \
    cudaError_t e_ = (expr);                             \
    if (e_ != cudaSuccess) return cuda_fail(e_, what);   \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

const char* kKernelNames[] = {"mla_q_absorb_plan", "mla_decode_splitkv", "mla_combine_uv"};
constexpr int kNumKernels = 3;
const char* kPrefillKernelNames[] = {"mla_prefill_expand", "mla_prefill_attention"};

mla_status_t check_config(const mla_config_t* c) {
  // Mandatory fields: a zero means "not given" and is reported by name.
  struct { const char* name; long v; } ints[] = {
      {"d_c (kv_lora_rank)", c->d_c}, {"d_rope (qk_rope_head_dim)", c->d_rope},
      {"n_h", c->n_h}, {"d_nope", c->d_nope}, {"d_v", c->d_v}, {"page_size", c->page_size},
      {"cache_dtype", c->cache_dtype}, {"max_position", c->max_position}};
  for (auto& f : ints) {
    if (f.v == 0)
      return fail(MLA_ERR_MISSING_FIELD, "mla_config_t.%s is missing (0); every field of mla_config_t is mandatory", f.name);
    if (f.v < 0)
      return fail(MLA_ERR_INVALID_ARG, "mla_config_t.%s = %ld is negative", f.name, f.v);
  }
  if (c->rope_base == 0.0f)
    return fail(MLA_ERR_MISSING_FIELD, "mla_config_t.rope_base is missing (0); every field of mla_config_t is mandatory");
  if (!(c->rope_base > 0.0f) || !std::isfinite(c->rope_base))
    return fail(MLA_ERR_INVALID_ARG, "mla_config_t.rope_base = %g must be positive and finite", c->rope_base);
  if (c->softmax_scale < 0.0f || !std::isfinite(c->softmax_scale))
    return fail(MLA_ERR_INVALID_ARG, "mla_config_t.softmax_scale = %g must be >= 0 (0 selects 1/sqrt(d_nope + d_rope))", c->softmax_scale);
  if (c->cache_dtype != MLA_CACHE_BF16 && c->cache_dtype != MLA_CACHE_FP8_E4M3 &&
      c->cache_dtype != MLA_CACHE_FP8_E4M3_BLOCK)
    return fail(MLA_ERR_INVALID_ARG, "mla_config_t.cache_dtype = %d is not an mla_cache_dtype_t", c->cache_dtype);
  if (c->cache_dtype == MLA_CACHE_FP8_E4M3) {
    if (c->fp8_scale == 0.0f)
      return fail(MLA_ERR_MISSING_FIELD, "mla_config_t.fp8_scale is missing (0); it is mandatory for MLA_CACHE_FP8_E4M3");
    if (!(c->fp8_scale > 0.0f) || !std::isfinite(c->fp8_scale))
      return fail(MLA_ERR_INVALID_ARG, "mla_config_t.fp8_scale = %g must be positive and finite", c->fp8_scale);
  }
  if (c->d_c != mla::kDc || c->d_rope != mla::kDr || c->d_nope != mla::kDn || c->d_v != mla::kDv)
    return fail(MLA_ERR_UNSUPPORTED,
                "shape d_c=%d d_rope=%d d_nope=%d d_v=%d is not built (built: 512 / 64 / 128 / 128)",
                c->d_c, c->d_rope, c->d_nope, c->d_v);
  if (c->n_h > mla::kMaxHeads)
    return fail(MLA_ERR_UNSUPPORTED, "n_h=%d is not built (built: 1..%d)", c->n_h, mla::kMaxHeads);
  if (c->page_size != mla::kPage)
    return fail(MLA_ERR_UNSUPPORTED, "page_size=%d is not built (built: 64)", c->page_size);
  if (c->max_position > mla::kMaxPosition)
    return fail(MLA_ERR_UNSUPPORTED, "max_position=%d exceeds the built limit %d", c->max_position, mla::kMaxPosition);
  return MLA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace mla {

void clear_last_error() { g_last_error.clear(); }

mla_status_t set_last_error(mla_status_t s, const char* msg) {
  g_last_error = msg;
  return s;
}

long long decode_unit_bound(const Handle& h, int batch, int max_ctx) {
  // The planner makes at most sum_b ceil(pages_b / target) <= batch + num_pairs units, or
  // batch * forced splits when the split count is forced; and never more units than a sequence
  // has pages, at most ceil(max_ctx / 64) each.  The decode grid is sized by this bound, so a
  // small step (one short sequence) launches one CTA pair, not one per SM pair.
  const long long by_pages = (long long)batch * ((max_ctx + kPage - 1) / kPage);
  // (a handle whose decode may run one CTA per unit plans a wave of num_sms units: sized for it
  // whatever MLA_OPT_SMALL_HEADS is set to when the workspace is sized)
  const int wave = (h.cfg.n_h <= kShMaxHeads && h.cfg.cache_dtype == MLA_CACHE_BF16) ? h.num_sms : h.num_pairs;
  const long long by_plan = (long long)batch * (h.force_splits > 0 ? h.force_splits : 1) + wave;
  return std::min<long long>(by_plan, std::max<long long>(1, by_pages));
}

size_t workspace_bytes(const Handle& h, int batch, int max_ctx, Workspace* ws, char* base) {
  const int n_h = h.cfg.n_h;
  const int max_units = (int)decode_unit_bound(h, batch, max_ctx);   // callers reject bounds > kMaxUnits
  const int max_parts = max_units;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return base ? base + o : nullptr; };
  char* counters = take(64 * sizeof(int32_t));
  char* units = take(sizeof(Unit) * (size_t)max_units);
  char* seqs = take(sizeof(SeqPlan) * (size_t)batch);
  char* q_abs = take(sizeof(__nv_bfloat16) * (size_t)batch * n_h * kRow);
  char* o_lat = take(sizeof(__nv_bfloat16) * (size_t)batch * n_h * kDc);
  char* part_o = take(sizeof(float) * (size_t)max_parts * n_h * kDc);
  char* part_lse = take(sizeof(float) * (size_t)max_parts * n_h);
  char* bad = take(sizeof(int32_t) * (size_t)batch);
  if (ws) {
    ws->counters = reinterpret_cast<int32_t*>(counters);
    ws->units = reinterpret_cast<Unit*>(units);
    ws->seqs = reinterpret_cast<SeqPlan*>(seqs);
    ws->q_abs = reinterpret_cast<__nv_bfloat16*>(q_abs);
    ws->o_lat = reinterpret_cast<__nv_bfloat16*>(o_lat);
    ws->part_o = reinterpret_cast<float*>(part_o);
    ws->part_lse = reinterpret_cast<float*>(part_lse);
    ws->bad = reinterpret_cast<int32_t*>(bad);
    ws->max_units = max_units;
    ws->max_parts = max_parts;
  }
  return off;
}

}  // namespace mla

using mla::Handle;

extern "C" {

const char* mla_last_error(void) { return g_last_error.c_str(); }

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_MISSING_FIELD: return "MLA_ERR_MISSING_FIELD";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_CHECK: return "MLA_ERR_DEVICE_CHECK";
  }
  return "MLA_ERR_UNKNOWN";
}

const char* mla_profile_kernel_name(int32_t index) {
  return (index >= 0 && index < kNumKernels) ? kKernelNames[index] : "";
}

const char* mla_profile_last_name(mla_handle_t hh, int32_t index) {
  const Handle* h = reinterpret_cast<const Handle*>(hh);
  if (!h || index < 0 || index >= h->n_ev_recorded - 1) return "";
  return h->prof_prefill ? kPrefillKernelNames[index] : kKernelNames[index];
}

mla_status_t mla_create(const mla_config_t* cfg, const void* w_uk, const void* w_uv,
                        mla_stream_t stream, mla_handle_t* out) {
  g_last_error.clear();
  if (!cfg) return fail(MLA_ERR_INVALID_ARG, "mla_create: cfg is NULL");
  if (!out) return fail(MLA_ERR_INVALID_ARG, "mla_create: out is NULL");
  *out = nullptr;
  mla_status_t s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (!w_uk) return fail(MLA_ERR_INVALID_ARG, "mla_create: w_uk is NULL");
  if (!w_uv) return fail(MLA_ERR_INVALID_ARG, "mla_create: w_uv is NULL");

  int dev = 0;
  MLA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  int major = 0, minor = 0, sms = 0;
  MLA_CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute");
  MLA_CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute");
  MLA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(MLA_ERR_UNSUPPORTED, "device %d is sm_%d%d; libmla.so is built for sm_103a only", dev, major, minor);

  Handle* h = new (std::nothrow) Handle();
  if (!h) return fail(MLA_ERR_CUDA, "mla_create: out of host memory");
  h->cfg = *cfg;
  h->scale = cfg->softmax_scale > 0.0f ? cfg->softmax_scale
                                       : (float)(1.0 / std::sqrt((double)(cfg->d_nope + cfg->d_rope)));
  h->device = dev;
  h->num_sms = sms;
  h->num_pairs = sms / 2;
  h->fp8_mma = 1;                           // MLA_OPT_FP8_MMA default
  h->small_heads = 0;                       // MLA_OPT_SMALL_HEADS default
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  auto cleanup = [&](mla_status_t err) { mla_destroy(reinterpret_cast<mla_handle_t>(h)); return err; };
  const size_t wbytes = sizeof(__nv_bfloat16) * (size_t)cfg->n_h * mla::kDn * mla::kDc;
  cudaError_t e;
  if ((e = cudaMalloc(&h->w_uk, wbytes)) != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(w_uk)"));
  if ((e = cudaMalloc(&h->w_uv, wbytes)) != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(w_uv)"));
  if ((e = cudaMalloc(&h->check_word, sizeof(unsigned))) != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(check)"));
  if ((e = cudaMemcpyAsync(h->w_uk, w_uk, wbytes, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
    return cleanup(cuda_fail(e, "copy w_uk"));
  if ((e = cudaMemcpyAsync(h->w_uv, w_uv, wbytes, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
    return cleanup(cuda_fail(e, "copy w_uv"));
  if ((e = cudaMemsetAsync(h->check_word, 0, sizeof(unsigned), st)) != cudaSuccess)
    return cleanup(cuda_fail(e, "clear check word"));

  // RoPE table: angle pos * base^(-2i/d_rope) in float64, cos / sin rounded to fp32.
  const int half = cfg->d_rope / 2;
  const size_t n_cs = (size_t)cfg->max_position * half;
  std::vector<float2> cs(n_cs);
  std::vector<double> inv(half);
  for (int i = 0; i < half; ++i) inv[i] = 1.0 / std::pow((double)cfg->rope_base, (2.0 * i) / cfg->d_rope);
  for (int p = 0; p < cfg->max_position; ++p)
    for (int i = 0; i < half; ++i) {
      const double th = (double)p * inv[i];
      cs[(size_t)p * half + i] = make_float2((float)std::cos(th), (float)std::sin(th));
    }
  if ((e = cudaMalloc(&h->rope_cs, sizeof(float2) * n_cs)) != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(rope)"));
  if ((e = cudaMemcpyAsync(h->rope_cs, cs.data(), sizeof(float2) * n_cs, cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return cleanup(cuda_fail(e, "copy rope table"));
  for (int i = 0; i < 8; ++i)
    if ((e = cudaEventCreate(&h->ev[i])) != cudaSuccess) return cleanup(cuda_fail(e, "cudaEventCreate"));
  if ((e = mla::prepare_weight_maps(*h)) != cudaSuccess) return cleanup(cuda_fail(e, "weight tensor maps"));
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cleanup(cuda_fail(e, "mla_create sync"));
  *out = reinterpret_cast<mla_handle_t>(h);
  return MLA_OK;
}

mla_status_t mla_destroy(mla_handle_t hh) {
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return MLA_OK;
  cudaDeviceSynchronize();
  cudaFree(h->w_uk);
  cudaFree(h->w_uv);
  cudaFree(h->rope_cs);
  cudaFree(h->check_word);
  for (int i = 0; i < 8; ++i)
    if (h->ev[i]) cudaEventDestroy(h->ev[i]);
  delete h;
  return MLA_OK;
}

mla_status_t mla_kv_append(mla_handle_t hh, const void* rows, const int32_t* seq, const int32_t* pos,
                           int32_t n, const int32_t* block_table, int32_t bt_rows, int32_t bt_stride,
                           void* cache, int32_t num_pages, mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_kv_append: handle is NULL");
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "mla_kv_append: n = %d is negative", n);
  if (n == 0) return MLA_OK;
  if (!rows || !seq || !pos || !block_table || !cache)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_append: a device pointer (rows, seq, pos, block_table, cache) is NULL");
  if (bt_rows <= 0 || bt_stride <= 0 || num_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_append: bt_rows=%d bt_stride=%d num_pages=%d must be positive",
                bt_rows, bt_stride, num_pages);
  if (!aligned(rows, 16) || !aligned(cache, 16))
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_append: rows and cache must be 16-byte aligned");
  cudaError_t e = mla::launch_kv_append(*h, static_cast<const __nv_bfloat16*>(rows), seq, pos, n, block_table,
                                        bt_rows, bt_stride, cache, num_pages, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return MLA_OK;
}

mla_status_t mla_kv_project_append(mla_handle_t hh, const void* x, int32_t hidden, const void* w_dkv,
                                   const int32_t* seq, const int32_t* pos, int32_t n, const int32_t* block_table,
                                   int32_t bt_rows, int32_t bt_stride, void* cache, int32_t num_pages,
                                   mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_kv_project_append: handle is NULL");
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "mla_kv_project_append: n = %d is negative", n);
  if (hidden <= 0 || hidden % 256 != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_project_append: hidden = %d must be a positive multiple of 256", hidden);
  if (n == 0) return MLA_OK;
  if (!x || !w_dkv || !seq || !pos || !block_table || !cache)
    return fail(MLA_ERR_INVALID_ARG,
                "mla_kv_project_append: a device pointer (x, w_dkv, seq, pos, block_table, cache) is NULL");
  if (bt_rows <= 0 || bt_stride <= 0 || num_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_project_append: bt_rows=%d bt_stride=%d num_pages=%d must be positive",
                bt_rows, bt_stride, num_pages);
  if (!aligned(x, 16) || !aligned(w_dkv, 16) || !aligned(cache, 16))
    return fail(MLA_ERR_INVALID_ARG, "mla_kv_project_append: x, w_dkv and cache must be 16-byte aligned");
  cudaError_t e = mla::launch_kv_project_append(*h, static_cast<const __nv_bfloat16*>(x), n, hidden,
                                                static_cast<const __nv_bfloat16*>(w_dkv), seq, pos, block_table,
                                                bt_rows, bt_stride, cache, num_pages,
                                                reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_project_append launch");
  return MLA_OK;
}

mla_status_t mla_project(mla_handle_t hh, const void* x, int32_t m, int32_t k, const void* w, int32_t n_out,
                         void* y, mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_project: handle is NULL");
  if (m < 0) return fail(MLA_ERR_INVALID_ARG, "mla_project: m = %d is negative", m);
  if (k <= 0 || k % 256 != 0) return fail(MLA_ERR_INVALID_ARG, "mla_project: k = %d must be a positive multiple of 256", k);
  if (n_out <= 0 || n_out % 16 != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_project: n_out = %d must be a positive multiple of 16", n_out);
  if (m == 0) return MLA_OK;
  if (!x || !w || !y) return fail(MLA_ERR_INVALID_ARG, "mla_project: a device pointer (x, w, y) is NULL");
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 4))
    return fail(MLA_ERR_INVALID_ARG, "mla_project: x and w must be 16-byte aligned, y 4-byte aligned");
  cudaError_t e = mla::launch_project(static_cast<const __nv_bfloat16*>(x), m, k, static_cast<const __nv_bfloat16*>(w),
                                      n_out, static_cast<__nv_bfloat16*>(y), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "project launch");
  return MLA_OK;
}

mla_status_t mla_rmsnorm(mla_handle_t hh, const void* x, int32_t m, int32_t n, int32_t ld_x, const void* w, float eps,
                         void* y, int32_t ld_y, mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_rmsnorm: handle is NULL");
  if (m < 0) return fail(MLA_ERR_INVALID_ARG, "mla_rmsnorm: m = %d is negative", m);
  if (n <= 0 || n % 8 != 0 || n > 8192)
    return fail(MLA_ERR_INVALID_ARG, "mla_rmsnorm: n = %d must be a positive multiple of 8, at most 8192", n);
  if (ld_x < n || ld_y < n || ld_x % 8 != 0 || ld_y % 8 != 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_rmsnorm: ld_x = %d and ld_y = %d must be multiples of 8, at least n = %d",
                ld_x, ld_y, n);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(MLA_ERR_INVALID_ARG, "mla_rmsnorm: eps = %g must be >= 0", eps);
  if (m == 0) return MLA_OK;
  if (!x || !w || !y) return fail(MLA_ERR_INVALID_ARG, "mla_rmsnorm: x, w or y is NULL");
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16))
    return fail(MLA_ERR_INVALID_ARG, "mla_rmsnorm: x, w and y must be 16-byte aligned");
  cudaError_t e = mla::launch_rmsnorm(static_cast<const __nv_bfloat16*>(x), m, n, ld_x,
                                      static_cast<const __nv_bfloat16*>(w), eps, static_cast<__nv_bfloat16*>(y), ld_y,
                                      reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm launch");
  return MLA_OK;
}

mla_status_t mla_expand_kv(mla_handle_t hh, const void* cache, int32_t num_pages, void* kvx, mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_expand_kv: handle is NULL");
  if (h->cfg.cache_dtype != MLA_CACHE_BF16)
    return fail(MLA_ERR_UNSUPPORTED, "mla_expand_kv: only a bf16 cache can be expanded");
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_expand_kv: num_pages = %d must be positive", num_pages);
  if (!cache || !kvx) return fail(MLA_ERR_INVALID_ARG, "mla_expand_kv: cache or kvx is NULL");
  if (!aligned(cache, 16) || !aligned(kvx, 16))
    return fail(MLA_ERR_INVALID_ARG, "mla_expand_kv: cache and kvx must be 16-byte aligned");
  cudaError_t e = mla::launch_expand_kv(*h, cache, num_pages, kvx, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "expand_kv launch");
  return MLA_OK;
}

mla_status_t mla_decode_naive_workspace_size(mla_handle_t hh, int32_t batch, int32_t max_ctx, size_t* bytes) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive_workspace_size: handle is NULL");
  if (!bytes) return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive_workspace_size: bytes is NULL");
  if (batch <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive_workspace_size: batch = %d must be positive", batch);
  if (max_ctx <= 0 || max_ctx > h->cfg.max_position)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive_workspace_size: max_ctx = %d must be in [1, max_position=%d]",
                max_ctx, h->cfg.max_position);
  *bytes = mla::naive_workspace_bytes(h->cfg.n_h, batch, max_ctx);
  return MLA_OK;
}

mla_status_t mla_decode_naive(mla_handle_t hh, const void* q, const int32_t* ctx_len, int32_t batch, int32_t max_ctx,
                              const int32_t* block_table, int32_t bt_stride, const void* kvx, int32_t num_pages,
                              void* workspace, size_t workspace_bytes, void* out, mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive: handle is NULL");
  if (batch <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive: batch = %d must be positive", batch);
  if (max_ctx <= 0 || max_ctx > h->cfg.max_position)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive: max_ctx = %d must be in [1, max_position=%d]", max_ctx,
                h->cfg.max_position);
  if (!q || !ctx_len || !block_table || !kvx || !workspace || !out)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive: a device pointer is NULL");
  const int need_pages = (max_ctx + mla::kPage - 1) / mla::kPage;
  if (bt_stride < need_pages)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive: bt_stride = %d holds fewer than the %d pages of max_ctx = %d",
                bt_stride, need_pages, max_ctx);
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive: num_pages = %d must be positive", num_pages);
  if (!aligned(q, 16) || !aligned(kvx, 16) || !aligned(out, 16))
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_naive: q, kvx and out must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(MLA_ERR_WORKSPACE, "mla_decode_naive: workspace must be 256-byte aligned");
  const size_t need = mla::naive_workspace_bytes(h->cfg.n_h, batch, max_ctx);
  if (workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE, "mla_decode_naive: workspace has %zu bytes, %zu needed", workspace_bytes, need);
  cudaError_t e = mla::launch_decode_naive(*h, q, ctx_len, batch, max_ctx, block_table, bt_stride, kvx, num_pages,
                                           workspace, out, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode_naive launch");
  return MLA_OK;
}

mla_status_t mla_prefill_workspace_size(mla_handle_t hh, int32_t batch, int32_t max_ctx, size_t* bytes) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_prefill_workspace_size: handle is NULL");
  if (!bytes) return fail(MLA_ERR_INVALID_ARG, "mla_prefill_workspace_size: bytes is NULL");
  if (batch <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_prefill_workspace_size: batch = %d must be positive", batch);
  if (max_ctx <= 0 || max_ctx > h->cfg.max_position)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill_workspace_size: max_ctx = %d must be in [1, max_position=%d]",
                max_ctx, h->cfg.max_position);
  *bytes = mla::prefill_workspace_bytes(h->cfg.n_h, batch, max_ctx);
  return MLA_OK;
}

mla_status_t mla_prefill(mla_handle_t hh, const void* q, const int32_t* q_start, const int32_t* q_len, int32_t total_q,
                         int32_t max_q, const int32_t* ctx_len, int32_t batch, int32_t max_ctx,
                         const int32_t* block_table, int32_t bt_stride, const void* cache, int32_t num_pages,
                         void* workspace, size_t workspace_bytes, void* out, mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: handle is NULL");
  if (batch <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: batch = %d must be positive", batch);
  if (max_ctx <= 0 || max_ctx > h->cfg.max_position)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: max_ctx = %d must be in [1, max_position=%d]", max_ctx,
                h->cfg.max_position);
  if (max_q <= 0 || max_q > max_ctx)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: max_q = %d must be in [1, max_ctx=%d]", max_q, max_ctx);
  if (total_q <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: total_q = %d must be positive", total_q);
  if (!q || !q_start || !q_len || !ctx_len || !block_table || !cache || !workspace || !out)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: a device pointer is NULL");
  const int need_pages = (max_ctx + mla::kPage - 1) / mla::kPage;
  if (bt_stride < need_pages)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: bt_stride = %d holds fewer than the %d pages of max_ctx = %d",
                bt_stride, need_pages, max_ctx);
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: num_pages = %d must be positive", num_pages);
  const long long rows = (long long)batch * h->cfg.n_h * ((max_ctx + 127) / 128 * 128);
  if (rows >= (1LL << 31))
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: batch x n_h x max_ctx = %lld expanded rows exceed 2^31", rows);
  if (!aligned(q, 16) || !aligned(cache, 128) || !aligned(out, 32))
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: q must be 16-byte aligned, out 32-byte, cache 128-byte");
  if (!aligned(workspace, 256)) return fail(MLA_ERR_WORKSPACE, "mla_prefill: workspace must be 256-byte aligned");
  const size_t need = mla::prefill_workspace_bytes(h->cfg.n_h, batch, max_ctx);
  if (workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE, "mla_prefill: workspace has %zu bytes, %zu needed", workspace_bytes, need);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool prof = h->profile != 0;
  if (prof) cudaEventRecord(h->ev[0], st);
  cudaError_t e = mla::launch_prefill(*h, q, q_start, q_len, total_q, max_q, ctx_len, batch, max_ctx, block_table,
                                      bt_stride, cache, num_pages, workspace, out, st, prof ? h->ev[1] : nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  if (prof) {
    cudaEventRecord(h->ev[2], st);
    h->n_ev_recorded = 3;
    h->prof_prefill = 1;
  }
  return MLA_OK;
}

mla_status_t mla_decode_workspace_size(mla_handle_t hh, int32_t batch, int32_t max_ctx, size_t* bytes) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_decode_workspace_size: handle is NULL");
  if (!bytes) return fail(MLA_ERR_INVALID_ARG, "mla_decode_workspace_size: bytes is NULL");
  if (batch <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode_workspace_size: batch = %d must be positive", batch);
  if (max_ctx <= 0 || max_ctx > h->cfg.max_position)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_workspace_size: max_ctx = %d must be in [1, max_position=%d]",
                max_ctx, h->cfg.max_position);
  if (mla::decode_unit_bound(*h, batch, max_ctx) > mla::kMaxUnits)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode_workspace_size: batch = %d with the split option gives more than %d work units",
                batch, mla::kMaxUnits);
  *bytes = mla::workspace_bytes(*h, batch, max_ctx, nullptr, nullptr);
  return MLA_OK;
}

mla_status_t mla_decode(mla_handle_t hh, const void* q, const int32_t* ctx_len, int32_t batch,
                        int32_t max_ctx, const int32_t* block_table, int32_t bt_stride,
                        const void* cache, int32_t num_pages, void* workspace, size_t workspace_bytes,
                        void* out, mla_stream_t stream) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_decode: handle is NULL");
  if (!q || !ctx_len || !block_table || !cache || !out)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: a device pointer (q, ctx_len, block_table, cache, out) is NULL");
  if (batch <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode: batch = %d must be positive", batch);
  if (max_ctx <= 0 || max_ctx > h->cfg.max_position)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: max_ctx = %d must be in [1, max_position=%d]", max_ctx,
                h->cfg.max_position);
  const int need_pages = (max_ctx + mla::kPage - 1) / mla::kPage;
  if (bt_stride < need_pages)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: bt_stride = %d < %d pages needed for max_ctx = %d", bt_stride,
                need_pages, max_ctx);
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode: num_pages = %d must be positive", num_pages);
  if (!aligned(q, 16) || !aligned(cache, 128) || !aligned(out, 16))
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: q and out must be 16-byte aligned, cache 128-byte aligned");
  if (!workspace) return fail(MLA_ERR_WORKSPACE, "mla_decode: workspace is NULL");
  if (!aligned(workspace, 256)) return fail(MLA_ERR_WORKSPACE, "mla_decode: workspace must be 256-byte aligned");
  if (mla::decode_unit_bound(*h, batch, max_ctx) > mla::kMaxUnits)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: batch = %d with the split option gives more than %d work units", batch,
                mla::kMaxUnits);
  mla::Workspace ws;
  const size_t need = mla::workspace_bytes(*h, batch, max_ctx, &ws, static_cast<char*>(workspace));
  if (workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE, "mla_decode: workspace has %zu bytes, %zu needed", workspace_bytes, need);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool prof = h->profile != 0;
  int ev = 0;
  auto mark = [&]() { if (prof) cudaEventRecord(h->ev[ev++], st); };
  cudaError_t e;
  // Kernel order: query absorption (with the split planner in one extra CTA), the split-KV
  // decode, then the merge + value up-projection.
  mark();
  if ((e = mla::launch_q_absorb(*h, static_cast<const __nv_bfloat16*>(q), ctx_len, batch, max_ctx, ws, st)) !=
      cudaSuccess)
    return cuda_fail(e, "q_absorb launch");
  mark();
  e = mla::small_head_decode(*h)
          ? mla::launch_decode_small_heads(*h, ctx_len, batch, block_table, bt_stride, cache, num_pages, ws, st)
          : mla::launch_decode(*h, ctx_len, batch, block_table, bt_stride, cache, num_pages, ws, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  mark();
  if ((e = mla::launch_combine_uv(*h, batch, ws, static_cast<__nv_bfloat16*>(out), st)) != cudaSuccess)
    return cuda_fail(e, "combine_uv launch");
  mark();
  h->n_ev_recorded = ev;
  h->prof_prefill = 0;
  return MLA_OK;
}

mla_status_t mla_get_status(mla_handle_t hh, mla_stream_t stream, uint32_t* device_flags) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_get_status: handle is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned word = 0;
  MLA_CUDA_TRY(cudaStreamSynchronize(st), "mla_get_status sync");
  MLA_CUDA_TRY(cudaMemcpy(&word, h->check_word, sizeof(unsigned), cudaMemcpyDeviceToHost), "read check word");
  MLA_CUDA_TRY(cudaMemset(h->check_word, 0, sizeof(unsigned)), "clear check word");
  if (device_flags) *device_flags = word;
  if (word == 0) return MLA_OK;
  std::string msg = "device check failed:";
  if (word & MLA_CHECK_CTX_LEN) msg += " ctx_len out of [1, max_ctx];";
  if (word & MLA_CHECK_PAGE_ID) msg += " page id out of [0, num_pages);";
  if (word & MLA_CHECK_APPEND_INDEX) msg += " append seq/pos out of range;";
  if (word & MLA_CHECK_TIMEOUT) msg += " a bounded in-kernel wait ran out;";
  return fail(MLA_ERR_DEVICE_CHECK, "%s", msg.c_str());
}

mla_status_t mla_set_option(mla_handle_t hh, int32_t option, int64_t value) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_set_option: handle is NULL");
  switch (option) {
    case MLA_OPT_SPLITS:
      if (value < 0 || value > 4096) return fail(MLA_ERR_INVALID_ARG, "MLA_OPT_SPLITS = %lld out of [0, 4096]", (long long)value);
      h->force_splits = (int)value;
      return MLA_OK;
    case MLA_OPT_PROFILE:
      h->profile = value != 0;
      h->n_ev_recorded = 0;
      return MLA_OK;
    case MLA_OPT_TEST_STALL:
      if (value < 0 || value > 5) return fail(MLA_ERR_INVALID_ARG, "MLA_OPT_TEST_STALL = %lld is not in 0..5", (long long)value);
      h->test_stall = (int)value;
      return MLA_OK;
    case MLA_OPT_FP8_MMA:
      if (value < 0 || value > 1) return fail(MLA_ERR_INVALID_ARG, "MLA_OPT_FP8_MMA = %lld is not 0 or 1", (long long)value);
      h->fp8_mma = (int)value;
      return MLA_OK;
    case MLA_OPT_SMALL_HEADS:
      if (value < 0 || value > 1)
        return fail(MLA_ERR_INVALID_ARG, "MLA_OPT_SMALL_HEADS = %lld is not 0 or 1", (long long)value);
      h->small_heads = (int)value;
      return MLA_OK;
  }
  return fail(MLA_ERR_INVALID_ARG, "mla_set_option: unknown option %d", option);
}

mla_status_t mla_profile_read(mla_handle_t hh, float* kernel_ms, int32_t capacity, int32_t* count) {
  g_last_error.clear();
  Handle* h = reinterpret_cast<Handle*>(hh);
  if (!h) return fail(MLA_ERR_INVALID_ARG, "mla_profile_read: handle is NULL");
  if (!count) return fail(MLA_ERR_INVALID_ARG, "mla_profile_read: count is NULL");
  *count = 0;
  if (!h->profile || h->n_ev_recorded < 2) return MLA_OK;
  const int n = h->n_ev_recorded - 1;
  MLA_CUDA_TRY(cudaEventSynchronize(h->ev[n]), "mla_profile_read sync");
  for (int i = 0; i < n && i < capacity && kernel_ms; ++i) {
    float ms = 0.0f;
    MLA_CUDA_TRY(cudaEventElapsedTime(&ms, h->ev[i], h->ev[i + 1]), "cudaEventElapsedTime");
    kernel_ms[i] = ms;
  }
  *count = n;
  return MLA_OK;
}

}  // extern "C"
