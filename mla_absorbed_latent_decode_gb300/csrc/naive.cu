// naive.cu -- standard-mode (expanded) MLA decode, the comparison the absorbed path is measured
// against ("80 行 PyTorch 从零写 DeepSeek 的 MLA" §3/§5: the naive mode caches per-head keys and
// values; "G5 MLA KV 访存建模设计规格": KV bytes read per token, absorbed vs standard).
//
//   expand:  for every cached token and head h, key_h = [W_UK[h] c ; k_r] (d_nope + d_rope) and
//            value_h = W_UV[h] c (d_v), rounded to bf16 -- what a standard MHA cache holds for
//            MLA (the RoPE key is shared by the heads and stored once per head);
//   decode:  per sequence and head, o_h = sum_t softmax_t(q_h . key_h,t * scale) value_h,t with
//            q_h = [q_nope ; RoPE(q_pe, ctx_len - 1)], no absorption and no up-projection.
//
// Expanded page layout: [page][64 slots][n_h][d_nope + d_rope + d_v] bf16 (640 B per token and
// head).  The decode streams it (HBM-bound, a GEMV per head): a CTA takes 16 heads of one
// sequence over one 256-token split, warp = head; a lane holds 6 of the 192 query values and
// 4 of the 128 output values, and loads the rows of 8 tokens before it uses any of them.
// Splits are merged by log-sum-exp (a standard identity).
#include "append_ops.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

constexpr int kKx = kDn + kDr;              // 192 key values per head
constexpr int kXRow = kKx + kDv;            // 320 values per (token, head)
constexpr int kNaiveSplit = 256;            // tokens per CTA
constexpr int kNaiveHeads = 16;             // heads (warps) per CTA
constexpr int kNaiveGroup = 8;              // tokens whose rows a warp loads together
constexpr int kSplitF = kDv + 4;            // floats per split record: m, l, 2 unused, o[128] (16-byte aligned)
constexpr int kExpandSmem = kDc * kPage * 2;   // the page's latent rows, transposed (64 KB)

// ---- expansion: CTA = (page, head); thread = (token t = tid % 64, rows r = tid / 64 + 4 i)
__global__ void __launch_bounds__(256) expand_kernel(const __nv_bfloat16* __restrict__ cache, int n_h,
                                                    const __nv_bfloat16* __restrict__ w_uk,
                                                    const __nv_bfloat16* __restrict__ w_uv,
                                                    __nv_bfloat16* __restrict__ kvx) {
  extern __shared__ __nv_bfloat16 ct_raw[];  // latent rows of the page, transposed: ct[j][t]
  __nv_bfloat16 (*ct)[kPage] = reinterpret_cast<__nv_bfloat16 (*)[kPage]>(ct_raw);
  const int page = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const __nv_bfloat16* rows = cache + (size_t)page * kPage * kRow;
  for (int i = tid; i < kPage * (kDc / 8); i += blockDim.x) {    // 8 values of row t per thread
    const int t = i % kPage, j8 = i / kPage;
    const uint4 v = *reinterpret_cast<const uint4*>(rows + (size_t)t * kRow + 8 * j8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ct[8 * j8 + 2 * e][t] = __float2bfloat16_rn(bf16_lo(w[e]));
      ct[8 * j8 + 2 * e + 1][t] = __float2bfloat16_rn(bf16_hi(w[e]));
    }
  }
  __syncthreads();
  const int t = tid % kPage;
  __nv_bfloat16* out = kvx + (((size_t)page * kPage + t) * n_h + h) * kXRow;
  for (int r = tid / kPage; r < kDn + kDv; r += 4) {
    const __nv_bfloat16* w = r < kDn ? w_uk + ((size_t)h * kDn + r) * kDc : w_uv + ((size_t)h * kDv + (r - kDn)) * kDc;
    float acc = 0.0f;
    for (int j = 0; j < kDc; j += 8) {
      const uint4 wv = *reinterpret_cast<const uint4*>(w + j);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(bf16_lo(ww[e]), __bfloat162float(ct[j + 2 * e][t]), acc);
        acc = fmaf(bf16_hi(ww[e]), __bfloat162float(ct[j + 2 * e + 1][t]), acc);
      }
    }
    out[r < kDn ? r : kKx + (r - kDn)] = __float2bfloat16_rn(acc);
  }
  if (tid < kPage) {                         // the RoPE key as cached (already rotated)
    const __nv_bfloat16* kr = rows + (size_t)t * kRow + kDc;
    for (int i = 0; i < kDr; ++i) out[kDn + i] = kr[i];
  }
}

// ---- decode: CTA = (split, head group, sequence); warp = head
__global__ void __launch_bounds__(kNaiveHeads * 32) naive_decode_kernel(
    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ ctx_len, int n_h, int max_ctx,
    const int32_t* __restrict__ block_table, int bt_stride, const __nv_bfloat16* __restrict__ kvx, int num_pages,
    const float2* __restrict__ rope_cs, int max_position, float scale_log2, int max_splits,
    float* __restrict__ part, __nv_bfloat16* __restrict__ out, unsigned* check) {
  const int split = blockIdx.x, b = blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kNaiveHeads + warp;
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  if (h >= n_h) return;
  const int L = ctx_len[b];
  const bool valid_len = L >= 1 && L <= max_ctx;
  const int nsplit = valid_len ? (L + kNaiveSplit - 1) / kNaiveSplit : 1;
  if (split >= nsplit) return;
  float* slot = part + (((size_t)b * n_h + h) * max_splits + split) * kSplitF;
  float o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float m = -INFINITY, l = 0.0f;
  bool bad = !valid_len;
  if (valid_len) {
    // query: lane holds values 6 lane .. 6 lane + 5; the RoPE part (values 128..191) rotated at L - 1
    const __nv_bfloat16* qh = q + ((size_t)b * n_h + h) * kKx;
    float qv[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) qv[i] = __bfloat162float(qh[6 * lane + i]);
    {
      const int pos = min(L - 1, max_position - 1);
#pragma unroll
      for (int i = 0; i < 6; i += 2) {        // pairs never straddle lanes: 6 lane and 128 are even
        const int idx = 6 * lane + i;
        if (idx >= kDn) rope_pair(qv[i], qv[i + 1], rope_cs[(size_t)pos * (kDr / 2) + (idx - kDn) / 2], &qv[i], &qv[i + 1]);
      }
    }
    // kNaiveGroup tokens per iteration: their rows are loaded before any of them is used, so a
    // warp keeps kNaiveGroup row reads in flight; a group never crosses a page (64 % 8 == 0 and
    // every split starts on a page boundary)
    const int t0 = split * kNaiveSplit, t1 = min(L, t0 + kNaiveSplit);
    for (int t = t0; t < t1 && !bad; t += kNaiveGroup) {
      const int n = min(kNaiveGroup, t1 - t);
      const int page = block_table[(size_t)b * bt_stride + t / kPage];
      if (page < 0 || page >= num_pages) { bad = true; break; }
      const __nv_bfloat16* row0 = kvx + (((size_t)page * kPage + t % kPage) * n_h + h) * kXRow;
      uint32_t kw[kNaiveGroup][3];
      uint2 vv[kNaiveGroup];
#pragma unroll
      for (int u = 0; u < kNaiveGroup; ++u) {
        if (u < n) {
          const __nv_bfloat16* row = row0 + (size_t)u * n_h * kXRow;
          const uint32_t* kp = reinterpret_cast<const uint32_t*>(row + 6 * lane);
          kw[u][0] = kp[0];
          kw[u][1] = kp[1];
          kw[u][2] = kp[2];
          vv[u] = *reinterpret_cast<const uint2*>(row + kKx + 4 * lane);
        } else {
          kw[u][0] = kw[u][1] = kw[u][2] = 0u;
          vv[u] = make_uint2(0u, 0u);
        }
      }
      float s[kNaiveGroup];
#pragma unroll
      for (int u = 0; u < kNaiveGroup; ++u) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          a = fmaf(qv[2 * i], bf16_lo(kw[u][i]), a);
          a = fmaf(qv[2 * i + 1], bf16_hi(kw[u][i]), a);
        }
        s[u] = a;
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
#pragma unroll
        for (int u = 0; u < kNaiveGroup; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
      }
      float m_new = m;
#pragma unroll
      for (int u = 0; u < kNaiveGroup; ++u) {
        s[u] = u < n ? s[u] * scale_log2 : -INFINITY;
        m_new = fmaxf(m_new, s[u]);
      }
      const float alpha = exp2f(m - m_new);
      l *= alpha;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] *= alpha;
#pragma unroll
      for (int u = 0; u < kNaiveGroup; ++u) {
        const float p = exp2f(s[u] - m_new);
        l += p;
        o[0] = fmaf(p, bf16_lo(vv[u].x), o[0]);
        o[1] = fmaf(p, bf16_hi(vv[u].x), o[1]);
        o[2] = fmaf(p, bf16_lo(vv[u].y), o[2]);
        o[3] = fmaf(p, bf16_hi(vv[u].y), o[3]);
      }
      m = m_new;
    }
  }
  if (bad) {
    if (lane == 0) atomicOr(check, valid_len ? kCheckPageId : kCheckCtxLen);
    m = -INFINITY;
    l = 0.0f;
    o[0] = o[1] = o[2] = o[3] = 0.0f;
  }
  if (nsplit == 1) {                         // the whole sequence: normalise and write
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    uint2* dst = reinterpret_cast<uint2*>(out + ((size_t)b * n_h + h) * kDv + 4 * lane);
    *dst = make_uint2(pack_bf16(o[0] * inv, o[1] * inv), pack_bf16(o[2] * inv, o[3] * inv));
  } else {
    if (lane == 0) {
      slot[0] = m;
      slot[1] = bad ? -1.0f : l;             // a negative sum marks a sequence to zero
    }
    *reinterpret_cast<float4*>(slot + 4 + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
  }
}

// ---- merge of the splits of a sequence (log-sum-exp): CTA = sequence, warp = head
__global__ void __launch_bounds__(256) naive_merge_kernel(const int32_t* __restrict__ ctx_len, int n_h, int max_ctx,
                                                          int max_splits, const float* __restrict__ part,
                                                          __nv_bfloat16* __restrict__ out) {
  const int b = blockIdx.x, lane = threadIdx.x & 31;
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  const int L = ctx_len[b];
  if (L < 1 || L > max_ctx) return;
  const int nsplit = (L + kNaiveSplit - 1) / kNaiveSplit;
  if (nsplit == 1) return;
  for (int h = threadIdx.x >> 5; h < n_h; h += blockDim.x >> 5) {
    const float* base = part + ((size_t)b * n_h + h) * max_splits * kSplitF;
    float mx = -INFINITY;
    bool bad = false;
    for (int k = 0; k < nsplit; ++k) {
      mx = fmaxf(mx, base[k * kSplitF]);
      bad = bad || base[k * kSplitF + 1] < 0.0f;
    }
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, den = 0.0f;
    for (int k = 0; k < nsplit && !bad; ++k) {
      const float* sl = base + k * kSplitF;
      const float w = exp2f(sl[0] - mx);
      den = fmaf(w, sl[1], den);
      const float4 v = *reinterpret_cast<const float4*>(sl + 4 + 4 * lane);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    }
    const float inv = (!bad && den > 0.0f) ? 1.0f / den : 0.0f;
    uint2* dst = reinterpret_cast<uint2*>(out + ((size_t)b * n_h + h) * kDv + 4 * lane);
    *dst = make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv));
  }
}

}  // namespace

size_t naive_workspace_bytes(int n_h, int batch, int max_ctx) {
  const int max_splits = (max_ctx + kNaiveSplit - 1) / kNaiveSplit;
  return sizeof(float) * (size_t)batch * n_h * max_splits * kSplitF;
}

cudaError_t launch_expand_kv(const Handle& h, const void* cache, int num_pages, void* kvx, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kExpandSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(expand_kernel, dim3(num_pages, h.cfg.n_h), dim3(256), kExpandSmem, st,
                    static_cast<const __nv_bfloat16*>(cache), h.cfg.n_h, (const __nv_bfloat16*)h.w_uk,
                    (const __nv_bfloat16*)h.w_uv, static_cast<__nv_bfloat16*>(kvx));
}

cudaError_t launch_decode_naive(const Handle& h, const void* q, const int32_t* ctx_len, int batch, int max_ctx,
                                const int32_t* block_table, int bt_stride, const void* kvx, int num_pages,
                                void* workspace, void* out, cudaStream_t st) {
  const int max_splits = (max_ctx + kNaiveSplit - 1) / kNaiveSplit;
  const float scale_log2 = h.scale * 1.4426950408889634f;
  const dim3 grid(max_splits, (h.cfg.n_h + kNaiveHeads - 1) / kNaiveHeads, batch);
  cudaError_t e = launch_pdl(naive_decode_kernel, grid, dim3(kNaiveHeads * 32), 0, st,
                             static_cast<const __nv_bfloat16*>(q), ctx_len, h.cfg.n_h, max_ctx, block_table, bt_stride,
                             static_cast<const __nv_bfloat16*>(kvx), num_pages, (const float2*)h.rope_cs,
                             h.cfg.max_position, scale_log2, max_splits, static_cast<float*>(workspace),
                             static_cast<__nv_bfloat16*>(out), h.check_word);
  if (e != cudaSuccess || max_splits == 1) return e;
  return launch_pdl(naive_merge_kernel, dim3(batch), dim3(256), 0, st, ctx_len, h.cfg.n_h, max_ctx, max_splits,
                    static_cast<const float*>(workspace), static_cast<__nv_bfloat16*>(out));
}

}  // namespace mla
