// project.cu -- the input and output projections around the absorbed decode, on the device:
//
//   kv rows   [c_kv | k_r] = x . W_DKV^T, then written into the paged cache exactly as
//             mla_kv_append writes rows (latent copied or e4m3-encoded, per tensor or per block of
//             128 values, RoPE key rotated at the token's position) -- "DeepSeek-V2-Lite 真实权重执行审计" §3.1: kv_a_proj_with_mqa
//             maps a hidden state to the 512 + 64 row; kv_norm is the identity here;
//   queries   q = x . W_Q^T, per head [q_nope | q_pe] ("80 行 PyTorch 从零写 DeepSeek 的 MLA" §2);
//   output    y = o . W_O^T over the heads' concatenated values.
//
// These are weight-bound products with few rows (one per token of the step).  A CTA computes 16
// output features for up to 32 rows: warp w owns features (2w, 2w + 1) -- in the RoPE range
// that is one interleaved pair -- and lane l accumulates, in fp32 and in a fixed order, the
// products of hidden elements [256 i + 8 l, 256 i + 8 l + 8) for every chunk i; a butterfly of
// warp shuffles then sums the lanes.  Both kernels share that arithmetic, so a fused
// projection + append writes the same bytes as mla_project followed by mla_kv_append.
#include "append_ops.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

constexpr int kPThreads = 256;   // 8 warps
constexpr int kPFeat = 16;       // output features per CTA
constexpr int kPTok = 32;        // rows per CTA

// acc[t][j] = sum over the hidden dimension of x[m0 + t] * w[f + j] (every lane holds the sums).
__device__ __forceinline__ void project_pair(const __nv_bfloat16* __restrict__ x, int m0, int mt,
                                             const __nv_bfloat16* __restrict__ w, int k, int f, int lane,
                                             float (&acc)[kPTok][2]) {
#pragma unroll
  for (int t = 0; t < kPTok; ++t) acc[t][0] = acc[t][1] = 0.0f;
  const uint4* w0p = reinterpret_cast<const uint4*>(w + (size_t)f * k) + lane;
  const uint4* w1p = reinterpret_cast<const uint4*>(w + (size_t)(f + 1) * k) + lane;
  for (int i = 0; i < k / 256; ++i) {
    const uint4 a = w0p[32 * i], b = w1p[32 * i];
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < kPTok; ++t) {
      if (t < mt) {
        const uint4 xv = reinterpret_cast<const uint4*>(x + (size_t)(m0 + t) * k)[32 * i + lane];
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[t][0] = fmaf(bf16_lo(xw[e]), bf16_lo(wa[e]), acc[t][0]);
          acc[t][0] = fmaf(bf16_hi(xw[e]), bf16_hi(wa[e]), acc[t][0]);
          acc[t][1] = fmaf(bf16_lo(xw[e]), bf16_lo(wb[e]), acc[t][1]);
          acc[t][1] = fmaf(bf16_hi(xw[e]), bf16_hi(wb[e]), acc[t][1]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kPTok; ++t) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      acc[t][0] += __shfl_xor_sync(0xffffffffu, acc[t][0], o);
      acc[t][1] += __shfl_xor_sync(0xffffffffu, acc[t][1], o);
    }
  }
}

// y[m][n_out] = bf16(x[m][k] . w[n_out][k]^T)
__global__ void __launch_bounds__(kPThreads) project_kernel(const __nv_bfloat16* __restrict__ x, int m, int k,
                                                           const __nv_bfloat16* __restrict__ w, int n_out,
                                                           __nv_bfloat16* __restrict__ y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.x * kPFeat + 2 * warp, m0 = blockIdx.y * kPTok, mt = min(kPTok, m - m0);
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  float acc[kPTok][2];
  project_pair(x, m0, mt, w, k, f, lane, acc);
#pragma unroll
  for (int t = 0; t < kPTok; ++t)
    if (t < mt && lane == t)
      *reinterpret_cast<uint32_t*>(y + (size_t)(m0 + t) * n_out + f) = pack_bf16(acc[t][0], acc[t][1]);
}

// rows = x . w_dkv^T, written into the paged cache as mla_kv_append writes them
template <bool kFp8>
__global__ void __launch_bounds__(kPThreads) kv_project_append_kernel(
    const __nv_bfloat16* __restrict__ x, int n, int k, const __nv_bfloat16* __restrict__ w,
    const int32_t* __restrict__ seq, const int32_t* __restrict__ pos, const int32_t* __restrict__ block_table,
    int bt_rows, int bt_stride, uint8_t* __restrict__ cache, int num_pages, const float2* __restrict__ rope_cs,
    int max_position, float fp8_scale, unsigned* check) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.x * kPFeat + 2 * warp, m0 = blockIdx.y * kPTok, mt = min(kPTok, n - m0);
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  // lane t's row: its cache slot, or -1 when its index is out of range (flagged once, by the
  // CTA holding features 0..15)
  uint8_t* dst = nullptr;
  int p = 0;
  if (lane < mt) {
    const int s = seq[m0 + lane];
    p = pos[m0 + lane];
    if (s < 0 || s >= bt_rows || p < 0 || p >= max_position || p / kPage >= bt_stride) {
      if (blockIdx.x == 0 && warp == 0) atomicOr(check, kCheckAppend);
    } else {
      const int page = block_table[(size_t)s * bt_stride + p / kPage];
      if (page < 0 || page >= num_pages) {
        if (blockIdx.x == 0 && warp == 0) atomicOr(check, kCheckPageId);
      } else {
        dst = cache + ((size_t)page * kPage + (p % kPage)) * (size_t)(kRow * (kFp8 ? 1 : 2));
      }
    }
  }
  float acc[kPTok][2];
  project_pair(x, m0, mt, w, k, f, lane, acc);
#pragma unroll
  for (int t = 0; t < kPTok; ++t) {
    if (t < mt && lane == t && dst) {
      // the row value is the bf16 rounding of the fp32 sum, as a row handed to mla_kv_append
      const uint32_t b = pack_bf16(acc[t][0], acc[t][1]);
      float v0 = bf16_lo(b), v1 = bf16_hi(b);
      if (f >= kDc) rope_pair(v0, v1, rope_cs[(size_t)p * (kDr / 2) + (f - kDc) / 2], &v0, &v1);
      if (!kFp8) {
        *reinterpret_cast<uint32_t*>(dst + 2 * f) = f >= kDc ? pack_bf16(v0, v1) : b;
      } else {
        const uint32_t c = pack_e4m3x4(__fdiv_rn(v0, fp8_scale), __fdiv_rn(v1, fp8_scale), 0.0f, 0.0f);
        *reinterpret_cast<uint16_t*>(dst + f) = (uint16_t)(c & 0xFFFFu);
      }
    }
  }
}

// Per-block FP8 cache: a block's scale needs all 128 of its values, so a CTA projects whole rows.
// It computes the 576 features of its kPTok rows in 36 passes of 16 (project_pair, as above, each
// bf16-rounded into a shared-memory row), then one warp per row writes it as mla_kv_append does.
__global__ void __launch_bounds__(kPThreads) kv_project_append_block_kernel(
    const __nv_bfloat16* __restrict__ x, int n, int k, const __nv_bfloat16* __restrict__ w,
    const int32_t* __restrict__ seq, const int32_t* __restrict__ pos, const int32_t* __restrict__ block_table,
    int bt_rows, int bt_stride, uint8_t* __restrict__ cache, int num_pages, const float2* __restrict__ rope_cs,
    int max_position, unsigned* check) {
  __shared__ __align__(16) uint32_t rows_s[kPTok][kRow / 2];      // bf16 pairs of the CTA's rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kPTok, mt = min(kPTok, n - m0);
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  for (int f0 = 0; f0 < kRow; f0 += kPFeat) {
    const int f = f0 + 2 * warp;
    float acc[kPTok][2];
    project_pair(x, m0, mt, w, k, f, lane, acc);
#pragma unroll
    for (int t = 0; t < kPTok; ++t)
      if (t < mt && lane == t) rows_s[t][f / 2] = pack_bf16(acc[t][0], acc[t][1]);
  }
  __syncthreads();
  for (int t = warp; t < mt; t += kPThreads / 32) {
    const int s = seq[m0 + t], p = pos[m0 + t];
    if (s < 0 || s >= bt_rows || p < 0 || p >= max_position || p / kPage >= bt_stride) {
      if (lane == 0) atomicOr(check, kCheckAppend);
      continue;
    }
    const int page = block_table[(size_t)s * bt_stride + p / kPage];
    if (page < 0 || page >= num_pages) {
      if (lane == 0) atomicOr(check, kCheckPageId);
      continue;
    }
    uint8_t* dst = cache + ((size_t)page * kPage + (p % kPage)) * (size_t)cache_row_bytes<kFp8Block>();
    write_cache_row<kFp8Block>(reinterpret_cast<const uint4*>(rows_s[t]), dst, p, lane, rope_cs, 0.0f);
  }
}

// RMSNorm of a row (Zhang & Sennrich 2019): y = x / sqrt(mean(x^2) + eps) * w, the sum of squares
// in fp32 (each lane over its 8-value chunks, then a shuffle tree), y = bf16((x * inv) * w).
// One warp per row; a lane reads its chunks in both passes and writes only them, so y may be x.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, int m, int n, int ld_x,
                                                      const __nv_bfloat16* __restrict__ w, float eps,
                                                      __nv_bfloat16* y, int ld_y) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  if (row >= m) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * ld_x);
  float ss = 0.0f;
  for (int c = lane; c < n / 8; c += 32) {
    const uint4 v = xr[c];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = bf16_lo(u[i]), b = bf16_hi(u[i]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = 1.0f / sqrtf(ss / (float)n + eps);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * ld_y);
  for (int c = lane; c < n / 8; c += 32) {
    const uint4 v = xr[c], g = wr[c];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w}, q[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = pack_bf16((bf16_lo(u[i]) * inv) * bf16_lo(q[i]), (bf16_hi(u[i]) * inv) * bf16_hi(q[i]));
    yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, int m, int n, int ld_x, const __nv_bfloat16* w, float eps,
                           __nv_bfloat16* y, int ld_y, cudaStream_t st) {
  return launch_pdl(rmsnorm_kernel, dim3((m + 7) / 8), dim3(256), 0, st, x, m, n, ld_x, w, eps, y, ld_y);
}

cudaError_t launch_project(const __nv_bfloat16* x, int m, int k, const __nv_bfloat16* w, int n_out,
                           __nv_bfloat16* y, cudaStream_t st) {
  const dim3 grid(n_out / kPFeat, (m + kPTok - 1) / kPTok);
  return launch_pdl(project_kernel, grid, dim3(kPThreads), 0, st, x, m, k, w, n_out, y);
}

cudaError_t launch_kv_project_append(const Handle& h, const __nv_bfloat16* x, int n, int k,
                                     const __nv_bfloat16* w, const int32_t* seq, const int32_t* pos,
                                     const int32_t* block_table, int bt_rows, int bt_stride, void* cache,
                                     int num_pages, cudaStream_t st) {
  if (h.cfg.cache_dtype == MLA_CACHE_FP8_E4M3_BLOCK)
    return launch_pdl(kv_project_append_block_kernel, dim3((n + kPTok - 1) / kPTok), dim3(kPThreads), 0, st, x, n, k,
                      w, seq, pos, block_table, bt_rows, bt_stride, static_cast<uint8_t*>(cache), num_pages,
                      (const float2*)h.rope_cs, h.cfg.max_position, h.check_word);
  const dim3 grid(kRow / kPFeat, (n + kPTok - 1) / kPTok);
  if (h.cfg.cache_dtype == MLA_CACHE_FP8_E4M3)
    return launch_pdl(kv_project_append_kernel<true>, grid, dim3(kPThreads), 0, st, x, n, k, w, seq, pos,
                      block_table, bt_rows, bt_stride, static_cast<uint8_t*>(cache), num_pages,
                      (const float2*)h.rope_cs, h.cfg.max_position, h.cfg.fp8_scale, h.check_word);
  return launch_pdl(kv_project_append_kernel<false>, grid, dim3(kPThreads), 0, st, x, n, k, w, seq, pos,
                    block_table, bt_rows, bt_stride, static_cast<uint8_t*>(cache), num_pages,
                    (const float2*)h.rope_cs, h.cfg.max_position, 0.0f, h.check_word);
}

}  // namespace mla
