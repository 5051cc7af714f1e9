// decode_simt.cu -- split-KV flash decode over the paged latent cache, CUDA-core version.
//
// For one unit (a page range of one sequence) and a group of 16 heads:
//   s_t    = scale * (q_abs[h] . row_t)          (576-wide: latent score + rope score)
//   online softmax over the unit's tokens (running max m, running sum l)
//   o[h]   = sum_t p_t row_t[0:512] / l
// "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2-§2.3; the
// flash-decode idea of streaming the latent cache once while computing is
// "G5 MLA KV 访存建模设计规格" 附录 B ("边搬边算").
//
// An FP8 cache is read as its e4m3 codes converted exactly to bf16; the tensor
// scale is folded into the softmax scale and the output.
#include <cuda_fp8.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

constexpr int kHeadsPerCta = 16;
constexpr int kThreads = 256;
constexpr size_t kSmemQ = sizeof(float) * kHeadsPerCta * kRow;
constexpr size_t kSmemTile = sizeof(__nv_bfloat16) * kPage * kRow;
constexpr size_t kSmemP = sizeof(float) * kHeadsPerCta * kPage;
constexpr size_t kSmemTotal = kSmemQ + kSmemTile + kSmemP + sizeof(float) * 3 * kHeadsPerCta;

__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 v) {
  uint32_t w[2] = {v.x, v.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i] >> (16 * k)) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      __nv_bfloat162 bf = __floats2bfloat162_rn(f.x, f.y);
      o[2 * i + k] = *reinterpret_cast<uint32_t*>(&bf);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(
    const int32_t* __restrict__ ctx_len, int n_h, const int32_t* __restrict__ block_table, int bt_stride,
    int num_pages, const uint8_t* __restrict__ cache, float score_scale, float out_scale, Workspace ws,
    unsigned* check) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem);
  __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem + kSmemQ);
  float* p_s = reinterpret_cast<float*>(smem + kSmemQ + kSmemTile);
  float* m_s = p_s + kHeadsPerCta * kPage;
  float* l_s = m_s + kHeadsPerCta;
  float* a_s = l_s + kHeadsPerCta;

  const int u = blockIdx.x;
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  if (u >= ws.counters[0]) return;
  const Unit unit = ws.units[u];
  const int b = unit.b;
  const int L = ctx_len[b];
  const int t_end = min(unit.page_end * kPage, L);
  const int h0 = blockIdx.y * kHeadsPerCta;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < kHeadsPerCta * kRow; i += kThreads) {
    const int hh = i / kRow, k = i % kRow;
    const int h = h0 + hh;
    q_s[i] = h < n_h ? __bfloat162float(ws.q_abs[((size_t)b * n_h + h) * kRow + k]) : 0.0f;
  }
  if (tid < kHeadsPerCta) { m_s[tid] = -INFINITY; l_s[tid] = 0.0f; }
  float2 acc[kHeadsPerCta];
#pragma unroll
  for (int hh = 0; hh < kHeadsPerCta; ++hh) acc[hh] = make_float2(0.0f, 0.0f);

  const int32_t* bt_row = block_table + (size_t)b * bt_stride;
  for (int pi = unit.page_begin; pi < unit.page_end; ++pi) {
    int page = bt_row[pi];
    if (page < 0 || page >= num_pages) {   // bad page id: read page 0 instead; the output is zeroed later
      if (tid == 0) {
        atomicOr(check, kCheckPageId);
        ws.bad[b] = 1;
      }
      page = 0;
    }
    const int valid = min(kPage, t_end - pi * kPage);
    __syncthreads();
    // stage the page: 64 rows x 72 chunks of 8 values, invalid rows zeroed
    for (int i = tid; i < kPage * (kRow / 8); i += kThreads) {
      const int r = i / (kRow / 8), k = i % (kRow / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < valid) {
        const size_t row = (size_t)page * kPage + r;
        if (kFp8)
          v = e4m3x8_to_bf16x8(reinterpret_cast<const uint2*>(cache + row * kRow)[k]);
        else
          v = reinterpret_cast<const uint4*>(cache + row * kRow * 2)[k];
      }
      reinterpret_cast<uint4*>(tile)[i] = v;
    }
    __syncthreads();
    // scores: 16 x 64 dot products of width 576, one warp each, lanes over pairs of columns
    for (int d = warp; d < kHeadsPerCta * kPage; d += kThreads / 32) {
      const int hh = d / kPage, t = d % kPage;
      const __nv_bfloat162* row = reinterpret_cast<const __nv_bfloat162*>(tile + t * kRow);
      const float2* qv = reinterpret_cast<const float2*>(q_s + hh * kRow);
      float s = 0.0f;
#pragma unroll
      for (int j = 0; j < kRow / 64; ++j) {
        const float2 x = __bfloat1622float2(row[lane + 32 * j]);
        const float2 y = qv[lane + 32 * j];
        s = fmaf(x.x, y.x, s);
        s = fmaf(x.y, y.y, s);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) p_s[hh * kPage + t] = t < valid ? s * score_scale : -INFINITY;
    }
    __syncthreads();
    // online softmax: warp w owns heads 2w, 2w + 1
    for (int hh = 2 * warp; hh < 2 * warp + 2; ++hh) {
      const float s0 = p_s[hh * kPage + lane], s1 = p_s[hh * kPage + lane + 32];
      float mt = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_old = m_s[hh];
      const float m_new = fmaxf(m_old, mt);
      const float alpha = m_old == -INFINITY ? 0.0f : expf(m_old - m_new);
      const float e0 = expf(s0 - m_new), e1 = expf(s1 - m_new);
      float sum = e0 + e1;
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      p_s[hh * kPage + lane] = e0;
      p_s[hh * kPage + lane + 32] = e1;
      __syncwarp();
      if (lane == 0) {
        m_s[hh] = m_new;
        l_s[hh] = l_s[hh] * alpha + sum;
        a_s[hh] = alpha;
      }
    }
    __syncthreads();
    // o[h][2 tid .. 2 tid + 1] = alpha * o + sum_t p[h][t] * row_t
#pragma unroll
    for (int hh = 0; hh < kHeadsPerCta; ++hh) {
      const float a = a_s[hh];
      acc[hh].x *= a;
      acc[hh].y *= a;
    }
    for (int t = 0; t < valid; ++t) {
      const float2 x = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(tile + t * kRow)[tid]);
#pragma unroll
      for (int hh = 0; hh < kHeadsPerCta; ++hh) {
        const float p = p_s[hh * kPage + t];
        acc[hh].x = fmaf(p, x.x, acc[hh].x);
        acc[hh].y = fmaf(p, x.y, acc[hh].y);
      }
    }
  }
  __syncthreads();
  for (int hh = 0; hh < kHeadsPerCta; ++hh) {
    const int h = h0 + hh;
    if (h >= n_h) break;
    const float inv = out_scale / l_s[hh];
    const float2 o = make_float2(acc[hh].x * inv, acc[hh].y * inv);
    if (unit.part < 0) {
      __nv_bfloat162 v = __floats2bfloat162_rn(o.x, o.y);
      reinterpret_cast<__nv_bfloat162*>(ws.o_lat + ((size_t)b * n_h + h) * kDc)[tid] = v;
    } else {
      reinterpret_cast<float2*>(ws.part_o + ((size_t)unit.part * n_h + h) * kDc)[tid] = o;
      if (tid == 0) ws.part_lse[(size_t)unit.part * n_h + h] = m_s[hh] + logf(l_s[hh]);
    }
  }
}

}  // namespace

cudaError_t launch_decode_simt(const Handle& h, const int32_t* ctx_len, int batch, const int32_t* block_table,
                          int bt_stride, const void* cache, int num_pages, const Workspace& ws, cudaStream_t st) {
  (void)batch;
  const bool fp8 = h.cfg.cache_dtype == MLA_CACHE_FP8_E4M3;
  static bool attr_set[2] = {false, false};
  auto kern = fp8 ? decode_simt_kernel<true> : decode_simt_kernel<false>;
  if (!attr_set[fp8]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTotal);
    if (e != cudaSuccess) return e;
    attr_set[fp8] = true;
  }
  const float sscale = h.scale * (fp8 ? h.cfg.fp8_scale : 1.0f);
  const float oscale = fp8 ? h.cfg.fp8_scale : 1.0f;
  dim3 grid(ws.max_units, (h.cfg.n_h + kHeadsPerCta - 1) / kHeadsPerCta);
  return launch_pdl(kern, grid, dim3(kThreads), kSmemTotal, st, ctx_len, h.cfg.n_h, block_table, bt_stride,
                    num_pages, static_cast<const uint8_t*>(cache), sscale, oscale, ws, h.check_word);
}

}  // namespace mla
