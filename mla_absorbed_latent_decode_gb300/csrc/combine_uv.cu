// combine_uv.cu -- merge split partials by log-sum-exp, then the value up-projection.
//
//   o_lat[b][h] = sum_j exp(lse_j - lse) o_j,  lse = log sum_j exp(lse_j)   (split sequences)
//   out[b][h]   = W_UV[h] o_lat[b][h]                                      (128 x 512 per head)
//
// The up-projection after the latent sum is value absorption ("DeepSeek MLA
// 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.3: sum_t p_t W^V c_t =
// W^V sum_t p_t c_t).  The log-sum-exp merge of chunk partials is the standard
// split-softmax identity (not on the pages).
//
// One CTA per (head, group of 8 sequences): the merged latents go to shared
// memory, then each warp computes 32 output values per sequence with lanes over
// the 512-wide dot product, so W_UV[h] is read once per 8 sequences.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kSeqPerCta = 8;
constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) combine_uv_kernel(int B, int n_h, const __nv_bfloat16* __restrict__ w_uv,
                                                             Workspace ws, __nv_bfloat16* __restrict__ out) {
  __shared__ float lat[kSeqPerCta][kDc];
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * kSeqPerCta;
  const int nb = min(kSeqPerCta, B - b0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int j = 0; j < kSeqPerCta; ++j) {
    const int b = b0 + j;
    const SeqPlan sp = j < nb ? ws.seqs[b] : SeqPlan{0, 0};
    for (int c = tid; c < kDc; c += kThreads) {
      float v = 0.0f;
      if (sp.nsplit == 1) {
        v = __bfloat162float(ws.o_lat[((size_t)b * n_h + h) * kDc + c]);
      } else if (sp.nsplit > 1) {
        float m = -INFINITY;
        for (int k = 0; k < sp.nsplit; ++k) {
          const int part = ws.units[sp.first_unit + k].part;
          m = fmaxf(m, ws.part_lse[(size_t)part * n_h + h]);
        }
        float num = 0.0f, den = 0.0f;
        for (int k = 0; k < sp.nsplit; ++k) {
          const int part = ws.units[sp.first_unit + k].part;
          const float w = expf(ws.part_lse[(size_t)part * n_h + h] - m);
          den += w;
          num = fmaf(w, ws.part_o[((size_t)part * n_h + h) * kDc + c], num);
        }
        v = num / den;
      }
      lat[j][c] = v;
    }
  }
  __syncthreads();
  // warp w computes rows v = 32 w .. 32 w + 31 of W_UV[h] against every staged latent
  const __nv_bfloat16* W = w_uv + (size_t)h * kDv * kDc;
  for (int vi = 0; vi < 32; ++vi) {
    const int v = 32 * warp + vi;
    const __nv_bfloat162* wr = reinterpret_cast<const __nv_bfloat162*>(W + (size_t)v * kDc);
    float2 wv[kDc / 64];
#pragma unroll
    for (int k = 0; k < kDc / 64; ++k) wv[k] = __bfloat1622float2(wr[lane + 32 * k]);
    for (int j = 0; j < nb; ++j) {
      const float2* lj = reinterpret_cast<const float2*>(lat[j]);
      float s = 0.0f;
#pragma unroll
      for (int k = 0; k < kDc / 64; ++k) {
        const float2 x = lj[lane + 32 * k];
        s = fmaf(wv[k].x, x.x, s);
        s = fmaf(wv[k].y, x.y, s);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) out[((size_t)(b0 + j) * n_h + h) * kDv + v] = __float2bfloat16_rn(s);
    }
  }
}

}  // namespace

cudaError_t launch_combine_uv(const Handle& h, int batch, const Workspace& ws, __nv_bfloat16* out, cudaStream_t st) {
  dim3 grid(h.cfg.n_h, (batch + kSeqPerCta - 1) / kSeqPerCta);
  combine_uv_kernel<<<grid, kThreads, 0, st>>>(batch, h.cfg.n_h, h.w_uv, ws, out);
  return cudaGetLastError();
}

}  // namespace mla
