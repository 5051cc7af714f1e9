// absorb.cu -- query preparation of a decode step.
//
//   q_abs[b][h][0:512]   = W_UK[h]^T q_nope[b][h]          (key absorption)
//   q_abs[b][h][512:576] = RoPE(q_pe[b][h], ctx_len[b] - 1)
//
// "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2 moves W_UK
// from every cached token to the query (q^T W^K c = (W^K^T q)^T c); the RoPE
// part cannot be absorbed (§2.4) and is rotated at the query position.
// fp32 accumulation, bf16 result.
//
// One CTA per (head, group of 8 sequences), one thread per latent index c: the
// thread walks the 128 no-RoPE rows of W_UK[h] (coalesced across c) and keeps
// 8 accumulators, so each weight element is read once per 8 sequences.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kSeqPerCta = 8;

__global__ void __launch_bounds__(kDc) q_absorb_kernel(
    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ ctx_len, int B, int n_h,
    const __nv_bfloat16* __restrict__ w_uk, const float2* __restrict__ rope_cs, int max_position,
    __nv_bfloat16* __restrict__ q_abs) {
  __shared__ float qn[kSeqPerCta][kDn];
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * kSeqPerCta;
  const int nb = min(kSeqPerCta, B - b0);
  const int c = threadIdx.x;
  for (int i = threadIdx.x; i < kSeqPerCta * kDn; i += blockDim.x) {
    const int j = i / kDn, n = i % kDn;
    qn[j][n] = j < nb ? __bfloat162float(q[((size_t)(b0 + j) * n_h + h) * kDq + n]) : 0.0f;
  }
  __syncthreads();
  float acc[kSeqPerCta];
#pragma unroll
  for (int j = 0; j < kSeqPerCta; ++j) acc[j] = 0.0f;
  const __nv_bfloat16* w = w_uk + (size_t)h * kDn * kDc + c;
  for (int n = 0; n < kDn; ++n) {
    const float wv = __bfloat162float(w[(size_t)n * kDc]);
#pragma unroll
    for (int j = 0; j < kSeqPerCta; ++j) acc[j] = fmaf(wv, qn[j][n], acc[j]);
  }
  for (int j = 0; j < nb; ++j) q_abs[((size_t)(b0 + j) * n_h + h) * kRow + c] = __float2bfloat16_rn(acc[j]);

  // RoPE of the query's rope part at position ctx_len - 1 (clamped into the table;
  // an invalid length's output is zeroed later).
  if (threadIdx.x < kSeqPerCta * (kDr / 2)) {
    const int j = threadIdx.x / (kDr / 2), i = threadIdx.x % (kDr / 2);
    if (j < nb) {
      const int b = b0 + j;
      const int pos = min(max(ctx_len[b] - 1, 0), max_position - 1);
      const __nv_bfloat16* src = q + ((size_t)b * n_h + h) * kDq + kDn;
      const float x0 = __bfloat162float(src[2 * i]), x1 = __bfloat162float(src[2 * i + 1]);
      const float2 cs = rope_cs[(size_t)pos * (kDr / 2) + i];
      __nv_bfloat16* dst = q_abs + ((size_t)b * n_h + h) * kRow + kDc;
      dst[2 * i] = __float2bfloat16_rn(x0 * cs.x - x1 * cs.y);
      dst[2 * i + 1] = __float2bfloat16_rn(x1 * cs.x + x0 * cs.y);
    }
  }
}

}  // namespace

cudaError_t launch_q_absorb(const Handle& h, const __nv_bfloat16* q, const int32_t* ctx_len, int batch,
                            const Workspace& ws, cudaStream_t st) {
  dim3 grid(h.cfg.n_h, (batch + kSeqPerCta - 1) / kSeqPerCta);
  q_absorb_kernel<<<grid, kDc, 0, st>>>(q, ctx_len, batch, h.cfg.n_h, h.w_uk, h.rope_cs, h.cfg.max_position,
                                        ws.q_abs);
  return cudaGetLastError();
}

}  // namespace mla
