// append.cu -- mla_kv_append: write token rows into the paged latent cache.
//
// A row is [c (512) | k_r (64)] bf16.  The latent is stored unchanged; the RoPE
// key is rotated at the token's absolute position ("DeepSeek MLA 吸收式缓存：真实
// 权重执行与 FlashMLA 架构边界" §2.4; rotation of interleaved pairs as in "80 行
// PyTorch 从零写 DeepSeek 的 MLA" 附录 A).  An FP8 cache stores every value
// divided by the tensor scale as OCP e4m3 (nearest even, saturating).  A per-block
// FP8 cache ("G5 MLA KV 访存建模设计规格" 附录 A: 656 bytes per token with per-block
// scales) stores [512 e4m3 latent codes | 4 fp32 scales | 64 bf16 RoPE values]: each
// block of 128 latent values is divided by its own scale max|x| / 448.
//
// One warp per row.  Lane l owns latent values [16 l, 16 l + 16) (32 bytes in,
// 32 bytes (bf16) or 16 bytes (e4m3) out; the 8 lanes of a 128-value block find its
// maximum by shuffles); lanes 0..3 also own RoPE values [16 l, 16 l + 16) of the key.
// HBM-bound: 1152 bytes read and 1152 (bf16), 576 (e4m3) or 656 bytes written per row.
#include "append_ops.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

template <int kMode>
__global__ void __launch_bounds__(256) kv_append_kernel(
    const __nv_bfloat16* __restrict__ rows, const int32_t* __restrict__ seq,
    const int32_t* __restrict__ pos, int n, const int32_t* __restrict__ block_table, int bt_rows,
    int bt_stride, uint8_t* __restrict__ cache, int num_pages, const float2* __restrict__ rope_cs,
    int max_position, float fp8_scale, unsigned* check) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  sm100::griddep_wait();
  sm100::griddep_launch_dependents();
  if (warp >= n) return;
  const int s = seq[warp];
  const int p = pos[warp];
  if (s < 0 || s >= bt_rows || p < 0 || p >= max_position || p / kPage >= bt_stride) {
    if (lane == 0) atomicOr(check, kCheckAppend);
    return;
  }
  const int page = block_table[(size_t)s * bt_stride + p / kPage];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) atomicOr(check, kCheckPageId);
    return;
  }
  constexpr int kRowBytes = cache_row_bytes<kMode>();
  const uint4* src = reinterpret_cast<const uint4*>(rows + (size_t)warp * kRow);
  uint8_t* dst = cache + ((size_t)page * kPage + (p % kPage)) * (size_t)kRowBytes;
  write_cache_row<kMode>(src, dst, p, lane, rope_cs, fp8_scale);
}

}  // namespace

cudaError_t launch_kv_append(const Handle& h, const __nv_bfloat16* rows, const int32_t* seq,
                             const int32_t* pos, int n, const int32_t* block_table, int bt_rows,
                             int bt_stride, void* cache, int num_pages, cudaStream_t st) {
  const int threads = 256;
  const int blocks = (int)(((long long)n * 32 + threads - 1) / threads);
  if (h.cfg.cache_dtype == MLA_CACHE_FP8_E4M3)
    return launch_pdl(kv_append_kernel<kFp8Tensor>, dim3(blocks), dim3(threads), 0, st, rows, seq, pos, n,
                      block_table, bt_rows, bt_stride, static_cast<uint8_t*>(cache), num_pages,
                      (const float2*)h.rope_cs, h.cfg.max_position, h.cfg.fp8_scale, h.check_word);
  if (h.cfg.cache_dtype == MLA_CACHE_FP8_E4M3_BLOCK)
    return launch_pdl(kv_append_kernel<kFp8Block>, dim3(blocks), dim3(threads), 0, st, rows, seq, pos, n,
                      block_table, bt_rows, bt_stride, static_cast<uint8_t*>(cache), num_pages,
                      (const float2*)h.rope_cs, h.cfg.max_position, 0.0f, h.check_word);
  return launch_pdl(kv_append_kernel<kBf16>, dim3(blocks), dim3(threads), 0, st, rows, seq, pos, n, block_table,
                    bt_rows, bt_stride, static_cast<uint8_t*>(cache), num_pages, (const float2*)h.rope_cs,
                    h.cfg.max_position, 0.0f, h.check_word);
}

}  // namespace mla
