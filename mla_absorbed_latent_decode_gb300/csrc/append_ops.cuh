// append_ops.cuh -- the per-value operations of a cache write, shared by mla_kv_append and the
// fused projection + append: bf16 unpacking and packing, e4m3 encoding (nearest even,
// saturating), and the RoPE rotation of one interleaved pair with every product and sum
// rounded to fp32.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace mla {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

// Rotate one interleaved pair by (cos, sin) with every product and sum rounded to fp32.
__device__ __forceinline__ void rope_pair(float x0, float x1, float2 cs, float* o0, float* o1) {
  *o0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
  *o1 = __fadd_rn(__fmul_rn(x1, cs.x), __fmul_rn(x0, cs.y));
}

}  // namespace mla
