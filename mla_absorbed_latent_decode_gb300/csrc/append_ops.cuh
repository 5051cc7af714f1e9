// append_ops.cuh -- the per-value operations of a cache write and read, shared by mla_kv_append,
// the fused projection + append and the kernels that read an FP8 cache: bf16 unpacking and
// packing, e4m3 encoding (nearest even, saturating) and exact decoding, the RoPE rotation of one
// interleaved pair with every product and sum rounded to fp32, and the row write itself.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.cuh"

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

// FP8 cache: e4m3 -> bf16, exact, in integer and fp32 arithmetic (no conversion instruction):
// the code's 7 magnitude bits placed at bit 20 of a float32, its sign at bit 31, make that
// value times 2^-120 (a normal e4m3 keeps its exponent and mantissa fields; a subnormal one
// becomes a float32 subnormal), so one multiply by 2^120 (denormals kept) gives the value; it
// has at most 4 significant bits, so the upper 16 bits of the float32 are its bf16.  Code k of
// the word is moved to bits 24..31, shifted arithmetically by 4 (the sign lands on bits 28..31)
// and masked.  Output: bf16 of codes (0, 1) and (2, 3), low half first.
__device__ __forceinline__ float e4m3_at_top_to_f32(uint32_t t) {
  const uint32_t bits = (uint32_t)((int32_t)t >> 4) & 0x87F00000u;
  float f;
  asm("mul.rn.f32 %0, %1, 0f7B800000;" : "=f"(f) : "f"(__uint_as_float(bits)));   // x 2^120
  return f;
}
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  const float f0 = e4m3_at_top_to_f32(w << 24), f1 = e4m3_at_top_to_f32(w << 16);
  const float f2 = e4m3_at_top_to_f32(w << 8), f3 = e4m3_at_top_to_f32(w);
  return make_uint2(__byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632),
                    __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632));
}

// Per-block FP8 cache: the exact values of four codes times their block scale, each product
// rounded to fp32 and then to bf16 (nearest even); low half first, as above.
__device__ __forceinline__ uint2 e4m3x4_scaled_to_bf16x4(uint32_t w, float scale) {
  const float f0 = e4m3_at_top_to_f32(w << 24) * scale, f1 = e4m3_at_top_to_f32(w << 16) * scale;
  const float f2 = e4m3_at_top_to_f32(w << 8) * scale, f3 = e4m3_at_top_to_f32(w) * scale;
  return make_uint2(pack_bf16(f0, f1), pack_bf16(f2, f3));
}

// cache formats of a row write: bf16, e4m3 with one tensor scale, per-block e4m3 (656 bytes)
enum AppendMode { kBf16 = 0, kFp8Tensor = 1, kFp8Block = 2 };

template <int kMode>
__host__ __device__ constexpr int cache_row_bytes() {
  return kMode == kBf16 ? kRow * 2 : kMode == kFp8Tensor ? kRow : kDc + 16 + 2 * kDr;
}

// One row [c (512) | k_r (64)] bf16 at `src` written to its cache slot `dst` by one warp (position
// p for the RoPE rotation).  Lane l owns latent values [16 l, 16 l + 16) (the 8 lanes of a
// 128-value block find its maximum by shuffles); lanes 0..3 also own RoPE values [16 l, 16 l + 16).
template <int kMode>
__device__ __forceinline__ void write_cache_row(const uint4* __restrict__ src, uint8_t* __restrict__ dst, int p,
                                                int lane, const float2* __restrict__ rope_cs, float fp8_scale) {
  // latent: values [16 lane, 16 lane + 16)
  const uint4 a = src[2 * lane];
  const uint4 b = src[2 * lane + 1];
  if (kMode == kBf16) {
    reinterpret_cast<uint4*>(dst)[2 * lane] = a;
    reinterpret_cast<uint4*>(dst)[2 * lane + 1] = b;
  } else {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float scale = fp8_scale;
    if (kMode == kFp8Block) {               // this lane's block: 128 values on lanes 8 k .. 8 k + 7
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
#pragma unroll
      for (int off = 4; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      scale = __fdiv_rn(m, 448.0f);
      if ((lane & 7) == 0) reinterpret_cast<float*>(dst + kDc)[lane >> 3] = scale;
    }
    uint32_t o[4];
    if (kMode == kFp8Block && !(scale > 0.0f)) {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = 0u;   // an all-zero block: zero codes
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = pack_e4m3x4(__fdiv_rn(bf16_lo(w[2 * i]), scale), __fdiv_rn(bf16_hi(w[2 * i]), scale),
                           __fdiv_rn(bf16_lo(w[2 * i + 1]), scale), __fdiv_rn(bf16_hi(w[2 * i + 1]), scale));
    }
    reinterpret_cast<uint4*>(dst)[lane] = make_uint4(o[0], o[1], o[2], o[3]);
  }

  // RoPE key: lanes 0..3 own values [16 lane, 16 lane + 16) = pairs [8 lane, 8 lane + 8)
  if (lane < 4) {
    const uint4 ra = src[kDc / 8 + 2 * lane];
    const uint4 rb = src[kDc / 8 + 2 * lane + 1];
    const uint32_t w[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
    const float2* cs = rope_cs + (size_t)p * (kDr / 2) + 8 * lane;
    float r[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) rope_pair(bf16_lo(w[i]), bf16_hi(w[i]), cs[i], &r[2 * i], &r[2 * i + 1]);
    if (kMode != kFp8Tensor) {             // bf16, after the latent (and, per-block, the 16 scale bytes)
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = pack_bf16(r[2 * i], r[2 * i + 1]);
      uint4* d = reinterpret_cast<uint4*>(dst + (kMode == kBf16 ? kDc * 2 : kDc + 16));
      d[2 * lane] = make_uint4(o[0], o[1], o[2], o[3]);
      d[2 * lane + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = pack_e4m3x4(__fdiv_rn(r[4 * i], fp8_scale), __fdiv_rn(r[4 * i + 1], fp8_scale),
                           __fdiv_rn(r[4 * i + 2], fp8_scale), __fdiv_rn(r[4 * i + 3], fp8_scale));
      reinterpret_cast<uint4*>(dst + kDc)[lane] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace mla
