// head_gemm.cu -- the two per-head weight contractions of a decode step, on
// tcgen05 tensor cores, batched over every sequence so each weight byte is read
// from HBM once:
//
//   query absorption ("DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2)
//     Q_lat^T[h] [512 x B] = W_UK[h]^T [512 x 128] . q_nope[:, h]^T [128 x B]
//     plus the RoPE part of the query rotated at ctx_len - 1 (§2.4);
//   value up-projection after the latent sum (§2.3)
//     out^T[h]   [128 x B] = W_UV[h] [128 x 512] . o_lat[:, h]^T [512 x B].
//
// Before the up-projection, split sequences' partial latent sums are merged by
// log-sum-exp into o_lat (a standard identity, not on the pages); invalid
// sequences get a zero latent, hence a zero output.
//
// One CTA per (head, 128-row block of M, tile of up to 256 sequences).  Operands
// arrive by TMA in 128-byte-swizzled 64-column chunks through a small ring of
// stages; one thread issues the loads and the MMAs; warps 0-3 (one per 32 TMEM
// lanes) run the epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr int kMaxN = 256;
constexpr int kRing = 4;                               // K-chunk stages
constexpr int kAChunk = 128 * 128;                     // 128 rows x 64 bf16 = 16 KB
constexpr int kBChunk = kMaxN * 128;                   // up to 256 rows x 64 bf16 = 32 KB
constexpr int kStage = kAChunk + kBChunk;
constexpr int kSmem = kRing * kStage + 1024 + 1024;

enum Mode { kQAbsorb = 0, kUpProject = 1 };

struct GemmBars {
  uint64_t full[kRing];
  uint64_t empty[kRing];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// grid: (n_h, M blocks, N tiles).  Mode kQAbsorb: A = W_UK (MN-major, K = 128, M = 512);
// mode kUpProject: A = W_UV (K-major, K = 512, M = 128).  B = one 64-column chunk of
// q_nope / o_lat rows per K chunk, K-major.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int B, int n_h,
                 int n_pad, const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ ctx_len,
                 const float2* __restrict__ rope_cs, int max_position, __nv_bfloat16* __restrict__ out,
                 unsigned* check) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + kRing * kStage);
  volatile int* abort_flag = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, mb = blockIdx.y, n0 = blockIdx.z * kMaxN;
  const int n_here = min(n_pad, kMaxN);              // MMA N (multiple of 16)
  const uint32_t b_bytes = (uint32_t)n_here * 128;

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) { mbar_init(smem_u32(&bars->full[s]), 1); mbar_init(smem_u32(&bars->empty[s]), 1); }
    mbar_init(smem_u32(&bars->done), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(smem_u32(&bars->tmem_base), 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, n_here, kMode == kQAbsorb, false);
    bool ok = true;
    auto load_b = [&](uint32_t dst, int col, uint32_t bar) {
      // B: rows = sequences n0 .., 64 columns of head h (3-D map: column, head, sequence)
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
              dst),
          "l"(reinterpret_cast<uint64_t>(&tm_b)), "r"(col), "r"(h), "r"(n0), "r"(bar)
          : "memory");
    };
    if (kMode == kQAbsorb) {
      // one stage: A = two MN-major boxes (c = 128 mb + [0, 64) and + [64, 128), all 128 K rows n),
      // B = two K-chunks of q_nope (n = [0, 64), [64, 128))
      const uint32_t full = smem_u32(&bars->full[0]);
      const uint32_t a_st = sbase, b_st = sbase + 2 * kAChunk;
      mbar_arrive_expect_tx(full, 2u * kAChunk + 2u * b_bytes);
      tma_load_2d(a_st, &tm_a, 128 * mb, 128 * h, full);
      tma_load_2d(a_st + kAChunk, &tm_a, 128 * mb + 64, 128 * h, full);
      load_b(b_st, 0, full);
      load_b(b_st + b_bytes, 64, full);
      if (!mbar_wait(full, 0, abort_flag)) ok = false;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8 && ok; ++k)   // A: 16 K-rows of 128 B per step; the M halves are kAChunk apart
        mma_ss(tmem, sdesc_sw128(a_st + 2048 * k, kAChunk, 1024),
               sdesc_sw128(b_st + (k >> 2) * b_bytes + 32 * (k & 3), 16, 1024), idesc, k > 0 ? 1u : 0u);
    } else {
      // ring over the 8 K-chunks of 64: A = W_UV rows v (K-major), B = o_lat rows (K-major)
      auto issue = [&](int c) {
        const int s = c % kRing;
        const uint32_t full = smem_u32(&bars->full[s]);
        mbar_arrive_expect_tx(full, (uint32_t)kAChunk + b_bytes);
        const uint32_t a_dst = sbase + s * kStage;
        tma_load_2d(a_dst, &tm_a, 64 * c, 128 * h, full);
        load_b(a_dst + kAChunk, 64 * c, full);
      };
      for (int c = 0; c < 8 && c < kRing; ++c) issue(c);
      for (int c = 0; c < 8 && ok; ++c) {
        const int s = c % kRing;
        if (!mbar_wait(smem_u32(&bars->full[s]), (c / kRing) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_st = sbase + s * kStage, b_st = a_st + kAChunk;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem, sdesc_sw128(a_st + 32 * k, 16, 1024), sdesc_sw128(b_st + 32 * k, 16, 1024), idesc,
                 (c > 0 || k > 0) ? 1u : 0u);
        mma_commit(smem_u32(&bars->empty[s]));
        if (c + kRing < 8) {
          if (!mbar_wait(smem_u32(&bars->empty[s]), (c / kRing) & 1, abort_flag)) { ok = false; break; }
          issue(c + kRing);
        }
      }
    }
    if (!ok && atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
    mma_commit(smem_u32(&bars->done));
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->done), 0, abort_flag));
  tc_fence_after();
  // epilogue: lane = output row (c within the block / v), column = sequence
  const int row = 32 * warp + lane;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  if (ok) {
    for (int c0 = 0; c0 < n_here; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(lane_addr + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int b = n0 + c0 + i;
        if (b >= B) break;
        const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(r[i]));
        if (kMode == kQAbsorb)
          out[((size_t)b * n_h + h) * kRow + 128 * mb + row] = v;
        else
          out[((size_t)b * n_h + h) * kDv + row] = v;
      }
    }
  }
  if (kMode == kQAbsorb && mb == 0) {
    // RoPE part of the query, rotated at position ctx_len - 1 (clamped into the table)
    for (int i = tid; i < min(B - n0, kMaxN) * (kDr / 2); i += kThreads) {
      const int b = n0 + i / (kDr / 2), p = i % (kDr / 2);
      const int pos = min(max(ctx_len[b] - 1, 0), max_position - 1);
      const __nv_bfloat162 x = reinterpret_cast<const __nv_bfloat162*>(q + ((size_t)b * n_h + h) * kDq + kDn)[p];
      const float2 cs = rope_cs[(size_t)pos * (kDr / 2) + p];
      const float x0 = __bfloat162float(x.x), x1 = __bfloat162float(x.y);
      reinterpret_cast<uint32_t*>(out + ((size_t)b * n_h + h) * kRow + kDc)[p] =
          bf16x2_bits(x0 * cs.x - x1 * cs.y, x1 * cs.x + x0 * cs.y);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// Log-sum-exp merge of split sequences' partials into o_lat (bf16); zero latent for
// invalid sequences; unsplit sequences already hold their latent.  One warp per (b, h).
__global__ void __launch_bounds__(128) combine_kernel(int B, int n_h, Workspace ws) {
  const int b = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= n_h) return;
  const SeqPlan sp = ws.seqs[b];
  if (sp.nsplit == 1) return;
  uint4* dst = reinterpret_cast<uint4*>(ws.o_lat + ((size_t)b * n_h + h) * kDc) + 2 * lane;   // 16 values
  if (sp.nsplit == 0) {
    dst[0] = make_uint4(0, 0, 0, 0);
    dst[1] = make_uint4(0, 0, 0, 0);
    return;
  }
  float m = -INFINITY;
  for (int k = 0; k < sp.nsplit; ++k)
    m = fmaxf(m, ws.part_lse[(size_t)ws.units[sp.first_unit + k].part * n_h + h]);
  float acc[16], den = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
  for (int k = 0; k < sp.nsplit; ++k) {
    const int part = ws.units[sp.first_unit + k].part;
    const float w = expf(ws.part_lse[(size_t)part * n_h + h] - m);
    den += w;
    const float4* src = reinterpret_cast<const float4*>(ws.part_o + ((size_t)part * n_h + h) * kDc) + 4 * lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = src[i];
      acc[4 * i] = fmaf(w, v.x, acc[4 * i]);
      acc[4 * i + 1] = fmaf(w, v.y, acc[4 * i + 1]);
      acc[4 * i + 2] = fmaf(w, v.z, acc[4 * i + 2]);
      acc[4 * i + 3] = fmaf(w, v.w, acc[4 * i + 3]);
    }
  }
  const float inv = 1.0f / den;
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = bf16x2_bits(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult qr;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Weight map: [n_h * 128 rows][512 bf16], 64 x 128 boxes, 128-byte swizzle.
cudaError_t weight_map(const void* w, int n_h, CUtensorMap* m) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)kDc, (cuuint64_t)n_h * 128};
  const cuuint64_t strides[1] = {(cuuint64_t)kDc * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

// Per-sequence rows of one head: tensor [B][n_h][width] bf16 viewed as (column, head, sequence),
// boxes of 64 columns x 1 head x n_box sequences, 128-byte swizzle; rows past B read as zero.
cudaError_t rows_map(const void* base, int B, int n_h, int width, int n_box, CUtensorMap* m) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)n_h, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * n_h};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)n_box};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

template <int kMode>
cudaError_t launch_head_gemm(const Handle& h, const CUtensorMap& ta, const CUtensorMap& tb, int batch,
                             const __nv_bfloat16* q, const int32_t* ctx_len, __nv_bfloat16* out, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(head_gemm_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int n_pad = ((batch + 15) / 16) * 16;
  dim3 grid(h.cfg.n_h, kMode == kQAbsorb ? 4 : 1, (batch + kMaxN - 1) / kMaxN);
  head_gemm_kernel<kMode><<<grid, kThreads, kSmem, st>>>(ta, tb, batch, h.cfg.n_h, n_pad, q, ctx_len, h.rope_cs,
                                                         h.cfg.max_position, out, h.check_word);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_weight_maps(Handle& h) {
  cudaError_t e = weight_map(h.w_uk, h.cfg.n_h, reinterpret_cast<CUtensorMap*>(h.tmap_wuk));
  if (e != cudaSuccess) return e;
  return weight_map(h.w_uv, h.cfg.n_h, reinterpret_cast<CUtensorMap*>(h.tmap_wuv));
}

cudaError_t launch_q_absorb(const Handle& h, const __nv_bfloat16* q, const int32_t* ctx_len, int batch,
                            const Workspace& ws, cudaStream_t st) {
  alignas(64) CUtensorMap tq;
  cudaError_t e = rows_map(q, batch, h.cfg.n_h, kDq, min(((batch + 15) / 16) * 16, kMaxN), &tq);
  if (e != cudaSuccess) return e;
  return launch_head_gemm<kQAbsorb>(h, *reinterpret_cast<const CUtensorMap*>(h.tmap_wuk), tq, batch, q, ctx_len,
                                    ws.q_abs, st);
}

cudaError_t launch_combine_uv(const Handle& h, int batch, const Workspace& ws, __nv_bfloat16* out, cudaStream_t st) {
  combine_kernel<<<dim3(batch, (h.cfg.n_h + 3) / 4), 128, 0, st>>>(batch, h.cfg.n_h, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap to;
  e = rows_map(ws.o_lat, batch, h.cfg.n_h, kDc, min(((batch + 15) / 16) * 16, kMaxN), &to);
  if (e != cudaSuccess) return e;
  return launch_head_gemm<kUpProject>(h, *reinterpret_cast<const CUtensorMap*>(h.tmap_wuv), to, batch, nullptr,
                                      nullptr, out, st);
}

}  // namespace mla
