// prefill.cu -- causal prefill over the latent cache in MHA mode, on tcgen05 tensor cores.
//
// Prefill handles every query token of a prompt (or of a chunk after a cached prefix) in one
// pass; with query length = context length it is compute-bound ("G5 MLA KV 访存建模设计规格",
// 名词定义 and 用例 2).  FlashMLA runs dense prefill in MHA mode, i.e. with the latent expanded
// per head ("DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §6.1 support matrix,
// §2.1 for the expansion), which costs 2 (d_nope + d_rope + d_v) = 640 flops per query, key
// and head against 2 (d_c + d_rope + d_c) = 2176 in the absorbed form.
//
//   1. expand_tc_kernel: for every cached row t of a sequence and head h,
//        K_nope[b][h][t] = W_UK[h] c_t,   V[b][h][t] = W_UV[h] c_t     (bf16),
//      and the (already rotated) RoPE key K_r[b][t] copied once per token (an FP8 cache's values
//      decoded: codes times the tensor scale, or times their block's scale);
//      item = (head, 128 tokens): D[128 tokens][256] = C[128][512] . [W_UK[h] ; W_UV[h]]^T,
//      A = two cache pages by TMA, B = the head's weight rows, K-major, 4-stage ring;
//      persistent CTAs, two TMEM accumulators (the epilogue of an item under the next's MMAs).
//   2. prefill_attn_kernel: item = (128 queries, head, sequence), persistent CTAs taking items in
//      turn; query i of sequence b sits at position ctx_len - q_len + i and sees keys 0 .. that
//      position.  Per 128-key tile j:
//        S = Q K^T (M = 128 queries, N = 128 keys, K = 128 + 64) into one of two TMEM score
//        buffers; online softmax (base 2, lazy rescale of O when the running maximum grows by
//        more than 2^8) by warps 0-3, one query row per thread; P (bf16) into TMEM; O += P V
//        (A = P from TMEM, B = V MN-major).  One thread issues the QK^T MMAs and another the
//        P V ones; K and V tiles arrive by TMA from two producer warps through 2-stage rings.
//
// TMEM of the attention CTA (512 columns): O [0, 128), S0 [128, 256), S1 [256, 384),
// P0 [384, 448), P1 [448, 512).  Shared memory: Q 48 KB, K ring 2 x 48 KB, V ring 2 x 32 KB.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "append_ops.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBox = 128 * 128;        // 64 bf16 columns x 128 rows, 128-byte swizzled: 16 KB
constexpr int kPageBox = 128 * 64;     // 64 bf16 columns x 64 rows (one cache page): 8 KB
constexpr int kTile = 128;             // tokens of an expansion tile = keys of an attention tile
constexpr int kQBlk = 128;             // queries of an attention CTA

// ------------------------------------------------------------------ expansion
// cache formats: bf16 rows; e4m3 rows with one tensor scale; per-block e4m3 rows (656 bytes: 512
// codes, 4 fp32 block scales, 64 bf16 RoPE values).  With an FP8 cache each page's 64 x 64 code
// box lands in the upper half of its bf16 box and one conversion warp per page turns it into the
// bf16 operand in place (exact values; per block: times the token's block scale, rounded to bf16);
// the tensor scale is applied in the epilogue, in fp32.
constexpr int kExBf16 = 0, kExFp8 = 1, kExFp8Block = 2;
constexpr int kExStages = 4;
constexpr int kExScaleBytes = kPage * 16;                    // per-block format: 64 tokens x 4 fp32 scales
template <int kMode>
__host__ __device__ constexpr int ex_stage_bytes() {                             // two pages x 64 columns, W_UK and W_UV boxes
  return 2 * kPageBox + 2 * kBox + (kMode == kExFp8Block ? 2 * kExScaleBytes : 0);
}
template <int kMode>
__host__ __device__ constexpr int ex_threads() {                                 // warps 0-3 epilogue, 4 producer, 5 MMA, 6-7 conversion
  return kMode == kExBf16 ? 192 : 256;
}
template <int kMode>
__host__ __device__ constexpr int ex_smem() {
  return kExStages * ex_stage_bytes<kMode>() + 1024 + 1024;
}

struct ExBars {
  uint64_t full[kExStages];
  uint64_t conv[kExStages];    // FP8 cache: both pages of the chunk converted (2 warps)
  uint64_t empty[kExStages];
  uint64_t acc_full[2];      // the MMAs of an item are done: its accumulator may be read
  uint64_t acc_empty[2];     // the epilogue has read the accumulator (4 warps arrive)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ bool page_ok(int p, int num_pages) { return p >= 0 && p < num_pages; }

// One 32-byte global store (a whole sector; the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_32B(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// One expansion item: 128 tokens of a sequence for one head.  Items are numbered with the head
// fastest, so the CTAs working at the same time share the token tile (its cache rows stay in L2).
struct ExItem {
  int h, t0, b, L, p0, p1;
  bool valid, ok0, ok1;
};

__device__ __forceinline__ ExItem ex_item(int idx, int n_h, int ntb, const int32_t* ctx_len, int max_ctx,
                                          const int32_t* block_table, int bt_stride, int num_pages) {
  ExItem it;
  it.h = idx % n_h;
  const int tb = (idx / n_h) % ntb;
  it.b = idx / (n_h * ntb);
  it.t0 = tb * kTile;
  it.L = ctx_len[it.b];
  it.valid = it.L >= 1 && it.L <= max_ctx && it.t0 < it.L;   // the attention kernel flags bad lengths
  const bool need1 = it.t0 + kPage < it.L;
  it.p0 = it.valid ? block_table[(size_t)it.b * bt_stride + 2 * tb] : -1;
  it.p1 = it.valid && need1 ? block_table[(size_t)it.b * bt_stride + 2 * tb + 1] : -1;
  it.ok0 = it.valid && page_ok(it.p0, num_pages);
  it.ok1 = it.valid && need1 && page_ok(it.p1, num_pages);
  return it;
}

// Persistent: CTA c takes items c, c + gridDim.x, ...; the K-chunk ring runs on across items and
// the accumulator alternates between two 256-column TMEM halves, so the epilogue of one item
// overlaps the loads and MMAs of the next.
template <int kMode>
__global__ void __launch_bounds__(ex_threads<kMode>(), 1)
expand_tc_kernel(const __grid_constant__ CUtensorMap tm_cache, const __grid_constant__ CUtensorMap tm_wuk,
                 const __grid_constant__ CUtensorMap tm_wuv, const __grid_constant__ CUtensorMap tm_scale,
                 const uint8_t* __restrict__ cache, float cache_scale,
                 const int32_t* __restrict__ ctx_len, int n_h, int max_ctx, const int32_t* __restrict__ block_table,
                 int bt_stride, int num_pages, int lpad, int n_items, __nv_bfloat16* __restrict__ kn,
                 __nv_bfloat16* __restrict__ vv, __nv_bfloat16* __restrict__ kr, int* sched, int stall,
                 unsigned* check) {
  constexpr bool kFp8 = kMode != kExBf16;
  constexpr int kStageB = ex_stage_bytes<kMode>();
  constexpr int kRowB = kMode == kExBf16 ? kRow * 2 : kMode == kExFp8 ? kRow : kDc + 16 + 2 * kDr;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  ExBars* bars = reinterpret_cast<ExBars*>(smem + kExStages * kStageB);
  volatile int* abort_flag = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntb = lpad / kTile;
  if (tid == 0) {
    for (int i = 0; i < kExStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->conv[i]), 2);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->acc_full[i]), 1);
      mbar_init(smem_u32(&bars->acc_empty[i]), 4);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) { tmem_alloc(smem_u32(&bars->tmem_base), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  griddep_wait();                          // the rows may have been appended by the previous kernel
  griddep_launch_dependents();
  // the attention kernel's work counter (after the wait: an earlier call's attention, still the
  // previous kernel in the stream, may have been using it)
  if (blockIdx.x == 0 && tid == 0) *sched = 0;

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_cache);
      if (kMode == kExFp8Block) prefetch_tmap(&tm_scale);
      int c = 0;                           // K chunks issued so far (ring position)
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        const ExItem it = ex_item(idx, n_h, ntb, ctx_len, max_ctx, block_table, bt_stride, num_pages);
        if (!it.valid) continue;
        if (it.h == 0 && (!it.ok0 || (it.t0 + kPage < it.L && !it.ok1))) atomicOr(check, kCheckPageId);
        constexpr uint32_t kPageTx = kMode == kExBf16 ? kPageBox : kPageBox / 2 + (kMode == kExFp8Block ? kExScaleBytes : 0);
        const uint32_t bytes = (it.ok0 ? kPageTx : 0) + (it.ok1 ? kPageTx : 0) + 2 * kBox;
        for (int kc = 0; kc < kDc / 64; ++kc, ++c) {
          const int s = c % kExStages;
          if (c >= kExStages && !mbar_wait(smem_u32(&bars->empty[s]), ((c / kExStages) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * kStageB, fb = smem_u32(&bars->full[s]);
          mbar_arrive_expect_tx(fb, bytes);
          // (an FP8 page's codes into the upper half of its bf16 box; per block, its scales after the weights)
          if (it.ok0) tma_load_2d(st + (kFp8 ? kPageBox / 2 : 0), &tm_cache, 64 * kc, it.p0 * kPage, fb);
          if (it.ok1) tma_load_2d(st + kPageBox + (kFp8 ? kPageBox / 2 : 0), &tm_cache, 64 * kc, it.p1 * kPage, fb);
          if (kMode == kExFp8Block) {
            if (it.ok0) tma_load_2d(st + 2 * kPageBox + 2 * kBox, &tm_scale, kDc, it.p0 * kPage, fb);
            if (it.ok1) tma_load_2d(st + 2 * kPageBox + 2 * kBox + kExScaleBytes, &tm_scale, kDc, it.p1 * kPage, fb);
          }
          tma_load_2d(st + 2 * kPageBox, &tm_wuk, 64 * kc, kDn * it.h, fb);
          // (a test of the bounded waits, stall == 4: CTA 0 never loads the W_UV box of its first
          // chunk, so that stage's barrier, armed for every byte, cannot complete)
          if (!(stall == 4 && blockIdx.x == 0 && c == 0))
            tma_load_2d(st + 2 * kPageBox + kBox, &tm_wuv, 64 * kc, kDv * it.h, fb);
        }
      }
      if (!ok && atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
      for (int k = max(0, c - kExStages); k < c; ++k) {   // every copy lands before exit
        volatile int never = 0;
        mbar_wait(smem_u32(&bars->full[k % kExStages]), (k / kExStages) & 1, &never);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // M = 128 tokens, N = 256 (the head's 128 W_UK rows, then its 128 W_UV rows), both K-major
      constexpr uint32_t idesc = idesc_bf16_f32(128, 256, false, false);
      int c = 0, v = 0;                    // K chunks consumed, items accumulated
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        const ExItem it = ex_item(idx, n_h, ntb, ctx_len, max_ctx, block_table, bt_stride, num_pages);
        if (!it.valid) continue;
        const int a = v & 1;
        // the accumulator's previous item (v - 2) has been read by the epilogue
        if (v >= 2 && !mbar_wait(smem_u32(&bars->acc_empty[a]), ((v >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int kc = 0; kc < kDc / 64; ++kc, ++c) {
          const int s = c % kExStages;
          if (!mbar_wait(smem_u32(kFp8 ? &bars->conv[s] : &bars->full[s]), (c / kExStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * kStageB;
          const uint64_t ad = sdesc_sw128(st, 16, 1024), wd = sdesc_sw128(st + 2 * kPageBox, 16, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)        // 16 latent columns per MMA: 32-byte steps in the 128-byte row
            mma_ss(tmem + 256 * a, ad + (uint64_t)(2 * k), wd + (uint64_t)(2 * k), idesc, (kc > 0 || k > 0) ? 1u : 0u);
          mma_commit(smem_u32(&bars->empty[s]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->acc_full[a]));
        ++v;
      }
      if (!ok && atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
      mma_commit(smem_u32(&bars->drain));    // every issued MMA has finished ...
      volatile int never = 0;
      mbar_wait(smem_u32(&bars->drain), 0, &never);   // ... before the CTA frees its TMEM
    }
  } else if (warp >= 6) {
    // ---------------------------------------------------------------- FP8 cache: codes -> bf16
    // (launched only with an FP8 cache) warp 6 + q converts page q of every chunk: lane = (row
    // 8 k + lane / 4, 16 codes 16 (lane % 4) ..) for k = 0..7; all of the box's codes are read
    // into registers before any bf16 row is written (the rows overlap the codes)
    if constexpr (kFp8) {
      const int q = warp - 6, pw = lane & 3;
      int c = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        const ExItem it = ex_item(idx, n_h, ntb, ctx_len, max_ctx, block_table, bt_stride, num_pages);
        if (!it.valid) continue;
        const bool loaded = q == 0 ? it.ok0 : it.ok1;
        for (int kc = 0; kc < kDc / 64; ++kc, ++c) {
          const int s = c % kExStages;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[s]), (c / kExStages) & 1, abort_flag))) {
            ok = false;
            break;
          }
          uint8_t* box = smem + s * kStageB + q * kPageBox;
          if (loaded) {
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              v[k] = *reinterpret_cast<const uint4*>(box + kPageBox / 2 + (8 * k + (lane >> 2)) * 64 + pw * 16);
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {       // 128-byte rows, 128-byte swizzle
              const int r = 8 * k + (lane >> 2);
              uint2 a, b, d, e;
              if constexpr (kMode == kExFp8Block) {   // times the token's scale of block kc / 2
                const float sc = reinterpret_cast<const float*>(smem + s * kStageB + 2 * kPageBox + 2 * kBox +
                                                                q * kExScaleBytes)[r * 4 + (kc >> 1)];
                a = e4m3x4_scaled_to_bf16x4(v[k].x, sc); b = e4m3x4_scaled_to_bf16x4(v[k].y, sc);
                d = e4m3x4_scaled_to_bf16x4(v[k].z, sc); e = e4m3x4_scaled_to_bf16x4(v[k].w, sc);
              } else {
                a = e4m3x4_to_bf16x4(v[k].x); b = e4m3x4_to_bf16x4(v[k].y);
                d = e4m3x4_to_bf16x4(v[k].z); e = e4m3x4_to_bf16x4(v[k].w);
              }
              *reinterpret_cast<uint4*>(box + r * 128 + (((2 * pw) ^ (r & 7)) * 16)) = make_uint4(a.x, a.y, b.x, b.y);
              *reinterpret_cast<uint4*>(box + r * 128 + (((2 * pw + 1) ^ (r & 7)) * 16)) = make_uint4(d.x, d.y, e.x, e.y);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->conv[s]));
        }
      }
      if (!ok && atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
    }
  } else {
    // ---------------------------------------------------------------- epilogue: thread = token
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    const int r = 32 * warp + lane;
    int v = 0;
    for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x) {
      const ExItem it = ex_item(idx, n_h, ntb, ctx_len, max_ctx, block_table, bt_stride, num_pages);
      if (!it.valid) continue;
      const int a = v & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->acc_full[a]), (v >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int t = it.t0 + r;
      const bool row_ok = t < it.L && (r < kPage ? it.ok0 : it.ok1);
      uint4* dk = reinterpret_cast<uint4*>(kn + (((size_t)it.b * n_h + it.h) * lpad + t) * kDn);
      uint4* dv = reinterpret_cast<uint4*>(vv + (((size_t)it.b * n_h + it.h) * lpad + t) * kDv);
#pragma unroll 1
      for (int g = 0; g < 8; ++g) {          // columns 32 g .. 32 g + 31: K_nope for g < 4, V after
        uint32_t x[32];
        tmem_ld32(lane_addr + 256 * a + 32 * g, x);
        tmem_ld_wait();
        uint4* d = (g < 4 ? dk : dv) + 4 * (g & 3);
#pragma unroll
        for (int i = 0; i < 2; ++i) {        // whole 32-byte sectors (a row's 64 bytes of the group)
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            w[e] = row_ok ? bf16x2(__uint_as_float(x[16 * i + 2 * e]) * cache_scale,
                                   __uint_as_float(x[16 * i + 2 * e + 1]) * cache_scale)
                          : 0u;
          st_global_32B(d + 2 * i, w);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[a]));
      if (it.h == 0) {                       // the RoPE key, shared by the heads, once per token
        uint4* d = reinterpret_cast<uint4*>(kr + ((size_t)it.b * lpad + t) * kDr);
        if (row_ok) {
          const uint8_t* row = cache + ((size_t)(r < kPage ? it.p0 : it.p1) * kPage + (r & (kPage - 1))) * kRowB;
          if constexpr (kMode == kExFp8) {    // 64 codes times the tensor scale
            const uint4* src = reinterpret_cast<const uint4*>(row + kDc);
#pragma unroll
            for (int i = 0; i < kDr / 16; ++i) {
              const uint4 v = src[i];
              const uint2 a = e4m3x4_scaled_to_bf16x4(v.x, cache_scale), b = e4m3x4_scaled_to_bf16x4(v.y, cache_scale);
              const uint2 g = e4m3x4_scaled_to_bf16x4(v.z, cache_scale), f = e4m3x4_scaled_to_bf16x4(v.w, cache_scale);
              d[2 * i] = make_uint4(a.x, a.y, b.x, b.y);
              d[2 * i + 1] = make_uint4(g.x, g.y, f.x, f.y);
            }
          } else {                            // bf16 after the latent (per block: after its scales too)
            const uint4* src = reinterpret_cast<const uint4*>(row + (kMode == kExBf16 ? kDc * 2 : kDc + 16));
#pragma unroll
            for (int i = 0; i < kDr / 8; ++i) d[i] = src[i];
          }
        } else {
#pragma unroll
          for (int i = 0; i < kDr / 8; ++i) d[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      ++v;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ attention
constexpr int kAtThreads = 256;        // warps 0-3 query RoPE + softmax + epilogue, 4 K / 5 V
                                       // producers, 6 QK^T / 7 P V issuers
constexpr int kWarpK = 4, kWarpV = 5, kWarpMma = 6, kWarpPv = 7;
constexpr int kOffQ = 0;                               // q_nope 0..63, q_nope 64..127, q_pe: 3 boxes
constexpr int kOffK = 3 * kBox;                        // 2 stages x (k_nope 0..63, 64..127, k_r)
constexpr int kOffV = kOffK + 2 * 3 * kBox;            // 2 stages x (v 0..63, 64..127)
constexpr int kOffBars = kOffV + 2 * 2 * kBox;
constexpr int kAtSmem = kOffBars + 1024 + 1024;
constexpr uint32_t kTmO = 0, kTmS = 128, kTmP = 384;   // TMEM columns
constexpr float kRescaleLog2 = 8.0f;                   // rescale O when the row maximum grows by > 2^8

struct AtBars {
  uint64_t qfull;            // the item's queries landed                    (K producer, tx)
  uint64_t qready;           // their RoPE part rotated in shared memory     (4 softmax warps)
  uint64_t qfree;            // every QK^T of the item done: the query buffer may be refilled
  uint64_t kfull[2], kempty[2], vfull[2], vempty[2];
  uint64_t sfull[2], sfree[2], pfull[2], pdone[2];
  uint64_t ofinal;           // the item's last P V done                     (MMA commit)
  uint64_t ofree;            // the epilogue has read O                      (4 softmax warps)
  uint64_t qkdrain, pvdrain;
  uint64_t item_full[4];     // ring entry written by the scheduling thread (the K producer)
  uint64_t item_free[4];     // ring entry read by the other six roles
  int ring[4];               // item indices handed out to this CTA, in order (-1: no more)
  uint32_t tmem_base;
  int abort;
};
constexpr int kRingReaders = 7;        // V producer, QK^T warp, P V issuer, 4 softmax warps

// The next item of a role that reads the ring: n-th entry, -1 when there are no more, -2 when
// a wait ran out (or another role aborted).  `arrive` is set on one thread per role.
__device__ __forceinline__ int at_next(AtBars* bars, int n, bool arrive, volatile int* abort_flag) {
  const int slot = n & 3;
  if (!mbar_wait(smem_u32(&bars->item_full[slot]), (n >> 2) & 1, abort_flag)) return -2;
  const int idx = *reinterpret_cast<volatile int*>(&bars->ring[slot]);
  if (arrive) mbar_arrive(smem_u32(&bars->item_free[slot]));
  return idx;
}

// Whether an item loop goes on with `idx`; a failed wait (-2) also clears ok.
__device__ __forceinline__ bool at_more(int idx, bool& ok) {
  if (idx == -2) ok = false;
  return idx >= 0;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum of 128 values (float bits) as a tree of three-input maxima, depth 5.
__device__ __forceinline__ float max128(const uint32_t (&x)[kTile]) {
  float a[44], b[15], c[5];
#pragma unroll
  for (int i = 0; i < 42; ++i)
    a[i] = max3(__uint_as_float(x[3 * i]), __uint_as_float(x[3 * i + 1]), __uint_as_float(x[3 * i + 2]));
  a[42] = __uint_as_float(x[126]);
  a[43] = __uint_as_float(x[127]);
#pragma unroll
  for (int i = 0; i < 14; ++i) b[i] = max3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[14] = fmaxf(a[42], a[43]);
#pragma unroll
  for (int i = 0; i < 5; ++i) c[i] = max3(b[3 * i], b[3 * i + 1], b[3 * i + 2]);
  return max3(max3(c[0], c[1], c[2]), c[3], c[4]);
}

__device__ __forceinline__ void at_fail(AtBars* bars, unsigned* check) {
  if (atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
}

// One attention item: 128 queries of one head of one sequence.  Items are numbered with the
// query block fastest (longest first), then the head, then the sequence, so the items in work
// at the same time share a head's keys and values in L2.  Every role of the CTA derives the
// same description from the same inputs.
struct AtItem {
  int b, h, qs, nq, L, r0, nrows, p_first, n_kt;
  bool rows_ok;              // q_start / q_len fit the query rows: outputs may be written
  bool live;                 // a valid item with queries: every role takes part
  bool zero;                 // queries of a sequence with an invalid length: zero rows only
};

__device__ __forceinline__ AtItem at_item(int idx, int nqb, int n_h, const int32_t* q_start, const int32_t* q_len,
                                          int total_q, int max_q, const int32_t* ctx_len, int max_ctx) {
  AtItem it;
  const int qb = nqb - 1 - idx % nqb;
  it.h = (idx / nqb) % n_h;
  it.b = idx / (nqb * n_h);
  it.L = ctx_len[it.b];
  it.nq = q_len[it.b];
  it.qs = q_start[it.b];
  it.rows_ok = it.nq >= 0 && it.nq <= max_q && it.qs >= 0 && (long long)it.qs + it.nq <= total_q;
  const bool seq_ok = it.rows_ok && it.L >= 1 && it.L <= max_ctx && it.nq <= it.L;
  it.r0 = qb * kQBlk;
  const bool has_rows = it.rows_ok && it.r0 < it.nq;
  it.nrows = has_rows ? min(kQBlk, it.nq - it.r0) : 0;
  it.live = has_rows && seq_ok;
  it.zero = has_rows && !seq_ok;
  it.p_first = it.live ? it.L - it.nq + it.r0 : 0;
  it.n_kt = it.live ? (it.p_first + it.nrows - 1 + kTile) / kTile : 0;   // key tiles 0 .. n_kt - 1
  return it;
}

// Persistent: each CTA takes the next item from a global counter (longest query blocks of a head
// first, a head's blocks together) and hands it to its roles through a 4-entry ring in shared
// memory, so a CTA that finishes early takes more work.  The key/value rings, the score buffers
// and their barriers run on across items (a global tile count g); the next item's queries load
// as soon as the previous item's last QK^T is done and the softmax warps rotate their RoPE part
// before the previous item's epilogue, so the next item's QK^T overlaps that epilogue; its first
// P V waits only for the epilogue to have read O.
__global__ void __launch_bounds__(kAtThreads, 1)
prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kn,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kr,
                    const int32_t* __restrict__ q_start, const int32_t* __restrict__ q_len, int total_q, int max_q,
                    const int32_t* __restrict__ ctx_len, int n_h, int max_ctx, const int32_t* __restrict__ block_table,
                    int bt_stride, int num_pages, const float2* __restrict__ rope_cs, int max_position,
                    float scale_log2, int lpad, int nqb, int n_items, int* sched, __nv_bfloat16* __restrict__ out,
                    int stall, unsigned* check) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  AtBars* bars = reinterpret_cast<AtBars*>(smem + kOffBars);
  volatile int* abort_flag = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(smem_u32(&bars->qfull), 1);
    mbar_init(smem_u32(&bars->qready), 4);
    mbar_init(smem_u32(&bars->qfree), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->kfull[i]), 1);
      mbar_init(smem_u32(&bars->kempty[i]), 1);
      mbar_init(smem_u32(&bars->vfull[i]), 1);
      mbar_init(smem_u32(&bars->vempty[i]), 1);
      mbar_init(smem_u32(&bars->sfull[i]), 1);
      mbar_init(smem_u32(&bars->sfree[i]), 4);
      mbar_init(smem_u32(&bars->pfull[i]), 4);
      mbar_init(smem_u32(&bars->pdone[i]), 1);
    }
    mbar_init(smem_u32(&bars->ofinal), 1);
    mbar_init(smem_u32(&bars->ofree), 4);
    mbar_init(smem_u32(&bars->qkdrain), 1);
    mbar_init(smem_u32(&bars->pvdrain), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&bars->item_full[i]), 1);
      mbar_init(smem_u32(&bars->item_free[i]), kRingReaders);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) { tmem_alloc(smem_u32(&bars->tmem_base), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  griddep_wait();                                      // the expanded keys and values
  griddep_launch_dependents();
// item loops of the ring readers: one thread (AT_ITEMS_T) or a whole warp whose lane 0 reads the
// entry and broadcasts it (AT_ITEMS_W); a failed wait ends the loop with ok = false
#define AT_ITEMS_T for (int n = 0, idx = 0; at_more(idx = at_next(bars, n, true, abort_flag), ok); ++n)
#define AT_ITEMS_W                                                                                      \
  for (int n = 0, idx = 0;                                                                              \
       at_more(idx = __shfl_sync(0xffffffffu, lane == 0 ? at_next(bars, n, true, abort_flag) : 0, 0), ok); ++n)
#define AT_ITEM() at_item(idx, nqb, n_h, q_start, q_len, total_q, max_q, ctx_len, max_ctx)

  if (warp == kWarpK) {
    // ---------------------------------------------------------------- queries, then the key tiles
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_kn);
      prefetch_tmap(&tm_kr);
      prefetch_tmap(&tm_v);
      int g = 0, u = 0;
      bool ok = true;
      for (int n = 0;; ++n) {
        // the scheduler: the next item from the global counter into ring entry n % 4, once the
        // six other roles have read that entry's previous item
        const int slot = n & 3;
        if (n >= 4 && !mbar_wait(smem_u32(&bars->item_free[slot]), ((n >> 2) - 1) & 1, abort_flag)) { ok = false; break; }
        int idx = atomicAdd(sched, 1);
        if (idx >= n_items) idx = -1;
        *reinterpret_cast<volatile int*>(&bars->ring[slot]) = idx;
        mbar_arrive(smem_u32(&bars->item_full[slot]));
        if (idx < 0) break;
        const AtItem it = AT_ITEM();
        if (!it.live) continue;
        // into L2 now (about two key tiles before the previous item ends): this item's queries,
        // which come from HBM, and its first key and value tiles
        for (int c = 0; c < 3; ++c) tma_prefetch_3d(&tm_q, 64 * c, it.h, it.qs + it.r0);
        {
          const int row0 = (it.b * n_h + it.h) * lpad;
          tma_prefetch_2d(&tm_kn, 0, row0);
          tma_prefetch_2d(&tm_kn, 64, row0);
          tma_prefetch_2d(&tm_kr, 0, it.b * lpad);
          tma_prefetch_2d(&tm_v, 0, row0);
          tma_prefetch_2d(&tm_v, 64, row0);
        }
        // the previous item's QK^T are done with the query buffer
        if (u >= 1 && !mbar_wait(smem_u32(&bars->qfree), (u - 1) & 1, abort_flag)) { ok = false; break; }
        const uint32_t qf = smem_u32(&bars->qfull);
        mbar_arrive_expect_tx(qf, 3 * kBox);
        for (int c = 0; c < 3; ++c) tma_load_3d(sbase + kOffQ + c * kBox, &tm_q, 64 * c, it.h, it.qs + it.r0, qf);
        ++u;
        const int kv_row0 = (it.b * n_h + it.h) * lpad;
        for (int j = 0; j < it.n_kt; ++j, ++g) {
          const int s = g & 1;
          if (g >= 2 && !mbar_wait(smem_u32(&bars->kempty[s]), ((g - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
          const uint32_t st = sbase + kOffK + s * 3 * kBox, fb = smem_u32(&bars->kfull[s]);
          mbar_arrive_expect_tx(fb, 3 * kBox);
          tma_load_2d(st, &tm_kn, 0, kv_row0 + kTile * j, fb);
          tma_load_2d(st + kBox, &tm_kn, 64, kv_row0 + kTile * j, fb);
          // (a test of the bounded waits, stall == 5: the CTA that takes the item of sequence 0, head
          // 0, first query block never loads the RoPE-key box of its first key tile, so that tile's
          // barrier, armed for every byte, cannot complete)
          if (!(stall == 5 && it.b == 0 && it.h == 0 && it.r0 == 0 && j == 0))
            tma_load_2d(st + 2 * kBox, &tm_kr, 0, it.b * lpad + kTile * j, fb);
        }
        if (!ok) break;
      }
      if (!ok) at_fail(bars, check);
      volatile int never = 0;                          // every copy lands before exit
      if (u >= 1) mbar_wait(smem_u32(&bars->qfull), (u - 1) & 1, &never);
      for (int k = max(0, g - 2); k < g; ++k) mbar_wait(smem_u32(&bars->kfull[k & 1]), (k >> 1) & 1, &never);
    }
  } else if (warp == kWarpV) {
    // ---------------------------------------------------------------- value tiles
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      int g = 0;
      bool ok = true;
      AT_ITEMS_T {
        const AtItem it = AT_ITEM();
        if (!it.live) continue;
        const int kv_row0 = (it.b * n_h + it.h) * lpad;
        for (int j = 0; j < it.n_kt; ++j, ++g) {
          const int s = g & 1;
          if (g >= 2 && !mbar_wait(smem_u32(&bars->vempty[s]), ((g - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
          const uint32_t st = sbase + kOffV + s * 2 * kBox, fb = smem_u32(&bars->vfull[s]);
          mbar_arrive_expect_tx(fb, 2 * kBox);
          tma_load_2d(st, &tm_v, 0, kv_row0 + kTile * j, fb);
          tma_load_2d(st + kBox, &tm_v, 64, kv_row0 + kTile * j, fb);
        }
        if (!ok) break;
      }
      if (!ok) at_fail(bars, check);
      volatile int never = 0;
      for (int k = max(0, g - 2); k < g; ++k) mbar_wait(smem_u32(&bars->vfull[k & 1]), (k >> 1) & 1, &never);
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- QK^T issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      const uint64_t qd = sdesc_sw128(sbase + kOffQ, 16, 1024);
      int g = 0, u = 0;
      bool ok = true;
      AT_ITEMS_T {
        const AtItem it = AT_ITEM();
        if (!it.live) continue;
        if (!mbar_wait(smem_u32(&bars->qready), u & 1, abort_flag)) { ok = false; break; }   // rotated queries
        for (int j = 0; j < it.n_kt; ++j, ++g) {
          const int s = g & 1;
          // K(g) has landed and the score buffer's previous tile, g - 2, has been read
          if (!mbar_wait(smem_u32(&bars->kfull[s]), (g >> 1) & 1, abort_flag) ||
              (g >= 2 && !mbar_wait(smem_u32(&bars->sfree[s]), ((g - 2) >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = sdesc_sw128(sbase + kOffK + s * 3 * kBox, 16, 1024);
#pragma unroll
          for (int k = 0; k < kDq / 16; ++k) {  // box k / 4 (k_nope, k_nope, k_r), 32-byte step k % 4
            const uint64_t off = (uint64_t)(((k >> 2) * kBox + (k & 3) * 32) >> 4);
            mma_ss(tmem + kTmS + 128 * s, qd + off, kd + off, idesc_qk, k > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars->sfull[s]));
          mma_commit(smem_u32(&bars->kempty[s]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->qfree));            // the item's QK^T are done with the queries
        ++u;
      }
      if (!ok) at_fail(bars, check);
      mma_commit(smem_u32(&bars->qkdrain));            // every QK^T issued above has finished ...
      volatile int never = 0;
      mbar_wait(smem_u32(&bars->qkdrain), 0, &never);  // ... before the CTA frees its TMEM
    }
  } else if (warp == kWarpPv) {
    // ---------------------------------------------------------------- P V issuer (its own thread:
    // a P V never waits behind a QK^T issue; the two write disjoint TMEM, O and P against S)
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
      int g = 0, u = 0;
      bool ok = true;
      AT_ITEMS_T {
        const AtItem it = AT_ITEM();
        if (!it.live) continue;
        for (int j = 0; j < it.n_kt; ++j, ++g) {
          const int s = g & 1;
          if (!mbar_wait(smem_u32(&bars->pfull[s]), (g >> 1) & 1, abort_flag) ||
              !mbar_wait(smem_u32(&bars->vfull[s]), (g >> 1) & 1, abort_flag) ||
              (j == 0 && u >= 1 && !mbar_wait(smem_u32(&bars->ofree), (u - 1) & 1, abort_flag))) {
            ok = false;                                // (j == 0: the previous item's O has been read)
            break;
          }
          tc_fence_after();
          // V tile: 128 key rows (K) x 128 value columns (N) in two 64-column boxes, MN-major
          const uint64_t vd = sdesc_sw128(sbase + kOffV + s * 2 * kBox, kBox, 1024);
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_ts(tmem + kTmO, tmem + kTmP + 64 * s + 8 * k, vd + (uint64_t)(128 * k), idesc_pv,
                   (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(smem_u32(&bars->vempty[s]));
          mma_commit(smem_u32(&bars->pdone[s]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->ofinal));
        ++u;
      }
      if (!ok) at_fail(bars, check);
      mma_commit(smem_u32(&bars->pvdrain));            // every P V issued above has finished
      volatile int never = 0;
      mbar_wait(smem_u32(&bars->pvdrain), 0, &never);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- query RoPE, softmax, epilogue:
    // thread = query row.  The warps rotate the next live item's queries as soon as they have
    // written the current item's last P, before its epilogue, so the next item's QK^T overlaps
    // the epilogue (one row per thread: each row's (cos, sin) in 16-byte loads, all in flight).
    const int r = 32 * warp + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    int g = 0, u = 0, n = 0;
    bool ok = true;
    // the next live item from the ring; queries of a sequence with a bad length are zeroed (and
    // flagged) on the way; false at the end of the work or on a failed wait
    auto next_live = [&](AtItem& it) -> bool {
      while (true) {
        const int idx = __shfl_sync(0xffffffffu, lane == 0 ? at_next(bars, n, true, abort_flag) : 0, 0);
        ++n;
        if (!at_more(idx, ok)) return false;
        it = AT_ITEM();
        if (it.zero || (!it.rows_ok && it.r0 == 0 && it.h == 0)) {
          if (r == 0) atomicOr(check, kCheckCtxLen);
          if (it.zero && r < it.nrows) {
            uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)(it.qs + it.r0 + r) * n_h + it.h) * kDv);
#pragma unroll
            for (int i = 0; i < kDv / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        if (it.live) return true;
      }
    };
    // row r's q_pe of live item number uu rotated in place at its position once the queries have
    // landed (swizzled box: chunk c at c ^ (r & 7))
    auto rotate = [&](const AtItem& it, int uu) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->qfull), uu & 1, abort_flag))) return false;
      const int lim = min(it.p_first + r, it.L - 1);    // rows past the block clamp (never stored)
      uint8_t* row = smem + kOffQ + 2 * kBox + r * 128;
      const float4* cs = reinterpret_cast<const float4*>(rope_cs + (size_t)min(lim, max_position - 1) * (kDr / 2));
      float4 cv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) cv[i] = cs[i];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4* p = reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4));
        const uint4 v = *p;
        const float2 cc[4] = {make_float2(cv[2 * c].x, cv[2 * c].y), make_float2(cv[2 * c].z, cv[2 * c].w),
                              make_float2(cv[2 * c + 1].x, cv[2 * c + 1].y), make_float2(cv[2 * c + 1].z, cv[2 * c + 1].w)};
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float y0, y1;
          rope_pair(bf16_lo(w[i]), bf16_hi(w[i]), cc[i], &y0, &y1);
          w[i] = pack_bf16(y0, y1);
        }
        *p = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();                          // the rotated rows, before the MMAs read them
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->qready));
      return true;
    };
    AtItem it;
    bool have = next_live(it);
    if (have && !rotate(it, 0)) { ok = false; have = false; }
    while (have) {
      // every page the item's keys come from must be a valid page id (else zero output rows)
      bool bad = false;
      const int npages = (it.p_first + it.nrows - 1 + kPage) / kPage;
      for (int i = lane; i < npages; i += 32) bad |= !page_ok(block_table[(size_t)it.b * bt_stride + i], num_pages);
      bad = __any_sync(0xffffffffu, bad);
      if (bad && r == 0) atomicOr(check, kCheckPageId);
      const int lim = min(it.p_first + r, it.L - 1);      // last visible key of this row
      float m_ref = -INFINITY, l = 0.0f;
      for (int j = 0; j < it.n_kt; ++j, ++g) {
        const int s = g & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->sfull[s]), (g >> 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t x[kTile];                               // scores, then scaled base-2 logits (float bits)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tmem_ld32(tmem + lane_off + kTmS + 128 * s + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&x[32 * q]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->sfree[s]));
        if (kTile * j + kTile - 1 > it.p_first) {        // a tile on the diagonal: hide keys past the row
#pragma unroll
          for (int c = 0; c < kTile; ++c)
            if (kTile * j + c > lim) x[c] = __float_as_uint(-INFINITY);
        }
        // the scale is positive, so the maximum of the raw scores gives the scaled one
        const float m_new = fmaxf(m_ref, max128(x) * scale_log2);
        if (__any_sync(0xffffffffu, m_new > m_ref + kRescaleLog2)) {
          const float alpha = ex2_approx(m_ref - m_new);
          l *= alpha;
          m_ref = m_new;
          if (j > 0) {                                   // O holds P V of the item's tiles < j: rescale it
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pdone[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const float2 al2 = make_float2(alpha, alpha);
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
              uint32_t o[32];
              tmem_ld32(tmem + lane_off + kTmO + 32 * q, o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), al2);
                o[2 * i] = __float_as_uint(v.x);
                o[2 * i + 1] = __float_as_uint(v.y);
              }
              tmem_st32(tmem + lane_off + kTmO + 32 * q, o);
            }
            tmem_st_wait();
          }
        }
        if (g >= 2) {                                    // P V(g - 2) has read this P buffer
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pdone[s]), ((g - 2) >> 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
        }
        // p = 2^(score * scale_log2 - m): one packed FMA per pair, four independent partial sums
        const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-m_ref, -m_ref);
        float2 ps[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ps[i] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 d = __ffma2_rn(make_float2(__uint_as_float(x[64 * hf + 2 * c]),
                                                    __uint_as_float(x[64 * hf + 2 * c + 1])), sc2, nm2);
            const float2 pp = make_float2(ex2_approx(d.x), ex2_approx(d.y));
            ps[c & 3] = __fadd2_rn(ps[c & 3], pp);
            pk[c] = bf16x2(pp.x, pp.y);
          }
          tmem_st32(tmem + lane_off + kTmP + 64 * s + 32 * hf, pk);
        }
        const float2 sum2 = __fadd2_rn(__fadd2_rn(ps[0], ps[1]), __fadd2_rn(ps[2], ps[3]));
        l += sum2.x + sum2.y;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->pfull[s]));
      }
      if (!ok) break;
      // the next live item's queries, rotated before this item's epilogue
      AtItem nxt;
      const bool have_next = next_live(nxt);
      if (!ok) break;
      if (have_next && !rotate(nxt, u + 1)) { ok = false; break; }
      // ---------------------------------------------------------------- epilogue of the item
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->ofinal), u & 1, abort_flag)) && !*abort_flag;
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;      // (a bad page id: zero rows)
      uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)(it.qs + it.r0 + r) * n_h + it.h) * kDv);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kTmO + 32 * q, o);
        tmem_ld_wait();
        if (r < it.nrows) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {                  // whole 32-byte sectors of this row
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = bad ? 0u : bf16x2(__uint_as_float(o[16 * i + 2 * e]) * inv, __uint_as_float(o[16 * i + 2 * e + 1]) * inv);
            st_global_32B(dst + 4 * q + 2 * i, w);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->ofree));   // the next item's first P V may overwrite O
      ++u;
      it = nxt;
      have = have_next;
    }
    if (!ok) at_fail(bars, check);
  }
#undef AT_ITEMS_T
#undef AT_ITEMS_W
#undef AT_ITEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
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

// bf16 matrix [rows][width] with boxes of 64 columns x 128 rows, 128-byte swizzle.
cudaError_t rows_map_2d(const void* base, long long rows, int width, CUtensorMap* m) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

// Queries [total_q][n_h][192] bf16 as (column, head, row): boxes of 64 columns x 1 head x 128 rows
// (rows past total_q read as zeros).
cudaError_t query_map(const void* q, int total_q, int n_h, CUtensorMap* m) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kDq, (cuuint64_t)n_h, (cuuint64_t)total_q};
  const cuuint64_t strides[2] = {(cuuint64_t)kDq * 2, (cuuint64_t)kDq * 2 * n_h};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kQBlk};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

int padded_ctx(int max_ctx) { return (max_ctx + kTile - 1) / kTile * kTile; }

}  // namespace

// Workspace of a prefill: K_nope and V [B][n_h][lpad][128] and K_r [B][lpad][64], bf16,
// lpad = max_ctx rounded up to 128 tokens, then the attention kernel's work counter.
size_t prefill_workspace_bytes(int n_h, int batch, int max_ctx) {
  return (size_t)batch * padded_ctx(max_ctx) * (2 * (size_t)n_h * kDn + kDr) * 2 + 256;   // + the work counter
}

cudaError_t launch_prefill(const Handle& h, const void* q, const int32_t* q_start, const int32_t* q_len, int total_q,
                           int max_q, const int32_t* ctx_len, int batch, int max_ctx, const int32_t* block_table,
                           int bt_stride, const void* cache, int num_pages, void* workspace, void* out,
                           cudaStream_t st, cudaEvent_t between) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(expand_tc_kernel<kExBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         ex_smem<kExBf16>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(expand_tc_kernel<kExFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize, ex_smem<kExFp8>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(expand_tc_kernel<kExFp8Block>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               ex_smem<kExFp8Block>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAtSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaError_t e = cache_maps(h, cache, num_pages);
  if (e != cudaSuccess) return e;
  const int n_h = h.cfg.n_h, lpad = padded_ctx(max_ctx);
  __nv_bfloat16* kn = static_cast<__nv_bfloat16*>(workspace);
  __nv_bfloat16* vv = kn + (size_t)batch * n_h * lpad * kDn;
  __nv_bfloat16* kr = vv + (size_t)batch * n_h * lpad * kDv;
  int* sched = reinterpret_cast<int*>(kr + (size_t)batch * lpad * kDr);   // 256-byte aligned: every region is
  alignas(64) CUtensorMap tm_q, tm_kn, tm_v, tm_kr;
  if ((e = query_map(q, total_q, n_h, &tm_q)) != cudaSuccess) return e;
  if ((e = rows_map_2d(kn, (long long)batch * n_h * lpad, kDn, &tm_kn)) != cudaSuccess) return e;
  if ((e = rows_map_2d(vv, (long long)batch * n_h * lpad, kDv, &tm_v)) != cudaSuccess) return e;
  if ((e = rows_map_2d(kr, (long long)batch * lpad, kDr, &tm_kr)) != cudaSuccess) return e;
  const int n_items = n_h * (lpad / kTile) * batch;
  const CUtensorMap& tm_cache = *reinterpret_cast<const CUtensorMap*>(h.tmap);
  const CUtensorMap& tm_wuk = *reinterpret_cast<const CUtensorMap*>(h.tmap_wuk);
  const CUtensorMap& tm_wuv = *reinterpret_cast<const CUtensorMap*>(h.tmap_wuv);
  const CUtensorMap& tm_scale = *reinterpret_cast<const CUtensorMap*>(h.tmap_scale);
  const uint8_t* cache8 = static_cast<const uint8_t*>(cache);
  const dim3 ex_grid(min(n_items, h.num_sms));
  if (h.cfg.cache_dtype == MLA_CACHE_FP8_E4M3)
    e = launch_pdl(expand_tc_kernel<kExFp8>, ex_grid, dim3(ex_threads<kExFp8>()), ex_smem<kExFp8>(), st, tm_cache,
                   tm_wuk, tm_wuv, tm_scale, cache8, h.cfg.fp8_scale, ctx_len, n_h, max_ctx, block_table, bt_stride,
                   num_pages, lpad, n_items, kn, vv, kr, sched, h.test_stall, h.check_word);
  else if (h.cfg.cache_dtype == MLA_CACHE_FP8_E4M3_BLOCK)
    e = launch_pdl(expand_tc_kernel<kExFp8Block>, ex_grid, dim3(ex_threads<kExFp8Block>()), ex_smem<kExFp8Block>(), st,
                   tm_cache, tm_wuk, tm_wuv, tm_scale, cache8, 1.0f, ctx_len, n_h, max_ctx, block_table, bt_stride,
                   num_pages, lpad, n_items, kn, vv, kr, sched, h.test_stall, h.check_word);
  else
    e = launch_pdl(expand_tc_kernel<kExBf16>, ex_grid, dim3(ex_threads<kExBf16>()), ex_smem<kExBf16>(), st, tm_cache,
                   tm_wuk, tm_wuv, tm_scale, cache8, 1.0f, ctx_len, n_h, max_ctx, block_table, bt_stride, num_pages,
                   lpad, n_items, kn, vv, kr, sched, h.test_stall, h.check_word);
  if (e != cudaSuccess) return e;
  if (between && (e = cudaEventRecord(between, st)) != cudaSuccess) return e;   // profiling: splits the two kernels
  const float scale_log2 = h.scale * 1.4426950408889634f;
  const int nqb = (max_q + kQBlk - 1) / kQBlk, n_att = nqb * n_h * batch;
  return launch_pdl(prefill_attn_kernel, dim3(min(n_att, h.num_sms)), dim3(kAtThreads), kAtSmem, st,
                    tm_q, tm_kn, tm_v, tm_kr, q_start, q_len, total_q, max_q, ctx_len, n_h, max_ctx, block_table,
                    bt_stride, num_pages, (const float2*)h.rope_cs, h.cfg.max_position, scale_log2, lpad, nqb, n_att,
                    sched, static_cast<__nv_bfloat16*>(out), h.test_stall, h.check_word);
}

}  // namespace mla
