// decode_tc.cu -- split-KV flash decode over the paged 576-wide latent cache on
// the 5th-generation tensor cores (tcgen05 + Tensor Memory), TMA-fed.
//
// What one work unit computes (a page range of one sequence, all heads):
//   s_t    = scale * ( q_lat[h] . c_t + q_pe'[h] . k_r,t )                 t in the unit
//   o[h]   = sum_t softmax(s)_t c_t, with the unit's log-sum-exp when split
// ("DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2-§2.4: the
// absorbed query is scored against the shared latent row, and the softmax
// weights sum latent rows; "G5 MLA KV 访存建模设计规格" 附录 B: the KV stream is
// consumed as it arrives -- flash decode).
//
// Design (one 2-CTA cluster per unit; heads are the 128-row M dimension, so one
// cache tile serves every head of the sequence):
//   * The 576 columns are split between the two CTAs of the cluster:
//       CTA 0: latent columns [0, 256)   and RoPE-key columns [512, 544)
//       CTA 1: latent columns [256, 512) and RoPE-key columns [544, 576)
//     Each CTA TMA-loads only its columns of every 64-token page (32 KB of latent
//     in 128-byte-swizzled boxes, 4 KB of RoPE key in a 64-byte-swizzled box) into
//     a 4-deep ring, so the pair reads each cache byte from HBM once and both CTAs
//     carry the same QK^T work.
//   * QK^T is split along K: each CTA computes a partial score tile
//       S_r[128 heads x 64 tokens] = Q_r . C_r^T
//     with Q_r's latent part resident in TMEM (A operand) and its half of the
//     RoPE query in shared memory.  Two groups of four warps take the tiles in
//     turn (group j % 2 takes tile j; thread = head = TMEM lane).  A group reads
//     S_r as soon as it lands, scales it to the base-2 softmax domain, rounds it
//     to fp16, stages it in a free receive slot of its own CTA and moves it into
//     the peer's receive slot with one 4 KB bulk copy per warp (16 KB per tile
//     each way, 4 slots): under load, bulk copies move distributed shared memory
//     faster than 16-byte remote stores.  It then forms x = x_own + fp16(x_peer);
//     fp16 keeps 11 bits of a logit, finer than the bf16 P it feeds.  The two CTAs'
//     logits agree up to that rounding, and each normalises its half of the output
//     with its own sum.  One tile's chain (read, send, wait for the peer, softmax,
//     write P) is longer than the QK^T that feeds it; two groups run two chains at
//     once, handing the running max from tile to tile through shared memory and
//     keeping separate sums, reconciled at the end.
//   * P (bf16) is written into one of two P slots in TMEM and used as the A operand
//     of O_r[128 x 256] += P . C_r[64 tokens x 256 latent]; the same shared-memory
//     tile is the B operand, read MN-major.  Each CTA accumulates its half of
//     the latent output in TMEM (256 columns).
//   * TMEM per CTA (512 columns): O_r [0,256), Q_r [256,384), S [384,448), P slots
//     [448,480) and [480,512).  The score buffer is free as soon as the tile's
//     group has loaded it, so QK^T of tile j+1 is issued when tile j's
//     softmax starts, not when it ends; P(j) keeps its own slot until P . C reads it.
//   * Online softmax in the base-2 domain with a lazy rescale: the running max
//     only moves (and O is rescaled in TMEM) when a tile's max exceeds it by more
//     than 8, so P <= 2^8.
//   * Warp roles per CTA: warps 0-3 and 4-7 the two tile groups (score exchange,
//     softmax, epilogue), warp 8 TMA producer, warp 9 issues QK^T, warp 10 issues
//     P . C; with an FP8 cache, warps 11-15 convert each tile to bf16 in place, one box each.
//     Every wait is bounded; on a timeout the kernel sets MLA_CHECK_TIMEOUT,
//     drains and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_fp16.h>

#include "append_ops.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kStagesMax = 4;              // cache tiles in flight per CTA (3 with FP8 MMAs)
constexpr int kChunkBytes = kPage * 128;   // one 64-token x 64-column bf16 box (SW128): 8 KB
constexpr int kRopeBytes = kPage * 64;     // one 64-token x 32-column bf16 box of the RoPE key (SW64): 4 KB
constexpr int kScaleBytes = kPage * 16;   // per-block FP8 cache: the 4 fp32 block scales of 64 tokens: 1 KB
constexpr int kQpeBytes = kMaxHeads * 64;              // 128 heads x 32 bf16 of the RoPE query, SW64 K-major
constexpr int kSlots = 4;                              // partial-score receive slots
constexpr int kSlotBytes = kMaxHeads * kPage * 2;      // 128 x 64 fp16 = 16 KB
constexpr int kXchgBytes = 3 * 2 * kMaxHeads * 4;      // running maxima / final sums of the two tile groups
constexpr int kThreads = 352;                          // 2 tile groups of 4 warps, producer, 2 MMA warps
constexpr int kThreadsFp8 = 512;                       // + 5 FP8 conversion warps (4 for the per-block format)
constexpr int kThreadsFp8Mma = 512;                    // + 4 warps transposing tiles, 1 converting the RoPE key
// cache modes of the kernel: bf16 rows, e4m3 rows with one tensor scale (converted to bf16 in shared
// memory, or used as they are by FP8 MMAs), per-block e4m3 rows
constexpr int kModeBf16 = 0, kModeFp8 = 1, kModeFp8Block = 2, kModeFp8Mma = 3;
// FP8 MMAs (kind::f8f6f4): the latent codes are the B operand of QK^T as stored; P . C reads P in
// e4m3 and a copy of the tile's latent codes transposed to token-contiguous rows (every operand
// K-major in shared memory)
constexpr int kCodeBox = kPage * 128;        // 64 tokens x 128 e4m3 codes, 128-byte swizzle: 8 KB
constexpr int kCtBytes = 256 * kPage;        // 256 latent columns x 64 token codes, 64-byte swizzle: 16 KB
constexpr int kQ8Bytes = kMaxHeads * 256;    // e4m3 latent query: two boxes of 128 heads x 128 codes (SW128)
constexpr int kP8Bytes = kMaxHeads * kPage;  // e4m3 P of one tile: 128 heads x 64 codes (SW64): 8 KB

// Shared-memory layout of a kernel mode (offsets from the 1024-byte aligned base).
template <int kMode>
struct Smem {
  static constexpr bool kMma8 = kMode == kModeFp8Mma;
  static constexpr int kStages = kMma8 ? 3 : 4;
  // a stage: the bf16 latent chunks (or two code boxes), the RoPE key in bf16, per-block scales
  // (FP8 MMAs: two code boxes, the RoPE key in bf16, then its 2 KB of codes, converted out of place)
  static constexpr int kStage = kMma8 ? 2 * kCodeBox + kRopeBytes + kRopeBytes / 2
                                      : 4 * kChunkBytes + kRopeBytes + kScaleBytes;
  static constexpr int kRopeOff = kMma8 ? 2 * kCodeBox : 4 * kChunkBytes;   // RoPE box inside a stage
  static constexpr int kRopeCodeOff = kMma8 ? 2 * kCodeBox + kRopeBytes : kRopeOff + kRopeBytes / 2;
  static constexpr int kOffCt = kStages * kStage;                           // two transposed-tile buffers
  static constexpr int kOffQ8 = kOffCt + (kMma8 ? 2 * kCtBytes : 0);
  static constexpr int kOffQpe = kOffQ8 + (kMma8 ? kQ8Bytes : 0);
  static constexpr int kOffRecv = kOffQpe + kQpeBytes;
  static constexpr int kOffP8 = kOffRecv + kSlots * kSlotBytes;              // two e4m3 P slots
  static constexpr int kOffBars = kOffP8 + (kMma8 ? 2 * kP8Bytes : 0);
  static constexpr int kOffXchg = kOffBars + 1024;
  static constexpr int kBytes = kOffXchg + kXchgBytes + 1024;                // + alignment slack
  static_assert(kBytes <= 232448, "the largest dynamic shared memory a CTA may opt into (227 KB)");
  static_assert(kOffQ8 >= 8 * 2 * 4096, "the epilogue stages its output in the first 64 KB");
  static_assert(kOffCt % 1024 == 0 && kOffQ8 % 1024 == 0 && kOffP8 % 1024 == 0 && kStage % 1024 == 0, "atoms");
};
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;                            // QK^T issuer (allocates TMEM)
constexpr int kWarpPv = 10;                            // P . C issuer
constexpr int kWarpConv = 11;                          // FP8 cache: warps 11-15 convert tiles

// TMEM column map
constexpr uint32_t kTmO = 0;
constexpr uint32_t kTmQ = 256;
constexpr uint32_t kTmS = 384;             // 64 columns of fp32 partial scores
constexpr uint32_t kTmP = 448;             // P slot b (64 bf16 per lane) at kTmP + 32 b

struct Bars {                               // mbarriers (8 bytes each) and flags
  uint64_t full[kStagesMax];                // TMA tile landed                      (producer, tx)
  uint64_t conv[kStagesMax];                // FP8 cache: tile converted to bf16    (5 or 4 conversion warps;
                                            //   FP8 MMAs: the RoPE key converted, 1 warp)
  uint64_t empty[kStagesMax];               // tile consumed by P . C               (MMA commit; FP8 MMAs:
                                            //   QK^T done (MMA commit) and the tile transposed (4 warps))
  uint64_t tready[2];                       // FP8 MMAs: tile j transposed into buffer j % 2 (4 warps)
  uint64_t sfull[2];                        // S_r(j) in TMEM, tile group j % 2     (MMA commit)
  uint64_t sfree[2];                        // S_r(j) loaded by its tile group      (4 warps)
  uint64_t mready[2];                       // a group's running max published     (4 warps)
  uint64_t efin;                            // single phase: both groups' sums out  (8 warps)
  uint64_t pfull[2];                        // P(j) written into P slot j % 2       (4 warps)
  uint64_t pdone[2];                        // P . C of a tile in P slot b done     (MMA commit)
  uint64_t ofinal;                          // single phase: the last P . C landed  (MMA commit)
  uint64_t qfull;                           // single phase: the absorbed query landed (producer, tx)
  uint64_t qfree;                           // FP8 MMAs, single phase: the peer has read its query out
                                            //   of its receive slots (1 remote arrival)
  uint64_t recvfull[kSlots][4];             // peer's partial scores of one lane quarter (32 heads) arrived
                                            //   (1 arrival + 4 KB tx, armed by the receiving warp)
  uint64_t drain[2];                        // every MMA of the QK^T / P . C issuer done
  uint32_t tmem_base;
  int abort;
  int peer_sent[8];                         // written by the peer: partial-score copies its group warp w sent here
  int peer_consumed[8];                     // written by the peer: copies its group warp w received from here
  int sent[8];                              // copies group warp w of this CTA sent to the peer
  int consumed[8];                          // copies group warp w of this CTA received and read
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// (lo, hi) -> fp16x2, round to nearest, saturating at +-65504
__device__ __forceinline__ uint32_t f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 f16x2_to_f32(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

__device__ __forceinline__ float2 bf16x2_to_f32(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// four values -> e4m3 codes (round to nearest even, saturating at +-448), the first in the low byte
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  unsigned short lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// three-input maximum (one instruction on sm_100 and later)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// maximum of 64 values in 32 three-input steps, as a tree of depth 5
__device__ __forceinline__ float max64(const float2 (&x2)[32]) {
  const float* v = reinterpret_cast<const float*>(x2);
  float a[22], b[8];
#pragma unroll
  for (int i = 0; i < 21; ++i) a[i] = max3f(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[21] = v[63];
#pragma unroll
  for (int i = 0; i < 7; ++i) b[i] = max3f(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[7] = a[21];
  return max3f(max3f(b[0], b[1], b[2]), max3f(b[3], b[4], b[5]), fmaxf(b[6], b[7]));
}

__device__ __forceinline__ void fail_timeout(Bars* bars, unsigned* check) {
  if (atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
}

// kMode != bf16: the cache holds e4m3 codes.  The producer TMA-loads each 64 x 64 code box into the
// upper half of the 8 KB slot its bf16 chunk will occupy; one conversion warp per box converts
// it in place (all its reads, then all its writes) before QK^T may use the tile.  The tensor
// scale is folded into the softmax scale and the output scale by the launcher.  The per-block
// format brings each page's block scales in a 1 KB box and its RoPE key already in bf16: four
// warps convert the latent boxes, each value times its token's block scale.
template <int kMode>
__global__ void __cluster_dims__(2, 1, 1)
__launch_bounds__(kMode == kModeFp8Mma ? kThreadsFp8Mma : kMode != kModeBf16 ? kThreadsFp8 : kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_rope,
                 const __grid_constant__ CUtensorMap tmap_scale,
                 const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_qpe,
                 const __grid_constant__ CUtensorMap tmap_o,
                 const int32_t* __restrict__ ctx_len, int n_h,
                 const int32_t* __restrict__ block_table, int bt_stride, int num_pages, float scale_log2,
                 float out_scale, int stall, const uint8_t* __restrict__ w_next, size_t w_next_bytes, Workspace ws,
                 unsigned* check) {
  constexpr bool kFp8 = kMode != kModeBf16;            // e4m3 codes (converted in shared memory, or FP8 MMAs)
  constexpr bool kBlock = kMode == kModeFp8Block;
  using L = Smem<kMode>;
  constexpr bool kMma8 = L::kMma8;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base: swizzle atoms and TMA destinations need it
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kOffBars);
  volatile int* abort_flag = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int unit_idx = blockIdx.x >> 1;
  const uint32_t stage0 = sbase;            // the ring starts the layout

  // barriers and descriptor prefetch need nothing from the earlier kernels of the step
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), kMma8 ? 5 : 1);
      mbar_init(smem_u32(&bars->conv[s]), kMma8 ? 1 : (kBlock ? 4 : 5));
    }
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bars->tready[i]), 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->sfull[i]), 1);
      mbar_init(smem_u32(&bars->sfree[i]), 4);
      mbar_init(smem_u32(&bars->mready[i]), 4);
      mbar_init(smem_u32(&bars->pfull[i]), 4);
    }
    mbar_init(smem_u32(&bars->efin), 8);
    for (int i = 0; i < kSlots; ++i)
      for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&bars->recvfull[i][q]), 1);
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bars->pdone[i]), 1);
    mbar_init(smem_u32(&bars->ofinal), 1);
    mbar_init(smem_u32(&bars->qfull), 1);
    mbar_init(smem_u32(&bars->qfree), 1);
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bars->drain[i]), 1);
    bars->abort = 0;
    // the first phase of every receive quarter (tiles 0..3) armed now, so that the cluster barrier
    // below also publishes it; later tiles are armed four tiles ahead, as each slot is consumed.
    // (A phase armed for a tile the unit does not have never completes and is never waited on.)
    for (int i = 0; i < kSlots; ++i)
      for (int q = 0; q < 4; ++q) mbar_arrive_expect_tx(smem_u32(&bars->recvfull[i][q]), 32 * 128);
    fence_mbar_init();
  }
  if (warp == kWarpProducer && lane == 0) {
    prefetch_tmap(&tmap);
    prefetch_tmap(&tmap_rope);
    if (kBlock) prefetch_tmap(&tmap_scale);
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_qpe);
    prefetch_tmap(&tmap_o);
  }
  __syncthreads();
  // the peer's barriers are initialised (and its first receive phases armed) before any copy into
  // this CTA: a cluster barrier, taken before the dependency wait so that it overlaps the previous
  // kernel (taken after the query's arrival it cost ~1 us on every CTA's critical path)
  cluster_sync();
  griddep_wait();                           // plan, absorbed queries and cache rows are inputs
  griddep_launch_dependents();
  // (the unit record is read together with the unit count: the grid never exceeds the workspace's units)
  const int n_units = ws.counters[0];
  const Unit unit = ws.units[unit_idx];
  if (unit_idx >= n_units) return;         // both CTAs of the cluster leave together
  const int b = unit.b;
  const int n_tiles = unit.page_end - unit.page_begin;

  // TMA of tile j into ring stage j % kStages (both CTAs: this CTA's 288 columns)
  const int32_t* bt_row = block_table + (size_t)b * bt_stride + unit.page_begin;
  auto issue_tile = [&](int j, int page) {
    const int s = j % kStages;
    if (page < 0 || page >= num_pages) {   // bad page id: read page 0 instead; the output is zeroed later
      if (rank == 0) {
        atomicOr(check, kCheckPageId);
        ws.bad[b] = 1;
      }
      page = 0;
    }
    const uint32_t full = smem_u32(&bars->full[s]);
    const uint32_t st = stage0 + s * L::kStage;
    constexpr uint32_t kTx = kMma8 ? 2 * kCodeBox + kRopeBytes / 2
                             : kBlock ? 2 * kChunkBytes + kRopeBytes + kScaleBytes
                                      : (kFp8 ? 2 * kChunkBytes + kRopeBytes / 2 : 4 * kChunkBytes + kRopeBytes);
    mbar_arrive_expect_tx(full, kTx);
    // (an evict-first L2 policy on these once-read rows was measured 4 us slower per step)
    if constexpr (kMma8) {                 // FP8 MMAs: two boxes of 128 codes, 128-byte swizzled, as stored
      for (int c = 0; c < 2; ++c) tma_load_2d(st + c * kCodeBox, &tmap, (int)(rank * 256 + c * 128), page * kPage, full);
    } else {
      for (int c = 0; c < 4; ++c)          // FP8: each code box into the upper half of its chunk slot
        tma_load_2d(st + c * kChunkBytes + (kFp8 ? kChunkBytes / 2 : 0), &tmap, (int)(rank * 256 + c * 64),
                    page * kPage, full);
    }
    // RoPE key: bf16 (its own map over the rows' last 128 bytes for the per-block format) or codes
    tma_load_2d(kMma8 ? st + L::kRopeCodeOff : st + L::kRopeOff + (kMode == kModeFp8 ? kRopeBytes / 2 : 0), &tmap_rope,
                (int)((kBlock ? 0 : kDc) + rank * 32), page * kPage, full);
    if (kBlock)                            // the 4 block scales of every token of the page
      tma_load_2d(st + 4 * kChunkBytes + kRopeBytes, &tmap_scale, kDc, page * kPage, full);
  };
  // the absorbed query of this CTA (latent half: 4 boxes of 64 columns x 128 heads, 128-byte
  // swizzle; RoPE half: straight into its 64-byte swizzled operand slot; heads past n_h read as
  // zeros), then the first tiles of the empty ring.  The latent boxes are staged where no copy
  // can land before they are read.  The peer copies tile j's scores into receive slot j % 4 of
  // this CTA; it sends tiles 2 and 3 only after it has received this CTA's copies of tiles 0 and
  // 1, which leave after this CTA's query has been read, so boxes 2-3 wait in slots 2-3.  Boxes
  // 0-1 wait in ring stage 3, whose tile is requested once they have been read.  With FP8 MMAs
  // (three smaller stages) all four boxes wait in the receive slots, and the peer sends its first
  // copies only after this CTA has signalled that it has read them (the qfree barrier).
  constexpr bool kQStage3 = !kMma8;
  static_assert(!kQStage3 || L::kStage >= 2 * kMaxHeads * 128, "query boxes 0-1 in one stage");
  auto q_box = [&](int c) -> uint32_t {   // shared-memory offset of latent query box c
    return (kQStage3 && c < 2) ? 3 * L::kStage + c * kMaxHeads * 128 : L::kOffRecv + c * kMaxHeads * 128;
  };
  const int n_pre = min(n_tiles, kQStage3 ? kStages - 1 : kStages);
  // a test of the bounded waits (stall == 2): CTA 0 of unit 0 never loads its tile 1
  const int withheld = (stall == 2 && unit_idx == 0 && rank == 0 && n_tiles > 1) ? 1 : -1;
  if (warp == kWarpProducer && lane == 0) {
    // tile 0 first, then the query, then the rest of the ring: every CTA of the grid requests its
    // ring at once, and the first QK^T needs only tile 0 and the query
    int pages[kStages];
#pragma unroll
    for (int j = 0; j < kStages; ++j) pages[j] = j < n_pre ? bt_row[j] : 0;
    if (withheld != 0) issue_tile(0, pages[0]);
    const uint32_t qf = smem_u32(&bars->qfull);
    mbar_arrive_expect_tx(qf, (uint32_t)(4 * kMaxHeads * 128 + kQpeBytes));
    for (int c = 0; c < 4; ++c)
      tma_load_3d(sbase + q_box(c), &tmap_q, (int)(rank * 256 + c * 64), 0, b, qf);
    tma_load_3d(sbase + L::kOffQpe, &tmap_qpe, (int)(kDc + rank * 32), 0, b, qf);
    for (int j = 1; j < n_pre; ++j)
      if (j != withheld) issue_tile(j, pages[j]);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  const int t_end = min(unit.page_end * kPage, ctx_len[b]);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // ---- latent half of the query: shared memory -> TMEM (A operand of QK^T).  Warp w moves heads
  // 32 (w % 4) .. + 31, latent columns 128 (w / 4) .. + 127 of this CTA's 256.  With FP8 MMAs the
  // latent half is quantised instead: one e4m3 scale per head and CTA, s = max |q| / 448 over the
  // CTA's 256 latent values, codes q / s into two 128-byte-swizzled boxes (box w / 4), and the RoPE
  // half divided by s in place, so that QK^T sums s-scaled units (times s in the score scale).
  float qscale = scale_log2;                // per-thread factor of the scores: scale (x s with FP8 MMAs)
  if (warp < 8) {
    const int q4 = warp & 3, half = warp >> 2;
    const int h = q4 * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const bool landed = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->qfull), 0, abort_flag));
    if (!landed) fail_timeout(bars, check);
    if constexpr (kMma8) {
      // two passes over the staged bf16 query (it stays in the receive slots until the exchange
      // starts): the head's maximum magnitude, then the codes
      float amax = 0.0f;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint8_t* row = smem + q_box(2 * half + part) + h * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 x = *reinterpret_cast<const uint4*>(row + ((k ^ (h & 7)) * 16));
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 v = bf16x2_to_f32(w4[i]);
            amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
          }
        }
      }
      float* amax_x = reinterpret_cast<float*>(smem + L::kOffXchg) + 2 * kMaxHeads;   // [half][head]
      amax_x[half * kMaxHeads + h] = amax;
      named_barrier(1, 256);                // the two halves of every head's amax are out
      amax = fmaxf(amax_x[h], amax_x[kMaxHeads + h]);
      const float sq = amax > 0.0f ? amax * (1.0f / 448.0f) : 1.0f, inv = 1.0f / sq;
      qscale = scale_log2 * sq;
      uint8_t* q8row = smem + L::kOffQ8 + half * (kQ8Bytes / 2) + h * 128;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint8_t* row = smem + q_box(2 * half + part) + h * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {        // 16 codes = 8 bf16 pairs (two 16-byte pieces of the row)
          const uint4 x0 = *reinterpret_cast<const uint4*>(row + (((2 * c) ^ (h & 7)) * 16));
          const uint4 x1 = *reinterpret_cast<const uint4*>(row + (((2 * c + 1) ^ (h & 7)) * 16));
          const uint32_t w8[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 v0 = bf16x2_to_f32(w8[2 * i]), v1 = bf16x2_to_f32(w8[2 * i + 1]);
            w[i] = e4m3x4(v0.x * inv, v0.y * inv, v1.x * inv, v1.y * inv);
          }
          const int chunk = 4 * part + c;
          *reinterpret_cast<uint4*>(q8row + ((chunk ^ (h & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (half == 0) {                       // the RoPE half, 32 bf16 of the head, divided by s in place
        uint8_t* pe = smem + L::kOffQpe + h * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4* p4 = reinterpret_cast<uint4*>(pe + ((c ^ ((h >> 1) & 3)) * 16));
          uint4 x = *p4;
          const float2 a = bf16x2_to_f32(x.x), bq = bf16x2_to_f32(x.y), cq = bf16x2_to_f32(x.z), d = bf16x2_to_f32(x.w);
          *p4 = make_uint4(bf16x2_bits(a.x * inv, a.y * inv), bf16x2_bits(bq.x * inv, bq.y * inv),
                           bf16x2_bits(cq.x * inv, cq.y * inv), bf16x2_bits(d.x * inv, d.y * inv));
        }
      }
      fence_proxy_async_smem();              // generic writes before the tensor core reads them
    } else if (landed) {
#pragma unroll
      for (int part = 0; part < 2; ++part) {      // box 2 half + part: 64 columns = 32 TMEM columns
        const uint8_t* row = smem + q_box(2 * half + part) + h * 128;
        uint32_t r[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 x = *reinterpret_cast<const uint4*>(row + ((k ^ (h & 7)) * 16));
          r[4 * k] = x.x; r[4 * k + 1] = x.y; r[4 * k + 2] = x.z; r[4 * k + 3] = x.w;
        }
        tmem_st32(lane_addr + kTmQ + 64 * half + 32 * part, r);
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();    // these reads come before the copies that later reuse the slots
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // FP8 MMAs: the query has left this CTA's receive slots, so the peer may now copy scores into
  // them (its group warps wait for this before their first copy)
  if (!kQStage3 && tid == 0) mbar_arrive_cluster(map_to_rank(smem_u32(&bars->qfree), peer));

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      auto prefetch_tile = [&](int pg) {     // a tile's boxes into L2 (no shared memory, no completion)
        if (pg >= 0 && pg < num_pages) {
          if constexpr (kMma8) {
            for (int c = 0; c < 2; ++c) tma_prefetch_2d(&tmap, (int)(rank * 256 + c * 128), pg * kPage);
          } else {
            for (int c = 0; c < 4; ++c) tma_prefetch_2d(&tmap, (int)(rank * 256 + c * 64), pg * kPage);
          }
          tma_prefetch_2d(&tmap_rope, (int)((kBlock ? 0 : kDc) + rank * 32), pg * kPage);
          if (kBlock) tma_prefetch_2d(&tmap_scale, kDc, pg * kPage);
        }
      };
      int issued = n_pre;
      // the first tile of a stage that held query boxes, now that they have been read
      for (; issued < min(n_tiles, kStages); ++issued) issue_tile(issued, bt_row[issued]);
      // the next user of each stage into L2, once tile 0 has landed (out of the start-up burst)
      if (n_tiles > kStages && mbar_wait(smem_u32(&bars->full[0]), 0, abort_flag)) {
        for (int j = kStages; j < min(n_tiles, 2 * kStages); ++j) prefetch_tile(bt_row[j]);
      }
      for (int j = issued; j < n_tiles; ++j) {
        const int s = j % kStages;
        const int page = bt_row[j];
        if (j + kStages < n_tiles) prefetch_tile(bt_row[j + kStages]);   // the stage's next tile, into L2
        if (!mbar_wait(smem_u32(&bars->empty[s]), ((j / kStages) & 1) ^ 1, abort_flag)) {
          fail_timeout(bars, check);
          break;
        }
        issue_tile(j, page);
        issued = j + 1;
      }
      // the value up-projection's weights (the next kernel) into L2 while the last tiles are
      // consumed: this CTA's share of them, 16 KB per request.  (bf16 cache only: with an FP8
      // cache the extra code in this register-bound variant measured 14 us slower per step)
      if (kMode == kModeBf16 && w_next) {
        const size_t n_cta = 2 * (size_t)__ldcg(&ws.counters[0]), me = 2 * (size_t)unit_idx + rank;
        const size_t lo = (w_next_bytes * me / n_cta) & ~(size_t)15, hi = (w_next_bytes * (me + 1) / n_cta) & ~(size_t)15;
        for (size_t off = lo; off < hi; off += 16384)
          bulk_prefetch_l2(w_next + off, (uint32_t)min((size_t)16384, hi - off));
      }
      // drain: every load issued has landed before the CTA may exit
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        volatile int never = 0;
        if (j != withheld) mbar_wait(smem_u32(&bars->full[j % kStages]), (j / kStages) & 1, &never);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ QK^T issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, 64, false, false);
      const uint32_t idesc_qk8 = idesc_e4m3_f32(128, 64);
      const uint64_t qpe_desc = sdesc_sw64(sbase + L::kOffQpe, 16, 512);
      const uint64_t q8_desc = sdesc_sw128(sbase + L::kOffQ8, 16, 1024);
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % kStages;
        // the tile has landed (and been converted), and S(j - 1) has been loaded by its group
        if (!mbar_wait(smem_u32(kFp8 ? &bars->conv[s] : &bars->full[s]), (j / kStages) & 1, abort_flag) ||
            (j > 0 && !mbar_wait(smem_u32(&bars->sfree[(j - 1) & 1]), ((j - 1) >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = stage0 + s * L::kStage;
        const uint64_t lat_desc = sdesc_sw128(st, 16, 1024), rope_desc = sdesc_sw64(st + L::kRopeOff, 16, 512);
        const uint32_t d = tmem + kTmS;
        if constexpr (kMma8) {
#pragma unroll
          for (int k = 0; k < 8; ++k)        // code box k / 4, 32-code step k % 4 inside the 128-byte row
            mma8_ss(d, q8_desc + (uint64_t)((((k >> 2) * (kQ8Bytes / 2)) + (k & 3) * 32) >> 4),
                    lat_desc + (uint64_t)((((k >> 2) * kCodeBox) + (k & 3) * 32) >> 4), idesc_qk8, k > 0);
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k)       // latent chunk k / 4, 32-byte step k % 4 inside the 128-byte row
            mma_ts(d, tmem + kTmQ + 8 * k, lat_desc + (uint64_t)((((k >> 2) * kChunkBytes) + (k & 3) * 32) >> 4),
                   idesc_qk, k > 0);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k)
          mma_ss(d, qpe_desc + (uint64_t)(2 * k), rope_desc + (uint64_t)(2 * k), idesc_qk, 1);
        mma_commit(smem_u32(&bars->sfull[j & 1]));
        if constexpr (kMma8) mma_commit(smem_u32(&bars->empty[s]));   // QK^T's share of releasing the stage
      }
      if (!ok) fail_timeout(bars, check);
      mma_commit(smem_u32(&bars->drain[0]));   // arrives once every MMA issued above has finished
      volatile int never = 0;
      mbar_wait(smem_u32(&bars->drain[0]), 0, &never);
    }
  } else if (warp == kWarpPv) {
    // ------------------------------------------------------------ P . C issuer (tile order)
    // A separate issuer: a P . C never waits behind the issue of a QK^T (they use disjoint
    // TMEM: P slots and O, against the score buffer).
    if (lane == 0) {
      const uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
      const uint32_t idesc_pv8 = idesc_e4m3_f32(128, 256);
      bool ok = true;
      for (int jj = 0; jj < n_tiles; ++jj) {
        const int s = jj % kStages, bb = jj & 1;
        // P(jj) written; with FP8 MMAs also tile jj transposed into buffer jj % 2
        if (!mbar_wait(smem_u32(&bars->pfull[bb]), (jj >> 1) & 1, abort_flag) ||
            (kMma8 && !mbar_wait(smem_u32(&bars->tready[bb]), (jj >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (kMma8) {               // e4m3 P (K-major, 64-byte rows) . transposed codes (K-major)
          const uint64_t p_desc = sdesc_sw64(sbase + L::kOffP8 + bb * kP8Bytes, 16, 512);
          const uint64_t ct_desc = sdesc_sw64(sbase + L::kOffCt + bb * kCtBytes, 16, 512);
#pragma unroll
          for (int k = 0; k < 2; ++k)        // 32 tokens per step: 32 bytes along both operands' rows
            mma8_ss(tmem + kTmO, p_desc + (uint64_t)(2 * k), ct_desc + (uint64_t)(2 * k), idesc_pv8,
                    (jj > 0 || k > 0) ? 1u : 0u);
        } else {
          const uint64_t c_desc = sdesc_sw128(stage0 + s * L::kStage, kChunkBytes, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + kTmO, tmem + kTmP + 32 * bb + 8 * k, c_desc + (uint64_t)(128 * k), idesc_pv,
                   (jj > 0 || k > 0) ? 1u : 0u);
          mma_commit(smem_u32(&bars->empty[s]));
        }
        mma_commit(smem_u32(&bars->pdone[bb]));
        if (jj == n_tiles - 1) mma_commit(smem_u32(&bars->ofinal));
      }
      if (!ok) fail_timeout(bars, check);
      mma_commit(smem_u32(&bars->drain[1]));
      volatile int never = 0;
      mbar_wait(smem_u32(&bars->drain[1]), 0, &never);
    }
  } else if (warp >= kWarpConv) {
    // ------------------------------------------------------------ FP8 cache: e4m3 -> bf16 in place
    // (launched only with an FP8 cache) warp 11 + c converts latent chunk c of every tile,
    // warp 15 the RoPE box.  A box's codes sit in the upper half of the slot its bf16 rows
    // fill, so all of them are read (into the warp's registers) before any row is written;
    // one warp per box makes that a warp-level order.  Every wait is bounded: a warp that
    // gives up aborts the kernel.
    if constexpr (kFp8) {
      const int c = warp - kWarpConv;         // 0..3 latent chunk, 4 RoPE box (codes with one tensor scale)
      bool ok = true;
      if (kMma8 && c < 4) {
        // FP8 MMAs: warp 11 + c transposes latent columns [64 c, 64 c + 64) of every tile into the
        // buffer of the tile's parity: row n = latent column, 64 token codes, 64-byte swizzle
        // (16-byte chunk k of row n at k ^ ((n >> 1) & 3)), token codes past the context zeroed.
        // Lane = (token group tg = lane & 3: tokens 16 tg .. + 15; column group cg = lane >> 2:
        // columns 8 cg .. + 7 of the warp's 64); 4 x 4 byte blocks are transposed with byte permutes.
        // Bank-conflict-free order: step r reads token 16 tg + (r ^ 2 tg) (the four token groups then
        // sit on rows of different swizzle phase), and odd column groups write their columns in
        // pairs swapped (the two column groups of a store phase then fill both halves of the bank
        // line); the byte permute and the selects below undo both orders.
        const int tg = lane & 3, cg = lane >> 2;
        const int box = c >> 1, chunk = 4 * (c & 1) + (cg >> 1), off8 = (cg & 1) * 8;
        const int xr = tg << 1;
        const uint32_t bsel = (tg & 1) ? 0x1032u : 0x3210u;   // token k ^ 2 (tg & 1) -> byte k of a block
        const bool bswap = (tg >> 1) != 0;                       // block i holds tokens 4 (i ^ (tg >> 1)) ..
        const bool cswap = (cg & 1) != 0;
        for (int t = 0; t < n_tiles; ++t) {
          const int s = t % kStages, bb = t & 1;
          // the tile has landed, and buffer bb's last reader, P . C of tile t - 2, has finished
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[s]), (t / kStages) & 1, abort_flag)) ||
              (t >= 2 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pdone[bb]), ((t - 2) >> 1) & 1, abort_flag)))) {
            ok = false;
            break;
          }
          const uint8_t* src = smem + s * L::kStage + box * kCodeBox;
          uint32_t a[16][2];                  // a[r]: the 8 codes of token 16 tg + (r ^ 2 tg)
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const int tok = 16 * tg + (r ^ xr);
            const uint2 v = *reinterpret_cast<const uint2*>(src + tok * 128 + ((chunk ^ (tok & 7)) * 16) + off8);
            a[r][0] = v.x;
            a[r][1] = v.y;
          }
          uint32_t o[8][4];                   // o[col][i] byte k: token 16 tg + 4 (i ^ (tg >> 1)) + (k ^ 2 (tg & 1))
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint32_t t0 = __byte_perm(a[4 * i][k], a[4 * i + 1][k], 0x5140);
              const uint32_t t1 = __byte_perm(a[4 * i][k], a[4 * i + 1][k], 0x7362);
              const uint32_t t2 = __byte_perm(a[4 * i + 2][k], a[4 * i + 3][k], 0x5140);
              const uint32_t t3 = __byte_perm(a[4 * i + 2][k], a[4 * i + 3][k], 0x7362);
              o[4 * k][i] = __byte_perm(t0, t2, 0x5410);
              o[4 * k + 1][i] = __byte_perm(t0, t2, 0x7632);
              o[4 * k + 2][i] = __byte_perm(t1, t3, 0x5410);
              o[4 * k + 3][i] = __byte_perm(t1, t3, 0x7632);
            }
          const int valid = min(kPage, t_end - (unit.page_begin + t) * kPage);
          uint8_t* dst = smem + L::kOffCt + bb * kCtBytes;
#pragma unroll
          for (int col = 0; col < 8; ++col) {
            const int n = 64 * c + 8 * cg + (col ^ (cswap ? 1 : 0));   // the column this lane writes now
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {     // block i of the output: tokens 16 tg + 4 i .. + 3 in order
              const uint32_t x0 = cswap ? o[col ^ 1][i] : o[col][i];
              const uint32_t x1 = cswap ? o[col ^ 1][i ^ 1] : o[col][i ^ 1];
              w[i] = __byte_perm(bswap ? x1 : x0, 0u, bsel);
            }
            if (valid < kPage) {              // a partial last page: codes of rows past the context become 0
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int nv = min(4, max(0, valid - (16 * tg + 4 * i)));
                w[i] &= nv >= 4 ? 0xFFFFFFFFu : ((1u << (8 * nv)) - 1u);
              }
            }
            *reinterpret_cast<uint4*>(dst + n * 64 + ((tg ^ ((n >> 1) & 3)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bars->tready[bb]));
            mbar_arrive(smem_u32(&bars->empty[s]));   // this warp is done with the stage's codes
          }
        }
      }
      for (int t = 0; t < n_tiles && !(kBlock && c == 4) && !(kMma8 && c < 4); ++t) {
        const int s = t % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[s]), (t / kStages) & 1, abort_flag))) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * L::kStage;
        if (c < 4 && kBlock) {
          // as below, each value times its token's scale for this chunk's block of 128 latent
          // values (block 2 rank + c / 2; the page's scales sit after the RoPE box, 16 bytes a token)
          const int p = lane & 3;
          uint8_t* box = st + c * kChunkBytes;
          const float* scl = reinterpret_cast<const float*>(st + 4 * kChunkBytes + kRopeBytes) + 2 * rank + (c >> 1);
          uint4 v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            v[k] = *reinterpret_cast<const uint4*>(box + kChunkBytes / 2 + (8 * k + (lane >> 2)) * 64 + p * 16);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {       // 128-byte rows, 128-byte swizzle (the scales are not rewritten)
            const int r = 8 * k + (lane >> 2);
            const float sc = scl[r * 4];
            const uint2 a = e4m3x4_scaled_to_bf16x4(v[k].x, sc), b = e4m3x4_scaled_to_bf16x4(v[k].y, sc);
            const uint2 d = e4m3x4_scaled_to_bf16x4(v[k].z, sc), e = e4m3x4_scaled_to_bf16x4(v[k].w, sc);
            *reinterpret_cast<uint4*>(box + r * 128 + (((2 * p) ^ (r & 7)) * 16)) = make_uint4(a.x, a.y, b.x, b.y);
            *reinterpret_cast<uint4*>(box + r * 128 + (((2 * p + 1) ^ (r & 7)) * 16)) = make_uint4(d.x, d.y, e.x, e.y);
          }
        } else if (c < 4) {
          // lane = (row 8 k + lane / 4, 16 codes 16 (lane % 4) ..) for k = 0..7
          const int p = lane & 3;
          uint8_t* box = st + c * kChunkBytes;
          uint4 v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            v[k] = *reinterpret_cast<const uint4*>(box + kChunkBytes / 2 + (8 * k + (lane >> 2)) * 64 + p * 16);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {       // 128-byte rows, 128-byte swizzle
            const int r = 8 * k + (lane >> 2);
            const uint2 a = e4m3x4_to_bf16x4(v[k].x), b = e4m3x4_to_bf16x4(v[k].y);
            const uint2 d = e4m3x4_to_bf16x4(v[k].z), e = e4m3x4_to_bf16x4(v[k].w);
            *reinterpret_cast<uint4*>(box + r * 128 + (((2 * p) ^ (r & 7)) * 16)) = make_uint4(a.x, a.y, b.x, b.y);
            *reinterpret_cast<uint4*>(box + r * 128 + (((2 * p + 1) ^ (r & 7)) * 16)) = make_uint4(d.x, d.y, e.x, e.y);
          }
        } else {
          // lane = (row 16 k + lane / 2, 16 codes 16 (lane % 2) ..) for k = 0..3; the codes sit in
          // the upper half of the box (or, with FP8 MMAs, in their own landing area)
          const int p = lane & 1;
          uint8_t* box = st + L::kRopeOff;
          const uint8_t* codes = st + L::kRopeCodeOff;
          uint4 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            v[k] = *reinterpret_cast<const uint4*>(codes + (16 * k + (lane >> 1)) * 32 + p * 16);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {       // 64-byte rows, 64-byte swizzle
            const int r = 16 * k + (lane >> 1);
            const uint2 a = e4m3x4_to_bf16x4(v[k].x), b = e4m3x4_to_bf16x4(v[k].y);
            const uint2 d = e4m3x4_to_bf16x4(v[k].z), e = e4m3x4_to_bf16x4(v[k].w);
            *reinterpret_cast<uint4*>(box + r * 64 + (((2 * p) ^ ((r >> 1) & 3)) * 16)) = make_uint4(a.x, a.y, b.x, b.y);
            *reinterpret_cast<uint4*>(box + r * 64 + (((2 * p + 1) ^ ((r >> 1) & 3)) * 16)) = make_uint4(d.x, d.y, e.x, e.y);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->conv[s]));
      }
      if (!ok) fail_timeout(bars, check);
    }
  } else {
    // ------------------------------------------------------------ tile groups: exchange, softmax, epilogue
    // Group g = warp / 4 takes the tiles j = g (mod 2); warp w holds heads 32 (w % 4) .. + 31
    // (thread = head = TMEM lane).  A tile's chain -- read S_r, send the fp16 copy, wait for the
    // peer's, softmax, write P -- is longer than the QK^T that feeds it, so two groups run
    // two tiles' chains at once.  The running max is handed from tile to tile through shared
    // memory; each group keeps its own sum, and the two are reconciled in the epilogue.
    const int g = warp >> 2, q4 = warp & 3;
    const int h = q4 * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t recv_peer = map_to_rank(sbase + L::kOffRecv, peer);
    float* m_pub = reinterpret_cast<float*>(smem + L::kOffXchg);    // [group][head]: running max after its last tile
    float* fin_x = m_pub + 2 * kMaxHeads;                         // [group][2][head]: final (max, sum)
    const float2 sc2 = make_float2(qscale, qscale), zero2 = make_float2(0.0f, 0.0f);
    float m_g = -INFINITY, l_g = 0.0f;        // this group's sum, relative to 2^m_g
    bool ok = true;
    int sent = 0, consumed = 0;               // this warp's partial-score copies sent / received (in tile order)
    // waits are made warp-uniform: tcgen05.ld / st below are .sync.aligned
    auto wait_cta = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, abort_flag));
    };
    auto wait_cluster = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait<true>(smem_u32(bar), parity, abort_flag));
    };
    for (int j = g; j < n_tiles; j += 2) {
      const int k = j >> 1, slot = j & (kSlots - 1);
      const int valid = min(kPage, t_end - (unit.page_begin + j) * kPage);
      if (!wait_cta(&bars->sfull[g], k & 1)) { ok = false; break; }
      // (FP8 MMAs) before this warp's first copy: the peer's query is out of the slots it lands in
      if (!kQStage3 && k == 0 && !wait_cluster(&bars->qfree, 0)) { ok = false; break; }
      tc_fence_after();
      // x2[i] = scores 2i, 2i + 1 in the log2 domain, as pairs for the packed fp32 ops
      float2 x2[32];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(lane_addr + kTmS, r0);      // own partial, kept in fp32 (the peer gets fp16)
        tmem_ld32(lane_addr + kTmS + 32, r1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->sfree[g]));   // QK^T of tile j + 1 may overwrite S
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x2[i] = __ffma2_rn(make_float2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1])), sc2, zero2);
          x2[16 + i] = __ffma2_rn(make_float2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1])), sc2, zero2);
        }
      }
      {
        // fp16 copy for the peer, staged in this CTA's own receive slot (j + 2) % 4 and moved
        // by one 4 KB bulk copy per warp into the peer's slot j % 4, completing on the peer's
        // barrier of that slot and lane quarter.  The staging rows last held tile j - 2 for
        // this same warp, which has consumed them; the peer refills them with tile j + 2 only
        // after its group g has finished tile j, which needed every copy of this tile, so
        // after the copies have read them.  The peer's slot j % 4 needs no "free" handshake
        // either: this CTA sends tile j after its group g finished tile j - 2, which needed
        // the peer's tile j - 2 copies, sent after the peer's group g finished tile j - 4,
        // the last user of the slot -- and re-armed the slot's quarter for tile j there, so
        // every copy lands in an armed phase.
        uint8_t* stg = smem + L::kOffRecv + ((j + 2) & (kSlots - 1)) * kSlotBytes;
#pragma unroll
        for (int qq = 0; qq < 8; ++qq)
          *reinterpret_cast<uint4*>(stg + h * 128 + ((qq ^ (h & 7)) * 16)) =
              make_uint4(f16x2_sat(x2[4 * qq].x, x2[4 * qq].y), f16x2_sat(x2[4 * qq + 1].x, x2[4 * qq + 1].y),
                         f16x2_sat(x2[4 * qq + 2].x, x2[4 * qq + 2].y), f16x2_sat(x2[4 * qq + 3].x, x2[4 * qq + 3].y));
        fence_proxy_async_smem();
        __syncwarp();
        // (a test of the bounded waits, stall == 3: CTA 1 of unit 0 withholds warp 4's copy of tile 1)
        const bool withhold = stall == 3 && unit_idx == 0 && rank == 1 && j == 1 && q4 == 0;
        if (lane == 0 && !withhold) {
          const uint32_t peer_bar = map_to_rank(smem_u32(&bars->recvfull[slot][q4]), peer);
          asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                       ::"r"(recv_peer + slot * kSlotBytes + q4 * 32 * 128), "r"(smem_u32(stg + q4 * 32 * 128)),
                       "r"(32 * 128), "r"(peer_bar) : "memory");
        }
        ++sent;                               // (a withheld copy counts: its receiver then waits out its limit at exit)
      }
      if (!wait_cluster(&bars->recvfull[slot][q4], (j >> 2) & 1)) { ok = false; break; }
      ++consumed;
      {
        // x = x_own + x_peer
        const uint4* rp = reinterpret_cast<const uint4*>(smem + L::kOffRecv + slot * kSlotBytes + h * 128);
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          const uint4 v = rp[qq ^ (h & 7)];
          const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) x2[4 * qq + kk] = __fadd2_rn(x2[4 * qq + kk], f16x2_to_f32(ww[kk]));
        }
      }
      // the quarter is read: arm it for tile j + 4, which the peer sends only after this warp has
      // sent tile j + 2, later in this loop
      if (lane == 0 && j + kSlots < n_tiles)
        mbar_arrive_expect_tx(smem_u32(&bars->recvfull[slot][q4]), 32 * 128);
      if (valid < kPage) {
        // a partial last page: rows past the context hold stale data; zero this CTA's latent
        // rows there so P = 0 meets finite values in P . C (with FP8 MMAs the transposing warps
        // zero those tokens' codes in the copy P . C reads)
        if constexpr (!kMma8) {
          uint8_t* st = smem + (j % kStages) * L::kStage;
          for (int rr = valid + (h >> 3); rr < kPage; rr += 16)     // 16 rows x 8 16-byte pieces per pass
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              *reinterpret_cast<uint4*>(st + cc * kChunkBytes + rr * 128 + (h & 7) * 16) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (2 * i >= valid) x2[i].x = -INFINITY;
          if (2 * i + 1 >= valid) x2[i].y = -INFINITY;
        }
      }
      const float mt = max64(x2);
      // P slot g's previous user, P . C of tile j - 2, has finished.  Waited before the max
      // is published: the other group then knows that this slot's phase for tile j - 2 is
      // complete, so its own wait for P . C of tile j (one phase later) is unambiguous.
      if (j >= 2 && !wait_cta(&bars->pdone[g], (k - 1) & 1)) { ok = false; break; }
      // the running max after tile j - 1 (the other group's), then this tile's
      float m_prev = -INFINITY;
      if (j > 0) {
        if (!wait_cta(&bars->mready[g ^ 1], ((j - 1) >> 1) & 1)) { ok = false; break; }
        m_prev = m_pub[(g ^ 1) * kMaxHeads + h];
      }
      const bool grow = mt > m_prev + 8.0f;
      const float m_new = grow ? mt : m_prev;
      m_pub[g * kMaxHeads + h] = m_new;       // read by the other group before it publishes again
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->mready[g]));
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // rescale this warp's rows of O once P . C of tile j - 1 has landed (the other slot;
        // its previous phase, tile j - 3, was seen complete by the other group before it
        // published the max this group has just read)
        if (!wait_cta(&bars->pdone[g ^ 1], ((j - 1) >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const float alpha = grow ? ex2_approx(m_prev - m_new) : 1.0f;
        const float2 al2 = make_float2(alpha, alpha);
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(lane_addr + kTmO + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 v = __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), al2, zero2);
            r[2 * i] = __float_as_uint(v.x);
            r[2 * i + 1] = __float_as_uint(v.y);
          }
          tmem_st32(lane_addr + kTmO + c0, r);
        }
        tmem_st_wait();
      }
      if (m_g != m_new) {
        l_g *= ex2_approx(m_g - m_new);       // 0 while this group has no sum yet
        m_g = m_new;
      }
      uint32_t pk[32];                        // P as bf16 pairs, or (FP8 MMAs) 16 words of 4 e4m3 codes
      float2 ps[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) ps[i] = zero2;
      const float2 negm2 = make_float2(-m_new, -m_new);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 d0 = __fadd2_rn(x2[i], negm2), d1 = __fadd2_rn(x2[i + 1], negm2);
        const float2 p0 = make_float2(ex2_approx(d0.x), ex2_approx(d0.y));
        const float2 p1 = make_float2(ex2_approx(d1.x), ex2_approx(d1.y));
        ps[i & 3] = __fadd2_rn(ps[i & 3], p0);
        ps[(i + 1) & 3] = __fadd2_rn(ps[(i + 1) & 3], p1);
        if constexpr (kMma8) {
          pk[i >> 1] = e4m3x4(p0.x, p0.y, p1.x, p1.y);
        } else {
          pk[i] = bf16x2_bits(p0.x, p0.y);
          pk[i + 1] = bf16x2_bits(p1.x, p1.y);
        }
      }
      {
        const float2 s2 = __fadd2_rn(__fadd2_rn(ps[0], ps[1]), __fadd2_rn(ps[2], ps[3]));
        l_g += s2.x + s2.y;
      }
      if constexpr (kMma8) {
        // P(j) as e4m3 codes (P <= 2^8 < 448) into this thread's row of P slot g (64-byte rows,
        // 16-byte chunk c at c ^ ((h >> 1) & 3)); its last reader, P . C of tile j - 2, is done
        uint8_t* prow = smem + L::kOffP8 + g * kP8Bytes + h * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c)            // 16 tokens per 16-byte chunk
          *reinterpret_cast<uint4*>(prow + ((c ^ ((h >> 1) & 3)) * 16)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        fence_proxy_async_smem();            // generic writes before the tensor core reads them
      } else {
        tmem_st32(lane_addr + kTmP + 32 * g, pk);
        tmem_st_wait();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->pfull[g]));
    }
    if (!ok) fail_timeout(bars, check);
    // tell the peer how many copies this warp sent into it and received from it (read after the
    // first cluster barrier below)
    if (lane == 0) {
      const uint32_t dst_s = map_to_rank(smem_u32(&bars->peer_sent[warp]), peer);
      const uint32_t dst_c = map_to_rank(smem_u32(&bars->peer_consumed[warp]), peer);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst_s), "r"(sent) : "memory");
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst_c), "r"(consumed) : "memory");
      bars->sent[warp] = sent;
      bars->consumed[warp] = consumed;
    }
    // ---- epilogue: reconcile the two groups' sums; group g writes latent columns
    // [128 g, 128 g + 128) of this CTA's half of every head
    // (ofinal is a single-phase barrier: a parity wait on pdone here could be two phases behind)
    fin_x[(g * 2) * kMaxHeads + h] = m_g;
    fin_x[(g * 2 + 1) * kMaxHeads + h] = l_g;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars->efin));
    bool fin = ok && n_tiles > 0;
    if (fin) {
      fin = wait_cta(&bars->efin, 0) && wait_cta(&bars->ofinal, 0);
      if (!fin) fail_timeout(bars, check);
    }
    if (fin) {
      tc_fence_after();
      const float m_o = fin_x[((g ^ 1) * 2) * kMaxHeads + h], l_o = fin_x[((g ^ 1) * 2 + 1) * kMaxHeads + h];
      const float m_fin = fmaxf(m_g, m_o);    // the running max after the last tile
      const float l_sum = l_g * ex2_approx(m_g - m_fin) + l_o * ex2_approx(m_o - m_fin);
      const float inv = out_scale / l_sum;
      const bool live = h < n_h;
      // a whole sequence: bf16 rows staged in the (now idle) ring, this warp's 32 heads x 2 boxes
      // of 64 columns, 128-byte swizzled, and written by TMA stores (heads past n_h are clipped)
      uint8_t* ob = smem + (g * 4 + q4) * 2 * 4096;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const int c0 = 128 * g + 32 * cc;
        uint32_t r[32];
        tmem_ld32(lane_addr + kTmO + c0, r);
        tmem_ld_wait();
        if (unit.part < 0) {
          uint8_t* row = ob + (cc >> 1) * 4096 + lane * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* f = reinterpret_cast<const float*>(r + 8 * i);
            *reinterpret_cast<uint4*>(row + (((((cc & 1) * 4) + i) ^ (lane & 7)) * 16)) =
                make_uint4(bf16x2_bits(f[0] * inv, f[1] * inv), bf16x2_bits(f[2] * inv, f[3] * inv),
                           bf16x2_bits(f[4] * inv, f[5] * inv), bf16x2_bits(f[6] * inv, f[7] * inv));
          }
        } else if (live) {
          float4* dst = reinterpret_cast<float4*>(ws.part_o + ((size_t)unit.part * n_h + h) * kDc + rank * 256 + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float* f = reinterpret_cast<const float*>(r + 4 * i);
            dst[i] = make_float4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
          }
        }
      }
      if (unit.part < 0) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && 32 * q4 < n_h) {
          for (int bx = 0; bx < 2; ++bx)
            tma_store_3d(&tmap_o, smem_u32(ob + bx * 4096), (int)(rank * 256 + 128 * g + 64 * bx), 32 * q4, b);
          bulk_commit_group();                // (its staging read is awaited at exit)
        }
      }
      if (live && unit.part >= 0 && rank == 0 && g == 0)
        ws.part_lse[(size_t)unit.part * n_h + h] = (m_fin + log2f(l_sum)) * 0.69314718055994531f;
    }
  }
  tc_fence_before();
  __syncthreads();
  // Every copy either CTA will ever send has been issued and its count published.  A copy
  // completes only on its receiver's barrier, and its source is this CTA's shared memory.  When
  // every copy sent either way was received (normal operation) none is in flight and the CTAs
  // may exit after this barrier.  Otherwise (after a timeout) each receiving warp waits for the
  // copies the peer sent it but it did not consume, and a second barrier keeps both CTAs, and so
  // the copies' sources and destinations, alive until then.  Both CTAs decide alike: each holds
  // the same four counts per warp pair.
  cluster_sync();
  bool all_received = true;
#pragma unroll
  for (int w = 0; w < 8; ++w)
    all_received &= bars->consumed[w] == bars->peer_sent[w] && bars->peer_consumed[w] == bars->sent[w];
  if (!all_received) {
    if (warp < 8 && lane == 0) {
      const int g = warp >> 2, q4 = warp & 3;
      volatile int never = 0;
      const int n_sent = bars->peer_sent[warp];
      for (int c = bars->consumed[warp]; c < n_sent; ++c) {
        const int j = g + 2 * c;
        mbar_wait<true>(smem_u32(&bars->recvfull[j & (kSlots - 1)][q4]), (j >> 2) & 1, &never);
      }
    }
    __syncthreads();
    cluster_sync();
  }
  if (warp < 8 && lane == 0) bulk_wait_read();   // the output staging read before the CTA exits
                                                 // (the writes complete with the grid)
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

// Tensor map of a bf16 cache [num_pages * 64 rows][576]: boxes of `width` columns x 64 rows,
// 128-byte swizzle for 64 columns (latent), 64-byte swizzle for 32 (RoPE key).
cudaError_t make_cache_tensor_map(const void* cache, int num_pages, int width, CUtensorMap* map) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)num_pages * kPage};
  const cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
  const cuuint32_t box[2] = {(cuuint32_t)width, (cuuint32_t)kPage};
  const cuuint32_t elem[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, width == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of an e4m3 cache [num_pages * 64 rows][576 bytes]: boxes of `width` bytes x 64
// rows, no swizzle (the kernel converts them into swizzled bf16 chunks), or, for 128-byte boxes,
// 128-byte swizzled (FP8 MMA operands as they land).
cudaError_t make_cache_tensor_map_fp8(const void* cache, int num_pages, int width, CUtensorMap* map) {
  // 128-byte boxes are MMA operands as loaded (128-byte swizzle); narrower ones are converted first
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)num_pages * kPage};
  const cuuint64_t strides[1] = {(cuuint64_t)kRow};
  const cuuint32_t box[2] = {(cuuint32_t)width, (cuuint32_t)kPage};
  const cuuint32_t elem[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, width == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of the absorbed query [B][n_h][576] bf16 as (column, head, sequence): boxes of
// `width` columns x 128 heads x 1 sequence (heads past n_h read as zeros), 128-byte swizzle for
// 64 columns, 64-byte swizzle for 32.
cudaError_t make_query_tensor_map(const void* q_abs, int batch, int n_h, int width, CUtensorMap* map) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kRow, (cuuint64_t)n_h, (cuuint64_t)batch};
  const cuuint64_t strides[2] = {(cuuint64_t)kRow * 2, (cuuint64_t)kRow * 2 * n_h};
  const cuuint32_t box[3] = {(cuuint32_t)width, (cuuint32_t)kMaxHeads, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q_abs), dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, width == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of the normalised latent sums o_lat [B][n_h][512] bf16 as (column, head, sequence):
// store boxes of 64 columns x 32 heads x 1 sequence, 128-byte swizzle.
cudaError_t make_latent_out_tensor_map(void* o_lat, int batch, int n_h, CUtensorMap* map) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kDc, (cuuint64_t)n_h, (cuuint64_t)batch};
  const cuuint64_t strides[2] = {(cuuint64_t)kDc * 2, (cuuint64_t)kDc * 2 * n_h};
  const cuuint32_t box[3] = {64, 32, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o_lat, dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Per-block FP8 cache [num_pages * 64 rows][656 bytes]: codes (boxes of 64 bytes x 64 rows,
// no swizzle), the 16 scale bytes of a row (box 16 x 64), and the bf16 RoPE key at byte 528
// of each row as its own bf16 matrix [rows][64] (boxes of 32 columns x 64 rows, 64-byte
// swizzle, the operand layout of the bf16 cache's RoPE box).
cudaError_t make_block_cache_maps(const void* cache, int num_pages, CUtensorMap* codes, CUtensorMap* scales,
                                  CUtensorMap* rope) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  constexpr int kRowB = kDc + 16 + 2 * kDr;
  const cuuint64_t rows = (cuuint64_t)num_pages * kPage;
  const cuuint64_t dims8[2] = {(cuuint64_t)kRowB, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kRowB};
  const cuuint32_t elem[2] = {1, 1};
  const cuuint32_t box_c[2] = {64, (cuuint32_t)kPage}, box_s[2] = {16, (cuuint32_t)kPage};
  CUresult r = enc(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims8, strides, box_c, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS)
    r = enc(scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims8, strides, box_s, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    const cuuint64_t dims[2] = {(cuuint64_t)kDr, rows};
    const cuuint32_t box_r[2] = {32, (cuuint32_t)kPage};
    r = enc(rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(static_cast<const void*>(static_cast<const uint8_t*>(cache) + kDc + 16)), dims, strides,
            box_r, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
template <int kMode>
cudaError_t launch_decode_tc(const Handle& h, const int32_t* ctx_len, int batch, const int32_t* block_table, int bt_stride,
                             int num_pages, const CUtensorMap& map, const CUtensorMap& map_rope,
                             const CUtensorMap& map_scale, const Workspace& ws, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_tc_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<kMode>::kBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  // an FP8 cache with one tensor scale holds codes of value / fp8_scale: the scale multiplies
  // every score and the output (the per-block format's values are scaled when converted)
  const float cache_scale = (kMode == kModeFp8 || kMode == kModeFp8Mma) ? h.cfg.fp8_scale : 1.0f;
  const float scale_log2 = h.scale * cache_scale * 1.4426950408889634f;
  // the absorbed query [B][n_h][576] as (column, head, sequence): 64- and 32-column boxes of 128 heads
  alignas(64) CUtensorMap map_q, map_qpe;
  alignas(64) CUtensorMap map_o;
  cudaError_t e = make_query_tensor_map(ws.q_abs, batch, h.cfg.n_h, 64, &map_q);
  if (e == cudaSuccess) e = make_query_tensor_map(ws.q_abs, batch, h.cfg.n_h, 32, &map_qpe);
  if (e == cudaSuccess) e = make_latent_out_tensor_map(ws.o_lat, batch, h.cfg.n_h, &map_o);
  if (e != cudaSuccess) return e;
  const int threads = kMode == kModeFp8Mma ? kThreadsFp8Mma : kMode != kModeBf16 ? kThreadsFp8 : kThreads;
  return launch_pdl(decode_tc_kernel<kMode>, dim3(2 * ws.max_units), dim3(threads),
                    Smem<kMode>::kBytes, st, map, map_rope, map_scale, map_q, map_qpe, map_o,
                    ctx_len,
                    h.cfg.n_h, block_table, bt_stride, num_pages, scale_log2, cache_scale, h.test_stall,
                    reinterpret_cast<const uint8_t*>(h.w_uv), sizeof(__nv_bfloat16) * (size_t)h.cfg.n_h * kDv * kDc, ws,
                    h.check_word);
}
}  // namespace

// TMA descriptors of a cache (64- and 32-column boxes of one page; for the per-block format
// also its scale boxes), rebuilt only when the cache pointer or its page count changes.
cudaError_t cache_maps(const Handle& h, const void* cache, int num_pages) {
  const int dt = h.cfg.cache_dtype;
  Handle& hm = const_cast<Handle&>(h);
  if (hm.tmap_cache != cache || hm.tmap_pages != num_pages) {
    CUtensorMap* m = reinterpret_cast<CUtensorMap*>(hm.tmap);
    CUtensorMap* mr = reinterpret_cast<CUtensorMap*>(hm.tmap_rope);
    CUtensorMap* ms = reinterpret_cast<CUtensorMap*>(hm.tmap_scale);
    cudaError_t e;
    if (dt == MLA_CACHE_FP8_E4M3_BLOCK) {
      e = make_block_cache_maps(cache, num_pages, m, ms, mr);
    } else {
      const bool fp8 = dt == MLA_CACHE_FP8_E4M3;
      e = fp8 ? make_cache_tensor_map_fp8(cache, num_pages, 64, m) : make_cache_tensor_map(cache, num_pages, 64, m);
      if (e == cudaSuccess)
        e = fp8 ? make_cache_tensor_map_fp8(cache, num_pages, 32, mr) : make_cache_tensor_map(cache, num_pages, 32, mr);
      if (e == cudaSuccess) *ms = *m;      // unused by these formats; any valid map
      CUtensorMap* m8 = reinterpret_cast<CUtensorMap*>(hm.tmap8);
      if (e == cudaSuccess) e = fp8 ? make_cache_tensor_map_fp8(cache, num_pages, 128, m8) : cudaSuccess;
      if (e == cudaSuccess && !fp8) *m8 = *m;
    }
    if (e != cudaSuccess) return e;
    hm.tmap_cache = cache;
    hm.tmap_pages = num_pages;
  }
  return cudaSuccess;
}

// Decode-kernel dispatch: the tensor-core kernel, with in-shared-memory e4m3 -> bf16
// conversion for an FP8 cache, or (per-tensor scale, MLA_OPT_FP8_MMA) FP8 tensor-core MMAs.
cudaError_t launch_decode(const Handle& h, const int32_t* ctx_len, int batch, const int32_t* block_table,
                          int bt_stride, const void* cache, int num_pages, const Workspace& ws, cudaStream_t st) {
  cudaError_t e = cache_maps(h, cache, num_pages);
  if (e != cudaSuccess) return e;
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(h.tmap);
  const CUtensorMap& map_rope = *reinterpret_cast<const CUtensorMap*>(h.tmap_rope);
  const CUtensorMap& map_scale = *reinterpret_cast<const CUtensorMap*>(h.tmap_scale);
  switch (h.cfg.cache_dtype) {
    case MLA_CACHE_FP8_E4M3:
      if (h.fp8_mma)
        return launch_decode_tc<kModeFp8Mma>(h, ctx_len, batch, block_table, bt_stride, num_pages,
                                             *reinterpret_cast<const CUtensorMap*>(h.tmap8), map_rope, map_scale, ws, st);
      return launch_decode_tc<kModeFp8>(h, ctx_len, batch, block_table, bt_stride, num_pages, map, map_rope,
                                        map_scale, ws, st);
    case MLA_CACHE_FP8_E4M3_BLOCK:
      return launch_decode_tc<kModeFp8Block>(h, ctx_len, batch, block_table, bt_stride, num_pages, map, map_rope,
                                             map_scale, ws, st);
    default:
      return launch_decode_tc<kModeBf16>(h, ctx_len, batch, block_table, bt_stride, num_pages, map, map_rope,
                                         map_scale, ws, st);
  }
}

}  // namespace mla
