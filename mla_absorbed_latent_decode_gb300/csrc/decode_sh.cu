// decode_sh.cu -- split-KV flash decode for few heads (n_h <= 32) over a bf16 paged cache: one
// CTA per work unit, heads on the N dimension of every MMA.
//
// What a unit computes is that of decode_tc.cu ("DeepSeek MLA 吸收式缓存：真实权重执行与
// FlashMLA 架构边界" §2.2-§2.4: the absorbed query scored against the shared 576-wide row,
// the softmax weights summing latent rows; "G5 MLA KV 访存建模设计规格" 附录 B: the stream
// consumed as it arrives).  With 128 heads the heads fill the MMAs' M dimension and O (128 x 512
// fp32) fills Tensor Memory, so a CTA pair splits the row and exchanges partial scores.  With
// 16 or 32 heads that layout wastes 3/4 or 7/8 of every MMA and of the exchange; here the
// operands swap instead:
//   S^T [64 tokens x N heads]   = C [64 x 576] . Q^T          (M = 64, K-major A = the cache tile)
//   O^T [512 latent x N heads] += C^T [512 x 64] . P^T [64 x N] (M = 128 per latent quarter; A = the
//                                                               same tile read MN-major)
// N = 16 or 32 (heads past n_h are zero rows of Q).  Tensor Memory then holds two score buffers
// (N columns each) and O^T (4 N columns), so one CTA takes the whole 576-wide row: no score
// exchange, and twice as many independent units as SM pairs.
//
// Roles (224 threads): warps 0-3 the softmax and the epilogue, warp 4 the TMA producer (a 2-deep
// ring of 72 KB stages: the tile's 9 boxes of 64 tokens x 64 columns, 128-byte swizzle), warp 5
// issues QK^T into score buffer j % 2, warp 6 issues P . C in tile order.  An M = 64 accumulator
// puts token r in lane 32 (r / 16) + r % 16, so lanes 0-15 of each softmax warp hold 16 tokens,
// each thread all N heads of its token.  The running maximum is per head and the same in every
// thread: the four warps exchange their tiles' maxima through shared memory (an mbarrier per
// tile parity), and the lazy rescale (only when a head's maximum grows by more than 8 in the
// log2 domain) rescales that head's O^T column in Tensor Memory after the previous P . C.  P^T
// (bf16, [N heads][64 tokens], 128-byte swizzle) is written by the softmax threads into one of
// two buffers, the K-major B operand of P . C.  Every wait is bounded; on a timeout the kernel
// sets MLA_CHECK_TIMEOUT, drains and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kShBox = 64 * 128;                     // one 64-token x 64-column bf16 box (8 KB)
constexpr int kShBoxes = kRow / 64;                  // 9: eight latent boxes and the RoPE key
constexpr int kShStage = kShBoxes * kShBox;          // 73,728 B
constexpr int kShThreads = 224;
constexpr int kShWarpProducer = 4, kShWarpQk = 5, kShWarpPv = 6;
constexpr float kShRescaleLog2 = 8.0f;

template <int N>
struct ShSmem {
  static constexpr int kQ = 2 * kShStage;            // the query: 9 boxes of N heads x 64 columns
  static constexpr int kQBox = N * 128;
  static constexpr int kP = kQ + kShBoxes * kQBox;   // P^T: two buffers of N heads x 64 tokens
  static constexpr int kPBuf = N * 128;
  static constexpr int kX = kP + 2 * kPBuf;          // per-warp maxima [2 parities][4][N], sums [4][N]
  static constexpr int kBars = kX + 3 * 4 * N * 4;
  static constexpr int kBytes = kBars + 256 + 1024;  // + alignment slack
  static_assert(kQ % 1024 == 0 && kP % 1024 == 0 && kQBox % 1024 == 0 && kPBuf % 1024 == 0, "swizzle atoms");
  static_assert(kBytes <= 232448, "dynamic shared memory");
};

struct ShBars {
  uint64_t full[2];           // tile landed (producer, tx)
  uint64_t empty[2];          // tile read by P . C (commit; QK^T of the tile finished before its softmax)
  uint64_t sfull[2];          // S^T(j) in score buffer j % 2 (commit)
  uint64_t sfree[2];          // S^T(j) loaded by the four softmax warps
  uint64_t pfull[2];          // P^T(j) written (four warps)
  uint64_t pdone[2];          // P . C of the tile in P buffer b done (commit)
  uint64_t xfull[2];          // the four warps' tile maxima written, by tile parity (four warps)
  uint64_t sums;              // the four warps' row sums written (four warps, single phase)
  uint64_t ofinal;            // single phase: the last P . C done (commit)
  uint64_t qfull;             // single phase: the query landed (producer, tx)
  uint64_t drain[2];          // every MMA of an issuer done
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(ShBars) <= 256, "barrier block");

__device__ __forceinline__ void sh_fail(ShBars* bars, unsigned* check) {
  if (atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
}

// Tensor Memory load of 16 or 32 consecutive columns of this warp's 32 lanes.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 32) {
    tmem_ld32(taddr, r);
  } else {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  }
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 32) {
    tmem_st32(taddr, r);
  } else {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
  }
}

template <int N>
__global__ void __launch_bounds__(kShThreads, 1)
decode_sh_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_q,
                 const int32_t* __restrict__ ctx_len, int n_h, const int32_t* __restrict__ block_table, int bt_stride,
                 int num_pages, float scale_log2, int stall, Workspace ws, unsigned* check) {
  using L = ShSmem<N>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  ShBars* bars = reinterpret_cast<ShBars*>(smem + L::kBars);
  volatile int* abort_flag = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit_idx = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
      mbar_init(smem_u32(&bars->sfull[i]), 1);
      mbar_init(smem_u32(&bars->sfree[i]), 4);
      mbar_init(smem_u32(&bars->pfull[i]), 4);
      mbar_init(smem_u32(&bars->pdone[i]), 1);
      mbar_init(smem_u32(&bars->xfull[i]), 4);
      mbar_init(smem_u32(&bars->drain[i]), 1);
    }
    mbar_init(smem_u32(&bars->sums), 4);
    mbar_init(smem_u32(&bars->ofinal), 1);
    mbar_init(smem_u32(&bars->qfull), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kShWarpProducer && lane == 0) {
    prefetch_tmap(&tmap);
    prefetch_tmap(&tmap_q);
  }
  __syncthreads();
  griddep_wait();                          // plan, absorbed queries and cache rows are inputs
  griddep_launch_dependents();
  // (the unit record is read together with the unit count: the grid never exceeds the workspace's units)
  const int n_units = ws.counters[0];
  const Unit unit = ws.units[unit_idx];
  if (unit_idx >= n_units) return;
  const int b = unit.b;
  const int n_tiles = unit.page_end - unit.page_begin;
  const int32_t* bt_row = block_table + (size_t)b * bt_stride + unit.page_begin;
  const int t_end = min(unit.page_end * kPage, ctx_len[b]);
  bool bad_page = false;                   // (producer thread) flagged after its last copy

  auto issue_tile = [&](int j, int page) {
    const int s = j & 1;
    if (page < 0 || page >= num_pages) {   // bad page id: read page 0 instead; the output is zeroed later
      bad_page = true;
      page = 0;
    }
    const uint32_t full = smem_u32(&bars->full[s]);
    mbar_arrive_expect_tx(full, (uint32_t)kShStage);
    for (int c = 0; c < kShBoxes; ++c) tma_load_2d(sbase + s * kShStage + c * kShBox, &tmap, 64 * c, page * kPage, full);
  };
  // a test of the bounded waits (stall == 2): the first unit never loads its tile 1
  const int withheld = (stall == 2 && unit_idx == 0 && n_tiles > 1) ? 1 : -1;
  if (warp == kShWarpProducer && lane == 0) {
    const int p0 = bt_row[0], p1 = n_tiles > 1 ? bt_row[1] : 0;
    issue_tile(0, p0);
    const uint32_t qf = smem_u32(&bars->qfull);
    mbar_arrive_expect_tx(qf, (uint32_t)(kShBoxes * L::kQBox));
    for (int c = 0; c < kShBoxes; ++c) tma_load_3d(sbase + L::kQ + c * L::kQBox, &tmap_q, 64 * c, 0, b, qf);
    if (n_tiles > 1 && withheld != 1) issue_tile(1, p1);
  }
  if (warp == kShWarpQk) {
    tmem_alloc(smem_u32(&bars->tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;   // columns: S^T buffers [0, N), [N, 2N); O^T quarter q at 2N + q N

  if (warp == kShWarpProducer) {
    if (lane == 0) {
      int issued = min(n_tiles, 2);
      for (int j = 2; j < n_tiles; ++j) {
        const int s = j & 1;
        const int page = bt_row[j];
        if (j + 2 < n_tiles) {             // the stage's next tile into L2
          const int pg = bt_row[j + 2];
          if (pg >= 0 && pg < num_pages)
            for (int c = 0; c < kShBoxes; ++c) tma_prefetch_2d(&tmap, 64 * c, pg * kPage);
        }
        if (!mbar_wait(smem_u32(&bars->empty[s]), ((j >> 1) & 1) ^ 1, abort_flag)) {
          sh_fail(bars, check);
          break;
        }
        issue_tile(j, page);
        issued = j + 1;
      }
      for (int j = max(0, issued - 2); j < issued; ++j) {   // every load issued lands before exit
        volatile int never = 0;
        if (j != withheld) mbar_wait(smem_u32(&bars->full[j & 1]), (j >> 1) & 1, &never);
      }
      if (bad_page && b >= 0) {
        atomicOr(check, kCheckPageId);
        ws.bad[b] = 1;
      }
    }
  } else if (warp == kShWarpQk) {
    // ------------------------------------------------------------ QK^T: S^T(j) = C(j) . Q^T
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(64, N, false, false);
      bool ok = mbar_wait(smem_u32(&bars->qfull), 0, abort_flag);
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        // the tile has landed, and S^T(j - 2) has been loaded from the buffer
        if (!mbar_wait(smem_u32(&bars->full[s]), (j >> 1) & 1, abort_flag) ||
            (j >= 2 && !mbar_wait(smem_u32(&bars->sfree[s]), ((j >> 1) - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = sbase + s * kShStage;
#pragma unroll
        for (int c = 0; c < kShBoxes; ++c) {
          const uint64_t a = sdesc_sw128(st + c * kShBox, 16, 1024);
          const uint64_t q = sdesc_sw128(sbase + L::kQ + c * L::kQBox, 16, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)      // 16 columns (32 bytes) per step inside the 128-byte rows
            mma_ss(tmem + s * N, a + (uint64_t)(2 * k), q + (uint64_t)(2 * k), idesc, (c | k) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->sfull[s]));
      }
      if (!ok) sh_fail(bars, check);
      mma_commit(smem_u32(&bars->drain[0]));
      volatile int never = 0;
      mbar_wait(smem_u32(&bars->drain[0]), 0, &never);
    }
  } else if (warp == kShWarpPv) {
    // ------------------------------------------------------------ P . C: O^T += C(j)^T . P^T(j)
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, N, true, false);
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j & 1;
        if (!mbar_wait(smem_u32(&bars->pfull[s]), (j >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t p = sdesc_sw128(sbase + L::kP + s * L::kPBuf, 16, 1024);
#pragma unroll
        for (int q = 0; q < 4; ++q) {      // latent quarter q: boxes 2q, 2q + 1 (128 columns)
          const uint64_t c = sdesc_sw128(sbase + s * kShStage + 2 * q * kShBox, kShBox, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)      // 16 tokens per step: 16 rows of the tile, 32 bytes of P^T's rows
            mma_ss(tmem + 2 * N + q * N, c + (uint64_t)(128 * k), p + (uint64_t)(2 * k), idesc,
                   (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->empty[s]));
        mma_commit(smem_u32(&bars->pdone[s]));
        if (j == n_tiles - 1) mma_commit(smem_u32(&bars->ofinal));
      }
      if (!ok) sh_fail(bars, check);
      mma_commit(smem_u32(&bars->drain[1]));
      volatile int never = 0;
      mbar_wait(smem_u32(&bars->drain[1]), 0, &never);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax and epilogue
    const int q4 = warp;
    const bool live = lane < 16;           // the M = 64 accumulator's rows sit in lanes 0-15
    const int tok = 16 * q4 + lane;        // this lane's token in the tile (live lanes)
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    float* xmax = reinterpret_cast<float*>(smem + L::kX);          // [parity][warp][N]
    float* xsum = xmax + 2 * 4 * N;                                  // [warp][N]
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, abort_flag));
    };
    float m[N], l[N];
#pragma unroll
    for (int h = 0; h < N; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
    }
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j & 1;
      if (!wait_all(&bars->sfull[s], (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      float x[N];
      {
        uint32_t r[N];
        tmem_ld_n<N>(lane_addr + s * N, r);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->sfree[s]));      // QK^T of tile j + 2 may overwrite
        const int valid = min(kPage, t_end - (unit.page_begin + j) * kPage);
        const bool use = live && tok < valid;
#pragma unroll
        for (int h = 0; h < N; ++h) x[h] = use ? __uint_as_float(r[h]) * scale_log2 : -INFINITY;
        if (live && !use) {                // a partial last page: its rows past the context become zeros,
          uint4* row = reinterpret_cast<uint4*>(smem + s * kShStage + tok * 128);   // so P = 0 meets finite values
#pragma unroll 1
          for (int c = 0; c < kShBoxes - 1; ++c)
#pragma unroll
            for (int k = 0; k < 8; ++k) row[c * (kShBox / 16) + k] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // the tile's maximum per head: over the 16 tokens of this warp, then over the four warps
      float* xw = xmax + (s * 4 + q4) * N;
#pragma unroll
      for (int h = 0; h < N; ++h) {
        float v = x[h];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
        if (lane == 0) xw[h] = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->xfull[s]));
      if (!wait_all(&bars->xfull[s], (j >> 1) & 1)) { ok = false; break; }
      bool grow = false;
      float alpha[N];
#pragma unroll
      for (int h = 0; h < N; ++h) {
        const float* xs = xmax + s * 4 * N + h;
        const float mt = fmaxf(fmaxf(xs[0], xs[N]), fmaxf(xs[2 * N], xs[3 * N]));
        const float m_new = mt > m[h] + kShRescaleLog2 ? mt : m[h];
        alpha[h] = m_new == m[h] ? 1.0f : (m[h] == -INFINITY ? 0.0f : exp2f(m[h] - m_new));
        grow |= m_new != m[h];
        m[h] = m_new;
      }
      if (grow) {                          // (the same decision in every thread: from the same maxima)
#pragma unroll
        for (int h = 0; h < N; ++h) l[h] *= alpha[h];
        if (j > 0) {
          // O^T's columns of the growing heads, times alpha, once P . C of tile j - 1 is done
          if (!wait_all(&bars->pdone[(j - 1) & 1], ((j - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t r[N];
            tmem_ld_n<N>(lane_addr + 2 * N + q * N, r);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < N; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * alpha[h]);
            tmem_st_n<N>(lane_addr + 2 * N + q * N, r);
          }
          tmem_st_wait();
          tc_fence_before();
        }
      }
      // P = 2^(x - m) (0 past the context), its sums, and P^T into buffer j % 2 once P . C of
      // tile j - 2 has read it: row h = head, 64 tokens (128 bytes, 128-byte swizzle)
      if (j >= 2 && !wait_all(&bars->pdone[s], ((j >> 1) - 1) & 1)) { ok = false; break; }
      uint8_t* pbuf = smem + L::kP + s * L::kPBuf;
#pragma unroll
      for (int h = 0; h < N; ++h) {
        const float p = exp2f(x[h] - m[h]);
        l[h] += live ? p : 0.0f;
        if (live)
          *reinterpret_cast<__nv_bfloat16*>(pbuf + h * 128 + ((((tok >> 3) ^ (h & 7))) << 4) + (tok & 7) * 2) =
              __float2bfloat16_rn(p);
      }
      fence_proxy_async_smem();            // generic writes before the tensor core reads them
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->pfull[s]));
    }
    if (!ok) sh_fail(bars, check);
    // ---- epilogue: the row sums over the 64 tokens of a tile, summed over the four warps
#pragma unroll
    for (int h = 0; h < N; ++h) {
      float v = live ? l[h] : 0.0f;
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) xsum[q4 * N + h] = v;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars->sums));
    bool fin = ok && n_tiles > 0;
    if (fin) {
      fin = wait_all(&bars->sums, 0) && wait_all(&bars->ofinal, 0);
      if (!fin) sh_fail(bars, check);
    }
    if (fin) {
      tc_fence_after();
      float inv[N];
#pragma unroll
      for (int h = 0; h < N; ++h) inv[h] = 1.0f / (xsum[h] + xsum[N + h] + xsum[2 * N + h] + xsum[3 * N + h]);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {        // lane = latent row 128 q + 32 q4 + lane of every head
        uint32_t r[N];
        tmem_ld_n<N>(lane_addr + 2 * N + q * N, r);
        tmem_ld_wait();
        const int col = 128 * q + 32 * q4 + lane;
        if (unit.part < 0) {
          __nv_bfloat16* dst = ws.o_lat + (size_t)b * n_h * kDc + col;
#pragma unroll
          for (int h = 0; h < N; ++h)
            if (h < n_h) dst[(size_t)h * kDc] = __float2bfloat16_rn(__uint_as_float(r[h]) * inv[h]);
        } else {
          float* dst = ws.part_o + (size_t)unit.part * n_h * kDc + col;
#pragma unroll
          for (int h = 0; h < N; ++h)
            if (h < n_h) dst[(size_t)h * kDc] = __uint_as_float(r[h]) * inv[h];
        }
      }
      if (unit.part >= 0 && q4 == 0 && lane == 0) {
#pragma unroll
        for (int h = 0; h < N; ++h)
          if (h < n_h) ws.part_lse[(size_t)unit.part * n_h + h] = (m[h] - log2f(inv[h])) * 0.69314718055994531f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kShWarpQk) tmem_dealloc(tmem, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 sh_encoder() {
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

// The absorbed query [B][n_h][576] as (column, head, sequence), boxes of 64 columns x N heads x 1
// sequence, 128-byte swizzle (heads past n_h arrive as zeros).
cudaError_t sh_query_map(const void* q_abs, int batch, int n_h, int N, CUtensorMap* map) {
  auto enc = sh_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kRow, (cuuint64_t)n_h, (cuuint64_t)batch};
  const cuuint64_t strides[2] = {(cuuint64_t)kRow * 2, (cuuint64_t)kRow * 2 * n_h};
  const cuuint32_t box[3] = {64, (cuuint32_t)N, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q_abs), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

template <int N>
cudaError_t launch_sh(const Handle& h, const int32_t* ctx_len, int batch, const int32_t* block_table, int bt_stride,
                      int num_pages, const Workspace& ws, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_sh_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         ShSmem<N>::kBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  alignas(64) CUtensorMap map_q;
  cudaError_t e = sh_query_map(ws.q_abs, batch, h.cfg.n_h, N, &map_q);
  if (e != cudaSuccess) return e;
  const float scale_log2 = h.scale * 1.4426950408889634f;
  return launch_pdl(decode_sh_kernel<N>, dim3(ws.max_units), dim3(kShThreads), ShSmem<N>::kBytes, st,
                    *reinterpret_cast<const CUtensorMap*>(h.tmap), map_q, ctx_len, h.cfg.n_h, block_table, bt_stride,
                    num_pages, scale_log2, h.test_stall, ws, h.check_word);
}

}  // namespace

bool small_head_decode(const Handle& h) {
  return h.small_heads && h.cfg.cache_dtype == MLA_CACHE_BF16 && h.cfg.n_h <= kShMaxHeads;
}

cudaError_t launch_decode_small_heads(const Handle& h, const int32_t* ctx_len, int batch, const int32_t* block_table,
                                      int bt_stride, const void* cache, int num_pages, const Workspace& ws,
                                      cudaStream_t st) {
  cudaError_t e = cache_maps(h, cache, num_pages);
  if (e != cudaSuccess) return e;
  if (h.cfg.n_h <= 16) return launch_sh<16>(h, ctx_len, batch, block_table, bt_stride, num_pages, ws, st);
  return launch_sh<32>(h, ctx_len, batch, block_table, bt_stride, num_pages, ws, st);
}

}  // namespace mla
