// head_gemm.cu -- the two per-head weight contractions of a decode step, on
// tcgen05 tensor cores, batched over every sequence so each weight byte is read
// from HBM once:
//
//   query absorption ("DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2)
//     Q_lat[:, h] [B x 512] = q_nope[:, h] [B x 128] . W_UK[h] [128 x 512]
//     plus the RoPE part of the query rotated at ctx_len - 1 (§2.4);
//   value up-projection after the latent sum (§2.3)
//     out^T[h]   [128 x B] = W_UV[h] [128 x 512] . o_lat[:, h]^T [512 x B].
//
// The query-absorption launch has one extra CTA that runs the split planner
// (plan.cuh) while the GEMM CTAs wait for their weights.  Before the
// up-projection, split sequences' partial latent sums are merged by log-sum-exp
// into the GEMM's operand tile (a standard identity, not on the pages); invalid sequences, and
// sequences whose block table held a bad page id, get a zero latent, hence a zero
// output.
//
// One CTA per (head, tile of sequences): the whole weight matrix of the head
// (128 KB) and the tile's rows arrive by TMA in 128-byte-swizzled 64-column
// boxes, all issued up front, each group of boxes on its own mbarrier so the MMAs
// over a group start as soon as it lands; one thread issues the MMAs from
// precomputed descriptors; warps 0-3 (one per 32 TMEM lanes) run the epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.cuh"
#include "plan.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr int kBox = 128 * 128;                        // one 64-column x 128-row bf16 box: 16 KB

// query absorption: one CTA per (head, tile of 128 sequences); sequences are the M rows
constexpr int kQaM = 128;
constexpr int kQaSmem = 8 * kBox + 2 * kBox + 1024 + 1024;
// value up-projection: one CTA per (head, tile of up to 64 sequences); the 128 value rows are M.
// The tile (the MMA's N) is 64, 32 or 16 sequences, chosen at launch so that small batches
// still spread over many SMs.
constexpr int kUpN = 64;
constexpr int kUpSmem = 8 * kBox + 8 * kUpN * 128 + 1024 + 1024;

struct GemmBars {
  uint64_t full[8];          // per 64-column box (up-projection: weight box + latent box)
  uint64_t done[2];          // MMAs of a half (query absorption) / of the whole tile (up-projection)
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 3-D TMA of one 64-column chunk of B rows (tensor [B][n_h][width]: column, head, sequence).
__device__ __forceinline__ void load_rows(uint32_t dst, const CUtensorMap* m, int col, int h, int n0, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(col), "r"(h), "r"(n0), "r"(bar)
      : "memory");
}

// Q_lat[n0 .. n0 + 128, h] = q_nope[n0 .., h] . W_UK[h]: M = 128 sequences (rows past B arrive
// as zeros), N = 2 x 256 latent columns, K = 128.  A = the query rows, K-major; B = W_UK[h]
// read MN-major (each box: 128 K-rows of 64 latent columns).  The CTA with blockIdx.x == n_h
// runs the split planner instead.
__global__ void __launch_bounds__(kThreads, 1)
q_absorb_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_out, int B, int n_h,
                int max_ctx, const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ ctx_len,
                const float2* __restrict__ rope_cs, int max_position, int num_pairs, int forced, int stall,
                Workspace ws, unsigned* check) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int red[64];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (blockIdx.x == n_h) {
    // ---- the split planner (one CTA; context lengths are inputs of the step)
    griddep_wait();
    griddep_launch_dependents();
    if (blockIdx.z == 0) plan_block(ctx_len, B, max_ctx, num_pairs, forced, ws, check, reinterpret_cast<int*>(smem), red);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + 10 * kBox);
  volatile int* abort_flag = &bars->abort;
  const int h = blockIdx.x, n0 = blockIdx.z * kQaM;
  // barriers: full[0] = the query rows, full[1 + hh] = weight boxes of latent half hh
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&bars->full[i]), 1);
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bars->done[i]), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(smem_u32(&bars->tmem_base), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t w_st = sbase, a_st = sbase + 8 * kBox;
  if (tid == 0) {
    for (int hh = 0; hh < 2; ++hh) {        // each latent half on its own barrier: its MMAs start as it lands
      const uint32_t wf = smem_u32(&bars->full[1 + hh]);
      mbar_arrive_expect_tx(wf, 4u * kBox);
      for (int i = 4 * hh; i < 4 * hh + 4; ++i) tma_load_2d(w_st + i * kBox, &tm_w, 64 * i, 128 * h, wf);
    }
    griddep_wait();                        // the queries may come from the previous kernel
    griddep_launch_dependents();
    const uint32_t qf = smem_u32(&bars->full[0]);
    if (stall != 1) {                      // (a test of the bounded waits, stall == 1, withholds the copy)
      mbar_arrive_expect_tx(qf, 2u * kBox);
      load_rows(a_st, &tm_q, 0, h, n0, qf);
      load_rows(a_st + kBox, &tm_q, 64, h, n0, qf);
    }
    bool ok = mbar_wait(qf, 0, abort_flag);
    constexpr uint32_t idesc = idesc_bf16_f32(128, 256, false, true);
    const uint64_t a0 = sdesc_sw128(a_st, 16, 1024), b0 = sdesc_sw128(w_st, kBox, 1024);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {       // latent columns [256 hh, 256 hh + 256): boxes 4 hh .. 4 hh + 3
      ok = ok && mbar_wait(smem_u32(&bars->full[1 + hh]), 0, abort_flag);
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int k = 0; k < 8; ++k)        // K rows [16 k, 16 k + 16): A box k / 4 at 32 B steps; B 2 KB steps
          mma_ss(tmem + 256 * hh, a0 + (uint64_t)(((k >> 2) * kBox + (k & 3) * 32) >> 4),
                 b0 + (uint64_t)((hh * 4 * kBox + k * 2048) >> 4), idesc, k > 0 ? 1u : 0u);
      }
      mma_commit(smem_u32(&bars->done[hh]));
    }
    if (!ok) {
      if (atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
      for (int i = 0; i < 3; ++i) {           // let every copy in flight land before the CTA exits
        volatile int never = 0;
        mbar_wait(smem_u32(&bars->full[i]), 0, &never);
      }
    }
  }
  griddep_wait();
  // RoPE part of the query, rotated at position ctx_len - 1 (clamped into the table): one
  // sequence per thread of warps 1-3 (warp 0 issues the copies and MMAs meanwhile), every
  // load of a sequence issued before any is used
  if (warp > 0) {
    for (int j = tid - 32; j < min(B - n0, kQaM); j += kThreads - 32) {
      const int b = n0 + j;
      const int pos = min(max(ctx_len[b] - 1, 0), max_position - 1);
      const uint4* qs = reinterpret_cast<const uint4*>(q + ((size_t)b * n_h + h) * kDq + kDn);
      const float4* cs = reinterpret_cast<const float4*>(rope_cs + (size_t)pos * (kDr / 2));
      uint4 qv[8];
      float4 cv[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = qs[i];
#pragma unroll
      for (int i = 0; i < 16; ++i) cv[i] = cs[i];
      uint4* dst = reinterpret_cast<uint4*>(ws.q_abs + ((size_t)b * n_h + h) * kRow + kDc);
#pragma unroll
      for (int i = 0; i < 8; ++i) {            // pairs 4 i .. 4 i + 3
        const uint32_t w[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
        const float4 c01 = cv[2 * i], c23 = cv[2 * i + 1];
        const float cs_c[4] = {c01.x, c01.z, c23.x, c23.z}, cs_s[4] = {c01.y, c01.w, c23.y, c23.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x0 = __uint_as_float(w[k] << 16), x1 = __uint_as_float(w[k] & 0xFFFF0000u);
          o[k] = bf16x2_bits(x0 * cs_c[k] - x1 * cs_s[k], x1 * cs_c[k] + x0 * cs_s[k]);
        }
        dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  __syncwarp();
  // epilogue, one latent half at a time (half 1's MMAs overlap half 0's epilogue): thread =
  // sequence (TMEM lane), 32 latent values per load.  The half is staged in its (now free)
  // weight boxes, 64 columns x 128 rows each, 128-byte swizzled, and written out by TMA
  // stores (rows past B are not written).
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  const int r = 32 * warp + lane;
  bool ok = true;
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    ok = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->done[hh]), 0, abort_flag));
    tc_fence_after();
    if (ok) {
#pragma unroll 1
      for (int g = 8 * hh; g < 8 * hh + 8; ++g) {
        uint32_t v[32];
        tmem_ld32(lane_addr + 32 * g, v);
        tmem_ld_wait();
        uint8_t* row = smem + (g >> 1) * kBox + r * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = (g & 1) * 4 + i;             // 16-byte chunk of the box row
          *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) * 16)) =
              make_uint4(bf16x2_bits(__uint_as_float(v[8 * i]), __uint_as_float(v[8 * i + 1])),
                         bf16x2_bits(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                         bf16x2_bits(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                         bf16x2_bits(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
        }
      }
      fence_proxy_async_smem();
    }
    __syncthreads();
    if (ok && tid == 0) {
      for (int i = 4 * hh; i < 4 * hh + 4; ++i) tma_store_3d(&tm_out, sbase + i * kBox, 64 * i, h, n0);
      bulk_commit_group();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
  if (tid == 0) bulk_wait_read();          // the staging read before the CTA exits (the writes complete with the grid)
}

// out^T[h] = W_UV[h] . o_lat[:, h]^T for the sequences n0 .. n0 + n_pad of this CTA, after
// merging split sequences' partials of head h by log-sum-exp straight into the operand tile in
// shared memory (zero latent for an invalid sequence or one with a bad page id; unsplit
// sequences' rows come from o_lat, written by the decode).  Eight warps take the merge; warps
// 0-3 (one per 32 TMEM lanes) run the epilogue.
constexpr int kUpThreads = 256;
__global__ void __launch_bounds__(kUpThreads, 1)
up_project_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_o, int B, int n_h,
                  int n_pad, int n_tile, Workspace ws, __nv_bfloat16* __restrict__ out, unsigned* check) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int2 plan_s[kUpN];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + 8 * kBox + 8 * kUpN * 128);
  volatile int* abort_flag = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, n0 = blockIdx.z * n_tile;
  // the TMA box height = the MMA's N, at least 16 (rows past B arrive as zeros; with a tile of 8
  // sequences the next tile's rows come along and their results are dropped)
  const int n_here = max(16, min(n_pad, n_tile));
  const uint32_t b_bytes = (uint32_t)n_here * 128;
  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(smem_u32(&bars->full[i]), 1);
    mbar_init(smem_u32(&bars->done[0]), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(smem_u32(&bars->tmem_base), 64); tmem_relinquish(); }
  // weights do not depend on the merge: start their loads at once.  Box i of the weights and
  // box i of the latent rows complete one barrier, so the MMAs over K box i start as it lands.
  const uint32_t a_st = sbase, b_st = sbase + 8 * kBox;
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < 8; ++i) {
      mbar_arrive_expect_tx(smem_u32(&bars->full[i]), (uint32_t)kBox + b_bytes);
      tma_load_2d(a_st + i * kBox, &tm_w, 64 * i, 128 * h, smem_u32(&bars->full[i]));
    }
  }
  // The latent rows of the tile's sequences (the B operand, 128-byte-swizzled boxes of 64
  // columns) are requested by TMA right after the dependency wait, whatever the tile holds; the
  // rows of split, invalid or bad-page sequences are then overwritten in shared memory, once the
  // boxes have landed, by the merge pass: one warp per such sequence (zeros for an invalid or
  // bad-page one).  The plan entries of the tile are loaded together first (one per thread),
  // before the dependency wait: the plan comes from the query-absorption launch, two launches
  // back and complete when this grid starts; the bad-page flags, written by the decode, after it.
  // A split sequence's partial slots are its unit indices first_unit .. first_unit + nsplit - 1;
  // lane k holds split k's log-sum-exp (32 splits per load, one load each), and the partials are
  // requested eight splits at a time, the first batch together with the log-sum-exps, merged
  // with a running maximum: one or two L2 round trips per merge.
  const int n_seq = min(B - n0, n_tile);
  int2 sp = make_int2(0, 0);
  if (tid < n_seq) sp = __ldcg(reinterpret_cast<const int2*>(ws.seqs) + n0 + tid);
  griddep_wait();                          // the latent sums and bad-page flags of the decode
  griddep_launch_dependents();
  if (tid == 0)
    for (int i = 0; i < 8; ++i) load_rows(b_st + i * b_bytes, &tm_o, 64 * i, h, n0, smem_u32(&bars->full[i]));
  const int bad = tid < n_seq ? ws.bad[n0 + tid] : 0;
  if (tid < n_seq) plan_s[tid] = make_int2(sp.x, bad ? 0 : sp.y);
  __syncthreads();
  bool rows_landed = false;                // (this warp has waited for the row boxes)
  auto wait_rows = [&]() {
    if (rows_landed) return;
    rows_landed = true;
    bool landed = true;
    for (int i = 0; i < 8; ++i) landed = mbar_wait(smem_u32(&bars->full[i]), 0, abort_flag) && landed;
    if (!landed && atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
  };
  // lane l's 16 values [16 l, 16 l + 16) of row j: box l / 4, 16-byte chunks 2 (l % 4) and
  // 2 (l % 4) + 1, each at its swizzled place (chunk c of row j at c ^ (j % 8))
  auto row_chunk = [&](int j, int c) -> uint4* {
    return reinterpret_cast<uint4*>(smem + 8 * kBox + (lane >> 2) * b_bytes + j * 128 + ((c ^ (j & 7)) * 16));
  };
  bool wrote = false;
  for (int j = warp; j < n_seq; j += kUpThreads / 32) {
    const int first = plan_s[j].x, nsplit = plan_s[j].y;
    if (nsplit == 1) continue;
    wrote = true;
    const int c0 = 2 * (lane & 3);
    if (nsplit == 0) {
      wait_rows();
      *row_chunk(j, c0) = make_uint4(0, 0, 0, 0);
      *row_chunk(j, c0 + 1) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const float* lse = ws.part_lse + (size_t)first * n_h + h;
    float acc[16], den = 0.0f, m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
    const float4* src0 = reinterpret_cast<const float4*>(ws.part_o + ((size_t)first * n_h + h) * kDc) + 4 * lane;
    const size_t slot4 = (size_t)n_h * kDc / 4;                 // one partial slot, in float4
    for (int k0 = 0; k0 < nsplit; k0 += 32) {
      const int kn = min(32, nsplit - k0);
      const float l_lane = lane < kn ? __ldcg(lse + (size_t)(k0 + lane) * n_h) : -INFINITY;
      for (int k1 = 0; k1 < kn; k1 += 8) {
        float4 v[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            v[u][i] = k1 + u < kn ? __ldcg(src0 + (size_t)(k0 + k1 + u) * slot4 + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        float lb[8], mb = m;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          lb[u] = __shfl_sync(0xffffffffu, l_lane, (k1 + u) & 31);
          if (k1 + u < kn) mb = fmaxf(mb, lb[u]);
        }
        if (mb > m) {                        // the running maximum grows: rescale what is summed
          const float sc = expf(m - mb);       // 0 on the first batch (m = -inf)
          den *= sc;
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] *= sc;
          m = mb;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float w = k1 + u < kn ? expf(lb[u] - m) : 0.0f;
          den += w;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[4 * i] = fmaf(w, v[u][i].x, acc[4 * i]);
            acc[4 * i + 1] = fmaf(w, v[u][i].y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(w, v[u][i].z, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(w, v[u][i].w, acc[4 * i + 3]);
          }
        }
      }
    }
    const float inv = 1.0f / den;
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = bf16x2_bits(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    wait_rows();                            // the TMA rows landed: this row may now be replaced
    *row_chunk(j, c0) = make_uint4(o[0], o[1], o[2], o[3]);
    *row_chunk(j, c0 + 1) = make_uint4(o[4], o[5], o[6], o[7]);
  }
  if (wrote) fence_proxy_async_smem();     // these rows are read below by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, n_here, false, false);
    const uint64_t a0 = sdesc_sw128(a_st, 16, 1024), b0 = sdesc_sw128(b_st, 16, 1024);
    bool ok = true;
    for (int c = 0; c < 8 && ok; ++c) {
      ok = mbar_wait(smem_u32(&bars->full[c]), 0, abort_flag);
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem, a0 + (uint64_t)((c * kBox + 32 * k) >> 4), b0 + (uint64_t)((c * b_bytes + 32 * k) >> 4), idesc,
                 (c > 0 || k > 0) ? 1u : 0u);
      }
    }
    if (!ok) {
      if (atomicExch(&bars->abort, 1) == 0) atomicOr(check, kCheckTimeout);
      for (int c = 0; c < 8; ++c) {           // let every copy in flight land before the CTA exits
        volatile int never = 0;
        mbar_wait(smem_u32(&bars->full[c]), 0, &never);
      }
    }
    mma_commit(smem_u32(&bars->done[0]));
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->done[0]), 0, abort_flag));
  tc_fence_after();
  // epilogue: thread = value row v (TMEM lane) holding up to 64 sequences; transposed through
  // shared memory (the weight region is free now) into [sequence][128 v] bf16 rows, then
  // written with 16-byte stores, one 256-byte row per sequence
  const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem);     // [64][128]
  const int v = 32 * warp + lane;
  if (ok && warp < 4) {
    for (int c0 = 0; c0 < n_here; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(lane_addr + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) tile[(c0 + i) * kDv + v] = __float2bfloat16_rn(__uint_as_float(r[i]));
    }
  }
  __syncthreads();
  if (ok) {
    for (int i = tid; i < n_seq * (kDv / 8); i += kUpThreads) {
      const int j = i / (kDv / 8), c = i % (kDv / 8);
      reinterpret_cast<uint4*>(out + ((size_t)(n0 + j) * n_h + h) * kDv)[c] =
          reinterpret_cast<const uint4*>(tile + j * kDv)[c];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
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

}  // namespace

cudaError_t prepare_weight_maps(Handle& h) {
  cudaError_t e = weight_map(h.w_uk, h.cfg.n_h, reinterpret_cast<CUtensorMap*>(h.tmap_wuk));
  if (e != cudaSuccess) return e;
  return weight_map(h.w_uv, h.cfg.n_h, reinterpret_cast<CUtensorMap*>(h.tmap_wuv));
}

cudaError_t launch_q_absorb(const Handle& h, const __nv_bfloat16* q, const int32_t* ctx_len, int batch,
                            int max_ctx, const Workspace& ws, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(q_absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQaSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  static_assert(kQaSmem - 2048 >= (int)sizeof(int) * plan_detail::kPlanSmemSeqs, "planner page counts");
  alignas(64) CUtensorMap tq, tout;
  cudaError_t e = rows_map(q, batch, h.cfg.n_h, kDq, kQaM, &tq);
  if (e != cudaSuccess) return e;
  if ((e = rows_map(ws.q_abs, batch, h.cfg.n_h, kRow, kQaM, &tout)) != cudaSuccess) return e;
  dim3 grid(h.cfg.n_h + 1, 1, (batch + kQaM - 1) / kQaM);     // + 1: the planner CTA
  return launch_pdl(q_absorb_kernel, grid, dim3(kThreads), kQaSmem, st,
                    *reinterpret_cast<const CUtensorMap*>(h.tmap_wuk), tq, tout, batch, h.cfg.n_h, max_ctx, q, ctx_len,
                    (const float2*)h.rope_cs, h.cfg.max_position, decode_wave(h), h.force_splits, h.test_stall, ws,
                    h.check_word);
}

cudaError_t launch_combine_uv(const Handle& h, int batch, const Workspace& ws, __nv_bfloat16* out, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(up_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUpSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int n_pad = ((batch + 15) / 16) * 16;
  // the largest tile of 64 / 32 / 16 / 8 sequences that still gives half the SMs a CTA (else 8):
  // with few heads, small tiles spread the split merges (one warp per sequence) over more CTAs
  int n_tile = kUpN;
  while (n_tile > 8 && (long long)h.cfg.n_h * ((batch + n_tile - 1) / n_tile) < h.num_sms / 2) n_tile /= 2;
  alignas(64) CUtensorMap to;
  cudaError_t e = rows_map(ws.o_lat, batch, h.cfg.n_h, kDc, max(16, min(n_pad, n_tile)), &to);
  if (e != cudaSuccess) return e;
  dim3 grid(h.cfg.n_h, 1, (batch + n_tile - 1) / n_tile);
  return launch_pdl(up_project_kernel, grid, dim3(kUpThreads), kUpSmem, st,
                    *reinterpret_cast<const CUtensorMap*>(h.tmap_wuv), to, batch, h.cfg.n_h, n_pad, n_tile, ws, out,
                    h.check_word);
}

}  // namespace mla
