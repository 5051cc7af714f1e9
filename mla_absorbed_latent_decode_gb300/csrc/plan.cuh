// plan.cuh -- the split-KV planner of a decode step (integer work, one CTA of any
// size that is a multiple of 32 threads).  It runs as an extra CTA of the query-
// absorption kernel, concurrently with the absorption GEMMs.
//
// Input: ctx_len[B].  Output (in the workspace): a list of units, each a
// contiguous page range of one sequence, per sequence the index of its first unit
// and its unit count, and a zeroed per-sequence "bad page" flag.
//
//   valid(b)   = 1 <= ctx_len[b] <= max_ctx; otherwise the sequence gets no unit,
//                its output is zeroed and a check bit is set.  (Page ids are
//                checked by the decode kernel as it reads them: a bad one sets
//                bad[b], and the sequence's output is zeroed after the decode.)
//   pages(b)   = ceil(ctx_len[b] / 64) for a valid sequence, else 0.
//   target     = the smallest page count >= ceil(sum_b pages(b) / num_pairs) with
//                sum_b ceil(pages(b) / target) <= max(num_pairs, valid sequences):
//                pages one SM pair streams, chosen so that the units fit in one wave
//                of SM pairs (no pair runs two units back to back while others idle).
//   nsplit(b)  = ceil(pages(b) / target), or min(forced, pages(b)) when the
//                split count is forced.
//   unit j of b covers pages [j * pages(b) / nsplit(b), (j+1) * pages(b) / nsplit(b)).
//
// Units are numbered sequence by sequence.  A unit that is a whole sequence
// writes the final latent sum; the others write partials (slot = unit index)
// merged later by log-sum-exp.  Splitting is not on the pages; it is needed
// because one sequence's context (up to 65536 tokens here) is far more work
// than one SM pair should take when the batch is small.
#pragma once

#include "internal.cuh"

namespace mla {
namespace plan_detail {

constexpr int kPlanSmemSeqs = 16384;     // page counts of up to this many sequences stay in shared memory

// Block-wide reductions over one value per thread (red: >= 33 ints of shared memory).
__device__ __forceinline__ int block_reduce(int v, int* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const int y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? max(v, y) : v + y;
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = is_max ? 0 : 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = is_max ? max(t, red[w]) : t + red[w];
  return t;
}

// Exclusive prefix sum over one value per thread; returns the block total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) red[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) before += red[w];
    all += red[w];
  }
  *total = all;
  return before + x - v;
}

__device__ __forceinline__ int pages_of(int b, const int* pages_s, const Workspace& ws) {
  return b < kPlanSmemSeqs ? pages_s[b] : ws.seqs[b].nsplit;
}

}  // namespace plan_detail

// The planner body.  `pages_s` is shared memory for min(B, kPlanSmemSeqs) ints, `red` for 33.
__device__ void plan_block(const int32_t* __restrict__ ctx_len, int B, int max_ctx, int num_pairs, int forced,
                           const Workspace& ws, unsigned* check, int* pages_s, int* red) {
  using namespace plan_detail;
  const int lane = threadIdx.x & 31;
  // 1. context lengths, one load per thread per pass; bad-page flags cleared
  unsigned flags = 0;
  int my_pages = 0, my_valid = 0, my_max = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int L = ctx_len[b];
    int np = 0;
    if (L < 1 || L > max_ctx) flags |= kCheckCtxLen;
    else np = (L + kPage - 1) / kPage;
    if (b < kPlanSmemSeqs) pages_s[b] = np; else ws.seqs[b].nsplit = np;
    ws.bad[b] = 0;
    my_pages += np;
    my_valid += np > 0;
    my_max = max(my_max, np);
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (flags && lane == 0) atomicOr(check, flags);
  const int total_pages = block_reduce(my_pages, red, false);
  __syncthreads();
  const int valid_seqs = block_reduce(my_valid, red, false);
  __syncthreads();
  const int max_pages = block_reduce(my_max, red, true);
  // 2. smallest page target whose split count fits in one wave of SM pairs (binary search
  //    from an even share of the pages); with at least as many sequences as pairs nothing
  //    is split
  const int pairs = max(1, num_pairs);
  int lo = max(1, (total_pages + pairs - 1) / pairs), hi = max(lo, max_pages);
  const int budget = max(pairs, valid_seqs);
  while (lo < hi) {
    const int mid = lo + (hi - lo) / 2;
    int n = 0;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      const int np = pages_of(b, pages_s, ws);
      n += np == 0 ? 0 : (np + mid - 1) / mid;
    }
    __syncthreads();
    if (block_reduce(n, red, false) <= budget) hi = mid; else lo = mid + 1;
  }
  const int target = lo;
  // 3. split counts, prefix-summed chunk by chunk into first_unit
  int base = 0;
  for (int b0 = 0; b0 < B; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    int ns = 0, np = 0;
    if (b < B) {
      np = pages_of(b, pages_s, ws);
      ns = np == 0 ? 0 : (forced > 0 ? min(forced, np) : (np + target - 1) / target);
    }
    __syncthreads();
    int chunk_total = 0;
    const int off = block_exclusive_scan(ns, red, &chunk_total);
    if (b < B) {
      const int first = base + off;
      for (int j = 0; j < ns; ++j) {
        Unit u;
        u.b = b;
        u.page_begin = (int)((long long)j * np / ns);
        u.page_end = (int)((long long)(j + 1) * np / ns);
        u.part = ns > 1 ? first + j : -1;
        ws.units[first + j] = u;
      }
      SeqPlan sp;
      sp.first_unit = first;
      sp.nsplit = ns;
      ws.seqs[b] = sp;
    }
    base += chunk_total;
  }
  if (threadIdx.x == 0) {
    ws.counters[0] = base;
    ws.counters[1] = base;
  }
}

}  // namespace mla
