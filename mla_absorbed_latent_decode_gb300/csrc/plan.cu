// plan.cu -- the split-KV planner of a decode step (integer work, one CTA).
//
// Input: ctx_len[B] and the block table.  Output (in the workspace): a list of
// units, each a contiguous page range of one sequence, and per sequence the
// index of its first unit and its unit count.
//
//   valid(b)   = 1 <= ctx_len[b] <= max_ctx and every page id of the sequence
//                lies in [0, num_pages); otherwise the sequence gets no unit,
//                its output is zeroed and a check bit is set.
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
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemSeqs = 16384;     // page counts of up to this many sequences stay in shared memory

__device__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = 0;
  if (threadIdx.x < 32) {
    t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// Exclusive prefix sum over one value per thread; returns the block total in *total.
__device__ int block_exclusive_scan(int v, int* red, int* total) {
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
  if (threadIdx.x < 32) {
    int w = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    red[threadIdx.x] = s - w;  // exclusive warp offsets
    if (threadIdx.x == 31) red[32] = s;
  }
  __syncthreads();
  const int r = red[warp] + x - v;
  *total = red[32];
  __syncthreads();
  return r;
}


// pages(b): from shared memory for the first kPlanSmemSeqs sequences, else parked in seqs[b].nsplit
__device__ __forceinline__ int pages_of(int b, const int* pages_s, const Workspace& ws) {
  return b < kPlanSmemSeqs ? pages_s[b] : ws.seqs[b].nsplit;
}
// Per-thread partial counts over this thread's sequences.
__device__ int count_units(int B, const int* pages_s, const Workspace& ws, int target) {
  int n = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int np = pages_of(b, pages_s, ws);
    n += np == 0 ? 0 : (np + target - 1) / target;
  }
  return n;
}
__device__ int count_valid(int B, const int* pages_s, const Workspace& ws) {
  int n = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) n += pages_of(b, pages_s, ws) > 0;
  return n;
}
__device__ int thread_max_pages(int B, const int* pages_s, const Workspace& ws) {
  int m = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) m = max(m, pages_of(b, pages_s, ws));
  return m;
}
__device__ int block_max(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (threadIdx.x == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(
    const int32_t* __restrict__ ctx_len, int B, int max_ctx, const int32_t* __restrict__ block_table,
    int bt_stride, int num_pages, int num_pairs, int forced, Workspace ws, unsigned* check) {
  __shared__ int red[64];
  extern __shared__ int pages_s[];     // [min(B, kPlanSmemSeqs)]
  // Runs as a programmatic dependent of the query-absorption kernel without waiting for it:
  // it starts only after every CTA of that kernel passed its own griddepcontrol.wait, so the
  // caller's inputs (context lengths, block table) are complete.  It waits for that kernel
  // at its end, so the decode kernel after it sees both.
  sm100::griddep_launch_dependents();
  // 1. validate and count pages, one warp per sequence (lanes check page ids in parallel);
  //    pages(b) is parked in seqs[b].nsplit
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  unsigned flags = 0;
  int my_pages = 0;
  for (int b = warp; b < B; b += nwarps) {
    const int L = ctx_len[b];
    int np = 0;
    if (L < 1 || L > max_ctx) {
      flags |= kCheckCtxLen;
    } else {
      np = (L + kPage - 1) / kPage;
      const int32_t* row = block_table + (size_t)b * bt_stride;
      bool bad = false;
      for (int i = lane; i < np; i += 32) {
        const int pg = row[i];
        bad |= (pg < 0 || pg >= num_pages);
      }
      if (__any_sync(0xffffffffu, bad)) { flags |= kCheckPageId; np = 0; }
    }
    if (lane == 0) {
      if (b < kPlanSmemSeqs) pages_s[b] = np; else ws.seqs[b].nsplit = np;
      my_pages += np;
    }
  }
  if (flags && lane == 0) atomicOr(check, flags);
  __syncthreads();   // seqs[].nsplit written by other warps is read below
  const int total_pages = block_sum(my_pages, red);
  const int max_pages = block_max(thread_max_pages(B, pages_s, ws), red);
  // Smallest page target whose split count fits in one wave of SM pairs: start from an
  // even share of the pages and grow it (binary search) until sum_b ceil(pages_b / target)
  // <= max(num_pairs, number of valid sequences).  With at least as many sequences as
  // pairs nothing is split.
  const int pairs = max(1, num_pairs);
  int lo = max(1, (total_pages + pairs - 1) / pairs), hi = max(lo, max_pages);
  const int valid_seqs = block_sum(count_valid(B, pages_s, ws), red);
  const int budget = max(pairs, valid_seqs);
  while (lo < hi) {
    const int mid = lo + (hi - lo) / 2;
    if (block_sum(count_units(B, pages_s, ws, mid), red) <= budget) hi = mid; else lo = mid + 1;
  }
  const int target = lo;

  // 2. split counts, prefix-summed chunk by chunk into first_unit
  int base = 0;
  for (int b0 = 0; b0 < B; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    int ns = 0;
    if (b < B) {
      const int np = pages_of(b, pages_s, ws);
      ns = np == 0 ? 0 : (forced > 0 ? min(forced, np) : (np + target - 1) / target);
    }
    int chunk_total = 0;
    const int off = block_exclusive_scan(ns, red, &chunk_total);
    if (b < B) {
      const int np = pages_of(b, pages_s, ws);
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
  sm100::griddep_wait();
}

}  // namespace

cudaError_t launch_plan(const Handle& h, const int32_t* ctx_len, int batch, int max_ctx,
                        const int32_t* block_table, int bt_stride, int num_pages, const Workspace& ws,
                        cudaStream_t st) {
  const size_t smem = sizeof(int) * (size_t)min(batch, kPlanSmemSeqs);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(int) * kPlanSmemSeqs));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), smem, st, ctx_len, batch, max_ctx, block_table,
                    bt_stride, num_pages, h.num_pairs, h.force_splits, ws, h.check_word);
}

}  // namespace mla
