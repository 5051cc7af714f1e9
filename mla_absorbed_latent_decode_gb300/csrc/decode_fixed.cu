// decode_fixed.cu -- mla_decode_fixed_scratch: the decode step with its scratch in one
// array that the library owns, so the call needs no workspace from the caller.
//
// Why it exists: mla_decode asks the caller for a workspace buffer.  Some callers have no
// way to provide one at the point of the call: a plain C host loop that links only this
// library and must not call cudaMalloc per step (cudaMalloc/cudaFree synchronise the
// device and can stall the stream that is being fed), or an engine whose memory pool is
// fully handed out to the KV cache.  For those, the scratch here is a file-scope device
// array of fixed size, created with the library's module on each device; nothing is
// allocated at call time, by this code or by any library it calls.
//
// Contract:
//   - the array holds kFixedScratchBytes (32 MiB); a call whose workspace (as
//     mla_decode_workspace_size reports it for the same batch) is larger is rejected
//     with MLA_ERR_WORKSPACE before anything is enqueued;
//   - every call writes each part of the scratch before reading it (plan counters, units,
//     absorbed queries, partials), so the array never has to start at zero;
//   - all calls on one device share the array, across handles and streams: two calls in
//     flight at the same time overwrite each other's scratch.  Callers order them (one
//     stream, or events between streams);
//   - the first call in a CUDA context looks up the array's device address
//     (cudaGetSymbolAddress), which may load the module in that context; make that first
//     call before any stream capture begins.  The address is cached together with the
//     context it belongs to (a device reset, or another context made current, gives a new
//     context and so a new lookup, which must also happen outside stream capture).  Later
//     calls in the same context only read the cached pointer.
#include <cuda.h>

#include <mutex>
#include <cstdio>

#include "internal.cuh"

namespace mla {
namespace {

constexpr size_t kFixedScratchBytes = size_t(MLA_FIXED_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

// One cached lookup per device: the context it was made in and the array's address there.
struct ScratchEntry {
  CUcontext ctx;
  void* ptr;
};
std::mutex g_lookup_mutex;
ScratchEntry g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (the library does not link
// libcuda directly).
cudaError_t current_context(CUcontext* ctx) {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return cudaErrorNotSupported;
    fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  return fn(ctx) == CUDA_SUCCESS && *ctx ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the array on `device` (which the caller has made current), looked up
// again whenever the current context is not the one the cached address was taken in.
cudaError_t scratch_on(int device, void** ptr) {
  std::lock_guard<std::mutex> lock(g_lookup_mutex);
  CUcontext ctx = nullptr;
  cudaError_t e = cudaFree(nullptr);      // make sure the runtime's context exists and is current
  if (e != cudaSuccess) return e;
  if ((e = current_context(&ctx)) != cudaSuccess) return e;
  ScratchEntry& ent = g_scratch[device];
  if (!ent.ptr || ent.ctx != ctx) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_fixed_scratch)) != cudaSuccess) return e;
    ent.ctx = ctx;
    ent.ptr = p;
  }
  *ptr = ent.ptr;
  return cudaSuccess;
}

mla_status_t report(mla_status_t s, const char* fmt, int a, long long b, long long c) {
  char buf[256];
  snprintf(buf, sizeof(buf), fmt, a, b, c);
  return set_last_error(s, buf);
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_decode_fixed_scratch(mla_handle_t hh, const void* q, const int32_t* ctx_len,
                                                 int32_t batch, int32_t max_ctx, const int32_t* block_table,
                                                 int32_t bt_stride, const void* cache, int32_t num_pages,
                                                 void* out, mla_stream_t stream) {
  mla::clear_last_error();
  const mla::Handle* h = reinterpret_cast<const mla::Handle*>(hh);
  if (!h) return mla::set_last_error(MLA_ERR_INVALID_ARG, "mla_decode_fixed_scratch: handle is NULL");
  size_t need = 0;
  mla_status_t s = mla_decode_workspace_size(hh, batch, max_ctx, &need);
  if (s != MLA_OK) return s;
  if (need > mla::kFixedScratchBytes)
    return mla::report(MLA_ERR_WORKSPACE,
                       "mla_decode_fixed_scratch: batch = %d needs %lld bytes of scratch, more than the "
                       "library's fixed %lld bytes; use mla_decode with a caller workspace",
                       batch, (long long)need, (long long)mla::kFixedScratchBytes);
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess)
    return mla::set_last_error(MLA_ERR_CUDA, "mla_decode_fixed_scratch: cudaGetDevice failed");
  if (cur != h->device || cur < 0 || cur >= mla::kMaxDevices)
    return mla::report(MLA_ERR_INVALID_ARG,
                       "mla_decode_fixed_scratch: device %d is current, the handle was created on device "
                       "%lld (at most %lld devices)",
                       cur, (long long)h->device, (long long)mla::kMaxDevices);
  void* scratch = nullptr;
  if ((e = mla::scratch_on(cur, &scratch)) != cudaSuccess) {
    char buf[256];
    snprintf(buf, sizeof(buf), "mla_decode_fixed_scratch: cudaGetSymbolAddress: %s (%s)", cudaGetErrorName(e),
             cudaGetErrorString(e));
    return mla::set_last_error(MLA_ERR_CUDA, buf);
  }
  return mla_decode(hh, q, ctx_len, batch, max_ctx, block_table, bt_stride, cache, num_pages, scratch,
                    mla::kFixedScratchBytes, out, stream);
}
