// fd_noalloc.cu -- fd_decode_attention_noalloc: decode attention that allocates nothing.
//
// Some callers cannot allocate device memory at the moment they run a decode step:
// a plugin whose host framework owns all device memory and forbids allocation while
// it enqueues work, a serving loop with a fixed memory budget decided at start-up, or
// any code path where a cudaMalloc would implicitly synchronise the device and stall
// other streams.  fd_decode_attention already allocates nothing, but it asks the caller
// for a workspace.  This entry point takes no workspace at all: the split partials go
// to a scratch array that is part of the library itself, a file-scope __device__
// array of kScratchBytes that every GPU that loads the library keeps until the process
// exits.  The caller still passes its inputs and outputs.
//
// Limits and sharing:
//   - A call needs fd_workspace_size(B, Q * Hq, Hkv, d, S) bytes of scratch, Q being the
//     query tokens per row (1 for q [B, Hq, d]) and S the split count the call resolves
//     (fd_resolve_num_splits_q); a call that needs more than kScratchBytes is rejected
//     with FD_ERR_UNSUPPORTED and nothing is launched.
//   - Every call on a device uses the same array, and the array keeps whatever the last
//     call left in it.  Two calls that can run on the GPU at the same time (different
//     streams without an ordering between them) race on the array and give wrong
//     results; order them on one stream or with events.
//   - The first call on each device does a one-time set-up with that device current:
//     it looks up the array's device address (cudaGetSymbolAddress), zero-fills the
//     array (cudaMemset, not an allocation) and waits for the whole device to finish
//     (cudaDeviceSynchronize).  cudaMemset of device memory returns before the fill is
//     done and is ordered only against the legacy default stream, so without that wait
//     a caller stream created non-blocking could run this call's kernels while the fill
//     still clears the scratch under them.  Make that first call before any stream
//     capture on the device.
//   - Device-side input flags (out-of-range lengths or page ids) are still acted on as
//     fd_decode_attention documents, but this entry point has no way to report them.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "fd.h"
#include "fd_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t{8} << 20;   // 8 MiB per device
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code the name g_scratch is only a host-side stand-in,
// never a device address: host code must use the address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device; set up once per device.
fd_status scratch_on_current_device(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fd::record_error(FD_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fd::record_error(FD_ERR_UNSUPPORTED, "device ordinal beyond the no-alloc table");
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) {
      return fd::record_error(FD_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                            : "no device address for scratch");
    }
    e = cudaMemset(p, 0, kScratchBytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();   // the fill is done before any launch
    if (e != cudaSuccess) return fd::record_error(FD_ERR_CUDA, cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return FD_OK;
}

// FD_ERR_UNSUPPORTED for a call that does not fit the scratch (need 0: size not known).
fd_status refuse_size(size_t need) {
  char msg[240];
  if (need > 0)
    snprintf(msg, sizeof msg,
             "this call needs %zu bytes of scratch but the built-in scratch holds %zu; "
             "use fd_decode_attention with a caller workspace (or fewer splits)",
             need, kScratchBytes);
  else
    snprintf(msg, sizeof msg,
             "this call needs more than the %zu bytes of the built-in scratch; "
             "use fd_decode_attention with a caller workspace (or fewer splits)",
             kScratchBytes);
  return fd::record_error(FD_ERR_UNSUPPORTED, msg);
}

}  // namespace

extern "C" fd_status fd_decode_attention_noalloc(const fd_tensor* q, const fd_tensor* k_cache,
                                                 const fd_tensor* v_cache,
                                                 const int32_t* seq_lens,
                                                 const fd_tensor* block_table, int32_t page_size,
                                                 int32_t num_splits, fd_tensor* out,
                                                 float* lse_out, void* stream) {
  // Size the request when the descriptors are readable: q [B, Hq, d] or [B, Q, Hq, d],
  // with the split count the call itself resolves.  Sizes that fd_workspace_size does
  // not accept (it returns 0) are left to fd_decode_attention's checks, which report
  // them the usual way.
  if (q && k_cache && (q->ndim == 3 || q->ndim == 4) && k_cache->ndim == 4 &&
      num_splits >= 0) {
    const bool multi = q->ndim == 4;
    const int64_t B = q->shape[0], Q = multi ? q->shape[1] : 1;
    const int64_t Hq = q->shape[multi ? 2 : 1], d = q->shape[multi ? 3 : 2];
    const int64_t Hkv = k_cache->shape[1];
    const int64_t L_cap = block_table ? (block_table->ndim == 2 ? block_table->shape[1] : 0) *
                                            (int64_t)page_size
                                      : k_cache->shape[2];
    const int64_t rows = B * Q * Hq;
    if (B > 0 && Q > 0 && Hq > 0 && Hkv > 0 && d > 0 && rows <= INT32_MAX && Q <= INT32_MAX &&
        B <= INT32_MAX && Hkv <= INT32_MAX && d <= INT32_MAX && L_cap > 0) {
      const int32_t S = fd_resolve_num_splits_q((int32_t)B, (int32_t)Q, (int32_t)Hq,
                                                (int32_t)Hkv, (int32_t)d, L_cap, num_splits);
      const size_t need = fd_workspace_size((int32_t)B, (int32_t)(Q * Hq), (int32_t)Hkv,
                                            (int32_t)d, S);
      if (need > kScratchBytes) return refuse_size(need);
    }
  }
  void* scratch = nullptr;
  fd_status st = scratch_on_current_device(&scratch);
  if (st != FD_OK) return st;
  st = fd_decode_attention(q, k_cache, v_cache, seq_lens, block_table, page_size, num_splits,
                           out, lse_out, scratch, kScratchBytes, stream);
  // Any size the check above could not read still ends here, with this entry point's code.
  if (st == FD_ERR_WORKSPACE_TOO_SMALL) return refuse_size(0);
  return st;
}
