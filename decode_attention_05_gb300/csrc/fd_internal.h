// fd_internal.h -- parameters shared by the host planner (fd_api.cu) and the kernels.
//
// Not part of the public ABI (that is include/fd.h).
#pragma once

#include <cuda.h>            // CUtensorMap (type only; the driver entry point is looked up)
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "fd.h"

namespace fd {

// Device error flag set when a bounded wait gives up (a kernel then writes empty
// partials for its split and returns; the host sees it via fd_read_device_error).
constexpr uint32_t kDevFlagTimeout = FD_DEVFLAG_TIMEOUT;

// Bytes of one K (or V) tile in shared memory; the tile height in tokens is
// kTileBytes / (d * element size): 64 tokens for bf16 d=128.
constexpr int kTileBytes = 16384;
// kv heads per CTA (and per TMA box) in the head-group tiling; one per consumer warp
constexpr int kHeadGroup = 4;

// Claim word of one work item (b, kv head, split) for tail sharing, in the workspace:
// claim = back << 32 | front, the item's tiles [front, back) that nobody has claimed yet;
// epoch = the call that opened it (its owner writes the claim, then the epoch).
struct StealWord {
  unsigned long long claim;
  uint32_t epoch;
  uint32_t pad;
};

// Everything one decode call needs on the device, resolved by the host planner.
struct Params {
  // sizes
  int32_t B, Hq, Hkv, d, G;
  int64_t L_cap;          // tokens of capacity per row
  int32_t S;              // number of splits
  int64_t split_len;      // ceil(L_cap / S)
  // query [B, Q, Hq, d] (Q = 1: single-token decode)
  const void* q;
  int64_t q_sb, q_sj, q_sh;   // strides (elements) of batch, query token and head
  int32_t Q;                  // query tokens per row; query j sees keys t < L_b - Q + 1 + j
  int32_t n_rows;             // query rows per (b, kv head) = Q * G
  // lengths and paging
  const int32_t* seq_lens;
  const int32_t* block_table;   // nullptr -> contiguous
  int64_t bt_sb;                // batch stride of the block table (elements)
  int32_t page_size;            // tokens per page (paged), else 0
  int32_t log2_page;            // log2(page_size)
  int32_t log2_box;             // log2(rows of one TMA box): the tile, or a page if shorter
  int32_t max_pages;            // block table width
  int64_t num_pages;            // pages in the pool
  // workspace
  uint32_t* flags;        // device error flags (workspace header)
  unsigned long long* counters;   // [B, Hkv] (epoch << 32 | arrivals) per (b, kv head) for
                                  // the fused merge, or nullptr: the partial pass then
                                  // leaves the merge to a separate kernel
  uint32_t epoch;                 // this call's ticket epoch (never 0)
  // Persistent schedule: work items (split, kv head, row) handed out by a queue word and
  // a finished-CTA word in the workspace header (zero between launches, 64-bit)
  int32_t persistent;
  // Head-group tiles (kHeadGroup): a CTA serves kHeadGroup kv heads of a split and a
  // tile is 16 tokens of one page x kHeadGroup heads, one TMA box; 0 = one head per CTA
  int32_t head_group;
  unsigned long long* item_queue;
  unsigned long long* ctas_done;
  // Tail sharing: claim words [B, Hkv, S] of the items (see fd_pipeline.cuh), and
  // whether this launch shares (0: every CTA streams exactly its own split)
  StealWord* steal;
  int32_t tail_share;
  // 1: split i covers its range with both ends rounded up to whole tiles (split_range in
  // fd_pipeline.cuh): no tile is loaded by two CTAs (the tcgen05 kernel)
  int32_t tile_owned;
  // Failure-path self-test only (fd_selftest_stalled_decode; 0 otherwise): n > 0 makes the
  // producer of CTA (0, 0, 0) stop before its tile n - 1 and publish nothing more, as if
  // those copies never arrived, so the CTA's bounded waits run out
  int32_t selftest_stall;
  float* lse_part;        // [B, Q, Hq, S]     natural-log LSE_i, -inf for an empty split
  float* o_part;          // [B, Q, Hq, S, d]  normalised partial output O_i
  // outputs
  void* out;                // [B, Q, Hq, d]
  int64_t out_sb, out_sj, out_sh;
  int32_t out_bf16;       // 1: bf16 out, 0: f32 out
  float* lse_out;         // [B, Q, Hq] or nullptr
  // 1: a single split whose result is the output: the partial pass writes out and
  // lse_out itself and no merge runs (put_* in fd_pipeline.cuh); 0: it writes partials
  int32_t direct;
  // CTAs of the grid resident at once (set by a launcher whose CTAs prefetch the first
  // tiles of the CTA `wave` places later once they have issued their own, which then
  // finds them in L2 when it starts; 0: no such prefetch)
  int32_t wave;
  float scale_log2;       // log2(e) / sqrt(d): scores are kept in base-2 units inside kernels
  // FP8 KV cache (E4M3 codes): per-kv-head dequantisation scales [Hkv] (nullptr = 1)
  int32_t kv_fp8;
  int32_t in_f32;         // 1: q, K and V are f32 (tensor-core path: 3xTF32 products)
  const float* k_scale;
  const float* v_scale;
};

// Launchers (each returns the launch's cudaError_t).
// tcgen05 kernel (fd_partial_tc.cu): bf16 q/K/V, d = 128, 1..64 query rows per kv head,
// contiguous caches or pages of at least 16 tokens, grid schedule.
bool partial_tc_supported(const Params& p);
cudaError_t launch_partial_tc(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              cudaStream_t stream);
cudaError_t launch_partial_simt(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                int dtype, cudaStream_t stream);
// Whether the mma.sync kernel launch_partial_mma picks for p writes a single split's
// result as the output when p.direct is set (otherwise the host runs the merge).
bool mma_writes_direct(const Params& p);
cudaError_t launch_partial_mma(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream);
cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool pdl);

// Launch a partial-pass kernel with programmatic dependent launch: its CTAs may be
// scheduled while the previous kernel in the stream finishes; the kernel waits
// (griddepcontrol.wait) before its first global memory access.
template <class Kernel>
cudaError_t launch_partial_kernel(Kernel kernel, dim3 grid, int threads, size_t smem,
                                  cudaStream_t stream, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tk, tv, p);
}

// Record `message` as the calling thread's fd_last_error() and return `st`.
fd_status record_error(fd_status st, const char* message);

// SM count of the current device, queried once per device (0 if it cannot be read).
int sm_count();

// The opt-in dynamic shared-memory size is a per-kernel, per-device attribute: each
// launcher keeps one of these (a function-local static per kernel instantiation) and
// sets the attribute the first time it launches on a device, not on every call.
struct SmemOptIn {
  std::atomic<uint64_t> done{0};   // bit i: set on device i (devices 0..63)
  template <class Kernel>
  cudaError_t apply(Kernel kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// Query rows per (b, kv head) group padded to the kernels' template size: a power of two
// up to kMaxRows (groups above kMaxNarrowRows run the wide tensor-core kernel only).
constexpr int kMaxNarrowRows = 16;
constexpr int kMaxRows = 64;
// FP8 KV caches take up to kMaxFp8Rows query rows per kv head (the wide kernel with 8
// rows a warp above kMaxNarrowRows).
constexpr int kMaxFp8Rows = 32;
// The automatic path sends groups of at least this many rows to the tcgen05 kernel
// (where it applies).  GQA 128K cache, one CTA's worth of splits per SM: 32 rows 91 us
// (tcgen05) vs 132 us (mma.sync wide kernel), 64 rows 93 us vs 228 us; up to 16 rows the
// mma.sync kernels stay at the HBM rate (79-82 us).
constexpr int kTcAutoMinRows = 17;
// f32 inputs run on the tensor cores (3xTF32) for groups of up to this many rows.
constexpr int kMaxF32MmaRows = 8;
inline int rows_template(int n) {
  int r = 1;
  while (r < n) r <<= 1;
  return n >= 1 && r <= kMaxRows ? r : 0;
}

// Tile height (tokens) used by the kernels for a dtype and head dim.
inline int tile_tokens(int d, int esz) { return kTileBytes / (d * esz); }

}  // namespace fd
