// fd_api.cu -- the C ABI of libfd (include/fd.h): argument validation, the split-count
// planner, workspace layout, TMA tensor maps, kernel dispatch, and plans.
//
// Host code only (the kernels live in fd_partial_*.cu and fd_combine.cu).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "fd.h"
#include "fd_internal.h"

namespace {

thread_local char g_last_error[512] = "";
std::atomic<int> g_path{FD_PATH_AUTO};
std::atomic<int> g_merge{FD_MERGE_KERNEL};
std::atomic<int> g_schedule{FD_SCHEDULE_AUTO};
std::atomic<uint32_t> g_epoch{0x5eed0001u};   // per-call ticket epochs of the fused merge

// The path, merge mode and schedule one call runs with: its fd_options, with the
// process-wide settings in the fields marked FD_FROM_PROCESS (or all of them for NULL).
struct Settings {
  int path, merge, schedule;
};

bool valid_path(int v) {
  return v == FD_PATH_AUTO || v == FD_PATH_SIMT || v == FD_PATH_MMA || v == FD_PATH_TCGEN05;
}
bool valid_merge(int v) { return v == FD_MERGE_KERNEL || v == FD_MERGE_IN_KERNEL; }
bool valid_schedule(int v) {
  return v == FD_SCHEDULE_AUTO || v == FD_SCHEDULE_GRID || v == FD_SCHEDULE_PERSISTENT ||
         v == FD_SCHEDULE_HEAD_GROUPS || v == FD_SCHEDULE_TAIL_SHARING;
}

// False if a field holds neither FD_FROM_PROCESS nor one of its enum values.
bool resolve_settings(const fd_options* o, Settings* s) {
  s->path = (!o || o->path == FD_FROM_PROCESS) ? g_path.load() : o->path;
  s->merge = (!o || o->merge_mode == FD_FROM_PROCESS) ? g_merge.load() : o->merge_mode;
  s->schedule = (!o || o->schedule == FD_FROM_PROCESS) ? g_schedule.load() : o->schedule;
  return valid_path(s->path) && valid_merge(s->merge) && valid_schedule(s->schedule);
}

// Which partial-pass kernel runs, from the call's settings and sizes.  The persistent
// and head-group kernels write only partials, so neither runs under the single-launch
// merge.
struct Schedule {
  bool heads, persistent, tail_share;
};

// rows: query rows per (b, kv head) group (Q x G); groups above kMaxNarrowRows always
// run the wide grid kernel.  pairs: the call's (b, kv head) pairs, B x Hkv, S its split
// count and split_len its tokens per split (0: not known -- the name-only queries).
// f32 inputs on the tensor-core path run on the grid schedule only.
//
// Automatic head groups: always for small pages (16 and 32 tokens bf16, 32 FP8: their
// one-page boxes become one 16 KB box); for contiguous caches and larger pages once the
// batch holds kHeadsMinPairsPerSm (b, kv head) pairs per SM, with up to 8 query rows per
// kv head.
// There one CTA streams four kv heads of a row without a cross-warp merge, and the grid
// schedule's many short CTAs lose a start-up and an epilogue each.  Measured on GB300
// (bf16, d = 128, 32 heads over 8 kv heads, one split, a step over 256-512 MiB of KV):
// 128 rows of 512 tokens 50.0 -> 39.8 us, 256 x 512 92.1 -> 77.8, 512 x 256 101.6 ->
// 84.8, 1024 x 128 127.7 -> 90.0, 96 x 1024 64.0 -> 60.1; below the threshold the grid
// wins (64 x 1024: 42.0 against 49.6, whose 128 CTAs leave SMs idle).  FP8 caches
// (32-token tiles of 4 heads), same batches: 128 x 512 31.0 -> 22.8 us, 256 x 256 36.8
// -> 26.3, 1024 x 128 102.5 -> 62.7; with 32-token pages 32 x 2048 41.7 -> 25.5.
constexpr int64_t kHeadsMinPairsPerSm = 5;
// ... and with head groups, the persistent schedule for items of at most
// kPersistMaxItemTokens tokens (split_len), kPersistMinItemsPerSm of them per SM or
// more: each short CTA of the head-group grid pays ~2.5 us of start-up and pipeline fill
// for little streaming.  Measured on GB300 (Hq 32 over Hkv 8, one split), head groups ->
// persistent head groups: bf16 1024 rows x 128 tokens 90.6 -> 81.5 us, 512 x 256 84.8 ->
// 83.1; FP8 1024 x 128 62.7 -> 52.1, 512 x 256 52.1 -> 50.5; 16-token pages 1024 x 128
// 94.8 -> 82.5.  With fewer items a CTA's last one is a large share of its work (256 x
// 256, 3.4 items per SM: bf16 42.2 against 43.9, FP8 26.3 against 28.9), and from 512
// tokens per item the grid is ahead (bf16 256 x 512: 77.3 against 80.2).
constexpr int64_t kPersistMaxItemTokens = 256;
constexpr int64_t kPersistMinItemsPerSm = 6;
// Splits of fewer tokens than this, with 17 to 32 query rows per kv head, run the
// persistent wide kernel rather than the tcgen05 kernel (resolve_path).
constexpr int64_t kTcMinSplitTokens = 513;

Schedule choose_schedule(int sched, int path, bool kv8, bool f32, int64_t d, int64_t Hkv,
                         int32_t page_size, bool fused, int64_t rows, int64_t pairs,
                         int64_t S, int64_t split_len) {
  const bool narrow = rows <= fd::kMaxNarrowRows && !f32;
  // A head-group tile holds head_tok tokens of each head (one 16 KB box of 4 heads): a
  // page must hold at least that many.
  const int32_t head_tok = kv8 ? 32 : 16;
  const bool head_ok = path == FD_PATH_MMA && d == 128 &&
                       (page_size == 0 || page_size >= head_tok) &&
                       Hkv % fd::kHeadGroup == 0 && !fused && narrow;
  // Pages whose one-page boxes are small on the grid schedule: 16 and 32 tokens for bf16
  // (4 and 8 KB), 32 for FP8 (4 KB).  (FP8 with 64-token pages keeps the grid for small
  // batches: 32 rows of 2048 tokens 26.3 us on the grid, 51.2 with head groups.)
  const bool small_pages = page_size == head_tok || (!kv8 && page_size == 2 * head_tok);
  const int sms = rows <= 8 && pairs > 0 ? fd::sm_count() : 0;   // 0: no device
  const bool big_batch = sms > 0 && pairs >= kHeadsMinPairsPerSm * sms;
  Schedule sc;
  // The tiling: head groups where the automatic rule takes them (the persistent schedule
  // follows it too), or everywhere they apply when asked for.
  sc.heads = head_ok && (((sched == FD_SCHEDULE_AUTO || sched == FD_SCHEDULE_PERSISTENT) &&
                          (small_pages || big_batch)) ||
                         sched == FD_SCHEDULE_HEAD_GROUPS);
  const bool short_items = split_len > 0 && split_len <= kPersistMaxItemTokens &&
                           pairs / fd::kHeadGroup * S >= kPersistMinItemsPerSm * sms;
  // Wide groups of up to 32 rows (the mma.sync wide kernel, 8 rows a warp) have a
  // persistent form too, taken automatically for the short splits that resolve_path
  // gives them (fewer than kTcMinSplitTokens tokens).
  const bool wide32 = rows > fd::kMaxNarrowRows && rows <= 32 && !f32;
  const bool short_wide = wide32 && split_len > 0 && split_len < kTcMinSplitTokens;
  sc.persistent = path == FD_PATH_MMA && !fused && (narrow || wide32) &&
                  (sched == FD_SCHEDULE_PERSISTENT ||
                   (sched == FD_SCHEDULE_AUTO &&
                    ((sc.heads && big_batch && short_items) || short_wide)));
  // Tail sharing: the tcgen05 kernel, when asked for (measured slower than the plain
  // grid on GB300: the owners' claim round trips cost more than the tail it recovers).
  sc.tail_share = path == FD_PATH_TCGEN05 && sched == FD_SCHEDULE_TAIL_SHARING;
  return sc;
}

// Whether the tcgen05 kernel takes a call: bf16 q/K/V, d = 128, contiguous or pages of
// at least 16 tokens (its per-page products need N >= 16), up to kMaxRows rows.
bool tc_takes(int32_t q_dtype, bool kv8, int64_t d, int32_t page_size, int64_t rows) {
  return q_dtype == FD_BF16 && !kv8 && d == 128 && (page_size == 0 || page_size >= 16) &&
         rows >= 1 && rows <= fd::kMaxRows;
}

// Automatic choice: groups of kTcAutoMinRows rows or more go to the tcgen05 kernel where
// it applies; otherwise the mma.sync path for bf16 and for f32 groups of up to
// kMaxF32MmaRows rows, and the CUDA-core path for larger f32 groups.  Exception: groups
// of up to 32 rows whose splits hold fewer than kTcMinSplitTokens tokens (split_len; 0:
// not known) take the mma.sync wide kernel on the persistent schedule (choose_schedule).
// The tcgen05 kernel holds one CTA per SM and pays its start-up and epilogue (~7.5 us)
// once per split with nothing to overlap them; the persistent wide kernel streams its
// items back to back, two CTAs per SM.  Measured on GB300 (Hq 64 over Hkv 8, 4 query
// tokens = 32 rows, one split), tcgen05 -> persistent wide: 256 rows x 256 tokens 140.0
// -> 78.0 us, 512 x 128 238.8 -> 94.2, 128 x 512 91.0 -> 77.7, 64 x 512 49.1 -> 43.4;
// from 1024 tokens a split the tcgen05 kernel is ahead (64 x 1024: 69.8 against 74.2,
// 32 x 2048: 54.4 against 71.6), and with 64 rows at any length.

int resolve_path(int path, int32_t q_dtype, bool kv8, int64_t d, int32_t page_size,
                 int64_t rows, int64_t split_len) {
  if (path != FD_PATH_AUTO) return path;
  const bool short_splits = rows <= 32 && split_len > 0 && split_len < kTcMinSplitTokens;
  if (rows >= fd::kTcAutoMinRows && tc_takes(q_dtype, kv8, d, page_size, rows) && !short_splits)
    return FD_PATH_TCGEN05;
  return q_dtype == FD_BF16 || rows <= fd::kMaxF32MmaRows ? FD_PATH_MMA : FD_PATH_SIMT;
}

// The partial-pass kernel a call runs (fd_partial_kernel_name*); pairs = B x Hkv and S
// the split count, or 0 when not known (then a call of few pairs and several splits).
const char* kernel_name(const Settings& cfg, int32_t dtype, int32_t kv_dtype, int32_t d,
                        int32_t Hkv, int32_t page_size, int32_t rows, int32_t with_output,
                        int64_t pairs, int32_t S, int64_t split_len) {
  const bool kv8 = kv_dtype == FD_F8E4M3;
  if ((dtype != FD_BF16 && dtype != FD_F32) || (!kv8 && kv_dtype != dtype) ||
      (kv8 && dtype != FD_BF16) || d <= 0 || Hkv <= 0 || page_size < 0 || rows < 1 ||
      rows > fd::kMaxRows)
    return nullptr;
  const int path = resolve_path(cfg.path, dtype, kv8, d, page_size, rows, split_len);
  if ((path == FD_PATH_MMA && dtype == FD_F32 && rows > fd::kMaxF32MmaRows) ||
      (kv8 && path != FD_PATH_MMA))
    return nullptr;
  if (path == FD_PATH_TCGEN05)
    return tc_takes(dtype, kv8, d, page_size, rows) ? "fd_partial_tc_kernel" : nullptr;
  if (rows > fd::kMaxNarrowRows && (path != FD_PATH_MMA || (kv8 && rows > fd::kMaxFp8Rows)))
    return nullptr;
  if (path == FD_PATH_SIMT) return "fd_partial_simt_kernel";
  // One split with an output writes the output from the partial pass: no in-kernel merge.
  const bool fused = with_output && S != 1 && cfg.merge == FD_MERGE_IN_KERNEL;
  const Schedule sc = choose_schedule(cfg.schedule, path, kv8, dtype == FD_F32, d, Hkv,
                                      page_size, fused, rows, pairs, S, split_len);
  if (rows > fd::kMaxNarrowRows)
    return sc.persistent ? "fd_partial_wide_persist_kernel" : "fd_partial_wide_kernel";
  if (sc.heads) return sc.persistent ? "fd_partial_heads_persist_kernel" : "fd_partial_heads_kernel";
  if (sc.persistent) return "fd_partial_persist_kernel";
  return "fd_partial_mma_kernel";
}

fd_status fail(fd_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

constexpr size_t kAlign = 256;
// Header: device error flags (u32 at 0), the persistent schedule's item queue and
// done counter (u64 at kQueueOff, kDoneOff: plain fetch-add counters, zero between
// launches -- a fresh header is zero and the last CTA of each launch resets them).
constexpr size_t kHeaderBytes = 256;
constexpr size_t kQueueOff = 64, kDoneOff = 128;
constexpr int32_t kMaxSplits = 4096;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int64_t x) {
  int r = 0;
  while ((int64_t{1} << r) < x) ++r;
  return r;
}

int esize(int32_t dtype) { return dtype == FD_F8E4M3 ? 1 : (dtype == FD_BF16 ? 2 : 4); }


// Workspace regions for given sizes: header | LSE_i [B, Hq, S] |
// O_i [B, Hq, S, d] | ticket counters [B, Hkv] (64-bit) of the fused merge | claim words
// [B, Hkv, S] (16 bytes) of tail sharing; each region 256-byte aligned.  Neither the
// counters nor the claim words need particular initial contents (take_ticket and
// produce_tiles_shared in fd_pipeline.cuh), so one workspace serves calls of any sizes
// that fit it.
struct WsLayout {
  size_t lse_off, o_off, cnt_off, steal_off, total;
};

WsLayout ws_layout(int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t S) {
  WsLayout w;
  w.lse_off = kHeaderBytes;
  w.o_off = align_up(w.lse_off + (size_t)(B * Hq * S) * sizeof(float), kAlign);
  w.cnt_off = align_up(w.o_off + (size_t)(B * Hq * S * d) * sizeof(float), kAlign);
  w.steal_off = align_up(w.cnt_off + (size_t)(B * Hkv) * sizeof(unsigned long long), kAlign);
  w.total = align_up(w.steal_off + (size_t)(B * Hkv * S) * sizeof(fd::StealWord), kAlign);
  return w;
}

// ---- cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda) ----
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

// A KV cache viewed as 5-D for TMA: {elements of one 128-byte line, tokens (L_cap or
// page_size), 128-byte lines per row, kv heads, batch rows (or pages)}, 128-byte swizzle.
// The line dimension sits outside the row dimension (its stride, 128 B, is smaller than
// the row stride) so that a box of R rows lands in shared memory line-slice by
// line-slice: [line][row][128 B].
struct MapKey {
  const void* ptr;
  int32_t dtype;
  uint64_t dims[5];
  uint64_t strides[4];
  uint32_t box_rows, box_heads;
  bool operator==(const MapKey& o) const { return memcmp(this, &o, sizeof *this) == 0; }
};

struct MapCache {
  std::mutex mu;
  std::vector<std::pair<MapKey, CUtensorMap>> entries;   // most recent last
};

MapCache& map_cache() {
  static MapCache c;
  return c;
}

fd_status make_kv_map(const fd_tensor* t, uint32_t box_rows, uint32_t box_heads,
                      CUtensorMap* out) {
  const int es = esize(t->dtype);
  const int d = (int)t->shape[3];
  MapKey key;
  memset(&key, 0, sizeof key);
  key.ptr = t->data;
  key.dtype = t->dtype;
  key.dims[0] = (uint64_t)(128 / es);              // elements of one 128-byte line
  key.dims[1] = (uint64_t)t->shape[2];              // token rows (L_cap or page_size)
  key.dims[2] = (uint64_t)(d * es / 128);           // 128-byte lines per row
  key.dims[3] = (uint64_t)t->shape[1];              // kv heads
  key.dims[4] = (uint64_t)t->shape[0];              // batch rows or pages
  key.strides[0] = (uint64_t)t->stride[2] * es;     // next row
  key.strides[1] = 128;                             // next line of the same row
  key.strides[2] = (uint64_t)t->stride[1] * es;
  key.strides[3] = (uint64_t)t->stride[0] * es;
  key.box_rows = box_rows;
  key.box_heads = box_heads;
  MapCache& c = map_cache();
  {
    std::lock_guard<std::mutex> lock(c.mu);
    for (size_t i = 0; i < c.entries.size(); ++i) {
      if (c.entries[i].first == key) {
        *out = c.entries[i].second;
        return FD_OK;
      }
    }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(FD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  // One box = `box_rows` token rows, all lines, of `box_heads` consecutive kv heads: it
  // lands as [head][line][row][128 B], so the lines of one column slice of consecutive
  // rows are consecutive 128-byte lines.
  const cuuint32_t box[5] = {(cuuint32_t)key.dims[0], box_rows, (cuuint32_t)key.dims[2],
                             box_heads, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUtensorMap m;
  const CUtensorMapDataType ty = t->dtype == FD_BF16     ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : t->dtype == FD_F8E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = enc(&m, ty,
                   5, t->data, key.dims, key.strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    return fail(FD_ERR_INVALID_ARG, "cuTensorMapEncodeTiled rejected the KV cache view (CUresult %d)",
                (int)r);
  }
  std::lock_guard<std::mutex> lock(c.mu);
  if (c.entries.size() >= 32) c.entries.erase(c.entries.begin());
  c.entries.emplace_back(key, m);
  *out = m;
  return FD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int current_sm_count() { return fd::sm_count(); }

// Split count for num_splits = 0.  Single-token groups (up to kMaxNarrowRows query rows
// per kv head) take fd_num_splits_heuristic.  Wider groups run the tcgen05 or mma.sync
// wide kernel, bound by tile math, which do best with one CTA's worth of splits per SM
// (GQA 128K cache, 64 rows: 19 splits 93 us, 38 splits 111 us); never more splits than
// the single-token plan, so a workspace sized by fd_resolve_num_splits always suffices.
int32_t heuristic_splits(int32_t B, int32_t Q, int32_t Hq, int32_t Hkv, int32_t d,
                         int64_t L_cap) {
  const int sms = current_sm_count();
  const int32_t S = fd_num_splits_heuristic(B, Hq, Hkv, d, L_cap, sms);
  if (Hkv <= 0 || (int64_t)Q * (Hq / Hkv) <= fd::kMaxNarrowRows) return S;
  const int64_t units = (int64_t)B * Hkv;
  int64_t s = std::max<int64_t>(1, sms / units);
  s = std::min<int64_t>(s, std::max<int64_t>(1, (L_cap + 255) / 256));
  return (int32_t)std::min<int64_t>(S, s);
}

}  // namespace

namespace fd {
// Lets other translation units of the library report a failure through fd_last_error.
fd_status record_error(fd_status st, const char* message) { return fail(st, "%s", message); }

// SM count of the current device, queried once per device (0 if it cannot be read).
int sm_count() {
  constexpr int kDevices = 64;
  static std::atomic<int> cached[kDevices];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kDevices) {
    n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kDevices && n > 0) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}
}  // namespace fd

extern "C" {

const char* fd_version(void) { return "fd 0.1.0 (sm_103a)"; }

const char* fd_last_error(void) { return g_last_error; }

const char* fd_status_string(fd_status s) {
  switch (s) {
    case FD_OK: return "FD_OK";
    case FD_ERR_INVALID_ARG: return "FD_ERR_INVALID_ARG";
    case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED";
    case FD_ERR_WORKSPACE_TOO_SMALL: return "FD_ERR_WORKSPACE_TOO_SMALL";
    case FD_ERR_CUDA: return "FD_ERR_CUDA";
    case FD_ERR_DEVICE_FLAG: return "FD_ERR_DEVICE_FLAG";
  }
  return "FD_ERR_UNKNOWN";
}

fd_status fd_set_path(int32_t path) {
  if (!valid_path(path)) return fail(FD_ERR_INVALID_ARG, "unknown kernel path %d", path);
  g_path.store(path);
  return FD_OK;
}

int32_t fd_get_path(void) { return g_path.load(); }

fd_status fd_set_merge_mode(int32_t mode) {
  if (!valid_merge(mode)) return fail(FD_ERR_INVALID_ARG, "unknown merge mode %d", mode);
  g_merge.store(mode);
  return FD_OK;
}

int32_t fd_get_merge_mode(void) { return g_merge.load(); }

fd_status fd_set_schedule(int32_t schedule) {
  if (!valid_schedule(schedule)) return fail(FD_ERR_INVALID_ARG, "unknown schedule %d", schedule);
  g_schedule.store(schedule);
  return FD_OK;
}

int32_t fd_get_schedule(void) { return g_schedule.load(); }

const char* fd_partial_kernel_name(int32_t dtype, int32_t kv_dtype, int32_t d, int32_t Hkv,
                                   int32_t page_size, int32_t rows, int32_t with_output) {
  return fd_partial_kernel_name_ex(nullptr, dtype, kv_dtype, d, Hkv, page_size, rows,
                                   with_output);
}

const char* fd_partial_kernel_name_ex(const fd_options* options, int32_t dtype,
                                      int32_t kv_dtype, int32_t d, int32_t Hkv,
                                      int32_t page_size, int32_t rows, int32_t with_output) {
  Settings cfg;
  if (!resolve_settings(options, &cfg)) return nullptr;
  return kernel_name(cfg, dtype, kv_dtype, d, Hkv, page_size, rows, with_output, 0, 0, 0);
}

const char* fd_partial_kernel_name_for(const fd_options* options, int32_t dtype,
                                       int32_t kv_dtype, int32_t B, int32_t Q, int32_t Hq,
                                       int32_t Hkv, int32_t d, int32_t page_size, int64_t L_cap,
                                       int32_t num_splits, int32_t with_output) {
  Settings cfg;
  if (!resolve_settings(options, &cfg) || B <= 0 || Q <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 ||
      Hq % Hkv != 0 || L_cap <= 0 || num_splits < 0 || num_splits > kMaxSplits)
    return nullptr;
  const int64_t rows = (int64_t)Q * (Hq / Hkv);
  if (rows > fd::kMaxRows) return nullptr;
  const int32_t S = num_splits > 0 ? num_splits : heuristic_splits(B, Q, Hq, Hkv, d, L_cap);
  return kernel_name(cfg, dtype, kv_dtype, d, Hkv, page_size, (int32_t)rows, with_output,
                     (int64_t)B * Hkv, S, (L_cap + S - 1) / S);
}

size_t fd_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || num_splits <= 0 || num_splits > kMaxSplits)
    return 0;
  return ws_layout(B, Hq, Hkv, d, num_splits).total;
}

int32_t fd_resolve_num_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int64_t L_cap,
                              int32_t num_splits) {
  if (num_splits > 0) return num_splits;
  return fd_num_splits_heuristic(B, Hq, Hkv, d, L_cap, current_sm_count());
}

int32_t fd_resolve_num_splits_q(int32_t B, int32_t Q, int32_t Hq, int32_t Hkv, int32_t d,
                                int64_t L_cap, int32_t num_splits) {
  if (num_splits > 0) return num_splits;
  return heuristic_splits(B, Q, Hq, Hkv, d, L_cap);
}

fd_status fd_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return fail(FD_ERR_INVALID_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
  return FD_OK;
}

fd_status fd_read_device_error(void* workspace, void* stream, uint32_t* flags) {
  if (!workspace) return fail(FD_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t f = 0;
  cudaError_t e = cudaMemcpyAsync(&f, workspace, sizeof f, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && f != 0) e = cudaMemsetAsync(workspace, 0, sizeof f, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "reading device flags: %s", cudaGetErrorString(e));
  if (flags) *flags = f;
  if (f) return fail(FD_ERR_DEVICE_FLAG, "device error flags 0x%x", f);
  return FD_OK;
}

}  // extern "C"

namespace {

// Everything a call resolved on the host: kernel parameters, tensor maps and path.
struct Prepared {
  fd::Params p;
  CUtensorMap tk, tv;
  int path;
  int32_t dtype;
  bool fused;   // the last CTA of each group merges it (FD_MERGE_IN_KERNEL with an output)
};

// Validate a decode call and resolve it.  `out` may be NULL (partial pass only).
fd_status prepare(const fd_tensor* q, const fd_tensor* k_cache, const fd_tensor* v_cache,
                  const int32_t* seq_lens, const fd_tensor* block_table, int32_t page_size,
                  int32_t num_splits, const fd_tensor* out, float* lse_out, void* workspace,
                  size_t workspace_bytes, bool need_out, const Settings& cfg, Prepared* pr,
                  bool kv8 = false, const float* k_scale = nullptr,
                  const float* v_scale = nullptr) {
  // ---- presence and ranks
  if (!q || !k_cache || !v_cache || (need_out && !out))
    return fail(FD_ERR_INVALID_ARG, "q, k_cache, v_cache and out are required");
  if (!q->data || !k_cache->data || !v_cache->data || (out && !out->data))
    return fail(FD_ERR_INVALID_ARG, "a tensor has a NULL data pointer");
  if (!seq_lens) return fail(FD_ERR_INVALID_ARG, "seq_lens is NULL");
  if (!workspace) return fail(FD_ERR_INVALID_ARG, "workspace is NULL");
  if ((q->ndim != 3 && q->ndim != 4) || k_cache->ndim != 4 || v_cache->ndim != 4 ||
      (out && out->ndim != q->ndim))
    return fail(FD_ERR_INVALID_ARG,
                "ranks must be q 3 or 4, k/v 4, out as q (got %d, %d, %d, %d)", q->ndim,
                k_cache->ndim, v_cache->ndim, out ? out->ndim : q->ndim);
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_INVALID_ARG, "num_splits must be in [0, %d], got %d", kMaxSplits, num_splits);

  // q [B, Hq, d] (one query token per row) or [B, Q, Hq, d] (Q tokens, causal).
  const bool multi = q->ndim == 4;
  const int64_t B = q->shape[0], Q = multi ? q->shape[1] : 1;
  const int64_t Hq = q->shape[multi ? 2 : 1], d = q->shape[multi ? 3 : 2];
  if (Q <= 0) return fail(FD_ERR_INVALID_ARG, "empty query token dimension");
  const int64_t Hkv = k_cache->shape[1];
  if (B <= 0 || Hq <= 0 || d <= 0 || Hkv <= 0) return fail(FD_ERR_INVALID_ARG, "empty shape");
  for (int i = 0; i < 4; ++i) {
    if (k_cache->shape[i] != v_cache->shape[i])
      return fail(FD_ERR_INVALID_ARG, "k_cache and v_cache shapes differ in dim %d", i);
  }
  if (k_cache->shape[3] != d) return fail(FD_ERR_INVALID_ARG, "k/v head dim %lld != q head dim %lld",
                                          (long long)k_cache->shape[3], (long long)d);
  if (out) {
    for (int i = 0; i < q->ndim; ++i) {
      if (out->shape[i] != q->shape[i]) return fail(FD_ERR_INVALID_ARG, "out must have q's shape");
    }
  }
  if (Hq % Hkv != 0) return fail(FD_ERR_INVALID_ARG, "Hq (%lld) is not a multiple of Hkv (%lld)",
                                 (long long)Hq, (long long)Hkv);
  // ---- dtypes
  if (kv8) {
    if (k_cache->dtype != FD_F8E4M3 || v_cache->dtype != FD_F8E4M3 || q->dtype != FD_BF16)
      return fail(FD_ERR_INVALID_ARG, "the FP8 KV entry point takes bf16 q and fp8 e4m3 k/v");
    if (q->shape[q->ndim - 1] != 128)
      return fail(FD_ERR_UNSUPPORTED, "the FP8 KV cache needs head dim 128");
    if ((k_scale && ((uintptr_t)k_scale & 3)) || (v_scale && ((uintptr_t)v_scale & 3)))
      return fail(FD_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  } else {
    if (k_cache->dtype == FD_F8E4M3 || v_cache->dtype == FD_F8E4M3)
      return fail(FD_ERR_INVALID_ARG, "an FP8 KV cache goes through fd_decode_attention_fp8kv");
    if (k_cache->dtype != q->dtype || v_cache->dtype != q->dtype)
      return fail(FD_ERR_INVALID_ARG, "q, k_cache and v_cache must share one dtype");
  }
  if (q->dtype != FD_BF16 && q->dtype != FD_F32)
    return fail(FD_ERR_UNSUPPORTED, "q/k/v dtype must be bf16 or f32");
  if (out && out->dtype != FD_F32 && !(out->dtype == FD_BF16 && q->dtype == FD_BF16))
    return fail(FD_ERR_UNSUPPORTED, "out must be f32, or bf16 with bf16 inputs");
  const int64_t G = Hq / Hkv;
  if (d != 64 && d != 128) return fail(FD_ERR_UNSUPPORTED, "head dim %lld not in {64, 128}", (long long)d);
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16 && G != 32 && G != 64)
    return fail(FD_ERR_UNSUPPORTED, "group size %lld not in {1, 2, 4, 8, 16, 32, 64}", (long long)G);
  if (Q * G > fd::kMaxRows)
    return fail(FD_ERR_UNSUPPORTED, "query tokens x group size = %lld exceeds %d rows per kv head",
                (long long)(Q * G), fd::kMaxRows);
  const int es = esize(k_cache->dtype);              // KV element size (TMA, tiles)
  const int qes = esize(q->dtype);
  // ---- strides and alignment (TMA: 16-byte base and strides; rows contiguous)
  if (q->stride[q->ndim - 1] != 1 || k_cache->stride[3] != 1 || v_cache->stride[3] != 1 ||
      (out && out->stride[out->ndim - 1] != 1))
    return fail(FD_ERR_INVALID_ARG, "the last dimension of q, k, v and out must be contiguous");
  if (!aligned16(q->data) || !aligned16(k_cache->data) || !aligned16(v_cache->data))
    return fail(FD_ERR_INVALID_ARG, "q, k_cache and v_cache must be 16-byte aligned");
  for (int i = 0; i + 1 < q->ndim; ++i) {
    if ((q->stride[i] * qes) % 16) return fail(FD_ERR_INVALID_ARG, "q strides must be multiples of 16 bytes");
  }
  for (int i = 0; i < 3; ++i) {
    if ((k_cache->stride[i] * es) % 16 || (v_cache->stride[i] * es) % 16 || k_cache->stride[i] <= 0 ||
        v_cache->stride[i] <= 0)
      return fail(FD_ERR_INVALID_ARG, "k/v strides must be positive multiples of 16 bytes");
  }
  if (k_cache->stride[2] < d || v_cache->stride[2] < d)
    return fail(FD_ERR_INVALID_ARG, "k/v token rows overlap");
  // ---- contiguous or paged
  const bool paged = block_table != nullptr;
  int64_t L_cap = 0;
  int32_t max_pages = 0;
  int64_t bt_sb = 0;
  if (!paged) {
    if (page_size != 0) return fail(FD_ERR_INVALID_ARG, "page_size must be 0 without a block table");
    if (k_cache->shape[0] != B) return fail(FD_ERR_INVALID_ARG, "contiguous k_cache must be [B, Hkv, L_cap, d]");
    L_cap = k_cache->shape[2];
  } else {
    if (!block_table->data) return fail(FD_ERR_INVALID_ARG, "block_table has a NULL data pointer");
    if (block_table->ndim != 2 || block_table->dtype != FD_I32)
      return fail(FD_ERR_INVALID_ARG, "block_table must be int32 [B, max_pages]");
    if (block_table->shape[0] != B || block_table->shape[1] <= 0 || block_table->stride[1] != 1)
      return fail(FD_ERR_INVALID_ARG, "block_table must be [B, max_pages] with contiguous rows");
    if (!is_pow2(page_size) || page_size < 8 || page_size > 65536)
      return fail(FD_ERR_INVALID_ARG, "page_size must be a power of two in [8, 65536], got %d", page_size);
    if (k_cache->shape[2] != page_size)
      return fail(FD_ERR_INVALID_ARG, "paged k_cache must be [num_pages, Hkv, page_size, d]");
    max_pages = (int32_t)block_table->shape[1];
    bt_sb = block_table->stride[0];
    L_cap = (int64_t)max_pages * page_size;
  }
  if (L_cap <= 0 || L_cap >= (int64_t{1} << 31))
    return fail(FD_ERR_INVALID_ARG, "cache capacity must be in [1, 2^31), got %lld", (long long)L_cap);
  if (lse_out && ((uintptr_t)lse_out & 3))
    return fail(FD_ERR_INVALID_ARG, "lse_out must be 4-byte aligned");
  // ---- splits and workspace
  int32_t S = num_splits > 0 ? num_splits
                             : heuristic_splits((int32_t)B, (int32_t)Q, (int32_t)Hq,
                                                (int32_t)Hkv, (int32_t)d, L_cap);
  const WsLayout wl = ws_layout(B, Q * Hq, Hkv, d, S);   // partial rows: [B, Q, Hq]
  if (((uintptr_t)workspace & (kAlign - 1)) != 0)
    return fail(FD_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < wl.total)
    return fail(FD_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", wl.total, workspace_bytes);
  if ((int64_t)S * Hkv > 65535 * 65535LL || Hkv > 65535 || B > 65535)
    return fail(FD_ERR_UNSUPPORTED, "grid too large");

  // ---- path
  const int path = resolve_path(cfg.path, q->dtype, kv8, d, paged ? page_size : 0, Q * G,
                                (L_cap + S - 1) / S);
  if (path == FD_PATH_TCGEN05 && !tc_takes(q->dtype, kv8, d, paged ? page_size : 0, Q * G))
    return fail(FD_ERR_UNSUPPORTED,
                "the tcgen05 kernel takes bf16 q/K/V with d = 128, up to %d query rows per kv "
                "head and pages of at least 16 tokens",
                fd::kMaxRows);
  if (path == FD_PATH_MMA && q->dtype == FD_F32 && Q * G > fd::kMaxF32MmaRows)
    return fail(FD_ERR_UNSUPPORTED,
                "the tensor-core path takes f32 inputs for up to %d query rows per kv head",
                fd::kMaxF32MmaRows);
  if (kv8 && path != FD_PATH_MMA)
    return fail(FD_ERR_UNSUPPORTED, "the FP8 KV cache runs on the tensor-core path only");
  if (Q * G > fd::kMaxNarrowRows && path == FD_PATH_SIMT)
    return fail(FD_ERR_UNSUPPORTED,
                "more than %d query rows per kv head (%lld) run on the tensor-core paths only",
                fd::kMaxNarrowRows, (long long)(Q * G));
  if (kv8 && Q * G > fd::kMaxFp8Rows)
    return fail(FD_ERR_UNSUPPORTED,
                "an FP8 KV cache takes up to %d query rows per kv head, not %lld",
                fd::kMaxFp8Rows, (long long)(Q * G));

  // ---- schedule (fd_set_schedule or the call's options).  One split with an output:
  // the partial pass writes the output itself (Params::direct) and nothing merges.
  const bool direct = need_out && S == 1;
  const bool fused = need_out && !direct && cfg.merge == FD_MERGE_IN_KERNEL;
  const Schedule sc = choose_schedule(cfg.schedule, path, kv8, q->dtype == FD_F32, d, Hkv,
                                     paged ? page_size : 0, fused, Q * G, B * Hkv, S,
                                     (L_cap + S - 1) / S);
  const bool heads = sc.heads, persistent = sc.persistent;

  // ---- tensor maps (box height: one tile, or one page when pages are shorter; with head
  // groups a quarter tile -- 16 bf16 or 32 FP8 rows -- of kHeadGroup heads)
  const int TT = fd::tile_tokens((int)d, es);
  const uint32_t box_rows = heads ? (uint32_t)(TT / fd::kHeadGroup)     // 16 bf16, 32 FP8
                                 : (uint32_t)(paged && page_size < TT ? page_size : TT);
  const uint32_t box_heads = heads ? (uint32_t)fd::kHeadGroup : 1u;
  fd_status st = make_kv_map(k_cache, box_rows, box_heads, &pr->tk);
  if (st != FD_OK) return st;
  st = make_kv_map(v_cache, box_rows, box_heads, &pr->tv);
  if (st != FD_OK) return st;

  fd::Params& p = pr->p;
  memset(&p, 0, sizeof p);
  p.B = (int32_t)B;
  p.Hq = (int32_t)Hq;
  p.Hkv = (int32_t)Hkv;
  p.d = (int32_t)d;
  p.G = (int32_t)G;
  p.L_cap = L_cap;
  p.S = S;
  p.split_len = (L_cap + S - 1) / S;
  p.q = q->data;
  p.Q = (int32_t)Q;
  p.n_rows = (int32_t)(Q * G);
  p.q_sb = q->stride[0];
  p.q_sj = multi ? q->stride[1] : 0;
  p.q_sh = q->stride[multi ? 2 : 1];
  p.seq_lens = seq_lens;
  p.block_table = paged ? static_cast<const int32_t*>(block_table->data) : nullptr;
  p.bt_sb = bt_sb;
  p.page_size = paged ? page_size : 0;
  p.log2_page = paged ? ilog2(page_size) : 0;
  p.log2_box = ilog2(box_rows);
  p.max_pages = max_pages;
  p.num_pages = paged ? k_cache->shape[0] : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.flags = reinterpret_cast<uint32_t*>(ws);
  p.counters = reinterpret_cast<unsigned long long*>(ws + wl.cnt_off);
  p.item_queue = reinterpret_cast<unsigned long long*>(ws + kQueueOff);
  p.ctas_done = reinterpret_cast<unsigned long long*>(ws + kDoneOff);
  uint32_t epoch = g_epoch.fetch_add(1u);
  if (epoch == 0u) epoch = g_epoch.fetch_add(1u);   // 0 would match a zeroed word
  p.epoch = epoch;
  p.lse_part = reinterpret_cast<float*>(ws + wl.lse_off);
  p.o_part = reinterpret_cast<float*>(ws + wl.o_off);
  p.out = out ? out->data : nullptr;
  p.out_sb = out ? out->stride[0] : 0;
  p.out_sj = out && multi ? out->stride[1] : 0;
  p.out_sh = out ? out->stride[multi ? 2 : 1] : 0;
  p.out_bf16 = out && out->dtype == FD_BF16 ? 1 : 0;
  p.lse_out = lse_out;
  p.direct = 0;                     // set below, once the kernel is known
  p.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)d));
  p.kv_fp8 = kv8 ? 1 : 0;
  p.in_f32 = q->dtype == FD_F32 ? 1 : 0;
  p.k_scale = kv8 ? k_scale : nullptr;
  p.v_scale = kv8 ? v_scale : nullptr;

  p.persistent = persistent ? 1 : 0;
  p.head_group = heads ? fd::kHeadGroup : 0;
  p.steal = reinterpret_cast<fd::StealWord*>(ws + wl.steal_off);
  p.tail_share = sc.tail_share ? 1 : 0;
  // The tcgen05 kernel gives a tile that straddles two splits to the lower one, so no
  // tile is read twice (split_len need not be a whole number of tiles: 128K tokens over
  // 19 splits, one CTA per SM, read 0.9% more bytes otherwise).
  p.tile_owned = path == FD_PATH_TCGEN05 ? 1 : 0;
  p.direct = direct && (path != FD_PATH_MMA || fd::mma_writes_direct(p)) ? 1 : 0;

  pr->path = path;
  pr->dtype = q->dtype;
  pr->fused = fused;
  return FD_OK;
}

fd_status launch_partial(const Prepared& pr, cudaStream_t s) {
  cudaError_t e = pr.path == FD_PATH_MMA      ? fd::launch_partial_mma(pr.p, pr.tk, pr.tv, s)
                  : pr.path == FD_PATH_TCGEN05 ? fd::launch_partial_tc(pr.p, pr.tk, pr.tv, s)
                                               : fd::launch_partial_simt(pr.p, pr.tk, pr.tv, pr.dtype, s);
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "partial-pass launch: %s", cudaGetErrorString(e));
  return FD_OK;
}

fd_status launch_merge(const fd::Params& p, cudaStream_t s) {
  cudaError_t e = fd::launch_combine(p, s, /*pdl=*/true);
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
  return FD_OK;
}

// Which cache format an entry point takes: bf16 / f32 only, FP8 E4M3 only, or whichever
// k_cache's dtype says (fd_decode_attention_ex).
enum class CacheKind { kPlain, kFp8, kByDtype };

// One decode call: resolve the settings, validate and plan, then launch the partial pass
// and, with an output, the merge (its own kernel, or inside the partial pass for
// FD_MERGE_IN_KERNEL).  need_out false: the partial pass only.
fd_status run_decode(CacheKind kind, const fd_tensor* q, const fd_tensor* k_cache,
                     const fd_tensor* v_cache, const float* k_scale, const float* v_scale,
                     const int32_t* seq_lens, const fd_tensor* block_table, int32_t page_size,
                     int32_t num_splits, fd_tensor* out, float* lse_out, void* workspace,
                     size_t workspace_bytes, void* stream, const fd_options* options,
                     bool need_out, int32_t selftest_stall = 0) {
  Settings cfg;
  if (!resolve_settings(options, &cfg))
    return fail(FD_ERR_INVALID_ARG, "fd_options holds an unknown path, merge mode or schedule");
  bool kv8 = kind == CacheKind::kFp8;
  if (kind == CacheKind::kByDtype) {
    kv8 = k_cache != nullptr && k_cache->dtype == FD_F8E4M3;
    if (!kv8 && (k_scale || v_scale))
      return fail(FD_ERR_INVALID_ARG, "k_scale / v_scale belong to an FP8 E4M3 cache only");
  }
  Prepared pr;
  fd_status st = prepare(q, k_cache, v_cache, seq_lens, block_table, page_size, num_splits,
                         need_out ? out : nullptr, need_out ? lse_out : nullptr, workspace,
                         workspace_bytes, need_out, cfg, &pr, kv8, k_scale, v_scale);
  if (st != FD_OK) return st;
  pr.p.selftest_stall = selftest_stall;
  const cudaStream_t s = (cudaStream_t)stream;
  if (need_out && pr.fused) return launch_partial(pr, s);   // one launch merges in-kernel
  pr.p.counters = nullptr;          // the merge, if any, is a separate kernel
  st = launch_partial(pr, s);
  if (st != FD_OK || !need_out || pr.p.direct) return st;   // direct: out is written
  return launch_merge(pr.p, s);
}

}  // namespace

extern "C" {

fd_status fd_decode_attention(const fd_tensor* q, const fd_tensor* k_cache,
                              const fd_tensor* v_cache, const int32_t* seq_lens,
                              const fd_tensor* block_table, int32_t page_size,
                              int32_t num_splits, fd_tensor* out, float* lse_out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kPlain, q, k_cache, v_cache, nullptr, nullptr, seq_lens,
                    block_table, page_size, num_splits, out, lse_out, workspace,
                    workspace_bytes, stream, nullptr, true);
}

fd_status fd_decode_partial(const fd_tensor* q, const fd_tensor* k_cache,
                            const fd_tensor* v_cache, const int32_t* seq_lens,
                            const fd_tensor* block_table, int32_t page_size, int32_t num_splits,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kPlain, q, k_cache, v_cache, nullptr, nullptr, seq_lens,
                    block_table, page_size, num_splits, nullptr, nullptr, workspace,
                    workspace_bytes, stream, nullptr, false);
}

fd_status fd_decode_attention_fp8kv(const fd_tensor* q, const fd_tensor* k_cache,
                                   const fd_tensor* v_cache, const float* k_scale,
                                   const float* v_scale, const int32_t* seq_lens,
                                   const fd_tensor* block_table, int32_t page_size,
                                   int32_t num_splits, fd_tensor* out, float* lse_out,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  return run_decode(CacheKind::kFp8, q, k_cache, v_cache, k_scale, v_scale, seq_lens,
                    block_table, page_size, num_splits, out, lse_out, workspace,
                    workspace_bytes, stream, nullptr, true);
}

fd_status fd_decode_partial_fp8kv(const fd_tensor* q, const fd_tensor* k_cache,
                                 const fd_tensor* v_cache, const float* k_scale,
                                 const float* v_scale, const int32_t* seq_lens,
                                 const fd_tensor* block_table, int32_t page_size,
                                 int32_t num_splits, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  return run_decode(CacheKind::kFp8, q, k_cache, v_cache, k_scale, v_scale, seq_lens,
                    block_table, page_size, num_splits, nullptr, nullptr, workspace,
                    workspace_bytes, stream, nullptr, false);
}

fd_status fd_decode_attention_ex(const fd_tensor* q, const fd_tensor* k_cache,
                                 const fd_tensor* v_cache, const float* k_scale,
                                 const float* v_scale, const int32_t* seq_lens,
                                 const fd_tensor* block_table, int32_t page_size,
                                 int32_t num_splits, fd_tensor* out, float* lse_out,
                                 void* workspace, size_t workspace_bytes, void* stream,
                                 const fd_options* options) {
  return run_decode(CacheKind::kByDtype, q, k_cache, v_cache, k_scale, v_scale, seq_lens,
                    block_table, page_size, num_splits, out, lse_out, workspace,
                    workspace_bytes, stream, options, out != nullptr);
}

fd_status fd_selftest_stalled_decode(const fd_tensor* q, const fd_tensor* k_cache,
                                     const fd_tensor* v_cache, const float* k_scale,
                                     const float* v_scale, const int32_t* seq_lens,
                                     const fd_tensor* block_table, int32_t page_size,
                                     int32_t num_splits, fd_tensor* out, float* lse_out,
                                     void* workspace, size_t workspace_bytes, void* stream,
                                     const fd_options* options, int32_t stall_tile) {
  if (stall_tile < 0) return fail(FD_ERR_INVALID_ARG, "stall_tile must be >= 0");
  return run_decode(CacheKind::kByDtype, q, k_cache, v_cache, k_scale, v_scale, seq_lens,
                    block_table, page_size, num_splits, out, lse_out, workspace,
                    workspace_bytes, stream, options, out != nullptr, stall_tile + 1);
}

fd_status fd_workspace_partials(void* workspace, int32_t B, int32_t Hq, int32_t d,
                                int32_t num_splits, float** lse_part, float** o_part) {
  if (!workspace || B <= 0 || Hq <= 0 || d <= 0 || num_splits <= 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_INVALID_ARG, "invalid workspace or sizes");
  const WsLayout wl = ws_layout(B, Hq, 1, d, num_splits);   // partial offsets need no Hkv
  if (lse_part) *lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + wl.lse_off);
  if (o_part) *o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + wl.o_off);
  return FD_OK;
}

fd_status fd_merge_partials(int32_t B, int32_t Hq, int32_t d, int32_t num_splits,
                            const float* lse_part, const float* o_part, fd_tensor* out,
                            float* lse_out, void* stream) {
  if (!lse_part || !o_part || !out || !out->data)
    return fail(FD_ERR_INVALID_ARG, "lse_part, o_part and out are required");
  if (B <= 0 || Hq <= 0 || num_splits <= 0 || num_splits > kMaxSplits)
    return fail(FD_ERR_INVALID_ARG, "invalid sizes");
  if (d != 64 && d != 128) return fail(FD_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", d);
  if (out->ndim != 3 || out->shape[0] != B || out->shape[1] != Hq || out->shape[2] != d ||
      out->stride[2] != 1)
    return fail(FD_ERR_INVALID_ARG, "out must be [B, Hq, d] with a contiguous last dim");
  if (out->dtype != FD_F32 && out->dtype != FD_BF16)
    return fail(FD_ERR_UNSUPPORTED, "out must be f32 or bf16");
  if (((uintptr_t)o_part & 15) || ((uintptr_t)lse_part & 3))
    return fail(FD_ERR_INVALID_ARG, "o_part must be 16-byte and lse_part 4-byte aligned");
  if (lse_out && ((uintptr_t)lse_out & 3)) return fail(FD_ERR_INVALID_ARG, "lse_out misaligned");
  fd::Params p;
  memset(&p, 0, sizeof p);
  p.B = B;
  p.Hq = Hq;
  p.d = d;
  p.S = num_splits;
  p.lse_part = const_cast<float*>(lse_part);
  p.o_part = const_cast<float*>(o_part);
  p.out = out->data;
  p.out_sb = out->stride[0];
  p.out_sh = out->stride[1];
  p.out_bf16 = out->dtype == FD_BF16 ? 1 : 0;
  p.lse_out = lse_out;
  p.Q = 1;
  p.G = 1;
  p.n_rows = 1;
  return launch_merge(p, (cudaStream_t)stream);
}


// ------------------------------------------------------------------------ plans
struct fd_plan {
  int32_t B, Q, Hq, Hkv, d;   // Q query tokens per row (1: single-token decode)
  int64_t L_cap;
  int32_t S;
  int device;
  void* ws;
  size_t ws_bytes;
  cudaEvent_t done;   // recorded after each decode's merge pass
  fd_options opts;    // fd_plan_set_options (every field FD_FROM_PROCESS by default)
};

static fd_status plan_alloc(fd_plan* p, int32_t S) {
  const int64_t rows = (int64_t)p->Q * p->Hq;
  const size_t bytes = rows <= INT32_MAX ? fd_workspace_size(p->B, (int32_t)rows, p->Hkv, p->d, S)
                                         : 0;
  if (bytes == 0) return fail(FD_ERR_INVALID_ARG, "invalid plan sizes");
  void* ws = nullptr;
  cudaError_t e = cudaMalloc(&ws, bytes);
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  e = cudaMemset(ws, 0, bytes);
  if (e != cudaSuccess) {
    cudaFree(ws);
    return fail(FD_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
  }
  cudaEvent_t ev;
  e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaFree(ws);
    return fail(FD_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(e));
  }
  p->ws = ws;
  p->ws_bytes = bytes;
  p->done = ev;
  p->S = S;
  return FD_OK;
}

fd_status fd_plan_create(fd_plan** plan, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                         int64_t L_cap, int32_t num_splits) {
  return fd_plan_create_q(plan, B, 1, Hq, Hkv, d, L_cap, num_splits);
}

fd_status fd_plan_create_q(fd_plan** plan, int32_t B, int32_t Q, int32_t Hq, int32_t Hkv,
                           int32_t d, int64_t L_cap, int32_t num_splits) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  *plan = nullptr;
  if (B <= 0 || Q <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || L_cap <= 0 || num_splits < 0 ||
      num_splits > kMaxSplits || Hq % Hkv != 0)
    return fail(FD_ERR_INVALID_ARG, "invalid plan sizes");
  fd_plan* p = new fd_plan();
  p->opts.path = p->opts.merge_mode = p->opts.schedule = FD_FROM_PROCESS;
  p->Q = Q;
  p->B = B;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->d = d;
  p->L_cap = L_cap;
  cudaGetDevice(&p->device);
  const int32_t S = num_splits > 0 ? num_splits : heuristic_splits(B, Q, Hq, Hkv, d, L_cap);
  fd_status st = plan_alloc(p, S);
  if (st != FD_OK) {
    delete p;
    return st;
  }
  *plan = p;
  return FD_OK;
}

int32_t fd_plan_num_splits(const fd_plan* plan) { return plan ? plan->S : 0; }
size_t fd_plan_workspace_bytes(const fd_plan* plan) { return plan ? plan->ws_bytes : 0; }
void* fd_plan_workspace(const fd_plan* plan) { return plan ? plan->ws : nullptr; }

// Whether q and the cache have the plan's sizes: q [B, Hq, d] for a plan of one query
// token per row, [B, Q, Hq, d] for Q > 1 (a 4-D q with Q = 1 is accepted too).
static bool plan_fits(const fd_plan* plan, const fd_tensor* q, const fd_tensor* k_cache) {
  if (!q || !k_cache || k_cache->ndim != 4 || k_cache->shape[1] != plan->Hkv) return false;
  if (q->ndim == 3)
    return plan->Q == 1 && q->shape[0] == plan->B && q->shape[1] == plan->Hq &&
           q->shape[2] == plan->d;
  return q->ndim == 4 && q->shape[0] == plan->B && q->shape[1] == plan->Q &&
         q->shape[2] == plan->Hq && q->shape[3] == plan->d;
}

static fd_status plan_run(fd_plan* plan, CacheKind kind, const fd_tensor* q,
                          const fd_tensor* k_cache, const fd_tensor* v_cache,
                          const float* k_scale, const float* v_scale, const int32_t* seq_lens,
                          const fd_tensor* block_table, int32_t page_size, fd_tensor* out,
                          float* lse_out, void* stream) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  if (!plan_fits(plan, q, k_cache)) return fail(FD_ERR_INVALID_ARG, "tensor sizes differ from the plan's");
  fd_status st = run_decode(kind, q, k_cache, v_cache, k_scale, v_scale, seq_lens, block_table,
                            page_size, plan->S, out, lse_out, plan->ws, plan->ws_bytes, stream,
                            &plan->opts, true);
  if (st != FD_OK) return st;
  cudaError_t e = cudaEventRecord(plan->done, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
  return FD_OK;
}

fd_status fd_plan_decode(fd_plan* plan, const fd_tensor* q, const fd_tensor* k_cache,
                         const fd_tensor* v_cache, const int32_t* seq_lens,
                         const fd_tensor* block_table, int32_t page_size, fd_tensor* out,
                         float* lse_out, void* stream) {
  return plan_run(plan, CacheKind::kPlain, q, k_cache, v_cache, nullptr, nullptr, seq_lens,
                  block_table, page_size, out, lse_out, stream);
}

fd_status fd_plan_decode_ex(fd_plan* plan, const fd_tensor* q, const fd_tensor* k_cache,
                            const fd_tensor* v_cache, const float* k_scale, const float* v_scale,
                            const int32_t* seq_lens, const fd_tensor* block_table,
                            int32_t page_size, fd_tensor* out, float* lse_out, void* stream) {
  if (!out) return fail(FD_ERR_INVALID_ARG, "out is required");
  return plan_run(plan, CacheKind::kByDtype, q, k_cache, v_cache, k_scale, v_scale, seq_lens,
                  block_table, page_size, out, lse_out, stream);
}

fd_status fd_plan_set_options(fd_plan* plan, const fd_options* options) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  fd_options o;
  o.path = o.merge_mode = o.schedule = FD_FROM_PROCESS;
  if (options) o = *options;
  Settings cfg;
  if (!resolve_settings(&o, &cfg))
    return fail(FD_ERR_INVALID_ARG, "fd_options holds an unknown path, merge mode or schedule");
  plan->opts = o;
  return FD_OK;
}

fd_status fd_plan_resize(fd_plan* plan, int32_t num_splits) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  if (num_splits < 0 || num_splits > kMaxSplits) return fail(FD_ERR_INVALID_ARG, "bad num_splits");
  const int32_t S = num_splits > 0 ? num_splits
                                   : heuristic_splits(plan->B, plan->Q, plan->Hq, plan->Hkv,
                                                      plan->d, plan->L_cap);
  if (S == plan->S) return FD_OK;
  // The old workspace may still be read by an in-flight merge: wait for it first.
  cudaError_t e = cudaEventSynchronize(plan->done);
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "cudaEventSynchronize: %s", cudaGetErrorString(e));
  void* old_ws = plan->ws;
  cudaEvent_t old_ev = plan->done;
  fd_status st = plan_alloc(plan, S);
  if (st != FD_OK) return st;   // plan unchanged (old buffers kept)
  cudaFree(old_ws);
  cudaEventDestroy(old_ev);
  return FD_OK;
}

void fd_plan_destroy(fd_plan* plan) {
  if (!plan) return;
  if (plan->done) {
    cudaEventSynchronize(plan->done);
    cudaEventDestroy(plan->done);
  }
  if (plan->ws) cudaFree(plan->ws);
  delete plan;
}

}  // extern "C"
