// fd_pipeline.cuh -- the memory side of the split-KV partial pass: which tokens a CTA
// owns, and a TMA producer warp that streams K and V tiles of those tokens from HBM
// into a ring of shared-memory stages guarded by mbarriers.
//
// Grid: blockIdx.x = split i, blockIdx.y = kv head g, blockIdx.z = batch row b.  The
// CTA serves all G = Hq / Hkv query heads of kv head g, so each KV byte of the split is
// read from HBM exactly once per step ("AI Infra: math and infra optimisation in large
// models", section 2.6, "Flash-Decoding Split-K": the KV cache is cut along the
// sequence and the pieces go to different SMs).
//
// Split i of row b covers logical tokens [i * split_len, min((i + 1) * split_len, L_b));
// it is empty when it starts at or past L_b.  Tiles are TT tokens long and aligned to
// multiples of TT in the logical token space, so a split that starts or ends mid-tile
// loads that boundary tile and masks the tokens outside its range.
//
// Paged caches: logical token t is slot t % ps of page block_table[b][t / ps]; the page
// ids are read in the table's order ("2kiu.com/news/6053916", section "the split count
// is a cost account": logical order must not be replaced by physical page numbers).
#pragma once

#include "fd_device.cuh"

namespace fd {

struct SplitInfo {
  int b, g, split;
  int64_t L;            // the row's length (clamped to [0, L_cap])
  int64_t lo, hi;       // valid logical tokens of this split: [lo, hi)
  int64_t T0;           // start of the first tile (a multiple of TT)
  int n_tiles;
  int64_t used_pages;   // pages of row b that hold tokens < L_b (paged)
};

// Logical tokens [lo, hi) that split `split` of a row of length L covers in this
// launch: [i split_len, (i + 1) split_len) clipped to L -- or, with p.tile_owned, the same
// with both ends rounded up to whole TT-token tiles, so that every tile belongs to exactly
// one split and is loaded once (the keys of a tile that straddles a boundary go to the
// lower split; every key still enters exactly one partial, so the merge is unchanged).
template <int TT>
__device__ __forceinline__ void split_range(const Params& p, int split, int64_t L, int64_t& lo,
                                            int64_t& hi) {
  lo = (int64_t)split * p.split_len;
  hi = lo + p.split_len;
  if (p.tile_owned) {
    lo = (lo + TT - 1) / TT * TT;
    hi = (hi + TT - 1) / TT * TT;
  }
  hi = min(hi, L);
}

// Resolve this CTA's split; clamps and flags an out-of-range sequence length.
template <int TT>
__device__ __forceinline__ SplitInfo split_info(const Params& p) {
  SplitInfo si;
  si.split = blockIdx.x;
  si.g = blockIdx.y;
  si.b = blockIdx.z;
  int64_t L = p.seq_lens[si.b];
  if (L < 0 || L > p.L_cap) {
    if (threadIdx.x == 0) atomicOr(p.flags, FD_DEVFLAG_SEQ_LEN);
    L = L < 0 ? 0 : p.L_cap;
  }
  si.L = L;
  split_range<TT>(p, si.split, L, si.lo, si.hi);
  si.T0 = (si.lo / TT) * TT;
  si.n_tiles = si.lo < si.hi ? (int)((si.hi - si.T0 + TT - 1) / TT) : 0;
  si.used_pages = p.page_size > 0 ? (L + p.page_size - 1) >> p.log2_page : 0;
  return si;
}

// L2 prefetch of the first `count` tiles of this CTA's split, contiguous caches (grid
// blockIdx = (split, kv head or head group, batch row); `head` = the first kv head of
// the CTA's TMA boxes), issued BEFORE griddepcontrol.wait.  Where a split starts depends only on the launch's
// sizes (split_len), and a prefetch is only a hint: L2 is the point of coherence, so the
// loads after the wait still see whatever the previous kernel of the stream wrote.  The
// inputs that kernel may still be changing -- the row's length, and for a paged cache
// the block-table entries -- are read relaxed and only steer the prefetch: a split past
// the length prefetches nothing, and a page id outside [0, num_pages) is skipped.  A CTA
// that becomes resident while the previous decode step finishes (programmatic dependent
// launch) thus has its first tiles on the way to L2 before it may read them, and the
// tail of the previous step's bandwidth is not left idle.
__device__ __forceinline__ int32_t ld_relaxed_s32(const int32_t* a) {
  int32_t v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
template <int TT>
__device__ __forceinline__ void prefetch_tiles_of(const Params& p, const CUtensorMap* tk,
                                                  const CUtensorMap* tv, int count, int split,
                                                  int head, int b) {
  if (p.block_table != nullptr) return;       // paged caches: prefetch_first_pages
  const int64_t L = min(max((int64_t)ld_relaxed_s32(p.seq_lens + b), (int64_t)0), p.L_cap);
  int64_t lo, hi;
  split_range<TT>(p, split, L, lo, hi);
  const int64_t T0 = lo / TT * TT;
#pragma unroll 1
  for (int k = 0; k < count; ++k) {
    const int64_t t0 = T0 + (int64_t)k * TT;
    if (t0 >= hi) break;
    tma_prefetch_5d(tk, 0, (int)t0, 0, head, b);
    tma_prefetch_5d(tv, 0, (int)t0, 0, head, b);
  }
}
template <int TT>
__device__ __forceinline__ void prefetch_first_tiles(const Params& p, const CUtensorMap* tk,
                                                     const CUtensorMap* tv, int count, int head) {
  prefetch_tiles_of<TT>(p, tk, tv, count, (int)blockIdx.x, head, (int)blockIdx.z);
}

// The next wave (contiguous caches, grid (S, Hkv / HPC, B) of HPC kv heads per CTA):
// once a CTA has issued its own tiles, the first `count` tiles of the CTA p.wave launch
// places later -- the one that will take a freed slot about when this one ends -- go to
// L2, so that CTA's first loads hit L2 instead of waiting on HBM.  A hint only: the
// lengths are read relaxed and a wrong guess costs bandwidth, not correctness.
template <int TT, int HPC = 1>
__device__ __forceinline__ void prefetch_next_wave(const Params& p, const CUtensorMap* tk,
                                                   const CUtensorMap* tv, int count) {
  if (p.wave <= 0 || p.block_table != nullptr) return;
  const int64_t linear = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
  const int64_t target = linear + p.wave;
  if (target >= (int64_t)gridDim.x * gridDim.y * gridDim.z) return;
  const int split = (int)(target % gridDim.x);
  const int64_t rest = target / gridDim.x;
  prefetch_tiles_of<TT>(p, tk, tv, count, split, (int)(rest % gridDim.y) * HPC,
                        (int)(rest / gridDim.y));
}

// The same for a paged cache whose boxes are TT rows of one page (TT <= page_size; the
// caller checks):
// the page ids of the split's first tiles come from the block table, read relaxed; a
// page id outside [0, num_pages) is skipped.  Kept apart from prefetch_first_tiles, and
// left out of the kernels with 16 query rows per kv head: there its extra registers
// spill (measured 7% slower).
template <int TT>
__device__ __forceinline__ void prefetch_first_pages(const Params& p, const CUtensorMap* tk,
                                                     const CUtensorMap* tv, int count, int head) {
  const int b = (int)blockIdx.z;
  const int64_t L = min(max((int64_t)ld_relaxed_s32(p.seq_lens + b), (int64_t)0), p.L_cap);
  const int64_t lo = (int64_t)blockIdx.x * p.split_len;
  const int64_t hi = min(lo + p.split_len, L);
  const int64_t T0 = lo / TT * TT;
#pragma unroll 1
  for (int k = 0; k < count; ++k) {
    const int64_t t0 = T0 + (int64_t)k * TT;
    if (t0 >= hi) break;
    const int64_t pi = t0 >> p.log2_page;
    const int32_t id = ld_relaxed_s32(p.block_table + (int64_t)b * p.bt_sb + pi);
    if (id < 0 || (int64_t)id >= p.num_pages) continue;
    const int slot = (int)(t0 & (p.page_size - 1));
    tma_prefetch_5d(tk, 0, slot, 0, head, id);
    tma_prefetch_5d(tv, 0, slot, 0, head, id);
  }
}

// Query rows of a (b, kv head) group: row rho (0 .. Q * G - 1) is query token j = rho / G
// of head h = rho mod G.  Its flat index over [B, Q, Hq] (partials, lse_out), its query
// vector, and its causal key bound: the Q query tokens are the last Q positions of the
// row, so token j sees keys t < L_b - Q + 1 + j ("AI Infra: math and infra optimisation
// in large models", section 2.5: a token sees itself and the past; with Q = 1 this is
// the plain length mask t < L_b).
__device__ __forceinline__ int64_t flat_row(const Params& p, int b, int g, int rho) {
  const int j = rho / p.G, h = rho - j * p.G;
  return ((int64_t)b * p.Q + j) * p.Hq + (int64_t)g * p.G + h;
}
__device__ __forceinline__ int64_t q_offset(const Params& p, int b, int g, int rho) {
  const int j = rho / p.G, h = rho - j * p.G;
  return (int64_t)b * p.q_sb + (int64_t)j * p.q_sj + ((int64_t)g * p.G + h) * p.q_sh;
}
__device__ __forceinline__ int64_t key_bound(const Params& p, int64_t L, int rho) {
  return L - p.Q + 1 + rho / p.G;
}

// ---------------------------------------------------------------- split results
//
// A split writes its normalised output O_i and LSE_i to the workspace partials -- except
// when the call has one split and asks for the output (Params::direct).  The merge is
// then the identity: the one weight is 2^(LSE_1 - LSE_1) = 1, so out = O_1 and
// lse_out = LSE_1, and the partial pass writes out and lse_out itself (no O_i round trip
// through memory, no merge launch).  A row that the split leaves without a key gets
// out = 0 and lse_out = -inf there, as the merge would give it.
__device__ __forceinline__ int64_t out_elem(const Params& p, int b, int g, int rho) {
  const int j = rho / p.G, h = rho - j * p.G;
  return (int64_t)b * p.out_sb + (int64_t)j * p.out_sj + ((int64_t)g * p.G + h) * p.out_sh;
}
__device__ __forceinline__ void put_out(const Params& p, int64_t e, float v) {
  if (p.out_bf16) {
    reinterpret_cast<__nv_bfloat16*>(p.out)[e] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<float*>(p.out)[e] = v;
  }
}
// LSE_i of row rho of group (b, g).  DIRECT = false: a kernel that never runs with
// Params::direct (its partials-only form, for instantiations at their register cap).
template <bool DIRECT = true>
__device__ __forceinline__ void put_lse(const Params& p, int b, int g, int rho, int split, float v) {
  const int64_t row = flat_row(p, b, g, rho);
  if (!DIRECT || !p.direct) {
    p.lse_part[row * p.S + split] = v;
  } else if (p.lse_out != nullptr) {
    p.lse_out[row] = v;
  }
}
// Direct output: dims j .. j + 3 of out for row rho of group (b, g).
__device__ __forceinline__ void put_out4(const Params& p, int b, int g, int rho, int j, float4 o) {
  const int64_t e = out_elem(p, b, g, rho) + j;
  put_out(p, e, o.x);
  put_out(p, e + 1, o.y);
  put_out(p, e + 2, o.z);
  put_out(p, e + 3, o.w);
}
// Row rho of group (b, g) has no key in the split (or its split was abandoned): LSE_i =
// -inf and no O_i -- weight 0 in the merge; with direct output, out = 0 and -inf.
template <bool DIRECT = true>
__device__ __forceinline__ void put_empty_row(const Params& p, int b, int g, int rho, int split) {
  put_lse<DIRECT>(p, b, g, rho, split, kNegInf);
  if (DIRECT && p.direct) {
    const int64_t e = out_elem(p, b, g, rho);
    for (int j = 0; j < p.d; ++j) put_out(p, e + j, 0.f);
  }
}

// Take a ticket on an epoch-tagged counter word (the fused merge's per-group
// arrivals).  A counter word holds
// (epoch << 32 | arrivals).  Each call brings a fresh epoch, so the first arrival of a
// call restarts the count whatever the word held before (a workspace reused with other
// sizes, stale data); the last arrival also puts the word back to 0, so a launch that
// is replayed as is starts from a clean count too.  Lock-free: a failed compare-and-swap
// means another CTA's succeeded.  Returns the arrival number (1 .. S), or 0 if the
// bounded loop gave up (flagged).
__device__ __forceinline__ unsigned take_ticket(const Params& p, unsigned long long* c) {
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(c);
  for (int it = 0; it < (1 << 20); ++it) {
    const unsigned long long want =
        ((unsigned)(cur >> 32) == p.epoch) ? cur + 1ull
                                           : (((unsigned long long)p.epoch << 32) | 1ull);
    const unsigned long long prev = atomicCAS(c, cur, want);
    if (prev == cur) return (unsigned)(want & 0xffffffffull);
    cur = prev;
  }
  atomicOr(p.flags, kDevFlagTimeout);
  return 0u;
}

// Shared-memory control block of the pipeline.
template <int STAGES>
struct PipeCtl {
  uint64_t full[STAGES];    // TMA bytes landed (count 1 + transaction bytes)
  uint64_t empty[STAGES];   // consumers released the stage (count = consumer warps)
  uint32_t bad[STAGES];     // bit j: page slot j of the tile had an invalid page id
  // Tile descriptors published by produce_tiles_shared with each stage: the tile's first
  // logical token, the valid range [lo, hi) of the split it belongs to, and done = 1 for
  // a stage that carries no tile but the end of the sequence (n_total tiles in all).
  int64_t t0[STAGES], lo[STAGES], hi[STAGES];
  int32_t done[STAGES];
  int32_t n_total;
  int32_t abort;            // a bounded wait gave up
  int32_t last;             // this CTA drew its group's last ticket (fused merge)
};

// Failure-path self-test (Params::selftest_stall): whether the producer of this CTA stops
// before its ring slot n.  Never true outside fd_selftest_stalled_decode.
__device__ __forceinline__ bool selftest_stops(const Params& p, int n) {
  return p.selftest_stall > 0 && n == p.selftest_stall - 1 && blockIdx.x == 0 &&
         blockIdx.y == 0 && blockIdx.z == 0;
}

// ---------------------------------------------------------------- persistent schedule
//
// Work item x (0 .. S * Hkv * B - 1) is split S - 1 - x / (Hkv * B) of kv head
// x mod Hkv of row (x / Hkv) mod B: the highest split indices, which only the longest
// rows have, go first, and the many short or empty items fill in at the end.
struct TileMeta {
  int32_t b, g, split, flags;   // flags: kFirst | kLast | kDone
  int64_t t0, lo, hi, L;        // tile start, the item's valid range, the row's length
  uint32_t bad;
};
constexpr int32_t kMetaFirst = 1, kMetaLast = 2, kMetaDone = 4;

template <int STAGES>
struct PersistCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t epi[3];              // consumer warps meet here around an item's epilogue
  TileMeta meta[STAGES];
  float mm[4 * 16], ml[4 * 16]; // per-warp running max and exp-sum of the item's rows
  int32_t abort;
};

// Item x of the persistent schedule: its split, (first) kv head and row.  HG kv heads per
// item: 1, or kHeadGroup with head-group tiles (then g is a multiple of kHeadGroup).
struct Item {
  int split, g, b;
};
template <int HG>
__device__ __forceinline__ Item item_of(const Params& p, int64_t x) {
  const int64_t groups = p.Hkv / HG;
  const int64_t per_split = groups * p.B;
  const int64_t r = x % per_split;
  return Item{p.S - 1 - (int)(x / per_split), (int)(r % groups) * HG, (int)(r / groups)};
}

// The first `count` tiles of the CTA's first item (item blockIdx.x: the first item of
// every CTA is its own, the queue hands out the rest) prefetched into L2 before the
// kernel waits for the previous kernel of the stream: the row length and page ids are
// read relaxed -- a hint only, the producer reads them again after the wait.  Pages
// shorter than a tile are not prefetched.
template <int TT, int HG>
__device__ __forceinline__ void prefetch_first_item(const Params& p, const CUtensorMap* tk,
                                                    const CUtensorMap* tv, int count) {
  const Item it = item_of<HG>(p, (int64_t)blockIdx.x);
  const int64_t L = min(max((int64_t)ld_relaxed_s32(p.seq_lens + it.b), (int64_t)0), p.L_cap);
  const int64_t lo = (int64_t)it.split * p.split_len;
  const int64_t hi = min(lo + p.split_len, L);
  const int64_t T0 = lo / TT * TT;
  const bool paged = p.block_table != nullptr;
  if (paged && p.page_size < TT) return;
#pragma unroll 1
  for (int k = 0; k < count; ++k) {
    const int64_t t0 = T0 + (int64_t)k * TT;
    if (t0 >= hi) break;
    if (!paged) {
      tma_prefetch_5d(tk, 0, (int)t0, 0, it.g, it.b);
      tma_prefetch_5d(tv, 0, (int)t0, 0, it.g, it.b);
    } else {
      const int32_t id = ld_relaxed_s32(p.block_table + (int64_t)it.b * p.bt_sb + (t0 >> p.log2_page));
      if (id < 0 || (int64_t)id >= p.num_pages) continue;
      const int slot = (int)(t0 & (p.page_size - 1));
      tma_prefetch_5d(tk, 0, slot, 0, it.g, id);
      tma_prefetch_5d(tv, 0, slot, 0, it.g, id);
    }
  }
}

// Producer warp of the persistent kernel: takes items from the queue and streams their
// tiles into the ring without a break between items; publishes a kDone stage at the
// end.  Empty items get their LSE_i = -inf written here and never reach the consumers.
// HG kv heads per item (1, or kHeadGroup with head-group tiles: TT is then one head's
// tokens of a tile, and one box of TT rows x HG heads fills the stage).
template <int TT, int STAGES, bool DIRECT, int HG = 1>
__device__ __forceinline__ void produce_items(const Params& p, const CUtensorMap* tk,
                                              const CUtensorMap* tv, uint8_t* stages,
                                              PersistCtl<STAGES>* ctl, int lane) {
  const uint64_t pol = policy_evict_first();
  const bool paged = p.block_table != nullptr;
  const int ps = p.page_size;
  const int pages_per_tile = paged ? (ps >= TT ? 1 : TT / ps) : 1;
  const int box_rows = paged ? (ps >= TT ? TT : ps) : TT;
  const uint32_t box_bytes = (uint32_t)(kTileBytes / TT) * box_rows;
  const int64_t n_items = (int64_t)p.S * (p.Hkv / HG) * p.B;
  int n = 0;                        // tiles published so far (ring position)
  bool aborted = false;

  // Acquire ring slot n (lane 0 waits, the warp agrees).
  auto acquire = [&](int slot_n) -> bool {
    if (slot_n < STAGES) return true;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->empty[slot_n % STAGES]), ((slot_n / STAGES) - 1) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) {
      ctl->abort = 1;
      atomicOr(p.flags, kDevFlagTimeout);
    }
    return ok != 0;
  };

  // The CTA's first item is item blockIdx.x (the grid never has more CTAs than items);
  // the others come from a plain fetch-and-add on the queue word, offset by the grid
  // size (the word is zero at launch: a fresh workspace header is zero and the last CTA
  // of every launch puts it back).  The next item's ticket is taken when an item starts,
  // so its latency hides behind the item.
  unsigned long long ticket = blockIdx.x;
  while (!aborted) {
    if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int32_t*>(&ctl->abort), 0)) break;
    const int64_t item = (int64_t)__shfl_sync(0xffffffffu, ticket, 0);
    if (item >= n_items) break;
    if (lane == 0) ticket = gridDim.x + atomicAdd(p.item_queue, 1ull);
    const Item it = item_of<HG>(p, item);
    const int split = it.split, g = it.g, b = it.b;
    int64_t L = p.seq_lens[b];
    if (L < 0 || L > p.L_cap) {
      if (lane == 0) atomicOr(p.flags, FD_DEVFLAG_SEQ_LEN);
      L = L < 0 ? 0 : p.L_cap;
    }
    const int64_t lo = (int64_t)split * p.split_len;
    const int64_t hi = min(lo + p.split_len, L);
    if (lo >= hi) {                 // empty split: weight 0 in the merge
      for (int i = lane; i < HG * p.n_rows; i += 32)
        put_empty_row<DIRECT>(p, b, g + i / p.n_rows, i % p.n_rows, split);
      continue;
    }
    const int64_t T0 = lo / TT * TT;
    const int n_tiles = (int)((hi - T0 + TT - 1) / TT);
    const int64_t used_pages = paged ? (L + ps - 1) >> p.log2_page : 0;
    int64_t cache_base = -64;
    int32_t cache = -2;
    for (int t = 0; t < n_tiles; ++t, ++n) {
      if (selftest_stops(p, n) || !acquire(n)) {
        aborted = true;
        break;
      }
      const int stage = n % STAGES;
      const int64_t t0 = T0 + (int64_t)t * TT;
      uint32_t bad = 0;
      int32_t pid[16];
      if (paged) {
        const int64_t pi0 = t0 >> p.log2_page;
        for (int j = 0; j < pages_per_tile; ++j) {
          const int64_t pi = pi0 + j;
          if (pi < cache_base || pi >= cache_base + 32) {
            cache_base = pi;
            const int64_t mine = pi + lane;
            cache = mine < used_pages ? p.block_table[(int64_t)b * p.bt_sb + mine] : -2;
          }
          int32_t id = __shfl_sync(0xffffffffu, cache, (int)(pi - cache_base));
          if (id == -2) {
            id = 0;
          } else if (id < 0 || (int64_t)id >= p.num_pages) {
            bad |= 1u << j;
            id = 0;
          }
          pid[j] = id;
        }
        if (bad && lane == 0) atomicOr(p.flags, FD_DEVFLAG_PAGE);
      }
      if (lane == 0) {
        TileMeta& m = ctl->meta[stage];
        m.b = b;
        m.g = g;
        m.split = split;
        m.flags = (t == 0 ? kMetaFirst : 0) | (t == n_tiles - 1 ? kMetaLast : 0);
        m.t0 = t0;
        m.lo = lo;
        m.hi = hi;
        m.L = L;
        m.bad = bad;
        const uint32_t full = smem_addr(&ctl->full[stage]);
        mbar_arrive_expect_tx(full, 2u * kTileBytes);
        const uint32_t dk = smem_addr(stages + (size_t)stage * 2 * kTileBytes);
        const uint32_t dv = dk + kTileBytes;
        if (!paged) {
          tma_load_5d(dk, tk, full, 0, (int)t0, 0, g, b, pol);
          tma_load_5d(dv, tv, full, 0, (int)t0, 0, g, b, pol);
        } else if (ps >= TT) {
          const int slot = (int)(t0 & (ps - 1));
          tma_load_5d(dk, tk, full, 0, slot, 0, g, pid[0], pol);
          tma_load_5d(dv, tv, full, 0, slot, 0, g, pid[0], pol);
        } else {
          for (int j = 0; j < pages_per_tile; ++j) {
            tma_load_5d(dk + j * box_bytes, tk, full, 0, 0, 0, g, pid[j], pol);
            tma_load_5d(dv + j * box_bytes, tv, full, 0, 0, 0, g, pid[j], pol);
          }
        }
      }
      __syncwarp();
    }
  }
  // Tell the consumers there is nothing more (a stage with kDone, completed by a plain
  // arrive), unless the ring is stuck.
  if (!aborted && acquire(n)) {
    if (lane == 0) {
      ctl->meta[n % STAGES].flags = kMetaDone;
      mbar_arrive(smem_addr(&ctl->full[n % STAGES]));
    }
    __syncwarp();
    ++n;
  }
  // Never leave with copies in flight (bounded waits on the last issued stages).
  if (lane == 0) {
    const int first = n > STAGES ? n - STAGES : 0;
    for (int m = first; m < n; ++m) {
      if (!mbar_wait(smem_addr(&ctl->full[m % STAGES]), (m / STAGES) & 1))
        atomicOr(p.flags, kDevFlagTimeout);
    }
    // The last CTA to finish puts the queue words back to zero, so that a launch that
    // is replayed as is starts from a clean queue too.  The fences order this CTA's
    // last queue ticket before its done ticket, and every done ticket before the reset.
    __threadfence();
    if (atomicAdd(p.ctas_done, 1ull) == gridDim.x - 1ull) {
      __threadfence();
      *p.item_queue = 0ull;
      *p.ctas_done = 0ull;
    }
  }
}

// Page-id window of a producer warp (paged caches): lane i holds the block-table entry
// of page (base + i) of the row, or -2 when that page holds no token of the row (never
// read from the table).
struct PageWindow {
  int64_t base = -64;            // no window loaded yet
  int32_t id = -2;
};

// Issue the K and V copies of the tile whose first logical token is t0 (row si.b, kv
// head si.g) into `stage`, completing on its full barrier.  All 32 lanes resolve page
// ids (they share the window); lane 0 records the invalid-page bits and issues.
//   stages: base of STAGES * 2 * kTileBytes bytes, 1024-byte aligned; stage s holds the
//           K tile at s * 2 * kTileBytes and the V tile kTileBytes after it.  A tile is
//           one TMA box (contiguous cache, or pages of at least a tile) or one box per
//           page; each box is laid out [line][row][128 B] (see tile_chunk), 128-byte
//           swizzled, and 1024-byte aligned (a box is at least 8 rows).
template <int TT, int STAGES>
__device__ __forceinline__ void issue_tile(const Params& p, const SplitInfo& si, int64_t t0,
                                           const CUtensorMap* tk, const CUtensorMap* tv,
                                           uint8_t* stages, PipeCtl<STAGES>* ctl, int stage,
                                           PageWindow& win, uint64_t pol, int lane) {
  const bool paged = p.block_table != nullptr;
  const int ps = p.page_size;
  const int pages_per_tile = paged ? (ps >= TT ? 1 : TT / ps) : 1;
  const int box_rows = paged ? (ps >= TT ? TT : ps) : TT;
  const uint32_t box_bytes = (uint32_t)(kTileBytes / TT) * box_rows;   // all lines of a box
  uint32_t bad = 0;
  int32_t pid[16];  // pages_per_tile <= TT / 8 <= 16 (page_size >= 8 is enforced)
  if (paged) {
    const int64_t pi0 = t0 >> p.log2_page;
    for (int j = 0; j < pages_per_tile; ++j) {
      const int64_t pi = pi0 + j;
      if (pi < win.base || pi >= win.base + 32) {             // warp-uniform refill
        win.base = pi;
        const int64_t mine = pi + lane;
        win.id = mine < si.used_pages ? p.block_table[(int64_t)si.b * p.bt_sb + mine] : -2;
      }
      int32_t id = __shfl_sync(0xffffffffu, win.id, (int)(pi - win.base));
      if (id == -2) {
        id = 0;                          // no token of the row here: any valid page
      } else if (id < 0 || (int64_t)id >= p.num_pages) {
        bad |= 1u << j;                  // a used entry out of range: exclude its tokens
        id = 0;
      }
      pid[j] = id;
    }
    if (bad && lane == 0) atomicOr(p.flags, FD_DEVFLAG_PAGE);
  }
  if (lane == 0) {
    ctl->bad[stage] = bad;
    const uint32_t full = smem_addr(&ctl->full[stage]);
    mbar_arrive_expect_tx(full, 2u * kTileBytes);
    const uint32_t dk = smem_addr(stages + (size_t)stage * 2 * kTileBytes);
    const uint32_t dv = dk + kTileBytes;
    // Coordinates: {element 0, token row, line 0, kv head, batch row | page}.
    if (!paged) {
      tma_load_5d(dk, tk, full, 0, (int)t0, 0, si.g, si.b, pol);
      tma_load_5d(dv, tv, full, 0, (int)t0, 0, si.g, si.b, pol);
    } else if (ps >= TT) {
      const int slot = (int)(t0 & (ps - 1));
      tma_load_5d(dk, tk, full, 0, slot, 0, si.g, pid[0], pol);
      tma_load_5d(dv, tv, full, 0, slot, 0, si.g, pid[0], pol);
    } else {
      for (int j = 0; j < pages_per_tile; ++j) {
        tma_load_5d(dk + j * box_bytes, tk, full, 0, 0, 0, si.g, pid[j], pol);
        tma_load_5d(dv + j * box_bytes, tv, full, 0, 0, 0, si.g, pid[j], pol);
      }
    }
  }
}

// Acquire ring slot n for the producer warp: wait (lane 0, bounded) until the consumers
// have released the tile that used the stage before; on a timeout the split is aborted
// and flagged.  Every lane returns the same answer.
template <int STAGES>
__device__ __forceinline__ bool acquire_slot(const Params& p, PipeCtl<STAGES>* ctl, int n,
                                             int lane) {
  if (n < STAGES) return true;
  int ok = 1;
  if (lane == 0) ok = mbar_wait(smem_addr(&ctl->empty[n % STAGES]), ((n / STAGES) - 1) & 1);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok && lane == 0) {
    ctl->abort = 1;
    atomicOr(p.flags, kDevFlagTimeout);
  }
  return ok != 0;
}

// Never leave with copies in flight: wait (bounded) for the last issued use of each
// stage (n slots issued in all).  Earlier uses of a stage completed before it was reused.
template <int STAGES>
__device__ __forceinline__ void drain_ring(const Params& p, PipeCtl<STAGES>* ctl, int n,
                                           int lane) {
  if (lane == 0) {
    const int first = n > STAGES ? n - STAGES : 0;
    for (int m = first; m < n; ++m) {
      if (!mbar_wait(smem_addr(&ctl->full[m % STAGES]), (m / STAGES) & 1)) {
        atomicOr(p.flags, kDevFlagTimeout);
      }
    }
  }
}

// Producer warp: streams tiles 0..n_tiles-1 of the split.  All 32 lanes run the loop
// (they share the page-id window); lane 0 issues the copies.
// HPC: kv heads per CTA of the grid (1, or kHeadGroup for head-group tiles).
template <int TT, int STAGES, int HPC = 1>
__device__ __forceinline__ void produce_tiles(const Params& p, const SplitInfo& si,
                                              const CUtensorMap* tk, const CUtensorMap* tv,
                                              uint8_t* stages, PipeCtl<STAGES>* ctl,
                                              int lane) {
  const uint64_t pol = policy_evict_first();
  PageWindow win;
  int n = 0;
  for (; n < si.n_tiles; ++n) {
    if (selftest_stops(p, n)) break;
    if (!acquire_slot(p, ctl, n, lane)) break;
    if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int32_t*>(&ctl->abort), 0)) break;
    issue_tile<TT, STAGES>(p, si, si.T0 + (int64_t)n * TT, tk, tv, stages, ctl, n % STAGES,
                           win, pol, lane);
    __syncwarp();
  }
  if (n == si.n_tiles && lane == 0) prefetch_next_wave<TT, HPC>(p, tk, tv, STAGES);
  drain_ring(p, ctl, n, lane);
}

// ---------------------------------------------------------------- tail sharing
//
// CTAs stream at rates that differ by a few percent (which memory channels their
// addresses hit), so with one split per CTA the last splits finish well after the
// average one.  Tail sharing lets a CTA that has finished its own split continue with
// tiles of a split of the SAME (b, kv head) that is still in progress: same query rows,
// so the extra keys simply join the helper's own running maximum, sum and accumulator,
// and its partial (O_i, LSE_i) then covers its split plus the stolen tiles.  Every key
// is still counted exactly once over the row's partials, and the LSE-weighted merge of
// "2kiu.com/news/6053916" (section "weight block results with log-sum-exp") is exact
// whatever keys each partial holds.  Each CTA's stream stays contiguous: the owner takes
// its tiles from the front of its split in chunks of kClaimChunk (fetch-and-add on the
// split's claim word), a helper takes the back half of the largest unclaimed remainder
// (compare-and-swap), so no address interleaving between CTAs arises.
constexpr uint32_t kClaimChunk = 2;   // tiles an owner claims at a time
constexpr int kClaimAhead = 2;        // an owner's claims in flight
constexpr uint32_t kMinSteal = 2;     // a helper takes half of at least this many tiles

__device__ __forceinline__ unsigned long long claim_pack(uint32_t front, uint32_t back) {
  return ((unsigned long long)back << 32) | front;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* a) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* a, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// The split of the helper's (b, kv head) group with the most unclaimed tiles (at least
// kMinSteal), whose back half the helper then claims.  Only splits whose owner has
// published this call's epoch are considered.  On success the piece is tiles [cur, end)
// of that split (relative to its first tile T0) with valid range [lo, hi).  Bounded: a
// lost compare-and-swap is retried a fixed number of times.
template <int TT>
__device__ __forceinline__ bool steal_piece(const Params& p, const SplitInfo& si,
                                            StealWord* group, int lane, int64_t& T0,
                                            int64_t& lo, int64_t& hi, uint32_t& cur,
                                            uint32_t& end) {
  for (int attempt = 0; attempt < 64; ++attempt) {
    uint32_t best_rem = 0;
    int best = -1;
    unsigned long long best_w = 0;
    for (int s = lane; s < p.S; s += 32) {
      if (ld_acquire_u32(&group[s].epoch) != p.epoch) continue;
      const unsigned long long w = ld_relaxed_u64(&group[s].claim);
      const uint32_t f = (uint32_t)w, bk = (uint32_t)(w >> 32);
      const uint32_t rem = bk > f ? bk - f : 0u;
      if (rem > best_rem) {
        best_rem = rem;
        best = s;
        best_w = w;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {      // arg-max over (remainder, split)
      const uint32_t r2 = __shfl_xor_sync(0xffffffffu, best_rem, off);
      const int s2 = __shfl_xor_sync(0xffffffffu, best, off);
      const unsigned long long w2 = __shfl_xor_sync(0xffffffffu, best_w, off);
      if (r2 > best_rem || (r2 == best_rem && s2 > best)) {
        best_rem = r2;
        best = s2;
        best_w = w2;
      }
    }
    if (best_rem < kMinSteal) return false;
    const uint32_t f = (uint32_t)best_w, bk = (uint32_t)(best_w >> 32);
    const uint32_t k = best_rem / 2;
    int ok = 0;
    if (lane == 0) ok = atomicCAS(&group[best].claim, best_w, claim_pack(f, bk - k)) == best_w;
    if (__shfl_sync(0xffffffffu, ok, 0)) {
      split_range<TT>(p, best, si.L, lo, hi);
      T0 = lo / TT * TT;
      cur = bk - k;
      end = bk;
      return true;
    }
  }
  return false;
}

// One fetch-and-add claim of kClaimChunk tiles on an owner's word, into ticket slot
// `slot` (lane 0 holds the tickets in separate registers).  Measured: the claims cost the
// producer 0.16-0.4 us each whatever the number in flight (1 to 3), so how long a claim
// takes to come back is not the whole cost.
__device__ __forceinline__ void claim_into(int slot, unsigned long long* word,
                                           unsigned long long& t0, unsigned long long& t1,
                                           unsigned long long& t2) {
  const unsigned long long add = (unsigned long long)kClaimChunk;
  if (slot == 0) t0 = atomicAdd(word, add);
  else if (slot == 1) t1 = atomicAdd(word, add);
  else t2 = atomicAdd(word, add);
}
__device__ __forceinline__ unsigned long long ticket_of(int slot, unsigned long long t0,
                                                        unsigned long long t1,
                                                        unsigned long long t2) {
  return __shfl_sync(0xffffffffu, slot == 0 ? t0 : (slot == 1 ? t1 : t2), 0);
}

// Producer warp of the kernels whose consumers read the tile descriptors (t0, lo, hi,
// done) of each stage: streams the CTA's own split and, with `share`, tiles taken from
// other splits of the same (b, kv head) afterwards (see above); then publishes two done
// stages (one for each tile parity: some consumers take every other tile) carrying
// n_total.  Without `share` the sequence is exactly the split's tiles, in order.
// The owner keeps kClaimAhead claims in flight; a helper looks for a piece when the
// current one is exhausted (the ring still holds the tiles it has issued).
template <int TT, int STAGES>
__device__ __forceinline__ void produce_tiles_shared(const Params& p, const SplitInfo& si,
                                                     const CUtensorMap* tk,
                                                     const CUtensorMap* tv, uint8_t* stages,
                                                     PipeCtl<STAGES>* ctl, int lane,
                                                     bool share) {
  static_assert(kClaimAhead >= 1 && kClaimAhead <= 3, "one to three claims in flight");
  const uint64_t pol = policy_evict_first();
  PageWindow win;
  const uint32_t n_own = (uint32_t)si.n_tiles;
  StealWord* group = share ? p.steal + ((int64_t)si.b * p.Hkv + si.g) * p.S : nullptr;
  StealWord* mine = share ? group + si.split : nullptr;
  // The piece being streamed: tiles [cur, end) of a split whose first tile starts at
  // logical token T0, valid range [lo, hi).  First the own split.
  int64_t T0 = si.T0, lo = si.lo, hi = si.hi;
  uint32_t cur = 0, end = share ? min(kClaimChunk, n_own) : n_own;
  // Own claims in flight: ticket slots used round robin, oldest at `head`.
  unsigned long long t0r = 0, t1r = 0, t2r = 0;
  int head = 0, live = 0;
  uint32_t next_f = end;                   // the front the next claim is expected to see
  bool own = true;
  if (share) {
    if (lane == 0) {
      // Publish the split's unclaimed range [end, n_own); the epoch (written last) tells
      // helpers that the word belongs to this call.
      atomicExch(&mine->claim, claim_pack(end, n_own));
      __threadfence();
      st_release_u32(&mine->epoch, p.epoch);
    }
    for (; next_f < n_own && live < kClaimAhead; next_f += kClaimChunk, ++live) {
      if (lane == 0) claim_into((head + live) % kClaimAhead, &mine->claim, t0r, t1r, t2r);
    }
  }
  int n = 0;
  bool aborted = false;
  for (;;) {
    if (cur >= end && own && live > 0) {       // the next chunk of the own split
      const unsigned long long old = ticket_of(head, t0r, t1r, t2r);
      const uint32_t f = (uint32_t)old, bk = (uint32_t)(old >> 32);
      head = (head + 1) % kClaimAhead;
      --live;
      cur = f;
      end = f < bk ? min(f + kClaimChunk, bk) : f;
      if (end >= bk) {
        live = 0;                              // the rest come back empty
      } else if (next_f < bk) {
        if (lane == 0) claim_into((head + live) % kClaimAhead, &mine->claim, t0r, t1r, t2r);
        ++live;
        next_f += kClaimChunk;
      }
    }
    if (cur >= end) {                          // the current piece is exhausted
      own = false;
      if (!share || !steal_piece<TT>(p, si, group, lane, T0, lo, hi, cur, end)) break;
    }
    if (selftest_stops(p, n) || !acquire_slot(p, ctl, n, lane) ||
        __shfl_sync(0xffffffffu, *reinterpret_cast<volatile int32_t*>(&ctl->abort), 0)) {
      aborted = true;
      break;
    }
    const int stage = n % STAGES;
    const int64_t t0 = T0 + (int64_t)cur * TT;
    if (lane == 0) {
      ctl->t0[stage] = t0;
      ctl->lo[stage] = lo;
      ctl->hi[stage] = hi;
      ctl->done[stage] = 0;
    }
    issue_tile<TT, STAGES>(p, si, t0, tk, tv, stages, ctl, stage, win, pol, lane);
    __syncwarp();
    ++cur;
    ++n;
  }
  const int n_total = n;
  if (!aborted && lane == 0) prefetch_next_wave<TT>(p, tk, tv, STAGES);
  if (!aborted) {
    for (int k = 0; k < 2; ++k) {            // the end, for each tile parity
      if (!acquire_slot(p, ctl, n, lane)) break;
      if (lane == 0) {
        const int stage = n % STAGES;
        ctl->done[stage] = 1;
        ctl->n_total = n_total;
        mbar_arrive(smem_addr(&ctl->full[stage]));
      }
      __syncwarp();
      ++n;
    }
  }
  // Close the own split's word: nothing more can be taken from it in this call or, for
  // a launch that is replayed as is, before its owner opens it again.
  if (share && lane == 0) atomicExch(&mine->claim, claim_pack(0x7fffffffu, 0u));
  drain_ring(p, ctl, n, lane);
}

}  // namespace fd
