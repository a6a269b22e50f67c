// fd_partial_simt.cuh -- split-KV partial pass with CUDA-core dot products.
//
// One CTA = one split of one (batch row b, kv head g) and all query rows that read kv
// head g: its G query heads, times Q query tokens in multi-token decode (template G is
// that row count rounded up to a power of two).  Warp 4 is the TMA producer
// (fd_pipeline.cuh); warps 0-3 consume tiles.
//
// Per tile, each consumer warp takes TT/4 token rows.  A lane owns EPL consecutive
// dims of a row (LPR lanes cover one row, RPW rows per warp step), keeps the matching
// slice of the G query vectors in registers (pre-scaled by log2(e)/sqrt(d), so scores
// are base-2 logits), and the G x EPL slice of the accumulator.  For a batch of rows:
//   s[h]   = q_h . k_t / sqrt(d)                 (dot over the lane's dims, then a
//                                                  butterfly sum across the LPR lanes)
//   s[h]   = -inf for t outside [lo, hi), on an invalid page, or past row h's causal
//            bound (excluded, not added)
//   m_new  = max(m, max_t s)                     (safe-softmax shift)
//   c      = 2^(m - m_new);  l = l c;  acc = acc c   (only when some m grows)
//   p      = 2^(s - m_new);  l += p;  acc += p v_t
// which is the online-softmax / FlashAttention loop of "AI Infra: math and infra
// optimisation in large models", section 2.6 ("Online Softmax" and the FlashAttention
// update: rescale the old sum and output by exp(m_old - m_new), then add the new tile).
// At the end the four warps' (m, l, acc) are merged with the same weights as the
// split merge, and the CTA writes O_i = acc / l and LSE_i = (m + log2 l) ln 2 for its
// split ("FlashDecoding interview notes", section two: O_i = acc_i / l_i; section three:
// LSE_i = m_i + log l_i).  A split with no valid key writes LSE_i = -inf and no O_i.
#pragma once

#include "fd_epilogue.cuh"

namespace fd {

template <int ESZ_, int D_, int G_>
struct SimtShape {
  static constexpr int ESZ = ESZ_;
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int ROW_BYTES = D * ESZ;
  static constexpr int TT = kTileBytes / ROW_BYTES;          // tokens per tile
  static constexpr int LINES = ROW_BYTES / 128;              // 128-byte lines per row
  static constexpr int EPL = (G >= 16 || ESZ == 4) ? 4 : 8;  // elements per lane
  static constexpr int BPL = EPL * ESZ;                      // bytes per lane: 8 or 16
  static constexpr int LPR = D / EPL;                        // lanes per row
  static constexpr int RPW = 32 / LPR;                       // rows per warp step
  static constexpr int NCW = 4;                              // consumer warps
  static constexpr int ROWS_PER_WARP = TT / NCW;
  static constexpr int NSTEP = ROWS_PER_WARP / RPW;
  static constexpr int SB0 = 32 / G > 2 ? 32 / G : 2;
  static constexpr int SB = NSTEP < SB0 ? NSTEP : SB0;       // rows steps per softmax batch
  static constexpr int STAGES = 3;
  static constexpr int THREADS = (NCW + 1) * 32;
  static_assert(LPR <= 32 && 32 % LPR == 0, "lane layout");
  static_assert(NSTEP % SB == 0, "batching");
  // Merge scratch (reuses the stage buffers once the pipeline has drained).
  static constexpr int MERGE_BYTES = NCW * G * D * 4 + 2 * NCW * G * 4;
  static_assert(MERGE_BYTES <= STAGES * 2 * kTileBytes, "merge scratch fits the stages");
  static constexpr size_t SMEM_BYTES =
      1024 /*alignment slack*/ + (size_t)STAGES * 2 * kTileBytes + sizeof(PipeCtl<STAGES>);
};

// Load this lane's EPL elements of token row r from a swizzled tile, widened to f32.
template <class SH>
__device__ __forceinline__ void load_row_slice(const uint8_t* tile, int r, int li, uint32_t lb,
                                               float (&f)[SH::EPL]) {
  const int off = li * SH::BPL;                               // byte offset in the row
  const uint32_t a = tile_chunk<SH::LINES>((uint32_t)r, (uint32_t)(off >> 4), lb) + (off & 15);
  if constexpr (SH::BPL == 16) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + a);
    if constexpr (SH::ESZ == 2) {
      f[0] = bf16lo_to_f32(u.x); f[1] = bf16hi_to_f32(u.x);
      f[2] = bf16lo_to_f32(u.y); f[3] = bf16hi_to_f32(u.y);
      f[4] = bf16lo_to_f32(u.z); f[5] = bf16hi_to_f32(u.z);
      f[6] = bf16lo_to_f32(u.w); f[7] = bf16hi_to_f32(u.w);
    } else {
      f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
      f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(tile + a);
    f[0] = bf16lo_to_f32(u.x); f[1] = bf16hi_to_f32(u.x);
    f[2] = bf16lo_to_f32(u.y); f[3] = bf16hi_to_f32(u.y);
  }
}

// Load EPL query elements from global memory, widened to f32.
template <class SH>
__device__ __forceinline__ void load_q_slice(const void* q, int64_t off, float (&f)[SH::EPL]) {
  if constexpr (SH::ESZ == 2) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(q) + off;
#pragma unroll
    for (int e = 0; e < SH::EPL; ++e) f[e] = __uint_as_float((uint32_t)p[e] << 16);
  } else {
    const float* p = reinterpret_cast<const float*>(q) + off;
#pragma unroll
    for (int e = 0; e < SH::EPL; ++e) f[e] = p[e];
  }
}

template <class SH>
// Two CTAs of 160 threads per SM leave 204 registers per thread; __launch_bounds__ would
// budget for 192-thread CTAs and cap at 168, which spills the wide GQA accumulators.
__global__ void __maxnreg__(200)
    fd_partial_simt_kernel(const __grid_constant__ CUtensorMap tk,
                           const __grid_constant__ CUtensorMap tv,
                           const __grid_constant__ Params p) {
  constexpr int G = SH::G, EPL = SH::EPL, LPR = SH::LPR, RPW = SH::RPW, TT = SH::TT;
  constexpr int STAGES = SH::STAGES;
  pdl_wait();                       // inputs of this step are visible
  const SplitInfo si = split_info<TT>(p);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<PipeCtl<STAGES>*>(stages + (size_t)STAGES * 2 * kTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (si.n_tiles == 0) {            // empty split: weight 0 in the merge, nothing to load
    write_empty_split(p, si, threadIdx.x);
    pdl_trigger();
    if (p.counters != nullptr && warp < SH::NCW)
      arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), SH::NCW);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == SH::NCW) {            // ---------------- producer warp
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    produce_tiles<TT, STAGES>(p, si, &tk, &tv, stages, ctl, lane);
    pdl_trigger();
    return;
  }

  // ---------------------------------------------------- consumer warps
  const int rg = lane / LPR;        // row within a warp step
  const int li = lane % LPR;        // lane within the row
  // Row h of the group (query token h / p.G, head h mod p.G); rows past p.n_rows pad
  // the template size and stay zero.
  float qv[G][EPL];
  int64_t lim[G];                   // causal key bound of each row
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const bool live = h < p.n_rows;
    load_q_slice<SH>(p.q, q_offset(p, si.b, si.g, live ? h : 0) + li * EPL, qv[h]);
#pragma unroll
    for (int e = 0; e < EPL; ++e) qv[h][e] = live ? qv[h][e] * p.scale_log2 : 0.f;
    lim[h] = key_bound(p, si.L, h);
  }
  float m[G], l[G], acc[G][EPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = kNegInf;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
  }
  const int ps = p.page_size;
  const bool multi_page = ps > 0 && ps < TT;
  const uint32_t lb = (uint32_t)p.log2_box;
  bool aborted = false;

  for (int n = 0; n < si.n_tiles; ++n) {
    const int stage = n % STAGES;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_addr(&ctl->full[stage]), (n / STAGES) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) {
        ctl->abort = 1;
        atomicOr(p.flags, kDevFlagTimeout);
      }
      aborted = true;
      break;
    }
    const uint8_t* kt = stages + (size_t)stage * 2 * kTileBytes;
    const uint8_t* vt = kt + kTileBytes;
    const uint32_t bad = ctl->bad[stage];
    const int64_t t0 = si.T0 + (int64_t)n * TT;

#pragma unroll 1
    for (int sb = 0; sb < SH::NSTEP; sb += SH::SB) {
      float s[SH::SB][G];
      bool valid[SH::SB];
      int64_t toks[SH::SB];
#pragma unroll
      for (int st = 0; st < SH::SB; ++st) {
        const int r = warp * SH::ROWS_PER_WARP + (sb + st) * RPW + rg;
        const int64_t tok = t0 + r;
        toks[st] = tok;
        const int pslot = multi_page ? (r >> p.log2_page) : 0;
        valid[st] = tok >= si.lo && tok < si.hi && !((bad >> pslot) & 1u);
        float kf[EPL];
        load_row_slice<SH>(kt, r, li, lb, kf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) a = fmaf(qv[h][e], kf[e], a);
          s[st][h] = a;
        }
      }
      // Sum the partial dots over the LPR lanes of each row.
#pragma unroll
      for (int st = 0; st < SH::SB; ++st)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int off = 1; off < LPR; off <<= 1)
            s[st][h] += __shfl_xor_sync(0xffffffffu, s[st][h], off);
      // Length / page mask: excluded keys get -inf (never a finite sentinel).
      float mx[G];
#pragma unroll
      for (int h = 0; h < G; ++h) mx[h] = kNegInf;
#pragma unroll
      for (int st = 0; st < SH::SB; ++st)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          s[st][h] = (valid[st] && toks[st] < lim[h]) ? s[st][h] : kNegInf;
          mx[h] = fmaxf(mx[h], s[st][h]);
        }
      bool grow = false;
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1)
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], off));
        grow |= mx[h] > m[h];
      }
      if (grow) {                   // uniform across the warp: m and mx are warp-wide
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mn = fmaxf(m[h], mx[h]);
          const float c = (mn == kNegInf) ? 1.f : ex2(m[h] - mn);   // ex2(-inf) = 0
          l[h] *= c;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[h][e] *= c;
          m[h] = mn;
        }
      }
#pragma unroll
      for (int st = 0; st < SH::SB; ++st) {
        const int r = warp * SH::ROWS_PER_WARP + (sb + st) * RPW + rg;
        float vf[EPL];
        load_row_slice<SH>(vt, r, li, lb, vf);
#pragma unroll
        for (int e = 0; e < EPL; ++e) vf[e] = valid[st] ? vf[e] : 0.f;   // stale rows may be NaN
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pr = s[st][h] != kNegInf ? ex2(s[st][h] - m[h]) : 0.f;
          l[h] += pr;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[h][e] = fmaf(pr, vf[e], acc[h][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl->empty[stage]));
  }
  pdl_trigger();

  // All consumer warps agree on abort (it is read after the barrier below).
  named_bar_sync(1, SH::NCW * 32);
  if (aborted || *reinterpret_cast<volatile int32_t*>(&ctl->abort)) {
    if (warp == 0) write_empty_split(p, si, threadIdx.x);
    if (p.counters != nullptr) arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
    return;
  }

  // Sum l and acc over the row groups of the warp (each group saw different rows).
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
    }
  }
  // Intra-CTA merge of the four warps' (m, l, acc), through the drained stage buffers.
  float* macc = reinterpret_cast<float*>(stages);                 // [NCW][G][D], swizzled
  float* mm = macc + SH::NCW * G * SH::D;                         // [NCW][G]
  float* ml = mm + SH::NCW * G;                                   // [NCW][G]
  if (rg == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
      if (h < p.n_rows)
#pragma unroll
        for (int e = 0; e < EPL; ++e) macc[macc_index<G, SH::D>(warp, h, li * EPL + e)] = acc[h][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      mm[warp * G + h] = m[h];
      ml[warp * G + h] = l[h];
    }
  }
  named_bar_sync(1, SH::NCW * 32);
  merge_warps_and_store<G, SH::D, SH::NCW>(p, si, macc, mm, ml, threadIdx.x, [] {
    named_bar_sync(1, SH::NCW * 32);
    return true;
  });
  if (p.counters != nullptr) arrive_and_merge<SH::D, SH::NCW>(p, si, threadIdx.x, &ctl->last);
}

}  // namespace fd
