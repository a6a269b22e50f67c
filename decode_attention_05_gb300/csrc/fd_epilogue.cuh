// fd_epilogue.cuh -- end of a split: merge the consumer warps' online-softmax states
// and write the split's partial output and LSE.
//
// Each of NCW warps saw a disjoint subset of the split's tokens and holds, per query
// head h, a running max m_w (base-2 logits), a shifted exp-sum l_w and an un-normalised
// accumulator acc_w = sum_t 2^(s_t - m_w) v_t.  They are merged with the same weights
// as the split merge ("2kiu.com/news/6053916", section "why this counter-example exposes
// averaging": the (max, exp-sum, weighted sum) and (normalised output, LSE) encodings
// are equivalent, but one's normalised output must not stand in for the other's raw
// accumulator):
//   M = max_w m_w,  c_w = 2^(m_w - M),  L = sum_w c_w l_w,  O = sum_w c_w acc_w / L.
// The split then writes O_i = O and LSE_i = (M + log2 L) ln 2 (natural log), i.e.
// "FlashDecoding interview notes" (gtnt.cn/news/53829), section two: O_i = acc_i / l_i,
// and section three: LSE_i = m_i + log(l_i).  A split whose keys were all excluded
// writes LSE_i = -inf and no O_i.
#pragma once

#include <cuda_bf16.h>

#include "fd_pipeline.cuh"

namespace fd {

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Split epilogue for an empty (or aborted) split: LSE_i = -inf for the whole group.
__device__ __forceinline__ void write_empty_split(const Params& p, const SplitInfo& si, int tid) {
  if (tid < p.n_rows) put_empty_row(p, si.b, si.g, tid, si.split);
}

// Index of (warp w, row h, dim j) in the merge scratch macc [NCW][G][D].  The dims of
// a row are XOR-swizzled by 8 x ((h / 2) mod 4): the tensor-core epilogue's lanes write
// rows 2 apart at the same dims, which then fall in different banks; groups of 4
// consecutive dims stay together (16-byte reads).
template <int G, int D>
__device__ __forceinline__ int macc_index(int w, int h, int j) {
  static_assert(D % 32 == 0, "the swizzle needs 32 dims per row");
  return (w * G + h) * D + (j ^ (((h >> 1) & 3) << 3));
}

// macc [NCW][G][D] (macc_index), mm [NCW][G], ml [NCW][G] in shared memory (G = query
// rows of the group, a power of two >= p.n_rows), filled by every warp for rows
// < p.n_rows; called by all NCW * 32 consumer threads (ctid = 0 .. NCW * 32 - 1) after
// they are visible.  One thread per row turns the warps' maxima into weights
// w_w = 2^(m_w - M) / L (kept in mm; L in ml[h]) and writes LSE_i; `sync` makes them
// visible to all (it returns false if the threads could not meet; nothing more is
// written then); every thread then forms 4 output dims at a time.  Returns sync's
// answer.
template <int G, int D, int NCW, bool DIRECT = true, class Sync>
__device__ __forceinline__ bool merge_warps_and_store(const Params& p, const SplitInfo& si,
                                                      const float* macc, float* mm, float* ml,
                                                      int ctid, Sync&& sync) {
  if (ctid < p.n_rows) {
    const int h = ctid;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, mm[w * G + h]);
    float c[NCW], L = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float mw = mm[w * G + h];
      c[w] = (M == kNegInf || mw == kNegInf) ? 0.f : ex2(mw - M);
      L = fmaf(ml[w * G + h], c[w], L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) mm[w * G + h] = c[w] * inv;
    ml[h] = L;
    put_lse<DIRECT>(p, si.b, si.g, h, si.split,
                    L > 0.f ? (M + lg2_approx(L)) * 0.6931471805599453f : kNegInf);
  }
  if (!sync()) return false;
  constexpr int D4 = D / 4;
  if (DIRECT && p.direct) {
    // A single split's result is the output: every row is written, zeros for a row
    // without keys.
    for (int idx = ctid; idx < p.n_rows * D4; idx += NCW * 32) {
      const int h = idx / D4, j = (idx - h * D4) * 4;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ml[h] > 0.f) {
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float f = mm[w * G + h];
          const float4 a = *reinterpret_cast<const float4*>(macc + macc_index<G, D>(w, h, j));
          o.x = fmaf(a.x, f, o.x);
          o.y = fmaf(a.y, f, o.y);
          o.z = fmaf(a.z, f, o.z);
          o.w = fmaf(a.w, f, o.w);
        }
      }
      put_out4(p, si.b, si.g, h, j, o);
    }
    return true;
  }
  for (int idx = ctid; idx < p.n_rows * D4; idx += NCW * 32) {
    const int h = idx / D4, j = (idx - h * D4) * 4;
    if (!(ml[h] > 0.f)) continue;                   // no key in the split: no O_i
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float f = mm[w * G + h];
      const float4 a = *reinterpret_cast<const float4*>(macc + macc_index<G, D>(w, h, j));
      o.x = fmaf(a.x, f, o.x);
      o.y = fmaf(a.y, f, o.y);
      o.z = fmaf(a.z, f, o.z);
      o.w = fmaf(a.w, f, o.w);
    }
    const int64_t row = flat_row(p, si.b, si.g, h);
    *reinterpret_cast<float4*>(p.o_part + (row * p.S + si.split) * D + j) = o;
  }
  return true;
}

// ---------------------------------------------------------------- fused merge
//
// Single-launch decode: every CTA of a (b, kv head) group -- empty splits included --
// publishes its partials, then takes a ticket on the group's counter; the CTA that
// draws the last ticket merges the group's G query heads.  No CTA ever waits for
// another: the last to arrive finds every partial already visible (each CTA fences
// once, after a barrier, before its ticket; the last one fences after it), so there is
// no second kernel and
// no grid-wide dependency ("2kiu.com/news/6053916", section "the split count is a cost
// account": the merge may start only when every partial it needs is visible).
//
// Merge of one output row by one warp (a lane holds D / 32 dims): the splits are
// folded BATCH at a time with a running maximum, the same online rule as inside a
// split, so all loads of a batch are issued before any result is needed:
//   M' = max(M, max_s LSE_s),  W = W 2^(M - M') + sum_s 2^(LSE_s - M'),
//   acc = acc 2^(M - M') + sum_s 2^(LSE_s - M') O_s          (base-2 of the natural LSEs)
// ending with out = acc / W and lse_out = M + log W.  An empty split (LSE = -inf) has
// weight 0 and its O_s never reaches the sum (it is selected away, never multiplied:
// its memory may hold anything).  A row with no non-empty split gives 0 and -inf.
// Row index: (b * Q + j) * Hq + h.  Loads bypass L1 (partials of the running grid).
template <int D, int BATCH>
__device__ __forceinline__ void merge_row(const Params& p, int64_t row, int lane) {
  constexpr int VEC = D / 32;
  constexpr float kLog2e = 1.4426950408889634f;
  const float* lse = p.lse_part + row * p.S;
  const float* ob = p.o_part + row * p.S * D + lane * VEC;
  float M = kNegInf, W = 0.f, acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < p.S; s0 += BATCH) {
    float ls[BATCH], v[BATCH][VEC];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const bool in = s0 + u < p.S;
      ls[u] = in ? __ldcg(lse + s0 + u) * kLog2e : kNegInf;
      if constexpr (VEC == 4) {
        const float4 t = in ? __ldcg(reinterpret_cast<const float4*>(ob + (int64_t)(s0 + u) * D))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
      } else {
        const float2 t = in ? __ldcg(reinterpret_cast<const float2*>(ob + (int64_t)(s0 + u) * D))
                            : make_float2(0.f, 0.f);
        v[u][0] = t.x; v[u][1] = t.y;
      }
    }
    float mb = ls[0];
#pragma unroll
    for (int u = 1; u < BATCH; ++u) mb = fmaxf(mb, ls[u]);
    const float mn = fmaxf(M, mb);
    if (mn == kNegInf) continue;                    // nothing non-empty yet
    const float c = (M == kNegInf) ? 0.f : ex2(M - mn);
    W *= c;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] *= c;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const bool live = ls[u] != kNegInf;
      const float w = live ? ex2(ls[u] - mn) : 0.f;
      W += w;
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, live ? v[u][e] : 0.f, acc[e]);
    }
    M = mn;
  }
  const int64_t bj = row / p.Hq;
  const int hq = (int)(row - bj * p.Hq);
  const int64_t b = bj / p.Q;
  const int j = (int)(bj - b * p.Q);
  const int64_t obase = b * p.out_sb + (int64_t)j * p.out_sj + (int64_t)hq * p.out_sh + lane * VEC;
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    const float o = acc[e] * inv;
    if (p.out_bf16) {
      reinterpret_cast<__nv_bfloat16*>(p.out)[obase + e] = __float2bfloat16_rn(o);
    } else {
      reinterpret_cast<float*>(p.out)[obase + e] = o;
    }
  }
  if (lane == 0 && p.lse_out != nullptr)
    p.lse_out[row] = W > 0.f ? (M + lg2_approx(W)) * 0.6931471805599453f : kNegInf;
}

// The merge of a (b, kv head) group's rows inside the partial pass: warp w of the NCW
// consumer warps takes rows w, w + NCW, ...
template <int D, int NCW>
__device__ __forceinline__ void merge_group(const Params& p, int b, int g, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  for (int rho = warp; rho < p.n_rows; rho += NCW) merge_row<D, 16>(p, flat_row(p, b, g, rho), lane);
}

// Called by the NCW * 32 consumer threads of a CTA after it has written its partials
// (or its empty-split LSE).  `flag` is a shared-memory word.
template <int D, int NCW>
__device__ __forceinline__ void arrive_and_merge(const Params& p, const SplitInfo& si, int ctid,
                                                 int32_t* flag) {
  unsigned long long* c = &p.counters[(int64_t)si.b * p.Hkv + si.g];
  // The barrier makes every consumer thread's partial writes visible to thread 0; its
  // gpu-scope fence then publishes them (cumulatively) before its ticket.
  named_bar_sync(1, NCW * 32);
  if (ctid == 0) {
    __threadfence();
    const bool last = take_ticket(p, c) == (unsigned)p.S;
    if (last) __threadfence();                       // acquire the other CTAs' partials
    *flag = last ? 1 : 0;
  }
  named_bar_sync(1, NCW * 32);
  if (*flag == 0) return;
  merge_group<D, NCW>(p, si.b, si.g, ctid);
  if (ctid == 0) *c = 0ull;                          // clean for a replay of this launch
}

}  // namespace fd
