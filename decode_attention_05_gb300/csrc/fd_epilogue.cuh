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

#include "fd_pipeline.cuh"

namespace fd {

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Split epilogue for an empty (or aborted) split: LSE_i = -inf for the whole group.
__device__ __forceinline__ void write_empty_split(const Params& p, const SplitInfo& si, int tid) {
  if (tid < p.G) {
    const int64_t row = (int64_t)si.b * p.Hq + (int64_t)si.g * p.G + tid;
    p.lse_part[row * p.S + si.split] = kNegInf;
  }
}

// macc [NCW][G][D], mm [NCW][G], ml [NCW][G] in shared memory, filled by every warp;
// called by all NCW * 32 consumer threads (ctid = 0 .. NCW * 32 - 1) after a barrier.
template <int G, int D, int NCW>
__device__ __forceinline__ void merge_warps_and_store(const Params& p, const SplitInfo& si,
                                                      const float* macc, const float* mm,
                                                      const float* ml, int ctid) {
  const int64_t row0 = (int64_t)si.b * p.Hq + (int64_t)si.g * G;
  for (int idx = ctid; idx < G * D; idx += NCW * 32) {
    const int h = idx / D, j = idx % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, mm[w * G + h]);
    float L = 0.f, O = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < NCW; ++w) {
        const float mw = mm[w * G + h];
        const float c = (mw == kNegInf) ? 0.f : ex2(mw - M);
        L = fmaf(ml[w * G + h], c, L);
        O = fmaf(macc[(w * G + h) * D + j], c, O);
      }
    }
    const int64_t row = row0 + h;
    if (L > 0.f) {
      p.o_part[(row * p.S + si.split) * D + j] = O / L;
      if (j == 0) p.lse_part[row * p.S + si.split] = (M + lg2_approx(L)) * 0.6931471805599453f;
    } else if (j == 0) {
      p.lse_part[row * p.S + si.split] = kNegInf;
    }
  }
}

}  // namespace fd
