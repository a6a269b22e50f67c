// fd_combine.cu -- the merge pass of split-KV decode: one CTA per (b, query token,
// query head) row, or, for calls with many rows, one warp per row.
//
// Reads the S partials (O_i, LSE_i) of its row and computes
//   M = max over non-empty splits of LSE_i,   w_i = exp(LSE_i - M)  in (0, 1],
//   out = sum_i w_i O_i / sum_i w_i,          lse_out = M + log(sum_i w_i)
// in one pass: the splits are folded with a running maximum (when M grows, what was
// summed so far is rescaled by exp(M_old - M_new)), so no load waits for a maximum.
// ("FlashDecoding interview notes" (gtnt.cn/news/53829), section three, point 2: the
// weights use LSE_i - LSE_global <= 0, so no exponent can overflow; "2kiu.com/news/
// 6053916", section "weight block results with log-sum-exp": a softmax over the block
// LSEs weights the block outputs).  An empty split (LSE_i = -inf) has weight 0 and its
// O_i never enters the sum: it is not a zero-output block with a normal weight.  A row whose
// splits are all empty gets out = 0 and lse_out = -inf.
//
// Launched with programmatic dependent launch: the CTA waits (griddepcontrol.wait) for
// the partial pass's memory to be visible before it reads the workspace, and lets the
// next kernel of the stream start launching at once (that kernel waits in turn).
#include <cuda_bf16.h>

#include "fd_device.cuh"
#include "fd_epilogue.cuh"

namespace fd {

template <int D>
__global__ void __launch_bounds__(128) fd_combine_kernel(const __grid_constant__ Params p) {
  constexpr int VEC = D / 32;                  // dims per lane: 4 (d=128) or 2 (d=64)
  constexpr int BATCH = 8;                     // splits whose loads are in flight at once
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.6931471805599453f;
  __shared__ float wm[4], ww[4];
  __shared__ __align__(16) float accs[4][D];
  pdl_trigger();                               // the next step's partial pass may launch
  pdl_wait();

  const int row = blockIdx.x;                  // (b * Q + j) * Hq + h
  const int S = p.S;
  const float* lse = p.lse_part + (int64_t)row * S;
  const float* ob = p.o_part + (int64_t)row * S * D + (threadIdx.x & 31) * VEC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Warp w folds splits w, w + 4, w + 8, ... with a running maximum (base-2 units): a
  // batch's loads are all issued before any of them is used.
  float M = kNegInf, W = 0.f, acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  for (int s0 = warp; s0 < S; s0 += 4 * BATCH) {
    float ls[BATCH], v[BATCH][VEC];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int s = s0 + 4 * u;
      const bool in = s < S;
      ls[u] = in ? lse[s] * kLog2e : kNegInf;
      if constexpr (VEC == 4) {
        const float4 t = in ? *reinterpret_cast<const float4*>(ob + (int64_t)s * D)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
      } else {
        const float2 t = in ? *reinterpret_cast<const float2*>(ob + (int64_t)s * D)
                            : make_float2(0.f, 0.f);
        v[u][0] = t.x; v[u][1] = t.y;
      }
    }
    float mb = ls[0];
#pragma unroll
    for (int u = 1; u < BATCH; ++u) mb = fmaxf(mb, ls[u]);
    const float mn = fmaxf(M, mb);
    if (mn == kNegInf) continue;               // only empty splits so far
    const float c = (M == kNegInf) ? 0.f : ex2(M - mn);
    W *= c;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] *= c;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      // An empty split (LSE = -inf) has weight 0 and its O_i is selected away, never
      // multiplied: that memory was not written by this call.
      const bool live = ls[u] != kNegInf;
      const float w = live ? ex2(ls[u] - mn) : 0.f;
      W += w;
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, live ? v[u][e] : 0.f, acc[e]);
    }
    M = mn;
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) accs[warp][lane * VEC + e] = acc[e];
  if (lane == 0) {
    wm[warp] = M;
    ww[warp] = W;
  }
  __syncthreads();

  // Merge the four warps' states with the same rule.
  const float Mt = fmaxf(fmaxf(wm[0], wm[1]), fmaxf(wm[2], wm[3]));
  float cw[4], Wt = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    cw[w] = (wm[w] == kNegInf) ? 0.f : ex2(wm[w] - Mt);
    Wt = fmaf(ww[w], cw[w], Wt);
  }
  const int h = row % p.Hq, bj = row / p.Hq, b = bj / p.Q, qj = bj % p.Q;
  for (int j = tid; j < D; j += 128) {
    float o = 0.f;
    if (Wt > 0.f) {
      o = accs[0][j] * cw[0] + accs[1][j] * cw[1] + accs[2][j] * cw[2] + accs[3][j] * cw[3];
      o /= Wt;
    }
    const int64_t off = (int64_t)b * p.out_sb + (int64_t)qj * p.out_sj + (int64_t)h * p.out_sh + j;
    if (p.out_bf16) {
      reinterpret_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(o);
    } else {
      reinterpret_cast<float*>(p.out)[off] = o;
    }
  }
  if (tid == 0 && p.lse_out != nullptr) {
    float lg;
    asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(Wt));
    p.lse_out[row] = (Wt > 0.f) ? (Mt + lg) * kLn2 : kNegInf;
  }
}

// Many rows with few splits: one warp per row, kRowWarps rows per CTA (merge_row, the
// same fold with the splits of a row in one warp, all kRowSplits loads in flight at
// once).  A CTA of four warps per row spreads a row's splits but lives only as long as
// one row's loads; with thousands of rows (large batches, usually with few splits each)
// the launch of those short CTAs, not their memory traffic, set the pass's time.  With
// more splits per row the four warps' parallel loads win (1024 rows of 19 splits:
// 41.8 us a step with four warps per row, 42.5 with one).
constexpr int kRowWarps = 8;
constexpr int kRowSplits = 8;
constexpr int64_t kRowsPerWarpMin = 1024;   // rows from which the warp-per-row form runs

template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) fd_combine_rows_kernel(const __grid_constant__ Params p) {
  pdl_trigger();                               // the next step's partial pass may launch
  pdl_wait();
  const int64_t row = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (row >= (int64_t)p.B * p.Q * p.Hq) return;
  merge_row<D, kRowSplits>(p, row, threadIdx.x & 31);
}

cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool pdl) {
  const int64_t rows = (int64_t)p.B * p.Q * p.Hq;
  const bool by_rows = rows >= kRowsPerWarpMin && p.S <= kRowSplits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(by_rows ? (rows + kRowWarps - 1) / kRowWarps : rows));
  cfg.blockDim = dim3(by_rows ? kRowWarps * 32 : 128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (by_rows) {
    if (p.d == 128) return cudaLaunchKernelEx(&cfg, fd_combine_rows_kernel<128>, p);
    return cudaLaunchKernelEx(&cfg, fd_combine_rows_kernel<64>, p);
  }
  if (p.d == 128) return cudaLaunchKernelEx(&cfg, fd_combine_kernel<128>, p);
  return cudaLaunchKernelEx(&cfg, fd_combine_kernel<64>, p);
}

}  // namespace fd
