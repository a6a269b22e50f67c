// fd_combine.cu -- the merge pass of split-KV decode: one CTA per (b, query head).
//
// Reads the S partials (O_i, LSE_i) of its row and computes
//   M = max over non-empty splits of LSE_i,   w_i = exp(LSE_i - M)  in (0, 1],
//   out = sum_i w_i O_i / sum_i w_i,          lse_out = M + log(sum_i w_i)
// ("FlashDecoding interview notes" (gtnt.cn/news/53829), section three, point 2: the
// weights use LSE_i - LSE_global <= 0, so no exponent can overflow; "2kiu.com/news/
// 6053916", section "weight block results with log-sum-exp": a softmax over the block
// LSEs weights the block outputs).  An empty split (LSE_i = -inf) has weight 0 and its
// O_i is never read: it is not a zero-output block with a normal weight.  A row whose
// splits are all empty gets out = 0 and lse_out = -inf.
//
// Launched with programmatic dependent launch: the CTA waits (griddepcontrol.wait) for
// the partial pass's memory to be visible before it reads the workspace.
#include <cuda_bf16.h>

#include "fd_device.cuh"

namespace fd {

template <int D>
__global__ void __launch_bounds__(128) fd_combine_kernel(const __grid_constant__ Params p) {
  constexpr int VEC = D / 32;                  // dims per lane: 4 (d=128) or 2 (d=64)
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.6931471805599453f;
  __shared__ float red[4];
  __shared__ float sw[4];
  __shared__ __align__(16) float accs[4][D];
  pdl_wait();

  const int row = blockIdx.x;                  // b * Hq + h
  const int S = p.S;
  const float* lse = p.lse_part + (int64_t)row * S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  float mx = kNegInf;
  for (int s = tid; s < S; s += 128) mx = fmaxf(mx, lse[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));

  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != kNegInf) {
    const float* ob = p.o_part + (int64_t)row * S * D + lane * VEC;
#pragma unroll 4
    for (int s = warp; s < S; s += 4) {
      const float ls = lse[s];
      if (ls == kNegInf) continue;             // empty split: weight 0, O_i never read
      const float w = ex2((ls - M) * kLog2e);
      wsum += w;
      if constexpr (VEC == 4) {
        const float4 o = *reinterpret_cast<const float4*>(ob + (int64_t)s * D);
        acc[0] = fmaf(w, o.x, acc[0]);
        acc[1] = fmaf(w, o.y, acc[1]);
        acc[2] = fmaf(w, o.z, acc[2]);
        acc[3] = fmaf(w, o.w, acc[3]);
      } else {
        const float2 o = *reinterpret_cast<const float2*>(ob + (int64_t)s * D);
        acc[0] = fmaf(w, o.x, acc[0]);
        acc[1] = fmaf(w, o.y, acc[1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) accs[warp][lane * VEC + e] = acc[e];
  if (lane == 0) sw[warp] = wsum;
  __syncthreads();

  const int b = row / p.Hq, h = row % p.Hq;
  const float W = sw[0] + sw[1] + sw[2] + sw[3];
  for (int j = tid; j < D; j += 128) {
    float o = 0.f;
    if (W > 0.f) o = (accs[0][j] + accs[1][j] + accs[2][j] + accs[3][j]) / W;
    const int64_t off = (int64_t)b * p.out_sb + (int64_t)h * p.out_sh + j;
    if (p.out_bf16) {
      reinterpret_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(o);
    } else {
      reinterpret_cast<float*>(p.out)[off] = o;
    }
  }
  if (tid == 0 && p.lse_out != nullptr) {
    float lg;
    asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(W));
    p.lse_out[row] = (W > 0.f) ? M + lg * kLn2 : kNegInf;
  }
}

cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.Hq));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.d == 128) return cudaLaunchKernelEx(&cfg, fd_combine_kernel<128>, p);
  return cudaLaunchKernelEx(&cfg, fd_combine_kernel<64>, p);
}

}  // namespace fd
