/*
 * c_abi_decode.c -- decode attention through libfd's C ABI alone: no Python, no torch.
 *
 * A plain C99 program that includes fd.h, allocates device buffers with the CUDA runtime,
 * runs one decode step three ways -- fd_decode_attention, fd_decode_attention_ex with
 * per-call options (the mma.sync path) and a plan (fd_plan_create / fd_plan_decode) --
 * asks fd_partial_kernel_name_for which kernel two calls would run,
 * and checks every output element against the fp64 oracle (oracle/fd_oracle.c, test
 * infrastructure, linked into this test only) with the parity tolerances of the Python
 * tests:  out |got - ref| <= 4e-3 + 8e-3 |ref|,  lse |got - ref| <= 1e-4 + 1e-5 |ref|.
 *
 * Workload: B = 2 rows, Hq = 16, Hkv = 2 (GQA, G = 8), d = 128, contiguous bf16 cache of
 * 3000 tokens, lengths {3000, 777}; q, K, V drawn from a seeded generator (below) and
 * rounded to bf16 once, so the kernels and the oracle read the same stored values.
 *
 * Exit status 0 and "c abi ok" on success; 1 with a message otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "fd.h"

/* The fp64 oracle (oracle/fd_oracle.c).  dtype 1 = bf16 bit patterns. */
int fd_oracle_decode(int B, int Hq, int Hkv, int d, int dtype, const void* q, const void* k,
                     const void* v, const int32_t* seq_lens, int64_t L_cap,
                     const int32_t* block_table, int max_pages, int page_size,
                     int64_t num_pages, const int64_t* rows, int64_t n_rows, double* out,
                     double* lse, int num_threads);

enum { B = 2, HQ = 16, HKV = 2, D = 128, LCAP = 3000 };

/* Test input generator: a 64-bit linear congruential stream, two uniforms per normal
 * (Box-Muller), then float -> bf16 bits by round-to-nearest-even. */
static uint64_t g_state = 0x5eed1234abcdULL;
static double uniform01(void) {
  g_state = g_state * 6364136223846793005ULL + 1442695040888963407ULL;
  return ((double)(g_state >> 11) + 0.5) / 9007199254740992.0;
}
static float normal(void) {
  const double u = uniform01(), v = uniform01();
  return (float)(sqrt(-2.0 * log(u)) * cos(6.283185307179586 * v));
}
static uint16_t to_bf16(float x) {
  uint32_t bits;
  memcpy(&bits, &x, sizeof bits);
  bits += 0x7fffu + ((bits >> 16) & 1u);
  return (uint16_t)(bits >> 16);
}

static int fail_cuda(const char* what, cudaError_t e) {
  fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
  return 1;
}

static fd_tensor desc(void* data, int32_t dtype, int ndim, const int64_t* shape) {
  fd_tensor t;
  int64_t acc = 1;
  int i;
  memset(&t, 0, sizeof t);
  t.data = data;
  t.dtype = dtype;
  t.ndim = ndim;
  for (i = ndim - 1; i >= 0; --i) {
    t.shape[i] = shape[i];
    t.stride[i] = acc;
    acc *= shape[i];
  }
  return t;
}

/* Compare a device result with the oracle; returns the number of violations. */
static int check(const char* name, const float* out, const float* lse, const double* ref_o,
                 const double* ref_l) {
  int bad = 0, i;
  for (i = 0; i < B * HQ * D; ++i) {
    const double err = fabs((double)out[i] - ref_o[i]);
    if (!(err <= 4e-3 + 8e-3 * fabs(ref_o[i]))) {
      if (bad < 5) fprintf(stderr, "%s: out[%d] = %g, oracle %g\n", name, i, out[i], ref_o[i]);
      ++bad;
    }
  }
  for (i = 0; i < B * HQ; ++i) {
    const double err = fabs((double)lse[i] - ref_l[i]);
    if (!(err <= 1e-4 + 1e-5 * fabs(ref_l[i]))) {
      if (bad < 5) fprintf(stderr, "%s: lse[%d] = %g, oracle %g\n", name, i, lse[i], ref_l[i]);
      ++bad;
    }
  }
  return bad;
}

int main(void) {
  const int64_t nq = (int64_t)B * HQ * D, nkv = (int64_t)B * HKV * LCAP * D;
  const int32_t lens[B] = {3000, 777};
  const int64_t q_shape[3] = {B, HQ, D}, kv_shape[4] = {B, HKV, LCAP, D};
  uint16_t *hq = malloc(nq * 2), *hk = malloc(nkv * 2), *hv = malloc(nkv * 2);
  float *out_h = malloc(nq * 4), *lse_h = malloc(B * HQ * 4);
  double *ref_o = malloc(nq * 8), *ref_l = malloc(B * HQ * 8);
  void *dq, *dk, *dv, *dlens, *dout, *dlse, *dws;
  fd_tensor tq, tk, tv, tout;
  fd_options opts;
  fd_plan* plan = NULL;
  size_t ws_bytes;
  int32_t S;
  uint32_t flags = 0;
  int64_t i;
  int bad = 0, pass;
  cudaError_t e;
  fd_status st;

  if (!hq || !hk || !hv || !out_h || !lse_h || !ref_o || !ref_l) return 1;
  for (i = 0; i < nq; ++i) hq[i] = to_bf16(normal());
  for (i = 0; i < nkv; ++i) hk[i] = to_bf16(normal());
  for (i = 0; i < nkv; ++i) hv[i] = to_bf16(normal());

  if (fd_oracle_decode(B, HQ, HKV, D, 1, hq, hk, hv, lens, LCAP, NULL, 0, 0, 0, NULL, 0, ref_o,
                       ref_l, 0) != 0) {
    fprintf(stderr, "oracle refused the inputs\n");
    return 1;
  }

  S = fd_resolve_num_splits(B, HQ, HKV, D, LCAP, 0);
  ws_bytes = fd_workspace_size(B, HQ, HKV, D, S);
  if (ws_bytes == 0) return 1;
  if ((e = cudaMalloc(&dq, nq * 2)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
  if ((e = cudaMalloc(&dk, nkv * 2)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
  if ((e = cudaMalloc(&dv, nkv * 2)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
  if ((e = cudaMalloc(&dlens, sizeof lens)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
  if ((e = cudaMalloc(&dout, nq * 4)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
  if ((e = cudaMalloc(&dlse, B * HQ * 4)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
  if ((e = cudaMalloc(&dws, ws_bytes)) != cudaSuccess) return fail_cuda("cudaMalloc", e);
  cudaMemcpy(dq, hq, nq * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dk, hk, nkv * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dv, hv, nkv * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dlens, lens, sizeof lens, cudaMemcpyHostToDevice);
  if (fd_workspace_init(dws, ws_bytes, NULL) != FD_OK) return 1;

  tq = desc(dq, FD_BF16, 3, q_shape);
  tk = desc(dk, FD_BF16, 4, kv_shape);
  tv = desc(dv, FD_BF16, 4, kv_shape);
  tout = desc(dout, FD_F32, 3, q_shape);

  for (pass = 0; pass < 3; ++pass) {
    const char* name = pass == 0 ? "fd_decode_attention"
                       : pass == 1 ? "fd_decode_attention_ex" : "fd_plan_decode";
    cudaMemset(dout, 0xff, nq * 4);                 /* NaN: every element must be written */
    if (pass == 0) {
      st = fd_decode_attention(&tq, &tk, &tv, (const int32_t*)dlens, NULL, 0, 0, &tout,
                               (float*)dlse, dws, ws_bytes, NULL);
    } else if (pass == 1) {
      opts.path = FD_PATH_MMA;
      opts.merge_mode = FD_FROM_PROCESS;
      opts.schedule = FD_FROM_PROCESS;
      st = fd_decode_attention_ex(&tq, &tk, &tv, NULL, NULL, (const int32_t*)dlens, NULL, 0, 0,
                                  &tout, (float*)dlse, dws, ws_bytes, NULL, &opts);
    } else {
      st = fd_plan_create(&plan, B, HQ, HKV, D, LCAP, 0);
      if (st == FD_OK)
        st = fd_plan_decode(plan, &tq, &tk, &tv, (const int32_t*)dlens, NULL, 0, &tout,
                            (float*)dlse, NULL);
    }
    if (st != FD_OK) {
      fprintf(stderr, "%s: %s (%s)\n", name, fd_status_string(st), fd_last_error());
      return 1;
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail_cuda(name, e);
    cudaMemcpy(out_h, dout, nq * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(lse_h, dlse, B * HQ * 4, cudaMemcpyDeviceToHost);
    if (fd_read_device_error(pass == 2 ? fd_plan_workspace(plan) : dws, NULL, &flags) != FD_OK) {
      fprintf(stderr, "%s: device flags 0x%x\n", name, flags);
      return 1;
    }
    bad += check(name, out_h, lse_h, ref_o, ref_l);
  }
  {
    /* The kernel a call of these sizes runs: a 1-split call over 16-token pages takes head
     * groups even under the single-launch merge (one split never merges in-kernel). */
    fd_options inkernel;
    const char* k;
    inkernel.path = FD_FROM_PROCESS;
    inkernel.merge_mode = FD_MERGE_IN_KERNEL;
    inkernel.schedule = FD_FROM_PROCESS;
    k = fd_partial_kernel_name_for(&inkernel, FD_BF16, FD_BF16, B, 1, HQ, HKV, D, 0, LCAP, S, 1);
    if (!k || strcmp(k, "fd_partial_mma_kernel") != 0) {
      fprintf(stderr, "fd_partial_kernel_name_for: %s\n", k ? k : "(null)");
      return 1;
    }
    k = fd_partial_kernel_name_for(&inkernel, FD_BF16, FD_BF16, 4, 1, 32, 8, D, 16, 4096, 1, 1);
    if (!k || strcmp(k, "fd_partial_heads_kernel") != 0) {
      fprintf(stderr, "fd_partial_kernel_name_for (pages): %s\n", k ? k : "(null)");
      return 1;
    }
  }
  fd_plan_destroy(plan);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(dlens);
  cudaFree(dout);
  cudaFree(dlse);
  cudaFree(dws);
  if (bad) {
    fprintf(stderr, "%d elements outside the tolerance\n", bad);
    return 1;
  }
  printf("c abi ok: %s, 3 entry points x %d outputs match the fp64 oracle\n", fd_version(),
         B * HQ * (D + 1));
  return 0;
}
