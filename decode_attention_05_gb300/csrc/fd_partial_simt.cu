// fd_partial_simt.cu -- instantiations and launcher of the CUDA-core partial pass.
#include "fd_partial_simt.cuh"

namespace fd {

namespace {

template <class SH>
cudaError_t launch_simt(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                        cudaStream_t stream) {
  auto kernel = fd_partial_simt_kernel<SH>;
  static SmemOptIn opt_in;          // set once per device
  cudaError_t e = opt_in.apply(kernel, (int)SH::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.S, (unsigned)p.Hkv, (unsigned)p.B);
  e = launch_partial_kernel(kernel, grid, SH::THREADS, SH::SMEM_BYTES, stream, tk, tv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int ESZ, int D>
cudaError_t dispatch_g(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream) {
  switch (rows_template(p.n_rows)) {   // query rows per (b, kv head), padded
    case 1: return launch_simt<SimtShape<ESZ, D, 1>>(p, tk, tv, stream);
    case 2: return launch_simt<SimtShape<ESZ, D, 2>>(p, tk, tv, stream);
    case 4: return launch_simt<SimtShape<ESZ, D, 4>>(p, tk, tv, stream);
    case 8: return launch_simt<SimtShape<ESZ, D, 8>>(p, tk, tv, stream);
    case 16: return launch_simt<SimtShape<ESZ, D, 16>>(p, tk, tv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_partial_simt(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                int dtype, cudaStream_t stream) {
  const int esz = dtype == FD_BF16 ? 2 : 4;
  if (esz == 2 && p.d == 128) return dispatch_g<2, 128>(p, tk, tv, stream);
  if (esz == 2 && p.d == 64) return dispatch_g<2, 64>(p, tk, tv, stream);
  if (esz == 4 && p.d == 128) return dispatch_g<4, 128>(p, tk, tv, stream);
  if (esz == 4 && p.d == 64) return dispatch_g<4, 64>(p, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fd
