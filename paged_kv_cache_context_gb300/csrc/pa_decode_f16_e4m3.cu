// Paged decode kernels: query/output __half, cache pa::E4M3 (all head dims, group sizes,
// block sizes and both work modes). One translation unit per dtype pair so
// they build in parallel.
#include "pa_decode.cuh"

cudaError_t pa_dispatch_decode_f16_e4m3(const pa::DecodeParams& prm, dim3 grid, int D, int GT, int BS,
                                  int mode, int* ctas, cudaStream_t stream) {
  return pa::dispatch_decode<__half, pa::E4M3>(prm, grid, D, GT, BS, mode, ctas, stream);
}
