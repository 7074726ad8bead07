// Paged decode kernels: query/output __nv_bfloat16, cache pa::I8 (INT8 codes with one
// fp32 scale per cached row; all head dims, group sizes, block sizes and both
// work modes). One translation unit per dtype pair so they build in parallel.
#include "pa_decode.cuh"

cudaError_t pa_dispatch_decode_bf16_i8(const pa::DecodeParams& prm, dim3 grid, int D, int GT,
                                      int BS, int mode, int* ctas, cudaStream_t stream) {
  return pa::dispatch_decode<__nv_bfloat16, pa::I8>(prm, grid, D, GT, BS, mode, ctas, stream);
}
