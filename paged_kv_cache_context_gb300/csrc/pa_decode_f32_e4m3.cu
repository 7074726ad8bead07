// Paged decode kernels: query/output float, cache pa::E4M3 (all head dims, group sizes
// and block sizes). One translation unit per dtype pair so they build in parallel.
#include "pa_decode.cuh"

cudaError_t pa_dispatch_decode_f32_e4m3(const pa::DecodeParams& prm, int num_seqs, int D, int GT,
                                  int BS, cudaStream_t stream) {
  return pa::dispatch_decode<float, pa::E4M3>(prm, num_seqs, D, GT, BS, stream);
}
