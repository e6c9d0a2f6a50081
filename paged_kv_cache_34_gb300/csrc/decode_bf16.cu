// decode_bf16.cu -- the paged decode over 16-bit pools, BF16 elements.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const DecodeArgs &a, const dec::DecodeParams &p, cudaStream_t s) {
  return dec::launch_family<BF16, 0>(a, p, s);
}

}  // namespace pa
