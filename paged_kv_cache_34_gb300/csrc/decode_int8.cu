// decode_int8.cu -- the paged decode over one-byte pools of INT8 codes with
// per-KV-head scales, for fp16 or bf16 queries and outputs.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f16_int8(const DecodeArgs &a, const dec::DecodeParams &p,
                                  cudaStream_t s) {
  return dec::launch_family<F16, 1>(a, p, s);
}
cudaError_t launch_decode_bf16_int8(const DecodeArgs &a, const dec::DecodeParams &p,
                                   cudaStream_t s) {
  return dec::launch_family<BF16, 1>(a, p, s);
}

}  // namespace pa
