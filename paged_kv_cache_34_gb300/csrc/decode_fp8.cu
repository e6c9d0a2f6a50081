// decode_fp8.cu -- the paged decode over one-byte pools of FP8-E4M3 codes with
// per-KV-head scales, for fp16 or bf16 queries and outputs.
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f16_fp8(const DecodeArgs &a, const dec::DecodeParams &p,
                                  cudaStream_t s) {
  return dec::launch_family<F16, 2>(a, p, s);
}
cudaError_t launch_decode_bf16_fp8(const DecodeArgs &a, const dec::DecodeParams &p,
                                   cudaStream_t s) {
  return dec::launch_family<BF16, 2>(a, p, s);
}

}  // namespace pa
