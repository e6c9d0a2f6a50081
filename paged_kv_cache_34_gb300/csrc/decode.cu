// decode.cu -- launcher of the paged decode (the kernels are in
// decode_kernel.cuh, instantiated per element type and pool format in
// decode_f16.cu, decode_bf16.cu, decode_int8.cu and decode_fp8.cu).
#include "decode_kernel.cuh"

namespace pa {

// Largest dynamic shared memory the decode kernel needs for this shape, so
// the host can reject shapes that cannot launch.
size_t decode_smem_bytes(int head_dim, int num_seqs, int partition_size, int block_size,
                         bool kv_int8) {
  const int max_ids = (partition_size > 0 ? partition_size : kDecodeChunkCap) / block_size + 2;
  if (kv_int8)
    return head_dim == 128 ? dec::DecodeSmem<128, true>::bytes(num_seqs, max_ids)
                           : dec::DecodeSmem<64, true>::bytes(num_seqs, max_ids);
  return head_dim == 128 ? dec::DecodeSmem<128>::bytes(num_seqs, max_ids)
                         : dec::DecodeSmem<64>::bytes(num_seqs, max_ids);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
  dec::DecodeParams p;
  p.out = a.out;
  p.out_row_stride = a.out_row_stride;
  p.q = a.query;
  p.q_row_stride = a.q_row_stride;
  p.block_table = a.block_table;
  p.bt_stride = a.block_table_stride;
  p.context_lens = a.context_lens;
  p.capacity = a.capacity;
  p.max_ctx = a.max_context_len;
  p.num_seqs = a.num_seqs;
  p.hq = a.num_q_heads;
  p.hkv = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.nc = a.slices.nc;
  p.hs = a.slices.hs;
  p.vh = a.num_kv_heads * a.slices.nc;
  p.box_rows = a.box_rows;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  p.partition_size = a.partition_size;
  p.num_partitions = a.num_partitions;
  p.balanced = a.partition_size == 0;
  p.chunk_cap = kDecodeChunkCap;
  p.num_workers = a.grid * dec::kWorkers;
  p.max_ids = (p.balanced ? kDecodeChunkCap : a.partition_size) / a.block_size + 2;
  p.ws_o = a.ws_o;
  p.ws_ml = a.ws_ml;
  p.ws_pref = a.ws_pref;
  p.nw = a.num_new;
  p.after_write = a.after_write ? 1 : 0;
  p.new_k = a.new_k;
  p.new_v = a.new_v;
  p.new_stride = a.new_stride;
  p.slot_mapping = a.slot_mapping;
  p.k_pool = a.k_pool;
  p.v_pool = a.v_pool;
  p.num_slots = a.num_blocks * a.block_size;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.err = a.d_error;
  p.wait_ns = a.wait_ns;
  if (a.head_dim != 64 && a.head_dim != 128) return cudaErrorInvalidValue;
  const bool bf = a.dtype == PA_BF16;
  if (a.kv_int8 && a.kv_fp8)
    return bf ? launch_decode_bf16_fp8(a, p, stream) : launch_decode_f16_fp8(a, p, stream);
  if (a.kv_int8)
    return bf ? launch_decode_bf16_int8(a, p, stream) : launch_decode_f16_int8(a, p, stream);
  return bf ? launch_decode_bf16(a, p, stream) : launch_decode_f16(a, p, stream);
}

}  // namespace pa
