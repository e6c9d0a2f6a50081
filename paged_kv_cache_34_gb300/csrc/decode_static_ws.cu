// decode_static_ws.cu -- pa_decode for callers that cannot allocate device
// memory.
//
// pa_decode needs a device workspace for its split-KV partial results when
// a sequence spans several partitions, and expects the caller to provide it.
// Some callers have no way to do that: code running where cudaMalloc is not
// allowed or not wanted (inside a region that records work for later replay,
// a real-time loop with a fixed memory budget, a plug-in whose host framework
// owns every allocation, or a plain C caller with no device allocator).  For
// them, pa_decode_static_ws runs the same decode with its workspace in a
// fixed-size array that lives in the library's own device image.
//
// The array is declared at file scope below.  Its name is only a host-side
// stand-in for the device object, so the host never passes it to a kernel:
// the first call on each device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it.  That first
// call should come before any stream capture.  Every later call, from any
// thread, reuses the cached address.
//
// All calls on a device share the one array and leave their partial results
// in it.  Nothing in it needs to start at zero: each call writes every
// partial it later reads.  Calls that can overlap on the GPU (different
// streams without ordering between them) would corrupt each other's
// partials; order them on one stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = PA_STATIC_WORKSPACE_BYTES;

// The shared workspace.  Every GPU that loads the library holds it until the
// process exits.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_workspace_addr[kMaxDevices] = {nullptr};

// Device address of the array on the current device (looked up once per
// device).  Returns the CUDA error of the lookup, if any.
cudaError_t static_workspace(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_workspace_addr[dev]) {
    void *addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_static_workspace);
    if (e != cudaSuccess) return e;
    g_workspace_addr[dev] = addr;
  }
  *out = g_workspace_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

pa_status pa_decode_static_ws(void *out, int64_t out_row_stride, const void *query,
                              int64_t q_row_stride, const void *key_cache,
                              const void *value_cache, const int32_t *block_table,
                              int64_t block_table_stride, int32_t max_blocks_per_seq,
                              const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, float scale, int32_t max_context_len,
                              int32_t partition_size, pa_dtype dtype, int32_t *d_error,
                              void *stream) {
  // Pick a plan whose workspace fits the array.  An explicit partition size
  // that does not fit is an error.  When the automatic plan does not fit,
  // fixed partitions are used instead, grown (fewer partial results) until
  // they fit.  A partition at least as long as max_context_len needs no
  // workspace at all, but a long partition needs more shared memory for its
  // block ids: a shape that fits the array only with partitions the decode
  // kernel cannot hold is refused with PA_ERR_WORKSPACE.
  int32_t part = 0;
  size_t need = 0;
  pa_status st = pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                partition_size, &part, &need);
  if (st != PA_OK) return st;
  if (need > kStaticWorkspaceBytes) {
    if (partition_size != 0) return PA_ERR_WORKSPACE;
    int64_t p64 = 64;
    while (true) {
      if (block_size > 0 &&
          pa::decode_smem_bytes(head_dim, num_seqs, static_cast<int>(p64), block_size) >
              227 * 1024)
        return PA_ERR_WORKSPACE;
      st = pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                          static_cast<int32_t>(p64), &part, &need);
      if (st != PA_OK) return st;
      if (need <= kStaticWorkspaceBytes) break;
      if (p64 >= max_context_len) return PA_ERR_WORKSPACE;  // need is 0 there: unreachable
      p64 *= 2;
      if (p64 > max_context_len) p64 = (static_cast<int64_t>(max_context_len) + 15) / 16 * 16;
    }
  }
  void *ws = nullptr;
  if (need > 0) {
    const cudaError_t e = static_workspace(&ws);
    if (e != cudaSuccess) {
      pa::record_cuda_error(e);
      return PA_ERR_CUDA;
    }
  }
  return pa_decode(out, out_row_stride, query, q_row_stride, key_cache, value_cache, block_table,
                   block_table_stride, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, scale, max_context_len, part, ws,
                   need > 0 ? kStaticWorkspaceBytes : 0, dtype, d_error, stream);
}

}  // extern "C"
