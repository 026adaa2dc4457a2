// Allocation-free variant of pkv_paged_attention_decode: the split-context
// scratch lives in a fixed-size array of this library's own device memory
// instead of a caller-provided workspace.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "pkv.h"

namespace {

// Scratch for the split-context partials of the no-allocation entry point.
// Every device that loads this library holds it until the process exits.
// Device code could name it directly; host code must not (on the host the
// name is only a stand-in, not a device address): it asks the runtime for the
// address on each device once, below.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_decode_scratch on the current device, looked up once
// per device (the first call on a device does the lookup).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, float scale, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int num_seqs, int max_blocks_per_seq, int num_blocks, int max_context_len,
    pkv_dtype dtype, int32_t* dev_err, pkv_stream_t stream) {
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len);
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  if (need == 0 || num_seqs <= 0)  // no partials to keep: nothing of the scratch is touched
    return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                      num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                      max_blocks_per_seq, num_blocks, max_context_len, dtype, nullptr,
                                      0, dev_err, stream);
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return PKV_ERR_CUDA;
  // The segment counters at the start of the scratch must be zero when the
  // kernel starts; a previous call that reported a device error may have left
  // some set, so clear them on the caller's stream (no allocation involved).
  const size_t counter_bytes = (size_t)num_seqs * num_heads * sizeof(int32_t);
  if (cudaMemsetAsync(scratch, 0, counter_bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                    num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                    max_blocks_per_seq, num_blocks, max_context_len, dtype, scratch,
                                    (size_t)PKV_NOALLOC_SCRATCH_BYTES, dev_err, stream);
}
