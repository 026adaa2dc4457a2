// Host launchers of the cache maintenance kernels (arguments already validated).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pkv {

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                     int row_bytes, int block_size, int num_blocks, int32_t* dev_err,
                                     cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                               int64_t block_bytes, int num_blocks, int32_t* dev_err, cudaStream_t stream);

}  // namespace pkv
