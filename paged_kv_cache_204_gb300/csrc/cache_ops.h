// Host launchers of the cache maintenance kernels (arguments already validated).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pkv {

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                     int row_bytes, int block_size, int num_blocks, int32_t* dev_err,
                                     cudaStream_t stream);

// fp8 e4m3 caches: 16-bit rows (is_bf16 selects bfloat16 over binary16) are
// divided by the scale and rounded to e4m3 on the way in.
cudaError_t launch_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                         int head_dim, int block_size, int num_blocks, int is_bf16, float k_scale,
                                         float v_scale, int32_t* dev_err, cudaStream_t stream);

// q4_0 caches: each 16-bit row (is_bf16 selects bfloat16 over binary16) is
// quantised on the way in, 32 values per block (one binary16 scale and 16
// code bytes; rows of 9 head_dim / 16 bytes).
cudaError_t launch_reshape_and_cache_q4(const void* k, const void* v, void* k_cache, void* v_cache,
                                        const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                        int head_dim, int block_size, int num_blocks, int is_bf16, int32_t* dev_err,
                                        cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                               int64_t block_bytes, int num_blocks, int32_t* dev_err, cudaStream_t stream);

}  // namespace pkv
