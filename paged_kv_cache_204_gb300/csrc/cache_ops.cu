// Cache maintenance kernels: slot-mapped write of new K/V rows and whole-block
// copies for copy-on-write ("PagedAttention: the KV cache was the bottleneck
// all along", section "Virtual memory for attention": sequences acquire
// blocks as they grow; shared blocks are copied when a sharer diverges).
// Both are byte moves in 16-byte vectors: results are bit-exact.
#include "cache_ops.h"
#include "common.cuh"

namespace pkv {

// grid = (new token, group of 128 chunks): each thread moves one 16-byte
// chunk of the token's K rows and of its V rows (all kv heads) to
// cache[slot / bs][h][slot % bs], so every load of the step is in flight at once.
__global__ void __launch_bounds__(128)
    reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                             const int64_t* __restrict__ slot_mapping, int num_kv_heads,
                             int row_chunks, int block_size, int64_t num_slots, int32_t* dev_err) {
  const int t = blockIdx.x;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_err(dev_err, PKV_DEV_ERR_SLOT);
    return;
  }
  const int n = num_kv_heads * row_chunks;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= n) return;
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot - blk * block_size);
  const int h = c / row_chunks;
  const int cc = c - h * row_chunks;
  const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row_chunks + cc;
  const uint4 kx = __ldg(k + (size_t)t * n + c);
  const uint4 vx = __ldg(v + (size_t)t * n + c);
  k_cache[dst] = kx;
  v_cache[dst] = vx;
}

// fp8 e4m3 cache write. grid = (new token, group of 128 eight-element runs):
// each thread reads 8 elements (16 bytes) of the token's K row and V row,
// divides them by k_scale / v_scale in fp32 (IEEE rounding) and stores the
// e4m3 codes (8 bytes) at cache[slot / bs][h][slot % bs].
template <typename T>
__global__ void __launch_bounds__(128)
    reshape_and_cache_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                                 const int64_t* __restrict__ slot_mapping, int num_kv_heads, int row_runs,
                                 int block_size, int64_t num_slots, float k_scale, float v_scale,
                                 int32_t* dev_err) {
  const int t = blockIdx.x;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_err(dev_err, PKV_DEV_ERR_SLOT);
    return;
  }
  const int n = num_kv_heads * row_runs;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= n) return;
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot - blk * block_size);
  const int h = c / row_runs;
  const int cc = c - h * row_runs;
  const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row_runs + cc;
  float fk[8], fv[8];
  Chunk<T>::widen(__ldg(k + (size_t)t * n + c), fk);
  Chunk<T>::widen(__ldg(v + (size_t)t * n + c), fv);
  uint32_t wk[4], wv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    wk[i] = narrow_e4m3x2(__fdiv_rn(fk[2 * i], k_scale), __fdiv_rn(fk[2 * i + 1], k_scale));
    wv[i] = narrow_e4m3x2(__fdiv_rn(fv[2 * i], v_scale), __fdiv_rn(fv[2 * i + 1], v_scale));
  }
  k_cache[dst] = make_uint2(wk[0] | (wk[1] << 16), wk[2] | (wk[3] << 16));
  v_cache[dst] = make_uint2(wv[0] | (wv[1] << 16), wv[2] | (wv[3] << 16));
}

// q4_0 cache write. grid = (new token, group of 4 kv heads), one warp per
// (token, kv head) row; the lanes of a 32-value block (8 at head_dim 128, 16
// at 64) hold values l, l + L, ... (L lanes per block), so lane l ends with
// code byte l (values l and l + 16) and, at head_dim 128, byte l + 8. Block
// rule, every step in binary32: m = the first value of largest magnitude
// (+0 if none is above 0), d = m / -8, inv = 1 / d (0 if d is 0), code =
// min(15, trunc(x inv + 8.5)) (0 below 0 or NaN); d is stored rounded to
// binary16.
template <typename T, int D>
__device__ __forceinline__ void quantize_row_q4(const T* __restrict__ src, unsigned char* __restrict__ dst,
                                                int lane) {
  constexpr int NBK = D / 32;
  constexpr int LPB = 32 / NBK;  // lanes per block
  constexpr int EPL = 32 / LPB;  // values per lane
  const int b = lane / LPB, l = lane % LPB;
  float x[EPL];
  float amax = 0.f, m = 0.f;
  int idx = 32;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    x[i] = to_float(src[32 * b + l + LPB * i]);
    const float a = fabsf(x[i]);
    if (a > amax) {
      amax = a;
      m = x[i];
      idx = l + LPB * i;
    }
  }
  // the block's first value of largest magnitude
#pragma unroll
  for (int o = 1; o < LPB; o <<= 1) {
    const float a2 = __shfl_xor_sync(0xffffffffu, amax, o);
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (a2 > amax || (a2 == amax && i2 < idx)) {
      amax = a2;
      m = m2;
      idx = i2;
    }
  }
  const float d = __fdiv_rn(m, -8.f);
  const float inv = d != 0.f ? __fdiv_rn(1.f, d) : 0.f;
  int q[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const float y = __fadd_rn(__fmul_rn(x[i], inv), 8.5f);
    q[i] = y >= 15.f ? 15 : (y >= 0.f ? static_cast<int>(y) : 0);
  }
  unsigned char* codes = dst + D / 16 + 16 * b;
  // values l (low bits) and l + 16 (high bits) make byte l
  if constexpr (LPB == 8) {
    codes[l] = static_cast<unsigned char>(q[0] | (q[2] << 4));
    codes[l + 8] = static_cast<unsigned char>(q[1] | (q[3] << 4));
  } else {
    codes[l] = static_cast<unsigned char>(q[0] | (q[1] << 4));
  }
  if (l == 0) *reinterpret_cast<unsigned short*>(dst + 2 * b) = __half_as_ushort(__float2half_rn(d));
}

template <typename T, int D>
__global__ void __launch_bounds__(128)
    reshape_and_cache_q4_kernel(const T* __restrict__ k, const T* __restrict__ v, unsigned char* __restrict__ k_cache,
                                unsigned char* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping,
                                int num_kv_heads, int block_size, int64_t num_slots, int32_t* dev_err) {
  const int t = blockIdx.x;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_err(dev_err, PKV_DEV_ERR_SLOT);
    return;
  }
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  if (h >= num_kv_heads) return;
  const int lane = threadIdx.x & 31;
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot - blk * block_size);
  constexpr int RB = D / 16 * 9;
  const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * RB;
  const size_t src = ((size_t)t * num_kv_heads + h) * D;
  quantize_row_q4<T, D>(k + src, k_cache + dst, lane);
  quantize_row_q4<T, D>(v + src, v_cache + dst, lane);
}

// grid = (pair, pool K|V, piece). Each piece streams part of one block with
// 4 independent 16-byte loads in flight per thread.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int64_t* __restrict__ pairs, int64_t block_chunks, int num_blocks,
                       int32_t* dev_err) {
  const int64_t src = __ldg(pairs + 2 * (size_t)blockIdx.x);
  const int64_t dst = __ldg(pairs + 2 * (size_t)blockIdx.x + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_err(dev_err, PKV_DEV_ERR_PAIR);
    return;
  }
  uint4* pool = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4* s = pool + (size_t)src * block_chunks;
  uint4* d = pool + (size_t)dst * block_chunks;
  const int64_t stride = (int64_t)gridDim.z * blockDim.x;
  int64_t c = (int64_t)blockIdx.z * blockDim.x + threadIdx.x;
  for (; c + 3 * stride < block_chunks; c += 4 * stride) {
    const uint4 a = s[c], b = s[c + stride], e = s[c + 2 * stride], f = s[c + 3 * stride];
    d[c] = a;
    d[c + stride] = b;
    d[c + 2 * stride] = e;
    d[c + 3 * stride] = f;
  }
  for (; c < block_chunks; c += stride) d[c] = s[c];
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                     int row_bytes, int block_size, int num_blocks, int32_t* dev_err,
                                     cudaStream_t stream) {
  const int n = num_kv_heads * (row_bytes / 16);
  const dim3 grid(num_tokens, (n + 127) / 128);
  reshape_and_cache_kernel<<<grid, 128, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, num_kv_heads, row_bytes / 16, block_size,
      (int64_t)num_blocks * block_size, dev_err);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                         int head_dim, int block_size, int num_blocks, int is_bf16, float k_scale,
                                         float v_scale, int32_t* dev_err, cudaStream_t stream) {
  const int runs = head_dim / 8;
  const int n = num_kv_heads * runs;
  const dim3 grid(num_tokens, (n + 127) / 128);
  const int64_t slots = (int64_t)num_blocks * block_size;
  if (is_bf16)
    reshape_and_cache_fp8_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint2*>(k_cache),
        static_cast<uint2*>(v_cache), slot_mapping, num_kv_heads, runs, block_size, slots, k_scale, v_scale, dev_err);
  else
    reshape_and_cache_fp8_kernel<__half><<<grid, 128, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint2*>(k_cache),
        static_cast<uint2*>(v_cache), slot_mapping, num_kv_heads, runs, block_size, slots, k_scale, v_scale, dev_err);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_q4(const void* k, const void* v, void* k_cache, void* v_cache,
                                        const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                        int head_dim, int block_size, int num_blocks, int is_bf16, int32_t* dev_err,
                                        cudaStream_t stream) {
  const dim3 grid(num_tokens, (num_kv_heads + 3) / 4);
  const int64_t slots = (int64_t)num_blocks * block_size;
  unsigned char* kc = static_cast<unsigned char*>(k_cache);
  unsigned char* vc = static_cast<unsigned char*>(v_cache);
#define PKV_Q4_LAUNCH(T, D)                                                                                    \
  reshape_and_cache_q4_kernel<T, D><<<grid, 128, 0, stream>>>(static_cast<const T*>(k), static_cast<const T*>(v), \
                                                             kc, vc, slot_mapping, num_kv_heads, block_size, slots, \
                                                             dev_err)
  if (is_bf16) {
    if (head_dim == 128) PKV_Q4_LAUNCH(__nv_bfloat16, 128);
    else PKV_Q4_LAUNCH(__nv_bfloat16, 64);
  } else {
    if (head_dim == 128) PKV_Q4_LAUNCH(__half, 128);
    else PKV_Q4_LAUNCH(__half, 64);
  }
#undef PKV_Q4_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                               int64_t block_bytes, int num_blocks, int32_t* dev_err, cudaStream_t stream) {
  const int64_t chunks = block_bytes / 16;
  int64_t pieces = (chunks + 256 * 4 - 1) / (256 * 4);
  if (pieces > 64) pieces = 64;
  dim3 grid(num_pairs, 2, static_cast<unsigned>(pieces));
  copy_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                               pairs, chunks, num_blocks, dev_err);
  return cudaGetLastError();
}

}  // namespace pkv
