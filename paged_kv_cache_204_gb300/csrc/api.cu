// C ABI of the paged KV-cache library: argument checks, launch-shape choice
// and dispatch. Owns no memory, keeps no per-call state, never synchronises.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "cache_ops.h"
#include "decode.cuh"
#include "pkv.h"

namespace {

std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool supported_head_dim(int d) { return d == 64 || d == 128; }
bool supported_block_size(int b) { return b == 8 || b == 16 || b == 32; }
bool valid_dtype(int t) { return t == PKV_F32 || t == PKV_F16 || t == PKV_BF16; }
int elem_bytes(int t) { return t == PKV_F32 ? 4 : 2; }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WorkspaceLayout {
  size_t counter_off = 0, ml_off = 0, o_off = 0, total = 0;
};

// Counters of the (sequence, head group) segments, then the partial slots of
// the persistent warps (two per warp, up to kMaxGroupPerWarp heads each).
WorkspaceLayout workspace_layout(int num_seqs, int num_heads, int head_dim) {
  WorkspaceLayout w;
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0) return w;
  const size_t slots = (size_t)pkv::kMaxDecodeWarps * 2 * pkv::kMaxGroupPerWarp;
  w.counter_off = 0;
  w.ml_off = align_up((size_t)num_seqs * num_heads * sizeof(int32_t), 256);
  w.o_off = w.ml_off + align_up(slots * sizeof(float2), 256);
  w.total = w.o_off + slots * head_dim * sizeof(float);
  return w;
}

pkv_status launch_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace

extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    default: return "PKV_ERR_UNKNOWN";
  }
}

int pkv_version(void) { return 100; }

void pkv_set_wait_timeout_ns(uint64_t ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }
uint64_t pkv_get_wait_timeout_ns(void) { return g_wait_limit_ns.load(std::memory_order_relaxed); }

size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len) {
  if (max_context_len < 0) return 0;
  return workspace_layout(num_seqs, num_heads, head_dim).total;
}

pkv_status pkv_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                 int head_dim, int block_size, int num_blocks, pkv_dtype dtype,
                                 int32_t* dev_err, pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || !supported_head_dim(head_dim) || !supported_block_size(block_size))
    return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8) || (dev_err && !aligned(dev_err, 4)))
    return PKV_ERR_INVALID_ARG;
  return launch_status(pkv::launch_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                                     num_kv_heads, head_dim * elem_bytes(dtype),
                                                     block_size, num_blocks, dev_err,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_pairs, int num_pairs,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           pkv_dtype dtype, int32_t* dev_err, pkv_stream_t stream) {
  if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || !supported_head_dim(head_dim) || !supported_block_size(block_size))
    return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 8) ||
      (dev_err && !aligned(dev_err, 4)))
    return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes = (int64_t)num_kv_heads * block_size * head_dim * elem_bytes(dtype);
  return launch_status(pkv::launch_copy_blocks(k_cache, v_cache, block_pairs, num_pairs, block_bytes,
                                               num_blocks, dev_err, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float scale, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size, int num_seqs,
                                      int max_blocks_per_seq, int num_blocks, int max_context_len,
                                      pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_err, pkv_stream_t stream) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0 || num_blocks <= 0 || max_context_len < 0 || !std::isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size) return PKV_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || !supported_head_dim(head_dim) || !supported_block_size(block_size))
    return PKV_ERR_UNSUPPORTED;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || (dev_err && !aligned(dev_err, 4)))
    return PKV_ERR_INVALID_ARG;

  const WorkspaceLayout ws = workspace_layout(num_seqs, num_heads, head_dim);
  if (!workspace || workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;

  const int group = num_heads / num_kv_heads;
  const int gpw = group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1);
  const int gpw_index = gpw == 4 ? 2 : (gpw == 2 ? 1 : 0);
  pkv::DecodeLauncher launch = dtype == PKV_F32   ? pkv::decode_launcher_f32(head_dim, gpw_index)
                               : dtype == PKV_F16 ? pkv::decode_launcher_f16(head_dim, gpw_index)
                                                  : pkv::decode_launcher_bf16(head_dim, gpw_index);
  if (!launch) return PKV_ERR_UNSUPPORTED;

  pkv::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.head_groups = num_heads / gpw;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.max_context_len = max_context_len;
  char* wsb = static_cast<char*>(workspace);
  p.ws_counter = reinterpret_cast<int32_t*>(wsb + ws.counter_off);
  p.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  p.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  p.dev_err = dev_err;
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  return launch_status(launch(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
