// C ABI of the paged KV-cache library: argument checks, launch-shape choice
// and dispatch. Owns no memory, keeps no per-call state, never synchronises.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "cache_ops.h"
#include "decode.cuh"
#include "decode_grouped.cuh"
#include "pkv.h"
#include "prefill.cuh"

namespace {

std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool supported_head_dim(int d) { return d == 64 || d == 128; }
bool supported_block_size(int b) { return b == 8 || b == 16 || b == 32; }
bool valid_dtype(int t) { return t == PKV_F32 || t == PKV_F16 || t == PKV_BF16; }
bool valid_cache_dtype(int t) { return valid_dtype(t) || t == PKV_FP8_E4M3 || t == PKV_Q4_0; }
int elem_bytes(int t) { return t == PKV_F32 ? 4 : (t == PKV_FP8_E4M3 ? 1 : 2); }
// bytes of one cache row of head_dim values
int64_t cache_row_bytes(int t, int head_dim) {
  return t == PKV_Q4_0 ? (int64_t)head_dim / 16 * 9 : (int64_t)head_dim * elem_bytes(t);
}
bool valid_scale(float s) { return std::isfinite(s) && s > 0.f; }
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

// Grouped decode: the grouping flag, usable prefix per group and per
// sequence, piece counters, each row's prefix result, the row counters and
// tail results of the single-launch kernel, then the warps' partial slots.
struct GroupedLayout {
  size_t flag = 0, group_S = 0, group_units = 0, seq_P = 0, seg_ctr = 0, row_ml = 0, row_o = 0;
  size_t row_ctr = 0, tail_ml = 0, tail_o = 0;
  size_t slot_ml = 0, slot_o = 0, total = 0;
};

GroupedLayout grouped_layout(int num_seqs, int num_heads, int head_dim, int num_groups) {
  GroupedLayout w;
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || num_groups <= 0) return w;
  const size_t rows = (size_t)num_seqs * num_heads;
  const size_t slots = (size_t)pkv::kMaxDecodeWarps * 2 * pkv::kMaxPrefixRows;
  size_t off = 0;
  w.flag = off;  // flag word (1 = grouping rejected)
  off += 256;
  w.group_S = off;
  off += align_up((size_t)num_groups * 4, 256);
  w.group_units = off;
  off += align_up((size_t)num_groups * 8, 256);
  w.seq_P = off;
  off += align_up((size_t)num_seqs * 4, 256);
  w.seg_ctr = off;
  off += align_up(2 * rows * 4, 256);
  w.row_ml = off;
  off += align_up(rows * sizeof(float2), 256);
  w.row_o = off;
  off += align_up(rows * head_dim * sizeof(float), 256);
  w.row_ctr = off;
  off += align_up(rows * 4, 256);
  w.tail_ml = off;
  off += align_up(rows * sizeof(float2), 256);
  w.tail_o = off;
  off += align_up(rows * head_dim * sizeof(float), 256);
  w.slot_ml = off;
  off += align_up(slots * sizeof(float2), 256);
  w.slot_o = off;
  off += slots * head_dim * sizeof(float);
  w.total = off;
  return w;
}

pkv_status launch_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// Host checks shared by the decode entry points (nothing is enqueued).
pkv_status check_decode_args(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens, float scale,
                             int num_heads, int num_kv_heads, int head_dim, int block_size, int num_seqs,
                             int max_blocks_per_seq, int num_blocks, int max_context_len, pkv_dtype dtype,
                             int32_t* dev_err) {
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
  return PKV_OK;
}

pkv::DecodeParams decode_params(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens, float scale,
                                int num_heads, int num_kv_heads, int block_size, int num_seqs,
                                int max_blocks_per_seq, int num_blocks, int max_context_len, int gpw,
                                int32_t* dev_err) {
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
  p.group = num_heads / num_kv_heads;
  p.head_groups = num_heads / gpw;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.max_context_len = max_context_len;
  p.dev_err = dev_err;
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.v_scale = 1.f;
  return p;
}

// Query heads one warp serves against one kv head: the largest of 4, 2, 1
// that divides the group.
int heads_per_warp(int group) { return group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1); }

}  // namespace

extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
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
  if (!valid_cache_dtype(dtype) || !supported_head_dim(head_dim) || !supported_block_size(block_size))
    return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 8) ||
      (dev_err && !aligned(dev_err, 4)))
    return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes = (int64_t)num_kv_heads * block_size * cache_row_bytes(dtype, head_dim);
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
  const pkv_status st = check_decode_args(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                          num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                          max_blocks_per_seq, num_blocks, max_context_len, dtype, dev_err);
  if (st != PKV_OK || num_seqs == 0) return st;
  const WorkspaceLayout ws = workspace_layout(num_seqs, num_heads, head_dim);
  if (!workspace || workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;

  const int gpw = heads_per_warp(num_heads / num_kv_heads);
  const int gpw_index = gpw == 4 ? 2 : (gpw == 2 ? 1 : 0);
  pkv::DecodeLauncher launch = dtype == PKV_F32   ? pkv::decode_launcher_f32(head_dim, gpw_index)
                               : dtype == PKV_F16 ? pkv::decode_launcher_f16(head_dim, gpw_index)
                                                  : pkv::decode_launcher_bf16(head_dim, gpw_index);
  if (!launch) return PKV_ERR_UNSUPPORTED;
  pkv::DecodeParams p = decode_params(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                      num_heads, num_kv_heads, block_size, num_seqs, max_blocks_per_seq,
                                      num_blocks, max_context_len, gpw, dev_err);
  char* wsb = static_cast<char*>(workspace);
  p.ws_counter = reinterpret_cast<int32_t*>(wsb + ws.counter_off);
  p.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  p.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  return launch_status(launch(p, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                     int head_dim, int block_size, int num_blocks, pkv_dtype src_dtype,
                                     float k_scale, float v_scale, int32_t* dev_err, pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
      !valid_scale(k_scale) || !valid_scale(v_scale))
    return PKV_ERR_INVALID_ARG;
  if ((src_dtype != PKV_F16 && src_dtype != PKV_BF16) || !supported_head_dim(head_dim) ||
      !supported_block_size(block_size))
    return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8) || (dev_err && !aligned(dev_err, 4)))
    return PKV_ERR_INVALID_ARG;
  return launch_status(pkv::launch_reshape_and_cache_fp8(
      k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, num_blocks,
      src_dtype == PKV_BF16 ? 1 : 0, k_scale, v_scale, dev_err, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_attention_decode_fp8(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* context_lens, float scale, float k_scale,
                                          float v_scale, int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_seqs, int max_blocks_per_seq,
                                          int num_blocks, int max_context_len, pkv_dtype dtype,
                                          void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                          pkv_stream_t stream) {
  if (!valid_scale(k_scale) || !valid_scale(v_scale)) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16 && valid_dtype(dtype)) return PKV_ERR_UNSUPPORTED;
  const pkv_status st = check_decode_args(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                          num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                          max_blocks_per_seq, num_blocks, max_context_len, dtype, dev_err);
  if (st != PKV_OK || num_seqs == 0) return st;
  const WorkspaceLayout ws = workspace_layout(num_seqs, num_heads, head_dim);
  if (!workspace || workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;
  const int gpw = heads_per_warp(num_heads / num_kv_heads);
  const int gpw_index = gpw == 4 ? 2 : (gpw == 2 ? 1 : 0);
  pkv::DecodeLauncher launch = pkv::decode_launcher_fp8(dtype == PKV_BF16 ? 1 : 0, head_dim, gpw_index);
  if (!launch) return PKV_ERR_UNSUPPORTED;
  pkv::DecodeParams p = decode_params(out, q, k_cache, v_cache, block_tables, context_lens, scale * k_scale,
                                      num_heads, num_kv_heads, block_size, num_seqs, max_blocks_per_seq,
                                      num_blocks, max_context_len, gpw, dev_err);
  p.v_scale = v_scale;
  char* wsb = static_cast<char*>(workspace);
  p.ws_counter = reinterpret_cast<int32_t*>(wsb + ws.counter_off);
  p.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  p.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  return launch_status(launch(p, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_reshape_and_cache_q4_0(const void* k, const void* v, void* k_cache, void* v_cache,
                                      const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks, pkv_dtype src_dtype,
                                      int32_t* dev_err, pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if ((src_dtype != PKV_F16 && src_dtype != PKV_BF16) || !supported_head_dim(head_dim) ||
      !supported_block_size(block_size))
    return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (num_kv_heads > 4 * 65535) return PKV_ERR_UNSUPPORTED;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8) || (dev_err && !aligned(dev_err, 4)))
    return PKV_ERR_INVALID_ARG;
  return launch_status(pkv::launch_reshape_and_cache_q4(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                                        num_kv_heads, head_dim, block_size, num_blocks,
                                                        src_dtype == PKV_BF16 ? 1 : 0, dev_err,
                                                        reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_attention_decode_q4_0(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* context_lens, float scale, int num_heads,
                                           int num_kv_heads, int head_dim, int block_size, int num_seqs,
                                           int max_blocks_per_seq, int num_blocks, int max_context_len,
                                           pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                           int32_t* dev_err, pkv_stream_t stream) {
  if (dtype != PKV_F16 && dtype != PKV_BF16 && valid_dtype(dtype)) return PKV_ERR_UNSUPPORTED;
  const pkv_status st = check_decode_args(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                          num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                          max_blocks_per_seq, num_blocks, max_context_len, dtype, dev_err);
  if (st != PKV_OK || num_seqs == 0) return st;
  const WorkspaceLayout ws = workspace_layout(num_seqs, num_heads, head_dim);
  if (!workspace || workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;
  pkv::DecodeLauncher launch = pkv::decode_launcher_q4(dtype == PKV_BF16 ? 1 : 0, head_dim);
  if (!launch) return PKV_ERR_UNSUPPORTED;
  // one query head per warp, whatever the grouping of query heads
  pkv::DecodeParams p = decode_params(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_heads,
                                      num_kv_heads, block_size, num_seqs, max_blocks_per_seq, num_blocks,
                                      max_context_len, 1, dev_err);
  char* wsb = static_cast<char*>(workspace);
  p.ws_counter = reinterpret_cast<int32_t*>(wsb + ws.counter_off);
  p.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  p.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  return launch_status(launch(p, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_attention_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       const int32_t* query_start, float scale, int num_heads,
                                       int num_kv_heads, int head_dim, int block_size, int num_seqs,
                                       int max_blocks_per_seq, int num_blocks, int max_query_len,
                                       pkv_dtype dtype, int32_t* dev_err, pkv_stream_t stream) {
  if (max_query_len < 0) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F16 && dtype != PKV_BF16 && valid_dtype(dtype)) return PKV_ERR_UNSUPPORTED;
  const pkv_status st = check_decode_args(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                          num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                          max_blocks_per_seq, num_blocks, 0, dtype, dev_err);
  if (st != PKV_OK || num_seqs == 0 || max_query_len == 0) return st;
  if (!query_start || !aligned(query_start, 4)) return PKV_ERR_INVALID_ARG;
  if (num_heads > 65535) return PKV_ERR_UNSUPPORTED;
  pkv::PrefillLauncher launch = pkv::prefill_launcher(dtype == PKV_BF16 ? 1 : 0, head_dim);
  if (!launch) return PKV_ERR_UNSUPPORTED;
  pkv::PrefillParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.dev_err = dev_err;
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  return launch_status(launch(p, max_query_len, reinterpret_cast<cudaStream_t>(stream)));
}

size_t pkv_decode_grouped_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                          int num_groups) {
  if (max_context_len < 0) return 0;
  return grouped_layout(num_seqs, num_heads, head_dim, num_groups).total;
}

pkv_status pkv_paged_attention_decode_grouped(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, float scale, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              int num_seqs, int max_blocks_per_seq, int num_blocks,
                                              int max_context_len, const int32_t* group_start,
                                              const int32_t* shared_blocks, int num_groups,
                                              pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                              int32_t* dev_err, pkv_stream_t stream) {
  const pkv_status st = check_decode_args(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                          num_heads, num_kv_heads, head_dim, block_size, num_seqs,
                                          max_blocks_per_seq, num_blocks, max_context_len, dtype, dev_err);
  if (st != PKV_OK || num_seqs == 0) return st;
  if (num_groups < 1 || !group_start || !shared_blocks || !aligned(group_start, 4) ||
      !aligned(shared_blocks, 4))
    return PKV_ERR_INVALID_ARG;
  const GroupedLayout ws = grouped_layout(num_seqs, num_heads, head_dim, num_groups);
  if (!workspace || workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;
  // 16-bit pools are read by TMA as rows of head_dim elements: the row index
  // (one past the pool included) must fit in int32
  if (dtype != PKV_F32 && (int64_t)num_blocks * num_kv_heads * block_size + 16 > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;

  const int gpw = heads_per_warp(num_heads / num_kv_heads);
  const int gpw_index = gpw == 4 ? 2 : (gpw == 2 ? 1 : 0);
  pkv::GroupedLauncher launch = dtype == PKV_F32   ? pkv::grouped_launcher_f32(head_dim, gpw_index)
                                : dtype == PKV_F16 ? pkv::grouped_launcher_f16(head_dim, gpw_index)
                                                   : pkv::grouped_launcher_bf16(head_dim, gpw_index);
  if (!launch) return PKV_ERR_UNSUPPORTED;
  pkv::GroupedParams gp{};
  gp.base = decode_params(out, q, k_cache, v_cache, block_tables, context_lens, scale, num_heads,
                          num_kv_heads, block_size, num_seqs, max_blocks_per_seq, num_blocks,
                          max_context_len, gpw, dev_err);
  char* wsb = static_cast<char*>(workspace);
  gp.base.ws_ml = reinterpret_cast<float2*>(wsb + ws.slot_ml);
  gp.base.ws_o = reinterpret_cast<float*>(wsb + ws.slot_o);
  gp.group_start = group_start;
  gp.shared_blocks = shared_blocks;
  gp.num_groups = num_groups;
  gp.ws_flag = reinterpret_cast<int32_t*>(wsb + ws.flag);
  gp.ws_group_S = reinterpret_cast<int32_t*>(wsb + ws.group_S);
  gp.ws_group_units = reinterpret_cast<long long*>(wsb + ws.group_units);
  gp.ws_seq_P = reinterpret_cast<int32_t*>(wsb + ws.seq_P);
  gp.ws_seg_ctr = reinterpret_cast<int32_t*>(wsb + ws.seg_ctr);
  gp.ws_row_ml = reinterpret_cast<float2*>(wsb + ws.row_ml);
  gp.ws_row_o = reinterpret_cast<float*>(wsb + ws.row_o);
  gp.ws_row_ctr = reinterpret_cast<int32_t*>(wsb + ws.row_ctr);
  gp.ws_tail_ml = reinterpret_cast<float2*>(wsb + ws.tail_ml);
  gp.ws_tail_o = reinterpret_cast<float*>(wsb + ws.tail_o);
  return launch_status(launch(gp, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
