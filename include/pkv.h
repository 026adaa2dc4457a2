/*
 * pkv.h — C ABI of the paged KV-cache decode library (GB300, sm_103a).
 *
 * The library implements the data-parallel hot path of PagedAttention
 * (Kwon et al., "Efficient Memory Management for Large Language Model Serving
 * with PagedAttention", SOSP 2023):
 *
 *   pkv_reshape_and_cache        write each step's new K/V rows into cache slots
 *   pkv_copy_blocks              copy whole physical blocks (copy-on-write)
 *   pkv_paged_attention_decode   single-token attention over a block-paged cache
 *
 * Sources for the semantics (page title, then section):
 *   [VM]  "PagedAttention: the KV cache was the bottleneck all along",
 *         section "Virtual memory for attention": the cache is cut into
 *         fixed-size blocks holding the keys and values of a fixed number of
 *         tokens; a sequence's blocks may sit anywhere in memory; a per-sequence
 *         block table translates logical block positions into physical blocks,
 *         the way a page table does; blocks are acquired as a sequence grows;
 *         the attention kernel reads K and V from those scattered blocks; sampled
 *         completions of one prompt share its blocks and copy a block only when
 *         they diverge (copy-on-write).
 *   [ABS] "Efficient Memory Management for Large Language Model Serving with
 *         PagedAttention", section "From the abstract": the attention algorithm
 *         is modelled on virtual memory and paging.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers to contiguous, row-major memory
 *    owned by the caller. The library allocates nothing, frees nothing, keeps
 *    no per-call state, never synchronises the stream and never reads device
 *    memory from the host. Work is enqueued on `stream` (a cudaStream_t; NULL
 *    means the legacy default stream).
 *  - Element type `dtype` is one of pkv_dtype. The kernels move 16-byte
 *    vectors: q, out, k, v, k_cache and v_cache must be 16-byte aligned.
 *  - Cache layout (one pool for K, one for V):
 *        cache[num_blocks][num_kv_heads][block_size][head_dim]
 *    so one (block, kv head) tile of block_size x head_dim elements is a
 *    contiguous run of memory. A cache slot is
 *        slot = physical_block * block_size + offset_in_block.
 *  - Supported: head_dim in {64, 128}, block_size in {8, 16, 32},
 *    num_heads % num_kv_heads == 0 (grouped-query heads h map to kv head
 *    h / (num_heads / num_kv_heads)).
 *  - Host-side checks run before anything is enqueued and return a
 *    pkv_status; nothing is launched when the status is not PKV_OK.
 *  - Device-side checks never trap. A kernel that meets a bad index skips (or
 *    clamps, see each entry point) the access and ORs a PKV_DEV_ERR_* bit into
 *    `*dev_err` when `dev_err` is not NULL. The caller reads that word after
 *    synchronising; a non-zero word means the outputs of that call are not
 *    valid.
 *  - Every wait inside a kernel is bounded (pkv_set_wait_timeout_ns); a wait
 *    that runs out sets PKV_DEV_ERR_TIMEOUT, lets its own copies land, and the
 *    kernel returns normally, leaving the CUDA context usable.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared here so that C callers need no CUDA
 * header to use this one. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum pkv_dtype {
  PKV_F32 = 0,      /* IEEE binary32 */
  PKV_F16 = 1,      /* IEEE binary16 */
  PKV_BF16 = 2,     /* bfloat16      */
  PKV_FP8_E4M3 = 3, /* 8-bit float, 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities,
                       largest finite 448 (OCP "E4M3"); cache element type only, see the fp8 entry points */
  PKV_Q4_0 = 4      /* 4-bit codes in blocks of 32 values with one binary16 scale (q4_0); cache type
                       only, rows of 9 * head_dim / 16 bytes, see the q4_0 entry points */
} pkv_dtype;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* NULL or misaligned pointer, negative or inconsistent size */
  PKV_ERR_UNSUPPORTED = 2, /* well-formed but not built: head_dim, block_size, dtype, grid limit */
  PKV_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than pkv_decode_workspace_bytes() */
  PKV_ERR_CUDA = 4,        /* a CUDA runtime call or a kernel launch failed */
  PKV_ERR_OUT_OF_BLOCKS = 5 /* host block manager: the free blocks cannot hold the request */
} pkv_status;

/* Bits ORed into *dev_err by the kernels. */
#define PKV_DEV_ERR_BLOCK_ID 0x1    /* block table entry outside [0, num_blocks) */
#define PKV_DEV_ERR_SLOT 0x2        /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEV_ERR_CONTEXT_LEN 0x4 /* context_lens entry < 0, > max_context_len or > max_blocks_per_seq * block_size */
#define PKV_DEV_ERR_TIMEOUT 0x8     /* a bounded wait inside a kernel ran out */
#define PKV_DEV_ERR_PAIR 0x10       /* copy_blocks pair entry outside [0, num_blocks) */
#define PKV_DEV_ERR_GROUP 0x20      /* grouped decode: grouping not a partition, or shared blocks differ */

/* Human-readable name of a pkv_status value (static string, never NULL). */
const char* pkv_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/*
 * Limit, in nanoseconds, of every bounded wait inside the kernels (default
 * 1e9 ns = 1 s). A value of 0 makes any wait that is not already satisfied on
 * its first test give up at once; it exists so that the timeout path can be
 * exercised. Process-wide; takes effect for launches enqueued after the call.
 */
void pkv_set_wait_timeout_ns(uint64_t ns);
uint64_t pkv_get_wait_timeout_ns(void);

/* -------------------------------------------------------------------------
 * pkv_reshape_and_cache
 *
 * Operation [VM]: a decoding step appends one K row and one V row per kv
 * head to each running sequence, into the cache slot of that token:
 *     for t in [0, num_tokens), h in [0, num_kv_heads):
 *         s = slot_mapping[t]; if s < 0: skip (padding token)
 *         k_cache[s / block_size][h][s % block_size][:] = k[t][h][:]
 *         v_cache[s / block_size][h][s % block_size][:] = v[t][h][:]
 * It is a pure byte copy: the result is bit-exact.
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim]   dtype, read
 *   k_cache,
 *   v_cache       [num_blocks][num_kv_heads][block_size][head_dim], written at the slots only
 *   slot_mapping  int64 [num_tokens]
 *   dev_err       optional int32 word (see PKV_DEV_ERR_*)
 *
 * Errors: host — INVALID_ARG for NULL/misaligned pointers or sizes < 0,
 * UNSUPPORTED for head_dim/block_size/dtype outside the supported sets.
 * Device — a slot >= num_blocks * block_size is skipped and sets
 * PKV_DEV_ERR_SLOT. Two tokens with the same slot race (undefined which wins).
 * num_tokens == 0 enqueues nothing.
 * ---------------------------------------------------------------------- */
pkv_status pkv_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                 int head_dim, int block_size, int num_blocks, pkv_dtype dtype,
                                 int32_t* dev_err, pkv_stream_t stream);

/* -------------------------------------------------------------------------
 * pkv_copy_blocks
 *
 * Operation [VM]: when sequences that share a block diverge, the writer gets
 * its own copy of that block first (copy-on-write). For every pair i:
 *     src = block_pairs[2*i], dst = block_pairs[2*i + 1]
 *     k_cache[dst][:][:][:] = k_cache[src][:][:][:]     (all kv heads)
 *     v_cache[dst][:][:][:] = v_cache[src][:][:][:]
 * A byte copy: bit-exact.
 *
 *   k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *   block_pairs       int64 [num_pairs][2] (device)
 *
 * Pairs are independent and may run in any order: a block that is the
 * destination of one pair must not be the source or destination of another
 * pair in the same call (undefined otherwise). Errors: host checks as for
 * pkv_reshape_and_cache; a pair with an entry outside [0, num_blocks) is
 * skipped and sets PKV_DEV_ERR_PAIR. num_pairs == 0 enqueues nothing.
 * ---------------------------------------------------------------------- */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_pairs, int num_pairs,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           pkv_dtype dtype, int32_t* dev_err, pkv_stream_t stream);

/* -------------------------------------------------------------------------
 * pkv_paged_attention_decode
 *
 * Operation [VM], [ABS]: softmax attention of one new query token per
 * sequence over the keys and values of that sequence's first context_lens[s]
 * tokens, which live in scattered physical blocks reached through the block
 * table. For sequence s, query head h, kv head g = h / (num_heads/num_kv_heads):
 *     token t (0 <= t < L = context_lens[s]) is stored in block
 *         p = block_tables[s][t / block_size], row t % block_size
 *     x_t   = scale * sum_d q[s][h][d] * k_cache[p][g][t % block_size][d]
 *     out[s][h][:] = sum_t softmax(x)_t * v_cache[p][g][t % block_size][:]
 * L == 0 gives an all-zero output row. Accumulation is fp32; the result is
 * rounded once to dtype.
 *
 *   out            [num_seqs][num_heads][head_dim]  dtype, written
 *   q              [num_seqs][num_heads][head_dim]  dtype
 *   k_cache,
 *   v_cache        [num_blocks][num_kv_heads][block_size][head_dim] dtype
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]; only the first
 *                  ceil(L / block_size) entries of row s are read
 *   context_lens   int32 [num_seqs]
 *   max_context_len  an upper bound of every context_lens entry, supplied by
 *                  the caller (it sizes the grid; the host never reads the
 *                  device array); must be <= max_blocks_per_seq * block_size
 *   workspace      device scratch of at least pkv_decode_workspace_bytes()
 *                  bytes (required whenever num_seqs > 0). Its first region
 *                  holds int32 counters that MUST be zero before the first call;
 *                  every call that ends with *dev_err == 0 leaves them zero
 *                  again. After a call that reports a device error, zero the
 *                  workspace again. Two calls that share a workspace must not
 *                  overlap on the GPU.
 *
 * Work split: the (sequence, head group) pairs are laid end to end as one
 * sequence of 16-token tiles and every warp of a device-sized, resident grid
 * takes an equal contiguous range of it. Pairs cut by range boundaries are
 * finished by a log-sum-exp merge of their pieces inside the same launch.
 *
 * Errors: host — INVALID_ARG (NULL/misaligned pointers, num_heads not a
 * multiple of num_kv_heads, max_context_len > max_blocks_per_seq*block_size,
 * negative sizes), UNSUPPORTED (head_dim, block_size, dtype, num_seqs > 65535),
 * WORKSPACE. Device — a block id outside [0, num_blocks) is read as block 0
 * and sets PKV_DEV_ERR_BLOCK_ID; a context length outside its bounds is
 * clamped and sets PKV_DEV_ERR_CONTEXT_LEN; a wait that runs out sets
 * PKV_DEV_ERR_TIMEOUT. num_seqs == 0 enqueues nothing.
 * ---------------------------------------------------------------------- */
pkv_status pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float scale, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size, int num_seqs,
                                      int max_blocks_per_seq, int num_blocks, int max_context_len,
                                      pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_err, pkv_stream_t stream);

/* -------------------------------------------------------------------------
 * pkv_paged_attention_decode_grouped
 *
 * Operation [VM]: the same result as pkv_paged_attention_decode, for batches
 * in which sampled completions (or beams) of one prompt share the prompt's
 * physical blocks. The caller groups such sequences:
 *     group g = sequences [group_start[g], group_start[g+1])
 *     the first shared_blocks[g] entries of their block-table rows are the
 *     same physical blocks
 * and the kernel then reads each shared K/V tile once for all members of the
 * group (up to 4 members per pass) instead of once per member, adding each
 * member's own tail afterwards with a log-sum-exp merge. Groups of one
 * sequence, or with shared_blocks 0, are plain sequences.
 *
 *   group_start    int32 [num_groups + 1] (device); must partition
 *                  [0, num_seqs): group_start[0] = 0, non-decreasing,
 *                  group_start[num_groups] = num_seqs
 *   shared_blocks  int32 [num_groups] (device)
 *   workspace      at least pkv_decode_grouped_workspace_bytes() bytes,
 *                  zeroed before the first call; left zeroed by every call
 *                  that ends with *dev_err == 0 (other rules as for
 *                  pkv_paged_attention_decode)
 *   other arguments as for pkv_paged_attention_decode.
 *
 * The grouping is checked on the device before use: if group_start is not a
 * partition the grouping is ignored, and a group whose members' block-table
 * entries differ inside the promised prefix uses only the part that matches;
 * both set PKV_DEV_ERR_GROUP and still give the plain result. The shared
 * prefix actually read once is cut to whole 16-token tiles, whole blocks and
 * the shortest member's context. Each call enqueues two kernels (the check,
 * then the attention). Host errors as for pkv_paged_attention_decode, plus
 * INVALID_ARG when num_groups < 1 or group_start / shared_blocks is NULL.
 * ---------------------------------------------------------------------- */
pkv_status pkv_paged_attention_decode_grouped(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, float scale, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              int num_seqs, int max_blocks_per_seq, int num_blocks,
                                              int max_context_len, const int32_t* group_start,
                                              const int32_t* shared_blocks, int num_groups,
                                              pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                              int32_t* dev_err, pkv_stream_t stream);

/* Bytes of workspace pkv_paged_attention_decode_grouped needs. Pure host
 * function; 0 for non-positive sizes. */
size_t pkv_decode_grouped_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                          int num_groups);

/* -------------------------------------------------------------------------
 * pkv_paged_attention_decode_noalloc
 *
 * No counterpart in the paper: this is a packaging variant, not part of the
 * method. Same operation, arguments, layouts and error reporting as
 * pkv_paged_attention_decode, minus the workspace: the scratch that holds
 * the partial results of long contexts is a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES bytes of device memory that the library itself
 * declares, so neither the library nor the caller allocates anything.
 *
 * It is meant for callers that cannot call cudaMalloc or any other device
 * allocator at the point where they run attention: for example a plugin
 * inside a host application that has already reserved all device memory for
 * its own allocator, or code with a fixed memory budget that must not grow
 * at run time, or a loop that cannot afford the latency and implicit
 * synchronisation of an allocation. Such callers cannot size and provide a
 * workspace; this entry point needs none.
 *
 * Limits and rules:
 *  - PKV_NOALLOC_SCRATCH_BYTES (32 MiB) is reserved on every device that
 *    loads the library, for the life of the process.
 *  - Sizes whose pkv_decode_workspace_bytes() exceeds that limit are rejected
 *    with PKV_ERR_WORKSPACE before anything is enqueued (the LLaMA-13B-shaped
 *    step, 128 sequences x 40 heads, needs 16.5 MB; the limit is reached near
 *    four million sequence x head pairs).
 *  - The first call on a device looks up the array's device address once for
 *    that device (with that device current); make that first call before any
 *    stream capture begins.
 *  - The address found then is kept for the life of the process. Do not use
 *    this entry point on a device after cudaDeviceReset() (or any other
 *    teardown of its primary context): the library's module is loaded again
 *    there and the array may move, so the kept address would be stale.
 *  - Every call on a device shares the same array and leaves its last
 *    contents in it. Each call first clears the segment counters it needs
 *    (an asynchronous memset on `stream`; this happens even when the call
 *    then fails its host-side checks, and touches only the library's own
 *    array). Two calls whose work overlaps on the GPU — different streams, or
 *    different host threads — race on the array and give wrong results:
 *    serialise them.
 * ---------------------------------------------------------------------- */
#define PKV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

pkv_status pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, float scale, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              int num_seqs, int max_blocks_per_seq, int num_blocks,
                                              int max_context_len, pkv_dtype dtype, int32_t* dev_err,
                                              pkv_stream_t stream);

/* ----------------------------------------------------------------------
 * fp8 KV cache
 *
 * [QKV] "Efficient Memory Management for Large Language Model Serving with
 * PagedAttention" (hackerpapers page), section "In the conversation": a
 * reader notes that quantising the KV cache cuts its memory footprint. The
 * format here is this library's choice: the two pools hold PKV_FP8_E4M3
 * codes (one byte per element, same [num_blocks][num_kv_heads][block_size]
 * [head_dim] layout, so a block is half the bytes of a 16-bit one) with one
 * scale per pool: element x is stored as e4m3(x / scale), the quotient taken
 * in binary32 with round-to-nearest-even, then rounded to the nearest e4m3
 * value (ties to even) and saturated to +-448; the value read back is
 * scale * code. Queries and outputs stay binary16 or bfloat16. Attention
 * over an fp8 cache computes exactly what pkv_paged_attention_decode
 * computes over the decoded values (in fp32, up to rounding order).
 * pkv_copy_blocks copies fp8 blocks when given dtype PKV_FP8_E4M3.
 * ---------------------------------------------------------------------- */

/* Write new K/V rows into fp8 caches ([QKV], [VM]): k, v [num_tokens]
 * [num_kv_heads][head_dim] of src_dtype (PKV_F16 or PKV_BF16, 16-byte
 * aligned); caches of PKV_FP8_E4M3 codes; slots as in pkv_reshape_and_cache.
 * k_scale, v_scale: finite and > 0 (PKV_ERR_INVALID_ARG otherwise). */
pkv_status pkv_reshape_and_cache_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                     int head_dim, int block_size, int num_blocks, pkv_dtype src_dtype,
                                     float k_scale, float v_scale, int32_t* dev_err, pkv_stream_t stream);

/* pkv_paged_attention_decode over fp8 caches ([QKV], [VM]): the same
 * arguments, layouts, workspace and error behaviour, with k_cache and v_cache
 * holding PKV_FP8_E4M3 codes and `dtype` (PKV_F16 or PKV_BF16) the type of q
 * and out. Logits are scale * (q . (k_scale * K_code)) and the output is the
 * softmax-weighted sum of v_scale * V_code. k_scale, v_scale: finite, > 0. */
pkv_status pkv_paged_attention_decode_fp8(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* context_lens, float scale, float k_scale,
                                          float v_scale, int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_seqs, int max_blocks_per_seq,
                                          int num_blocks, int max_context_len, pkv_dtype dtype,
                                          void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                          pkv_stream_t stream);

/* ----------------------------------------------------------------------
 * 4-bit (q4_0) KV cache
 *
 * [QKV], "In the conversation": a reader notes that 4-bit KV-cache
 * quantisation (the cache type q4_0) cuts the cache to about a quarter. The
 * pages name the format without defining it; this library reads it as the
 * q4_0 block of the ggml tensor library. Every 32 consecutive values of a
 * K or V row form a block with one binary16 scale d and a 4-bit code q per
 * value, read back as d * (q - 8). Quantising a block x[0..31], every step
 * in binary32:
 *     m    = the first value of largest magnitude, sign kept (+0 when no
 *            |x| is above 0; NaN values never qualify)
 *     d    = m / -8, inv = 1 / d (0 when d is 0)
 *     q_j  = 15 if y >= 15, trunc(y) if 0 <= y < 15, else 0 (NaN too),
 *            where y = x_j * inv + 8.5 (a product and a sum, each rounded)
 *     d is stored rounded to binary16 (nearest, ties to even; a block whose
 *     largest magnitude exceeds 8 * 65504 gets an infinite scale).
 * Pools hold bytes, [num_blocks][num_kv_heads][block_size][9 * head_dim / 16]:
 * each row is its head_dim / 32 scales (little-endian binary16), then 16
 * code bytes per block, byte j holding q_j in its low and q_(j+16) in its
 * high four bits. A 16-bit row of 2 * head_dim bytes takes 9 * head_dim / 16
 * (0.28 of the bytes). Queries and outputs stay binary16 or bfloat16.
 * pkv_copy_blocks copies q4_0 blocks when given dtype PKV_Q4_0.
 * ---------------------------------------------------------------------- */

/* Write new K/V rows into q4_0 caches ([QKV], [VM]): k, v [num_tokens]
 * [num_kv_heads][head_dim] of src_dtype (PKV_F16 or PKV_BF16, 16-byte
 * aligned), quantised as above into the slot's row; slots, skipped
 * padding tokens and errors as in pkv_reshape_and_cache. The result is
 * bit-exact: the same bytes as the rule above computed on any IEEE host. */
pkv_status pkv_reshape_and_cache_q4_0(const void* k, const void* v, void* k_cache, void* v_cache,
                                      const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks, pkv_dtype src_dtype,
                                      int32_t* dev_err, pkv_stream_t stream);

/* pkv_paged_attention_decode over q4_0 caches ([QKV], [VM]): the same
 * arguments, layouts, workspace and error behaviour, with k_cache and
 * v_cache holding q4_0 rows and `dtype` (PKV_F16 or PKV_BF16) the type of q
 * and out. Every K and V value is d * (q - 8) of its block: logits are
 * scale * (q . K) and the output is the softmax-weighted sum of V, with
 * fp32 accumulation (the codes enter tensor-core MMAs exactly, the scales
 * multiply fp32 partial sums). */
pkv_status pkv_paged_attention_decode_q4_0(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* context_lens, float scale, int num_heads,
                                           int num_kv_heads, int head_dim, int block_size, int num_seqs,
                                           int max_blocks_per_seq, int num_blocks, int max_context_len,
                                           pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                           int32_t* dev_err, pkv_stream_t stream);

/* ----------------------------------------------------------------------
 * Paged prefill
 *
 * [WL] "PagedAttention: the KV cache was the bottleneck all along", section
 * "What is left": the wish for shared blocks for common system prompts
 * across users, i.e. the prompt side running over the same paged cache. With
 * the host block manager, users fork a sequence holding the system prompt,
 * so the prompt's blocks are shared and its K/V is written once; each user's
 * own tokens are then written with pkv_reshape_and_cache and attended with
 * this call.
 * ---------------------------------------------------------------------- */

/* Causal attention of each sequence's newest tokens over its paged context
 * ([WL], [VM]). Sequence s holds context_lens[s] = L tokens in the cache,
 * its new ones included; its n = query_start[s+1] - query_start[s] queries
 * (0 <= n <= L) are its last n tokens, and query i (position L - n + i)
 * attends to tokens 0 .. L - n + i:
 *     out[query_start[s] + i][h] = softmax_t(scale * q . K_t) . V_t.
 * q, out: [query_start[num_seqs]][num_heads][head_dim], packed by sequence;
 * query_start: int32 [num_seqs + 1], non-decreasing, query_start[0] = 0;
 * max_query_len >= every n (it sizes the grid); caches, block tables and
 * context lengths as in pkv_paged_attention_decode. dtype: PKV_F16 or
 * PKV_BF16 (tensor-core path). No workspace. Host checks as in the decode
 * call, plus PKV_ERR_INVALID_ARG for a NULL query_start or max_query_len < 0.
 * Device: a sequence with n < 0, n > L or L out of range sets
 * PKV_DEV_ERR_CONTEXT_LEN and is skipped; a bad block id sets
 * PKV_DEV_ERR_BLOCK_ID (its rows read as zeros). */
pkv_status pkv_paged_attention_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       const int32_t* query_start, float scale, int num_heads,
                                       int num_kv_heads, int head_dim, int block_size, int num_seqs,
                                       int max_blocks_per_seq, int num_blocks, int max_query_len,
                                       pkv_dtype dtype, int32_t* dev_err, pkv_stream_t stream);

/* Bytes of workspace pkv_paged_attention_decode needs for these sizes: the
 * segment counters (num_seqs * num_heads int32) plus a fixed area for the
 * partial results of the split segments (independent of the context lengths;
 * about 16.3 MB for head_dim 128). Pure host function; returns 0 for
 * non-positive sizes. */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
