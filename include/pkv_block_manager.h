/*
 * pkv_block_manager.h — host-side block manager of the paged KV cache.
 *
 * The bookkeeping that runs on the CPU right before each decode step: it
 * decides which physical cache block holds which token of which sequence,
 * and hands the attention kernels their block tables, context lengths, cache
 * slots for the new K/V rows and copy-on-write block pairs.
 *
 * Semantics (page title, then section):
 *   [VM]  "PagedAttention: the KV cache was the bottleneck all along",
 *         section "Virtual memory for attention": the cache is cut into
 *         fixed-size blocks; a sequence takes a new block only when it
 *         grows past its last one, so the only waste is the unfilled tail of
 *         its final block; a block table maps logical block positions to
 *         physical blocks; samples of one prompt (and beams) share blocks and
 *         copy a block only when one of them writes into it while others
 *         still use it (copy-on-write); sharing saves memory.
 *   [NUM] same page, section "The number that made us read the code":
 *         reserving one contiguous region of the maximum length per
 *         sequence wastes most of the cache; this manager never reserves.
 *
 * Conventions
 * -----------
 *  - Plain host code: every pointer argument is HOST memory owned by the
 *    caller; no CUDA call is made and no GPU is needed. A manager is not
 *    thread-safe: one thread at a time per manager.
 *  - Sequence ids are small non-negative integers. The id of a freed
 *    sequence is handed out again by a later pkv_bm_add_seq / pkv_bm_fork.
 *  - Physical blocks are ids in [0, num_blocks). Free blocks are handed out
 *    from a stack whose initial order is a seeded permutation (seed 0:
 *    ascending ids), and a freed block goes back on top of it.
 *  - Every call returns PKV_OK or an error status and changes nothing when it
 *    fails: PKV_ERR_INVALID_ARG for a NULL manager or output pointer, a
 *    negative count or an id that is not a live sequence;
 *    PKV_ERR_OUT_OF_BLOCKS when the free blocks cannot hold the request.
 */
#ifndef PKV_BLOCK_MANAGER_H_
#define PKV_BLOCK_MANAGER_H_

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* Counters of the current state ([VM]). A block is "used" while at least one
 * live sequence's table holds it. `filled_slots` counts, for every used block,
 * the slots up to the furthest token any live sequence keeps in it;
 * `logical_blocks` is the sum over live sequences of their table lengths (the
 * blocks they would need with private copies). */
typedef struct pkv_bm_stats {
  int64_t num_blocks;      /* pool size */
  int64_t free_blocks;     /* blocks on the free stack */
  int64_t used_blocks;     /* num_blocks - free_blocks */
  int64_t shared_blocks;   /* used blocks held by more than one live sequence */
  int64_t filled_slots;    /* slots of used blocks that hold a token */
  int64_t logical_blocks;  /* sum of the live sequences' table lengths */
  int64_t logical_tokens;  /* sum of the live sequences' lengths */
  int64_t live_seqs;       /* live sequences */
  int64_t cow_copies;      /* copy-on-write pairs emitted since creation */
} pkv_bm_stats;

/* Create a manager of `num_blocks` blocks of `block_size` token slots, all
 * free. `seed` fixes the order in which free blocks are first handed out
 * (0: ascending ids; otherwise a permutation drawn from the seed, which
 * scatters a sequence's blocks over the pool). *out receives the manager.
 * PKV_ERR_INVALID_ARG: out NULL, num_blocks or block_size < 1. */
pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, uint64_t seed, pkv_block_manager** out);

/* Release the manager and everything it holds (NULL is ignored). */
void pkv_bm_destroy(pkv_block_manager* bm);

/* New empty sequence (length 0, no blocks). *seq receives its id. */
pkv_status pkv_bm_add_seq(pkv_block_manager* bm, int32_t* seq);

/* New sequence sharing every block of live sequence `parent` ([VM]: a
 * sampled completion or a beam starts as a copy of its parent's table; the
 * reference count of each block goes up by one, no block is copied).
 * *child receives its id. */
pkv_status pkv_bm_fork(pkv_block_manager* bm, int32_t parent, int32_t* child);

/* End live sequence `seq`: its blocks' reference counts go down by one and
 * blocks no longer held by any sequence return to the free stack. */
pkv_status pkv_bm_free_seq(pkv_block_manager* bm, int32_t seq);

/* Reserve cache slots for the next `n` tokens of live sequence `seq` ([VM]).
 * Token t of the sequence lives at slot table[t / block_size] * block_size +
 * t % block_size. A new block is taken only when a token starts one. If the
 * first new token falls into a partly filled last block that another live
 * sequence also holds, that block is first replaced by a fresh private copy:
 * the (source, destination) pair is written to cow_pair[0..1] and *num_cow is
 * set to 1 (else 0); the caller must copy the block's K/V rows (for example
 * with pkv_copy_blocks) before writing the new rows. slots (n entries),
 * cow_pair (2 entries) and num_cow may each be NULL when not wanted.
 * PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the free stack holds fewer
 * blocks than the request needs. n = 0 is a no-op. */
pkv_status pkv_bm_append(pkv_block_manager* bm, int32_t seq, int32_t n, int64_t* slots, int64_t* cow_pair,
                         int32_t* num_cow);

/* One decode step's reservations in one call: counts[i] more tokens for each
 * of the `n` distinct live sequences seqs[i], in order, each exactly as
 * pkv_bm_append would do it (a sibling's copy made earlier in the batch
 * counts: the last holder of a shared block writes into it in place). The
 * slots of all sequences are packed in order into slots (sum of counts
 * entries, may be NULL); the copy-on-write pairs into cow_pairs ([n][2],
 * may be NULL), their number into *num_cow (may be NULL). All or nothing:
 * PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the whole batch does not fit;
 * PKV_ERR_INVALID_ARG when an id repeats, is not live, or a count is < 0. */
pkv_status pkv_bm_append_batch(pkv_block_manager* bm, const int32_t* seqs, const int32_t* counts, int32_t n,
                               int64_t* slots, int64_t* cow_pairs, int32_t* num_cow);

/* One beam-search step of one request ([VM]: beams share long prefixes and
 * are forked and discarded all the time). beams[0..width) are the request's
 * current beams (distinct live sequences); new beam i continues beam
 * beams[parents[i]] (parents[i] in [0, width)) with n_new more tokens.
 * After the call new_beams[i] is the sequence of new beam i: the first new
 * beam (lowest i) of a parent takes over the parent's sequence id, further
 * ones are forks of it, and beams that no new beam continues are ended
 * (their blocks freed unless other sequences hold them). Then every new beam
 * appends n_new tokens in order i = 0, 1, ..., exactly as pkv_bm_append_batch
 * does, so children writing into a shared partly filled block get private
 * copies except the last, which writes in place. slots ([width * n_new],
 * packed by i), cow_pairs ([width][2]) and num_cow as in
 * pkv_bm_append_batch; each may be NULL. All or nothing:
 * PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the step does not fit even
 * after the ended beams' blocks return; PKV_ERR_INVALID_ARG when width < 1,
 * n_new < 0, a beam repeats or is not live, or a parent index is out of
 * range. */
pkv_status pkv_bm_beam_step(pkv_block_manager* bm, const int32_t* beams, const int32_t* parents, int32_t width,
                            int32_t n_new, int32_t* new_beams, int64_t* slots, int64_t* cow_pairs,
                            int32_t* num_cow);

/* One beam-search step of `requests` requests of `width` beams each, in one
 * call (the host side of a batched beam-search decode step). beams and
 * parents are [requests][width]; row r is one request's current beams and
 * the parent index (in [0, width), within row r) of each of its new beams,
 * as in pkv_bm_beam_step. The step runs in three passes over all requests:
 * first every beam that no new beam continues is ended, then every new beam
 * takes its sequence id (a parent's first child keeps the parent's id,
 * further children are forks), then every new beam appends n_new tokens in
 * row-major order (r, i), exactly as pkv_bm_append_batch over that order.
 * Per request this gives the same tables as pkv_bm_beam_step; across
 * requests the physical block and sequence ids handed out may differ from
 * calling it once per request, because every request's ended blocks return
 * before any request appends. new_beams is [requests][width]; slots
 * ([requests * width * n_new], packed row-major), cow_pairs
 * ([requests * width][2]) and num_cow as in pkv_bm_append_batch;
 * shared_blocks ([requests]) receives, per request, the number of leading
 * blocks its new beams all share (pkv_bm_common_prefix). Each output but
 * new_beams may be NULL. All or nothing across all requests:
 * PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the whole step does not fit
 * after the ended beams' blocks return; PKV_ERR_INVALID_ARG when
 * requests < 0, width < 1, n_new < 0, a beam repeats anywhere in beams or is
 * not live, or a parent index is out of range. requests = 0 is a no-op. */
pkv_status pkv_bm_beam_step_many(pkv_block_manager* bm, const int32_t* beams, const int32_t* parents,
                                 int32_t requests, int32_t width, int32_t n_new, int32_t* new_beams, int64_t* slots,
                                 int64_t* cow_pairs, int32_t* num_cow, int32_t* shared_blocks);

/* Length (tokens) and table length (blocks) of live sequence `seq`. */
pkv_status pkv_bm_seq_info(const pkv_block_manager* bm, int32_t seq, int64_t* length, int32_t* num_blocks);

/* Block-table rows and context lengths of `n` live sequences, in the layout
 * the decode entry points take: block_tables[i][j] (row length max_blocks,
 * int32) = physical block of logical block j of seqs[i], -1 past the end of
 * its table; context_lens[i] = its length. PKV_ERR_INVALID_ARG when a table
 * is longer than max_blocks or a length exceeds INT32_MAX (nothing written). */
pkv_status pkv_bm_export(const pkv_block_manager* bm, const int32_t* seqs, int32_t n, int32_t max_blocks,
                         int32_t* block_tables, int32_t* context_lens);

/* Number of leading block-table entries that the `n` live sequences seqs[]
 * all hold in common (the same physical blocks): the shared prefix, in
 * blocks, that pkv_paged_attention_decode_grouped takes for one group. */
pkv_status pkv_bm_common_prefix(const pkv_block_manager* bm, const int32_t* seqs, int32_t n, int32_t* blocks);

/* Current counters (see pkv_bm_stats). */
pkv_status pkv_bm_get_stats(const pkv_block_manager* bm, pkv_bm_stats* stats);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCK_MANAGER_H_ */
