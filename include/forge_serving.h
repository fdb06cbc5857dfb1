/*
 * forge_serving.h — the KV block pool and the continuous-batching decode
 * step driver that feed forge_paged.h's append and decode calls.
 *
 * What this covers (page title, section):
 *   - forge-engine README, "What it implements", row "KV cache": a paged
 *     block allocator with deterministic cleanup; row "Scheduling":
 *     continuous, bounded, token-budgeted batching; the sample run's report
 *     ends with zero KV blocks still allocated.
 *   - "Make the Engine Talk", 1.2: each decode pass adds exactly one token
 *     to every running sequence's cache.
 *
 * The pages name these properties and give no algorithm.  The policies
 * below are this library's reading, stated so they can be checked:
 *
 * Pool (forge_kv_pool).  NB blocks of block_size tokens, ids 0..NB-1, held
 * on a free stack.  A fresh pool hands out 0, 1, 2, ...; a released block
 * goes back on top, so it is the next one handed out; a sequence's blocks
 * are pushed back last block first, so releasing a sequence and adding an
 * equally long one hands out the same ids in the same order.  A sequence
 * owns ceil(tokens / block_size) blocks; its table row lists them in token
 * order.  The pool never reads or writes KV data: it only decides block
 * ids.  Identical call sequences give identical ids on every host.
 *
 * Batch (forge_batch).  A fixed number of rows (the decode batch width).
 * Requests are queued by forge_batch_submit, in order.  Each
 * forge_batch_step performs, in this order:
 *   1. retire: every row whose sequence has run its max_new_tokens decode
 *      steps frees its row and all its blocks;
 *   2. preempt: while the running rows need more new blocks for this step's
 *      token than the pool has free, the most recently admitted running
 *      sequence is released and put back at the FRONT of the queue with
 *      prompt = its current length (its cache is rebuilt on re-admission)
 *      and its remaining decode steps unchanged;
 *   3. admit, first come first served: the queue's head is admitted into the
 *      lowest-numbered free row while (a) a row is free, (b) the pool can
 *      hold its prompt plus this step's token on top of what the running
 *      rows need, and (c) the prompt tokens admitted this step stay within
 *      token_budget; a prompt longer than the whole budget is admitted only
 *      as the step's first admission.  Admission stops at the first request
 *      that does not fit (no overtaking).  The caller writes an admitted
 *      sequence's prompt K/V (prefill) into its blocks;
 *   4. grow: every running row takes one new token at position len (a new
 *      block when len % block_size == 0); its context length becomes len+1
 *      and its slot is table[len / block_size] * block_size + len % block_size.
 * After the last request retires the pool holds zero allocated blocks.
 *
 * forge_batch_apply uploads one step's changes (per row: the new length
 * and the block taken, if any; per admitted row: its whole table row; every
 * running row whole when the step before was never applied) and one kernel
 * updates the caller's device block_tables and context_lens in
 * place and writes slot_mapping from the device table.  Rows without a
 * sequence get length 0 and slot -1, which forge_paged_kv_append skips and
 * forge_paged_gqa_decode answers with zeros.
 *
 * Ownership: the caller owns the device tensors; a forge_batch owns a small
 * ring of pinned host and device staging buffers (freed by
 * forge_batch_destroy).  The pool must outlive every batch that uses it,
 * and a pool serves one batch at a time.  All functions are thread-safe.
 * Host-side functions make no CUDA call.
 */
#ifndef FORGE_SERVING_H
#define FORGE_SERVING_H

#include "forge_paged.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct forge_kv_pool forge_kv_pool;
typedef struct forge_batch forge_batch;

/* A pool of num_blocks blocks of block_size tokens; no sequence may own more
 * than max_blocks_per_seq blocks (the width of a block-table row).  NULL for
 * num_blocks < 0, block_size <= 0, max_blocks_per_seq <= 0 or no memory. */
FORGE_API forge_kv_pool *forge_kv_pool_create(int32_t num_blocks, int32_t block_size,
                                              int32_t max_blocks_per_seq);
FORGE_API void forge_kv_pool_destroy(forge_kv_pool *pool);

/* Register sequence seq_id holding num_tokens tokens (its blocks are taken
 * now).  FORGE_ERR_VALUE: seq_id already present, num_tokens < 0, or more
 * than max_blocks_per_seq blocks needed; FORGE_ERR_CAPACITY: not enough free
 * blocks (nothing taken). */
FORGE_API int forge_kv_pool_add(forge_kv_pool *pool, int64_t seq_id, int32_t num_tokens);

/* Add one token to seq_id; *slot_out (may be NULL) = its cache slot
 * (block * block_size + offset).  FORGE_ERR_VALUE: unknown seq_id or the
 * table row is full; FORGE_ERR_CAPACITY: a new block is needed and none is
 * free (nothing changed). */
FORGE_API int forge_kv_pool_grow(forge_kv_pool *pool, int64_t seq_id, int64_t *slot_out);

/* Return all of seq_id's blocks to the pool.  FORGE_ERR_VALUE: unknown id. */
FORGE_API int forge_kv_pool_release(forge_kv_pool *pool, int64_t seq_id);

/* Free / allocated block counts; -1 for a NULL pool. */
FORGE_API int32_t forge_kv_pool_free_blocks(const forge_kv_pool *pool);
FORGE_API int32_t forge_kv_pool_used_blocks(const forge_kv_pool *pool);

/* seq_id's token count and block list (blocks_out may be NULL; else it holds
 * capacity entries, FORGE_ERR_SHAPE when too few). */
FORGE_API int forge_kv_pool_sequence(const forge_kv_pool *pool, int64_t seq_id, int32_t *len_out,
                                     int32_t *blocks_out, int32_t capacity, int32_t *nblocks_out);

/* A decode batch of `rows` rows over `pool`; at most token_budget prompt
 * tokens are admitted per step (see 3. above).  NULL for a NULL pool,
 * rows <= 0, token_budget <= 0, or no memory. */
FORGE_API forge_batch *forge_batch_create(forge_kv_pool *pool, int32_t rows, int32_t token_budget);

/* Waits for this batch's staging copies, frees them and releases every
 * sequence the batch still holds back to the pool. */
FORGE_API void forge_batch_destroy(forge_batch *batch);

/* Queue a request.  FORGE_ERR_VALUE: seq_id already queued or running,
 * prompt_tokens < 0, max_new_tokens < 1, or prompt + max_new longer than a
 * table row; FORGE_ERR_CAPACITY: it could not fit in the pool even alone. */
FORGE_API int forge_batch_submit(forge_batch *batch, int64_t seq_id, int32_t prompt_tokens,
                                 int32_t max_new_tokens);

typedef struct {
    int32_t running;     /* rows holding a sequence after the step */
    int32_t waiting;     /* requests still queued */
    int32_t admitted;    /* sequences admitted by the step (their prompts need prefill) */
    int32_t retired;     /* sequences that finished at the start of the step */
    int32_t preempted;   /* sequences sent back to the queue by the step */
    int32_t free_blocks; /* pool blocks free after the step */
    int64_t tokens;      /* sum of the rows' context lengths after the step */
} forge_batch_report;

/* One host step (retire, preempt, admit, grow).  report may be NULL.
 * Host only: the device sees the step after forge_batch_apply. */
FORGE_API int forge_batch_step(forge_batch *batch, forge_batch_report *report);

/* The last step's row state, each array [rows] or NULL: the sequence in the
 * row (-1 = none), its context length (0 = none), its new token's slot
 * (-1 = none) and the block the step took for it (-1 = none). */
FORGE_API int forge_batch_rows(const forge_batch *batch, int64_t *seq_ids, int32_t *context_lens,
                               int64_t *slots, int32_t *new_blocks);

#define FORGE_BATCH_ADMITTED 0  /* row = the row it took, tokens = its prompt length */
#define FORGE_BATCH_RETIRED 1   /* row = the row it left, tokens = its final length */
#define FORGE_BATCH_PREEMPTED 2 /* row = the row it left, tokens = its length (new prompt) */

/* The last step's events of one kind, in the order they happened.  Writes
 * up to `capacity` entries into each non-NULL array and returns how many
 * events there were (which may exceed capacity), or a negative status. */
FORGE_API int forge_batch_events(const forge_batch *batch, int kind, int32_t capacity,
                                 int64_t *seq_ids, int32_t *rows, int32_t *tokens);

/*
 * Apply the last step on the device, on `stream`:
 *   block_tables  int32 [rows, MB], MB >= the pool's max_blocks_per_seq,
 *                 inner stride 1: rows admitted by the step are rewritten
 *                 whole (entries past the sequence's blocks set to -1), and
 *                 so is every running row if the previous step was never
 *                 applied; other running rows get the block their new token
 *                 opened.  Rows without a sequence are left as they are;
 *   context_lens  int32 [rows], contiguous: every row's length (0 = none);
 *   slot_mapping  int64 [rows], contiguous: per row
 *                 block_tables[r][(len-1)/bs] * bs + (len-1) % bs, read from
 *                 the device table after the update, or -1 for an empty row.
 * The step's description goes through a pinned staging buffer with one
 * cudaMemcpyAsync, then one single-CTA kernel; the call does not wait for
 * the device except when a staging buffer (one of a ring of 4) is reused
 * before the apply kernel that last read it has ended.  Applies of one batch
 * may go to different streams.  Not capturable into a CUDA graph (FORGE_ERR_UNSUPPORTED while
 * the stream captures).  A batch stays on the device of its first apply
 * (FORGE_ERR_VALUE on another).  FORGE_ERR_DTYPE / FORGE_ERR_SHAPE on
 * tensors that do not match, FORGE_ERR_CUDA on a failed CUDA call.
 */
FORGE_API int forge_batch_apply(forge_batch *batch, forge_tensor *block_tables, forge_tensor *context_lens,
                                forge_tensor *slot_mapping, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FORGE_SERVING_H */
