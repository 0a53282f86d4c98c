/*
 * pkv_pool.h -- host-side block pool that generates the inputs of libpkv.
 *
 * Plain C99, no CUDA.  The pool never touches K/V bytes: it decides which
 * physical block ids a request's logical blocks map to, produces the slot
 * mapping consumed by pkv_kv_append, the (src, dst) pairs consumed by
 * pkv_kv_block_copy, and the dense block tables consumed by the attention
 * calls.  It is never on a timed device path.
 *
 * Sources:
 *   "M5.3 - KV Memory Layout and Exact Reuse", 0x04B (refcount = committed
 *   request references; a block with no reference returns to the free list),
 *   0x04E (append has three physical paths: offset 0 takes a new block, a
 *   private tail is written in place, a shared tail is copied on write first),
 *   0x05A (copy-on-write copies the valid tail rows), 0x0AB (ragged requests in
 *   a dense [B, n_max] table).
 *   "Cache Concepts: Prefix Matching vs. Storage": the free FIFO of the block
 *   pool, and the slot invariant table[req, pos // P] * P + pos % P computed
 *   with int64 page ids.
 *   "7. Memory Management and Local Model State", "Sharing and copy-on-write".
 *
 * Ownership: every object is created and destroyed by the caller through the
 * functions below.  Not thread-safe; one pool per thread.
 *
 * Errors: functions returning int give 0 on success and a negative value on
 * failure (-1 bad argument, -2 pool exhausted); nothing is modified on
 * failure.
 */
#ifndef PKV_POOL_H
#define PKV_POOL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_pool pkv_pool;
typedef struct pkv_seq pkv_seq;

/* A pool of num_blocks block ids 0..num_blocks-1, each holding block_size
 * token rows.  The free FIFO starts in id order, or in a seeded
 * Fisher-Yates order (splitmix64 stream seeded with `seed`) when shuffle != 0.
 * Returns NULL on a bad argument or out of host memory. */
pkv_pool* pkv_pool_create(int64_t num_blocks, int32_t block_size,
                          uint64_t seed, int shuffle);
void pkv_pool_destroy(pkv_pool* pool);

int64_t pkv_pool_num_blocks(const pkv_pool* pool);
int32_t pkv_pool_block_size(const pkv_pool* pool);
int64_t pkv_pool_num_free(const pkv_pool* pool);

/* Pop the FIFO head with refcount 1; -2 if the pool is exhausted. */
int32_t pkv_pool_alloc(pkv_pool* pool);
/* Current refcount of a block id (-1 for an id outside the pool). */
int32_t pkv_pool_refcount(const pkv_pool* pool, int32_t block);
int pkv_pool_incref(pkv_pool* pool, int32_t block);
/* Drop one reference; at zero the block goes to the FIFO tail. */
int pkv_pool_decref(pkv_pool* pool, int32_t block);

/* A request's block list and committed length. */
pkv_seq* pkv_seq_create(pkv_pool* pool);
/* A child sharing every block of parent (each block's refcount + 1). */
pkv_seq* pkv_seq_fork(pkv_pool* pool, const pkv_seq* parent);
/* Drop every block reference of seq and free it. */
void pkv_seq_release(pkv_pool* pool, pkv_seq* seq);

int64_t pkv_seq_len(const pkv_seq* seq);
int32_t pkv_seq_num_blocks(const pkv_seq* seq);
/* Physical id of logical block j (-1 if j is out of range). */
int32_t pkv_seq_block(const pkv_seq* seq, int32_t j);

/* Append n tokens to seq.  slots_out[i] receives the slot id of token
 * len + i.  If the first token lands in a shared tail block, the tail is
 * copied on write: a new block is allocated, the pair (old, new) is written to
 * cow_pair_out[0..1] and *cow_count is set to 1 (else 0); the caller must run
 * that copy on the device before the append.  Returns -2 without changing
 * anything if the pool lacks the blocks. */
int pkv_seq_append_tokens(pkv_pool* pool, pkv_seq* seq, int64_t n,
                          int64_t* slots_out, int64_t* cow_pair_out,
                          int32_t* cow_count);

/* Dense [num_seqs, max_blocks] int32 table, padded with -1, and the int32
 * context lengths.  Returns -1 if a sequence has more than max_blocks
 * blocks. */
int pkv_build_block_tables(pkv_seq* const* seqs, int32_t num_seqs,
                           int32_t max_blocks, int32_t* tables_out,
                           int32_t* lens_out);

#ifdef __cplusplus
}
#endif
#endif
