/*
 * pkv_pool.c -- host block pool: free FIFO, refcounts, append planning.
 * Generates inputs only; see include/pkv_pool.h for the contract.
 */
#include "pkv_pool.h"

#include <stdlib.h>
#include <string.h>

struct pkv_pool {
  int64_t num_blocks;
  int32_t block_size;
  int32_t* refcount; /* per block id */
  int32_t* fifo;     /* ring buffer of free ids */
  int64_t head, count;
};

struct pkv_seq {
  int64_t len;
  int32_t nblocks, cap;
  int32_t* blocks;
};

/* splitmix64: a published 64-bit mixing generator (Steele, Lea, Flood). */
static uint64_t splitmix64(uint64_t* state) {
  uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

pkv_pool* pkv_pool_create(int64_t num_blocks, int32_t block_size,
                          uint64_t seed, int shuffle) {
  if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return NULL;
  pkv_pool* p = (pkv_pool*)calloc(1, sizeof(pkv_pool));
  if (!p) return NULL;
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->refcount = (int32_t*)calloc((size_t)num_blocks, sizeof(int32_t));
  p->fifo = (int32_t*)malloc((size_t)num_blocks * sizeof(int32_t));
  if (!p->refcount || !p->fifo) {
    free(p->refcount);
    free(p->fifo);
    free(p);
    return NULL;
  }
  for (int64_t i = 0; i < num_blocks; ++i) p->fifo[i] = (int32_t)i;
  if (shuffle) {
    uint64_t st = seed;
    for (int64_t i = num_blocks - 1; i > 0; --i) {
      int64_t j = (int64_t)(splitmix64(&st) % (uint64_t)(i + 1));
      int32_t t = p->fifo[i];
      p->fifo[i] = p->fifo[j];
      p->fifo[j] = t;
    }
  }
  p->head = 0;
  p->count = num_blocks;
  return p;
}

void pkv_pool_destroy(pkv_pool* pool) {
  if (!pool) return;
  free(pool->refcount);
  free(pool->fifo);
  free(pool);
}

int64_t pkv_pool_num_blocks(const pkv_pool* pool) { return pool->num_blocks; }
int32_t pkv_pool_block_size(const pkv_pool* pool) { return pool->block_size; }
int64_t pkv_pool_num_free(const pkv_pool* pool) { return pool->count; }

int32_t pkv_pool_alloc(pkv_pool* pool) {
  if (pool->count == 0) return -2;
  int32_t id = pool->fifo[pool->head];
  pool->head = (pool->head + 1) % pool->num_blocks;
  pool->count -= 1;
  pool->refcount[id] = 1;
  return id;
}

int32_t pkv_pool_refcount(const pkv_pool* pool, int32_t block) {
  if (block < 0 || block >= pool->num_blocks) return -1;
  return pool->refcount[block];
}

int pkv_pool_incref(pkv_pool* pool, int32_t block) {
  if (block < 0 || block >= pool->num_blocks || pool->refcount[block] <= 0) return -1;
  pool->refcount[block] += 1;
  return 0;
}

int pkv_pool_decref(pkv_pool* pool, int32_t block) {
  if (block < 0 || block >= pool->num_blocks || pool->refcount[block] <= 0) return -1;
  pool->refcount[block] -= 1;
  if (pool->refcount[block] == 0) {
    int64_t tail = (pool->head + pool->count) % pool->num_blocks;
    pool->fifo[tail] = block;
    pool->count += 1;
  }
  return 0;
}

static int seq_reserve(pkv_seq* s, int32_t n) {
  if (n <= s->cap) return 0;
  int32_t cap = s->cap ? s->cap : 8;
  while (cap < n) cap *= 2;
  int32_t* b = (int32_t*)realloc(s->blocks, (size_t)cap * sizeof(int32_t));
  if (!b) return -1;
  s->blocks = b;
  s->cap = cap;
  return 0;
}

pkv_seq* pkv_seq_create(pkv_pool* pool) {
  (void)pool;
  return (pkv_seq*)calloc(1, sizeof(pkv_seq));
}

pkv_seq* pkv_seq_fork(pkv_pool* pool, const pkv_seq* parent) {
  pkv_seq* s = (pkv_seq*)calloc(1, sizeof(pkv_seq));
  if (!s) return NULL;
  if (seq_reserve(s, parent->nblocks) != 0) {
    free(s);
    return NULL;
  }
  for (int32_t j = 0; j < parent->nblocks; ++j) {
    s->blocks[j] = parent->blocks[j];
    pkv_pool_incref(pool, parent->blocks[j]);
  }
  s->nblocks = parent->nblocks;
  s->len = parent->len;
  return s;
}

void pkv_seq_release(pkv_pool* pool, pkv_seq* seq) {
  if (!seq) return;
  for (int32_t j = 0; j < seq->nblocks; ++j) pkv_pool_decref(pool, seq->blocks[j]);
  free(seq->blocks);
  free(seq);
}

int64_t pkv_seq_len(const pkv_seq* seq) { return seq->len; }
int32_t pkv_seq_num_blocks(const pkv_seq* seq) { return seq->nblocks; }
int32_t pkv_seq_block(const pkv_seq* seq, int32_t j) {
  return (j < 0 || j >= seq->nblocks) ? -1 : seq->blocks[j];
}

int pkv_seq_append_tokens(pkv_pool* pool, pkv_seq* seq, int64_t n,
                          int64_t* slots_out, int64_t* cow_pair_out,
                          int32_t* cow_count) {
  if (n < 0) return -1;
  const int64_t P = pool->block_size;
  *cow_count = 0;
  if (n == 0) return 0;
  /* Blocks this append needs: new blocks past the current capacity, plus one
   * private copy if the first token falls into a shared partial tail. */
  const int64_t first_off = seq->len % P;
  const int tail_shared = first_off != 0 && seq->nblocks > 0 &&
                          pool->refcount[seq->blocks[seq->nblocks - 1]] > 1;
  const int64_t need_blocks = (seq->len + n + P - 1) / P;
  const int64_t new_blocks = need_blocks - seq->nblocks + (tail_shared ? 1 : 0);
  if (new_blocks > pool->count) return -2;
  if (need_blocks > INT32_MAX || seq_reserve(seq, (int32_t)need_blocks) != 0) return -1;

  if (tail_shared) {
    /* copy-on-write of the shared tail before the first divergent append */
    int32_t old = seq->blocks[seq->nblocks - 1];
    int32_t fresh = pkv_pool_alloc(pool);
    cow_pair_out[0] = old;
    cow_pair_out[1] = fresh;
    *cow_count = 1;
    seq->blocks[seq->nblocks - 1] = fresh;
    pkv_pool_decref(pool, old);
  }
  for (int64_t i = 0; i < n; ++i) {
    const int64_t pos = seq->len + i;
    const int64_t j = pos / P;
    if (pos % P == 0) {
      /* offset 0: a new block */
      seq->blocks[seq->nblocks] = pkv_pool_alloc(pool);
      seq->nblocks += 1;
    }
    /* slot = table[pos // P] * P + pos % P, with the id widened to int64 */
    slots_out[i] = (int64_t)seq->blocks[j] * P + pos % P;
  }
  seq->len += n;
  return 0;
}

int pkv_build_block_tables(pkv_seq* const* seqs, int32_t num_seqs,
                           int32_t max_blocks, int32_t* tables_out,
                           int32_t* lens_out) {
  for (int32_t r = 0; r < num_seqs; ++r) {
    const pkv_seq* s = seqs[r];
    if (s->nblocks > max_blocks || s->len > INT32_MAX) return -1;
    int32_t* row = tables_out + (int64_t)r * max_blocks;
    for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < s->nblocks ? s->blocks[j] : -1;
    lens_out[r] = (int32_t)s->len;
  }
  return 0;
}
